// K1: token-parallel prep kernel of the KDA chunked forward.
//
// One CTA per (chunk of 64 tokens, head), heads fastest, two CTAs per SM. It does the work of
// the FlashKDA "K1" stage (FlashKDA page, section "커널 퓨전(Kernel Fusion)
// 전략의 분리": gate activation, L2 normalisation, decay and the triangular
// inverse, all parallel over tokens) and the cuLA "kda chunk intra" stage
// (cuLA launch blog, section "Status & Roadmap"), and hands the recurrence
// kernel, per (chunk, head), everything it needs besides v, each in the layout of
// its shared-memory operand so that one bulk copy places it:
//   * M = [ -Tb ; P Tb ] (128 x 64 fp16, rows in 128-byte-swizzled order),
//       Tb = (I + A)^{-1} diag(beta)
//       A_ij = beta_i sum_k khat_ik khat_jk 2^{G_ik - G_jk}   (j < i)
//       P_ij = scale  sum_k qhat_ik khat_jk 2^{G_ik - G_jk}   (j <= i)
//   * khat Gamma, khat Gamma_last / Gamma and scale qhat Gamma (64 x K fp16 each, as
//     images of 64-channel panels of 128-byte swizzled token rows) and
//     Gamma_last (K fp32),
// with G the in-chunk inclusive cumulative base-2 log decay and Gamma = 2^G. The output
// scale sits in P and in the q image, so the recurrence kernel's O rows come out scaled.
// With these the recurrence kernel forms w = Tb (khat Gamma), u = Tb v, P w and
// P u as plain products. The log decay per token and channel is
// la2 = lb log2(e) sigmoid(exp(A_log)(g + dt_bias)).
//
// Norms. khat = k / |k| and qhat = q / |q| are per-row scalings, so they are
// taken out of the A/P sums: the products run on the raw bf16 values and the
// read back scales entry (i, j) by beta_i |k_i|^-1 |k_j|^-1 (A) or
// |q_i|^-1 |k_j|^-1 (P). The norms are computed first, for the hand-off.
//
// Exponent range. With lower_bound >= -5 one token decays by at most e^-5, so
// over 16 tokens |G| <= 80 ln-units (about 115.4 in base 2), which fits in
// fp32. Each 16-row block J keeps its own reference (the decay before the
// block). With alpha = 2^{la2} per token and channel:
//   X_i  = prod of alpha over the block's rows up to and including i   (<= 1)
//   Ys_j = prod of alpha over the block's rows after j                 (<= 1)
//   Y_j  = 2^{-Gb_j} = Ys_j 2^{-B_J}                                   (>= 1)
// with Gb the block-local inclusive cumulative sum and B_J the whole-block sum.
// For j in block J < i in block I,  2^{G_i - G_j} = X_i Ys_j c_IJ, where
// c_IJ = 2^{sum of the blocks strictly between J and I} <= 1: no factor
// overflows, and one only underflows when the true product is already below the
// fp32 range. Diagonal blocks use X_i Y_j (<= 2^115.4). This is the
// "intra-chunk rescaling" that large chunks need (FlashKDA page, section
// "Flash Linear Attention과 비교").
//
// All block products of A and P come from ONE tensor-core product (tcgen05,
// tf32 operands, fp32 accumulators in tensor memory), accumulated over two
// halves of the channels so that the operands fit twice per SM:
//   D = [k X ; q X] (128 x K)  x  [k Y ; k Ys_{0..2} ; k Ys_0 2^{B_1} ; k Ys_1 2^{B_2} ; k Ys_0 c_30]^T
// Columns 0-63 give the diagonal blocks, 64-111 the blocks next to the
// diagonal, 112-159 the three blocks further out. The unit lower triangular
// inverse T = (I + A)^{-1} is blocked: the two 32 x 32 diagonal halves by forward
// substitution in fp32 (one thread per column), then the lower-left 32 x 32 block
// -T_[23] A_[23][01] T_[01] as two small tensor-core products (fp16 operands, fp32
// accumulators): Z = A_[23][01] T_[01], then (T_[23] Z)^T = Z^T T_[23]^T. All of T lands, scaled as
// Tb = T diag(beta), in the fp16 operand of M = [-I ; P] Tb, a third tensor-core
// product (128 x 64 x 64).
#include <cstddef>
#include <type_traits>

#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {

constexpr int kPrepThreads = 256;
constexpr int kOpBRows = 160;                 // J-side operand rows
constexpr uint32_t kPrepTmemCols = 256;       // D_AP: cols 0..159; D_M: cols 192..255
constexpr long long kPrepWaitLimit = 4000000000LL;

// Shared memory (byte offsets from the 1024-aligned base). The operands hold one half of the
// channels (64) at a time, as tf32 in 128-byte-swizzled panels of 32 channels.
struct PrepLayout {
  static constexpr uint32_t opA = 0;                            // [k X ; q X]: 2 panels x 128 rows x 128 B
  static constexpr uint32_t opB = opA + 2 * 128 * 128;          // J side:      2 panels x 160 rows x 128 B
  static constexpr uint32_t opEnd = opB + 2 * kOpBRows * 128;
  // after the A/P product the operands are dead. In their place: A's two diagonal halves
  // transposed (fp32 [2 x 32][36]), the fp16 operands of the lower-left merge (32 rows of 128-byte
  // swizzled rows each, 32 columns used), the Tb^T operand and the [-I ; P] operand.
  static constexpr int LDQ = 36;                                // 16-byte aligned rows of 32 + 4
  static constexpr uint32_t matAt = 0;
  static constexpr uint32_t opAll = 10 * 1024;                  // A_[23][01]        (A of Z = A T_[01])
  static constexpr uint32_t opT01 = 14 * 1024;                  // T_[01]^T, K-major (B of Z)
  static constexpr uint32_t opT23 = 18 * 1024;                  // T_[23]^T, MN-major (B of Z^T T_[23]^T)
  static constexpr uint32_t opZ = 22 * 1024;                    // Z^T, MN-major      (A of Z^T T_[23]^T)
  static constexpr uint32_t opT = 26 * 1024;                    // Tb^T:      64 rows x 128 B (fp16)
  static constexpr uint32_t opM = 34 * 1024;                    // [-I ; P]: 128 rows x 128 B (fp16)
  static constexpr uint32_t mstage = 0;                         // M, staged for its copy-out: 128 rows x 128 B
  static constexpr uint32_t end = (opM + 128 * 128 > opEnd) ? opM + 128 * 128 : opEnd;
  static_assert(matAt + 64 * LDQ * 4 <= opAll, "transposed A overlaps the merge operands");
  static_assert(opT + 64 * 128 <= opM, "Tb^T operand overlaps the [-I ; P] operand");
  // the merge's A operands span 128 rows (K-major A_[23][01]: 128 rows of 128 B; MN-major Z^T: a
  // second 64-row panel 8 KB on, 32 K rows of 128 B): rows 32..127 are other data of this block,
  // whose products land in tensor-memory lanes that are never read
  static_assert(opAll + 128 * 128 <= end && opZ + 8192 + 32 * 128 <= end, "merge operand span");
  static_assert(end >= opEnd, "layout end");
  static_assert(mstage + 128 * 128 <= opT, "the M staging copy overlaps the M product's operands");
};

struct PrepMisc {
  uint64_t bar;
  uint32_t tmem_slot;
  int err;
  // 16-byte aligned: the norms are read four rows at a time
  alignas(16) float beta[kChunk];
  alignas(16) float kn[kChunk];
  alignas(16) float qn[kChunk];
  // per (4-row sub-block j, channel quad): the sum of la2 over the sub-block, then, in place, the
  // exclusive prefix over the sub-blocks (E[j] = sum over rows < 4 j; E[16] = the whole chunk)
  float4 epre[17][16];
};
static_assert(offsetof(PrepMisc, kn) % 16 == 0 && offsetof(PrepMisc, qn) % 16 == 0, "float4 reads of the norms");

__device__ __forceinline__ uint32_t ldg_u32(const __nv_bfloat16 *p) {
  return __ldg(reinterpret_cast<const unsigned int *>(p));
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ float2 ex2_2(float2 x) { return make_float2(ex2_approx(x.x), ex2_approx(x.y)); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
// tf32 operands: the tensor core reads the top 19 bits of each 32-bit word and drops the low 13,
// so adding half a tf32 unit in the last place first makes that truncation round to nearest
// (ties away from zero) in one integer add.
__device__ __forceinline__ float tf32_rn(float x) { return __uint_as_float(__float_as_uint(x) + 0x1000u); }
// Four channels of one row, as two packed pairs.
struct F4 {
  float2 lo, hi;
};
__device__ __forceinline__ F4 mul4(F4 a, F4 b) { return {__fmul2_rn(a.lo, b.lo), __fmul2_rn(a.hi, b.hi)}; }
__device__ __forceinline__ F4 add4(F4 a, F4 b) { return {__fadd2_rn(a.lo, b.lo), __fadd2_rn(a.hi, b.hi)}; }
__device__ __forceinline__ F4 ex2_4(F4 x) { return {ex2_2(x.lo), ex2_2(x.hi)}; }
__device__ __forceinline__ F4 splat4(float v) { return {make_float2(v, v), make_float2(v, v)}; }
__device__ __forceinline__ F4 f4_of(float4 v) { return {make_float2(v.x, v.y), make_float2(v.z, v.w)}; }
__device__ __forceinline__ float4 float4_of(F4 v) { return make_float4(v.lo.x, v.lo.y, v.hi.x, v.hi.y); }
__device__ __forceinline__ F4 bf4_to_f4(uint2 u) { return {bf2_to_f2(u.x), bf2_to_f2(u.y)}; }
__device__ __forceinline__ uint2 ldg_u64(const __nv_bfloat16 *p) { return __ldg(reinterpret_cast<const uint2 *>(p)); }
// two floats as an fp16 pair (round to nearest), low half first
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}
// four tf32-rounded values, one 16-byte store
__device__ __forceinline__ void st_tf32x4(unsigned char *p, F4 v) {
  *reinterpret_cast<float4 *>(p) = make_float4(tf32_rn(v.lo.x), tf32_rn(v.lo.y), tf32_rn(v.hi.x), tf32_rn(v.hi.y));
}
// four fp16 values, one 8-byte store
__device__ __forceinline__ void st_half4(unsigned char *p, F4 v) {
  const __half2 a = __float22half2_rn(v.lo), b = __float22half2_rn(v.hi);
  *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
}

// VF: the variant flags that change this kernel's code: kGatePerHead (one gate per token and
// head), kBetaF32 (fp32 beta logits), kExp2Poly (the per-token decays 2^la on the FMA pipe).
// Separate instantiations, so that the default kernel carries no code for them.
template <int K, uint32_t VF>
__global__ void __launch_bounds__(kPrepThreads, 2)
prep_kernel(const Problem p) {
  constexpr bool PH = (VF & kGatePerHead) != 0, BF32 = (VF & kBetaF32) != 0, POLY = (VF & kExp2Poly) != 0;
  using Lay = PrepLayout;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so that the
  // compiler keeps every access in the shared address space
  unsigned char *sm = smem_raw + ((1024u - (umma::smem_u32(smem_raw) & 1023u)) & 1023u);
  PrepMisc &ms = *reinterpret_cast<PrepMisc *>(sm + Lay::end);
  float (*matAt)[Lay::LDQ] = reinterpret_cast<float (*)[Lay::LDQ]>(sm + Lay::matAt);     // -A[32 h + c][32 h + r] at [32 h + r][c]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // block = chunk * H + head: the blocks of one wave take whole token rows across the heads
  const long long c = blockIdx.x / (unsigned)p.H;
  const int h = (int)(blockIdx.x - c * p.H);
  // The recurrence kernel may be scheduled once every CTA of this grid has started (its CTAs wait
  // for this grid to finish); this grid in turn waits here for the schedule kernel, when it was
  // launched to overlap it.
  pdl_launch_dependents();
  pdl_wait();
  if (p.flag && *p.flag != kDevOk) return;
  const long long total = p.cu ? (long long)p.chunk_off[p.N] : (long long)p.B * p.nc_fixed;
  if (c >= total) return;
  const int s = chunk_to_seq(p, c);
  const SeqInfo si = seq_info(p, s);
  const int n = (int)(c - si.chunk0);
  const int t0 = si.t0 + n * kChunk;
  const int len = min(kChunk, si.len - n * kChunk);
  const uint32_t sbase = umma::smem_u32(sm);

  // Elementwise unit of this thread: channel quad cq = lane % 16 of the current half (channels
  // 4 cq .. 4 cq + 3) and the 4-row sub-block sb4 = 2 warp + lane / 16 (rows 4 sb4 .. + 3), which
  // is sub-block sbi = sb4 % 4 of the 16-row block J = sb4 / 4. A warp covers two rows of 64
  // channels, so every global access of a row is one 128-byte line.
  const int cq = lane & 15, sb4 = 2 * warp + (lane >> 4), J = sb4 >> 2, sbi = sb4 & 3;
  const int row0 = 4 * sb4;
  const int nrows = max(0, min(4, len - row0));
  const float lbl2 = p.lb * kLog2e;
  const long long rstride = (long long)p.H * K;  // elements between consecutive tokens
  const long long rbase = tok_row(p, si.b, t0 + row0, h) * K;
  const uint32_t r7 = (uint32_t)(sb4 & 1) << 2;  // (row0 + r) & 7 == r7 + r
  // Swizzled byte offsets of this thread's quad in its rows, computed once:
  //   tf32 operand (32 channels per 128-byte row): the quad is one 16-byte chunk;
  //   16-bit image (64 channels per 128-byte row): the quad is half a chunk.
  uint32_t op_x[4], img_x[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    op_x[r] = (uint32_t)(row0 + r) * 128u + ((((uint32_t)cq & 7u) ^ (r7 + (uint32_t)r)) << 4);
    img_x[r] = (uint32_t)(row0 + r) * 128u + (((((uint32_t)cq >> 1) ^ (r7 + (uint32_t)r)) << 4) | (((uint32_t)cq & 1u) << 3));
  }
  unsigned char *const opA_q = sm + Lay::opA + (uint32_t)(cq >> 3) * (128 * 128);
  unsigned char *const opB_q = sm + Lay::opB + (uint32_t)(cq >> 3) * (kOpBRows * 128);
  // operand row `base + row0 + r` (base a multiple of 8) of this thread's quad
  auto opA_at = [&](int base, int r) -> unsigned char * { return opA_q + (uint32_t)base * 128u + op_x[r]; };
  auto opB_at = [&](int base, int r) -> unsigned char * { return opB_q + (uint32_t)base * 128u + op_x[r]; };

  // Rows of the sub-block past the sequence end are read from its last valid row (every load is
  // unconditional, so all of them are in flight at once) and their values are zeroed after.
  long long roff[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) roff[r] = rbase + (long long)min(r, max(nrows - 1, 0)) * rstride;
  auto row_off = [&](int r) -> long long { return roff[r]; };

  // The global loads of the norm pass (k and q of this thread's rows, both halves) and beta are
  // issued before the setup below, so that their latency overlaps it.
  uint2 rk[K / 64][4], rq[K / 64][4];
  if (nrows > 0) {
#pragma unroll
    for (int hf = 0; hf < K / 64; ++hf) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const long long off = row_off(r) + 64 * hf + 4 * cq;
        rk[hf][r] = ldg_u64(p.k + off);
        rq[hf][r] = ldg_u64(p.q + off);
      }
    }
    if (!PH && cq < 4 * (K / 64)) {   // g of the sub-block to L2: one prefetch per (row, 128-byte line)
      const int r = cq / (K / 64), line = cq % (K / 64);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.g + rbase + (long long)min(r, nrows - 1) * rstride + 64 * line));
    }
  }
  // beta logit of token tid (tid < 64), converted where it is used
  using BetaT = typename std::conditional<BF32, float, __nv_bfloat16>::type;
  BetaT beta_raw = BetaT(0.f);
  if (tid < len) beta_raw = static_cast<const BetaT *>(p.beta)[tok_row(p, si.b, t0 + tid, h)];
  const float a_log = p.A_log[h];

  // ---- pass 0: TMEM, barrier
  if (warp == 0) {
    umma::tmem_alloc(&ms.tmem_slot, kPrepTmemCols);
    umma::tmem_relinquish();
  }
  if (tid == 32) {
    umma::mbar_init(&ms.bar, 1);
    umma::mbar_fence_init();
    ms.err = 0;
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = ms.tmem_slot;
  const float cg = -expf(a_log) * kLog2e;   // sigmoid(a) = 1 / (1 + 2^{cg (g + dt)})
  uint32_t waits = 0;   // completed waits on ms.bar (its phase parity)
  auto wait_mma = [&]() {
    if (!umma::mbar_wait_bounded(&ms.bar, waits & 1, kPrepWaitLimit)) atomicExch(&ms.err, 1);
    ++waits;
    umma::fence_after_sync();
  };

  // ---- pass 1: row norms |k_i|, |q_i| over all channels (this thread's 4 rows)
  {
    float red[8];   // per row: |k|^2 (0..3) and |q|^2 (4..7) over this lane's channel quads
#pragma unroll
    for (int r = 0; r < 8; ++r) red[r] = 0.f;
    if (nrows > 0) {
      float2 acc[8];   // the same sums as two packed partial sums (even and odd channels)
#pragma unroll
      for (int r = 0; r < 8; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
      for (int hf = 0; hf < K / 64; ++hf) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const F4 kv = bf4_to_f4(rk[hf][r]), qv = bf4_to_f4(rq[hf][r]);
          acc[r] = __ffma2_rn(kv.hi, kv.hi, __ffma2_rn(kv.lo, kv.lo, acc[r]));
          acc[4 + r] = __ffma2_rn(qv.hi, qv.hi, __ffma2_rn(qv.lo, qv.lo, acc[4 + r]));
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        red[r] = r < nrows ? acc[r].x + acc[r].y : 0.f;
        red[4 + r] = r < nrows ? acc[4 + r].x + acc[4 + r].y : 0.f;
      }
    }
    // reduce-scatter of the 8 row sums over the 16 lanes of this sub-block: after the four steps
    // lane l holds the full sum of value v(l) = 4 b3 + 2 b2 + b1 (b = bits of l)
#pragma unroll
    for (int w = 4, bit = 8; w >= 1; w >>= 1, bit >>= 1) {
      const bool up = (lane & bit) != 0;
#pragma unroll
      for (int j = 0; j < w; ++j) {
        const float send = up ? red[j] : red[j + w];
        const float keep = up ? red[j + w] : red[j];
        red[j] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
      }
    }
    red[0] += __shfl_xor_sync(0xffffffffu, red[0], 1);
    if ((lane & 1) == 0) {
      const int v = ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
      const int i = row0 + (v & 3);
      const float nv = (i < len) ? rsqrtf(red[0] + kNormEps) : 0.f;
      if (v < 4) ms.kn[i] = nv;
      else ms.qn[i] = nv;
    }
  }
  // per (chunk, head) hand-off slots
  const long long slot = c * p.H + h;
  unsigned char *hb = p.hand + slot * p.hand_stride;
  unsigned char *kg_img = hb + hand_off_kg(K), *kt_img = hb + hand_off_kt(K), *qt_img = hb + hand_off_qt(K);

#pragma unroll   // two channel halves: unrolled, the second half's gate work can overlap the first half's stores
  for (int hf = 0; hf < K / 64; ++hf) {
    // ---- pass 2a: gate and log decay of 4 rows x 4 channels (k and q as loaded by pass 1). With
    // one gate per token and head (kGatePerHead) g is [B,T,H]: its element index is the token
    // row, and the row's pre-activation is shared by all channels.
    constexpr bool per_head = PH;
    const int kk = 64 * hf + 4 * cq;
    uint2 rawk[4], rawq[4], rawg[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) rawk[r] = rawq[r] = rawg[r] = make_uint2(0u, 0u);
    if (nrows > 0) {   // no load at all when the whole sub-block is past the sequence end
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        if (per_head) rawg[r].x = static_cast<uint32_t>(reinterpret_cast<const unsigned short &>(p.g[row_off(r) / K]));
        else rawg[r] = ldg_u64(p.g + row_off(r) + kk);
        rawk[r] = rk[0][r];   // this half's k and q (the second half is moved down after the first)
        rawq[r] = rq[0][r];
      }
    }
    F4 dt = splat4(0.f);
    if (p.dt_bias) dt = per_head ? splat4(p.dt_bias[h]) : f4_of(*reinterpret_cast<const float4 *>(p.dt_bias + h * K + kk));
    const F4 cdt = mul4(splat4(cg), dt);
    F4 al[4], kv[4], qv[4], la[4];
    F4 ssum = splat4(0.f);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      // per head: the token's gate (low half of rawg[r].x) in every channel
      const F4 g4 = per_head ? splat4(__uint_as_float(rawg[r].x << 16)) : bf4_to_f4(rawg[r]);
      const F4 e = {__ffma2_rn(make_float2(cg, cg), g4.lo, cdt.lo), __ffma2_rn(make_float2(cg, cg), g4.hi, cdt.hi)};
      // la = lb log2(e) / (1 + 2^e), the additions and multiplications as packed pairs
      const F4 d = add4(ex2_4(e), splat4(1.f));
      la[r] = mul4(splat4(lbl2), {make_float2(rcp_approx(d.lo.x), rcp_approx(d.lo.y)),
                                  make_float2(rcp_approx(d.hi.x), rcp_approx(d.hi.y))});
      kv[r] = bf4_to_f4(rawk[r]);
      qv[r] = bf4_to_f4(rawq[r]);
    }
    // rows past the sequence end (their k and q repeat the last row's, or are zero) decay nothing
    if (nrows < 4) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (r >= nrows) la[r] = splat4(0.f);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      ssum = add4(ssum, la[r]);
      if constexpr (POLY) al[r] = {make_float2(ex2_poly(la[r].lo.x), ex2_poly(la[r].lo.y)),
                                   make_float2(ex2_poly(la[r].hi.x), ex2_poly(la[r].hi.y))};
      else al[r] = ex2_4(la[r]);
    }
    if constexpr (K == 128) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        rk[0][r] = rk[K / 64 - 1][r];
        rq[0][r] = rq[K / 64 - 1][r];
      }
    }
    ms.epre[sb4][cq] = float4_of(ssum);
    if (hf == 0 && tid < kChunk) ms.beta[tid] = (tid < len) ? sigmoid_fast(static_cast<float>(beta_raw)) : 0.f;
    __syncthreads();
    if (tid < 16) {   // the exclusive prefix of channel quad tid over the 16 sub-blocks, in place
      F4 run = splat4(0.f);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const F4 v = f4_of(ms.epre[j][tid]);
        ms.epre[j][tid] = float4_of(run);
        run = add4(run, v);
      }
      ms.epre[16][tid] = float4_of(run);
    }
    __syncthreads();

    // ---- pass 2b: operands of the A/P product for this half (tf32, rounded to nearest), and the
    // hand-off khat Gamma, qhat Gamma, khat Gamma_last / Gamma, Gamma_last
    // Decay sums from the prefix E: blocks before J (E[4 J]), in block J before this sub-block
    // (E[sb4] - E[4 J]) and after it (E[4 J + 4] - E[sb4 + 1]), blocks after J (E[16] - E[4 J + 4]).
    // The differences lose at most a few units in the last place of sums of magnitude at most
    // 64 * 5 log2(e) (about 462), about 2e-5 relative in the decays, far below the tf32 rounding
    // of the operands.
    const F4 e_b0 = f4_of(ms.epre[4 * J][cq]), e_b1 = f4_of(ms.epre[4 * J + 4][cq]);
    const F4 e_own = f4_of(ms.epre[sb4][cq]), e_next = f4_of(ms.epre[sb4 + 1][cq]);
    const F4 e_tot = f4_of(ms.epre[16][cq]);
    auto sub4 = [](F4 a, F4 b) -> F4 {
      return {make_float2(a.lo.x - b.lo.x, a.lo.y - b.lo.y), make_float2(a.hi.x - b.hi.x, a.hi.y - b.hi.y)};
    };
    const F4 BJ = sub4(e_b1, e_b0), Xs = sub4(e_own, e_b0), Ss = sub4(e_b1, e_next), after = sub4(e_tot, e_b1);
    const F4 PJ = ex2_4(e_b0), SJ = ex2_4(after);   // decay of the blocks before / after J
    if (J == 0 && sbi == 0)
      *reinterpret_cast<float4 *>(hb + hand_off_gam(K) + 4 * kk) = float4_of(ex2_4(e_tot));
    // byte offset of (row0 + r, kk .. kk + 3) in a 16-bit image of 64-channel panels
    auto img_off = [&](int r) -> uint32_t { return (uint32_t)hf * 8192u + img_x[r]; };
    F4 X = ex2_4(Xs);     // decay from the block start to row0 - 1
    F4 suf = ex2_4(Ss);   // decay over the block rows after the sub-block
    const F4 eBinv = ex2_4({make_float2(-BJ.lo.x, -BJ.lo.y), make_float2(-BJ.hi.x, -BJ.hi.y)});
    F4 x1 = splat4(0.f), x2 = splat4(0.f);
    if (J == 0) {   // blocks 1 and 1..2
      const F4 e_12 = f4_of(ms.epre[12][cq]);
      x1 = ex2_4(sub4(f4_of(ms.epre[8][cq]), e_b1));
      x2 = ex2_4(sub4(e_12, e_b1));
    } else if (J == 1) {   // block 2
      x1 = ex2_4(sub4(f4_of(ms.epre[12][cq]), e_b1));
    }
    const int xrow = ((J == 0) ? 112 : 128) + 4 * sbi, yrow = 144 + 4 * sbi;
    const float4 kn4 = *reinterpret_cast<const float4 *>(&ms.kn[row0]);   // this thread's four rows
    const float4 qn4 = *reinterpret_cast<const float4 *>(&ms.qn[row0]);
    const float knr[4] = {kn4.x, kn4.y, kn4.z, kn4.w};
    const float qnr[4] = {qn4.x * p.scale, qn4.y * p.scale, qn4.z * p.scale, qn4.w * p.scale};
    if (hf > 0) wait_mma();   // the previous half's product has read the operands
#pragma unroll
    for (int r = 0; r < 4; ++r) {   // I side; Gamma = X 2^{blocks before J}
      X = mul4(X, al[r]);
      const F4 kx = mul4(kv[r], X), qx = mul4(qv[r], X);
      st_tf32x4(opA_at(0, r), kx);
      st_tf32x4(opA_at(64, r), qx);
      const uint32_t io = img_off(r);
      st_half4(kg_img + io, mul4(kx, mul4(PJ, splat4(knr[r]))));
      st_half4(qt_img + io, mul4(qx, mul4(PJ, splat4(qnr[r]))));
    }
#pragma unroll
    for (int r = 3; r >= 0; --r) {  // J side; Gamma_last / Gamma = Ys 2^{blocks after J}
      const F4 ys = mul4(kv[r], suf);
      suf = mul4(suf, al[r]);
      st_tf32x4(opB_at(0, r), mul4(ys, eBinv));
      if (J < 3) st_tf32x4(opB_at(64, r), ys);   // no block lies to the right of the last one
      if (J < 2) st_tf32x4(opB_at(xrow - row0, r), mul4(ys, x1));
      if (J == 0) st_tf32x4(opB_at(yrow - row0, r), mul4(ys, x2));
      st_half4(kt_img + img_off(r), mul4(ys, mul4(SJ, splat4(knr[r]))));
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      umma::fence_after_sync();
      const uint32_t id = umma::idesc_tf32(128, kOpBRows, 0, 0);
      const uint64_t a0 = umma::sdesc_sw128(sbase + Lay::opA, 16, 1024), b0 = umma::sdesc_sw128(sbase + Lay::opB, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma::mma_tf32_ss(tmem, umma::desc_add(a0, (ks >> 2) * (128 * 128) + (ks & 3) * 32),
                          umma::desc_add(b0, (ks >> 2) * (kOpBRows * 128) + (ks & 3) * 32), id, (hf > 0) || (ks > 0));
      umma::commit(&ms.bar);
    }
  }

  // ---- pass 3: read A and P back from TMEM (cols 0..159)
  wait_mma();
  __syncthreads();
  // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (lane = D row): the row blocks {Ilo, Ilo + 1}, with
  // Ilo = 0 (quadrants 0, 2) or 2 (quadrants 1, 3), one per half-warp. Each step of a warp handles
  // one block column J for both row blocks at once: it loads the D column block of (Ilo, J) and of
  // (Ilo + 1, J) and each half-warp keeps its own. The two warps of a quadrant split the J values
  // (below) so that warps 0 and 1, which then solve the two diagonal halves, write every diagonal
  // block of -A they read themselves.
  // A rows (< 64) go to fp32 matAt (blocks of the diagonal halves, negated and transposed) or to
  // the fp16 operand of the lower-left merge (the lower-left quarter), times
  // beta_i |k_i|^-1 |k_j|^-1, strictly lower; P rows to the [-I ; P] operand (times
  // |q_i|^-1 |k_j|^-1, lower with the diagonal).
  {
    const int quad = warp & 3, row = 32 * quad + lane, I = (row & 63) >> 4;
    const int Ilo = 2 * (quad & 1);
    const bool hi = (lane >> 4) != 0;   // this lane's row block is Ilo + 1
    const bool isA = row < 64;
    const float rowf = isA ? ms.beta[row] * ms.kn[row] : ms.qn[row - 64] * p.scale;
    const int thr = isA ? row : row - 63;   // column j is kept when j < thr
    // D column block of row block I2, block column J2 <= I2: 0-3 the diagonal, 4-6 the blocks next
    // to it, 7 (2, 0), 8 (3, 1), 9 (3, 0)
    auto col_block = [](int I2, int J2) { return J2 == I2 ? I2 : J2 == I2 - 1 ? 4 + J2 : (I2 == 2 ? 7 : J2 == 1 ? 8 : 9); };
    int Js[2];
    // upper quadrants (row blocks 0, 1): the first warp takes both block columns, the second none;
    // lower quadrants (row blocks 2, 3): the first warp the diagonal columns 2, 3, the second 0, 1.
    // So warps 0 and 1 write every diagonal block of -A that their substitution reads.
    Js[0] = Ilo == 0 ? ((warp >> 2) ? -1 : 0) : ((warp >> 2) ? 0 : 2);
    Js[1] = Ilo == 0 ? ((warp >> 2) ? -1 : 1) : ((warp >> 2) ? 1 : 3);
    float xlo[2][16], xhi[2][16];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int J = Js[e];
      if (J < 0) continue;
      const uint32_t lane_base = (uint32_t)quad * 32 << 16;
      if (J <= Ilo) {
        umma::tmem_ld16(tmem + lane_base + col_block(Ilo, J) * 16, xlo[e]);
      } else {   // no block (Ilo, J): the lower half-warp skips this step
#pragma unroll
        for (int t = 0; t < 16; ++t) xlo[e][t] = 0.f;
      }
      umma::tmem_ld16(tmem + lane_base + col_block(Ilo + 1, J) * 16, xhi[e]);
    }
    umma::tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int Jb = Js[e];
      if (Jb < 0 || Jb > I) continue;
      float x[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) x[t] = hi ? xhi[e][t] : xlo[e][t];
      if (isA && (I >> 1) == (Jb >> 1)) {   // block of a diagonal half of -A: transposed, scalar stores
        float *atc = &matAt[32 * (Jb >> 1) + 16 * (Jb & 1)][row & 31];
        const float nrowf = -rowf;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 knj = *reinterpret_cast<const float4 *>(&ms.kn[16 * Jb + 4 * q]);
          const float2 nr2 = make_float2(nrowf, nrowf);
          const float2 y01 = __fmul2_rn(make_float2(x[4 * q], x[4 * q + 1]), __fmul2_rn(nr2, make_float2(knj.x, knj.y)));
          const float2 y23 = __fmul2_rn(make_float2(x[4 * q + 2], x[4 * q + 3]), __fmul2_rn(nr2, make_float2(knj.z, knj.w)));
          const float y[4] = {y01.x, y01.y, y23.x, y23.y};
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) atc[(4 * q + e2) * Lay::LDQ] = (16 * Jb + 4 * q + e2 < thr) ? y[e2] : 0.f;
        }
        continue;
      }
      // lower-left quarter of A (rows >= 32, columns < 32), or a P row of the [-I ; P] operand:
      // fp16, 8 columns per swizzled 16-byte chunk
      unsigned char *rowp = isA ? sm + Lay::opAll + (uint32_t)(row - 32) * 128 : sm + Lay::opM + (uint32_t)row * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 knj = *reinterpret_cast<const float4 *>(&ms.kn[16 * Jb + 4 * q]);
        const float2 r2 = make_float2(rowf, rowf);
        const float2 y01 = __fmul2_rn(make_float2(x[4 * q], x[4 * q + 1]), __fmul2_rn(r2, make_float2(knj.x, knj.y)));
        const float2 y23 = __fmul2_rn(make_float2(x[4 * q + 2], x[4 * q + 3]), __fmul2_rn(r2, make_float2(knj.z, knj.w)));
        float y[4] = {y01.x, y01.y, y23.x, y23.y};
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) y[e2] = (16 * Jb + 4 * q + e2 < thr) ? y[e2] : 0.f;
        const uint32_t cc = (uint32_t)(2 * Jb + (q >> 1));
        *reinterpret_cast<uint2 *>(rowp + (((cc ^ (uint32_t)(row & 7)) << 4) | ((uint32_t)(q & 1) << 3))) =
            make_uint2(pack_h2(y[0], y[1]), pack_h2(y[2], y[3]));
      }
    }
  }
  // The diagonal blocks of -A that the substitution reads (matAt) were written by the same warp
  // (warp 0 the upper half, warp 1 the lower one): the lanes of that warp meet here.
  if (warp < 2) __syncwarp();
  // Tb^T operand (row j, column m: T[m][j] beta_j, fp16): the 16-byte chunk of (row j, columns
  // 8 c8 .. 8 c8 + 7)
  auto opT_chunk = [&](int j, int c8) -> unsigned char * { return sm + Lay::opT + umma::sw128_chunk(j, c8); };
  if (tid < 64) {
    // ---- pass 4a (warps 0-1): the 32 x 32 diagonal halves of T by forward substitution. Thread =
    // column col of half hh, its 32 rows in registers as 16 pairs. Step j, with x_j final,
    // adds (-A_ij) x_j to every x_i below it: independent packed FMAs on row pairs, column j of -A
    // read as broadcast 16-byte loads of the transposed half. A pair that holds row j itself
    // takes the coefficient -A_jj = 0, so x_j stays as it is. The column goes, times beta, to row
    // o + col of the Tb^T operand and, as is, to the fp16 operands of the lower-left merge (T_[01]
    // as a K-major B, T_[23] as a K-major A).
    const int hh = tid >> 5, col = tid & 31, o = 32 * hh;
    float2 x2[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) x2[m] = make_float2(2 * m == col ? 1.f : 0.f, 2 * m + 1 == col ? 1.f : 0.f);
#pragma unroll
    for (int j = 0; j < 31; ++j) {
      const float xj = (j & 1) ? x2[j >> 1].y : x2[j >> 1].x;
      const float2 xjj = make_float2(xj, xj);
#pragma unroll
      for (int q = (j + 1) / 4; q < 8; ++q) {
        const float4 na = *reinterpret_cast<const float4 *>(&matAt[o + j][4 * q]);
        if (4 * q + 1 > j) x2[2 * q] = __ffma2_rn(make_float2(na.x, na.y), xjj, x2[2 * q]);
        if (4 * q + 3 > j) x2[2 * q + 1] = __ffma2_rn(make_float2(na.z, na.w), xjj, x2[2 * q + 1]);
      }
    }
    float x[32];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      x[2 * m] = x2[m].x;
      x[2 * m + 1] = x2[m].y;
    }
    const float bj = ms.beta[o + col];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4 *>(opT_chunk(o + col, (o >> 3) + c)) =
          make_uint4(pack_h2(x[8 * c] * bj, x[8 * c + 1] * bj), pack_h2(x[8 * c + 2] * bj, x[8 * c + 3] * bj),
                     pack_h2(x[8 * c + 4] * bj, x[8 * c + 5] * bj), pack_h2(x[8 * c + 6] * bj, x[8 * c + 7] * bj));
    // row col of T_[01]^T (K-major B of Z = A_[23][01] T_[01]) or of T_[23]^T (MN-major B of
    // Z^T T_[23]^T): column col of the half, T[o + i][o + col], i = 0..31
    unsigned char *tdst = sm + (hh == 0 ? Lay::opT01 : Lay::opT23);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4 *>(tdst + umma::sw128_chunk(col, c)) =
          make_uint4(pack_h2(x[8 * c], x[8 * c + 1]), pack_h2(x[8 * c + 2], x[8 * c + 3]),
                     pack_h2(x[8 * c + 4], x[8 * c + 5]), pack_h2(x[8 * c + 6], x[8 * c + 7]));
  } else {
    // warps 2-7 meanwhile, as 16-byte stores of 8 fp16 columns: the -I half of [-I ; P] and the
    // zeros above the block diagonal of P (row i, chunk cc), then the zero upper-right quarter of
    // Tb^T (rows j >= 32, columns m < 32). A above its block diagonal is never read.
    constexpr uint32_t kHalfMinusOne = 0xBC00u;   // fp16 -1.0
#pragma unroll 1
    for (int x = tid - 64; x < 64 * 8 + 32 * 4; x += kPrepThreads - 64) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      if (x >= 64 * 8) {
        const int y = x - 64 * 8;
        *reinterpret_cast<uint4 *>(opT_chunk(32 + (y >> 2), y & 3)) = z;
        continue;
      }
      const int i = x >> 3, cc = x & 7;
      uint4 v = z;
      if ((i >> 3) == cc) {   // this chunk holds the diagonal entry (i, i)
        const uint32_t w = ((i & 1) ? kHalfMinusOne << 16 : kHalfMinusOne);
        const int word = (i & 7) >> 1;
        v = make_uint4(word == 0 ? w : 0u, word == 1 ? w : 0u, word == 2 ? w : 0u, word == 3 ? w : 0u);
      }
      *reinterpret_cast<uint4 *>(sm + Lay::opM + umma::sw128_chunk(i, cc)) = v;
      if (cc >= 2 * ((i >> 4) + 1)) *reinterpret_cast<uint4 *>(sm + Lay::opM + umma::sw128_chunk(64 + i, cc)) = z;
    }
  }
  umma::fence_proxy_async_smem();   // the merge operands (readback and solve) to the tensor core
  umma::fence_before_sync();
  __syncthreads();
  // ---- pass 4b: the lower-left 32 x 32 block of T, -T_[23] A_[23][01] T_[01], as two tensor-core
  // products on fp16 operands with fp32 accumulators in tensor-memory columns 0..63 (free after
  // the readback): Z = A_[23][01] T_[01], then (T_[23] Z)^T = Z^T T_[23]^T, whose row b is row b of
  // the block's part of the Tb^T operand. Rows 0..31 of each product (lanes of warp 0) are the
  // result.
  if (tid == 0) {
    umma::fence_after_sync();
    const uint32_t id = umma::idesc_f16(128, 32, 0, 0);
    const uint64_t a0 = umma::sdesc_sw128(sbase + Lay::opAll, 16, 1024), b0 = umma::sdesc_sw128(sbase + Lay::opT01, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) umma::mma_f16_ss(tmem, umma::desc_add(a0, ks * 32), umma::desc_add(b0, ks * 32), id, ks > 0);
    umma::commit(&ms.bar);
  }
  wait_mma();
  if (warp == 0) {   // Z row = lane -> fp16 row of the MN-major A operand Z^T of Z^T T_[23]^T
    float x[32];
    umma::tmem_ld32(tmem, x);
    umma::tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4 *>(sm + Lay::opZ + umma::sw128_chunk(lane, c)) =
          make_uint4(pack_h2(x[8 * c], x[8 * c + 1]), pack_h2(x[8 * c + 2], x[8 * c + 3]),
                     pack_h2(x[8 * c + 4], x[8 * c + 5]), pack_h2(x[8 * c + 6], x[8 * c + 7]));
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    umma::fence_after_sync();
    const uint32_t id = umma::idesc_f16(128, 32, 1, 1);   // A = Z^T and B = T_[23]^T, both MN-major
    const uint64_t a0 = umma::sdesc_sw128(sbase + Lay::opZ, 8192, 1024), b0 = umma::sdesc_sw128(sbase + Lay::opT23, 8192, 1024);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks)
      umma::mma_f16_ss(tmem + 32, umma::desc_add(a0, ks * 2048), umma::desc_add(b0, ks * 2048), id, ks > 0);
    umma::commit(&ms.bar);
  }
  wait_mma();
  if (warp == 0) {   // row b = lane of (T_[23] Z)^T: T[32 + i][b] beta_b = -(T_[23] Z)[i][b] beta_b, Tb^T row b
    float x[32];
    umma::tmem_ld32(tmem + 32, x);
    umma::tmem_ld_wait();
    const float nb = -ms.beta[lane];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4 *>(opT_chunk(lane, 4 + c)) =
          make_uint4(pack_h2(x[8 * c] * nb, x[8 * c + 1] * nb), pack_h2(x[8 * c + 2] * nb, x[8 * c + 3] * nb),
                     pack_h2(x[8 * c + 4] * nb, x[8 * c + 5] * nb), pack_h2(x[8 * c + 6] * nb, x[8 * c + 7] * nb));
  }

  // ---- pass 5: M = [-I ; P] Tb on the tensor cores
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    umma::fence_after_sync();
    const uint32_t id = umma::idesc_f16(128, 64, 0, 0);   // fp16 A and B, K-major
    const uint64_t a0 = umma::sdesc_sw128(sbase + Lay::opM, 16, 1024), b0 = umma::sdesc_sw128(sbase + Lay::opT, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma::mma_f16_ss(tmem + 192, umma::desc_add(a0, ks * 32), umma::desc_add(b0, ks * 32), id, ks > 0);
    umma::commit(&ms.bar);
  }
  wait_mma();
  // output: row r of M (TMEM lane r) -> fp16 row r in the swizzled chunk order r*8 + (cc ^ (r & 7)),
  // staged in shared memory (the operands are dead), then copied to the hand-off block with
  // coalesced 16-byte stores; warp w takes lanes 32 (w % 4) .. + 31 and columns 32 (w / 4) .. + 31
  {
    const int r = 32 * (warp & 3) + lane;
    uint4 *stage = reinterpret_cast<uint4 *>(sm + Lay::mstage) + r * 8;
#pragma unroll 1
    for (int c0 = 32 * (warp >> 2); c0 < 32 * (warp >> 2) + 32; c0 += 16) {
      float x[16];
      umma::tmem_ld16(tmem + 192 + ((uint32_t)(warp & 3) * 32 << 16) + c0, x);
      umma::tmem_ld_wait();
#pragma unroll
      for (int hc = 0; hc < 2; ++hc)
        stage[((c0 >> 3) + hc) ^ (r & 7)] =
            make_uint4(pack_h2(x[8 * hc], x[8 * hc + 1]), pack_h2(x[8 * hc + 2], x[8 * hc + 3]),
                       pack_h2(x[8 * hc + 4], x[8 * hc + 5]), pack_h2(x[8 * hc + 6], x[8 * hc + 7]));
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (tid == 0 && ms.err) atomicExch(p.dev_status, kDevWaitTimeout);
  // the staged 16 KB to the hand-off block: eight threads per 128-byte row, 16 bytes each, four
  // rows per thread (every load and store a whole line per eight lanes)
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(sm + Lay::mstage);
    uint4 *dst = reinterpret_cast<uint4 *>(p.mats + slot * p.mat_stride);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[tid + kPrepThreads * i] = src[tid + kPrepThreads * i];
  }
  if (warp == 0) umma::tmem_dealloc(tmem, kPrepTmemCols);
}

template <int K, uint32_t VF>
static cudaError_t launch_prep_t(const Problem &p, cudaStream_t stream, bool overlap) {
  using Lay = PrepLayout;
  const size_t smem = Lay::end + sizeof(PrepMisc) + 1024;
  static PerDeviceOnce attr;
  cudaError_t e = attr([&](int) {
    return cudaFuncSetAttribute(prep_kernel<K, VF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  return launch_kernel(prep_kernel<K, VF>, dim3((unsigned)(p.max_chunks * p.H)), dim3(kPrepThreads), smem, stream,
                       overlap, p);
}

template <int K>
static cudaError_t launch_prep_k(const Problem &p, cudaStream_t stream, bool overlap) {
  constexpr uint32_t G = kGatePerHead, B = kBetaF32, X = kExp2Poly;
  switch (p.flags & (G | B | X)) {
    case 0: return launch_prep_t<K, 0>(p, stream, overlap);
    case G: return launch_prep_t<K, G>(p, stream, overlap);
    case B: return launch_prep_t<K, B>(p, stream, overlap);
    case G | B: return launch_prep_t<K, G | B>(p, stream, overlap);
    case X: return launch_prep_t<K, X>(p, stream, overlap);
    case G | X: return launch_prep_t<K, G | X>(p, stream, overlap);
    case B | X: return launch_prep_t<K, B | X>(p, stream, overlap);
    default: return launch_prep_t<K, G | B | X>(p, stream, overlap);
  }
}

cudaError_t launch_prep(const Problem &p, cudaStream_t stream, bool overlap) {
  if (p.max_chunks == 0) return cudaSuccess;
  return p.K == 64 ? launch_prep_k<64>(p, stream, overlap) : launch_prep_k<128>(p, stream, overlap);
}

}  // namespace kda
