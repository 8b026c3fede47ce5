// K1: token-parallel prep kernel of the KDA chunked forward.
//
// One CTA per (chunk of 64 tokens, head), two CTAs per SM. It does the work of
// the FlashKDA "K1" stage (FlashKDA page, section "커널 퓨전(Kernel Fusion)
// 전략의 분리": gate activation, L2 normalisation, decay and the triangular
// inverse, all parallel over tokens) and the cuLA "kda chunk intra" stage
// (cuLA launch blog, section "Status & Roadmap"), and hands the recurrence
// kernel, per (chunk, head), everything it needs besides v, each in the layout of
// its shared-memory operand so that one bulk copy places it:
//   * M = [ -Tb ; P Tb ] (128 x 64 fp16, rows in 128-byte-swizzled order),
//       Tb = (I + A)^{-1} diag(beta)
//       A_ij = beta_i sum_k khat_ik khat_jk 2^{G_ik - G_jk}   (j < i)
//       P_ij =        sum_k qhat_ik khat_jk 2^{G_ik - G_jk}   (j <= i)
//   * khat Gamma, khat Gamma_last / Gamma and qhat Gamma (64 x K fp16 each, as
//     images of 64-channel panels of 128-byte swizzled token rows) and
//     Gamma_last (K fp32),
// with G the in-chunk inclusive cumulative base-2 log decay and Gamma = 2^G.
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
//   D = [k X ; q X] (128 x K)  x  [k Y ; k Ys ; k Ys_0 2^{B_1} ; k Ys_1 2^{B_2} ; k Ys_0 c_30]^T
// Columns 0-63 give the diagonal blocks, 64-127 the blocks next to the
// diagonal, 128-175 the three blocks further out. The unit lower triangular
// inverse T = (I + A)^{-1} is blocked: the four 16 x 16 diagonal blocks by
// forward substitution (one thread per column), then the off-diagonal blocks by
// doubling, in fp32: the 32 x 32 halves T_10 = -T_11 A_10 T_00 and T_32 = -T_33 A_32 T_22,
// then the lower-left 32 x 32 block -T_[23] A_[23][01] T_[01]. Finally
// M = [-I ; P] Tb is a second tensor-core product (128 x 64 x 64).
#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {

constexpr int kPrepThreads = 256;
constexpr int kOpBRows = 176;                 // J-side operand rows
constexpr uint32_t kPrepTmemCols = 256;       // D_AP: cols 0..175; D_M: cols 192..255
constexpr long long kPrepWaitLimit = 4000000000LL;

// Shared memory (byte offsets from the 1024-aligned base). The operands hold one half of the
// channels (64) at a time, as tf32 in 128-byte-swizzled panels of 32 channels.
struct PrepLayout {
  static constexpr uint32_t opA = 0;                            // [k X ; q X]: 2 panels x 128 rows x 128 B
  static constexpr uint32_t opB = opA + 2 * 128 * 128;          // J side:      2 panels x 176 rows x 128 B
  static constexpr uint32_t opEnd = opB + 2 * kOpBRows * 128;
  // after the A/P product the operands are dead: A and T (fp32 [64][68]), the merge scratch,
  // the Tb^T operand and the [-I ; P] operand take their place
  static constexpr int LD = 68;                                 // 68 = 4 (mod 32) words: conflict-free rows
  static constexpr uint32_t matA = 0;
  static constexpr uint32_t matT = matA + 64 * LD * 4;
  static constexpr uint32_t Z = matT + 64 * LD * 4;             // [4][16][16] fp32 merge scratch
  static constexpr uint32_t opT = 38 * 1024;                    // Tb^T:     2 panels x  64 rows x 128 B
  static constexpr uint32_t opM = 54 * 1024;                    // [-I ; P]: 2 panels x 128 rows x 128 B
  static constexpr uint32_t end = opM + 2 * 128 * 128;
  static_assert(Z + 4 * 16 * 16 * 4 <= opT, "A/T/Z overlap the Tb^T operand");
  static_assert(opT + 2 * 64 * 128 <= opM, "Tb^T operand overlaps the [-I ; P] operand");
  static_assert(end >= opEnd, "layout end");
};

struct PrepMisc {
  uint64_t bar;
  uint32_t tmem_slot;
  int err;
  float beta[kChunk], kn[kChunk], qn[kChunk];
  float2 ssub[4][2][32];                  // per (block, 8-row sub-block, channel pair): sum of la2
};

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
__device__ __forceinline__ void st_tf32x2(unsigned char *p, float2 v) {
  *reinterpret_cast<float2 *>(p) = make_float2(tf32_rn(v.x), tf32_rn(v.y));
}

template <int K>
__global__ void __launch_bounds__(kPrepThreads, 2)
prep_kernel(const Problem p) {
  using Lay = PrepLayout;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so that the
  // compiler keeps every access in the shared address space
  unsigned char *sm = smem_raw + ((1024u - (umma::smem_u32(smem_raw) & 1023u)) & 1023u);
  PrepMisc &ms = *reinterpret_cast<PrepMisc *>(sm + Lay::end);
  float (*matA)[Lay::LD] = reinterpret_cast<float (*)[Lay::LD]>(sm + Lay::matA);
  float (*matT)[Lay::LD] = reinterpret_cast<float (*)[Lay::LD]>(sm + Lay::matT);
  float (*Zs)[16][16] = reinterpret_cast<float (*)[16][16]>(sm + Lay::Z);   // [4][16][16]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long c = blockIdx.x;
  const int h = blockIdx.y;
  if (p.flag && *p.flag != kDevOk) return;
  const long long total = p.cu ? (long long)p.chunk_off[p.N] : (long long)p.B * p.nc_fixed;
  if (c >= total) return;
  const int s = chunk_to_seq(p, c);
  const SeqInfo si = seq_info(p, s);
  const int n = (int)(c - si.chunk0);
  const int t0 = si.t0 + n * kChunk;
  const int len = min(kChunk, si.len - n * kChunk);
  const uint32_t sbase = umma::smem_u32(sm);

  // ---- pass 0: beta sigmoid, TMEM, barrier
  if (tid < kChunk)
    ms.beta[tid] = (tid < len) ? sigmoid_fast(__bfloat162float(p.beta[tok_row(p, si.b, t0 + tid, h)])) : 0.f;
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
  uint32_t waits = 0;   // completed waits on ms.bar (its phase parity)
  auto wait_mma = [&]() {
    if (!umma::mbar_wait_bounded(&ms.bar, waits & 1, kPrepWaitLimit)) atomicExch(&ms.err, 1);
    ++waits;
    umma::fence_after_sync();
  };

  // Elementwise unit of this thread: channel pair `lane` of the current half, 16-row block
  // J = warp / 2, 8-row sub-block sb = warp % 2.
  const int J = warp >> 1, sb = warp & 1;
  const int row0 = 16 * J + 8 * sb;
  const int nrows = max(0, min(8, len - row0));
  const float ea = expf(p.A_log[h]);
  const float cg = -ea * kLog2e;                 // sigmoid(a) = 1 / (1 + 2^{cg (g + dt)})
  const float lbl2 = p.lb * kLog2e;
  const long long rstride = (long long)p.H * K;  // elements between consecutive tokens
  const long long rbase = tok_row(p, si.b, t0 + row0, h) * K;
  // swizzled byte offset of this lane's channel pair inside a row (row & 7 == r for row0 + r)
  const uint32_t pan = (uint32_t)(lane >> 4), chk = (uint32_t)((lane & 15) >> 1), sub8 = (uint32_t)(lane & 1) * 8;
  auto op_at = [&](uint32_t region, uint32_t rows_per_panel, int row, int r) -> unsigned char * {
    return sm + region + pan * (rows_per_panel * 128) + (uint32_t)row * 128 + (((chk ^ (uint32_t)r) << 4) | sub8);
  };

  // Rows of the sub-block past the sequence end are read from its last valid row (every load is
  // unconditional, so all of them are in flight at once) and their values are zeroed after.
  auto row_off = [&](int r) -> long long { return rbase + (long long)min(r, max(nrows - 1, 0)) * rstride; };

  // ---- pass 1: row norms |k_i|, |q_i| over all channels (this warp's 8 rows); g goes to L2 meanwhile
  {
    float red[16];   // per row: |k|^2 and |q|^2 over this lane's channel pairs
#pragma unroll
    for (int r = 0; r < 16; ++r) red[r] = 0.f;
    if (nrows > 0) {
      uint32_t rk[K / 64][8], rq[K / 64][8];
#pragma unroll
      for (int hf = 0; hf < K / 64; ++hf) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const long long off = row_off(r) + 64 * hf + 2 * lane;
          rk[hf][r] = ldg_u32(p.k + off);
          rq[hf][r] = ldg_u32(p.q + off);
        }
      }
      if (lane < 8 * (K / 64)) {   // g of the sub-block to L2: one prefetch per (row, 128-byte line)
        const int r = lane / (K / 64), line = lane % (K / 64);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.g + row_off(r) + 64 * line));
      }
#pragma unroll
      for (int hf = 0; hf < K / 64; ++hf) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float2 kv = bf2_to_f2(rk[hf][r]), qv = bf2_to_f2(rq[hf][r]);
          red[r] = fmaf(kv.x, kv.x, fmaf(kv.y, kv.y, red[r]));
          red[8 + r] = fmaf(qv.x, qv.x, fmaf(qv.y, qv.y, red[8 + r]));
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r >= nrows) red[r] = red[8 + r] = 0.f;
      }
    }
    // reduce-scatter of the 16 row sums over the warp: after the five steps lane l holds the
    // full sum of value v(l) = 8 b4 + 4 b3 + 2 b2 + b1 (b = bits of l)
#pragma unroll
    for (int w = 8, bit = 16; w >= 1; w >>= 1, bit >>= 1) {
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
      const int v = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
      const int i = row0 + (v & 7);
      const float nv = (i < len) ? rsqrtf(red[0] + kNormEps) : 0.f;
      if (v < 8) ms.kn[i] = nv;
      else ms.qn[i] = nv;
    }
  }
  // per (chunk, head) hand-off slots
  const long long slot = c * p.H + h;
  unsigned char *hb = p.hand + slot * p.hand_stride;
  unsigned char *kg_img = hb + hand_off_kg(K), *kt_img = hb + hand_off_kt(K), *qt_img = hb + hand_off_qt(K);

#pragma unroll 1
  for (int hf = 0; hf < K / 64; ++hf) {
    // ---- pass 2a: gate and log decay of 8 rows x 2 channels
    const int kk = 64 * hf + 2 * lane;
    uint32_t rawk[8], rawq[8], rawg[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) rawk[r] = rawq[r] = rawg[r] = 0u;
    if (nrows > 0) {   // no load at all when the whole sub-block is past the sequence end
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const long long off = row_off(r) + kk;
        rawg[r] = ldg_u32(p.g + off);
        rawk[r] = ldg_u32(p.k + off);
        rawq[r] = ldg_u32(p.q + off);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r >= nrows) rawk[r] = rawq[r] = rawg[r] = 0u;
      }
    }
    float2 dt = make_float2(0.f, 0.f);
    if (p.dt_bias) dt = *reinterpret_cast<const float2 *>(p.dt_bias + h * K + kk);
    const float2 cdt = make_float2(cg * dt.x, cg * dt.y);
    float2 al[8], kv[8], qv[8];
    float2 ssum = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float2 g2 = bf2_to_f2(rawg[r]);
      const float2 e = __ffma2_rn(make_float2(cg, cg), g2, cdt);
      float2 la = make_float2(lbl2 * rcp_approx(1.f + ex2_approx(e.x)), lbl2 * rcp_approx(1.f + ex2_approx(e.y)));
      if (r >= nrows) la = make_float2(0.f, 0.f);
      ssum.x += la.x;
      ssum.y += la.y;
      al[r] = ex2_2(la);
      kv[r] = bf2_to_f2(rawk[r]);
      qv[r] = bf2_to_f2(rawq[r]);
    }
    ms.ssub[J][sb][lane] = ssum;
    __syncthreads();

    // ---- pass 2b: operands of the A/P product for this half (tf32, rounded to nearest), and the
    // hand-off khat Gamma, qhat Gamma, khat Gamma_last / Gamma, Gamma_last
    float2 Bm[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float2 a = ms.ssub[m][0][lane], b = ms.ssub[m][1][lane];
      Bm[m] = make_float2(a.x + b.x, a.y + b.y);
    }
    const float2 S0 = ms.ssub[J][0][lane], S1 = ms.ssub[J][1][lane];
    const float2 BJ = Bm[J];
    float2 before = make_float2(0.f, 0.f), after = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      if (m < J) before = make_float2(before.x + Bm[m].x, before.y + Bm[m].y);
      if (m > J) after = make_float2(after.x + Bm[m].x, after.y + Bm[m].y);
    }
    const float2 PJ = ex2_2(before), SJ = ex2_2(after);   // decay of the blocks before / after J
    if (J == 0 && sb == 0) {
      const float2 tot = make_float2(BJ.x + after.x, BJ.y + after.y);
      *reinterpret_cast<float2 *>(hb + hand_off_gam(K) + 4 * kk) = ex2_2(tot);
    }
    // byte offset of (row, kk .. kk+1) in a 16-bit MN-major swizzled image (row & 7 == r)
    const uint32_t img_pan = (uint32_t)hf * 8192u, img_chk = (uint32_t)(lane >> 2), img_sub = (uint32_t)(lane & 3) * 4;
    float2 X = sb ? ex2_2(S0) : make_float2(1.f, 1.f);     // decay from the block start to row0 - 1
    float2 suf = sb ? make_float2(1.f, 1.f) : ex2_2(S1);   // decay over the block rows after the sub-block
    const float2 eBinv = ex2_2(make_float2(-BJ.x, -BJ.y));
    float2 x1 = make_float2(0.f, 0.f), x2 = make_float2(0.f, 0.f);
    if (J == 0) {
      x1 = ex2_2(Bm[1]);
      x2 = ex2_2(make_float2(Bm[1].x + Bm[2].x, Bm[1].y + Bm[2].y));
    } else if (J == 1) {
      x1 = ex2_2(Bm[2]);
    }
    const int xrow = (J == 0) ? 128 : 144;
    if (hf > 0) wait_mma();   // the previous half's product has read the operands
#pragma unroll
    for (int r = 0; r < 8; ++r) {   // I side; Gamma = X 2^{blocks before J}
      const int i = row0 + r;
      X = mul2(X, al[r]);
      st_tf32x2(op_at(Lay::opA, 128, i, r), mul2(kv[r], X));
      st_tf32x2(op_at(Lay::opA, 128, 64 + i, r), mul2(qv[r], X));
      const float2 G = mul2(X, PJ);
      const float kn = ms.kn[i], qn = ms.qn[i];
      const uint32_t io = (uint32_t)i * 128u + img_pan + (((img_chk ^ (uint32_t)r) << 4) | img_sub);
      *reinterpret_cast<__half2 *>(kg_img + io) = __float22half2_rn(mul2(kv[r], mul2(G, make_float2(kn, kn))));
      *reinterpret_cast<__half2 *>(qt_img + io) = __float22half2_rn(mul2(qv[r], mul2(G, make_float2(qn, qn))));
    }
#pragma unroll
    for (int r = 7; r >= 0; --r) {  // J side; Gamma_last / Gamma = Ys 2^{blocks after J}
      const int i = row0 + r;
      const float2 ys = mul2(kv[r], suf);
      suf = mul2(suf, al[r]);
      st_tf32x2(op_at(Lay::opB, kOpBRows, i, r), mul2(ys, eBinv));
      st_tf32x2(op_at(Lay::opB, kOpBRows, 64 + i, r), ys);
      if (J < 2) st_tf32x2(op_at(Lay::opB, kOpBRows, xrow + 8 * sb + r, r), mul2(ys, x1));
      if (J == 0) st_tf32x2(op_at(Lay::opB, kOpBRows, 160 + 8 * sb + r, r), mul2(ys, x2));
      const float kn = ms.kn[i];
      const uint32_t io = (uint32_t)i * 128u + img_pan + (((img_chk ^ (uint32_t)r) << 4) | img_sub);
      *reinterpret_cast<__half2 *>(kt_img + io) = __float22half2_rn(mul2(ys, mul2(SJ, make_float2(kn, kn))));
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

  // ---- pass 3: read A and P back from TMEM (cols 0..175)
  wait_mma();
  __syncthreads();
  // Warp w reads TMEM lanes 32 (w % 4) .. + 31 (lane = D row). A lane quadrant holds the row
  // blocks {0, 1} (quadrants 0, 2) or {2, 3} (quadrants 1, 3), which need the 16-column blocks
  // {0, 1, 4} or {2, 3, 5, 6, 8, 9, 10}; the two warps of a quadrant split them and load all of
  // theirs before one wait. A rows (< 64) go to fp32 matA (times beta_i |k_i|^-1 |k_j|^-1,
  // strictly lower), P rows to the [-I ; P] operand (times |q_i|^-1 |k_j|^-1, lower with the
  // diagonal, tf32).
  {
    const int row = 32 * (warp & 3) + lane, I = (row & 63) >> 4;
    const bool isA = row < 64;
    const float rowf = isA ? ms.beta[row] * ms.kn[row] : ms.qn[row - 64];
    const int thr = isA ? row : row - 63;   // column j is kept when j < thr
    const int xs = isA ? 0 : (row & 7);
    const int sel = (warp & 1) * 2 + (warp >> 2);   // (upper row blocks, second warp of the quadrant)
    const int cbs[4] = {sel == 0 ? 0 : sel == 1 ? 4 : sel == 2 ? 2 : 6, sel == 0 ? 1 : sel == 2 ? 3 : sel == 3 ? 8 : -1,
                        sel == 2 ? 5 : sel == 3 ? 9 : -1, sel == 3 ? 10 : -1};
    float xb[4][16];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (cbs[e] >= 0) umma::tmem_ld16(tmem + ((uint32_t)(warp & 3) * 32 << 16) + cbs[e] * 16, xb[e]);
    umma::tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int cb = cbs[e];
      if (cb < 0) continue;
      const float *x = xb[e];
      // block column Jb of D column block cb for row block I, or -1 if it is not one of row I's
      int Jb = -1;
      if (cb < 4) Jb = (cb == I) ? cb : -1;
      else if (cb < 8) Jb = (cb - 4 == I - 1) ? cb - 4 : -1;
      else if (cb == 8) Jb = (I == 2) ? 0 : -1;
      else Jb = (I == 3) ? (cb == 9 ? 1 : 0) : -1;
      if (Jb < 0) continue;
      unsigned char *rowp = isA ? reinterpret_cast<unsigned char *>(&matA[row][0])
                                : sm + Lay::opM + (uint32_t)(Jb >> 1) * (128 * 128) + (uint32_t)row * 128;
      const int c0 = isA ? 4 * Jb : 4 * (Jb & 1);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 knj = *reinterpret_cast<const float4 *>(&ms.kn[16 * Jb + 4 * q]);
        const float kj[4] = {knj.x, knj.y, knj.z, knj.w};
        float4 v;
        float *pv = &v.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float y = (16 * Jb + 4 * q + e < thr) ? x[4 * q + e] * rowf * kj[e] : 0.f;
          pv[e] = isA ? y : tf32_rn(y);
        }
        *reinterpret_cast<float4 *>(rowp + (((c0 + q) ^ xs) << 4)) = v;
      }
    }
  }
  // the -I half of [-I ; P], and zeros above the block diagonal of P and T, as 16-byte stores of
  // (row i, 4-column group cq); A above its block diagonal is never read
#pragma unroll 1
  for (int x = tid; x < 64 * 16; x += kPrepThreads) {
    const int i = x >> 4, cq = x & 15;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool dg = (i >> 2) == cq;   // this group holds the diagonal entry (i, i)
    const float4 v = make_float4(dg && (i & 3) == 0 ? -1.f : 0.f, dg && (i & 3) == 1 ? -1.f : 0.f,
                                 dg && (i & 3) == 2 ? -1.f : 0.f, dg && (i & 3) == 3 ? -1.f : 0.f);
    unsigned char *pan = sm + Lay::opM + (uint32_t)(cq >> 3) * (128 * 128);
    *reinterpret_cast<float4 *>(pan + umma::sw128_chunk(i, cq & 7)) = v;
    if (cq >= 4 * ((i >> 4) + 1)) {
      *reinterpret_cast<float4 *>(pan + umma::sw128_chunk(64 + i, cq & 7)) = z;
      *reinterpret_cast<float4 *>(&matT[i][4 * cq]) = z;
    }
  }
  __syncthreads();

  // ---- pass 4a: diagonal blocks of T by forward substitution (thread = (block, column)). The
  // column lives in a shift register: at step j the head x[0] is final (T row j), and x[s] then
  // takes the update of row j + 1 + s.
  if (tid < kChunk) {
    const int Jd = tid >> 4, col = tid & 15, o = 16 * Jd;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
      const float head = x[0];
      matT[o + j][o + col] = head;
      const float *aj = &matA[o + j][o + j];
#pragma unroll
      for (int s2 = 1; s2 < 16; ++s2) x[s2 - 1] = fmaf((j + s2 < 16) ? -aj[s2 * Lay::LD] : 0.f, head, x[s2]);
    }
  }
  __syncthreads();
  // ---- pass 4b: off-diagonal blocks of T by doubling (four steps). A thread computes a strip of
  // four columns of one row of a 16 x 16 block with 16-byte loads of T and Z rows.
  auto fma4 = [](float a, const float4 b, float4 &acc) {
    acc.x = fmaf(a, b.x, acc.x);
    acc.y = fmaf(a, b.y, acc.y);
    acc.z = fmaf(a, b.z, acc.z);
    acc.w = fmaf(a, b.w, acc.w);
  };
  // acc += X[xr][xc .. xc + 15] (row of a 16-column block of X) times the 16 x 4 strip of Y
  // starting at row yr, column yc (Y with leading dimension ldy)
  auto strip = [&](const float *xrow, const float *y, int ldy, float4 &acc) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 a = *reinterpret_cast<const float4 *>(xrow + 4 * q);
      fma4(a.x, *reinterpret_cast<const float4 *>(y + (4 * q + 0) * ldy), acc);
      fma4(a.y, *reinterpret_cast<const float4 *>(y + (4 * q + 1) * ldy), acc);
      fma4(a.z, *reinterpret_cast<const float4 *>(y + (4 * q + 2) * ldy), acc);
      fma4(a.w, *reinterpret_cast<const float4 *>(y + (4 * q + 3) * ldy), acc);
    }
  };
  {
    const int i = (tid >> 2) & 15, c4 = 4 * (tid & 3);
    // level 1, blocks (I, I - 1) for I = 1, 3: Z = A_{I,I-1} T_{I-1,I-1}, then T_{I,I-1} = -T_II Z
    const int p1 = tid >> 6, I1 = 2 * p1 + 1;   // threads 0..127
    if (tid < 128) {
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      strip(&matA[16 * I1 + i][16 * (I1 - 1)], &matT[16 * (I1 - 1)][16 * (I1 - 1) + c4], Lay::LD, z);
      *reinterpret_cast<float4 *>(&Zs[p1][i][c4]) = z;
    }
    __syncthreads();
    if (tid < 128) {
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      strip(&matT[16 * I1 + i][16 * I1], &Zs[p1][0][c4], 16, t);
      *reinterpret_cast<float4 *>(&matT[16 * I1 + i][16 * (I1 - 1) + c4]) = make_float4(-t.x, -t.y, -t.z, -t.w);
    }
    __syncthreads();
    // level 2, the lower-left 32 x 32 block (row blocks a = 2, 3; column blocks b = 0, 1):
    // Z_ab = sum_{b <= c <= 1} A_ac T_cb, then T_ab = -sum_{2 <= c <= a} T_ac Z_cb
    const int a = 2 + (tid >> 7), b = (tid >> 6) & 1;
    {
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = b; c <= 1; ++c) strip(&matA[16 * a + i][16 * c], &matT[16 * c][16 * b + c4], Lay::LD, z);
      *reinterpret_cast<float4 *>(&Zs[2 * (a - 2) + b][i][c4]) = z;
    }
    __syncthreads();
    {
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = 2; c <= a; ++c) strip(&matT[16 * a + i][16 * c], &Zs[2 * (c - 2) + b][0][c4], 16, t);
      *reinterpret_cast<float4 *>(&matT[16 * a + i][16 * b + c4]) = make_float4(-t.x, -t.y, -t.z, -t.w);
    }
    __syncthreads();
  }

  // ---- pass 5: Tb^T operand (row j, column m: T[m][j] beta_j), then M = [-I ; P] Tb on the tensor cores
  // thread = (row j of Tb^T, 4-column group m4): one 16-byte store per item
#pragma unroll 1
  for (int x = tid; x < 64 * 16; x += kPrepThreads) {
    const int j = x & 63, m4 = 4 * (x >> 6);
    const float bj = ms.beta[j];
    const float4 v = make_float4(tf32_rn(matT[m4][j] * bj), tf32_rn(matT[m4 + 1][j] * bj),
                                 tf32_rn(matT[m4 + 2][j] * bj), tf32_rn(matT[m4 + 3][j] * bj));
    *reinterpret_cast<float4 *>(sm + Lay::opT + (uint32_t)(m4 >> 5) * (64 * 128) +
                                umma::sw128_chunk(j, (m4 & 31) >> 2)) = v;
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    umma::fence_after_sync();
    const uint32_t id = umma::idesc_tf32(128, 64, 0, 0);
    const uint64_t a0 = umma::sdesc_sw128(sbase + Lay::opM, 16, 1024), b0 = umma::sdesc_sw128(sbase + Lay::opT, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma::mma_tf32_ss(tmem + 192, umma::desc_add(a0, (ks >> 2) * (128 * 128) + (ks & 3) * 32),
                        umma::desc_add(b0, (ks >> 2) * (64 * 128) + (ks & 3) * 32), id, ks > 0);
    umma::commit(&ms.bar);
  }
  wait_mma();
  // output: row r of M (TMEM lane r) -> fp16, written in the swizzled chunk order r*8 + (cc ^ (r & 7));
  // warp w takes lanes 32 (w % 4) .. + 31 and columns 32 (w / 4) .. + 31
  {
    const int r = 32 * (warp & 3) + lane;
    uint4 *dst = reinterpret_cast<uint4 *>(p.mats + slot * p.mat_stride) + r * 8;
#pragma unroll 1
    for (int c0 = 32 * (warp >> 2); c0 < 32 * (warp >> 2) + 32; c0 += 16) {
      float x[16];
      umma::tmem_ld16(tmem + 192 + ((uint32_t)(warp & 3) * 32 << 16) + c0, x);
      umma::tmem_ld_wait();
      if (ms.err) continue;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int cc = (c0 >> 3) + hc;
        __half2 hv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) hv[e] = __floats2half2_rn(x[8 * hc + 2 * e], x[8 * hc + 2 * e + 1]);
        dst[cc ^ (r & 7)] = *reinterpret_cast<const uint4 *>(hv);
      }
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (ms.err && tid == 0) atomicExch(p.dev_status, kDevWaitTimeout);
  if (warp == 0) umma::tmem_dealloc(tmem, kPrepTmemCols);
}

template <int K>
static cudaError_t launch_prep_t(const Problem &p, cudaStream_t stream) {
  using Lay = PrepLayout;
  const size_t smem = Lay::end + sizeof(PrepMisc) + 1024;
  cudaError_t e = cudaFuncSetAttribute(prep_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.max_chunks, (unsigned)p.H);
  prep_kernel<K><<<grid, kPrepThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prep(const Problem &p, cudaStream_t stream) {
  if (p.max_chunks == 0) return cudaSuccess;
  return p.K == 64 ? launch_prep_t<64>(p, stream) : launch_prep_t<128>(p, stream);
}

}  // namespace kda
