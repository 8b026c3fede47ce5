// K1: token-parallel prep kernel of the KDA chunked forward.
//
// One CTA per (chunk of 64 tokens, head). It does the work of the FlashKDA
// "K1" stage (FlashKDA page, section "커널 퓨전(Kernel Fusion) 전략의 분리":
// gate activation, L2 normalisation, decay, and the triangular inverse, all
// parallel over tokens) and the cuLA "kda chunk intra" stage (cuLA launch
// blog, section "Status & Roadmap"), and hands the recurrence kernel:
//   * the per-token base-2 log decay la2 = lb log2(e) sigmoid(exp(A_log)(g + dt_bias)),
//     rounded to fp16 (both kernels use the rounded value);
//   * one 128 x 64 fp16 matrix per (chunk, head), stored in the 128-byte-swizzled
//     row order of its shared-memory operand image (so one bulk copy places it):
//
//   M = [ -Tb ; P Tb ],   Tb = (I + A)^{-1} diag(beta)
//   A_ij = beta_i sum_k khat_ik khat_jk 2^{G_ik - G_jk}   (j < i)
//   P_ij =        sum_k qhat_ik khat_jk 2^{G_ik - G_jk}   (j <= i)
//
// with G the in-chunk cumulative base-2 log decay. With M the recurrence kernel
// forms w = Tb (khat 2^G), u = Tb v, P w and P u as plain products.
//
// Exponent range. With lower_bound >= -5 one token decays by at most e^-5, so
// over 16 tokens |G| <= 80 ln-units (about 115.4 in base 2), which fits in
// fp32. Each 16-row block J keeps its own reference (the decay before the
// block): X_i = 2^{Gb_i} <= 1 and Y_j = 2^{-Gb_j} >= 1 with Gb the block-local
// cumulative sum. For j in block J < i in block I,
//   2^{G_i - G_j} = [X_i] [Y_j 2^{B_J} c_IJ],
// where B_J is the whole-block sum of block J and c_IJ = 2^{sum of the blocks
// strictly between J and I}: the J-side factor Y_j 2^{B_J} is <= 1 and so is
// c_IJ, so nothing overflows and a factor only underflows when the true
// product is already below the fp32 range. Diagonal blocks use X_i Y_j
// directly (<= 2^115.4). This is the "intra-chunk rescaling" that large
// chunks need (FlashKDA page, section "Flash Linear Attention과 비교").
//
// All block products of A and P come from ONE tensor-core product (tcgen05,
// tf32 operands, fp32 accumulators in tensor memory):
//   D = [khat X ; qhat X] (128 x K)  x  [khat Y ; Ys ; Ys_0 2^{B_1} ; Ys_1 2^{B_2} ; Ys_0 c_30]^T
// with Ys = khat Y 2^{B_J}: columns 0-63 give the diagonal blocks, 64-127 the
// blocks next to the diagonal, 128-175 the three blocks further out.
// The unit lower triangular inverse T = (I + A)^{-1} is blocked: the four
// 16 x 16 diagonal blocks by right-looking forward substitution (one thread
// per column, the column in registers), then the off-diagonal blocks level by
// level, T_IJ = -T_II sum_{J<=M<I} A_IM T_MJ, in fp32. Finally M = [-I ; P] Tb
// is a second tensor-core product (128 x 64 x 64).
#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {

constexpr int kPrepThreads = 512;
constexpr int kOpBRows = 176;                 // J-side operand rows
constexpr uint32_t kPrepTmemCols = 256;       // D_AP: cols 0..175; D_M: cols 192..255
constexpr long long kPrepWaitLimit = 4000000000LL;

template <int K>
struct PrepLayout {
  static constexpr uint32_t NP = K / 32;                    // tf32 panels along K
  static constexpr uint32_t raw = 0;                        // bf16 q, k, g [64][K]
  static constexpr uint32_t opA = 3 * 64 * K * 2;           // [khat X ; qhat X]: NP x 128 rows x 128 B
  static constexpr uint32_t opB = opA + NP * 128 * 128;     // J side: NP x 176 rows x 128 B
  static constexpr uint32_t end = opB + NP * kOpBRows * 128;
  // after the A/P product the raw inputs and the I-side operand are dead: A and T (fp32
  // [64][68]), the merge scratch and the Tb^T operand reuse them; the [-I ; P] operand
  // reuses the J-side operand
  static constexpr int LD = 68;                             // 68 = 4 (mod 32) words: conflict-free rows
  static constexpr uint32_t matA = 0;
  static constexpr uint32_t matT = matA + 64 * LD * 4;
  static constexpr uint32_t Z = matT + 64 * LD * 4;         // [3][16][17] fp32
  static constexpr uint32_t opT = 38 * 1024;                // Tb^T:     2 panels x  64 rows x 128 B
  static constexpr uint32_t opM = opB;                      // [-I ; P]: 2 panels x 128 rows x 128 B
  static_assert(Z + 3 * 16 * 17 * 4 <= opT, "A/T/Z overlap the Tb^T operand");
  static_assert(opT + 2 * 64 * 128 <= opB, "Tb^T operand overlaps the [-I ; P] operand");
  static_assert(opM + 2 * 128 * 128 <= end, "[-I ; P] operand must fit in the J-side region");
};

struct PrepMisc {
  uint64_t bar;
  uint32_t tmem_slot;
  int err;
  float kn[kChunk], qn[kChunk], beta[kChunk];
};

template <int K>
__global__ void __launch_bounds__(kPrepThreads, 1)
prep_kernel(const Problem p) {
  using Lay = PrepLayout<K>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // 1024-byte aligned base, derived from the __shared__ array by pointer arithmetic so that the
  // compiler keeps every access in the shared address space
  unsigned char *sm = smem_raw + ((1024u - (umma::smem_u32(smem_raw) & 1023u)) & 1023u);
  __nv_bfloat16 *rq = reinterpret_cast<__nv_bfloat16 *>(sm + Lay::raw);
  __nv_bfloat16 *rk = rq + 64 * K;
  __nv_bfloat16 *rg = rk + 64 * K;
  float *Bs = reinterpret_cast<float *>(sm + Lay::end);      // [4][K] whole-block log2 decay
  float *eB = Bs + 4 * K;                                     // [4][K] 2^{B_J}
  float *c12 = eB + 4 * K;                                    // [K]    (spare)
  PrepMisc &ms = *reinterpret_cast<PrepMisc *>(c12 + K);
  float (*matA)[Lay::LD] = reinterpret_cast<float (*)[Lay::LD]>(sm + Lay::matA);
  float (*matT)[Lay::LD] = reinterpret_cast<float (*)[Lay::LD]>(sm + Lay::matT);
  float (*Zs)[16][17] = reinterpret_cast<float (*)[16][17]>(sm + Lay::Z);

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

  // ---- pass 0: stage q, k, g rows (zero-filled past the chunk end); beta sigmoid; TMEM, barrier
  stage_rows_async<K, kPrepThreads>(rq, p.q, p, si.b, t0, h, len, 0, K, tid);
  stage_rows_async<K, kPrepThreads>(rk, p.k, p, si.b, t0, h, len, 0, K, tid);
  stage_rows_async<K, kPrepThreads>(rg, p.g, p, si.b, t0, h, len, 0, K, tid);
  cp_async_commit();
  if (tid < kChunk)
    ms.beta[tid] = (tid < len) ? sigmoid_fast(__bfloat162float(p.beta[tok_row(p, si.b, t0 + tid, h)])) : 0.f;
  if (warp == 0) {
    umma::tmem_alloc(&ms.tmem_slot, kPrepTmemCols);
    umma::tmem_relinquish();
  }
  if (tid == 0) {
    umma::mbar_init(&ms.bar, 1);
    umma::mbar_fence_init();
    ms.err = 0;
  }
  cp_async_wait_all();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = ms.tmem_slot;

  // ---- pass 1: row norms (one warp per row, lanes across channels)
#pragma unroll 1
  for (int i = warp; i < kChunk; i += kPrepThreads / 32) {
    float ssk = 0.f, ssq = 0.f;
    const __nv_bfloat162 *kr = reinterpret_cast<const __nv_bfloat162 *>(rk + i * K);
    const __nv_bfloat162 *qr = reinterpret_cast<const __nv_bfloat162 *>(rq + i * K);
#pragma unroll
    for (int x = lane; x < K / 2; x += 32) {
      const float2 a = __bfloat1622float2(kr[x]), b = __bfloat1622float2(qr[x]);
      ssk += a.x * a.x + a.y * a.y;
      ssq += b.x * b.x + b.y * b.y;
    }
    ssk = warp_sum(ssk);
    ssq = warp_sum(ssq);
    if (lane == 0) {
      ms.kn[i] = (i < len) ? rsqrtf(ssk + kNormEps) : 0.f;
      ms.qn[i] = (i < len) ? rsqrtf(ssq + kNormEps) : 0.f;
    }
  }
  __syncthreads();

  // ---- pass 2: per (channel, 16-row block): gate and block-local decay, operands of the A/P product.
  // The loops over the 16 rows are kept rolled: the kernel runs once per CTA, so its speed is set
  // by instruction fetch as much as by issue, and short loop bodies keep the code small.
  auto opA_at = [&](int row, int kc) -> float * {
    return reinterpret_cast<float *>(sm + Lay::opA + (uint32_t)(kc >> 5) * (128 * 128) +
                                     umma::sw128_offset32(row, kc & 31));
  };
  auto opB_at = [&](int row, int kc) -> float * {
    return reinterpret_cast<float *>(sm + Lay::opB + (uint32_t)(kc >> 5) * (kOpBRows * 128) +
                                     umma::sw128_offset32(row, kc & 31));
  };
  const bool unit_on = tid < 4 * K;
  const int kk = tid % K, J = tid / K;   // unit = (channel kk, block J) when unit_on
  // the fp16 log decay of (row, kk) replaces g in place: only this unit reads either
  __half *rla = reinterpret_cast<__half *>(rg);
  if (unit_on) {
    const float ea = expf(p.A_log[h]);
    const float lbl2 = p.lb * kLog2e;
    const float dt = p.dt_bias ? p.dt_bias[h * K + kk] : 0.f;
    const long long gstride = (long long)p.H * K;
    __half *la_out = p.la2 + tok_row(p, si.b, t0 + 16 * J, h) * K + kk;
    float Bsum = 0.f;
#pragma unroll 1
    for (int r = 0; r < 16; ++r) {
      const int i = 16 * J + r;
      __half la = __float2half_rn(0.f);
      if (i < len) {
        // rounded to fp16 once; this kernel and the recurrence kernel both use the rounded value
        la = __float2half_rn(log2_decay(__bfloat162float(rg[i * K + kk]), dt, ea, lbl2));
        la_out[r * gstride] = la;
      }
      rla[i * K + kk] = la;
      Bsum += __half2float(la);
    }
    Bs[J * K + kk] = Bsum;
  }
  __syncthreads();
  if (unit_on) {
    // row i of block J (Gb = block-local inclusive cumulative decay):
    //   I side   kX, qX with X = 2^{Gb}
    //   J side   kY (row i), Ys = k 2^{B_J - Gb} (row 64 + i), and for the blocks two and three
    //            away from the diagonal Ys 2^{B_1} (J = 0, row 128 + r), Ys 2^{B_2} (J = 1,
    //            row 144 + r) and Ys 2^{B_1 + B_2} (J = 0, row 160 + r); every exponent is <= 0
    const float BJ = Bs[J * K + kk], B1 = Bs[K + kk], B2 = Bs[2 * K + kk];
    const int xrow = (J == 0) ? 128 : 144;
    const float xe = (J == 0) ? B1 : B2;
    float Gb = 0.f;
#pragma unroll 1
    for (int r = 0; r < 16; ++r) {
      const int i = 16 * J + r;
      Gb += __half2float(rla[i * K + kk]);
      const float kv = __bfloat162float(rk[i * K + kk]) * ms.kn[i];
      const float qv = __bfloat162float(rq[i * K + kk]) * ms.qn[i];
      const float X = ex2_approx(Gb), e = BJ - Gb;
      *opA_at(i, kk) = to_tf32(kv * X);      // operands rounded to nearest tf32
      *opA_at(64 + i, kk) = to_tf32(qv * X);
      *opB_at(i, kk) = to_tf32(kv * ex2_approx(-Gb));
      *opB_at(64 + i, kk) = to_tf32(kv * ex2_approx(e));
      if (J < 2) *opB_at(xrow + r, kk) = to_tf32(kv * ex2_approx(e + xe));
      if (J == 0) *opB_at(160 + r, kk) = to_tf32(kv * ex2_approx(e + B1 + B2));
    }
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();

  // ---- pass 3: all A and P blocks in one tcgen05 product (tf32), accumulator in TMEM cols 0..175
  if (tid == 0) {
    umma::fence_after_sync();
    const uint32_t id = umma::idesc_tf32(128, kOpBRows, 0, 0);
#pragma unroll 1
    for (int ks = 0; ks < K / 8; ++ks) {
      const uint64_t a = umma::sdesc_sw128(sbase + Lay::opA + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
      const uint64_t b =
          umma::sdesc_sw128(sbase + Lay::opB + (ks >> 2) * (kOpBRows * 128) + (ks & 3) * 32, 16, 1024);
      umma::mma_tf32_ss(tmem, a, b, id, ks > 0);
    }
    umma::commit(&ms.bar);
  }
  if (!umma::mbar_wait_bounded(&ms.bar, 0, kPrepWaitLimit)) atomicExch(&ms.err, 1);
  umma::fence_after_sync();
  // readback: warp w reads TMEM lanes 32 (w % 4) .. + 31 (lane = D row) and the 16-column blocks
  // cb = w / 4, w / 4 + 4, w / 4 + 8. A rows (< 64) go to fp32 matA (times beta, strictly lower),
  // P rows to the [-I ; P] operand (tf32, lower with the diagonal).
  {
    const int row = 32 * (warp & 3) + lane, I = (row & 63) >> 4;
    const bool isA = row < 64;
    const float mul = isA ? ms.beta[row] : 1.f;
    const int thr = isA ? row : row - 63;   // column j is kept when j < thr
    const int xs = isA ? 0 : (row & 7);
#pragma unroll 1
    for (int cb = warp >> 2; cb < kOpBRows / 16; cb += 4) {
      float x[16];
      umma::tmem_ld16(tmem + ((uint32_t)(warp & 3) * 32 << 16) + cb * 16, x);
      umma::tmem_ld_wait();
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
        float4 v;
        float *pv = &v.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float y = (16 * Jb + 4 * q + e < thr) ? x[4 * q + e] * mul : 0.f;
          pv[e] = isA ? y : to_tf32(y);
        }
        *reinterpret_cast<float4 *>(rowp + (((c0 + q) ^ xs) << 4)) = v;
      }
    }
  }
  // the -I half of [-I ; P], and zeros above the block diagonal of A, P and T
#pragma unroll 1
  for (int x = tid; x < 64 * 64; x += kPrepThreads) {
    const int i = x >> 6, m = x & 63;
    auto opM_at = [&](int row, int col) -> float * {
      return reinterpret_cast<float *>(sm + Lay::opM + (uint32_t)(col >> 5) * (128 * 128) +
                                       umma::sw128_offset32(row, col & 31));
    };
    *opM_at(i, m) = (i == m) ? -1.f : 0.f;
    if ((m >> 4) > (i >> 4)) {
      matA[i][m] = 0.f;
      matT[i][m] = 0.f;
      *opM_at(64 + i, m) = 0.f;
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
#pragma unroll 1
    for (int j = 0; j < 16; ++j) {
      const float head = x[0];
      matT[o + j][o + col] = head;
      const float *aj = &matA[o + j][o + j];
#pragma unroll
      for (int s = 1; s < 16; ++s) x[s - 1] = fmaf((j + s < 16) ? -aj[s * Lay::LD] : 0.f, head, x[s]);
    }
  }
  __syncthreads();
  // ---- pass 4b: off-diagonal blocks, level d = I - J: Z = sum_{J<=M<I} A_IM T_MJ; T_IJ = -T_II Z
#pragma unroll 1
  for (int d = 1; d < 4; ++d) {
    const int npairs = 4 - d;
#pragma unroll 1
    for (int x = tid; x < npairs * 256; x += kPrepThreads) {
      const int Jp = x >> 8, Ip = Jp + d, i = (x >> 4) & 15, col = x & 15;
      float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int M = Jp; M < Ip; ++M) {
#pragma unroll
        for (int m = 0; m < 16; ++m)
          z[m & 3] = fmaf(matA[16 * Ip + i][16 * M + m], matT[16 * M + m][16 * Jp + col], z[m & 3]);
      }
      Zs[Jp][i][col] = (z[0] + z[1]) + (z[2] + z[3]);
    }
    __syncthreads();
#pragma unroll 1
    for (int x = tid; x < npairs * 256; x += kPrepThreads) {
      const int Jp = x >> 8, Ip = Jp + d, i = (x >> 4) & 15, col = x & 15;
      float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int m = 0; m < 16; ++m) t[m & 3] = fmaf(matT[16 * Ip + i][16 * Ip + m], Zs[Jp][m][col], t[m & 3]);
      matT[16 * Ip + i][16 * Jp + col] = -((t[0] + t[1]) + (t[2] + t[3]));
    }
    __syncthreads();
  }

  // ---- pass 5: Tb^T operand (row j, column m: T[m][j] beta_j), then M = [-I ; P] Tb on the tensor cores
#pragma unroll 2
  for (int x = tid; x < 64 * 64; x += kPrepThreads) {
    const int m = x >> 6, j = x & 63;   // consecutive threads: consecutive j of one T row
    *reinterpret_cast<float *>(sm + Lay::opT + (uint32_t)(m >> 5) * (64 * 128) +
                               umma::sw128_offset32(j, m & 31)) = to_tf32(matT[m][j] * ms.beta[j]);
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    umma::fence_after_sync();
    const uint32_t id = umma::idesc_tf32(128, 64, 0, 0);
#pragma unroll 1
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t a = umma::sdesc_sw128(sbase + Lay::opM + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
      const uint64_t b = umma::sdesc_sw128(sbase + Lay::opT + (ks >> 2) * (64 * 128) + (ks & 3) * 32, 16, 1024);
      umma::mma_tf32_ss(tmem + 192, a, b, id, ks > 0);
    }
    umma::commit(&ms.bar);
  }
  if (!umma::mbar_wait_bounded(&ms.bar, 1, kPrepWaitLimit)) atomicExch(&ms.err, 1);
  umma::fence_after_sync();
  // output: row r of M (TMEM lane r) -> fp16, written in the swizzled chunk order r*8 + (cc ^ (r & 7));
  // warp w takes lanes 32 (w % 4) .. + 31 and columns 16 (w / 4) .. + 15
  {
    const int r = 32 * (warp & 3) + lane, c0 = 16 * (warp >> 2);
    uint4 *dst = reinterpret_cast<uint4 *>(p.mats + ((long long)c * p.H + h) * (2 * kChunk * kChunk)) + r * 8;
    float x[16];
    umma::tmem_ld16(tmem + 192 + ((uint32_t)(warp & 3) * 32 << 16) + c0, x);
    umma::tmem_ld_wait();
    if (!ms.err) {
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
  using Lay = PrepLayout<K>;
  const size_t smem = Lay::end + (9 * K) * sizeof(float) + sizeof(PrepMisc) + 1024;
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
