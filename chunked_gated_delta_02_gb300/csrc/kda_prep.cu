// K1: token-parallel prep kernel of the KDA chunked forward.
//
// One CTA per (chunk of 64 tokens, head). It does the work of the FlashKDA
// "K1" stage (FlashKDA page, section "커널 퓨전(Kernel Fusion) 전략의 분리":
// gate activation, L2 normalisation, decay, and the triangular inverse, all
// parallel over tokens) and the cuLA "kda chunk intra" stage (cuLA launch
// blog, section "Status & Roadmap"), and hands the recurrence kernel one
// 128 x 64 fp16 matrix per (chunk, head), stored in the 128-byte-swizzled row
// order of its shared-memory operand image (so one bulk copy places it):
//
//   M = [ -Tb ; P Tb ],   Tb = (I + A)^{-1} diag(beta)
//   A_ij = beta_i sum_k khat_ik khat_jk 2^{G_ik - G_jk}   (j < i)
//   P_ij =        sum_k qhat_ik khat_jk 2^{G_ik - G_jk}   (j <= i)
//
// with G the in-chunk cumulative base-2 log decay. With it the recurrence
// kernel forms w = Tb (khat 2^G), u = Tb v, P w and P u as plain products.
//
// Exponent range. With lower_bound >= -5 one token decays by at most e^-5,
// so over 16 tokens |G| <= 80 ln-units (about 115.4 in base 2), which fits in
// fp32. Each 16-row block J keeps its own reference (the decay before the
// block): X_i = 2^{Gb_i} <= 1 and Y_j = 2^{-Gb_j} >= 1 with Gb the
// block-local cumulative sum. For j in block J < i in block I,
//   2^{G_i - G_j} = [X_i c_IJ] [Y_j 2^{B_J}],
// where B_J is the whole-block sum of block J and c_IJ = 2^{sum of the
// blocks strictly between J and I}: every factor is <= 1, so nothing
// overflows and a factor only underflows when the true product is already
// below the fp32 range. Diagonal blocks use X_i Y_j directly (<= 2^115.4).
// This is the "intra-chunk rescaling" that large chunks need (FlashKDA page,
// section "Flash Linear Attention과 비교"); the block products run on the
// tensor cores in tf32 (mma.sync m16n8k8, operands rounded to nearest).
//
// The unit lower triangular inverse T = (I + A)^{-1} is blocked: the four
// 16 x 16 diagonal blocks by right-looking forward substitution (one thread
// per column, the column held in registers), then the off-diagonal blocks
// level by level, T_IJ = -T_II sum_{J<=M<I} A_IM T_MJ, in fp32.
#include "kda_common.cuh"

namespace kda {

constexpr int kPrepThreads = 512;

template <int K>
struct PrepSmem {
  static constexpr int KF = K + 4;   // fp32 row stride (floats)
  static constexpr int LD = kChunk + 4;   // row stride = 4 (mod 32) words: conflict-free A fragments
  union {
    struct {                          // passes 0-2: raw staged inputs
      __nv_bfloat16 q[kChunk * K], k[kChunk * K], g[kChunk * K];
    } raw;
    struct {                          // passes 3-5: chunk matrices
      float A[kChunk][LD], P[kChunk][LD], T[kChunk][LD];
    } mat;
  } u1;
  union {
    struct {                          // passes 2-3: decay-scaled operands, fp32: in diagonal
      float kX[kChunk][KF], qX[kChunk][KF];   // blocks the tiny 2^{Gb_i} meets 2^{-Gb_j} up to
      float kY[kChunk][KF];                   // 2^115, so neither side may flush to zero
    } op;
    struct {                          // passes 4-5
      float Z[3][16][17];
      __half out[2 * kChunk][kChunk + 8];    // padded rows: conflict-free fragment stores
    } post;
  } u2;
  float Bs[4][K];                     // whole-block log2 decay B_J
  float eB[4][K];                     // 2^{B_J}
  float c12[K];                       // 2^{B_1 + B_2}
  float kn[kChunk], qn[kChunk], beta[kChunk];
};

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t tf32_bits(float x) { return __float_as_uint(to_tf32(x)); }

template <int K>
__global__ void __launch_bounds__(kPrepThreads, 1)
prep_kernel(const Problem p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PrepSmem<K> &sm = *reinterpret_cast<PrepSmem<K> *>(smem_raw);
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

  // ---- pass 0: stage q, k, g rows (zero-filled past the chunk end); beta sigmoid
  stage_rows_async<K, kPrepThreads>(sm.u1.raw.q, p.q, p, si.b, t0, h, len, 0, K, tid);
  stage_rows_async<K, kPrepThreads>(sm.u1.raw.k, p.k, p, si.b, t0, h, len, 0, K, tid);
  stage_rows_async<K, kPrepThreads>(sm.u1.raw.g, p.g, p, si.b, t0, h, len, 0, K, tid);
  cp_async_commit();
  if (tid < kChunk)
    sm.beta[tid] = (tid < len) ? sigmoid_fast(__bfloat162float(p.beta[tok_row(p, si.b, t0 + tid, h)])) : 0.f;
  cp_async_wait_all();
  __syncthreads();

  // ---- pass 1: row norms (one warp per row, lanes across channels)
  for (int i = warp; i < kChunk; i += kPrepThreads / 32) {
    float ssk = 0.f, ssq = 0.f;
    const __nv_bfloat162 *kr = reinterpret_cast<const __nv_bfloat162 *>(sm.u1.raw.k + i * K);
    const __nv_bfloat162 *qr = reinterpret_cast<const __nv_bfloat162 *>(sm.u1.raw.q + i * K);
#pragma unroll
    for (int x = lane; x < K / 2; x += 32) {
      const float2 a = __bfloat1622float2(kr[x]), b = __bfloat1622float2(qr[x]);
      ssk += a.x * a.x + a.y * a.y;
      ssq += b.x * b.x + b.y * b.y;
    }
    ssk = warp_sum(ssk);
    ssq = warp_sum(ssq);
    if (lane == 0) {
      sm.kn[i] = (i < len) ? rsqrtf(ssk + kNormEps) : 0.f;
      sm.qn[i] = (i < len) ? rsqrtf(ssq + kNormEps) : 0.f;
    }
  }
  __syncthreads();

  // ---- pass 2: per (channel, 16-row block): gate, block-local cumulative decay, scaled operands
  {
    const float ea = expf(p.A_log[h]);
    const float lbl2 = p.lb * kLog2e;
    for (int unit = tid; unit < 4 * K; unit += kPrepThreads) {
      const int kk = unit % K, J = unit / K;
      const float dt = p.dt_bias ? p.dt_bias[h * K + kk] : 0.f;
      float Gb = 0.f;
#pragma unroll 4
      for (int r = 0; r < 16; ++r) {
        const int i = 16 * J + r;
        if (i < len) {
          // the log decay is rounded to fp16 once; this kernel and the recurrence kernel both use
          // the rounded value, so the two stay consistent
          const __half la = __float2half_rn(log2_decay(__bfloat162float(sm.u1.raw.g[i * K + kk]), dt, ea, lbl2));
          p.la2[tok_row(p, si.b, t0 + i, h) * K + kk] = la;
          Gb += __half2float(la);
        }
        const float kv = __bfloat162float(sm.u1.raw.k[i * K + kk]) * sm.kn[i];
        const float qv = __bfloat162float(sm.u1.raw.q[i * K + kk]) * sm.qn[i];
        const float X = ex2_approx(Gb), Y = ex2_approx(-Gb);
        sm.u2.op.kX[i][kk] = kv * X;
        sm.u2.op.qX[i][kk] = qv * X;
        sm.u2.op.kY[i][kk] = kv * Y;
      }
      sm.Bs[J][kk] = Gb;
      sm.eB[J][kk] = ex2_approx(Gb);
    }
  }
  __syncthreads();
  if (tid < K) sm.c12[tid] = ex2_approx(sm.Bs[1][tid] + sm.Bs[2][tid]);
  __syncthreads();   // the raw inputs are dead from here on: A/P/T reuse their space

  // ---- pass 3: A and P block products on the tensor cores (tf32); items = (block pair, n-tile)
  {
    const int gq = lane >> 2, tq = lane & 3;
    for (int item = warp; item < 20; item += kPrepThreads / 32) {
      const int pr = item >> 1, nt = item & 1;
      int I = 0;
      while ((I + 1) * (I + 2) / 2 <= pr) ++I;   // pair index -> (I, J), J <= I
      const int J = pr - I * (I + 1) / 2;
      float accA[4] = {0.f, 0.f, 0.f, 0.f}, accP[4] = {0.f, 0.f, 0.f, 0.f};
      const int r0 = 16 * I + gq, r1 = r0 + 8, jr = 16 * J + 8 * nt + gq;
#pragma unroll 4
      for (int k0 = 0; k0 < K; k0 += 8) {
        const int ka = k0 + tq, kb = k0 + tq + 4;
        float cia = 1.f, cib = 1.f, sja = 1.f, sjb = 1.f;
        if (I != J) {
          sja = sm.eB[J][ka];
          sjb = sm.eB[J][kb];
          if (I - J == 2) { cia = sm.eB[J + 1][ka]; cib = sm.eB[J + 1][kb]; }
          if (I - J == 3) { cia = sm.c12[ka]; cib = sm.c12[kb]; }
        }
        uint32_t aK[4], aQ[4], b[2];
        aK[0] = tf32_bits(sm.u2.op.kX[r0][ka] * cia);
        aK[1] = tf32_bits(sm.u2.op.kX[r1][ka] * cia);
        aK[2] = tf32_bits(sm.u2.op.kX[r0][kb] * cib);
        aK[3] = tf32_bits(sm.u2.op.kX[r1][kb] * cib);
        aQ[0] = tf32_bits(sm.u2.op.qX[r0][ka] * cia);
        aQ[1] = tf32_bits(sm.u2.op.qX[r1][ka] * cia);
        aQ[2] = tf32_bits(sm.u2.op.qX[r0][kb] * cib);
        aQ[3] = tf32_bits(sm.u2.op.qX[r1][kb] * cib);
        b[0] = tf32_bits(sm.u2.op.kY[jr][ka] * sja);
        b[1] = tf32_bits(sm.u2.op.kY[jr][kb] * sjb);
        mma_tf32(accA, aK, b);
        mma_tf32(accP, aQ, b);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * I + gq + ((e >> 1) << 3);
        const int j = 16 * J + 8 * nt + 2 * tq + (e & 1);
        sm.u1.mat.A[i][j] = (j < i) ? sm.beta[i] * accA[e] : 0.f;
        sm.u1.mat.P[i][j] = (j <= i) ? accP[e] : 0.f;
      }
    }
  }
  // upper blocks of A and P are zero; T starts as zero off the lower blocks
  for (int x = tid; x < kChunk * kChunk; x += kPrepThreads) {
    const int i = x / kChunk, j = x % kChunk;
    if ((j >> 4) > (i >> 4)) {
      sm.u1.mat.A[i][j] = 0.f;
      sm.u1.mat.P[i][j] = 0.f;
      sm.u1.mat.T[i][j] = 0.f;
    }
  }
  __syncthreads();

  // ---- pass 4a: diagonal blocks of T by right-looking substitution (thread = (block, column))
  if (tid < kChunk) {
    const int J = tid >> 4, col = tid & 15, o = 16 * J;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
#pragma unroll
      for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-sm.u1.mat.A[o + i][o + j], x[j], x[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) sm.u1.mat.T[o + i][o + col] = x[i];
  }
  __syncthreads();
  // ---- pass 4b: off-diagonal blocks, level d = I - J: Z = sum_{J<=M<I} A_IM T_MJ; T_IJ = -T_II Z
  for (int d = 1; d < 4; ++d) {
    const int npairs = 4 - d;
    for (int x = tid; x < npairs * 256; x += kPrepThreads) {
      const int J = x >> 8, I = J + d, i = (x >> 4) & 15, col = x & 15;
      float z = 0.f;
      for (int M = J; M < I; ++M) {
#pragma unroll
        for (int m = 0; m < 16; ++m) z = fmaf(sm.u1.mat.A[16 * I + i][16 * M + m], sm.u1.mat.T[16 * M + m][16 * J + col], z);
      }
      sm.u2.post.Z[J][i][col] = z;
    }
    __syncthreads();
    for (int x = tid; x < npairs * 256; x += kPrepThreads) {
      const int J = x >> 8, I = J + d, i = (x >> 4) & 15, col = x & 15;
      float t = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) t = fmaf(sm.u1.mat.T[16 * I + i][16 * I + m], sm.u2.post.Z[J][m][col], t);
      sm.u1.mat.T[16 * I + i][16 * J + col] = -t;
    }
    __syncthreads();
  }

  // ---- pass 5: M = [-T diag(beta) ; P T diag(beta)] in fp16, staged for coalesced stores.
  // P T on the tensor cores: output tile (16-row mt, 8-col nt); P is lower, T lower, so only
  // tiles with 8 nt <= 16 mt + 15 are non-zero and their k range is [8 nt, 16 mt + 16).
  {
    const int gq = lane >> 2, tq = lane & 3;
    for (int item = warp; item < 20; item += kPrepThreads / 32) {
      int mt = 0;
      while (item >= (mt + 1) * (mt + 2)) ++mt;   // items per mt: 2, 4, 6, 8
      const int nt = item - mt * (mt + 1);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int ks = nt; ks <= 2 * mt + 1; ++ks) {
        uint32_t a[4], b[2];
        const int r0 = 16 * mt + gq, c0 = 8 * ks + tq;
        a[0] = tf32_bits(sm.u1.mat.P[r0][c0]);
        a[1] = tf32_bits(sm.u1.mat.P[r0 + 8][c0]);
        a[2] = tf32_bits(sm.u1.mat.P[r0][c0 + 4]);
        a[3] = tf32_bits(sm.u1.mat.P[r0 + 8][c0 + 4]);
        b[0] = tf32_bits(sm.u1.mat.T[8 * ks + tq][8 * nt + gq]);
        b[1] = tf32_bits(sm.u1.mat.T[8 * ks + tq + 4][8 * nt + gq]);
        mma_tf32(acc, a, b);
      }
      const int j0 = 8 * nt + 2 * tq;
      const float b0 = sm.beta[j0], b1 = sm.beta[j0 + 1];
#pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) {
        const int i = 16 * mt + gq + 8 * hrow;
        *reinterpret_cast<__half2 *>(&sm.u2.post.out[kChunk + i][j0]) =
            __floats2half2_rn(j0 <= i ? acc[2 * hrow] * b0 : 0.f, j0 + 1 <= i ? acc[2 * hrow + 1] * b1 : 0.f);
      }
    }
    // zero tiles of P T (above the block diagonal) and the -T diag(beta) half
    for (int x = tid; x < kChunk * kChunk / 2; x += kPrepThreads) {
      const int i = x / (kChunk / 2), j = 2 * (x % (kChunk / 2));
      *reinterpret_cast<__half2 *>(&sm.u2.post.out[i][j]) =
          __floats2half2_rn(-sm.u1.mat.T[i][j] * sm.beta[j], -sm.u1.mat.T[i][j + 1] * sm.beta[j + 1]);
      if ((j >> 3) > 2 * (i >> 4) + 1)
        *reinterpret_cast<__half2 *>(&sm.u2.post.out[kChunk + i][j]) = __floats2half2_rn(0.f, 0.f);
    }
  }
  __syncthreads();
  {
    uint4 *dst = reinterpret_cast<uint4 *>(p.mats + ((long long)c * p.H + h) * (2 * kChunk * kChunk));
#pragma unroll
    for (int x = tid; x < 2 * kChunk * kChunk / 8; x += kPrepThreads) {
      // stored as the 128-byte-swizzled shared-memory image of the K-major operand:
      // 16-byte chunk cc of row r at position r * 8 + (cc ^ (r & 7))
      const int r = x >> 3, cc = x & 7;
      dst[r * 8 + (cc ^ (r & 7))] = *reinterpret_cast<const uint4 *>(&sm.u2.post.out[r][8 * cc]);
    }
  }
}

template <int K>
static cudaError_t launch_prep_t(const Problem &p, cudaStream_t stream) {
  const size_t smem = sizeof(PrepSmem<K>);
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
