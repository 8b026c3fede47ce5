// K2: head-parallel chunk recurrence of the KDA chunked forward.
//
// One CTA per (sequence, head, 32-wide slice of V). The CTA walks the chunks
// of its sequence in order and carries the K x 32 slice of the state S on
// chip (the FlashKDA "K2" stage, FlashKDA page, section "커널 퓨전(Kernel
// Fusion) 전략의 분리"; the cuLA "chunk gated delta h" + "chunk fwd o"
// stages, cuLA launch blog, section "Status & Roadmap"). Per chunk, with
// M = [-Tb ; P Tb] from the prep kernel and G the in-chunk cumulative base-2
// log decay measured from the chunk start:
//
//   [-w ; P w] = M (khat 2^G)          q~ = qhat 2^G,   Q' = q~ - P w
//   [-u ; P u] = M v                    k~ = khat 2^{G_last - G},  gamma = 2^{G_last}
//   R = [-u ; P u] + [w ; Q'] S        ->  U = -R[0:64],  o = scale R[64:128]
//   S <- Diag(gamma) S + k~^T U
//
// which is the WY/UT form of the delta rule inside a chunk: U are the
// residuals v - prediction, o mixes the inter-chunk term q~ S with the
// intra-chunk term P U. All factors 2^G, 2^{G_last-G} are <= 1.
// This version computes in fp32 on the CUDA cores.
#include "kda_common.cuh"

namespace kda {

constexpr int kRecThreads = 256;
constexpr int kBV = 32;

template <int K>
struct RecSmem {
  static constexpr int KP = K + 1;
  float bufA[kChunk][KP];   // khat 2^G, then v tile / U
  float bufB[kChunk][KP];   // q~, then Q'
  float bufC[kChunk][KP];   // G, then k~
  float bufD[kChunk][KP];   // khat, then w
  float M[2 * kChunk][kChunk + 1];
  float S[K][kBV + 1];
  float gam[K];
  float kn[kChunk], qn[kChunk];
};

template <int K>
__global__ void __launch_bounds__(kRecThreads)
recur_simt_kernel(const Problem p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RecSmem<K> &sm = *reinterpret_cast<RecSmem<K> *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int VT = p.V / kBV;
  const int bid = blockIdx.x;
  const int r = bid / (p.H * VT);
  const int h = (bid / VT) % p.H;
  const int v0 = (bid % VT) * kBV;
  if (p.flag && *p.flag != kDevOk) return;
  const int s = p.cu ? p.order[r] : r;
  const SeqInfo si = seq_info(p, s);
  // v tile and U reuse bufA (khat 2^G is dead by then): 2 * 64 * 32 floats <= 64 * (K+1)
  float *vt = &sm.bufA[0][0];
  float *U = vt + kChunk * kBV;
  static_assert(2 * kChunk * kBV <= kChunk * (K + 1), "v tile + U must fit in bufA");

  // state slice: S[k][v] = state[s,h,v0+v,k]
  for (int x = tid; x < K * kBV; x += kRecThreads) {
    const int kk = x % K, vv = x / K;
    sm.S[kk][vv] = p.init ? p.init[(((long long)s * p.H + h) * p.V + v0 + vv) * K + kk] : 0.f;
  }
  const float ea = expf(p.A_log[h]);
  const float lbl2 = p.lb * kLog2e;
  const int nch = (si.len + kChunk - 1) / kChunk;
  __syncthreads();

  for (int n = 0; n < nch; ++n) {
    const int t0 = si.t0 + n * kChunk;
    const int L = min(kChunk, si.len - n * kChunk);
    const long long cidx = (long long)si.chunk0 + n;
    // -- norms
    for (int i = warp; i < kChunk; i += kRecThreads / 32) {
      float ssk = 0.f, ssq = 0.f;
      if (i < L) {
        const long long row = tok_row(p, si.b, t0 + i, h);
        for (int kk = lane; kk < K; kk += 32) {
          const float a = __bfloat162float(p.k[row * K + kk]), b = __bfloat162float(p.q[row * K + kk]);
          ssk += a * a;
          ssq += b * b;
        }
      }
      ssk = warp_sum(ssk);
      ssq = warp_sum(ssq);
      if (lane == 0) {
        sm.kn[i] = (i < L) ? rsqrtf(ssk + kNormEps) : 0.f;
        sm.qn[i] = (i < L) ? rsqrtf(ssq + kNormEps) : 0.f;
      }
    }
    __syncthreads();
    // -- per-channel cumulative decay and decayed operands
    if (tid < K) {
      const int kk = tid;
      const float dt = p.dt_bias ? p.dt_bias[h * K + kk] : 0.f;
      float G = 0.f;
      for (int i = 0; i < kChunk; ++i) {
        float kv = 0.f, qv = 0.f;
        if (i < L) {
          const long long row = tok_row(p, si.b, t0 + i, h);
          G += log2_decay(__bfloat162float(p.g[row * K + kk]), dt, ea, lbl2);
          kv = __bfloat162float(p.k[row * K + kk]) * sm.kn[i];
          qv = __bfloat162float(p.q[row * K + kk]) * sm.qn[i];
        }
        const float X = ex2_approx(G);
        sm.bufA[i][kk] = kv * X;
        sm.bufB[i][kk] = qv * X;
        sm.bufC[i][kk] = G;
        sm.bufD[i][kk] = kv;
      }
      sm.gam[kk] = ex2_approx(G);
      for (int i = 0; i < kChunk; ++i) sm.bufC[i][kk] = sm.bufD[i][kk] * ex2_approx(G - sm.bufC[i][kk]);
    }
    // -- hand-off matrix of this chunk
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(p.mats + (cidx * p.H + h) * (2 * kChunk * kChunk));
      for (int x = tid; x < 2 * kChunk * kChunk / 8; x += kRecThreads) {
        const uint4 u = src[x];
        const __half *hv = reinterpret_cast<const __half *>(&u);
        const int rr = (x * 8) / kChunk, cc = (x * 8) % kChunk;
#pragma unroll
        for (int e = 0; e < 8; ++e) sm.M[rr][cc + e] = __half2float(hv[e]);
      }
    }
    __syncthreads();
    // -- [-w ; P w] = M (khat 2^G)
    for (int x = tid; x < 2 * kChunk * K; x += kRecThreads) {
      const int kk = x % K, rr = x / K;
      float acc = 0.f;
#pragma unroll 8
      for (int j = 0; j < kChunk; ++j) acc += sm.M[rr][j] * sm.bufA[j][kk];
      if (rr < kChunk) sm.bufD[rr][kk] = -acc;
      else sm.bufB[rr - kChunk][kk] -= acc;
    }
    __syncthreads();
    // -- v tile
    for (int x = tid; x < kChunk * kBV; x += kRecThreads) {
      const int vv = x % kBV, i = x / kBV;
      vt[i * kBV + vv] = (i < L) ? __bfloat162float(p.v[tok_row(p, si.b, t0 + i, h) * p.V + v0 + vv]) : 0.f;
    }
    __syncthreads();
    // -- R = M v + [w ; Q'] S ; o = scale R[64:], U = -R[:64]
    for (int x = tid; x < 2 * kChunk * kBV; x += kRecThreads) {
      const int vv = x % kBV, rr = x / kBV;
      float acc = 0.f;
#pragma unroll 8
      for (int j = 0; j < kChunk; ++j) acc += sm.M[rr][j] * vt[j * kBV + vv];
      const float *X = (rr < kChunk) ? &sm.bufD[rr][0] : &sm.bufB[rr - kChunk][0];
#pragma unroll 8
      for (int kk = 0; kk < K; ++kk) acc += X[kk] * sm.S[kk][vv];
      if (rr < kChunk) {
        U[rr * kBV + vv] = -acc;
      } else {
        const int i = rr - kChunk;
        if (i < L) p.o[tok_row(p, si.b, t0 + i, h) * p.V + v0 + vv] = __float2bfloat16_rn(p.scale * acc);
      }
    }
    __syncthreads();
    // -- S <- Diag(gamma) S + k~^T U
    for (int x = tid; x < K * kBV; x += kRecThreads) {
      const int vv = x % kBV, kk = x / kBV;
      float acc = 0.f;
#pragma unroll 8
      for (int i = 0; i < kChunk; ++i) acc += sm.bufC[i][kk] * U[i * kBV + vv];
      sm.S[kk][vv] = sm.gam[kk] * sm.S[kk][vv] + acc;
    }
    __syncthreads();
  }
  if (p.final_state) {
    for (int x = tid; x < K * kBV; x += kRecThreads) {
      const int kk = x % K, vv = x / K;
      p.final_state[(((long long)s * p.H + h) * p.V + v0 + vv) * K + kk] = sm.S[kk][vv];
    }
  }
}

template <int K>
static cudaError_t launch_recur_t(const Problem &p, cudaStream_t stream) {
  const size_t smem = sizeof(RecSmem<K>);
  cudaError_t e = cudaFuncSetAttribute(recur_simt_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.N * p.H * (p.V / kBV);
  recur_simt_kernel<K><<<(unsigned)grid, kRecThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_recur(const Problem &p, cudaStream_t stream) {
  if (p.N == 0) return cudaSuccess;
  return p.K == 64 ? launch_recur_t<64>(p, stream) : launch_recur_t<128>(p, stream);
}

}  // namespace kda
