// Intracard context parallelism for long sequences: the segments of a sequence run in parallel.
//
// The recurrence of one (sequence, head) is sequential over its chunks, so a problem with few
// sequences and heads leaves most SMs idle however narrow the V slices (the cuLA README mirror,
// section "Benchmarks", reports the FlashKDA intracard CP; the FlashQLA page, section "핵심 기능",
// names gate-driven automatic intracard context parallelism). The chunk recurrence is affine in the
// state: over a segment of chunks, S_end = Phi S_start + S_loc, where S_loc is the end state of the
// segment run from a zero state and Phi (K x K) is the product of the per-chunk transitions
// Diag(gamma) - k~^T w. Running the same recurrence from the start state e_j (column j of the
// identity) with v = 0 gives column j of Phi. So:
//
//   pass 1 (recurrence kernel, kSegLocal): every segment but the last, all at once. Segment 0
//           starts from the true initial state and writes its o; segments g >= 1 start from zero
//           and carry K extra state columns from the identity, giving [S_loc | Phi].
//   combine (this file): start(1) = end(0); start(g + 1) = Phi_g start(g) + S_loc_g.
//   pass 2 (recurrence kernel, kSegFinal): every segment but the first, all at once, from its
//           true start state, writing o and, for the last segment, the final state.
//
// This costs about (3 n - 4) / n times the recurrence work of the plain kernel (with K = V) for a
// critical path of about 2 / n of it, so it pays only where the plain kernel leaves SMs idle; the
// host plan below estimates both and picks. Segments are whole chunks, so the in-chunk algebra is
// unchanged; only the last segment of a sequence can end with a partial chunk.
#include "kda_common.cuh"

namespace kda {

// One CTA per (sequence, head, 32 value columns); 256 threads. Thread (k, cg) owns state row k of
// the columns [cg * CPT, cg * CPT + CPT) of the tile, S[c][k] = S_state[k][c0 + c], in fp32.
template <int K>
__global__ void __launch_bounds__(256) cp_combine_kernel(const Problem p) {
  constexpr int kCols = 32, CPT = kCols * K / 256;
  __shared__ float S[kCols][K];
  const int sh = blockIdx.x;
  const int s = sh / p.H, h = sh % p.H;
  const int c0 = blockIdx.y * kCols;
  const int k = threadIdx.x % K, cb = (threadIdx.x / K) * CPT;
  const int V = p.V;
  auto state_blk = [&](int g) -> const float * {
    return p.seg_state + (((long long)s * p.n_seg + g) * p.H + h) * (long long)(V + K) * K;
  };
  const float *e0 = state_blk(0);   // true end state of segment 0 (value columns)
#pragma unroll
  for (int c = 0; c < CPT; ++c) S[cb + c][k] = e0[(long long)(c0 + cb + c) * K + k];
  __syncthreads();
  for (int g = 1; g < p.n_seg; ++g) {
    float *dst = p.seg_start + (((long long)s * p.n_seg + g) * p.H + h) * (long long)V * K;
#pragma unroll
    for (int c = 0; c < CPT; ++c) dst[(long long)(c0 + cb + c) * K + k] = S[cb + c][k];
    if (g == p.n_seg - 1) break;
    // start(g + 1)[k][c] = sum_j Phi_g[k][j] start(g)[j][c] + S_loc_g[k][c], Phi_g[k][j] stored at
    // column V + j, row k of segment g's block
    const float *blk = state_blk(g);
    float acc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) acc[c] = blk[(long long)(c0 + cb + c) * K + k];
#pragma unroll 8
    for (int j = 0; j < K; ++j) {
      const float phi = blk[(long long)(V + j) * K + k];
#pragma unroll
      for (int c = 0; c < CPT; ++c) acc[c] = fmaf(phi, S[cb + c][j], acc[c]);
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < CPT; ++c) S[cb + c][k] = acc[c];
    __syncthreads();
  }
}

cudaError_t launch_cp_combine(const Problem &p, cudaStream_t stream) {
  if (p.N == 0 || p.n_seg < 2) return cudaSuccess;
  const dim3 grid((unsigned)(p.N * p.H), (unsigned)(p.V / 32));
  if (p.K == 64) cp_combine_kernel<64><<<grid, 256, 0, stream>>>(p);
  else cp_combine_kernel<128><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// Host plan: the largest segment count the workspace is sized for, and the automatic choice.
//
// Automatic context parallelism is considered for fixed-length batches whose plain recurrence
// cannot fill a large GPU even with 16-column V slices (N H V / 16 < 256 CTAs), with segments of
// at least 16 chunks and at most 16 segments.
int cp_max_segments(int T, int H, int V, int N, bool varlen, uint32_t cp_flags) {
  if (varlen || (cp_flags & kCpOff) || N == 0 || T == 0) return 0;
  const int n_c = (T + kChunk - 1) / kChunk;
  const int forced = (int)((cp_flags >> kCpSegShift) & 0xFFu);
  if (forced) return forced >= 2 ? forced : 0;
  if ((long long)N * H * (V / 16) >= 256) return 0;
  const int n = std::min(16, n_c / 16);
  return n >= 2 ? n : 0;
}

// Estimated time (SM cycles) of the plain recurrence and of context parallelism with n segments,
// from the measured chain periods per chunk of the recurrence kernel on GB300: about 3.05k cycles
// with 64-column slices and 2.15k with 16-column slices (the kernel is bound by that chain, so a
// wave of CTAs takes its chunk count times the period).
int cp_auto_segments(int T, int H, int K, int V, int N, int sms, int n_max, int plain_bv) {
  if (n_max < 2 || sms <= 0) return 0;
  const double c64 = 3050.0, c16 = 2150.0, combine_step = 6000.0, extra_launches = 10000.0;
  const long long n_c = (T + kChunk - 1) / kChunk;
  auto waves = [&](long long ctas) { return (double)((ctas + sms - 1) / sms); };
  const double t_plain = waves((long long)N * H * (V / plain_bv)) * n_c * (plain_bv == 64 ? c64 : c16);
  int best = 0;
  double t_best = 0.85 * t_plain;   // a clear gain only
  for (int n = 2; n <= n_max; ++n) {
    const long long m = (n_c + n - 1) / n;
    const long long ctas1 = (long long)N * H * (V / 64 + (long long)(n - 2) * ((V + K) / 64));
    const long long ctas2 = (long long)N * H * (n - 1) * (V / 64);
    const double t = (waves(ctas1) + waves(ctas2)) * m * c64 + (n - 2) * combine_step + extra_launches;
    if (t < t_best) {
      t_best = t;
      best = n;
    }
  }
  return best;
}

}  // namespace kda
