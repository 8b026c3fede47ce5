// K0: varlen scheduler for packed sequences (cu_seqlens).
//
// Packed variable-length input with int32 cu_seqlens is how the cuLA README
// (shadowgraph.io mirror, "Quick Start" notes) and the FlashKDA FLA example
// (FlashKDA page, section "flash-linear-attention 백엔드로 사용") pass ragged
// batches. One CTA:
//   1. checks cu_seqlens (starts at 0, never decreases, ends at T) and raises
//      the per-call flag plus the sticky device status on a violation;
//   2. writes chunk_off[s] = sum_{j<s} ceil(len_j / 64) (exclusive scan);
//   3. writes a longest-first order of the sequences (counting sort on the
//      chunk count), so that the recurrence kernel starts the longest
//      sequential chains first.
// Everything stays on the device: the host never waits for the schedule.
#include "kda_common.cuh"

namespace kda {

constexpr int kSchedThreads = 1024;
constexpr int kSchedBins = 8192;   // counting-sort bins (chunk counts) held in shared memory

__global__ void __launch_bounds__(kSchedThreads)
varlen_schedule_kernel(const int32_t *__restrict__ cu, int N, int T, int32_t *__restrict__ chunk_off,
                       int32_t *__restrict__ order, int32_t *__restrict__ flag,
                       int *__restrict__ dev_status) {
  __shared__ int s_bad;
  __shared__ int s_scan[kSchedThreads];
  __shared__ int s_bins[kSchedBins];
  pdl_launch_dependents();   // the prep kernel's CTAs may take their SMs now and wait there
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = (cu[0] != 0 || cu[N] != T) ? 1 : 0;
  __syncthreads();
  for (int i = tid; i < N; i += kSchedThreads)
    if (cu[i + 1] < cu[i]) atomicOr(&s_bad, 1);
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      *flag = kDevBadCuSeqlens;
      atomicExch(dev_status, kDevBadCuSeqlens);
    }
    return;
  }
  if (tid == 0) *flag = kDevOk;

  // Exclusive scan of chunk counts, in tiles of kSchedThreads with a carry.
  int carry = 0;
  for (int base = 0; base < N; base += kSchedThreads) {
    const int i = base + tid;
    const int nc = (i < N) ? (cu[i + 1] - cu[i] + kChunk - 1) / kChunk : 0;
    s_scan[tid] = nc;
    __syncthreads();
    for (int off = 1; off < kSchedThreads; off <<= 1) {  // Hillis-Steele inclusive scan
      const int x = (tid >= off) ? s_scan[tid - off] : 0;
      __syncthreads();
      s_scan[tid] += x;
      __syncthreads();
    }
    if (i < N) chunk_off[i] = carry + s_scan[tid] - nc;
    carry += s_scan[kSchedThreads - 1];
    __syncthreads();
  }
  if (tid == 0) chunk_off[N] = carry;

  // Longest-first order: counting sort on the chunk count, descending.
  const int max_nc = (T + kChunk - 1) / kChunk;
  if (max_nc + 1 > kSchedBins) {  // too many distinct lengths for the bins: keep input order
    for (int i = tid; i < N; i += kSchedThreads) order[i] = i;
    return;
  }
  for (int b = tid; b <= max_nc; b += kSchedThreads) s_bins[b] = 0;
  __syncthreads();
  for (int i = tid; i < N; i += kSchedThreads)
    atomicAdd(&s_bins[(cu[i + 1] - cu[i] + kChunk - 1) / kChunk], 1);
  __syncthreads();
  // bins -> start positions, longest (largest count) first: an exclusive scan
  // over the bins in descending order, 8 bins per thread.
  constexpr int kPer = kSchedBins / kSchedThreads;
  int local[kPer];
  int lsum = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = max_nc - (tid * kPer + j);
    local[j] = (b >= 0) ? s_bins[b] : 0;
    lsum += local[j];
  }
  s_scan[tid] = lsum;
  __syncthreads();
  for (int off = 1; off < kSchedThreads; off <<= 1) {
    const int x = (tid >= off) ? s_scan[tid - off] : 0;
    __syncthreads();
    s_scan[tid] += x;
    __syncthreads();
  }
  int pos = s_scan[tid] - lsum;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = max_nc - (tid * kPer + j);
    if (b >= 0) s_bins[b] = pos;
    pos += local[j];
  }
  __syncthreads();
  for (int i = tid; i < N; i += kSchedThreads) {
    const int b = (cu[i + 1] - cu[i] + kChunk - 1) / kChunk;
    order[atomicAdd(&s_bins[b], 1)] = i;
  }
}

cudaError_t launch_varlen_schedule(const Problem &p, cudaStream_t stream) {
  varlen_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(p.cu, p.N, p.T, p.chunk_off, p.order,
                                                          p.flag, p.dev_status);
  return cudaGetLastError();
}

}  // namespace kda
