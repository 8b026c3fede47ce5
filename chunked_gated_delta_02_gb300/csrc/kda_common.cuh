// Shared device-side definitions of the KDA chunked forward (sm_103a).
//
// Everything here is plumbing used by several kernels: the problem descriptor,
// the mapping from (sequence, chunk) to token rows, and a few hardware math
// instructions (ex2.approx / rcp.approx are single PTX instructions of the SFU;
// the FlashKDA page, section "저수준(Low-level) 명령어 및 메모리 활용", uses the
// same base-2 exponential trick).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "exp2_poly.cuh"

namespace kda {

constexpr int kChunk = 64;          // tokens per chunk
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNormEps = 1e-6f;   // L2-norm epsilon inside the square root

// Device data-error codes (mirrors KDA_DEVICE_* in include/kda.h).
constexpr int kDevOk = 0;
constexpr int kDevBadCuSeqlens = 1;
constexpr int kDevWaitTimeout = 2;
constexpr int kDevNonFinite = 3;     // the recurrence's last state of a (sequence, head) is not finite

// Variant flags (mirrors KDA_GATE_PER_HEAD, KDA_BETA_F32, KDA_STATE_BF16, KDA_STATE_KV in
// include/kda.h).
constexpr uint32_t kGatePerHead = 0x1u;   // g [B,T,H], dt_bias [H]: one decay per token and head
constexpr uint32_t kBetaF32 = 0x2u;       // beta logits in fp32
constexpr uint32_t kStateBf16 = 0x4u;     // initial / final state in bf16
constexpr uint32_t kStateKV = 0x8u;       // state layout [N,H,K,V] instead of [N,H,V,K]
constexpr uint32_t kExp2Poly = 0x10u;     // per-token decays 2^la by a polynomial on the FMA pipe
// Context parallelism (mirrors KDA_CP_OFF and KDA_CP_SEGMENTS(n) in include/kda.h): off, or forced
// with n segments in bits 8..15; otherwise chosen by the host plan (kda_cp.cu).
constexpr uint32_t kCpOff = 0x20u;
constexpr int kCpSegShift = 8;
constexpr uint32_t kCpFlagsMask = kCpOff | (0xFFu << kCpSegShift);

struct Problem {
  const __nv_bfloat16 *q, *k, *v, *g;  // g [B,T,H,K], or [B,T,H] with kGatePerHead
  const void *beta;                  // [B,T,H] logits, bf16 or fp32 (kBetaF32)
  const float *A_log, *dt_bias;      // dt_bias [H,K] ([H] with kGatePerHead) or null
  const void *init;                  // [N,H,V,K] or [N,H,K,V] (kStateKV), fp32 or bf16, or null
  void *final_state;                 // same type and layout as init, or null
  const int32_t *cu;                 // [N+1] or null (fixed length)
  __nv_bfloat16 *o;                  // [B,T,H,V]
  // prep -> recurrence hand-off: one block per (chunk, head) slot s = chunk * H + head at
  // hand + s * hand_stride, laid out as described at hand_off_* below; M of slot s is at
  // mats + s * mat_stride (inside the block, or in a caller buffer for the stage export)
  unsigned char *hand;
  long long hand_stride;             // bytes
  __half *mats;
  long long mat_stride;              // halves
  int32_t *chunk_off;                // [N+1] varlen chunk offsets (K0 output)
  int32_t *order;                    // [N] varlen longest-first order (K0 output)
  int32_t *flag;                     // per-call data-error flag (varlen) or null
  int *dev_status;                   // sticky per-device status word
  float lb, scale;
  int B, T, H, K, V, N;
  int nc_fixed;                      // ceil(T / C) in fixed-length mode
  long long max_chunks;
  uint32_t flags;                    // variant flags above
  // Context parallelism (kda_cp.cu): every sequence is cut into n_seg segments of whole chunks,
  // segment g holding chunks [n_c g / n_seg, n_c (g + 1) / n_seg) of its n_c.
  //   seg_state [N][n_seg][H][V + K][K] fp32: end state of each segment run from zero (value
  //             columns 0..V-1) and its transition (columns V + j: the state reached from the
  //             unit start column e_j with v = 0); for segment 0, the true end state (V columns)
  //   seg_start [N][n_seg][H][V][K] fp32: true start state of each segment
  int n_seg;
  float *seg_state;
  float *seg_start;
};

// Chunk range [lo, hi) of segment g of a sequence of n_c chunks cut into n_seg segments.
__host__ __device__ inline void segment_chunks(int n_c, int g, int n_seg, int &lo, int &hi) {
  lo = (int)((long long)n_c * g / n_seg);
  hi = (int)((long long)n_c * (g + 1) / n_seg);
}

// TMA descriptor of v, viewed as 4D [B][T][H][V] (innermost V) with a box of
// (V-slice width) columns x 1 head x 64 tokens x 1 batch row: one copy per chunk and
// V slice; tokens past T read as zeros.
struct TmaMaps {
  CUtensorMap v;
};

// Hand-off block of one (chunk, head) slot, in bytes. The images are stored in the 128-byte
// swizzled layout of the recurrence kernel's shared-memory operands (64-channel panels of 64
// token rows), so bulk copies place them:
//   [0, 16K)             M = [-Tb ; P Tb], 128 x 64 fp16, rows in swizzled order
//   [16K, 16K + 128K)    khat Gamma          (64 x K fp16)
//   next 128K bytes      qhat Gamma
//   next 128K bytes      khat Gamma_last / Gamma
//   next 4K bytes        Gamma_last (K fp32)
// M and khat Gamma are contiguous (one copy), and so are the last two.
constexpr long long kMatBytes = 2ll * kChunk * kChunk * 2;
__host__ __device__ constexpr long long hand_off_kg(int K) { return kMatBytes; }
__host__ __device__ constexpr long long hand_off_qt(int K) { return kMatBytes + 128ll * K; }
__host__ __device__ constexpr long long hand_off_kt(int K) { return kMatBytes + 256ll * K; }
__host__ __device__ constexpr long long hand_off_gam(int K) { return kMatBytes + 384ll * K; }
__host__ __device__ constexpr long long hand_bytes(int K) { return (kMatBytes + 388ll * K + 255) / 256 * 256; }

// Element index of S[k][v] of (sequence s, head h) in the state tensors, and the state's
// load and store in its storage type (the state is fp32 inside the kernels).
__device__ __forceinline__ long long state_index(const Problem &p, int s, int h, int k, int v) {
  return (p.flags & kStateKV) ? (((long long)s * p.H + h) * p.K + k) * p.V + v
                              : (((long long)s * p.H + h) * p.V + v) * p.K + k;
}
__device__ __forceinline__ float state_load(const Problem &p, long long i) {
  return (p.flags & kStateBf16) ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.init)[i])
                                : static_cast<const float *>(p.init)[i];
}
__device__ __forceinline__ void state_store(const Problem &p, long long i, float x) {
  if (p.flags & kStateBf16) static_cast<__nv_bfloat16 *>(p.final_state)[i] = __float2bfloat16_rn(x);
  else static_cast<float *>(p.final_state)[i] = x;
}

// Host: per-device state set once per process. A kernel's dynamic shared-memory limit and the SM
// count are device properties; the per-call launch path only looks them up after the first call
// on a device. (Up to 64 devices; beyond that the calls are simply made every time.)
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};
  // runs f() the first time it is called for the current device; f returns cudaSuccess on success
  template <typename F>
  cudaError_t operator()(F &&f) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t e = f(dev);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// Programmatic dependent launch (PTX griddepcontrol). A kernel launched with `overlap` set
// (launch_kernel below) may be scheduled before the kernel ahead of it in the stream has
// finished, once every CTA of that kernel has called pdl_launch_dependents() or exited; it
// must call pdl_wait(), which returns once the kernel ahead has completed and its writes are
// visible, before it reads or writes anything that kernel touches. Without the launch
// attribute pdl_wait() returns at once.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool overlap, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
  const cudaError_t last = cudaGetLastError();
  return e != cudaSuccess ? e : last;
}

struct SeqInfo {
  int b;        // batch row
  int t0;       // first token
  int len;      // number of tokens
  int chunk0;   // global chunk index of the first chunk
};

__device__ __forceinline__ SeqInfo seq_info(const Problem &p, int s) {
  SeqInfo r;
  if (p.cu) {
    r.b = 0;
    r.t0 = p.cu[s];
    r.len = p.cu[s + 1] - r.t0;
    r.chunk0 = p.chunk_off[s];
  } else {
    r.b = s;
    r.t0 = 0;
    r.len = p.T;
    r.chunk0 = s * p.nc_fixed;
  }
  return r;
}

// Row index of token t of batch row b, head h in a [B,T,H,*] tensor.
__device__ __forceinline__ long long tok_row(const Problem &p, int b, int t, int h) {
  return ((long long)b * p.T + t) * p.H + h;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x on the FMA pipe instead of the SFU, for x >= -126 (smaller x give 0, as the flush-to-zero
// ex2.approx does): n = round(x) by adding and subtracting 1.5 * 2^23 (the sum's low mantissa bits
// hold round(x)), f = x - n in [-1/2, 1/2], 2^f by the fitted polynomial of exp2_poly.cuh in
// Horner form, and 2^n added to the exponent field. Relative error about 1.1e-7 plus the
// rounding of five fused multiply-adds.
__device__ __forceinline__ float ex2_poly(float x) {
  const float xc = fmaxf(x, -126.f);
  const float t = xc + 12582912.f;
  const float f = xc - (t - 12582912.f);
  float p = kExp2PolyC5;
  p = fmaf(p, f, kExp2PolyC4);
  p = fmaf(p, f, kExp2PolyC3);
  p = fmaf(p, f, kExp2PolyC2);
  p = fmaf(p, f, kExp2PolyC1);
  p = fmaf(p, f, kExp2PolyC0);
  const uint32_t n = (uint32_t)(__float_as_int(t) - 0x4B400000);   // round(x) (two's complement)
  const float r = __int_as_float((int)((uint32_t)__float_as_int(p) + (n << 23)));
  return x < -126.f ? 0.f : r;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Logistic function from one base-2 exponential and one reciprocal.
// Saturates correctly: x -> +inf gives 1, x -> -inf gives 0.
__device__ __forceinline__ float sigmoid_fast(float x) {
  return rcp_approx(1.0f + ex2_approx(-x * kLog2e));
}

// Per-token base-2 log decay:  log2(alpha) = lb * log2(e) * sigmoid(ea * (g + dt)).
__device__ __forceinline__ float log2_decay(float g, float dt, float ea, float lb_log2e) {
  return lb_log2e * sigmoid_fast(ea * (g + dt));
}

__device__ __forceinline__ float to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// 16-byte global -> shared asynchronous copy (L2 only); src_valid == false zero-fills.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool src_valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
               "r"(src_valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Stage rows [0, 64) of a chunk of a [B,T,H,D] bf16 tensor into shared memory
// as bf16 [64][D] (rows >= L zero-filled). D * 2 bytes must be a multiple of 16.
template <int D, int NT>
__device__ __forceinline__ void stage_rows_async(__nv_bfloat16 *dst, const __nv_bfloat16 *src, const Problem &p,
                                                 int b, int t0, int h, int L, int col0, int ld, int tid) {
  constexpr int kChunks = D * 2 / 16;   // 16-byte chunks per row
  for (int x = tid; x < kChunk * kChunks; x += NT) {
    const int i = x / kChunks, c = x % kChunks;
    const bool ok = i < L;
    const __nv_bfloat16 *g = ok ? src + tok_row(p, b, t0 + i, h) * ld + col0 + c * 8 : src;
    cp_async16(dst + i * D + c * 8, g, ok);
  }
}

// Global chunk index -> sequence (binary search over the varlen chunk offsets).
__device__ __forceinline__ int chunk_to_seq(const Problem &p, long long c) {
  if (!p.cu) return (int)(c / p.nc_fixed);
  int lo = 0, hi = p.N;  // chunk_off[lo] <= c < chunk_off[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (p.chunk_off[mid] <= c) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace kda
