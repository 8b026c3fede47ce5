// Host side of the C ABI declared in include/kda.h: argument validation,
// workspace layout, and the K0 -> K1 -> K2 launch sequence on one stream.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "umma.cuh"

namespace kda {
cudaError_t launch_varlen_schedule(const Problem &p, cudaStream_t stream);
// overlap: launch so that the kernel may be scheduled while the kernel ahead of it in the stream
// (the schedule kernel, the prep kernel) is still running
cudaError_t launch_prep(const Problem &p, cudaStream_t stream, bool overlap);
cudaError_t launch_recur(const Problem &p, const TmaMaps &maps, int bv, cudaStream_t stream, bool overlap);
cudaError_t launch_recur_segments(const Problem &p, const TmaMaps &maps, int pass, cudaStream_t stream,
                                  bool overlap);
cudaError_t launch_cp_combine(const Problem &p, cudaStream_t stream);
int recur_slice_width(const Problem &p);
int slice_width_for(long long N, int H, int V, int sms);
int device_sm_count();
int cp_max_segments(int T, int H, int V, int N, bool varlen, uint32_t cp_flags);
int cp_auto_segments(int T, int H, int K, int V, int N, int sms, int n_max, int plain_bv);
}  // namespace kda

// Sticky per-device data-error word (KDA_DEVICE_* codes).
static __device__ int g_kda_device_status = 0;

// One bounded wait on an mbarrier that nothing arrives on (see kda_debug_wait_timeout).
static __global__ void wait_timeout_kernel(long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    kda::umma::mbar_init(&bar, 1);
    kda::umma::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !kda::umma::mbar_wait_bounded(&bar, 0, limit))
    atomicExch(&g_kda_device_status, kda::kDevWaitTimeout);
}

// NVTX range for the host-side enqueue of one stage (shows up around the launches in a trace).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t flag_off, chunk_off_off, order_off, hand_off, hand_stride, seg_state_off, seg_start_off, total;
  int n_seg_max;   // segments the context-parallel buffers hold (0: none)
};

bool sizes_ok(int B, int T, int H, int K, int V, int N) {
  return B >= 1 && T >= 0 && H >= 1 && K >= 1 && V >= 1 && N >= 0;
}

int64_t max_chunks_of(int B, int T, int N) {
  return (int64_t)B * ((T + kda::kChunk - 1) / kda::kChunk) + (int64_t)N;
}

Layout layout_of(int B, int T, int H, int K, int V, int N, int n_seg_max) {
  Layout L;
  size_t off = 0;
  L.flag_off = off;
  off = align_up(off + sizeof(int32_t));
  L.chunk_off_off = off;
  off = align_up(off + sizeof(int32_t) * ((size_t)N + 1));
  L.order_off = off;
  off = align_up(off + sizeof(int32_t) * ((size_t)N + 1));
  const size_t ch = (size_t)max_chunks_of(B, T, N) * (size_t)H;   // (chunk, head) slots
  L.hand_off = off;
  L.hand_stride = (size_t)kda::hand_bytes(K);
  off = align_up(off + ch * L.hand_stride);
  L.n_seg_max = n_seg_max;
  const size_t seg_blocks = (size_t)N * (size_t)(n_seg_max > 1 ? n_seg_max : 0) * (size_t)H;
  L.seg_state_off = off;
  off = align_up(off + seg_blocks * (size_t)(V + K) * K * sizeof(float));
  L.seg_start_off = off;
  off = align_up(off + seg_blocks * (size_t)V * K * sizeof(float));
  L.total = off;
  return L;
}

bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

// 4D view [B][T][H][D] of a 16-bit token tensor, box = (box_d, 1, 64, 1).
bool encode_token_map(CUtensorMap *m, const void *base, int D, int H, int T, int B, int box_d,
                      CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
  const cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)kda::kChunk, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, dtype, 4, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

kda_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// Segments per sequence of context parallelism (0: the plain recurrence): forced by
// KDA_CP_SEGMENTS, or where the host plan (kda_cp.cu) estimates a clear gain on this device.
int cp_segments_of(int n_seg_max, uint32_t flags, int T, int H, int K, int V, int N, int plain_bv) {
  if (n_seg_max < 2) return 0;
  if ((flags >> kda::kCpSegShift) & 0xFFu) return n_seg_max;
  return kda::cp_auto_segments(T, H, K, V, N, kda::device_sm_count(), n_seg_max, plain_bv);
}

static_assert(KDA_GATE_PER_HEAD == kda::kGatePerHead && KDA_BETA_F32 == kda::kBetaF32 &&
                  KDA_STATE_BF16 == kda::kStateBf16 && KDA_STATE_KV == kda::kStateKV &&
                  KDA_EXP2_POLY == kda::kExp2Poly,
              "variant flags of include/kda.h and the kernels");
static_assert(KDA_CP_OFF == kda::kCpOff && KDA_CP_SEGMENTS(3) == (3u << kda::kCpSegShift),
              "context-parallel flags of include/kda.h and the kernels");
constexpr uint32_t kAllFlags = KDA_GATE_PER_HEAD | KDA_BETA_F32 | KDA_STATE_BF16 | KDA_STATE_KV | KDA_EXP2_POLY |
                               KDA_CP_OFF | KDA_CP_SEGMENTS(0xFFu);

// Context-parallel part of the flags: at most one of KDA_CP_OFF and KDA_CP_SEGMENTS(n), n in [2, 64].
bool cp_flags_ok(uint32_t flags) {
  const uint32_t n = (flags >> kda::kCpSegShift) & 0xFFu;
  if (n == 0) return true;
  return !(flags & KDA_CP_OFF) && n >= 2 && n <= 64;
}

// Shared argument checks of kda_fwd_ex and kda_debug_chunk_matrices.
kda_status_t check_common(const void *q, const void *k, const void *g, const void *beta,
                          const float *A_log, const float *dt_bias, float lower_bound,
                          const int32_t *cu_seqlens, int B, int T, int H, int K, int num_seqs,
                          uint32_t flags) {
  if ((flags & ~kAllFlags) || !cp_flags_ok(flags)) return KDA_ERR_INVALID_ARG;
  if (!sizes_ok(B, T, H, K, K, num_seqs)) return KDA_ERR_INVALID_ARG;
  // token tensors may be null only when they hold no elements (T == 0)
  if (!A_log || (T > 0 && (!q || !k || !g || !beta))) return KDA_ERR_INVALID_ARG;
  if (K != 64 && K != 128) return KDA_ERR_UNSUPPORTED;
  if (!std::isfinite(lower_bound) || lower_bound < -5.0f || lower_bound > 0.0f) return KDA_ERR_INVALID_ARG;
  if (cu_seqlens) {
    if (B != 1) return KDA_ERR_INVALID_ARG;
    if (!aligned(cu_seqlens, 4)) return KDA_ERR_INVALID_ARG;
  } else if (num_seqs != B) {
    return KDA_ERR_INVALID_ARG;
  }
  const bool per_head = (flags & KDA_GATE_PER_HEAD) != 0;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(g, per_head ? 2 : 16) ||
      !aligned(beta, (flags & KDA_BETA_F32) ? 4 : 2) || !aligned(A_log, 4) ||
      (dt_bias && !aligned(dt_bias, per_head ? 4 : 16)))
    return KDA_ERR_INVALID_ARG;
  // element counts must fit the 64-bit index arithmetic of the kernels
  const double elems = (double)B * (double)T * (double)H * (double)K;
  if (elems > 9.0e15) return KDA_ERR_INVALID_ARG;
  if ((double)max_chunks_of(B, T, num_seqs) * H > 2.0e9) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

struct Scratch {
  void *ptr = nullptr;
  bool owned = false;
};

kda_status_t get_scratch(void *workspace, size_t workspace_bytes, size_t need, cudaStream_t stream,
                         Scratch &out) {
  if (workspace) {
    if (workspace_bytes < need || !aligned(workspace, kAlign)) return KDA_ERR_WORKSPACE;
    out.ptr = workspace;
    out.owned = false;
    return KDA_OK;
  }
  if (cudaMallocAsync(&out.ptr, need, stream) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_WORKSPACE;
  }
  out.owned = true;
  return KDA_OK;
}

void release_scratch(Scratch &s, cudaStream_t stream) {
  if (s.owned && s.ptr) cudaFreeAsync(s.ptr, stream);
  s.ptr = nullptr;
}

kda_status_t fill_problem(kda::Problem &p, const Layout &L, void *ws, const void *q, const void *k,
                          const void *v, const void *g, const void *beta, const float *A_log,
                          const float *dt_bias, float lower_bound, float scale,
                          const void *initial_state, void *final_state, const int32_t *cu,
                          int B, int T, int H, int K, int V, int N, uint32_t flags, void *o) {
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.k = static_cast<const __nv_bfloat16 *>(k);
  p.v = static_cast<const __nv_bfloat16 *>(v);
  p.g = static_cast<const __nv_bfloat16 *>(g);
  p.beta = beta;
  p.flags = flags;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.init = initial_state;
  p.final_state = final_state;
  p.cu = cu;
  p.o = static_cast<__nv_bfloat16 *>(o);
  char *base = static_cast<char *>(ws);
  p.flag = cu ? reinterpret_cast<int32_t *>(base + L.flag_off) : nullptr;
  p.chunk_off = reinterpret_cast<int32_t *>(base + L.chunk_off_off);
  p.order = reinterpret_cast<int32_t *>(base + L.order_off);
  p.hand = reinterpret_cast<unsigned char *>(base + L.hand_off);
  p.hand_stride = (long long)L.hand_stride;
  p.seg_state = reinterpret_cast<float *>(base + L.seg_state_off);
  p.seg_start = reinterpret_cast<float *>(base + L.seg_start_off);
  p.n_seg = 0;
  p.mats = reinterpret_cast<__half *>(p.hand);
  p.mat_stride = p.hand_stride / 2;
  static kda::PerDeviceOnce once;
  static std::atomic<int *> status_addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  const cudaError_t e = once([&](int d) {
    int *a = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(reinterpret_cast<void **>(&a), g_kda_device_status);
    if (r == cudaSuccess && d >= 0 && d < 64) status_addr[d].store(a, std::memory_order_relaxed);
    return r;
  });
  p.dev_status = (dev >= 0 && dev < 64) ? status_addr[dev].load(std::memory_order_relaxed) : nullptr;
  if (e == cudaSuccess && !p.dev_status &&
      cudaGetSymbolAddress(reinterpret_cast<void **>(&p.dev_status), g_kda_device_status) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  p.lb = lower_bound;
  p.scale = scale;
  p.B = B;
  p.T = T;
  p.H = H;
  p.K = K;
  p.V = V;
  p.N = N;
  p.nc_fixed = (T + kda::kChunk - 1) / kda::kChunk;
  p.max_chunks = cu ? max_chunks_of(1, T, N) : (long long)B * p.nc_fixed;
  return KDA_OK;
}

}  // namespace

extern "C" {

int kda_version(void) { return 100; }

int64_t kda_max_chunks(int B, int T, int num_seqs) {
  if (B < 1 || T < 0 || num_seqs < 0) return 0;
  return max_chunks_of(B, T, num_seqs);
}

size_t kda_fwd_workspace_size_ex(int B, int T, int H, int K, int V, int num_seqs, int varlen, uint32_t flags) {
  if (!sizes_ok(B, T, H, K, V, num_seqs) || !cp_flags_ok(flags)) return 0;
  const int n_max = kda::cp_max_segments(T, H, V, num_seqs, varlen != 0, flags);
  return layout_of(B, T, H, K, V, num_seqs, n_max).total;
}

size_t kda_fwd_workspace_size(int B, int T, int H, int K, int V, int num_seqs) {
  return kda_fwd_workspace_size_ex(B, T, H, K, V, num_seqs, 0, 0u);
}

const char *kda_status_string(kda_status_t s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported head dimension or size";
    case KDA_ERR_WORKSPACE: return "workspace too small, misaligned, or allocation failed";
    case KDA_ERR_CUDA: return "CUDA runtime error";
    case KDA_ERR_DEVICE_STATUS: return "device reported a data error";
  }
  return "unknown status";
}

kda_status_t kda_get_device_status(kda_stream_t stream, int *device_code) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
  int code = 0;
  if (cudaMemcpyFromSymbol(&code, g_kda_device_status, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_kda_device_status, &zero, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
  if (device_code) *device_code = code;
  return code == 0 ? KDA_OK : KDA_ERR_DEVICE_STATUS;
}

kda_status_t kda_fwd_with_events(const void *q, const void *k, const void *v, const void *g,
                                 const void *beta, const float *A_log, const float *dt_bias,
                                 float lower_bound, float scale, const float *initial_state,
                                 float *final_state, const int32_t *cu_seqlens, int B, int T, int H,
                                 int K, int V, int num_seqs, void *o, void *workspace,
                                 size_t workspace_bytes, kda_stream_t stream,
                                 const kda_stage_events_t *events) {
  return kda_fwd_ex(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state, final_state,
                    cu_seqlens, B, T, H, K, V, num_seqs, 0u, o, workspace, workspace_bytes, stream, events);
}

kda_status_t kda_fwd_ex(const void *q, const void *k, const void *v, const void *g, const void *beta,
                        const float *A_log, const float *dt_bias, float lower_bound, float scale,
                        const void *initial_state, void *final_state, const int32_t *cu_seqlens, int B,
                        int T, int H, int K, int V, int num_seqs, uint32_t flags, void *o,
                        void *workspace, size_t workspace_bytes, kda_stream_t stream,
                        const kda_stage_events_t *events) {
  kda_status_t st = check_common(q, k, g, beta, A_log, dt_bias, lower_bound, cu_seqlens, B, T, H, K,
                                 num_seqs, flags);
  if (st != KDA_OK) return st;
  if (V < 1) return KDA_ERR_INVALID_ARG;
  if (T > 0 && (!v || !o)) return KDA_ERR_INVALID_ARG;
  if (V != 64 && V != 128) return KDA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
  if (!aligned(v, 16) || !aligned(o, 16) || (initial_state && !aligned(initial_state, 16)) ||
      (final_state && !aligned(final_state, 16)))
    return KDA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (num_seqs == 0) return KDA_OK;
  const Layout L = layout_of(B, T, H, K, V, num_seqs,
                             kda::cp_max_segments(T, H, V, num_seqs, cu_seqlens != nullptr, flags));
  Scratch scr;
  st = get_scratch(workspace, workspace_bytes, L.total, s, scr);
  if (st != KDA_OK) return st;
  kda::Problem p;
  st = fill_problem(p, L, scr.ptr, q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                    final_state, cu_seqlens, B, T, H, K, V, num_seqs, flags & ~kda::kCpFlagsMask, o);
  auto mark = [&](void *ev) {
    if (st == KDA_OK && ev) st = from_cuda(cudaEventRecord(static_cast<cudaEvent_t>(ev), s));
  };
  mark(events ? events->prep_start : nullptr);
  if (st == KDA_OK && cu_seqlens) {
    NvtxRange r("kda K0 varlen schedule");
    st = from_cuda(kda::launch_varlen_schedule(p, s));
  }
  if (st == KDA_OK) {
    NvtxRange r("kda K1 prep");
    st = from_cuda(kda::launch_prep(p, s, cu_seqlens != nullptr));
  }
  // With an event recorded between them the two kernels run one after the other, so that the
  // event splits the time between them; otherwise the recurrence kernel's launch overlaps the end
  // of the prep kernel.
  const bool split = events && events->prep_done;
  mark(split ? events->prep_done : nullptr);
  kda::TmaMaps maps;
  std::memset(&maps, 0, sizeof maps);
  const int bv = kda::recur_slice_width(p);
  p.n_seg = cp_segments_of(L.n_seg_max, flags, T, H, K, V, num_seqs, bv);
  const int map_bv = p.n_seg >= 2 ? 64 : bv;
  if (st == KDA_OK && T > 0 && !encode_token_map(&maps.v, v, V, H, T, B, map_bv)) st = KDA_ERR_CUDA;
  if (st == KDA_OK && p.n_seg >= 2) {
    NvtxRange r("kda K2 recurrence, context parallel");
    st = from_cuda(kda::launch_recur_segments(p, maps, 1, s, !split));
    if (st == KDA_OK) st = from_cuda(kda::launch_cp_combine(p, s));
    if (st == KDA_OK) st = from_cuda(kda::launch_recur_segments(p, maps, 2, s, false));
  } else if (st == KDA_OK) {
    NvtxRange r("kda K2 recurrence");
    st = from_cuda(kda::launch_recur(p, maps, bv, s, !split));
  }
  mark(events ? events->recur_done : nullptr);
  release_scratch(scr, s);
  return st;
}

kda_status_t kda_fwd_plan(int B, int T, int H, int K, int V, int num_seqs, int varlen, uint32_t flags,
                          int *n_segments, int *slice_width) {
  if (!sizes_ok(B, T, H, K, V, num_seqs) || (flags & ~kAllFlags) || !cp_flags_ok(flags))
    return KDA_ERR_INVALID_ARG;
  if ((K != 64 && K != 128) || (V != 64 && V != 128)) return KDA_ERR_UNSUPPORTED;
  const int sms = kda::device_sm_count();
  if (sms <= 0) return KDA_ERR_CUDA;
  const int bv = kda::slice_width_for(num_seqs, H, V, sms);
  const int n_max = kda::cp_max_segments(T, H, V, num_seqs, varlen != 0, flags);
  const int n_seg = cp_segments_of(n_max, flags, T, H, K, V, num_seqs, bv);
  if (n_segments) *n_segments = n_seg;
  if (slice_width) *slice_width = n_seg >= 2 ? 64 : bv;
  return KDA_OK;
}

kda_status_t kda_debug_wait_timeout(long long limit_cycles, kda_stream_t stream) {
  if (limit_cycles < 1 || limit_cycles >= (1ll << 32)) return KDA_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_cycles);
  return from_cuda(cudaGetLastError());
}

kda_status_t kda_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                     const float *A_log, const float *dt_bias, float lower_bound, float scale,
                     const float *initial_state, float *final_state, const int32_t *cu_seqlens,
                     int B, int T, int H, int K, int V, int num_seqs, void *o, void *workspace,
                     size_t workspace_bytes, kda_stream_t stream) {
  return kda_fwd_with_events(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                             final_state, cu_seqlens, B, T, H, K, V, num_seqs, o, workspace,
                             workspace_bytes, stream, nullptr);
}

kda_status_t kda_debug_chunk_matrices(const void *q, const void *k, const void *g, const void *beta,
                                      const float *A_log, const float *dt_bias, float lower_bound,
                                      const int32_t *cu_seqlens, int B, int T, int H, int K,
                                      int num_seqs, void *chunk_mats, void *workspace,
                                      size_t workspace_bytes, kda_stream_t stream) {
  kda_status_t st = check_common(q, k, g, beta, A_log, dt_bias, lower_bound, cu_seqlens, B, T, H, K,
                                 num_seqs, 0u);
  if (st != KDA_OK) return st;
  if (!chunk_mats || !aligned(chunk_mats, 16)) return KDA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (num_seqs == 0) return KDA_OK;
  const Layout L = layout_of(B, T, H, K, K, num_seqs, 0);
  Scratch scr;
  st = get_scratch(workspace, workspace_bytes, L.total, s, scr);
  if (st != KDA_OK) return st;
  kda::Problem p;
  st = fill_problem(p, L, scr.ptr, q, k, k, g, beta, A_log, dt_bias, lower_bound, 1.0f, nullptr, nullptr,
                    cu_seqlens, B, T, H, K, K, num_seqs, 0u, nullptr);
  p.mats = static_cast<__half *>(chunk_mats);
  p.mat_stride = 2 * kda::kChunk * kda::kChunk;
  if (st == KDA_OK && cu_seqlens) st = from_cuda(kda::launch_varlen_schedule(p, s));
  if (st == KDA_OK) st = from_cuda(kda::launch_prep(p, s, cu_seqlens != nullptr));
  release_scratch(scr, s);
  return st;
}

}  // extern "C"
