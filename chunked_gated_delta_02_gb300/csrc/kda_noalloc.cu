// kda_fwd_noalloc(): the KDA forward for callers that are not allowed to
// allocate device memory.
//
// Some hosts of this library own every byte of device memory themselves: a
// serving runtime that reserves the whole GPU pool at start-up and hands a
// kernel plug-in only its input and output buffers, or a latency-critical
// path where a cudaMalloc / cudaMallocAsync (which can synchronise the device
// or grow a memory pool) is not permitted. kda_fwd() needs scratch memory for
// the prep -> recurrence hand-off and either takes it from the caller or
// allocates it; this entry point instead uses a fixed array that is part of
// the loaded library image, so it allocates nothing at all.
//
// The array lives in device global memory of every GPU that loads the
// library, for as long as the library stays loaded. In host code its name is
// only a host-side stand-in; the real device address is obtained once per
// device with cudaGetSymbolAddress() while that device is current, and that
// address is what the kernels receive.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda.h"

static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_MAX_SCRATCH];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device ordinal

// Device address of the scratch array on the current device (looked up once).
kda_status_t scratch_on_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_kda_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return KDA_ERR_CUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_fwd_noalloc(const void *q, const void *k, const void *v, const void *g,
                                        const void *beta, const float *A_log, const float *dt_bias,
                                        float lower_bound, float scale, const float *initial_state,
                                        float *final_state, const int32_t *cu_seqlens, int B, int T,
                                        int H, int K, int V, int num_seqs, void *o,
                                        kda_stream_t stream) {
  // Size check first, before any CUDA call: reject what the fixed array cannot hold.
  // (context parallelism stays off: its segment states would take scratch from the problem)
  const size_t need = kda_fwd_workspace_size_ex(B, T, H, K, V, num_seqs, cu_seqlens != nullptr, KDA_CP_OFF);
  if (need > (size_t)KDA_NOALLOC_MAX_SCRATCH) return KDA_ERR_WORKSPACE;
  void *scratch = nullptr;
  const kda_status_t st = scratch_on_current_device(&scratch);
  if (st != KDA_OK) return st;
  // The scratch needs no clearing: every call writes all the scratch it later reads.
  return kda_fwd_ex(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state, final_state,
                    cu_seqlens, B, T, H, K, V, num_seqs, KDA_CP_OFF, o, scratch,
                    (size_t)KDA_NOALLOC_MAX_SCRATCH, stream, nullptr);
}
