// kda_noalloc.cu -- kda_fwd for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a host framework that reserves all
// device memory up front and hands a plugin only its input and output buffers,
// or an embedded runtime with a fixed memory budget that forbids allocations
// after start-up.  kda_fwd_static_scratch runs the same forward as kda_fwd,
// with the workspace (status word, schedule tables, segment-scan state slots)
// in a file-scope device array instead of a caller buffer.
#include <mutex>

#include "kda_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)KDA_STATIC_SCRATCH_BYTES;

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_kda_static_scratch[kStaticScratchBytes];

// Device address of the array on each device, looked up with that device
// current.  In host code the array's name is only a stand-in for the symbol,
// never a usable address.  The address belongs to the context it was looked up
// in, so the cache is keyed by the context: after a device reset (or any
// teardown and re-creation of the primary context) it is looked up again.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    tried = true;
  }
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64];
CUcontext g_scratch_ctx[64];

kda_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  // cudaGetDevice does not create the context; the symbol lookup below does, so
  // the context is read after it on a first call
  CUcontext ctx = current_context();
  if (!g_scratch_ptr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_kda_static_scratch) != cudaSuccess || !ptr)
      return KDA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = current_context();
  }
  *out = g_scratch_ptr[dev];
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_fwd_static_scratch(
    const void* q, const void* k, const void* v, const void* g, const void* beta, float scale,
    void* out, const float* A_log, const float* dt_bias, float lower_bound,
    const void* initial_state, void* final_state, const int64_t* cu_seqlens, int64_t B, int64_t T,
    int32_t H, int32_t N, int32_t state_dtype, const kda_options* opts, cudaStream_t stream) {
  // kda_fwd's argument checks first, so a bad call gets the status kda_fwd gives it
  int32_t HV = 0, n = N;
  kda_status st = kda::validate_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                                    initial_state, final_state, cu_seqlens, B, T, H, &n,
                                    state_dtype, nullptr, false, opts, &HV);
  if (st != KDA_OK) return st;
  size_t need = 0;
  st = kda_get_workspace_size(B * T, HV, &need);
  if (st != KDA_OK) return st;
  if (need > kStaticScratchBytes) return KDA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != KDA_OK) return st;
  // kda_fwd clears the header (status word, schedule counts) on every call;
  // everything else it reads in the array is written earlier in the same call.
  return kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                 final_state, cu_seqlens, B, T, H, N, state_dtype, scratch, kStaticScratchBytes,
                 opts, stream);
}

extern "C" kda_status kda_static_scratch_device_status(kda_status* status, cudaStream_t stream) {
  if (!status) return KDA_ERR_NULL_POINTER;
  void* scratch = nullptr;
  const kda_status st = scratch_address(&scratch);
  if (st != KDA_OK) return st;
  return kda_get_device_status(scratch, status, stream);
}
