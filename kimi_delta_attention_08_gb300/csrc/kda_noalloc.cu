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

// Device address of the array on each device, looked up once per device (with
// that device current).  In host code the array's name is only a stand-in for
// the symbol, never a usable address.
std::mutex g_scratch_mutex;
void* g_scratch_ptr[64];

kda_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_kda_static_scratch) != cudaSuccess || !ptr)
      return KDA_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
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
  if (B < 1 || T < 0 || H < 1) return KDA_ERR_INVALID_SHAPE;
  // the workspace is sized by the value heads (kda_fwd validates num_v_heads)
  const int32_t HV = (opts && opts->num_v_heads > 0) ? opts->num_v_heads : H;
  size_t need = 0;
  const kda_status st = kda_get_workspace_size(B * T, HV, &need);
  if (st != KDA_OK) return st;
  if (need > kStaticScratchBytes) return KDA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const kda_status sa = scratch_address(&scratch);
  if (sa != KDA_OK) return sa;
  // kda_fwd clears the header (status word, schedule counts) on every call;
  // everything else it reads in the array is written earlier in the same call.
  return kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                 final_state, cu_seqlens, B, T, H, N, state_dtype, scratch, kStaticScratchBytes,
                 opts, stream);
}
