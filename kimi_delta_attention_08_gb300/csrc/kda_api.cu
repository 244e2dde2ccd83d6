// kda_api.cu -- the C ABI declared in include/kda.h: argument validation,
// workspace sizing and carve-up, planning and kernel launches.  Host only: it
// never synchronises (except kda_get_device_status) and never allocates.
#include <cmath>
#include <cstring>

#include "kda_internal.h"

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Compute capability check, cached per device ordinal.
kda_status check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KDA_ERR_CUDA;
  static int cached[64];  // 0 unknown, 1 ok, 2 unsupported
  if (dev < 64 && cached[dev]) return cached[dev] == 1 ? KDA_OK : KDA_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return KDA_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev < 64) cached[dev] = ok ? 1 : 2;
  return ok ? KDA_OK : KDA_ERR_UNSUPPORTED_DEVICE;
}

// Streaming multiprocessor count of the current device, cached per ordinal.
kda_status sm_count(int* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KDA_ERR_CUDA;
  static int cached[64];
  if (dev < 64 && cached[dev]) {
    *out = cached[dev];
    return KDA_OK;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return KDA_ERR_CUDA;
  if (dev < 64) cached[dev] = n;
  *out = n;
  return KDA_OK;
}

}  // namespace

namespace kda {

kda_status validate_fwd(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, float scale, const void* out, const float* A_log,
                        const float* dt_bias, float lower_bound, const void* initial_state,
                        const void* final_state, const int64_t* cu_seqlens, int64_t B, int64_t T,
                        int32_t H, int32_t* N, int32_t state_dtype, const void* workspace,
                        bool check_workspace, const kda_options* opts, int32_t* HV_out) {
  if (!A_log || !dt_bias || (check_workspace && !workspace)) return KDA_ERR_NULL_POINTER;
  if (B < 1 || T < 0 || H < 1) return KDA_ERR_INVALID_SHAPE;
  // each below 2^31 first, so that B * T cannot overflow
  if (B >= (int64_t(1) << 31) || T >= (int64_t(1) << 31)) return KDA_ERR_INVALID_SHAPE;
  // token tensors may be NULL only when there are no tokens (empty tensors)
  if (B * T > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL_POINTER;
  if (cu_seqlens) {
    if (B != 1 || *N < 1) return KDA_ERR_INVALID_SHAPE;
  } else {
    *N = (int32_t)B;
    if ((int64_t)*N != B) return KDA_ERR_INVALID_SHAPE;
  }
  // grouped value heads: HV heads of v / g / beta / out / states, H of q / k
  if (opts && opts->num_v_heads < 0) return KDA_ERR_INVALID_SHAPE;
  const int32_t HV = (opts && opts->num_v_heads > 0) ? opts->num_v_heads : H;
  if (HV % H != 0) return KDA_ERR_INVALID_SHAPE;
  const int64_t total = B * T;
  if (total >= (int64_t(1) << 31) || (int64_t)*N * HV >= (int64_t(1) << 31))
    return KDA_ERR_INVALID_SHAPE;
  if (state_dtype != KDA_STATE_FP32 && state_dtype != KDA_STATE_BF16) return KDA_ERR_INVALID_ARG;
  if (!(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
  if (opts) {
    if (opts->cp_mode < KDA_CP_AUTO || opts->cp_mode > KDA_CP_FORCE || opts->seg_chunks < 0)
      return KDA_ERR_INVALID_ARG;
    if (opts->path < KDA_PATH_AUTO || opts->path > KDA_PATH_RECURRENT) return KDA_ERR_INVALID_ARG;
    if (opts->g_dtype != KDA_GATE_BF16 && opts->g_dtype != KDA_GATE_FP32) return KDA_ERR_INVALID_ARG;
    if (opts->debug_stall != 0 && opts->debug_stall != 1) return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < 2; ++i)
      if (opts->reserved[i] != 0) return KDA_ERR_INVALID_ARG;
    // chunk start states come from the chunked kernel only
    if (opts->chunk_states && opts->path == KDA_PATH_RECURRENT) return KDA_ERR_INVALID_ARG;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) ||
      (opts && !aligned(opts->chunk_states, 16)) ||
      !aligned(out, 16) || !aligned(beta, 2) || !aligned(A_log, 4) || !aligned(dt_bias, 4) ||
      (initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)) ||
      (cu_seqlens && !aligned(cu_seqlens, 8)) || (check_workspace && !aligned(workspace, 128)))
    return KDA_ERR_MISALIGNED;
  *HV_out = HV;
  return KDA_OK;
}

}  // namespace kda

extern "C" {

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case KDA_ERR_INVALID_SHAPE: return "invalid shape (B, T, H, N) or varlen with B != 1";
    case KDA_ERR_INVALID_ARG: return "invalid argument (lower_bound, scale, dtype or option)";
    case KDA_ERR_MISALIGNED: return "misaligned pointer (tensors 16 B, workspace 128 B)";
    case KDA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than kda_get_workspace_size";
    case KDA_ERR_UNSUPPORTED_DEVICE: return "current device is not an sm_103 GPU";
    case KDA_ERR_CUDA: return "CUDA runtime or driver error";
    case KDA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait expired";
    case KDA_ERR_BAD_SEQLENS: return "cu_seqlens is not a valid prefix sum of the token axis";
  }
  return "unknown status";
}

kda_status kda_get_workspace_size(int64_t total_tokens, int32_t H, size_t* bytes) {
  if (!bytes) return KDA_ERR_NULL_POINTER;
  if (total_tokens < 0 || H < 0 || total_tokens >= (int64_t(1) << 31)) return KDA_ERR_INVALID_SHAPE;
  *bytes = kda::ws_layout(total_tokens, H).total;
  return KDA_OK;
}

kda_status kda_get_chunk_states_size(int64_t total_tokens, int32_t N, int32_t HV, size_t* bytes) {
  if (!bytes) return KDA_ERR_NULL_POINTER;
  if (total_tokens < 0 || N < 0 || HV < 0 || total_tokens >= (int64_t(1) << 31))
    return KDA_ERR_INVALID_SHAPE;
  const size_t slots = (size_t)(total_tokens / kda::kChunk) + 2 * (size_t)N + 1;
  *bytes = slots * (size_t)HV * kda::kHeadDim * kda::kHeadDim * sizeof(uint16_t);
  return KDA_OK;
}

kda_status kda_fwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                   float scale, void* out, const float* A_log, const float* dt_bias,
                   float lower_bound, const void* initial_state, void* final_state,
                   const int64_t* cu_seqlens, int64_t B, int64_t T, int32_t H, int32_t N,
                   int32_t state_dtype, void* workspace, size_t workspace_bytes,
                   const kda_options* opts, cudaStream_t stream) {
  int32_t HV = 0;
  kda_status st = kda::validate_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                                    initial_state, final_state, cu_seqlens, B, T, H, &N,
                                    state_dtype, workspace, true, opts, &HV);
  if (st != KDA_OK) return st;
  const int32_t qk_group = HV / H;
  const int64_t total = B * T;
  size_t need = 0;
  st = kda_get_workspace_size(total, HV, &need);
  if (st != KDA_OK) return st;
  if (workspace_bytes < need) return KDA_ERR_WORKSPACE_TOO_SMALL;
  if (opts && opts->chunk_states) {
    size_t cs = 0;
    st = kda_get_chunk_states_size(total, N, HV, &cs);
    if (st != KDA_OK) return st;
    if (opts->chunk_states_bytes < cs) return KDA_ERR_WORKSPACE_TOO_SMALL;
  }
  st = check_device();
  if (st != KDA_OK) return st;

  if (cu_seqlens && (int64_t)N > total + 1) return KDA_ERR_INVALID_SHAPE;  // workspace bound
  int num_sms = 0;
  if (sm_count(&num_sms) != KDA_OK) return KDA_ERR_CUDA;
  const int cp_mode = opts ? opts->cp_mode : KDA_CP_AUTO;
  const int seg_chunks = opts ? opts->seg_chunks : 0;
  const bool gate_f32 = opts && opts->g_dtype == KDA_GATE_FP32;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const kda::WsLayout L = kda::ws_layout(total, HV);
  kda::WsHeader* hdr = reinterpret_cast<kda::WsHeader*>(ws);
  if (cudaMemsetAsync(hdr, 0, sizeof(kda::WsHeader), stream) != cudaSuccess) return KDA_ERR_CUDA;

  const int path = opts ? opts->path : KDA_PATH_AUTO;
  void* const chunk_states = opts ? opts->chunk_states : nullptr;
  if (path == KDA_PATH_RECURRENT || (path == KDA_PATH_AUTO && cu_seqlens == nullptr &&
                                     T <= kda::kRecurrentMaxT && !chunk_states)) {
    kda::RecParams rp;
    std::memset(&rp, 0, sizeof(rp));
    rp.q = static_cast<const uint16_t*>(q);
    rp.k = static_cast<const uint16_t*>(k);
    rp.v = static_cast<const uint16_t*>(v);
    rp.g = g;
    rp.beta = static_cast<const uint16_t*>(beta);
    rp.A_log = A_log;
    rp.dt_bias = dt_bias;
    rp.out = static_cast<uint16_t*>(out);
    rp.init_state = initial_state;
    rp.final_state = final_state;
    rp.cu_seqlens = cu_seqlens;
    rp.seq_len = T;
    rp.total_tokens = total;
    rp.H = HV;
    rp.N = N;
    rp.qk_group = qk_group;
    rp.gate_f32 = gate_f32 ? 1 : 0;
    rp.debug_stall = opts ? opts->debug_stall : 0;
    rp.state_bf16 = state_dtype == KDA_STATE_BF16 ? 1 : 0;
    rp.scale = scale;
    rp.lower_bound = lower_bound;
    rp.status = &hdr->status;
    // rows of the first token box: all of a short batched sequence, else 16
    rp.tok_rows = (cu_seqlens == nullptr && T >= 1 && T < 16) ? (int32_t)T : 16;
    if (kda::launch_recurrent(rp, num_sms, stream) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
  }

  CUtensorMap maps[4];
  if (kda::make_qkvg_maps(q, k, v, g, total, HV, qk_group, gate_f32, maps) != cudaSuccess)
    return KDA_ERR_CUDA;
  kda::ChunkFwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.g32 = gate_f32 ? static_cast<const float*>(g) : nullptr;
  p.beta = static_cast<const uint16_t*>(beta);
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.out = static_cast<uint16_t*>(out);
  p.init_state = initial_state;
  p.final_state = final_state;
  p.cu_seqlens = cu_seqlens;
  p.seq_len = T;
  p.total_tokens = total;
  p.H = HV;
  p.N = N;
  p.qk_group = qk_group;
  p.gate_f32 = gate_f32 ? 1 : 0;
  p.debug_stall = opts ? opts->debug_stall : 0;
  p.state_bf16 = state_dtype == KDA_STATE_BF16 ? 1 : 0;
  p.scale = scale;
  p.lower_bound = lower_bound;
  p.status = &hdr->status;
  p.ckpt_out = static_cast<uint16_t*>(chunk_states);

  // Batched sequences of one known length need no device schedule unless the
  // segment scan engages (same rule as the device planner).
  bool need_plan = cu_seqlens != nullptr;
  if (!need_plan && cp_mode != KDA_CP_OFF) {
    const long long ch = (T + kda::kChunk - 1) / kda::kChunk;
    if (cp_mode == KDA_CP_FORCE) {
      need_plan = ch >= 2;
    } else {
      const long long avg = ((long long)B * ch * HV + num_sms - 1) / num_sms;
      need_plan = ch >= 2 * kda::kMinSegChunks && ch > 2 * avg;
    }
  }
  if (!need_plan) {
    if (kda::launch_chunk_fwd(maps, p, (int64_t)N * HV, stream) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
  }

  kda::PlanParams pp;
  std::memset(&pp, 0, sizeof(pp));
  pp.cu_seqlens = cu_seqlens;
  pp.seq_len = T;
  pp.total_tokens = total;
  pp.N = N;
  pp.H = HV;
  pp.cp_mode = cp_mode;
  pp.seg_chunks = seg_chunks;
  pp.num_sms = num_sms;
  pp.seg_cap = L.seg_cap;
  pp.hdr = hdr;
  pp.seg_units = reinterpret_cast<kda::Unit*>(ws + L.seg_units);
  pp.pre_units = reinterpret_cast<kda::Unit*>(ws + L.pre_units);
  pp.merge_units = reinterpret_cast<kda::Unit*>(ws + L.merge_units);
  pp.order = reinterpret_cast<int32_t*>(ws + L.order);
  pp.seq_info = reinterpret_cast<int32_t*>(ws + L.seq_info);
  if (kda::launch_plan(pp, stream) != cudaSuccess) return KDA_ERR_CUDA;

  p.hdr = hdr;
  p.order = pp.order;
  p.seq_info = pp.seq_info;
  p.slots = reinterpret_cast<float*>(ws + L.slots);
  p.seg_cap = L.seg_cap;
  if (cp_mode != KDA_CP_OFF && L.seg_cap > 0) {
    // segment scan: the prescan units (segment 0 of each split sequence writes its
    // outputs) together with every unsplit sequence, the serial merge of segment
    // transitions, then the reruns of segments 1 .. nseg - 1
    p.units = pp.pre_units;
    p.prescan = 1;
    p.unsplit_base = 2 * L.seg_cap;
    if (kda::launch_chunk_fwd(maps, p, 2 * (int64_t)L.seg_cap + (int64_t)N * HV, stream) !=
        cudaSuccess)
      return KDA_ERR_CUDA;
    kda::MergeParams mp;
    mp.hdr = hdr;
    mp.merge_units = pp.merge_units;
    mp.slots = p.slots;
    if (kda::launch_merge(mp, L.seg_cap, stream) != cudaSuccess) return KDA_ERR_CUDA;
    p.units = pp.seg_units;
    p.prescan = 0;
    p.unsplit_base = L.seg_cap;
    if (kda::launch_chunk_fwd(maps, p, (int64_t)L.seg_cap, stream) != cudaSuccess)
      return KDA_ERR_CUDA;
    return KDA_OK;
  }
  p.units = pp.seg_units;  // no segment scan: the plan holds no reruns
  p.prescan = 0;
  p.unsplit_base = L.seg_cap;
  if (kda::launch_chunk_fwd(maps, p, (int64_t)L.seg_cap + (int64_t)N * HV, stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  return KDA_OK;
}

kda_status kda_fwd_transition(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const float* A_log, const float* dt_bias,
                              float lower_bound, const int64_t* cu_seqlens, int64_t B, int64_t T,
                              int32_t H, int32_t N, float* M_out, float* B_out, void* workspace,
                              size_t workspace_bytes, const kda_options* opts,
                              cudaStream_t stream) {
  if (!M_out || !B_out) return KDA_ERR_NULL_POINTER;
  if (opts && opts->chunk_states) return KDA_ERR_INVALID_ARG;  // no outputs, no chunk states
  // kda_fwd's checks; M_out stands in for `out` (non-null, 16-byte aligned)
  int32_t HV = 0;
  kda_status st = kda::validate_fwd(q, k, v, g, beta, 1.0f, M_out, A_log, dt_bias, lower_bound,
                                    nullptr, nullptr, cu_seqlens, B, T, H, &N, KDA_STATE_FP32,
                                    workspace, true, opts, &HV);
  if (st != KDA_OK) return st;
  if (!aligned(B_out, 16)) return KDA_ERR_MISALIGNED;
  const int64_t total = B * T;
  if (cu_seqlens && (int64_t)N > total + 1) return KDA_ERR_INVALID_SHAPE;
  if (2 * (int64_t)N * HV >= (int64_t(1) << 31)) return KDA_ERR_INVALID_SHAPE;
  size_t need = 0;
  st = kda_get_workspace_size(total, HV, &need);
  if (st != KDA_OK) return st;
  if (workspace_bytes < need) return KDA_ERR_WORKSPACE_TOO_SMALL;
  st = check_device();
  if (st != KDA_OK) return st;
  const bool gate_f32 = opts && opts->g_dtype == KDA_GATE_FP32;
  kda::WsHeader* hdr = reinterpret_cast<kda::WsHeader*>(workspace);
  if (cudaMemsetAsync(hdr, 0, sizeof(kda::WsHeader), stream) != cudaSuccess) return KDA_ERR_CUDA;
  CUtensorMap maps[4];
  if (kda::make_qkvg_maps(q, k, v, g, total, HV, HV / H, gate_f32, maps) != cudaSuccess)
    return KDA_ERR_CUDA;
  kda::ChunkFwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.g32 = gate_f32 ? static_cast<const float*>(g) : nullptr;
  p.beta = static_cast<const uint16_t*>(beta);
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.cu_seqlens = cu_seqlens;
  p.seq_len = T;
  p.total_tokens = total;
  p.H = HV;
  p.N = N;
  p.qk_group = HV / H;
  p.gate_f32 = gate_f32 ? 1 : 0;
  p.debug_stall = opts ? opts->debug_stall : 0;
  p.scale = 1.0f;
  p.lower_bound = lower_bound;
  p.status = &hdr->status;
  p.trans_M = M_out;
  p.trans_B = B_out;
  if (kda::launch_chunk_fwd(maps, p, 2 * (int64_t)N * HV, stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  return KDA_OK;
}

kda_status kda_compose_states(const float* M, const float* B, int32_t R, int64_t num_states,
                              const float* S_in, float* S_out, cudaStream_t stream) {
  if (!S_out || (R > 0 && (!M || !B))) return KDA_ERR_NULL_POINTER;
  if (R < 0 || num_states < 0 || num_states >= (int64_t(1) << 27)) return KDA_ERR_INVALID_SHAPE;
  if (!aligned(S_out, 16) || (M && !aligned(M, 16)) || (B && !aligned(B, 16)) ||
      (S_in && !aligned(S_in, 16)))
    return KDA_ERR_MISALIGNED;
  const kda_status st = check_device();
  if (st != KDA_OK) return st;
  kda::ComposeParams cp;
  cp.M = M;
  cp.B = B;
  cp.S_in = S_in;
  cp.S_out = S_out;
  cp.R = R;
  cp.num_states = num_states;
  if (kda::launch_compose(cp, stream) != cudaSuccess) return KDA_ERR_CUDA;
  return KDA_OK;
}

kda_status kda_get_device_status(const void* workspace, kda_status* status, cudaStream_t stream) {
  if (!workspace || !status) return KDA_ERR_NULL_POINTER;
  if (!aligned(workspace, 128)) return KDA_ERR_MISALIGNED;
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (word & kda::kDevStatusBadSeqlens)
    *status = KDA_ERR_BAD_SEQLENS;
  else if (word & kda::kDevStatusTimeout)
    *status = KDA_ERR_DEVICE_TIMEOUT;
  else
    *status = KDA_OK;
  return KDA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ backward --
namespace kda {
int64_t bwd_scratch_ctas(int64_t units);
}

namespace {

struct BwdWs {
  size_t unit_part, ckpt, scratch, dq_part, dk_part, total;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

BwdWs bwd_layout(int64_t total_tokens, int32_t N, int32_t HV, int32_t G) {
  BwdWs w;
  size_t off = 256;  // header: the device status word
  w.unit_part = off;
  off += align256((size_t)N * HV * (kda::kHeadDim + 1) * sizeof(float));
  w.ckpt = off;
  off += (size_t)(total_tokens / kda::kBwdBlock + N + 1) * HV * kda::kHeadDim * kda::kHeadDim *
         sizeof(float);
  w.scratch = off;
  off += (size_t)kda::bwd_scratch_ctas((int64_t)N * HV) * (kda::kBwdBlock / kda::kBwdKeep) *
         kda::kHeadDim * kda::kHeadDim * sizeof(float);
  w.dq_part = w.dk_part = 0;
  if (G > 1) {
    const size_t part = align256((size_t)total_tokens * HV * kda::kHeadDim * sizeof(float));
    w.dq_part = off;
    off += part;
    w.dk_part = off;
    off += part;
  }
  w.total = off;
  return w;
}

}  // namespace

extern "C" {

kda_status kda_bwd_get_workspace_size(int64_t total_tokens, int32_t N, int32_t H,
                                      int32_t num_v_heads, size_t* bytes) {
  if (!bytes) return KDA_ERR_NULL_POINTER;
  const int32_t HV = num_v_heads > 0 ? num_v_heads : H;
  if (total_tokens < 0 || N < 0 || H < 1 || num_v_heads < 0 || HV % H != 0 ||
      total_tokens >= (int64_t(1) << 31))
    return KDA_ERR_INVALID_SHAPE;
  *bytes = bwd_layout(total_tokens, N, HV, HV / H).total;
  return KDA_OK;
}

kda_status kda_bwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                   float scale, const float* A_log, const float* dt_bias, float lower_bound,
                   const void* initial_state, const void* dout, const void* dfinal_state,
                   const int64_t* cu_seqlens, float* dq, float* dk, float* dv, float* dg,
                   float* dbeta, float* dA_log, float* ddt_bias, float* dinitial_state, int64_t B,
                   int64_t T, int32_t H, int32_t N, int32_t state_dtype, void* workspace,
                   size_t workspace_bytes, const kda_options* opts, cudaStream_t stream) {
  if (!A_log || !dt_bias || !dA_log || !ddt_bias || !workspace) return KDA_ERR_NULL_POINTER;
  if (B < 1 || T < 0 || H < 1) return KDA_ERR_INVALID_SHAPE;
  if (B >= (int64_t(1) << 31) || T >= (int64_t(1) << 31)) return KDA_ERR_INVALID_SHAPE;
  if (B * T > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta))
    return KDA_ERR_NULL_POINTER;
  if (cu_seqlens) {
    if (B != 1 || N < 1) return KDA_ERR_INVALID_SHAPE;
  } else {
    N = (int32_t)B;
    if ((int64_t)N != B) return KDA_ERR_INVALID_SHAPE;
  }
  if (opts && opts->num_v_heads < 0) return KDA_ERR_INVALID_SHAPE;
  const int32_t HV = (opts && opts->num_v_heads > 0) ? opts->num_v_heads : H;
  if (HV % H != 0) return KDA_ERR_INVALID_SHAPE;
  const int64_t total = B * T;
  if (total >= (int64_t(1) << 31) || (int64_t)N * HV >= (int64_t(1) << 31))
    return KDA_ERR_INVALID_SHAPE;
  if (state_dtype != KDA_STATE_FP32 && state_dtype != KDA_STATE_BF16) return KDA_ERR_INVALID_ARG;
  if (!(lower_bound >= -5.0f && lower_bound <= 0.0f) || !std::isfinite(scale))
    return KDA_ERR_INVALID_ARG;
  const int path = opts ? opts->path : KDA_PATH_AUTO;
  const bool chunked = path != KDA_PATH_RECURRENT;
  if (opts) {
    if (opts->g_dtype != KDA_GATE_BF16 && opts->g_dtype != KDA_GATE_FP32) return KDA_ERR_INVALID_ARG;
    if (opts->path < KDA_PATH_AUTO || opts->path > KDA_PATH_RECURRENT) return KDA_ERR_INVALID_ARG;
    // the stall hook exists on the chunked path only (its waits are bounded)
    if (opts->debug_stall != 0 && (opts->debug_stall != 1 || !chunked)) return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < 2; ++i)
      if (opts->reserved[i] != 0) return KDA_ERR_INVALID_ARG;
    if (opts->chunk_states && !chunked) return KDA_ERR_INVALID_ARG;
  }
  const void* const chunk_states = opts ? opts->chunk_states : nullptr;
  if (!aligned(q, 8) || !aligned(k, 8) || !aligned(v, 8) || !aligned(g, 16) || !aligned(dout, 8) ||
      !aligned(beta, 2) || !aligned(A_log, 4) || !aligned(dt_bias, 4) || !aligned(dq, 16) ||
      !aligned(dk, 16) || !aligned(dv, 4) || !aligned(dg, 16) || !aligned(dbeta, 4) ||
      !aligned(dA_log, 4) || !aligned(ddt_bias, 4) ||
      (initial_state && !aligned(initial_state, 16)) || (dfinal_state && !aligned(dfinal_state, 16)) ||
      (dinitial_state && !aligned(dinitial_state, 16)) || (cu_seqlens && !aligned(cu_seqlens, 8)) ||
      !aligned(workspace, 128) ||
      (chunked && (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))) ||  // tensor maps
      !aligned(chunk_states, 16))
    return KDA_ERR_MISALIGNED;
  const BwdWs L = bwd_layout(total, N, HV, HV / H);
  if (workspace_bytes < L.total) return KDA_ERR_WORKSPACE_TOO_SMALL;
  if (chunk_states) {
    size_t cs = 0;
    const kda_status cst = kda_get_chunk_states_size(total, N, HV, &cs);
    if (cst != KDA_OK) return cst;
    if (opts->chunk_states_bytes < cs) return KDA_ERR_WORKSPACE_TOO_SMALL;
  }
  kda_status st = check_device();
  if (st != KDA_OK) return st;
  int num_sms = 0;
  if (sm_count(&num_sms) != KDA_OK) return KDA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  kda::WsHeader* hdr = reinterpret_cast<kda::WsHeader*>(ws);
  if (cudaMemsetAsync(hdr, 0, sizeof(kda::WsHeader), stream) != cudaSuccess) return KDA_ERR_CUDA;

  kda::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.g = g;
  p.beta = static_cast<const uint16_t*>(beta);
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.init_state = initial_state;
  p.dout = static_cast<const uint16_t*>(dout);
  p.dfinal = dfinal_state;
  p.cu_seqlens = cu_seqlens;
  p.seq_len = T;
  p.total_tokens = total;
  p.H = HV;
  p.N = N;
  p.qk_group = HV / H;
  p.gate_f32 = (opts && opts->g_dtype == KDA_GATE_FP32) ? 1 : 0;
  p.state_bf16 = state_dtype == KDA_STATE_BF16 ? 1 : 0;
  p.scale = scale;
  p.lower_bound = lower_bound;
  p.dq = dq;
  p.dk = dk;
  p.dq_part = L.dq_part ? reinterpret_cast<float*>(ws + L.dq_part) : nullptr;
  p.dk_part = L.dk_part ? reinterpret_cast<float*>(ws + L.dk_part) : nullptr;
  p.dv = dv;
  p.dg = dg;
  p.dbeta = dbeta;
  p.dinit = dinitial_state;
  p.unit_part = reinterpret_cast<float*>(ws + L.unit_part);
  p.ckpt = reinterpret_cast<float*>(ws + L.ckpt);
  p.scratch = reinterpret_cast<float*>(ws + L.scratch);
  p.status = &hdr->status;
  if (!chunked) {
    if (kda::launch_bwd(p, num_sms, dA_log, ddt_bias, stream) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
  }
  // chunked path: the fused forward kernel in its state-checkpoint mode (no outputs)
  // writes every chunk's start state, then the reverse sweep on the tensor cores.
  // States that a kda_fwd of the same inputs wrote to opts->chunk_states are read
  // from there instead.
  p.debug_stall = opts ? opts->debug_stall : 0;
  if (chunk_states) p.ckpt = static_cast<float*>(const_cast<void*>(chunk_states));
  if (total > 0 && !chunk_states) {
    const bool gate_f32 = opts && opts->g_dtype == KDA_GATE_FP32;
    CUtensorMap maps[4];
    if (kda::make_qkvg_maps(q, k, v, g, total, HV, HV / H, gate_f32, maps) != cudaSuccess)
      return KDA_ERR_CUDA;
    kda::ChunkFwdParams fp;
    std::memset(&fp, 0, sizeof(fp));
    fp.g32 = gate_f32 ? static_cast<const float*>(g) : nullptr;
    fp.beta = static_cast<const uint16_t*>(beta);
    fp.A_log = A_log;
    fp.dt_bias = dt_bias;
    fp.init_state = initial_state;
    fp.cu_seqlens = cu_seqlens;
    fp.seq_len = T;
    fp.total_tokens = total;
    fp.H = HV;
    fp.N = N;
    fp.qk_group = HV / H;
    fp.gate_f32 = gate_f32 ? 1 : 0;
    fp.state_bf16 = p.state_bf16;
    fp.scale = scale;
    fp.lower_bound = lower_bound;
    fp.status = &hdr->status;
    fp.ckpt_out = reinterpret_cast<uint16_t*>(ws + L.ckpt);
    fp.no_out = 1;
    if (kda::launch_chunk_fwd(maps, fp, (int64_t)N * HV, stream) != cudaSuccess)
      return KDA_ERR_CUDA;
  }
  if (kda::launch_bwd_chunk(p, num_sms, dA_log, ddt_bias, stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  return KDA_OK;
}

}  // extern "C"
