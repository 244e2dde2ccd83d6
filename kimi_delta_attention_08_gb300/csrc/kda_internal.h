// kda_internal.h -- declarations shared by the translation units of the KDA
// library (not part of the public C ABI in include/kda.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;     // tokens per chunk of the chunked WY form
constexpr int kHeadDim = 128;  // K = V
constexpr int kMinSegChunks = 16;      // automatic segment length floor (1024 tokens)
constexpr int kMaxSegHeads = 256;      // workspace cap on (segment, head) pairs
constexpr int kMergeRowBlocks = 8;     // merge CTAs per (sequence, head): 16 rows each

// Device status word values (first 4 bytes of the workspace).
constexpr unsigned kDevStatusTimeout = 1u;
constexpr unsigned kDevStatusBadSeqlens = 2u;

// Kinds of work unit the chunk kernel runs.
enum UnitKind : int32_t {
  kUnitSerial = 0,  // a whole sequence: user initial state -> user final state, outputs
  kUnitRerun = 1,   // segment of a split sequence, from its merged start state, outputs
  kUnitPreS1 = 2,   // segment 0 of a split sequence: user initial state -> slot S_1
  kUnitPreM = 3,    // segment s: identity start, v = 0 -> slot M_s (transition)
  kUnitPreB = 4,    // segment s: zero start -> slot S_{s+1} (offset B_s)
};

struct Unit {        // 32 bytes
  int32_t n, h, seg, nseg;
  int32_t L;         // segment length in chunks
  int32_t kind;      // UnitKind
  int32_t slot_base; // first state slot of this (sequence, head)
  int32_t pad;
};

// Per (sequence, head) the state slots are: S_1 .. S_{nseg-1} at
// slot_base + (s - 1), then M_1 .. M_{nseg-2} at slot_base + (nseg - 1) + (s - 1).
__host__ __device__ inline int32_t slot_S(const Unit& u, int32_t s) { return u.slot_base + s - 1; }
__host__ __device__ inline int32_t slot_M(const Unit& u, int32_t s) {
  return u.slot_base + (u.nseg - 1) + (s - 1);
}

struct WsHeader {     // at workspace offset 0
  unsigned status;
  int32_t n_seg_units;  // rerun units of split sequences
  int32_t n_pre_units;  // prescan units
  int32_t n_merge;      // (sequence, head) chains to merge
  int32_t plan_ok;
};

struct WsLayout {
  size_t seg_units, pre_units, merge_units, order, seq_info, slots, total;
  int32_t seg_cap, max_slots;
  int64_t nmax;
};
WsLayout ws_layout(int64_t total_tokens, int32_t H);

// Heads: H below is the number of value heads -- one state, one output head and
// one gate / beta / A_log / dt_bias row each.  q and k have H / qk_group heads;
// value head h reads q/k head h / qk_group (qk_group = 1: one q/k head each).
struct ChunkFwdParams {
  const float* g32;          // fp32 gate [T_total][H][128] (fp32-gate kernel), else null
  const uint16_t* beta;      // bf16 bits [T_total][H]
  const float* A_log;        // [H]
  const float* dt_bias;      // [H][128]
  uint16_t* out;             // bf16 bits [T_total][H][128]
  const void* init_state;    // [N][H][V][K] or null
  void* final_state;         // [N][H][V][K] or null
  const int64_t* cu_seqlens; // [N+1] device, or null (batched)
  int64_t seq_len;           // batched mode: tokens per sequence
  int64_t total_tokens;      // B*T (packed token count)
  int32_t H;
  int32_t N;
  int32_t qk_group;          // value heads per q/k head (>= 1)
  int32_t gate_f32;          // 1: fp32 gate through g32 (selects the kernel instance)
  int32_t state_bf16;        // 1: bf16 state, 0: fp32 state
  float scale;
  float lower_bound;
  unsigned* status;          // device status word
  // schedule (null tables: one serial unit per blockIdx = n * H + h)
  const WsHeader* hdr;
  const Unit* units;         // rerun units (main pass) or prescan units (prescan pass)
  const int32_t* order;      // [N] sequence order, longest first
  const int32_t* seq_info;   // [N][4]: segments (1 = not split), L, slot base, chunks
  float* slots;              // fp32 state slots [.][128][128]
  int32_t seg_cap;           // rerun units per launch of the plan (workspace bound)
  int32_t unsplit_base;      // blockIdx < unsplit_base: table units (prescan or rerun);
                             // from it on, whole unsplit sequences in `order`
  int32_t prescan;           // 1: this launch runs the prescan units
  int32_t debug_stall;       // 1: the prep group never releases a chunk (timeout test)
  // transition mode (non-null trans_M): 2 N H blocks; block 2u / 2u + 1 writes the
  // transition M / offset B of (sequence, value head) u = n H + h over the whole
  // sequence, fp32 [N][H][V][K] like the states
  float* trans_M;
  float* trans_B;
  // state checkpoints (serial units only; null: none): the bf16 start state of
  // every chunk c of (sequence n, value head h), [V][K], at slot
  // bos / 64 + 2 n + c of a [slot][H][128][128] array (the chunked backward's input)
  uint16_t* ckpt_out;
  int32_t no_out;            // 1: no outputs (serial units run only for the states)
};

// Token-by-token path (kda_recurrent.cu), one CTA per (sequence, head).
struct RecParams {
  const uint16_t* q;         // bf16 bits [T_total][H / qk_group][128]
  const uint16_t* k;
  const uint16_t* v;         // bf16 bits [T_total][H][128]
  const void* g;             // [T_total][H][128], bf16 bits or fp32 (gate_f32)
  const uint16_t* beta;      // bf16 bits [T_total][H]
  const float* A_log;        // [H]
  const float* dt_bias;      // [H][128]
  uint16_t* out;             // bf16 bits [T_total][H][128]
  const void* init_state;    // [N][H][V][K] or null
  void* final_state;         // [N][H][V][K] or null
  const int64_t* cu_seqlens; // [N+1] device, or null (batched)
  int64_t seq_len;           // batched mode: tokens per sequence
  int64_t total_tokens;
  int32_t H;                 // value heads (units are (sequence, value head))
  int32_t N;
  int32_t qk_group;          // value heads per q/k head (>= 1)
  int32_t gate_f32;          // 1: g is fp32
  int32_t state_bf16;
  float scale;
  float lower_bound;
  unsigned* status;          // device status word
  int32_t tok_rows;          // token rows per TMA box (<= 16)
  int32_t debug_stall;       // 1: fetch only each CTA's first two units (timeout test)
};

// Batched sequences of at most this many tokens take the token-by-token path
// under KDA_PATH_AUTO (where it is measured faster than the chunked path).
constexpr int64_t kRecurrentMaxT = 16;

// Backward pass (kda_bwd.cu): token-by-token reverse mode, one unit (sequence,
// value head) at a time per persistent CTA.  Gradients are fp32.
constexpr int kBwdBlock = 16;  // tokens per checkpoint / recomputation block
constexpr int kBwdKeep = 4;    // tokens per decayed state kept in the scratch
static_assert(kBwdBlock % kBwdKeep == 0, "kept states align with the block");

struct BwdParams {
  const uint16_t* q;         // bf16 bits [T_total][H / qk_group][128]
  const uint16_t* k;
  const uint16_t* v;         // bf16 bits [T_total][H][128]
  const void* g;             // [T_total][H][128], bf16 bits or fp32 (gate_f32)
  const uint16_t* beta;      // bf16 bits [T_total][H]
  const float* A_log;        // [H]
  const float* dt_bias;      // [H][128]
  const void* init_state;    // [N][H][V][K] or null
  const uint16_t* dout;      // bf16 bits [T_total][H][128]
  const void* dfinal;        // [N][H][V][K] (state dtype) or null
  const int64_t* cu_seqlens; // [N+1] device, or null (batched)
  int64_t seq_len;           // batched mode: tokens per sequence
  int64_t total_tokens;
  int32_t H;                 // value heads
  int32_t N;
  int32_t qk_group;          // value heads per q/k head
  int32_t gate_f32;
  int32_t state_bf16;
  float scale;
  float lower_bound;
  float* dq;                 // [T_total][H / qk_group][128] (written directly when qk_group == 1)
  float* dk;
  float* dq_part;            // [T_total][H][128] per value head when qk_group > 1, else null
  float* dk_part;
  float* dv;                 // [T_total][H][128]
  float* dg;                 // [T_total][H][128]
  float* dbeta;              // [T_total][H]
  float* dinit;              // [N][H][V][K]
  float* unit_part;          // [N][H][129]: dt_bias gradient (128) and A_log gradient per unit
  float* ckpt;               // checkpoint slots [slots][H][128][128]
  float* scratch;            // [gridDim.x][kBwdBlock / kBwdKeep][128][128]
  unsigned* status;
  int32_t debug_stall;       // chunked path, timeout test: 1 = a chunk's first MMAs are never issued
};

// Checkpoint slot of block m of sequence n (collision-free over sequences:
// floor(bos / 64) + n + m); slots needed: floor(T_total / 64) + N + 1.
__host__ __device__ inline int64_t bwd_slot(int64_t bos, int32_t n, int64_t m) {
  return bos / kBwdBlock + n + m;
}

struct PlanParams {
  const int64_t* cu_seqlens;
  int64_t seq_len, total_tokens;
  int32_t N, H, cp_mode, seg_chunks, num_sms, seg_cap;
  WsHeader* hdr;
  Unit* seg_units;
  Unit* pre_units;
  Unit* merge_units;
  int32_t* order;
  int32_t* seq_info;  // [N][4]: nseg, L, slot_base, chunks
};

struct ComposeParams {
  const float* M;        // [R][num_states][128][128] stored transitions
  const float* B;        // [R][num_states][128][128] stored offsets
  const float* S_in;     // [num_states][128][128] or null (zero)
  float* S_out;          // [num_states][128][128]
  int32_t R;
  int64_t num_states;
};
cudaError_t launch_compose(const ComposeParams& cp, cudaStream_t stream);

struct MergeParams {
  const WsHeader* hdr;
  const Unit* merge_units;
  float* slots;
};

// Encode the tile maps of q, k ([T_total, H / qk_group, 128]) and v, g
// ([T_total, H, 128]): bf16 boxes of 64 tokens x 64 channels with 128-byte
// swizzle.  An fp32 gate gets a map of 64 tokens x 128 channels without swizzle,
// used only to prefetch it into L2.  Returns cudaSuccess or an error.
// cuTensorMapEncodeTiled through the runtime's driver entry point (strides in
// bytes for dimensions 1 .. rank-1, element strides 1, no interleave).
cudaError_t encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* ptr,
                             const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                             CUtensorMapSwizzle swizzle);
cudaError_t make_qkvg_maps(const void* q, const void* k, const void* v, const void* g,
                           int64_t T_total, int32_t H, int32_t qk_group, bool gate_f32,
                           CUtensorMap maps[4]);

// Raise a kernel's dynamic shared memory limit to `bytes` on the current device.
// The attribute is per device, so it is set once per device ordinal (`done` is
// the caller's table for that kernel); setting it twice is harmless.
inline cudaError_t ensure_smem_attr(const void* func, int bytes, bool (&done)[64]) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// Host-side argument checks of kda_fwd, in its order (everything but the workspace
// size and the device): returns the status kda_fwd would return for them, and on
// success the value-head count in *HV_out and, for batched input, N = B in *N.
// check_workspace = false skips the workspace pointer's NULL and alignment checks.
kda_status validate_fwd(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, float scale, const void* out, const float* A_log,
                        const float* dt_bias, float lower_bound, const void* initial_state,
                        const void* final_state, const int64_t* cu_seqlens, int64_t B, int64_t T,
                        int32_t H, int32_t* N, int32_t state_dtype, const void* workspace,
                        bool check_workspace, const kda_options* opts, int32_t* HV_out);

// Enqueue the chunk kernel over `grid` units.
cudaError_t launch_chunk_fwd(const CUtensorMap maps[4], const ChunkFwdParams& p, int64_t grid,
                             cudaStream_t stream);
cudaError_t launch_recurrent(const RecParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_plan(const PlanParams& pp, cudaStream_t stream);
// Backward: the per-unit kernel (grid = min(N * H, num_sms)), then the fixed-order
// sums over value heads (dq, dk when qk_group > 1) and over sequences (dA_log, dt_bias).
cudaError_t launch_bwd(const BwdParams& p, int num_sms, float* dA_log, float* ddt_bias,
                       cudaStream_t stream);
// Backward in the chunked form on the tensor cores (the same outputs and sums);
// its chunk-state checkpoints (bf16, 32 KiB per 64-token chunk) reuse p.ckpt.
cudaError_t launch_bwd_chunk(const BwdParams& p, int num_sms, float* dA_log, float* ddt_bias,
                             cudaStream_t stream);
// The fixed-order sums that follow either backward kernel.
cudaError_t launch_bwd_reduce(const BwdParams& p, float* dA_log, float* ddt_bias,
                              cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& mp, int32_t seg_cap, cudaStream_t stream);

}  // namespace kda
