// kda_internal.h -- declarations shared by the host-side translation units of
// the KDA library (not part of the public C ABI in include/kda.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;     // tokens per chunk of the chunked WY form
constexpr int kHeadDim = 128;  // K = V

// Device status word values (first 4 bytes of the workspace).
constexpr unsigned kDevStatusTimeout = 1u;
constexpr unsigned kDevStatusBadSeqlens = 2u;

// Byte offsets inside the caller's workspace.
constexpr size_t kWsStatusBytes = 256;  // status word + padding

struct ChunkFwdParams {
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
  int32_t state_bf16;        // 1: bf16 state, 0: fp32 state
  float scale;
  float lower_bound;
  unsigned* status;          // device status word
};

// Encode the four [T_total, H, 128] bf16 tile maps (box 64 tokens x 64 channels,
// 128-byte swizzle) for q, k, v, g.  Returns cudaSuccess or an error.
cudaError_t make_qkvg_maps(const void* q, const void* k, const void* v, const void* g,
                           int64_t T_total, int32_t H, CUtensorMap maps[4]);

// Enqueue the serial chunked forward over all N*H (sequence, head) units.
cudaError_t launch_chunk_fwd(const CUtensorMap maps[4], const ChunkFwdParams& p,
                             cudaStream_t stream);

}  // namespace kda
