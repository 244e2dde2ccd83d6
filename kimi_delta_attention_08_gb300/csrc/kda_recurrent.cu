// kda_recurrent.cu -- token-by-token forward for short sequences (decode and
// prompts of a few tokens).
//
// The chunked kernel pays a full warp-specialised pipeline per (sequence, head)
// even for one token; here the cost is what such a step fundamentally moves:
// the 128 x 128 state in and out, plus one row of q, k, v, g per token.  Per
// token, in the order of the recurrence S_t = (I - b k k^T) Diag(a) S_{t-1} +
// b k v^T, o_t = scale S_t^T q:
//   S <- Diag(alpha) S;   u = beta (v - S^T k);   S <- S + k u^T;   o = scale S^T q
// with the same gate, l2-norm and sigmoid preprocessing as the chunked path.
//
// Persistent CTAs (one per SM, 512 threads) walk the (sequence, head) units
// with two units' fetches in flight: TMA brings a unit's initial state (as
// 128-byte swizzled boxes, so the per-thread reads below are bank-conflict free)
// and its first token rows of q, k, v, g into one half of a double buffer, and
// a unit refills its half with the unit two ahead as soon as it has read it.
// The final state goes from registers straight to global memory (per value
// column a warp writes 128 contiguous k values), so no store holds a buffer.
// Warp w holds the value columns v = 8w .. 8w+7 of S in registers, lane l the
// four key channels k = 4l .. 4l+3 of each, so every token's k, q and alpha are
// read from shared memory once per warp (no redundant loads) and the two dot
// products over k reduce across the warp with a reduce-scatter butterfly.
// Tokens come in blocks of 16: one warp per token computes the gate, the l2
// norms and beta into shared memory, then the block's recurrence steps run from
// there with no barrier.
#include <cuda_bf16.h>

#include <cstring>

#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kRecThreads = 512;
constexpr int kCols = 8;        // value columns per warp
constexpr int kTokBlock = 16;   // tokens prepared together: one warp per token
constexpr float kLog2eR = 1.4426950408889634f;
constexpr uint64_t kRecWaitNs = 500ull * 1000ull * 1000ull;

// dynamic shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kStBytes = 65536;                 // one fp32 state (4 boxes of 128 x 32)
constexpr uint32_t kOffSt = 0;                       // [2] state buffers
constexpr uint32_t kTokBytes = 3 * kTokBlock * 256 + kTokBlock * 512;  // q, k, v, g rows
                                                                          // (g up to fp32)
constexpr uint32_t kOffTok = 2 * kStBytes;           // [2] token buffers
constexpr uint32_t kOffVec = kOffTok + 2 * kTokBytes;
constexpr uint32_t kVecBytes = 4 * kTokBlock * 128 * 4;  // k, q, alpha, v
constexpr uint32_t kOffBeta = kOffVec + kVecBytes;
constexpr uint32_t kOffBar = kOffBeta + kTokBlock * 4;
constexpr uint32_t kRecSmem = kOffBar + 64 + 1024;   // + alignment slack
static_assert(kRecSmem <= 232448, "shared memory budget");

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ bool unit_bounds(const RecParams& p, int n, int64_t& bos, int64_t& eos) {
  if (p.cu_seqlens) {
    bos = p.cu_seqlens[n];
    eos = p.cu_seqlens[n + 1];
  } else {
    bos = (int64_t)n * p.seq_len;
    eos = bos + p.seq_len;
  }
  return !(bos < 0 || eos < bos || eos > p.total_tokens || (p.cu_seqlens && n == 0 && bos != 0) ||
           (p.cu_seqlens && n == p.N - 1 && eos != p.total_tokens));
}

}  // namespace

__global__ void __launch_bounds__(kRecThreads, 1)
    kda_recurrent_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tg,
                         const __grid_constant__ CUtensorMap ts,
                         const RecParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* const sm = smem_align1024(smem_raw);
  float (*s_k)[128] = reinterpret_cast<float (*)[128]>(sm + kOffVec);
  float (*s_q)[128] = s_k + kTokBlock;
  float (*s_a)[128] = s_q + kTokBlock;
  float (*s_v)[128] = s_a + kTokBlock;
  float* const s_beta = reinterpret_cast<float*>(sm + kOffBeta);
  uint64_t* const bar = reinterpret_cast<uint64_t*>(sm + kOffBar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H;
  const int units = p.N * H;
  const bool has_init = p.init_state != nullptr;
  const uint32_t st_bytes = has_init ? (p.state_bf16 ? kStBytes / 2 : kStBytes) : 0u;
  const uint32_t g_row = p.gate_f32 ? 512u : 256u;  // bytes of one gate row
  const uint32_t tok_bytes = (3u * 256u + g_row) * (uint32_t)p.tok_rows;
  const int G = p.qk_group;  // value heads per q/k head

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // thread 0: fetch unit u's state and first token rows into buffer b
  auto issue = [&](int u, int b) {
    const int n = u / H, h = u % H;
    int64_t bos, eos;
    const bool ok = unit_bounds(p, n, bos, eos);
    const bool toks = ok && eos > bos;
    mbar_arrive_expect_tx(&bar[b], (ok ? st_bytes : 0u) + (toks ? tok_bytes : 0u));
    if (ok && has_init) {
      uint8_t* dst = sm + kOffSt + b * kStBytes;
      if (p.state_bf16) {
        for (int x = 0; x < 2; ++x) tma_load_2d(dst + x * 16384, &ts, &bar[b], 64 * x, u * 128);
      } else {
        for (int x = 0; x < 4; ++x) tma_load_2d(dst + x * 16384, &ts, &bar[b], 32 * x, u * 128);
      }
    }
    if (toks) {
      uint8_t* dst = sm + kOffTok + b * kTokBytes;
      const uint32_t tb = 256u * (uint32_t)p.tok_rows;  // one tensor's rows
      tma_load_3d(dst + 0 * tb, &tq, &bar[b], 0, h / G, (int32_t)bos);
      tma_load_3d(dst + 1 * tb, &tk, &bar[b], 0, h / G, (int32_t)bos);
      tma_load_3d(dst + 2 * tb, &tv, &bar[b], 0, h, (int32_t)bos);
      tma_load_3d(dst + 3 * tb, &tg, &bar[b], 0, h, (int32_t)bos);
    }
  };

  const int v0 = kCols * warp;   // this warp's first value column
  const int c0 = 4 * lane;        // this lane's four key channels (also its prep channels)
  const float lb2 = p.lower_bound * kLog2eR;
  const int64_t rstride = (int64_t)H * kHeadDim;           // v, g token stride (elements)
  const int64_t qkstride = (int64_t)(H / G) * kHeadDim;    // q, k token stride

  // Two units in flight: units i and i + 1 are fetched ahead; unit i refills its
  // buffer with unit i + 2 as soon as its state and first token rows are read.
  const int grid = (int)gridDim.x;
  int u = (int)blockIdx.x;
  if (tid == 0 && u < units) issue(u, 0);
  if (tid == 0 && u + grid < units) issue(u + grid, 1);
  bool aborted = false;
#pragma unroll 1
  for (int i = 0; u < units; ++i, u += grid) {
    const int b = i & 1;
    // call after a barrier that follows every read of buffer b by this unit
    auto refill = [&]() {
      if (tid == 0 && u + 2 * grid < units && !p.debug_stall) issue(u + 2 * grid, b);
    };
    bool landed = true;
    if (tid == 0) landed = mbar_wait(&bar[b], (uint32_t)((i >> 1) & 1), kRecWaitNs);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) atomicOr(p.status, kDevStatusTimeout);
      aborted = true;
      break;
    }
    const int n = u / H, h = u % H;
    int64_t bos, eos;
    if (!unit_bounds(p, n, bos, eos)) {
      if (tid == 0) atomicOr(p.status, kDevStatusBadSeqlens);
      __syncthreads();
      refill();
      continue;
    }

    // ---- state S[k][v] for this lane's k and the warp's v, from the swizzled
    // boxes (128 rows v of 128 bytes; 16-byte chunk j of row v at j ^ (v % 8))
    float4 S[kCols];
    if (!has_init) {
#pragma unroll
      for (int c = 0; c < kCols; ++c) S[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (p.state_bf16) {  // box x: channels 64x .. 64x+63
      const uint8_t* box = sm + kOffSt + b * kStBytes + (lane >> 4) * 16384;
      const int j = (lane & 15) >> 1, hb = (lane & 1) * 8;
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        const uint2 w = *reinterpret_cast<const uint2*>(box + (v0 + c) * 128 + ((j ^ c) << 4) + hb);
        S[c] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      }
    } else {  // box x: channels 32x .. 32x+31
      const uint8_t* box = sm + kOffSt + b * kStBytes + (lane >> 3) * 16384;
      const int j = lane & 7;
#pragma unroll
      for (int c = 0; c < kCols; ++c)
        S[c] = *reinterpret_cast<const float4*>(box + (v0 + c) * 128 + ((j ^ c) << 4));
    }

    const float nea = -expf(p.A_log[h]) * kLog2eR;
    const float* db = p.dt_bias + h * kHeadDim + c0;  // only 4-byte alignment is guaranteed
    const float ndb[4] = {nea * db[0], nea * db[1], nea * db[2], nea * db[3]};
    const uint8_t* tok = sm + kOffTok + b * kTokBytes;

#pragma unroll 1
    for (int64_t blk = bos; blk < eos; blk += (blk == bos ? p.tok_rows : kTokBlock)) {
      const int rows = blk == bos ? p.tok_rows : kTokBlock;  // the first block is one TMA box
      const int nt = (int)((eos - blk) < rows ? (eos - blk) : rows);
      // ---- prep of the block's tokens, one warp per token: gate, l2 norms, beta
      if (warp < nt) {
        uint2 kw, qw, vw;
        float gx[4];
        if (blk == bos) {  // the first block came with the unit's TMA fetch
          const int tb = 256 * p.tok_rows;
          const uint8_t* r = tok + warp * 256 + c0 * 2;
          qw = *reinterpret_cast<const uint2*>(r);
          kw = *reinterpret_cast<const uint2*>(r + tb);
          vw = *reinterpret_cast<const uint2*>(r + 2 * tb);
          const uint8_t* gr = tok + 3 * tb + warp * (int)g_row;
          if (p.gate_f32) {
            const float4 g4 = *reinterpret_cast<const float4*>(gr + c0 * 4);
            gx[0] = g4.x; gx[1] = g4.y; gx[2] = g4.z; gx[3] = g4.w;
          } else {
            const uint2 gw = *reinterpret_cast<const uint2*>(gr + c0 * 2);
            gx[0] = __uint_as_float(gw.x << 16); gx[1] = __uint_as_float(gw.x & 0xFFFF0000u);
            gx[2] = __uint_as_float(gw.y << 16); gx[3] = __uint_as_float(gw.y & 0xFFFF0000u);
          }
        } else {
          const int64_t row = (blk + warp) * rstride + (int64_t)h * kHeadDim + c0;
          const int64_t rowk = (blk + warp) * qkstride + (int64_t)(h / G) * kHeadDim + c0;
          kw = *reinterpret_cast<const uint2*>(p.k + rowk);
          qw = *reinterpret_cast<const uint2*>(p.q + rowk);
          vw = *reinterpret_cast<const uint2*>(p.v + row);
          if (p.gate_f32) {
            const float4 g4 = *reinterpret_cast<const float4*>(static_cast<const float*>(p.g) + row);
            gx[0] = g4.x; gx[1] = g4.y; gx[2] = g4.z; gx[3] = g4.w;
          } else {
            const uint2 gw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.g) + row);
            gx[0] = __uint_as_float(gw.x << 16); gx[1] = __uint_as_float(gw.x & 0xFFFF0000u);
            gx[2] = __uint_as_float(gw.y << 16); gx[3] = __uint_as_float(gw.y & 0xFFFF0000u);
          }
        }
        const float kx[4] = {__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xFFFF0000u),
                             __uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xFFFF0000u)};
        const float qx[4] = {__uint_as_float(qw.x << 16), __uint_as_float(qw.x & 0xFFFF0000u),
                             __uint_as_float(qw.y << 16), __uint_as_float(qw.y & 0xFFFF0000u)};
        float kk = 0.f, qq = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          kk = fmaf(kx[e], kx[e], kk);
          qq = fmaf(qx[e], qx[e], qq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          kk += __shfl_xor_sync(0xffffffffu, kk, o);
          qq += __shfl_xor_sync(0xffffffffu, qq, o);
        }
        const float rk = rsqrtf(kk + 1e-6f), rq = rsqrtf(qq + 1e-6f);
        float a4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          a4[e] = ex2_approx(lb2 * rcp_approx(1.0f + ex2_approx(fmaf(nea, gx[e], ndb[e]))));
        *reinterpret_cast<float4*>(&s_k[warp][c0]) =
            make_float4(kx[0] * rk, kx[1] * rk, kx[2] * rk, kx[3] * rk);
        *reinterpret_cast<float4*>(&s_q[warp][c0]) =
            make_float4(qx[0] * rq, qx[1] * rq, qx[2] * rq, qx[3] * rq);
        *reinterpret_cast<float4*>(&s_a[warp][c0]) = make_float4(a4[0], a4[1], a4[2], a4[3]);
        *reinterpret_cast<float4*>(&s_v[warp][c0]) =
            make_float4(__uint_as_float(vw.x << 16), __uint_as_float(vw.x & 0xFFFF0000u),
                        __uint_as_float(vw.y << 16), __uint_as_float(vw.y & 0xFFFF0000u));
        if (lane == 0) {
          const float bx = bf16_to_f(p.beta[(blk + warp) * H + h]);
          s_beta[warp] = rcp_approx(1.0f + ex2_approx(-bx * kLog2eR));
        }
      }
      __syncthreads();
      if (blk == bos) refill();  // state and first token rows are in registers / vectors

      // ---- the recurrence over the block, token by token, from shared memory
#pragma unroll 1
      for (int j = 0; j < nt; ++j) {
        const float4 a4 = *reinterpret_cast<const float4*>(&s_a[j][c0]);
        const float4 k4 = *reinterpret_cast<const float4*>(&s_k[j][c0]);
        const float4 q4 = *reinterpret_cast<const float4*>(&s_q[j][c0]);
        // S <- Diag(alpha) S ; d = S^T k for the warp's columns
        float x[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const float2 lo = f2mul(make_float2(a4.x, a4.y), make_float2(S[c].x, S[c].y));
          const float2 hi = f2mul(make_float2(a4.z, a4.w), make_float2(S[c].z, S[c].w));
          S[c] = make_float4(lo.x, lo.y, hi.x, hi.y);
          const float2 dp = f2fma(hi, make_float2(k4.z, k4.w), f2mul(lo, make_float2(k4.x, k4.y)));
          x[c] = dp.x + dp.y;
        }
        const float d = reduce_scatter8(x, lane);  // column v0 + (lane >> 2)
        const float uu = s_beta[j] * (s_v[j][v0 + (lane >> 2)] - d);
        // S <- S + k u^T ; o = S^T q
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const float uc = __shfl_sync(0xffffffffu, uu, 4 * c);
          const float2 u2 = make_float2(uc, uc);
          const float2 lo = f2fma(make_float2(k4.x, k4.y), u2, make_float2(S[c].x, S[c].y));
          const float2 hi = f2fma(make_float2(k4.z, k4.w), u2, make_float2(S[c].z, S[c].w));
          S[c] = make_float4(lo.x, lo.y, hi.x, hi.y);
          const float2 op = f2fma(hi, make_float2(q4.z, q4.w), f2mul(lo, make_float2(q4.x, q4.y)));
          x[c] = op.x + op.y;
        }
        const float o = reduce_scatter8(x, lane);
        if ((lane & 3) == 0) {
          const __nv_bfloat16 ob = __float2bfloat16_rn(p.scale * o);
          p.out[(blk + j) * rstride + (int64_t)h * kHeadDim + v0 + (lane >> 2)] =
              *reinterpret_cast<const uint16_t*>(&ob);
        }
      }
      __syncthreads();  // the next block's prep overwrites the token vectors
    }

    if (eos == bos) {  // no token block: the state buffer is read, free it here
      __syncthreads();
      refill();
    }

    if (p.final_state) {
      // straight from registers: per column v, a warp writes 128 contiguous k values
      if (p.state_bf16) {
        uint16_t* dst = static_cast<uint16_t*>(p.final_state) + ((int64_t)u * 128 + v0) * 128 + c0;
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          __nv_bfloat162 h0 = __floats2bfloat162_rn(S[c].x, S[c].y);
          __nv_bfloat162 h1 = __floats2bfloat162_rn(S[c].z, S[c].w);
          *reinterpret_cast<uint2*>(dst + c * 128) =
              make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
        }
      } else {
        float* dst = static_cast<float*>(p.final_state) + ((int64_t)u * 128 + v0) * 128 + c0;
#pragma unroll
        for (int c = 0; c < kCols; ++c) *reinterpret_cast<float4*>(dst + c * 128) = S[c];
      }
    }
  }
  if (aborted && tid == 0) {  // let copies in flight land before the CTA exits (bounded)
    (void)mbar_wait(&bar[0], 0, kRecWaitNs / 16);
    (void)mbar_wait(&bar[0], 1, kRecWaitNs / 16);
    (void)mbar_wait(&bar[1], 0, kRecWaitNs / 16);
    (void)mbar_wait(&bar[1], 1, kRecWaitNs / 16);
  }
}

cudaError_t launch_recurrent(const RecParams& p, int num_sms, cudaStream_t stream) {
  static bool attr_done[64];
  const cudaError_t ea = ensure_smem_attr(reinterpret_cast<const void*>(kda_recurrent_kernel),
                                          (int)kRecSmem, attr_done);
  if (ea != cudaSuccess) return ea;
  const int64_t units = (int64_t)p.N * p.H;
  if (units <= 0) return cudaSuccess;
  CUtensorMap maps[5];
  if (p.qk_group < 1 || p.H % p.qk_group != 0) return cudaErrorInvalidValue;
  const void* ptrs[4] = {p.q, p.k, p.v, p.g};
  const int32_t heads[4] = {p.H / p.qk_group, p.H / p.qk_group, p.H, p.H};
  const uint32_t tbox[3] = {(uint32_t)kHeadDim, 1, (uint32_t)p.tok_rows};
  for (int i = 0; i < 4; ++i) {  // token rows, no swizzle (one 256- or 512-byte row per token)
    const bool f32 = (i == 3 && p.gate_f32);
    const uint64_t esz = f32 ? 4 : 2;
    const uint64_t tdims[3] = {(uint64_t)kHeadDim, (uint64_t)heads[i],
                               (uint64_t)(p.total_tokens > 0 ? p.total_tokens : 1)};
    const uint64_t tstr[2] = {(uint64_t)kHeadDim * esz, (uint64_t)heads[i] * kHeadDim * esz};
    cudaError_t e = encode_tiled_map(
        &maps[i], f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
        ptrs[i], tdims, tstr, tbox, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  }
  std::memset(&maps[4], 0, sizeof(CUtensorMap));
  const uint64_t sdims[2] = {(uint64_t)kHeadDim, (uint64_t)units * kHeadDim};
  const uint64_t sstr[1] = {(uint64_t)kHeadDim * (p.state_bf16 ? 2 : 4)};
  const uint32_t sbox[2] = {p.state_bf16 ? 64u : 32u, (uint32_t)kHeadDim};
  const CUtensorMapDataType sdt =
      p.state_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (p.init_state) {  // the initial state: 128-byte-swizzled boxes of 128 rows
    cudaError_t e = encode_tiled_map(&maps[4], sdt, 2, p.init_state, sdims, sstr, sbox,
                                     CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  const int64_t grid = units < num_sms ? units : num_sms;
  kda_recurrent_kernel<<<(unsigned)grid, kRecThreads, kRecSmem, stream>>>(maps[0], maps[1], maps[2],
                                                                          maps[3], maps[4], p);
  return cudaGetLastError();
}

}  // namespace kda
