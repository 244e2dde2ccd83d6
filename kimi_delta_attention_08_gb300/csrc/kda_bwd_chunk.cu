// kda_bwd_chunk.cu -- backward pass of Kimi Delta Attention in the chunked WY
// form, on the tcgen05 tensor cores of sm_103a.
//
// The pages' kernels are forward only ("feat(kda): SM90 FlashKDA prefill,
// intracard CP, and backend dispatch", commit notes); this reverse mode is
// derived from the chunked forward that those notes describe (K1: decayed q/k,
// beta and the WY inverse; K2: the inter-chunk recurrence).  Per 64-token chunk,
// with hats for the l2-normalised rows, gam_t the in-chunk cumulative log2 decay
// per channel, F_t = 2^gam_t, E_t = 2^(gam_63 - gam_t):
//   Kt = K^ o F,  Kw = K^ o E,  Qt = Q^ o F          (all factors <= 1)
//   P = strict_lower pairs k^_t k^_s 2^(gam_t - gam_s),  Mq = lower_incl q^_t ...
//   A = Diag(beta) P,  T = (I + A)^-1
//   R = V - Kt S,  U = T Diag(beta) R                 (U = U~ - W S of the forward)
//   O = scale (Qt S + Mq U),  S' = Diag(F_63) S + Kw^T U
// Reverse, given dO and dS' (the gradient of S'):
//   dU  = Kw dS' + scale Mq^T dO          dR~ = T^T dU     dV = Diag(beta) dR~
//   dA  = -strict_lower(dR~ U^T)          dMq = scale lower_incl(dO U^T)
//   dS  = Diag(F_63) dS' + scale Qt^T dO - Kt^T Diag(beta) dR~
//   dbeta_t = rowsum(dR~ o R)_t + rowsum(dA o P)_t
//   dq^ = scale (dO S^T) o F + pairs(dMq, k^)
//   dk^ = -(Diag(beta) dR~ S^T) o F + (U dS'^T) o E + pairs(dP, k^) + pairs^T(dMq q^ + dP k^)
// and the gate through the in-chunk cumulative sums.  Two rearrangements keep the
// gate gradient accurate in bf16 (each removes a cancellation between large
// terms): the chunk-end term enters as 2^gam_63 <S, dS'> with the (U dS'^T) o E
// part of each token added to the LATER tokens' sums (an exclusive forward
// cumulative sum); and the diagonal pairs q^_t k^_t of Mq, which carry no decay,
// go straight into dq^ and dk^ instead of through the pair products.
//
// Pair products with the per-channel factor 2^(gam_t - gam_s) are split at two
// reference points rho1 = gam_15 (columns s < 32) and rho2 = gam_47 (s >= 32), so
// every factor stays inside [2^-116, 2^116] for lower_bound >= -5, as in the
// forward kernel.
//
// One CTA (kCT = 512 threads: four column groups of four warps) per (sequence,
// value head) unit, persistent over units.
// The chunk start states come from the fused forward kernel (kda_chunk_fwd.cu),
// run first in its state-checkpoint mode (bf16, one per chunk); this kernel walks
// the chunks backward with the state gradient dS in TMEM.  Every contraction is an M = 128 tcgen05.mma with
// bf16 operands built in shared memory (128-byte swizzle) by the CUDA cores and
// an fp32 accumulator in TMEM; one thread issues, every thread waits on an
// mbarrier (bounded wait).  Per-channel results live in TMEM lanes (lane =
// channel, column = token) until the chunk's final pass.  Every output has one
// writer; sums run in a fixed order, so results are bitwise reproducible.
#include <cuda_bf16.h>

#include <cstring>

#include "kda_internal.h"
#include "kda_ptx.cuh"
#include "kda_inverse.cuh"

namespace kda {
namespace {

using namespace ptx;

// Warps 4w .. 4w+3 form column group w: in every per-channel phase lane quarter
// w & 3 holds TMEM lanes (channels) 32 (w & 3) .. + 31 and group w the token
// columns [kCols w, kCols (w + 1)).  Four groups (16 warps) hide the latency of
// the CUDA-core phases better than two; each thread then holds half the columns.
#ifndef KDA_BWD_WG
#define KDA_BWD_WG 4
#endif
constexpr int kWG = KDA_BWD_WG;
static_assert(kWG == 2 || kWG == 4, "two or four column groups");
constexpr int kCT = 128 * kWG;  // threads per CTA
constexpr int kWarps = kCT / 32;
constexpr int kCols = 64 / kWG;  // token columns per group
constexpr uint64_t kWaitNsB = 500ull * 1000ull * 1000ull; // bounded waits: 0.5 s
constexpr float kL2e = 1.4426950408889634f;

// ---- shared memory: ten 16 KB operand slots, then fp32 arrays --------------
constexpr uint32_t kSlot = 16384;
constexpr uint32_t kNumSlots = 10;
constexpr uint32_t kOffGam = kNumSlots * kSlot;          // gam [64][128] fp32 (log2 units)
constexpr uint32_t kLdP = 65;                             // fp32 row stride of P
constexpr uint32_t kOffP = kOffGam + 64 * 128 * 4;        // P [64][65] fp32 (strict lower)
constexpr uint32_t kOffMisc = kOffP + 16896;
constexpr uint32_t kOffBar = kOffMisc;                    // one mbarrier
constexpr uint32_t kOffTaddr = kOffMisc + 8;
constexpr uint32_t kOffAbort = kOffMisc + 12;
constexpr uint32_t kOffBeta = kOffMisc + 256;             // [64] fp32
constexpr uint32_t kOffRq = kOffBeta + 256;               // [64]
constexpr uint32_t kOffRk = kOffRq + 256;                 // [64]
constexpr uint32_t kOffDd = kOffRk + 256;                 // [64] diagonal of dMq
constexpr uint32_t kOffDb1 = kOffDd + 256;                // [64] rowsum(dR~ o R)
constexpr uint32_t kOffDb2 = kOffDb1 + 256;               // [kWG][64] rowsum(dA o P), per group
constexpr uint32_t kOffEend = kOffDb2 + 256 * kWG;        // [128] chunk-end gate term
constexpr uint32_t kOffRed = kOffEend + 512;              // [4][128] per-lane-quarter partials
constexpr uint32_t kOffRed2 = kOffRed + 2048;             // [4][128]
constexpr uint32_t kOffCarry = kOffRed2 + 2048;           // [2][kWG][128] cumulative-sum carries
constexpr uint32_t kOffAcc = kOffCarry + 1024 * kWG;      // [kWG][128] dt_bias sums; [kCT] A_log
constexpr uint32_t kOffDots = kOffAcc + 512 * kWG + 4 * kCT;  // [2][64] per-token norm dots (q, k)
constexpr uint32_t kOffOnes = kOffDots + 512;             // [64] ones (the inverse's beta)
constexpr uint32_t kOffWmax = kOffOnes + 256;             // [kWarps] per-warp max |X|, then 2^shift
constexpr int kShiftIdx = kWarps;                         // index of 2^shift in the kOffWmax array
constexpr uint32_t kSmemUsed = kOffWmax + 4 * (kWarps + 1);
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;         // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffP % 16 == 0 && kOffMisc % 256 == 0, "alignment");

// slot roles; a slot is reused once its previous content is dead
constexpr int bKr = 0, bQr = 2, bBr = 4, bDOT = 5, bTM = 6 /* Tb | MqS */, bS = 7, bKt = 9,
              bBRT = 3, bUT = 4, bDSp = 0, bKw = 2, bDUT = 3, bDRt = 2, bNdR = 9, bX = 3,
              bQtS = 0, bKt2 = 1, bBr2 = 2, bKr2 = 4, bQr2 = 6;
// The inverse works in slots 0..1 (A, then its blocks of L^{-1}) once the Gram is read.
constexpr uint32_t kOffA = 0;
static_assert(64 * inv::kLdM * 4 <= 2 * kSlot, "inverse workspace");

// ---- TMEM columns ------------------------------------------------------------
constexpr uint32_t kTCols = 512;
constexpr uint32_t tDS = 0;     // state gradient dS, [v lane][k]
// per-channel accumulators [channel lane][t] (each 64 columns), then scratch
constexpr uint32_t tAQ = 128;   // dq^ (inter-chunk and pair parts)
constexpr uint32_t tAKt = 192;  // dk^ through Kt (inter-chunk and pair parts)
constexpr uint32_t tAKp = 256;  // dk^ through Kb, pair part (first: R = V - Kt S)
constexpr uint32_t tAKi = 320;  // dk^ through Kb, inter-chunk part (U dS'^T) o E
constexpr uint32_t tSC = 384;   // MMA scratch, 128 columns

__device__ __forceinline__ float bflo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bfhi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf1(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint32_t packbf(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// sigmoid(x) = 1 / (1 + 2^(-x log2 e)) with the hardware ex2 / rcp (the forward's form)
__device__ __forceinline__ float sigm(float x) { return rcp_approx(1.0f + ex2_approx(-x * kL2e)); }
// sigmoid(x) sigmoid(-x) = e / (1 + e)^2 with e = 2^(-|x| log2 e) <= 1: no cancellation
__device__ __forceinline__ float sig_prod(float x) {
  const float e = ex2_approx(-fabsf(x) * kL2e);
  const float r = rcp_approx(1.0f + e);
  return e * r * r;
}
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// Eight consecutive bf16 values into row `row` of a 128-byte-swizzled tile whose
// 64-element column blocks are `blk` bytes apart, starting at element e0 (a
// multiple of 8).
__device__ __forceinline__ void st8(uint8_t* tile, uint32_t blk, int row, int e0, const float (&x)[8]) {
  uint4 w;
  w.x = packbf(x[0], x[1]);
  w.y = packbf(x[2], x[3]);
  w.z = packbf(x[4], x[5]);
  w.w = packbf(x[6], x[7]);
  *reinterpret_cast<uint4*>(tile + (uint32_t)(e0 >> 6) * blk + sw128(row, (e0 & 63) * 2)) = w;
}
// 32 consecutive values (e0 a multiple of 32) of one row.
[[maybe_unused]] __device__ __forceinline__ void st32(uint8_t* tile, uint32_t blk, int row, int e0, const float (&x)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = x[8 * c + i];
    st8(tile, blk, row, e0 + 8 * c, y);
  }
}

// 16 consecutive values (e0 a multiple of 16) of one row.
__device__ __forceinline__ void st16(uint8_t* tile, uint32_t blk, int row, int e0, const float (&x)[16]) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = x[8 * c + i];
    st8(tile, blk, row, e0 + 8 * c, y);
  }
}

// kN (16 or 32) consecutive values (e0 a multiple of kN) of one row.
template <int kN>
__device__ __forceinline__ void stn(uint8_t* tile, uint32_t blk, int row, int e0, const float (&x)[kN]) {
  static_assert(kN == 16 || kN == 32, "16 or 32 columns");
  if constexpr (kN == 32) st32(tile, blk, row, e0, x); else st16(tile, blk, row, e0, x);
}

// Reduce-scatter over the 32 lanes of a warp: on entry lane l holds x[0..kN-1] (one
// value per column, kN = 8 or 16); on return every lane l holds the sum over the
// warp's lanes of column l & (kN - 1).  kN - 1 + log2(32 / kN) shuffles.
template <int kN>
__device__ __forceinline__ float warp_rs(float (&x)[kN], int lane) {
  static_assert(kN == 8 || kN == 16, "8 or 16 columns");
#pragma unroll
  for (int w = kN / 2; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? x[i] : x[i + w];
      const float keep = up ? x[i + w] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  float r = x[0];
#pragma unroll
  for (int o = kN; o < 32; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}
__device__ __forceinline__ float warp_rs16(float (&x)[16], int lane) { return warp_rs<16>(x, lane); }

struct Ctx {
  uint8_t* sm;
  float* gam;   // [64][128]
  float* P;     // [64][kLdP]
  float* beta;  // [64]
  float* rq;
  float* rk;
  uint64_t* bar;
  volatile int* abort;
  uint32_t tbase, lane_off;  // TMEM base; this warp's lane quarter (<< 16)
  int tid, warp, lane, wg, row;  // wg: column half; row: TMEM lane = 32 (warp & 3) + lane
  uint32_t phase;
};

__device__ __forceinline__ uint8_t* slot(const Ctx& c, int i) { return c.sm + (uint32_t)i * kSlot; }

// Stage 64 rows of 128 bf16 (256 bytes each, `stride` elements apart; rows past n
// are zero) into shared memory, row-major without swizzle: the loads are 16-byte
// vectors (kStageIt per thread); lane j of a warp then reads column j of a row without
// bank conflicts.  The caller synchronises before anyone reads the rows.
constexpr int kStageIt = 1024 / kCT;  // 16-byte pieces per thread of 64 rows of 256 bytes
__device__ __forceinline__ void stage_load(const Ctx& c, const uint16_t* src, int64_t stride, int n,
                                           uint4 (&w)[kStageIt]) {
#pragma unroll
  for (int it = 0; it < kStageIt; ++it) {
    const int idx = c.tid + it * kCT, t = idx >> 4, e0 = (idx & 15) * 8;
    w[it] = t < n ? *reinterpret_cast<const uint4*>(src + (int64_t)t * stride + e0)
                  : make_uint4(0u, 0u, 0u, 0u);
  }
}
__device__ __forceinline__ void stage_store(const Ctx& c, uint8_t* dst, const uint4 (&w)[kStageIt]) {
#pragma unroll
  for (int it = 0; it < kStageIt; ++it) {
    const int idx = c.tid + it * kCT;
    *reinterpret_cast<uint4*>(dst + (uint32_t)idx * 16u) = w[it];
  }
}
// Asynchronous 16-byte global -> shared copies (no registers); src_bytes 0 fills
// zeros.  A thread waits for its own copies with cp_async_wait_all; a barrier
// after that makes every thread's copies visible.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// The 64 rows of 128 bf16 at `src` (rows `stride` elements apart, rows past n zero)
// into `dst` as unswizzled [64][128] rows, asynchronously.
__device__ __forceinline__ void stage_async(const Ctx& c, uint8_t* dst, const uint16_t* src,
                                            int64_t stride, int n) {
#pragma unroll
  for (int it = 0; it < kStageIt; ++it) {
    const int idx = c.tid + it * kCT, t = idx >> 4, e0 = (idx & 15) * 8;
    const bool ok = t < n;
    cp_async16(dst + (uint32_t)idx * 16u, src + (ok ? (int64_t)t * stride + e0 : 0), ok ? 16u : 0u);
  }
}

__device__ __forceinline__ float staged(const uint8_t* rows, int t, int j) {
  return bf1(reinterpret_cast<const uint16_t*>(rows)[t * kHeadDim + j]);
}

// Every thread waits for the MMAs committed to the CTA's barrier (bounded).
__device__ __noinline__ bool mma_wait_slow(uint64_t* bar, uint32_t phase, volatile int* abort,
                                           unsigned* status) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, phase, 20000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitNsB) {
      *abort = 1;
      atomicOr(status, kDevStatusTimeout);
      return false;
    }
  }
}
// An expired wait sets the CTA's abort flag (and the status word); every thread
// then leaves at the next publish(), which all threads reach.
__device__ __forceinline__ void mma_wait(Ctx& c, unsigned* status) {
  if (!mbar_try_wait(c.bar, c.phase)) (void)mma_wait_slow(c.bar, c.phase, c.abort, status);
  c.phase ^= 1u;
  tc_fence_after();
}
// Operands written by the CUDA cores (shared memory, TMEM) become visible to the
// tensor cores; returns true if any thread has aborted.
__device__ __forceinline__ bool publish(const Ctx& c) {
  fence_proxy_async();
  tmem_wait_st();
  tc_fence_before();
  return __syncthreads_or(*c.abort != 0) != 0;
}

// ---- MMA issue (one thread) ------------------------------------------------
// Descriptors: K-major tiles step 32 bytes per 16 K-elements inside a 64-element
// column block and `blk` bytes between blocks; MN-major tiles step 2048 bytes
// (16 rows) per K-step.
__device__ __forceinline__ uint64_t dK(const uint8_t* p) { return sw128_desc(smem_u32(p), 16, 1024); }
__device__ __forceinline__ uint64_t dMN(const uint8_t* p, uint32_t lbo) {
  return sw128_desc(smem_u32(p), lbo, 1024);
}
__device__ __forceinline__ uint32_t kstep(int k, uint32_t blk) {  // K-major, in 16-byte units
  return (uint32_t)(k & 3) * 2u + (uint32_t)(k >> 2) * (blk >> 4);
}

// ---- per-chunk inputs ------------------------------------------------------
struct Chunk {
  int64_t tok0;  // first token (packed index)
  int n;         // valid tokens (1..64); rows n..63 are padding
  int last;      // chunk index within the unit
};

// beta, l2-norm reciprocals and the cumulative log2 decay of one chunk.  Padding
// rows get beta = 0, zero rows and no decay, so they contribute nothing.
// The chunk's q and k rows are at qx / kx (xs elements apart: global memory, or
// rows staged in shared memory by the previous chunk); its bf16 g rows at gx (gs
// apart), or null for the global fp32 / bf16 gate.
__device__ void prep_chunk(Ctx& c, const BwdParams& p, const Chunk& ch, int h, float ea,
                           const uint16_t* qx, const uint16_t* kx, int64_t xs, const uint16_t* gx,
                           int64_t gs) {
  // norms: warp w takes rows kNr w .. kNr w + kNr - 1, lane l channels 4l .. 4l+3
  constexpr int kNr = 64 / kWarps;
  uint2 qa[kNr], ka[kNr];
#pragma unroll
  for (int i = 0; i < kNr; ++i) {
    const int t = kNr * c.warp + i;
    const int64_t o = (int64_t)t * xs + 4 * c.lane;
    qa[i] = t < ch.n ? *reinterpret_cast<const uint2*>(qx + o) : make_uint2(0u, 0u);
    ka[i] = t < ch.n ? *reinterpret_cast<const uint2*>(kx + o) : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < kNr; ++i) {
    const int t = kNr * c.warp + i;
    float sq = bflo(qa[i].x) * bflo(qa[i].x) + bfhi(qa[i].x) * bfhi(qa[i].x) +
               bflo(qa[i].y) * bflo(qa[i].y) + bfhi(qa[i].y) * bfhi(qa[i].y);
    float sk = bflo(ka[i].x) * bflo(ka[i].x) + bfhi(ka[i].x) * bfhi(ka[i].x) +
               bflo(ka[i].y) * bflo(ka[i].y) + bfhi(ka[i].y) * bfhi(ka[i].y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (c.lane == 0) {
      c.rq[t] = t < ch.n ? rsqrtf(sq + 1e-6f) : 0.f;
      c.rk[t] = t < ch.n ? rsqrtf(sk + 1e-6f) : 0.f;
    }
  }
  if (c.tid < 64)
    c.beta[c.tid] = c.tid < ch.n ? sigm(bf1(p.beta[(ch.tok0 + c.tid) * p.H + h])) : 0.f;
  // gate, row by row (16-byte loads): log2 alpha into gam [t][j]; padding rows 0
  const float lb2 = p.lower_bound * kL2e;
  const float* dtb = p.dt_bias + h * kHeadDim;
  if (p.gate_f32) {
    const float* g = static_cast<const float*>(p.g) + (ch.tok0 * p.H + h) * kHeadDim;
#pragma unroll
    for (int it = 0; it < 2048 / kCT; ++it) {
      const int idx = c.tid + it * kCT, t = idx >> 5, e0 = (idx & 31) * 4;
      const float4 w = t < ch.n ? *reinterpret_cast<const float4*>(g + (int64_t)t * p.H * kHeadDim + e0)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 d = *reinterpret_cast<const float4*>(dtb + e0);
      float4 o;
      o.x = t < ch.n ? lb2 * sigm(ea * (w.x + d.x)) : 0.f;
      o.y = t < ch.n ? lb2 * sigm(ea * (w.y + d.y)) : 0.f;
      o.z = t < ch.n ? lb2 * sigm(ea * (w.z + d.z)) : 0.f;
      o.w = t < ch.n ? lb2 * sigm(ea * (w.w + d.w)) : 0.f;
      *reinterpret_cast<float4*>(c.gam + t * 128 + e0) = o;
    }
  } else {
    const uint16_t* g = gx ? gx : static_cast<const uint16_t*>(p.g) + (ch.tok0 * p.H + h) * kHeadDim;
    uint4 w[kStageIt];
    stage_load(c, g, gx ? gs : (int64_t)p.H * kHeadDim, ch.n, w);
#pragma unroll
    for (int it = 0; it < kStageIt; ++it) {
      const int idx = c.tid + it * kCT, t = idx >> 4, e0 = (idx & 15) * 8;
      const float gx[8] = {bflo(w[it].x), bfhi(w[it].x), bflo(w[it].y), bfhi(w[it].y),
                           bflo(w[it].z), bfhi(w[it].z), bflo(w[it].w), bfhi(w[it].w)};
      float o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = t < ch.n ? lb2 * sigm(ea * (gx[i] + dtb[e0 + i])) : 0.f;
      *reinterpret_cast<float4*>(c.gam + t * 128 + e0) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(c.gam + t * 128 + e0 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
  }
  __syncthreads();
  // cumulative sums: thread (channel j, group w) over the group's kCols tokens;
  // later groups add the earlier groups' totals
  const int j = c.tid & 127, grp = c.tid >> 7;
  float run = 0.f;
#pragma unroll
  for (int i = 0; i < kCols; ++i) {
    const int t = kCols * grp + i;
    run += c.gam[t * 128 + j];
    c.gam[t * 128 + j] = run;
  }
  __syncthreads();
  float carry = 0.f;
  if (grp > 0) {
    carry = c.gam[(kCols - 1) * 128 + j];
    for (int q = 1; q < grp; ++q) carry += c.gam[(kCols * (q + 1) - 1) * 128 + j];
  }
  if constexpr (kWG > 2) __syncthreads();  // every group total is read before any is raised
  if (grp > 0) {
#pragma unroll 4
    for (int i = kCols * grp; i < kCols * (grp + 1); ++i) c.gam[i * 128 + j] += carry;
  }
  __syncthreads();
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned start) into L2.
__device__ __forceinline__ void pf_l2(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// Pull a chunk's start-state checkpoint `ck` (32 KiB) into L2 while the current
// chunk computes.  (The chunk's rows arrive through 16-byte row loads, whose
// latency is short enough: a bulk prefetch per row cost more than it saved.)
__device__ __forceinline__ void prefetch_ckpt(const Ctx& c, const uint16_t* ck) {
  if (c.tid == 0) pf_l2(ck, kHeadDim * kHeadDim * 2);
}

// Tile kinds: rows r of a K-major bf16 tile [rows][128] with 64-column blocks
// rows*128 bytes apart; token t = r (or r - 64 for the second half of 128 rows).
enum TileKind { kTKt, kTKw, kTRho, kTBrho };

// value(r, j) = x[t][j] * rx[t] * s * factor, x = q or k of the chunk (bf16 rows).
// Every thread issues all its global loads first, then converts and stores.
template <int kKind, int kRows>
__device__ void build_tile(Ctx& c, uint8_t* tile, const uint16_t* x, int64_t xstride,
                           const float* rx, const Chunk& ch, float s) {
  constexpr int kIt = kRows * 16 / kCT;
  constexpr uint32_t blk = (uint32_t)kRows * 128u;
  const float* g = c.gam;
  uint4 w[kIt];
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int idx = c.tid + it * kCT, r = idx >> 4, e0 = (idx & 15) * 8, t = r & 63;
    const bool zero = t >= ch.n || (kKind == kTRho && r >= 64 && t < 32);
    w[it] = zero ? make_uint4(0u, 0u, 0u, 0u)
                 : *reinterpret_cast<const uint4*>(x + (int64_t)t * xstride + e0);
  }
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int idx = c.tid + it * kCT, r = idx >> 4, e0 = (idx & 15) * 8, t = r & 63;
    const float sc = rx[t] * s;
    const float4 g0 = *reinterpret_cast<const float4*>(g + t * 128 + e0);
    const float4 g1 = *reinterpret_cast<const float4*>(g + t * 128 + e0 + 4);
    const float gt[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float rf[8];
    if (kKind == kTKt) {
#pragma unroll
      for (int i = 0; i < 8; ++i) rf[i] = 0.f;
    } else {
      const int rr = (kKind == kTKw) ? 63 : ((kKind == kTRho ? (r >= 64) : (t >= 32)) ? 47 : 15);
      const float4 a0 = *reinterpret_cast<const float4*>(g + rr * 128 + e0);
      const float4 a1 = *reinterpret_cast<const float4*>(g + rr * 128 + e0 + 4);
      rf[0] = a0.x; rf[1] = a0.y; rf[2] = a0.z; rf[3] = a0.w;
      rf[4] = a1.x; rf[5] = a1.y; rf[6] = a1.z; rf[7] = a1.w;
    }
    const float xv[8] = {bflo(w[it].x), bfhi(w[it].x), bflo(w[it].y), bfhi(w[it].y),
                         bflo(w[it].z), bfhi(w[it].z), bflo(w[it].w), bfhi(w[it].w)};
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // exponent: gam_t (Kt), gam_63 - gam_t (Kw), gam_t - rho (rho rows), rho - gam_t (B);
      // zero rows have x = 0 and finite factors
      const float e = (kKind == kTKt) ? gt[i]
                      : (kKind == kTKw) ? rf[i] - gt[i]
                      : (kKind == kTRho) ? gt[i] - rf[i]
                                         : rf[i] - gt[i];
      y[i] = (kKind == kTRho && r >= 64 && t < 32) ? 0.f : (xv[i] * sc) * ex2_approx(e);
    }
    st8(tile, blk, r, e0, y);
  }
}

// The Gram operands and Kt in one pass over the chunk's q and k rows: K-rho and
// Q-rho [128][128], B-rho [64][128] and Kt [64][128] (see build_tile for each).
__device__ void build_gram_tiles(Ctx& c, const uint16_t* qx, const uint16_t* kx, int64_t xstride,
                                 const Chunk& ch, uint8_t* kr, uint8_t* qr, uint8_t* br,
                                 uint8_t* kt) {
  const float* g = c.gam;
  uint4 wq[kStageIt], wk[kStageIt];
#pragma unroll
  for (int it = 0; it < kStageIt; ++it) {
    const int idx = c.tid + it * kCT, t = idx >> 4, e0 = (idx & 15) * 8;
    const bool z = t >= ch.n;
    wq[it] = z ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(qx + (int64_t)t * xstride + e0);
    wk[it] = z ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(kx + (int64_t)t * xstride + e0);
  }
#pragma unroll
  for (int it = 0; it < kStageIt; ++it) {
    const int idx = c.tid + it * kCT, t = idx >> 4, e0 = (idx & 15) * 8;
    const float sq = c.rq[t], sk = c.rk[t];
    float gt[8], r1[8], r2[8];
#pragma unroll
    for (int h4 = 0; h4 < 2; ++h4) {
      const float4 a = *reinterpret_cast<const float4*>(g + t * 128 + e0 + 4 * h4);
      const float4 b = *reinterpret_cast<const float4*>(g + 15 * 128 + e0 + 4 * h4);
      const float4 d = *reinterpret_cast<const float4*>(g + 47 * 128 + e0 + 4 * h4);
      gt[4 * h4] = a.x; gt[4 * h4 + 1] = a.y; gt[4 * h4 + 2] = a.z; gt[4 * h4 + 3] = a.w;
      r1[4 * h4] = b.x; r1[4 * h4 + 1] = b.y; r1[4 * h4 + 2] = b.z; r1[4 * h4 + 3] = b.w;
      r2[4 * h4] = d.x; r2[4 * h4 + 1] = d.y; r2[4 * h4 + 2] = d.z; r2[4 * h4 + 3] = d.w;
    }
    const float qv[8] = {bflo(wq[it].x), bfhi(wq[it].x), bflo(wq[it].y), bfhi(wq[it].y),
                         bflo(wq[it].z), bfhi(wq[it].z), bflo(wq[it].w), bfhi(wq[it].w)};
    const float kv[8] = {bflo(wk[it].x), bfhi(wk[it].x), bflo(wk[it].y), bfhi(wk[it].y),
                         bflo(wk[it].z), bfhi(wk[it].z), bflo(wk[it].w), bfhi(wk[it].w)};
    float k1[8], q1[8], k2[8], q2[8], bb[8], tt[8];
    const bool up = t >= 32;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float qh = qv[i] * sq, kh = kv[i] * sk;
      const float f1 = ex2_approx(gt[i] - r1[i]);
      const float f2 = up ? ex2_approx(gt[i] - r2[i]) : 0.f;
      k1[i] = kh * f1;
      q1[i] = qh * f1;
      k2[i] = kh * f2;
      q2[i] = qh * f2;
      bb[i] = kh * ex2_approx((up ? r2[i] : r1[i]) - gt[i]);
      tt[i] = kh * ex2_approx(gt[i]);
    }
    st8(kr, 16384, t, e0, k1);
    st8(kr, 16384, 64 + t, e0, k2);
    st8(qr, 16384, t, e0, q1);
    st8(qr, 16384, 64 + t, e0, q2);
    st8(br, 8192, t, e0, bb);
    st8(kt, 8192, t, e0, tt);
  }
}

// Gram of the chunk: [R_k; R_q] rows against the B columns.  Scratch columns
// 0..63: k rows; 64..127: q rows (reverse sweep only).  Row t of D holds the
// s < 32 columns (rho1), row 64 + t the s >= 32 columns (rho2).
__device__ __forceinline__ void issue_gram(const Ctx& c, const uint8_t* kr, const uint8_t* qr,
                                           const uint8_t* br, bool commit) {
  const uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
  const uint64_t a1 = dK(kr), a2 = dK(qr), b = dK(br);
#pragma unroll 1
  for (int k = 0; k < 8; ++k)
    mma_bf16_ss(c.tbase + tSC, a1 + kstep(k, 16384), b + kstep(k, 8192), id, k > 0);
#pragma unroll 1
  for (int k = 0; k < 8; ++k)
    mma_bf16_ss(c.tbase + tSC + 64, a2 + kstep(k, 16384), b + kstep(k, 8192), id, k > 0);
  if (commit) mma_commit(c.bar);
}

__device__ __forceinline__ void ld32f(const Ctx& c, uint32_t col, uint32_t (&u)[32]) {
  tmem_ld32(c.tbase + c.lane_off + col, u);
}
__device__ __forceinline__ void st32f(const Ctx& c, uint32_t col, const float (&x)[32]) {
  uint32_t u[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(x[i]);
  tmem_st32(c.tbase + c.lane_off + col, u);
}

__device__ __forceinline__ void ld16f(const Ctx& c, uint32_t col, uint32_t (&u)[16]) {
  tmem_ld16(c.tbase + c.lane_off + col, u);
}
__device__ __forceinline__ void st16f(const Ctx& c, uint32_t col, const float (&x)[16]) {
  uint32_t u[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(x[i]);
  tmem_st16(c.tbase + c.lane_off + col, u);
}
// 32 lanes x 8 consecutive 32-bit columns
__device__ __forceinline__ void ld8f(const Ctx& c, uint32_t col, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(c.tbase + c.lane_off + col));
}
__device__ __forceinline__ void st8f(const Ctx& c, uint32_t col, const float (&x)[8]) {
  uint32_t u[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) u[i] = __float_as_uint(x[i]);
  tmem_st8(c.tbase + c.lane_off + col, u);
}
// kN (8, 16 or 32) columns of this warp's lanes
template <int kN>
__device__ __forceinline__ void ldnf(const Ctx& c, uint32_t col, uint32_t (&u)[kN]) {
  static_assert(kN == 8 || kN == 16 || kN == 32, "8, 16 or 32 columns");
  if constexpr (kN == 32) ld32f(c, col, u);
  else if constexpr (kN == 16) ld16f(c, col, u);
  else ld8f(c, col, u);
}
template <int kN>
__device__ __forceinline__ void stnf(const Ctx& c, uint32_t col, const float (&x)[kN]) {
  static_assert(kN == 8 || kN == 16 || kN == 32, "8, 16 or 32 columns");
  if constexpr (kN == 32) st32f(c, col, x);
  else if constexpr (kN == 16) st16f(c, col, x);
  else st8f(c, col, x);
}

// Gram epilogue.  A = Diag(beta) P (strict lower, fp32, inverse workspace); with
// mq: P (fp32) and the bf16 tile scale*Mq [t][s] (lower incl.).  Warps with
// lanes 0..63 read columns 0..31 (rho1), warps with lanes 64..127 columns 32..63.
__device__ void gram_epilogue(Ctx& c, float* A, uint8_t* mq, float scale) {
  const int wq = c.warp & 3;
  const bool lowrows = wq < 2;
  // lanes 0..63 with the groups of columns 0..31, lanes 64..127 with those of 32..63
  if ((c.wg < kWG / 2) != lowrows) return;
  const int t = c.row & 63;
  const int s0 = kCols * c.wg;
  uint32_t u[kCols];
  ldnf<kCols>(c, tSC + s0, u);
  uint32_t m[kCols];
  if (mq) ldnf<kCols>(c, tSC + 64 + s0, m);
  tmem_wait_ld();
  const float bt = c.beta[t];
  float mv[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) {
    const int s = s0 + i;
    const float pv = (s < t) ? u2f(u[i]) : 0.f;
    A[t * inv::kLdM + s] = bt * pv;
    if (mq) {
      c.P[t * kLdP + s] = pv;
      mv[i] = (s <= t) ? scale * u2f(m[i]) : 0.f;
    }
  }
  if (mq) stn<kCols>(mq, 8192, t, s0, mv);
}


// R = V - (Kt S) from the AKp columns (lane v, columns t; V from staged rows):
// beta R to the tile [v][t], and R itself back to AKp (kept for rowsum(dR~ o R)).
__device__ void r_epilogue(const Ctx& c, const uint8_t* vrows, uint8_t* brt) {
  const int s0 = kCols * c.wg;
  uint32_t u[kCols];
  ldnf<kCols>(c, tAKp + s0, u);
  float vv[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) vv[i] = staged(vrows, s0 + i, c.row);
  tmem_wait_ld();
  float r[kCols], br[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) {
    r[i] = vv[i] - u2f(u[i]);
    br[i] = c.beta[s0 + i] * r[i];
  }
  stn<kCols>(brt, 16384, c.row, s0, br);
  stnf<kCols>(c, tAKp + s0, r);
}

// bf16 tile [lane][cols] from the scratch columns at `col` (this group's kCols).
__device__ void tile_from_tmem(const Ctx& c, uint32_t col, uint8_t* tile) {
  uint32_t u[kCols];
  ldnf<kCols>(c, col + kCols * c.wg, u);
  tmem_wait_ld();
  float x[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) x[i] = u2f(u[i]);
  stn<kCols>(tile, 16384, c.row, kCols * c.wg, x);
}

// T = (I + A)^-1 of the strictly lower A (fp32 [64][inv::kLdM] at M, written by
// the Gram epilogue) as the bf16 tile [t][s] `tb`: the forward kernel's blocked
// inverse (kda_inverse.cuh) with beta = 1, on warps 0..3; the other warps meanwhile
// zero the six strictly upper 16x16 blocks, which it does not write.  All threads call.
__device__ void inverse_tile(const Ctx& c, float* M, uint8_t* tb, const float* ones) {
  if (c.tid < 64) inv::inverse_level0(M, c.tid);
  if (c.tid < 128) {
    named_sync(inv::kBarF, inv::kSubThreads);
    inv::lbeta_inverse(M, tb, ones, c.tid);
  } else {
    for (int idx = c.tid - 128; idx < 6 * 32; idx += kCT - 128) {  // block, row, 8-column half
      const int blk = idx >> 5, r = (idx >> 1) & 15, hh = idx & 1;
      const int a = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
      const int b = blk < 3 ? 1 + blk : (blk < 5 ? blk - 1 : 3);
      *reinterpret_cast<uint4*>(tb + sw128(16 * a + r, (16 * b + 8 * hh) * 2)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// ---- the reverse sweep -----------------------------------------------------
// One chunk, given dS' in tDS (replaced by the chunk's start-state gradient).
// Accumulates the dt_bias / A_log sums of this thread into *acc_dt, *acc_a.
// `staged_in`: this chunk's q, k (and bf16 g) rows were staged by the previous
// chunk in slots kStQ, kStK (kStG); `next_n` > 0: stage the next chunk's (tokens
// tok0 - 64 ..) likewise, once the slots are free.
constexpr int kStQ = 6, kStK = 7, kStG = 5;
#ifndef KDA_BWD_STAGE_NEXT
#define KDA_BWD_STAGE_NEXT 1
#endif
constexpr bool kStageNext = KDA_BWD_STAGE_NEXT != 0;
__device__ bool reverse_chunk(Ctx& c, const BwdParams& p, const Chunk& ch, int h, int hk, float ea,
                              float dtbj, const uint16_t* ck_start, float* acc_dt, float* acc_a,
                              bool staged_in, int next_n) {
  const int HK = p.H / p.qk_group;
  const int64_t xs = (int64_t)HK * kHeadDim;
  const uint16_t* qx = p.q + (ch.tok0 * HK + hk) * kHeadDim;
  const uint16_t* kx = p.k + (ch.tok0 * HK + hk) * kHeadDim;
  // the chunk's start rows: staged copies (row stride 128) or global memory
  const bool stg = kStageNext && staged_in && !p.gate_f32;
  const uint16_t* qs = stg ? reinterpret_cast<const uint16_t*>(slot(c, kStQ)) : qx;
  const uint16_t* ks = stg ? reinterpret_cast<const uint16_t*>(slot(c, kStK)) : kx;
  const int64_t ss = stg ? kHeadDim : xs;
  const float scale = p.scale;
  const int lq = c.warp & 3, wg = c.wg, row = c.row;
  float* red = reinterpret_cast<float*>(c.sm + kOffRed);    // [4][128]
  float* red2 = reinterpret_cast<float*>(c.sm + kOffRed2);  // [4][128]
  float* eend = reinterpret_cast<float*>(c.sm + kOffEend);
  float* dd = reinterpret_cast<float*>(c.sm + kOffDd);
  float* db1 = reinterpret_cast<float*>(c.sm + kOffDb1);
  float* db2 = reinterpret_cast<float*>(c.sm + kOffDb2);     // [2][64]
  float* carry = reinterpret_cast<float*>(c.sm + kOffCarry); // [2][kWG][128]
  float* dots = reinterpret_cast<float*>(c.sm + kOffDots);   // [2][64]
  const float* gam = c.gam;

  if (stg) {
    cp_async_wait_all();
    __syncthreads();
  }
  prep_chunk(c, p, ch, h, ea, qs, ks, ss,
             stg ? reinterpret_cast<const uint16_t*>(slot(c, kStG)) : nullptr, kHeadDim);
  const int64_t vs = (int64_t)p.H * kHeadDim;  // row stride of v, g and dout
  {  // dout rows staged in slot bTM (free until the Gram epilogue)
    uint4 w[kStageIt];
    stage_load(c, p.dout + (ch.tok0 * p.H + h) * kHeadDim, vs, ch.n, w);
    build_gram_tiles(c, qs, ks, ss, ch, slot(c, bKr), slot(c, bQr), slot(c, bBr), slot(c, bKt));
    __syncthreads();  // the staged q / k rows (slots kStQ, kStK) are read before bTM, bS reuse
    stage_store(c, slot(c, bTM), w);
  }
  {  // S tile [v][k] from the checkpoint (bf16 row-major): 2048 16-byte pieces
    uint8_t* st = slot(c, bS);
    constexpr int kIt = 2048 / kCT;
    uint4 w[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int idx = c.tid + it * kCT, v = idx >> 4, e0 = (idx & 15) * 8;
      w[it] = *reinterpret_cast<const uint4*>(ck_start + v * kHeadDim + e0);
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int idx = c.tid + it * kCT, v = idx >> 4, e0 = (idx & 15) * 8;
      *reinterpret_cast<uint4*>(st + (uint32_t)(e0 >> 6) * 16384u + sw128(v, (e0 & 63) * 2)) = w[it];
    }
  }
  __syncthreads();
  {  // dO^T tile [v][t] from the staged rows: lane v, tokens of this group
    float x[kCols];
#pragma unroll
    for (int i = 0; i < kCols; ++i) x[i] = staged(slot(c, bTM), kCols * wg + i, row);
    stn<kCols>(slot(c, bDOT), 16384, row, kCols * wg, x);
  }
  if (publish(c)) return false;
  uint4 vw[kStageIt];  // v rows, loaded while the Gram runs, staged in slot bBr once it is read
  stage_load(c, p.v + (ch.tok0 * p.H + h) * kHeadDim, vs, ch.n, vw);
  if (c.tid == 0 && !p.debug_stall) {  // (timeout test: nothing is issued, nothing commits)
    tc_fence_after();
    issue_gram(c, slot(c, bKr), slot(c, bQr), slot(c, bBr), false);
    // (1) Kt S (R = V - Kt S) into the AKp columns: A = S [v][k], B = Kt [t][k]
    const uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
    const uint64_t a = dK(slot(c, bS)), b = dK(slot(c, bKt));
#pragma unroll 1
    for (int k = 0; k < 8; ++k) mma_bf16_ss(c.tbase + tAKp, a + kstep(k, 16384), b + kstep(k, 8192), id, k > 0);
    mma_commit(c.bar);
  }
  mma_wait(c, p.status);
  stage_store(c, slot(c, bBr), vw);
  __syncthreads();  // the staged dout rows are read (dO^T tile) and the v rows written
  float* A = reinterpret_cast<float*>(slot(c, 0) + kOffA);
  uint8_t* tb = slot(c, bTM);
  uint8_t* mqs = slot(c, bTM) + 8192;
  gram_epilogue(c, A, mqs, scale);
  r_epilogue(c, slot(c, bBr), slot(c, bBRT));
  __syncthreads();
  inverse_tile(c, A, tb, reinterpret_cast<const float*>(c.sm + kOffOnes));
  if (publish(c)) return false;
  if (c.tid == 0) {  // (2) U = T (beta R)
    tc_fence_after();
    const uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
    const uint64_t a = dK(slot(c, bBRT)), b = dK(tb);
#pragma unroll 1
    for (int k = 0; k < 4; ++k) mma_bf16_ss(c.tbase + tSC + 64, a + 2 * k, b + 2 * k, id, k > 0);
    mma_commit(c.bar);
  }
  mma_wait(c, p.status);
  tile_from_tmem(c, tSC + 64, slot(c, bUT));
  {  // dS' -> bf16 tile [v][k]; chunk-end gate term <S, dS'> per k; dS <- Diag(F_63) dS'
    uint8_t* dsp = slot(c, bDSp);
    const uint8_t* st = slot(c, bS);
#pragma unroll 1
    for (int h4 = 0; h4 < 8 / kWG; ++h4) {
      const int k0 = (128 / kWG) * wg + 16 * h4;
      uint32_t u[16];
      ld16f(c, tDS + k0, u);
      tmem_wait_ld();
      float x[16], pr[16];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 w = *reinterpret_cast<const uint4*>(
            st + (uint32_t)(k0 >> 6) * 16384u + sw128(row, ((k0 & 63) + 8 * q) * 2));
        const float sv[8] = {bflo(w.x), bfhi(w.x), bflo(w.y), bfhi(w.y),
                             bflo(w.z), bfhi(w.z), bflo(w.w), bfhi(w.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) pr[8 * q + i] = sv[i] * u2f(u[8 * q + i]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = u2f(u[i]);
      st16(dsp, 16384, row, k0, x);
      const float part = warp_rs16(pr, c.lane);
      if (c.lane < 16) red[lq * 128 + k0 + c.lane] = part;
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] *= ex2_approx(gam[63 * 128 + k0 + i]);
      st16f(c, tDS + k0, x);
    }
  }
  build_tile<kTKw, 64>(c, slot(c, bKw), kx, xs, c.rk, ch, 1.f);
  if (publish(c)) return false;
  if (c.tid < 128)
    eend[c.tid] = ex2_approx(gam[63 * 128 + c.tid]) *
                  (((red[c.tid] + red[128 + c.tid]) + red[256 + c.tid]) + red[384 + c.tid]);
  if (c.tid == 0) {
    tc_fence_after();
    // (3) dU = Kw dS' + scale Mq^T dO:  A = dS'^T [v][k], B = Kw [t][k];  A = dO^T [v][t'],
    //     B = scale Mq [t'][s] (MN-major)
    const uint32_t id = idesc_bf16_f32(128, 64, 0, 0), idm = idesc_bf16_f32(128, 64, 0, 1);
    const uint64_t a = dK(slot(c, bDSp)), b = dK(slot(c, bKw));
#pragma unroll 1
    for (int k = 0; k < 8; ++k) mma_bf16_ss(c.tbase + tSC, a + kstep(k, 16384), b + kstep(k, 8192), id, k > 0);
    const uint64_t a2 = dK(slot(c, bDOT)), b2 = dMN(mqs, 8192);
#pragma unroll 1
    for (int k = 0; k < 4; ++k) mma_bf16_ss(c.tbase + tSC, a2 + 2 * k, b2 + 128 * k, idm, 1u);
    // (8) (U dS'^T)^T = dS' U^T into AKi:  A = dS' (MN-major over [v][k]), B = U (MN-major)
    const uint32_t id8 = idesc_bf16_f32(128, 64, 1, 1);
    const uint64_t a8 = dMN(slot(c, bDSp), 16384), b8 = dMN(slot(c, bUT), 16384);
#pragma unroll 1
    for (int k = 0; k < 8; ++k) mma_bf16_ss(c.tbase + tAKi, a8 + 128 * k, b8 + 128 * k, id8, k > 0);
    mma_commit(c.bar);
  }
  mma_wait(c, p.status);
  tile_from_tmem(c, tSC, slot(c, bDUT));
  {  // AKi: (U dS'^T) o E, the inter-chunk part of dk^ through Kb
    uint32_t u[kCols];
    ldnf<kCols>(c, tAKi + kCols * wg, u);
    tmem_wait_ld();
    float a[kCols];
#pragma unroll
    for (int i = 0; i < kCols; ++i)
      a[i] = u2f(u[i]) * ex2_approx(gam[63 * 128 + row] - gam[(kCols * wg + i) * 128 + row]);
    stnf<kCols>(c, tAKi + kCols * wg, a);
  }
  if (publish(c)) return false;
  if (c.tid == 0) {  // (4) dR~ = T^T dU: A = dU^T [v][t], B = Tb [t][s] (MN-major)
    tc_fence_after();
    const uint32_t id = idesc_bf16_f32(128, 64, 0, 1);
    const uint64_t a = dK(slot(c, bDUT)), b = dMN(tb, 8192);
#pragma unroll 1
    for (int k = 0; k < 4; ++k) mma_bf16_ss(c.tbase + tSC + 64, a + 2 * k, b + 128 * k, id, k > 0);
    mma_commit(c.bar);
  }
  mma_wait(c, p.status);
#pragma unroll 1
  for (int hh = 0; hh < kCols / 16; ++hh) {  // dV = Diag(beta) dR~; rowsum(dR~ o R); dR~^T, -(beta dR~)^T
    const int s0 = kCols * wg + 16 * hh;
    uint32_t u[16], rr[16];
    ld16f(c, tSC + 64 + s0, u);
    ld16f(c, tAKp + s0, rr);
    float bt[16];  // read ahead of the dv stores (see the final pass)
#pragma unroll
    for (int i = 0; i < 16; ++i) bt[i] = c.beta[s0 + i];
    tmem_wait_ld();
    float x[16], y[16], pr[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int s = s0 + i;
      x[i] = u2f(u[i]);
      y[i] = -bt[i] * x[i];
      pr[i] = x[i] * u2f(rr[i]);
      if (s < ch.n) p.dv[((ch.tok0 + s) * p.H + h) * kHeadDim + row] = bt[i] * x[i];
    }
    st16(slot(c, bDRt), 16384, row, s0, x);
    st16(slot(c, bNdR), 16384, row, s0, y);
    const float part = warp_rs16(pr, c.lane);
    if (c.lane < 16) red2[lq * 128 + s0 + c.lane] = part;
  }
  if (publish(c)) return false;
  if (c.tid < 64)
    db1[c.tid] = ((red2[c.tid] + red2[128 + c.tid]) + red2[256 + c.tid]) + red2[384 + c.tid];
  if (c.tid == 0) {
    tc_fence_after();
    // (5) [dR~ ; dO] U^T: A = [dR~^T | dO^T] MN-major, B = U^T MN-major
    const uint32_t id = idesc_bf16_f32(128, 64, 1, 1);
    const uint64_t a = dMN(slot(c, bDRt), (uint32_t)(bDOT - bDRt) * kSlot), b = dMN(slot(c, bUT), 16384);
#pragma unroll 1
    for (int k = 0; k < 8; ++k) mma_bf16_ss(c.tbase + tSC, a + 128 * k, b + 128 * k, id, k > 0);
    // (9) S [dO ; -dR]^T straight into AQ | AKt: A = S (MN-major over [v][k]),
    //     B = [dO^T | NdR^T] MN-major
    const uint32_t id9 = idesc_bf16_f32(128, 128, 1, 1);
    const uint64_t a9 = dMN(slot(c, bS), 16384), b9 = dMN(slot(c, bDOT), (uint32_t)(bNdR - bDOT) * kSlot);
#pragma unroll 1
    for (int k = 0; k < 8; ++k) mma_bf16_ss(c.tbase + tAQ, a9 + 128 * k, b9 + 128 * k, id9, k > 0);
    mma_commit(c.bar);
  }
  mma_wait(c, p.status);
  {  // rows t: dA = -(dR~ U^T) (strict), dP = beta dA -> X rows 64 + t; rows 64 + t:
     // dMq = scale (dO U^T) (strict) -> X rows t, diagonal -> dd.  X is stored at
     // 2^-shift (a power of two: exact) with |X| 2^-shift <= 16, so that the pair
     // products, whose operands reach 2^115 under saturated decay, stay in fp32 range
     // for any value magnitude; the folds multiply by 2^shift last.
    uint32_t u[kCols];
    ldnf<kCols>(c, tSC + kCols * wg, u);
    tmem_wait_ld();
    const int t = row & 63;
    float x[kCols];
    float mx = 0.f;
    if (row < 64) {
      const float bt = c.beta[t];
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kCols; ++i) {
        const int s = kCols * wg + i;
        const float da = s < t ? -u2f(u[i]) : 0.f;
        acc = fmaf(da, c.P[t * kLdP + s], acc);
        x[i] = bt * da;
        mx = fmaxf(mx, fabsf(x[i]));
      }
      db2[wg * 64 + t] = acc;
    } else {
#pragma unroll
      for (int i = 0; i < kCols; ++i) {
        const int s = kCols * wg + i;
        const float m = scale * u2f(u[i]);
        x[i] = s < t ? m : 0.f;
        if (s == t) dd[t] = m;
        mx = fmaxf(mx, fabsf(x[i]));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float* wmax = reinterpret_cast<float*>(c.sm + kOffWmax);
    if (c.lane == 0) wmax[c.warp] = mx;
    __syncthreads();
    mx = wmax[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) mx = fmaxf(mx, wmax[w]);
    // floor(log2 mx) from the exponent field (mx >= 0; inf / nan make the gradients
    // non-finite anyway); shift = floor(log2 mx) - 3 when positive
    const int e2 = (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127;
    const int shift = e2 > 3 ? (e2 - 3 < 124 ? e2 - 3 : 124) : 0;
    const float down = __uint_as_float((uint32_t)(127 - shift) << 23);
    if (c.tid == 0) wmax[kShiftIdx] = __uint_as_float((uint32_t)(127 + shift) << 23);
#pragma unroll
    for (int i = 0; i < kCols; ++i) x[i] *= down;
    stn<kCols>(slot(c, bX), 16384, row < 64 ? 64 + t : t, kCols * wg, x);
  }
#pragma unroll 1
  for (int hh = 0; hh < kCols / 16; ++hh) {  // D9 in place: AQ = scale (dO S^T) o F, AKt = -(dR S^T) o F
    const int t0 = kCols * wg + 16 * hh;
    uint32_t u1[16], u2[16];
    ld16f(c, tAQ + t0, u1);
    ld16f(c, tAKt + t0, u2);
    tmem_wait_ld();
    float a[16], b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float f = ex2_approx(gam[(t0 + i) * 128 + row]);
      a[i] = scale * u2f(u1[i]) * f;
      b[i] = u2f(u2[i]) * f;
    }
    st16f(c, tAQ + t0, a);
    st16f(c, tAKt + t0, b);
  }
  build_tile<kTKt, 64>(c, slot(c, bQtS), qx, xs, c.rq, ch, scale);
  build_tile<kTKt, 64>(c, slot(c, bKt2), kx, xs, c.rk, ch, 1.f);
  if (publish(c)) return false;
  if (c.tid < 64) {
    float b = db2[c.tid] + db2[64 + c.tid];
    for (int q = 2; q < kWG; ++q) b += db2[64 * q + c.tid];
    db2[c.tid] = b;
  }
  if (c.tid == 0) {
    tc_fence_after();
    // (10) dS += scale Qt^T dO - Kt^T dR: A = [dO^T | NdR^T] (K-major), B = [QtS | Kt] (MN-major)
    const uint32_t id = idesc_bf16_f32(128, 128, 0, 1);
    const uint64_t a1 = dK(slot(c, bDOT)), b1 = dMN(slot(c, bQtS), 8192);
    const uint64_t a2 = dK(slot(c, bNdR)), b2 = dMN(slot(c, bKt2), 8192);
#pragma unroll 1
    for (int k = 0; k < 4; ++k) mma_bf16_ss(c.tbase + tDS, a1 + 2 * k, b1 + 128 * k, id, 1u);
#pragma unroll 1
    for (int k = 0; k < 4; ++k) mma_bf16_ss(c.tbase + tDS, a2 + 2 * k, b2 + 128 * k, id, 1u);
  }
  build_tile<kTBrho, 64>(c, slot(c, bBr2), kx, xs, c.rk, ch, 1.f);
  if (publish(c)) return false;
  // (6) pairs(X, k^): A = B-rho (MN-major over [s][j]), B = X [n][s] (K-major); two passes
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (c.tid == 0) {
      tc_fence_after();
      const uint32_t id = idesc_bf16_f32(128, 128, 1, 0);
      const uint64_t a = dMN(slot(c, bBr2), 8192), b = dK(slot(c, bX));
#pragma unroll 1
      for (int k = 2 * pass; k < 2 * pass + 2; ++k)
        mma_bf16_ss(c.tbase + tSC, a + 128 * k, b + 2 * k, id, k > 2 * pass);
      mma_commit(c.bar);
    }
    mma_wait(c, p.status);
    if (pass == 0 || kCols * wg >= 32) {  // rho2 only meets tokens t >= 32
      const float ref = gam[(pass ? 47 : 15) * 128 + row];
      const float up = reinterpret_cast<const float*>(c.sm + kOffWmax)[kShiftIdx];  // 2^shift of X
#pragma unroll 1
      for (int hh = 0; hh < kCols / 16; ++hh) {
        const int t0 = kCols * wg + 16 * hh;
        uint32_t u1[16], u2[16], aq[16], ak[16];
        ld16f(c, tSC + t0, u1);
        ld16f(c, tSC + 64 + t0, u2);
        ld16f(c, tAQ + t0, aq);
        ld16f(c, tAKt + t0, ak);
        tmem_wait_ld();
        float o1[16], o2[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float f = ex2_approx(gam[(t0 + i) * 128 + row] - ref);
          o1[i] = u2f(aq[i]) + (u2f(u1[i]) * f) * up;
          o2[i] = u2f(ak[i]) + (u2f(u2[i]) * f) * up;
        }
        st16f(c, tAQ + t0, o1);
        st16f(c, tAKt + t0, o2);
      }
    }
    if (publish(c)) return false;
  }
  // every MMA so far has completed (including (10)): slots 0, 1 and 4..9 are free.
  // q, k and g rows for the final pass: q -> slot 0, k -> slot 1, g -> slot 8 (fp32: 8, 9)
  {
    uint4 wq[kStageIt], wk[kStageIt];
    stage_load(c, qx, xs, ch.n, wq);
    stage_load(c, kx, xs, ch.n, wk);
    build_tile<kTRho, 128>(c, slot(c, bKr2), kx, xs, c.rk, ch, 1.f);
    build_tile<kTRho, 128>(c, slot(c, bQr2), qx, xs, c.rq, ch, 1.f);
    stage_store(c, slot(c, 0), wq);
    stage_store(c, slot(c, 1), wk);
    if (p.gate_f32) {
      const float* g = static_cast<const float*>(p.g) + (ch.tok0 * p.H + h) * kHeadDim;
      float* dst = reinterpret_cast<float*>(slot(c, 8));
#pragma unroll
      for (int it = 0; it < 2048 / kCT; ++it) {
        const int idx = c.tid + it * kCT, t = idx >> 5, e0 = (idx & 31) * 4;
        *reinterpret_cast<float4*>(dst + t * 128 + e0) =
            t < ch.n ? *reinterpret_cast<const float4*>(g + (int64_t)t * vs + e0)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
      uint4 wg4[kStageIt];
      stage_load(c, static_cast<const uint16_t*>(p.g) + (ch.tok0 * p.H + h) * kHeadDim, vs, ch.n, wg4);
      stage_store(c, slot(c, 8), wg4);
    }
  }
  if (publish(c)) return false;
  if (c.tid == 0) {  // (7) pairs^T: A = [Q-rho | K-rho] rows (MN-major), B = X rows (MN-major)
    tc_fence_after();
    const uint32_t id = idesc_bf16_f32(128, 64, 1, 1);
    const uint64_t aq = dMN(slot(c, bQr2), 16384), ak = dMN(slot(c, bKr2), 16384);
    const uint64_t bx = dMN(slot(c, bX), 16384);
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {  // rows 0..63 (rho1) -> cols 0..63; 64..127 -> 64..127
      const uint32_t ro = half ? 512u : 0u;
#pragma unroll 1
      for (int k = 0; k < 4; ++k)
        mma_bf16_ss(c.tbase + tSC + 64 * half, aq + ro + 128 * k, bx + 128 * k, id, k > 0);
#pragma unroll 1
      for (int k = 0; k < 4; ++k)
        mma_bf16_ss(c.tbase + tSC + 64 * half, ak + ro + 128 * k, bx + 512 + 128 * k, id, 1u);
    }
    mma_commit(c.bar);
  }
  mma_wait(c, p.status);
  if (kStageNext && next_n > 0 && !p.gate_f32) {  // slots 4..7 free: the next chunk's q, k, g
    const int64_t t1 = ch.tok0 - kChunk;
    stage_async(c, slot(c, kStQ), p.q + (t1 * HK + hk) * kHeadDim, xs, next_n);
    stage_async(c, slot(c, kStK), p.k + (t1 * HK + hk) * kHeadDim, xs, next_n);
    stage_async(c, slot(c, kStG), static_cast<const uint16_t*>(p.g) + (t1 * p.H + h) * kHeadDim,
                vs, next_n);
    cp_async_commit();
  }
  {  // AKp = 2^(rho - gam_s) (...): tokens s < 32 from the rho1 half (columns s),
     // s >= 32 from the rho2 half (columns 64 + s)
    const int s0 = kCols * wg;
    const bool hi = s0 >= 32;
    uint32_t u[kCols];
    ldnf<kCols>(c, tSC + s0 + (hi ? 64 : 0), u);
    tmem_wait_ld();
    const float ref = gam[(hi ? 47 : 15) * 128 + row];
    const float up = reinterpret_cast<const float*>(c.sm + kOffWmax)[kShiftIdx];  // 2^shift of X
    float o[kCols];
#pragma unroll
    for (int i = 0; i < kCols; ++i)
      o[i] = (u2f(u[i]) * ex2_approx(ref - gam[(s0 + i) * 128 + row])) * up;
    stnf<kCols>(c, tAKp + s0, o);
  }
  tmem_wait_st();
  // ---- final pass (lane j, tokens of this half): diagonal pairs, gate terms and
  // their cumulative sums, the gate, l2-norm and sigmoid reverses, outputs.
  {
    // (a) dq^, dk^ with the diagonal pairs (AQ, AKt); the gate terms summed over
    // later tokens (AKp: suffix sums within each 16-token group) and over earlier
    // ones (AKi: exclusive prefix sums within the group); per-token dots of the norms
    constexpr int kS = kCols / 2;  // tokens per sub-group: two sub-groups per thread
    float lsum0 = 0.f, lsum1 = 0.f, isum0 = 0.f, isum1 = 0.f;
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      const int t0 = kCols * wg + kS * hh;
      uint32_t uq[kS], ut[kS], up[kS], ui[kS];
      ldnf<kS>(c, tAQ + t0, uq);
      ldnf<kS>(c, tAKt + t0, ut);
      ldnf<kS>(c, tAKp + t0, up);
      ldnf<kS>(c, tAKi + t0, ui);
      float qh[kS], kh[kS];
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        qh[i] = staged(slot(c, 0), t0 + i, row) * c.rq[t0 + i];
        kh[i] = staged(slot(c, 1), t0 + i, row) * c.rk[t0 + i];
      }
      tmem_wait_ld();
      float dq[kS], dk[kS], gl[kS], gi[kS];
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const float d = dd[t0 + i];
        const float aq = u2f(uq[i]), at = u2f(ut[i]), ap = u2f(up[i]), ai = u2f(ui[i]);
        dq[i] = aq + d * kh[i];
        dk[i] = ((at + ap) + ai) + d * qh[i];
        gl[i] = qh[i] * aq + kh[i] * (at - ap);
        gi[i] = kh[i] * ai;
      }
      float run = 0.f;
#pragma unroll
      for (int i = kS - 1; i >= 0; --i) {
        run += gl[i];
        gl[i] = run;
      }
      if (hh == 0) lsum0 = run; else lsum1 = run;
      run = 0.f;
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const float x = gi[i];
        gi[i] = run;
        run += x;
      }
      if (hh == 0) isum0 = run; else isum1 = run;
      stnf<kS>(c, tAQ + t0, dq);
      stnf<kS>(c, tAKt + t0, dk);
      stnf<kS>(c, tAKp + t0, gl);
      stnf<kS>(c, tAKi + t0, gi);
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        dq[i] *= qh[i];
        dk[i] *= kh[i];
      }
      const float pq = warp_rs<kS>(dq, c.lane), pk = warp_rs<kS>(dk, c.lane);
      if (c.lane < kS) {
        red[lq * 128 + t0 + c.lane] = pq;
        red2[lq * 128 + t0 + c.lane] = pk;
      }
    }
    {  // this group's totals: suffix sums for the earlier groups, prefix sums for the later
      carry[wg * 128 + row] = lsum0 + lsum1;
      carry[(kWG + wg) * 128 + row] = isum0 + isum1;
    }
    tmem_wait_st();
    __syncthreads();
    if (c.tid < 64) {
      const int t = c.tid;
      dots[t] = ((red[t] + red[128 + t]) + red[256 + t]) + red[384 + t];
      dots[64 + t] = ((red2[t] + red2[128 + t]) + red2[256 + t]) + red2[384 + t];
    }
    __syncthreads();
    // (c) per token: gate reverse, l2-norm reverse, outputs
    float cl0 = 0.f, ci0 = 0.f;
    for (int q = kWG - 1; q > wg; --q) cl0 += carry[q * 128 + row];
    for (int q = 0; q < wg; ++q) ci0 += carry[(kWG + q) * 128 + row];
    const float e = eend[row];
    const float lb = p.lower_bound;
    const int j = row;
    float adt = 0.f, aa = 0.f;
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
      const int t0 = kCols * wg + kS * hh;
      // sub-group offsets: the later sub-group's total for the suffix sums, the
      // earlier one's for the prefix sums
      const float cl = cl0 + (hh == 0 ? lsum1 : 0.f);
      const float ci = ci0 + (hh == 1 ? isum0 : 0.f);
      uint32_t uq[kS], uk[kS], ul[kS], ui[kS];
      ldnf<kS>(c, tAQ + t0, uq);
      ldnf<kS>(c, tAKt + t0, uk);
      ldnf<kS>(c, tAKp + t0, ul);
      ldnf<kS>(c, tAKi + t0, ui);
      // every shared-memory operand of the token loop is read here, ahead of the
      // global stores: the compiler does not move a read through a generic pointer
      // past a store that it cannot prove to be elsewhere
      float qh[kS], kh[kS], gv[kS], rq[kS], rk[kS];
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const int t = t0 + i;
        rq[i] = c.rq[t];
        rk[i] = c.rk[t];
        qh[i] = staged(slot(c, 0), t, j) * rq[i] * dots[t];
        kh[i] = staged(slot(c, 1), t, j) * rk[i] * dots[64 + t];
        gv[i] = p.gate_f32 ? reinterpret_cast<const float*>(slot(c, 8))[t * kHeadDim + j]
                           : staged(slot(c, 8), t, j);
      }
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const int t = t0 + i;
        if (t < ch.n) {
          const float dla = (e + (u2f(ul[i]) + cl)) + (u2f(ui[i]) + ci);
          const int64_t o = ((ch.tok0 + t) * p.H + h) * kHeadDim + j;
          const float x = ea * (gv[i] + dtbj);
          const float dpre = dla * lb * sig_prod(x);
          const float dgv = dpre * ea;
          p.dg[o] = dgv;
          adt += dgv;
          aa = fmaf(dpre, x, aa);
          const float gq = rq[i] * (u2f(uq[i]) - qh[i]);
          const float gk = rk[i] * (u2f(uk[i]) - kh[i]);
          if (p.qk_group == 1) {
            const int64_t oq = ((ch.tok0 + t) * HK + hk) * kHeadDim + j;
            p.dq[oq] = gq;
            p.dk[oq] = gk;
          } else {
            p.dq_part[o] = gq;
            p.dk_part[o] = gk;
          }
        }
      }
    }
    *acc_dt += adt;
    *acc_a += aa;
    if (c.tid < 64 && c.tid < ch.n) {
      const int t = c.tid;
      const float br = bf1(p.beta[(ch.tok0 + t) * p.H + h]);
      p.dbeta[(ch.tok0 + t) * p.H + h] = (db1[t] + db2[t]) * sig_prod(br);
    }
  }
  __syncthreads();  // the chunk's shared arrays are read before the next chunk's prep
  return true;
}

// bounds of sequence n; false for inconsistent cu_seqlens
__device__ __forceinline__ bool seq_bounds(const BwdParams& p, int n, int64_t& bos, int64_t& eos) {
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

// Load a [V][K] state (fp32 / bf16 / null = zero) into the TMEM state columns.
__device__ void state_in(const Ctx& c, const void* src, bool is_bf16) {
#pragma unroll 1
  for (int h2 = 0; h2 < 4 / kWG; ++h2) {
    const int k0 = (128 / kWG) * c.wg + 32 * h2;
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int64_t o = (int64_t)c.row * kHeadDim + k0 + i;
      x[i] = !src ? 0.f
                  : (is_bf16 ? bf1(static_cast<const uint16_t*>(src)[o])
                             : static_cast<const float*>(src)[o]);
    }
    st32f(c, tDS + k0, x);
  }
  tmem_wait_st();
}

__global__ void __launch_bounds__(kCT, 1) kda_bwd_chunk_kernel(const BwdParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = smem_align1024(smraw);
  Ctx c;
  c.sm = sm;
  c.gam = reinterpret_cast<float*>(sm + kOffGam);
  c.P = reinterpret_cast<float*>(sm + kOffP);
  c.beta = reinterpret_cast<float*>(sm + kOffBeta);
  c.rq = reinterpret_cast<float*>(sm + kOffRq);
  c.rk = reinterpret_cast<float*>(sm + kOffRk);
  c.bar = reinterpret_cast<uint64_t*>(sm + kOffBar);
  c.abort = reinterpret_cast<volatile int*>(sm + kOffAbort);
  c.tid = threadIdx.x;
  c.warp = c.tid >> 5;
  c.lane = c.tid & 31;
  c.wg = c.warp >> 2;
  c.row = 32 * (c.warp & 3) + c.lane;
  c.lane_off = (uint32_t)(32 * (c.warp & 3)) << 16;
  c.phase = 0;
  if (c.tid < 64) reinterpret_cast<float*>(sm + kOffOnes)[c.tid] = 1.f;
  if (c.tid == 0) {
    mbar_init(c.bar, 1);
    *c.abort = 0;
    fence_mbar_init();
  }
  if (c.warp == 0) {
    tmem_alloc(reinterpret_cast<uint32_t*>(sm + kOffTaddr), kTCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tbase = *reinterpret_cast<volatile uint32_t*>(sm + kOffTaddr);

  const int H = p.H;
  const int units = p.N * H;
  float* accs = reinterpret_cast<float*>(sm + kOffAcc);  // [kWG][128] dt_bias, then [kCT] A_log
  uint16_t* ck = reinterpret_cast<uint16_t*>(p.ckpt);
#pragma unroll 1
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int n = u / H, h = u % H, hk = h / p.qk_group;
    int64_t bos, eos;
    if (!seq_bounds(p, n, bos, eos)) {
      if (c.tid == 0) atomicOr(p.status, kDevStatusBadSeqlens);
      if (c.tid <= kHeadDim) p.unit_part[(int64_t)u * (kHeadDim + 1) + c.tid] = 0.f;
      continue;
    }
    const int64_t len = eos - bos;
    const int nch = (int)((len + kChunk - 1) / kChunk);
    const float ea = expf(p.A_log[h]);
    const float dtbj = p.dt_bias[h * kHeadDim + c.row];
    const int64_t slot0 = bos / kChunk + 2 * (int64_t)n;  // checkpoint slots slot0 .. slot0 + nch
    uint16_t* ckbase = ck + (slot0 * H + h) * (int64_t)(kHeadDim * kHeadDim);
    const int64_t st_off = (int64_t)u * kHeadDim * kHeadDim;
    const void* dfin = p.dfinal ? (p.state_bf16 ? (const void*)(static_cast<const uint16_t*>(p.dfinal) + st_off)
                                                : (const void*)(static_cast<const float*>(p.dfinal) + st_off))
                                : nullptr;
    bool ok = true;
    float acc_dt = 0.f, acc_a = 0.f;
    {
      state_in(c, dfin, p.state_bf16 != 0);
      const int64_t ckstride = (int64_t)H * kHeadDim * kHeadDim;
#pragma unroll 1
      for (int ci = nch - 1; ci >= 0 && ok; --ci) {
        Chunk ch;
        ch.tok0 = bos + (int64_t)ci * kChunk;
        ch.n = (int)((len - (int64_t)ci * kChunk) < kChunk ? (len - (int64_t)ci * kChunk) : kChunk);
        ch.last = ci;
        if (ci > 0) {  // the chunk before this one is next: its checkpoint into L2
          prefetch_ckpt(c, ckbase + (int64_t)(ci - 1) * ckstride);
        } else if (u + (int)gridDim.x < units) {  // the next unit's last chunk comes next
          const int u2 = u + (int)gridDim.x, n2 = u2 / H, h2 = u2 % H;
          int64_t b2, e2;
          if (seq_bounds(p, n2, b2, e2) && e2 > b2) {
            const int64_t s2 = b2 / kChunk + 2 * (int64_t)n2 + (e2 - b2 - 1) / kChunk;
            prefetch_ckpt(c, ck + (s2 * H + h2) * (int64_t)(kHeadDim * kHeadDim));
          }
        }
        ok = reverse_chunk(c, p, ch, h, hk, ea, dtbj, ckbase + (int64_t)ci * ckstride, &acc_dt,
                           &acc_a, ci < nch - 1, ci > 0 ? kChunk : 0);
      }
    }
    if (__syncthreads_or(!ok || *c.abort)) break;  // an expired wait: the status word has it
    // dinitial_state (lane v, columns k) and the unit's dt_bias / A_log partial sums
    tmem_wait_st();
    if (p.dinit) {
#pragma unroll 1
      for (int h2 = 0; h2 < 4 / kWG; ++h2) {
        const int k0 = (128 / kWG) * c.wg + 32 * h2;
        uint32_t w[32];
        ld32f(c, tDS + k0, w);
        tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(p.dinit + st_off + (int64_t)c.row * kHeadDim + k0);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(u2f(w[4 * q]), u2f(w[4 * q + 1]), u2f(w[4 * q + 2]), u2f(w[4 * q + 3]));
      }
    }
    accs[c.wg * 128 + c.row] = acc_dt;
    accs[kWG * 128 + c.tid] = acc_a;
    __syncthreads();
    if (c.tid < kHeadDim) {
      float s = accs[c.tid] + accs[128 + c.tid];
      for (int q = 2; q < kWG; ++q) s += accs[128 * q + c.tid];
      p.unit_part[(int64_t)u * (kHeadDim + 1) + c.tid] = s;
    } else if (c.tid == kHeadDim) {
      float s = 0.f;
      for (int i = 0; i < kCT; ++i) s += accs[kWG * 128 + i];
      p.unit_part[(int64_t)u * (kHeadDim + 1) + kHeadDim] = s;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  if (c.warp == 0) tmem_dealloc(c.tbase, kTCols);
}

}  // namespace

cudaError_t launch_bwd_chunk(const BwdParams& p, int num_sms, float* dA_log, float* ddt_bias,
                             cudaStream_t stream) {
  static bool attr_done[64];
  const cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kda_bwd_chunk_kernel),
                                         (int)kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)p.N * p.H;
  const int64_t grid = units < num_sms ? units : num_sms;
  if (grid > 0) kda_bwd_chunk_kernel<<<(unsigned)grid, kCT, kSmemBytes, stream>>>(p);
  return launch_bwd_reduce(p, dA_log, ddt_bias, stream);
}

}  // namespace kda
