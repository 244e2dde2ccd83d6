// kda_chunk_fwd.cu -- fused, warp-specialised chunked forward of Kimi Delta
// Attention on sm_103a.
//
// One CTA owns one (sequence, value head) unit and walks its 64-token chunks; q
// and k come from the unit's key head (value heads per key head: qk_group).
// Three warp groups work concurrently, each on a different chunk:
//
//   prep group   (warps 8-15)  chunk c+1: gate
//       log2 a = lower_bound*log2(e)*sigmoid(exp(A_log)(g + dt_bias)), in-chunk
//       cumulative decay gam_r per channel, q/k l2-norm, beta = sigmoid(beta),
//       and the decayed bf16 operands of the Gram product       (CUDA cores)
//       Gram  A = beta K Diag(decay) K^T (strict lower), P = Q Diag(decay) K^T
//             (lower incl.), issued when the chunk is prepared    (tcgen05)
//       and the store of the outputs O of chunk c-2, out of TMEM  (CUDA cores)
//   factor group (warps 4-7)   chunk c:
//       L^{-1} of L = I + A: 16x16 diagonal blocks by forward substitution,
//             off-diagonal blocks with tf32 mma.sync
//       W = L^{-1} Diag(beta)(K o Gam), U~ = L^{-1} Diag(beta) V  (tcgen05)
//       Q' = Q o Gam - P W,  O_intra = P U~                       (tcgen05)
//       (the state group writes the U~^T tile and half of Q'^T)
//   state group  (warps 0-3)   chunk c-1: the inter-chunk recurrence
//       U = U~ - W S,  O = scale (Q' S + O_intra)                 (tcgen05)
//       S <- Diag(Gam_last) S + (K o Gam_last/Gam)^T U             (tcgen05 + registers)
//
// This is the chunked WY / UT form that the FlashKDA kernels split into K1 (the
// prep and factor groups here) and K2 (the state group) ("feat(kda): SM90
// FlashKDA prefill, intracard CP, and backend dispatch", commit notes).
// Differences from that SM90 design: 64-token chunks so every contraction is an
// M=128 tcgen05.mma with the accumulator in TMEM; the decay factorisation inside
// a chunk uses two reference points (tokens 15 and 47) so every exp() factor
// stays inside [e^-80, e^80] for lower_bound >= -5; K1 and K2 live in one kernel
// and overlap, so only the raw inputs and the output touch HBM.
//
// The 128x128 fp32 state stays in TMEM next to its bf16 copy and the bf16 U
// operand, which the MMAs read from there.
// Raw q/k/v/g chunk tiles arrive by TMA with 128-byte swizzle straight into the
// layout the MMAs read.  An fp32 gate has no room in shared memory: the kernel
// is instantiated for it (kGateF32) and its prep group reads g from L2.
#include <cuda_bf16.h>

#include <cstring>

#include "kda_internal.h"
#include "kda_ptx.cuh"
#include "kda_inverse.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kStateThreads = 128;             // warps 0-3
constexpr int kSubThreads = 128;               // factor group, warps 4-7
constexpr int kPrepThreads = 256;              // prep group, warps 8-15
constexpr uint32_t kBarP = 1, kBarK2 = 2, kBarF = 3, kBarF0 = 4;  // named barrier ids
static_assert(kBarF == inv::kBarF && kBarF0 == inv::kBarF0 && kSubThreads == inv::kSubThreads,
              "the shared inverse's barriers");
constexpr uint64_t kWaitNs = 500ull * 1000ull * 1000ull;  // bounded waits: 0.5 s
constexpr float kLog2e = 1.4426950408889634f;
// Largest in-chunk factor 2^(rho2 - gam63) of the C2 columns that the state MMA
// takes unshifted; above it the update is accumulated at 2^-m scale (see prep).
constexpr int kShiftFree = 64;

// ---- shared memory map (byte offsets from a 1024-aligned base) -------------
constexpr uint32_t kStageBytes = 65536;
constexpr uint32_t kOffQK = 0;      // [k_h0 | q_h0 | k_h1 | q_h1], 8 KB each; decayed in place
constexpr uint32_t kOffG = 32768;   // [g_h0 | g_h1]; C1 over rows 0..31 of each; then [P | Lbeta]
constexpr uint32_t kOffV = 49152;   // [v_h0 | v_h1] -> U~^T (bf16)
constexpr uint32_t kOffPlo = 2 * kStageBytes;   // P_lo [t][s]
constexpr uint32_t kOffC2 = kOffPlo + 8192;     // C2[2]: 2 halves x 64 rows each
constexpr uint32_t kOffNW = kOffC2 + 2 * 16384; // -W^T [c][t]
constexpr uint32_t kOffQP = kOffNW + 16384;     // Q'^T [c][t]
constexpr uint32_t kLdM = inv::kLdM;            // fp32 row stride of the A / L^{-1} buffer
constexpr uint32_t kOffM = kOffQP + 16384;      // A + L^{-1} (fp32)
constexpr uint32_t kOffMisc = kOffM + 64 * kLdM * 4;
constexpr uint32_t kOffBar = kOffMisc;          // kNumBars mbarriers
constexpr uint32_t kOffTmem = kOffMisc + 160;
constexpr uint32_t kOffAbort = kOffMisc + 164;
constexpr uint32_t kOffMdown = kOffMisc + 168;  // 2^-m of the state update [2] (fp32)
constexpr uint32_t kOffBeta = kOffMisc + 256;   // fp32 [2][64]
constexpr uint32_t kOffRk = kOffMisc + 768;     // fp32 [2][64]
constexpr uint32_t kOffRq = kOffMisc + 1280;    // fp32 [2][64]
constexpr uint32_t kOffQsum = kOffMisc + 1792;  // per-8-token-group decay sums [8][128]
constexpr uint32_t kOffE1 = kOffMisc + 5888;    // 2^rho1 [2][128]
constexpr uint32_t kOffE2 = kOffMisc + 6912;    // 2^rho2 [2][128]
constexpr uint32_t kOffF = kOffMisc + 7936;     // 2^(gam63-rho2) [2][128]
constexpr uint32_t kSmemUsed = kOffMisc + 8960;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffNW % 1024 == 0 && kOffC2 % 1024 == 0 && kOffPlo % 1024 == 0 &&
                  kOffM % 1024 == 0, "alignment");

// mbarrier slots
// kBarTma0 + s: stage s's tiles have landed; kBarPrep0 + s: the prep group has
// prepared the chunk in stage s; kBarGram: that chunk's Gram has completed.
// kBarK1Mma: the factor group's own MMA groups have completed (two commits, one
// per issuer); kBarWMma / kBarQMma: the W, U~ and the Q', O_intra MMA groups of a
// chunk have completed (for the state group, which takes part in their
// epilogues); kBarWDone / kBarQDone: the state group's part of those epilogues is
// written; kBarK1Ready: the chunk's -W^T and Q'^T tiles are complete.
// kBarMma1 / kBarMma2: the state group's output / state MMA has completed;
// kBarD1UFree: the U half of D1 has been read by the state group's U conversion
// (the next chunk's U~ may land there); kBarD1OFree: the O half has been stored by
// the prep group (the next chunk's O_intra may land there).
// kBarSlot0 + j: TMEM scratch slot j is free again (chunk c's use of slot c & 1
// ended); kBarSlotF0 + j: C2, e2 and f of parity j are free (the rescale of the
// chunk that used them is done).
constexpr int kNumBars = 19;
constexpr int kBarTma0 = 0, kBarPrep0 = 2, kBarK1Mma = 4, kBarK1Ready = 5, kBarMma1 = 6,
              kBarMma2 = 7, kBarD1UFree = 8, kBarSlot0 = 9, kBarSlotF0 = 11, kBarWMma = 13,
              kBarWDone = 14, kBarQMma = 15, kBarQDone = 16, kBarGram = 17, kBarD1OFree = 18;
static_assert(kNumBars * 8 <= 160, "mbarriers overlap the TMEM address slot");

// ---- TMEM columns ----------------------------------------------------------
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTD1 = 0;       // [U~^T | O_intra^T] then [U^T | O^T]   (128)
constexpr uint32_t kTState = 128;  // fp32 state S (pre-scaled around the state MMA) (128)
// S^T bf16 (A operand of the output MMA, 64 columns) and U^T bf16 hi / lo (A of
// the state MMA, 32 + 32) share these columns: S^T is dead once the output MMA
// has completed, U^T once the state MMA has, and each is rewritten only then.
constexpr uint32_t kTSA = 256, kTUA = 256, kTULA = 288;
// Two factor scratch slots of 96 columns, chunk c in slot c & 1: the Gram
// [C1 32 | C2 64], then the W^T halves [t < 32 part over all t: 64 | t >= 32: 32],
// then the Q'^T accumulator (64).  Chunk c + 1's Gram can land while chunk c
// still holds its slot.
constexpr uint32_t kTSlot = 320, kSlotCols = 96;

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f2(float2 x) { return pack_bf2(x.x, x.y); }
// sigmoid(x) = 1 / (1 + 2^(-x log2 e)) with hardware ex2 / rcp
__device__ __forceinline__ float sigmoid_fast(float x) {
  return rcp_approx(1.0f + ex2_approx(-x * kLog2e));
}

// Store 32 consecutive bf16 values into row `row` of a 128-byte-swizzled tile,
// starting at element e0 (multiple of 8).
__device__ __forceinline__ void store_row32_bf16(uint8_t* tile, int row, int e0,
                                                 const float (&x)[32]) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint4 w;
    w.x = pack_bf2(x[8 * ch + 0], x[8 * ch + 1]);
    w.y = pack_bf2(x[8 * ch + 2], x[8 * ch + 3]);
    w.z = pack_bf2(x[8 * ch + 4], x[8 * ch + 5]);
    w.w = pack_bf2(x[8 * ch + 6], x[8 * ch + 7]);
    *reinterpret_cast<uint4*>(tile + sw128(row, (e0 + 8 * ch) * 2)) = w;
  }
}

// Gram epilogue, k rows: A[r][j0 + j] = beta_r (K C^T)[r][j0 + j] as fp32 (whole
// 32-column pieces: entries on and above the diagonal are overwritten by the
// inverse before anything reads them).
__device__ __forceinline__ void a_row_out(const uint32_t (&u)[32], int j0, int r, float bb,
                                          float* M) {
  float4* dst = reinterpret_cast<float4*>(M + r * kLdM + j0);
  const float2 b2 = make_float2(bb, bb);
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float2 x = f2mul(b2, make_float2(__uint_as_float(u[j]), __uint_as_float(u[j + 1])));
    const float2 y = f2mul(b2, make_float2(__uint_as_float(u[j + 2]), __uint_as_float(u[j + 3])));
    dst[j >> 2] = make_float4(x.x, x.y, y.x, y.y);
  }
}
// Gram epilogue, q rows: P[r][j0 + j] as bf16 hi + lo tiles; entries with
// j > lim are zeroed (lim = r - j0 on the diagonal piece, else no limit).
__device__ __forceinline__ void p_row_out(const uint32_t (&u)[32], int j0, int r, int lim,
                                          uint8_t* p_hi, uint8_t* p_lo) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    float x[8];
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (8 * ch + e <= lim) ? __uint_as_float(u[8 * ch + e]) : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hi[e] = pack_bf2(x[2 * e], x[2 * e + 1]);
      lo[e] = pack_bf2(x[2 * e] - bf_lo(hi[e]), x[2 * e + 1] - bf_hi(hi[e]));
    }
    const uint32_t off = sw128(r, (j0 + 8 * ch) * 2);
    *reinterpret_cast<uint4*>(p_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(p_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Same, from fp32 bit patterns.
__device__ __forceinline__ void store_row32_bits(uint8_t* tile, int row, int e0,
                                                 const uint32_t (&u)[32]) {
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    uint4 w;
    w.x = pack_bf2(__uint_as_float(u[8 * ch + 0]), __uint_as_float(u[8 * ch + 1]));
    w.y = pack_bf2(__uint_as_float(u[8 * ch + 2]), __uint_as_float(u[8 * ch + 3]));
    w.z = pack_bf2(__uint_as_float(u[8 * ch + 4]), __uint_as_float(u[8 * ch + 5]));
    w.w = pack_bf2(__uint_as_float(u[8 * ch + 6]), __uint_as_float(u[8 * ch + 7]));
    *reinterpret_cast<uint4*>(tile + sw128(row, (e0 + 8 * ch) * 2)) = w;
  }
}

__device__ __forceinline__ void store_row16_bits(uint8_t* tile, int row, int e0,
                                                 const uint32_t (&u)[16]) {
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    uint4 w;
    w.x = pack_bf2(__uint_as_float(u[8 * ch + 0]), __uint_as_float(u[8 * ch + 1]));
    w.y = pack_bf2(__uint_as_float(u[8 * ch + 2]), __uint_as_float(u[8 * ch + 3]));
    w.z = pack_bf2(__uint_as_float(u[8 * ch + 4]), __uint_as_float(u[8 * ch + 5]));
    w.w = pack_bf2(__uint_as_float(u[8 * ch + 6]), __uint_as_float(u[8 * ch + 7]));
    *reinterpret_cast<uint4*>(tile + sw128(row, (e0 + 8 * ch) * 2)) = w;
  }
}

// Gate of one channel pair, log2 units: lb2 sigmoid(exp(A_log)(g + dt_bias)) =
// lb2 / (1 + 2^(nea g + ndb)), from the pair's raw gate values.
__device__ __forceinline__ float2 gate_pair_f(float2 gx, float2 nea2, float2 ndb2, float2 lb22) {
  const float2 z = f2fma(nea2, gx, ndb2);
  const float2 d = f2add(make_float2(1.f, 1.f), make_float2(ex2_approx(z.x), ex2_approx(z.y)));
  return f2mul(lb22, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}
// Same, from the pair's packed bf16 g word.
__device__ __forceinline__ float2 gate_pair(uint32_t gv, float2 nea2, float2 ndb2, float2 lb22) {
  return gate_pair_f(make_float2(bf_lo(gv), bf_hi(gv)), nea2, ndb2, lb22);
}
struct Shared {
  uint8_t* sm;
  uint64_t* bar;
  volatile int* abort;
};

// Slow path of wait_bar, out of line so the many wait sites share one copy.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           unsigned* status) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    // suspended, not spinning, while the phase is incomplete
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitNs) {
      *abort = 1;
      atomicOr(status, kDevStatusTimeout);
      return false;
    }
  }
}

// Bounded mbarrier wait that also gives up as soon as another thread aborted.
__device__ __forceinline__ bool wait_bar(const Shared& S, int idx, uint32_t parity,
                                         unsigned* status) {
  uint64_t* bar = &S.bar[idx];
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, S.abort, status);
}

// Pull one chunk's q/k/v/g tiles into L2 so the later tiled load (or, for an
// fp32 gate, the prep group's plain loads) hits L2.  hk: q/k head; h: value head.
template <bool kGateF32>
__device__ __forceinline__ void prefetch_chunk_l2(const CUtensorMap* tq, const CUtensorMap* tk,
                                                  const CUtensorMap* tv, const CUtensorMap* tg,
                                                  int h, int hk, int64_t tok0) {
  const int32_t t32 = (int32_t)tok0;
#pragma unroll
  for (int c0 = 0; c0 < 128; c0 += 64) {
    tma_prefetch_3d(tk, c0, hk, t32);
    tma_prefetch_3d(tq, c0, hk, t32);
    if (!kGateF32) tma_prefetch_3d(tg, c0, h, t32);
    tma_prefetch_3d(tv, c0, h, t32);
  }
  if (kGateF32) tma_prefetch_3d(tg, 0, h, t32);  // one box covers all 128 channels
}

// q/k (head hk), g and v (value head h) tiles of one chunk into stage `st`; an
// fp32 gate is not staged (the prep group reads it from L2).
template <bool kGateF32>
__device__ __forceinline__ void issue_chunk_loads(uint8_t* st, uint64_t* bar, const CUtensorMap* tq,
                                                  const CUtensorMap* tk, const CUtensorMap* tv,
                                                  const CUtensorMap* tg, int h, int hk,
                                                  int64_t tok0, bool load_v = true) {
  mbar_arrive_expect_tx(bar, 32768u + (kGateF32 ? 0u : 16384u) + (load_v ? 16384u : 0u));
  const int32_t t32 = (int32_t)tok0;
  tma_load_3d(st + kOffQK + 0, tk, bar, 0, hk, t32);
  tma_load_3d(st + kOffQK + 8192, tq, bar, 0, hk, t32);
  tma_load_3d(st + kOffQK + 16384, tk, bar, 64, hk, t32);
  tma_load_3d(st + kOffQK + 24576, tq, bar, 64, hk, t32);
  if (!kGateF32) {
    tma_load_3d(st + kOffG + 0, tg, bar, 0, h, t32);
    tma_load_3d(st + kOffG + 8192, tg, bar, 64, h, t32);
  }
  if (load_v) {
    tma_load_3d(st + kOffV + 0, tv, bar, 0, h, t32);
    tma_load_3d(st + kOffV + 8192, tv, bar, 64, h, t32);
  }
}


// Rq[t][k] of rows t = t0 .. t0 + 31 (bf16 pairs, t0 + 2i in the low half of
// r[i]) for channel k = row, from the decayed q tile of stage `st`.  A warp reads
// 64 consecutive bytes of one row per step (conflict free).
__device__ __forceinline__ void load_rq_col(const uint8_t* st, int row, int t0, uint32_t (&r)[16]) {
  const uint8_t* base = st + kOffQK + (row >> 6) * 16384 + 8192;
  const uint32_t cbyte = 2u * (uint32_t)(row & 63);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t lo = *reinterpret_cast<const uint16_t*>(base + sw128(t0 + 2 * i, cbyte));
    const uint32_t hi = *reinterpret_cast<const uint16_t*>(base + sw128(t0 + 2 * i + 1, cbyte));
    r[i] = lo | (hi << 16);
  }
}

// Q'^T row (32 columns) = acc + e Rq^T -> QP tile, columns c0 .. c0 + 31.
__device__ __forceinline__ void qprime_store(uint8_t* qp, int row, int c0, const uint32_t (&acc)[32],
                                             const uint32_t (&rq)[16], float e) {
  float x[32];
  const float2 e2 = make_float2(e, e);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 v = f2fma(make_float2(bf_lo(rq[j]), bf_hi(rq[j])), e2,
                           make_float2(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1])));
    x[2 * j] = v.x;
    x[2 * j + 1] = v.y;
  }
  store_row32_bf16(qp, row, c0, x);
}

// Gram of one chunk into a scratch slot: D[i][col] = R[i] . [C1 | C2][col] over the
// 128 rows [R_k; R_q] (stage st), C1 columns 0..31 (rows t < 32 of the g area) and
// C2 columns 32..95; issued by one thread, completion on `bar`.
__device__ __forceinline__ void issue_gram(uint32_t slot, const uint8_t* st, const uint8_t* c2,
                                           uint64_t* bar) {
  // descriptors advance by (byte offset >> 4) in their address field
  const uint64_t dA = sw128_desc(smem_u32(st + kOffQK), 16, 1024);
  const uint64_t dB1 = sw128_desc(smem_u32(st + kOffG), 16, 1024), dB2 = sw128_desc(smem_u32(c2), 16, 1024);
  const uint32_t id1 = idesc_bf16_f32(128, 32, 0, 0), id2 = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll 1
  for (int j = 0; j < 8; ++j) {
    const uint32_t oa = (j >> 2) * 1024 + (j & 3) * 2, ob = (j >> 2) * 512 + (j & 3) * 2;
    mma_bf16_ss(slot, dA + oa, dB1 + ob, id1, j > 0);
    mma_bf16_ss(slot + 32, dA + oa, dB2 + ob, id2, j > 0);
  }
  mma_commit(bar);
}

}  // namespace

template <bool kGateF32>
__global__ void __launch_bounds__(kThreads, 1)
    kda_chunk_fwd_kernel(const __grid_constant__ CUtensorMap tq,
                         const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv,
                         const __grid_constant__ CUtensorMap tg, const ChunkFwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* const sm = smem_align1024(smem_raw);
  Shared S;
  S.sm = sm;
  S.bar = reinterpret_cast<uint64_t*>(sm + kOffBar);
  S.abort = reinterpret_cast<volatile int*>(sm + kOffAbort);
  const int tid = threadIdx.x, warp = tid >> 5;

  const int H = p.H;
  // ---- which unit this CTA runs (CTA-uniform)
  Unit U;
  U.seg = 0;
  U.nseg = 1;
  U.L = 0;
  U.kind = kUnitSerial;
  U.slot_base = 0;
  if (p.trans_M) {
    // transition mode: whole sequences, block 2u runs unit u from the identity
    // with v = 0 (its final state is M), block 2u + 1 from zero (B)
    const int u = (int)blockIdx.x >> 1;
    U.n = u / H;
    U.h = u % H;
    U.kind = (blockIdx.x & 1) ? kUnitPreB : kUnitPreM;
    U.L = 0x7FFFFFFF / kChunk;
  } else if (p.hdr) {
    if (!p.hdr->plan_ok) return;
    if ((int)blockIdx.x < p.unsplit_base) {
      const int cnt = p.prescan ? p.hdr->n_pre_units : p.hdr->n_seg_units;
      if ((int)blockIdx.x >= cnt) return;
      U = p.units[blockIdx.x];
    } else {
      const int u = (int)blockIdx.x - p.unsplit_base;
      U.n = p.order[u / H];
      U.h = u % H;
      if (p.seq_info[4 * U.n] > 1) return;  // split: run as segments
    }
  } else {
    U.n = (int)blockIdx.x / H;
    U.h = (int)blockIdx.x % H;
  }
  const int n = U.n, h = U.h;
  const int hk = h / p.qk_group;  // q/k head of value head h
  int64_t bos, eos;
  if (p.cu_seqlens) {
    bos = p.cu_seqlens[n];
    eos = p.cu_seqlens[n + 1];
  } else {
    bos = (int64_t)n * p.seq_len;
    eos = bos + p.seq_len;
  }
  // A unit whose bounds leave [0, T_total] (or run backwards) is skipped and
  // reported: every unit checking its own pair validates the whole prefix sum.
  if (bos < 0 || eos < bos || eos > p.total_tokens || (p.cu_seqlens && n == 0 && bos != 0) ||
      (p.cu_seqlens && n == p.N - 1 && eos != p.total_tokens)) {
    if (tid == 0) atomicOr(p.status, kDevStatusBadSeqlens);
    return;
  }
  if (U.kind != kUnitSerial) {  // one segment of a split sequence
    const int64_t sb = bos + (int64_t)U.seg * U.L * kChunk;
    eos = (sb + (int64_t)U.L * kChunk) < eos ? (sb + (int64_t)U.L * kChunk) : eos;
    bos = sb;
  }
  const int64_t len = eos - bos;
  const int nchunks = (int)((len + kChunk - 1) / kChunk);
  // initial state, final state, outputs and values for this unit
  constexpr int64_t kSlotElems = (int64_t)kHeadDim * kHeadDim;
  const int64_t user_off = ((int64_t)n * H + h) * kSlotElems;
  const void* init_ptr = nullptr;
  bool init_bf16 = false, init_identity = false;
  void* fin_ptr = nullptr;
  bool fin_bf16 = false;
  // segment 0 of a split sequence starts from the true initial state, so its
  // prescan unit writes the outputs; transition / offset units write none and
  // skip the work that only serves the outputs (Q', O_intra, the O half)
  const bool write_out =
      (U.kind == kUnitSerial || U.kind == kUnitRerun || U.kind == kUnitPreS1) && !p.no_out;
  // bf16 chunk start states for the backward, slot bos / 64 + 2 n + c of the
  // sequence's chunk c: written by every unit whose chunks produce outputs (a
  // whole sequence, or a segment: bos is then the segment's first token, a whole
  // number of chunks after the sequence's)
  uint16_t* const ck_unit =
      (p.ckpt_out && (U.kind == kUnitSerial || U.kind == kUnitRerun || U.kind == kUnitPreS1))
          ? p.ckpt_out + ((bos / kChunk + 2 * (int64_t)n) * H + h) * kSlotElems
          : nullptr;
  const bool zero_v = (U.kind == kUnitPreM);
  const bool first_seg = (U.kind == kUnitSerial || U.kind == kUnitPreS1 ||
                          (U.kind == kUnitRerun && U.seg == 0));
  if (first_seg) {
    if (p.init_state) {
      init_ptr = p.state_bf16
                     ? (const void*)(static_cast<const uint16_t*>(p.init_state) + user_off)
                     : (const void*)(static_cast<const float*>(p.init_state) + user_off);
      init_bf16 = p.state_bf16 != 0;
    }
  } else if (U.kind == kUnitRerun) {
    init_ptr = p.slots + (int64_t)slot_S(U, U.seg) * kSlotElems;
  } else if (U.kind == kUnitPreM) {
    init_identity = true;
  }
  if (U.kind == kUnitSerial || (U.kind == kUnitRerun && U.seg == U.nseg - 1)) {
    if (p.final_state) {
      fin_ptr = p.state_bf16 ? (void*)(static_cast<uint16_t*>(p.final_state) + user_off)
                             : (void*)(static_cast<float*>(p.final_state) + user_off);
      fin_bf16 = p.state_bf16 != 0;
    }
  } else if (p.trans_M) {
    fin_ptr = (U.kind == kUnitPreM ? p.trans_M : p.trans_B) + user_off;
  } else if (U.kind == kUnitPreS1) {
    fin_ptr = p.slots + (int64_t)slot_S(U, 1) * kSlotElems;
  } else if (U.kind == kUnitPreM) {
    fin_ptr = p.slots + (int64_t)slot_M(U, U.seg) * kSlotElems;
  } else if (U.kind == kUnitPreB) {
    fin_ptr = p.slots + (int64_t)slot_S(U, U.seg + 1) * kSlotElems;
  }

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(&S.bar[i], (i == kBarK1Mma || i == kBarWMma || i == kBarQMma) ? 2u : 1u);
    *S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(reinterpret_cast<uint32_t*>(sm + kOffTmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sm + kOffTmem);
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

  if (warp >= 8) {
    // =====================================================================
    // prep group: gate, decay, norms and decayed operands of chunk c.  Thread
    // = (token group qt of 8 tokens, channel quad cq): 4 channels x 8 tokens,
    // 8-byte shared-memory accesses; the swizzle of a row is fixed by its index
    // inside the group (t & 7 = i), so every address is known per thread.
    // =====================================================================
    const int ptid = tid - 256;
    const bool leader = (ptid == 0);
    const int cq = ptid & 31, qt = ptid >> 5;   // channel quad, token group
    const int c0 = 4 * cq, hh = c0 >> 6, cb = (c0 & 63) * 2;
    const float nea = -expf(p.A_log[h]) * kLog2e;  // -exp(A_log) log2(e)
    const float* dtb = p.dt_bias + h * kHeadDim + c0;
    const float2 nea2 = make_float2(nea, nea), lb22 = make_float2(p.lower_bound * kLog2e,
                                                                 p.lower_bound * kLog2e);
    const float2 ndbA = make_float2(nea * dtb[0], nea * dtb[1]);
    const float2 ndbB = make_float2(nea * dtb[2], nea * dtb[3]);
    // byte offset of row qt * 8 + i, channels c0 .. c0 + 3, in a 128-byte-swizzled tile
    auto rowoff = [&](int i) -> uint32_t {
      return (uint32_t)(qt * 8 + i) * 128u + ((((uint32_t)cb >> 4) ^ (uint32_t)i) << 4) +
             ((uint32_t)cb & 15u);
    };
    float* const s_qsum = reinterpret_cast<float*>(sm + kOffQsum);
    // raw beta of token ptid of the chunk being prepared (threads ptid < 64),
    // loaded one chunk ahead so its global-memory latency is hidden
    uint16_t beta_raw = 0;
    if (ptid < 64 && ptid < eos - bos) beta_raw = p.beta[(bos + ptid) * H + h];
    // O of chunk cc -> global, from the O half of D1 once the state group's output
    // MMA of cc has completed; then that half is released (kBarD1OFree).  Warps 8-11
    // take tokens 0..31, warps 12-15 tokens 32..63; lanes are consecutive value
    // channels, and lane pairs swap halves so that the even lane writes channels
    // (v, v + 1) of token 2j and the odd lane channels (v - 1, v) of token 2j + 1
    // (4-byte stores).  false: a wait gave up.
    const int orow = 32 * (warp & 3) + (tid & 31);
    const uint32_t olane = (uint32_t)(32 * (warp & 3)) << 16;
    const int oth = (warp - 8) >> 2;
    auto store_o = [&](int cc) -> bool {
      bool okw = true;
      if (leader) okw = wait_bar(S, kBarMma1, (uint32_t)(cc & 1), p.status);
      if (named_sync_or(kBarP, kPrepThreads, !okw)) return false;
      tc_fence_after();
      const int64_t t0c = bos + (int64_t)cc * kChunk;
      const int lenc = (int)((eos - t0c) < kChunk ? (eos - t0c) : kChunk);
      const bool odd = (orow & 1) != 0;
      const uint32_t sel = odd ? 0x3276u : 0x5410u;
      uint32_t* op = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) +
                                                 (t0c * H + h) * kHeadDim + (orow & ~1) +
                                                 (odd ? (int64_t)H * kHeadDim : 0));
      const int64_t tstride2 = (int64_t)H * kHeadDim;  // two tokens, in 4-byte words
      const int jmax = (lenc - (odd ? 1 : 0) + 1) >> 1;  // tokens 2j (+1) < lenc
      const float2 sc2 = make_float2(p.scale, p.scale);
#pragma unroll 1
      for (int q4 = 0; q4 < 2; ++q4) {
        uint32_t a[16];
        tmem_ld16(tbase + kTD1 + olane + 64 + 32 * oth + 16 * q4, a);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 o = f2mul(sc2, make_float2(__uint_as_float(a[2 * j]), __uint_as_float(a[2 * j + 1])));
          const uint32_t w = pack_bf2(o.x, o.y);
          const uint32_t x = __shfl_xor_sync(0xffffffffu, w, 1);
          const int jj = 16 * oth + 8 * q4 + j;
          if (jj < jmax) op[jj * tstride2] = __byte_perm(w, x, sel);
        }
      }
      tc_fence_before();
      named_sync(kBarP, kPrepThreads);
      if (leader) mbar_arrive(&S.bar[kBarD1OFree]);
      return true;
    };

#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      uint8_t* const st = sm + s * kStageBytes;
      uint8_t* const kq = st + kOffQK + hh * 16384;    // k rows; q rows at + 8192
      uint8_t* const gq = st + kOffG + hh * 8192;      // g rows, then C1 (rows < 32)
      uint8_t* const c2h = sm + kOffC2 + s * 16384 + hh * 8192;
      float* const s_beta = reinterpret_cast<float*>(sm + kOffBeta) + s * 64;
      float* const s_rk = reinterpret_cast<float*>(sm + kOffRk) + s * 64;
      float* const s_rq = reinterpret_cast<float*>(sm + kOffRq) + s * 64;
      float* const s_e1 = reinterpret_cast<float*>(sm + kOffE1) + s * 128;
      float* const s_e2 = reinterpret_cast<float*>(sm + kOffE2) + s * 128;
      float* const s_f = reinterpret_cast<float*>(sm + kOffF) + s * 128;
      const int64_t tok0 = bos + (int64_t)c * kChunk;
      const int clen = (int)((eos - tok0) < kChunk ? (eos - tok0) : kChunk);

      bool ok = wait_bar(S, kBarTma0 + s, (uint32_t)((c >> 1) & 1), p.status);
      if (named_sync_or(kBarP, kPrepThreads, !ok)) break;

      if (zero_v) {  // transition prescan: the values are zero
        uint4* vt = reinterpret_cast<uint4*>(st + kOffV);
#pragma unroll
        for (int i = 0; i < 4; ++i) vt[ptid + 256 * i] = make_uint4(0u, 0u, 0u, 0u);
      }
      // ---- beta (this chunk's, loaded last chunk) and the next chunk's raw beta
      if (ptid < 64) {
        s_beta[ptid] = (ptid < clen) ? sigmoid_fast(__uint_as_float((uint32_t)beta_raw << 16)) : 0.f;
        const int64_t tn = tok0 + kChunk + ptid;
        beta_raw = (tn < eos) ? p.beta[tn * H + h] : (uint16_t)0;
      }
      // ---- reciprocal row norms (two threads per row: k rows, then q rows); four
      // packed accumulators keep the dependent chains short
      {
        const int r = ptid >> 1, half = ptid & 1, t = r & 63;
        const uint8_t* rp = st + kOffQK + half * 16384 + (r < 64 ? 0 : 8192) + t * 128;
        float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 w = *reinterpret_cast<const uint4*>(rp + 16 * (j ^ (t & 7)));
          const float2 x0 = make_float2(bf_lo(w.x), bf_hi(w.x)), x1 = make_float2(bf_lo(w.y), bf_hi(w.y));
          const float2 x2 = make_float2(bf_lo(w.z), bf_hi(w.z)), x3 = make_float2(bf_lo(w.w), bf_hi(w.w));
          a0 = f2fma(x0, x0, a0);
          a1 = f2fma(x1, x1, a1);
          a2 = f2fma(x2, x2, a2);
          a3 = f2fma(x3, x3, a3);
        }
        const float2 b = f2add(f2add(a0, a1), f2add(a2, a3));
        float ss = b.x + b.y;
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        const float rs = (t < clen) ? rsqrtf(ss + 1e-6f) : 0.f;
        if (half == 0) (r < 64 ? s_rk : s_rq)[t] = rs;
      }

      // ---- gate pairs (log2 units) of the thread's 8 tokens x 4 channels, kept in
      // registers for the operand pass; tokens past the sequence end count 0
      float2 lgA[8], lgB[8];  // channels c0, c0 + 1 / c0 + 2, c0 + 3
      if constexpr (kGateF32) {  // all 8 loads in flight before the first use
        float4 gx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          gx[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (qt * 8 + i < clen)
            gx[i] = __ldg(reinterpret_cast<const float4*>(
                p.g32 + ((tok0 + qt * 8 + i) * H + h) * kHeadDim + c0));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          lgA[i] = gate_pair_f(make_float2(gx[i].x, gx[i].y), nea2, ndbA, lb22);
          lgB[i] = gate_pair_f(make_float2(gx[i].z, gx[i].w), nea2, ndbB, lb22);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint2 w = *reinterpret_cast<const uint2*>(gq + rowoff(i));
          lgA[i] = gate_pair(w.x, nea2, ndbA, lb22);
          lgB[i] = gate_pair(w.y, nea2, ndbB, lb22);
        }
      }
      if (clen < kChunk) {  // ragged last chunk (cold path)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (qt * 8 + i >= clen) lgA[i] = lgB[i] = make_float2(0.f, 0.f);
      }
      float2 runA = lgA[0], runB = lgB[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) {
        runA = f2add(runA, lgA[i]);
        runB = f2add(runB, lgB[i]);
      }
      *reinterpret_cast<float4*>(s_qsum + qt * 128 + c0) = make_float4(runA.x, runA.y, runB.x, runB.y);
      named_sync(kBarP, kPrepThreads);
      // group sums left to right: offset of this group, rho1 (after group 1), rho2
      // (after group 5) and gam63 (after group 7), all in the same order
      float4 sum = *reinterpret_cast<const float4*>(s_qsum + c0), off = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 r1 = sum, r2 = sum;
#pragma unroll
      for (int q = 1; q < 8; ++q) {
        if (q == qt) off = sum;
        const float4 x = *reinterpret_cast<const float4*>(s_qsum + q * 128 + c0);
        sum = make_float4(sum.x + x.x, sum.y + x.y, sum.z + x.z, sum.w + x.w);
        if (q == 1) r1 = sum;
        if (q == 5) r2 = sum;
      }
      // sum is now gam63 (decay to the chunk's last token, per channel)
      const float4 rho = qt < 4 ? r1 : r2;

      // ---- decayed bf16 operands (fp32 products, one rounding each), in place; C1 (rows
      // t < 32) over this thread's own g words, which it has read already.  The C2
      // words wait in registers until the state MMA of chunk c-2 has released C2[s].
      // a = gam_t - rho runs from (offset - rho); C2 of rows t < 32 uses
      // rho2 - gam_t = -(a + rho1 - rho2) in one exponent (factoring it through
      // 2^(rho2 - rho1) would underflow while the product is still significant).
      uint2 c2w[8];
      {
        float2 aA = make_float2(off.x - rho.x, off.y - rho.y), aB = make_float2(off.z - rho.z, off.w - rho.w);
        const float2 dA = make_float2(r1.x - r2.x, r1.y - r2.y), dB = make_float2(r1.z - r2.z, r1.w - r2.w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = qt * 8 + i;
          const uint32_t ro = rowoff(i);
          aA = f2add(aA, lgA[i]);
          aB = f2add(aB, lgB[i]);
          const float2 EA = make_float2(ex2_approx(aA.x), ex2_approx(aA.y));
          const float2 EB = make_float2(ex2_approx(aB.x), ex2_approx(aB.y));
          const float2 IA = make_float2(ex2_approx(-aA.x), ex2_approx(-aA.y));
          const float2 IB = make_float2(ex2_approx(-aB.x), ex2_approx(-aB.y));
          const float rk = s_rk[t], rq = s_rq[t];
          const float2 rk2 = make_float2(rk, rk), rq2 = make_float2(rq, rq);
          uint2* kp = reinterpret_cast<uint2*>(kq + ro);
          uint2* qp = reinterpret_cast<uint2*>(kq + 8192 + ro);
          const uint2 kv = *kp, qv = *qp;
          // the normalized rows in fp32, then one bf16 rounding per decayed operand
          const float2 kA0 = f2mul(rk2, make_float2(bf_lo(kv.x), bf_hi(kv.x)));
          const float2 kB0 = f2mul(rk2, make_float2(bf_lo(kv.y), bf_hi(kv.y)));
          const float2 qA0 = f2mul(rq2, make_float2(bf_lo(qv.x), bf_hi(qv.x)));
          const float2 qB0 = f2mul(rq2, make_float2(bf_lo(qv.y), bf_hi(qv.y)));
          *kp = make_uint2(pack_f2(f2mul(kA0, EA)), pack_f2(f2mul(kB0, EB)));
          *qp = make_uint2(pack_f2(f2mul(qA0, EA)), pack_f2(f2mul(qB0, EB)));
          const uint2 ck = make_uint2(pack_f2(f2mul(kA0, IA)), pack_f2(f2mul(kB0, IB)));
          if (qt < 4) {
            *reinterpret_cast<uint2*>(gq + ro) = ck;  // C1
            const float2 gA = f2add(aA, dA), gB = f2add(aB, dB);
            c2w[i] = make_uint2(
                pack_f2(f2mul(kA0, make_float2(ex2_approx(-gA.x), ex2_approx(-gA.y)))),
                pack_f2(f2mul(kB0, make_float2(ex2_approx(-gB.x), ex2_approx(-gB.y)))));
          } else {
            c2w[i] = ck;
          }
        }
        if (clen < kChunk) {  // rows past the sequence end are zero operands (cold path)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (qt * 8 + i >= clen) {
              const uint32_t ro = rowoff(i);
              *reinterpret_cast<uint2*>(kq + ro) = make_uint2(0u, 0u);
              *reinterpret_cast<uint2*>(kq + 8192 + ro) = make_uint2(0u, 0u);
              if (qt < 4) *reinterpret_cast<uint2*>(gq + ro) = make_uint2(0u, 0u);
              *reinterpret_cast<uint2*>(st + kOffV + hh * 8192 + ro) = make_uint2(0u, 0u);
              c2w[i] = make_uint2(0u, 0u);
            }
          }
        }
      }
      // Overflow guard of the state update.  Its MMA accumulates 2^rho2 S + U^T C2,
      // and the C2 factors reach 2^(rho2 - gam63) per channel (up to 2^115 at
      // lower_bound = -5), so large values would overflow fp32 there.  Where that
      // factor exceeds 2^kShiftFree on some channel, the update is accumulated
      // at 2^-m scale, m = ceil(max_c(rho2 - gam63)) - kShiftFree: U and the
      // pre-scale are multiplied by 2^-m and the post-scale f by 2^m.  Powers of
      // two, so nothing changes but the exponent range (m = 0: the same bits).
      // Warp 7 of the group holds every channel's gam63.
      int m = 0;
      if (qt == 7) {
        const float d = fmaxf(fmaxf(r2.x - sum.x, r2.y - sum.y), fmaxf(r2.z - sum.z, r2.w - sum.w));
        m = (int)__reduce_max_sync(0xffffffffu, (unsigned)max(0, (int)ceilf(d) - kShiftFree));
      }
      // O of chunk c - 2 (the prep group runs two chunks ahead of the state group,
      // whose output MMA of that chunk has run by now)
      if (write_out && c >= 2 && !store_o(c - 2)) break;
      // the state group's rescale of chunk c-2 (after its state MMA) is done: C2[s],
      // e2[s] and f[s] are free
      ok = true;
      if (leader && c >= 2) ok = wait_bar(S, kBarSlotF0 + s, (uint32_t)(((c >> 1) - 1) & 1), p.status);
      if (named_sync_or(kBarP, kPrepThreads, !ok)) break;
#pragma unroll
      for (int i = 0; i < 8; ++i) *reinterpret_cast<uint2*>(c2h + rowoff(i)) = c2w[i];
      if (qt == 7) {  // 0 <= m <= 52
        const float up = __int_as_float((127 + m) << 23);  // 2^m
        *reinterpret_cast<float4*>(s_f + c0) =
            make_float4(ex2_approx(sum.x - r2.x) * up, ex2_approx(sum.y - r2.y) * up,
                        ex2_approx(sum.z - r2.z) * up, ex2_approx(sum.w - r2.w) * up);
        *reinterpret_cast<float4*>(s_e1 + c0) =
            make_float4(ex2_approx(r1.x), ex2_approx(r1.y), ex2_approx(r1.z), ex2_approx(r1.w));
        *reinterpret_cast<float4*>(s_e2 + c0) =
            make_float4(ex2_approx(r2.x), ex2_approx(r2.y), ex2_approx(r2.z), ex2_approx(r2.w));
        if (cq == 0) reinterpret_cast<float*>(sm + kOffMdown)[s] = __int_as_float((127 - m) << 23);
      }
      fence_proxy_async();
      named_sync(kBarP, kPrepThreads);
      // the Gram's issuer is on sub-partition 3 (warp 11; see the factor group)
      if (ptid == 96 && !p.debug_stall) {  // (timeout test: never)
        mbar_arrive(&S.bar[kBarPrep0 + s]);
        // this chunk's Gram, into scratch slot s once chunk c - 2 has released it,
        // so that the factor group finds it done when it takes up chunk c
        const bool okg = c < 2 || wait_bar(S, kBarSlot0 + s, (uint32_t)(((c >> 1) - 1) & 1), p.status);
        if (okg) {
          tc_fence_after();
          issue_gram(tbase + kTSlot + kSlotCols * (uint32_t)s, st, sm + kOffC2 + s * 16384,
                     &S.bar[kBarGram]);
        }
      }
    }
    // O of the last two chunks (unless a wait gave up)
    if (write_out && !named_sync_or(kBarP, kPrepThreads, *S.abort != 0)) {
#pragma unroll 1
      for (int cc = nchunks >= 2 ? nchunks - 2 : 0; cc < nchunks; ++cc)
        if (!store_o(cc)) break;
    }
  } else if (warp >= 4) {
    // =====================================================================
    // factor group: Gram, inverse, W, U~, Q', O_intra of chunk c
    // =====================================================================
    const int ftid = tid - 128;
    const int row = ftid;                 // TMEM lane owned by this thread
    const bool leader = (ftid == 0);
    // The two MMA-issuing threads sit on sub-partitions 2 and 1 (warps 6 and 5):
    // a tcgen05.mma issue slows down several-fold while other warps of its
    // sub-partition keep the FMA pipe busy, so the issuers of the three groups
    // (state: warp 0, prep: warp 11, factor: warps 5 and 6) each get their own.
    const bool issuer1 = (ftid == 64), issuer2 = (ftid == 32), issuer = issuer1 || issuer2;
    float* const M = reinterpret_cast<float*>(sm + kOffM);
    const uint32_t tD1 = tbase + kTD1;
    uint32_t k1ph = 0;

    if (leader) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tg);
      if (nchunks > 0)
        issue_chunk_loads<kGateF32>(sm, &S.bar[kBarTma0], &tq, &tk, &tv, &tg, h, hk, bos, !zero_v);
      if (nchunks > 1)
        issue_chunk_loads<kGateF32>(sm + kStageBytes, &S.bar[kBarTma0 + 1], &tq, &tk, &tv, &tg,
                                    h, hk, bos + kChunk, !zero_v);
      for (int c = 2; c < 4 && c < nchunks; ++c)
        prefetch_chunk_l2<kGateF32>(&tq, &tk, &tv, &tg, h, hk, bos + (int64_t)c * kChunk);
    }

#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      uint8_t* const st = sm + s * kStageBytes;
      const float* s_beta = reinterpret_cast<const float*>(sm + kOffBeta) + s * 64;
      const float* s_e1 = reinterpret_cast<const float*>(sm + kOffE1) + s * 128;
      const float* s_e2 = reinterpret_cast<const float*>(sm + kOffE2) + s * 128;
      const uint32_t tScr = tbase + kTSlot + kSlotCols * (uint32_t)s;  // scratch slot of chunk c

      // the prep group has prepared chunk c and issued its Gram into slot s
      bool ok = wait_bar(S, kBarPrep0 + s, (uint32_t)((c >> 1) & 1), p.status);
      if (ok) ok = wait_bar(S, kBarGram, (uint32_t)(c & 1), p.status);
      if (named_sync_or(kBarF, kSubThreads, !ok)) break;
      tc_fence_after();

      // ---- warps 4-5: A (fp32, strict lower, x beta_r), then level 0 of the inverse;
      //      warps 6-7 meanwhile: P (bf16 hi + lo, lower incl.).  Rows t < 32 use
      //      the C1 columns (0..31), rows t >= 32 the C2 columns (32..95).  Blocks
      //      strictly above the diagonal are never read and are not written.
      {
        const int r = row & 63;
        const bool lowrow = (warp & 1) == 0;  // r < 32
        const int nhalf = lowrow ? 1 : 2;
        const uint32_t col0 = tScr + lane_base + (lowrow ? 0u : 32u);
        if (row < 64) {
          const float bb = s_beta[r];
#pragma unroll 1
          for (int hh = 0; hh < nhalf; ++hh) {
            uint32_t u[32];
            tmem_ld32(col0 + 32 * hh, u);
            tmem_wait_ld();
            a_row_out(u, 32 * hh, r, bb, M);
          }
          tc_fence_before();
          named_sync(kBarF0, 64);
          inv::inverse_level0(M, ftid);
        } else {
#pragma unroll 1
          for (int hh = 0; hh < nhalf; ++hh) {
            uint32_t u[32];
            tmem_ld32(col0 + 32 * hh, u);
            tmem_wait_ld();
            // the diagonal piece is the first half for rows < 32, the second above
            const int lim = (hh == nhalf - 1) ? r - 32 * hh : 64;
            p_row_out(u, 32 * hh, r, lim, st + kOffG, sm + kOffPlo);
          }
          tc_fence_before();
        }
      }
      named_sync(kBarF, kSubThreads);

      // ---- Lbeta[t][s] = L^{-1}[t][s] beta_s (bf16)
      inv::lbeta_inverse(M, st + kOffG + 8192, s_beta, ftid);
      fence_proxy_async();
      named_sync(kBarF, kSubThreads);

      // ---- W^T halves (first issuer) and U~^T (second issuer, once the U half of D1
      // is free of the previous chunk)
      ok = true;
      if (issuer2 && c >= 1) ok = wait_bar(S, kBarD1UFree, (uint32_t)((c - 1) & 1), p.status);
      if (issuer && ok) {
        tc_fence_after();
        const uint32_t lbt = smem_u32(st + kOffG + 8192);
        // K-step j (s = 16j..16j+15) only meets rows t >= 16j of Lbeta (the rest is
        // zero): N = 64 - 16j rows from t = 16j, written from D column 16j on.
        // The second W^T half therefore holds columns t >= 32 only.
        // K-step j: A + 2048 j bytes, B (Lbeta rows from 16j, columns 16j..) + 2080 j,
        // N = 64 - 16j (the N / 8 field of the instruction descriptor drops by 2)
        const uint64_t dB = sw128_desc(lbt, 16, 1024);
        const uint32_t id0 = idesc_bf16_f32(128, 64, 1, 0);
        if (issuer1) {
          const uint64_t dA = sw128_desc(smem_u32(st + kOffQK), 16384, 1024);
#pragma unroll 1
          for (int j = 0; j < 4; ++j)
            mma_bf16_ss(tScr + 16 * j + (j >= 2 ? 32 : 0), dA + 128 * j, dB + 130 * j,
                        id0 - (uint32_t)j * (2u << 17), (uint32_t)(j & 1));
        } else {
          const uint64_t dA = sw128_desc(smem_u32(st + kOffV), 8192, 1024);
#pragma unroll 1
          for (int j = 0; j < 4; ++j)
            mma_bf16_ss(tD1 + 16 * j, dA + 128 * j, dB + 130 * j, id0 - (uint32_t)j * (2u << 17), j > 0);
        }
        mma_commit(&S.bar[kBarK1Mma]);
        mma_commit(&S.bar[kBarWMma]);  // the state group's share of the epilogue waits here
      }
      if (ok) ok = wait_bar(S, kBarK1Mma, k1ph, p.status);
      k1ph ^= 1u;
      // NW / QP are free once the previous chunk's output MMA has completed
      if (ok && c >= 1) ok = wait_bar(S, kBarMma1, (uint32_t)((c - 1) & 1), p.status);
      if (named_sync_or(kBarF, kSubThreads, !ok)) break;
      tc_fence_after();

      // ---- -W^T -> NW tile.  The state group meanwhile writes the U~^T tile and
      // refills the stage once its last reader is done.
      {
        const float ne1 = -s_e1[row], ne2 = -s_e2[row];
        {  // t < 32: the first half only
          uint32_t w1[32];
          tmem_ld32(tScr + lane_base, w1);
          tmem_wait_ld();
          const float2 n1 = make_float2(ne1, ne1);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 x = f2mul(n1, make_float2(__uint_as_float(w1[j]), __uint_as_float(w1[j + 1])));
            w1[j] = __float_as_uint(x.x);
            w1[j + 1] = __float_as_uint(x.y);
          }
          store_row32_bits(sm + kOffNW, row, 0, w1);
        }
        // t >= 32, 16 columns at a time
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t w1[16], w2[16];
          tmem_ld16(tScr + lane_base + 32 + 16 * q, w1);
          tmem_ld16(tScr + lane_base + 64 + 16 * q, w2);
          tmem_wait_ld();
          const float2 n1 = make_float2(ne1, ne1), n2 = make_float2(ne2, ne2);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float2 x = f2fma(n2, make_float2(__uint_as_float(w2[j]), __uint_as_float(w2[j + 1])),
                                   f2mul(n1, make_float2(__uint_as_float(w1[j]),
                                                         __uint_as_float(w1[j + 1]))));
            w1[j] = __float_as_uint(x.x);
            w1[j + 1] = __float_as_uint(x.y);
          }
          store_row16_bits(sm + kOffNW, row, 32 + 16 * q, w1);
        }
      }
      // Rq of rows t < 32 for this thread's channel, read before the stage is refilled
      uint32_t rq_lo[16];
      if (write_out) load_rq_col(st, row, 0, rq_lo);
      fence_proxy_async();
      tc_fence_before();
      ok = wait_bar(S, kBarWDone, (uint32_t)(c & 1), p.status);
      // O_intra lands in the O half of D1: free once the prep group has stored the
      // previous chunk's O
      if (ok && write_out && issuer2 && c >= 1)
        ok = wait_bar(S, kBarD1OFree, (uint32_t)((c - 1) & 1), p.status);
      if (named_sync_or(kBarF, kSubThreads, !ok)) break;

      if (write_out) {
        // ---- first issuer: Q'^T acc = (-W)^T P^T (the Rq term is added in the
        //      epilogue); second issuer: O_intra^T = U~^T (P + P_lo)^T
        if (issuer) {
          tc_fence_after();
          // K-step j meets P rows from 16j (B + 2080 j bytes), N = 64 - 16j
          const uint64_t dP = sw128_desc(smem_u32(st + kOffG), 16, 1024);
          const uint32_t id0 = idesc_bf16_f32(128, 64, 0, 0);
          if (issuer1) {
            const uint64_t dW = sw128_desc(smem_u32(sm + kOffNW), 16, 1024);
#pragma unroll 1
            for (int j = 0; j < 4; ++j)  // rows t >= 16j of P only (see the W / U~ MMAs)
              mma_bf16_ss(tScr + 16 * j, dW + 2 * j, dP + 130 * j, id0 - (uint32_t)j * (2u << 17), j > 0);
          } else {
            const uint64_t dU = sw128_desc(smem_u32(st + kOffV), 16, 1024);
            const uint64_t dPl = sw128_desc(smem_u32(sm + kOffPlo), 16, 1024);
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {  // P_hi, then P_lo
              const int jj = j & 3;
              mma_bf16_ss(tD1 + 64 + 16 * jj, dU + 2 * jj, (j < 4 ? dP : dPl) + 130 * jj,
                          id0 - (uint32_t)jj * (2u << 17), j > 0);
            }
          }
          mma_commit(&S.bar[kBarK1Mma]);
          mma_commit(&S.bar[kBarQMma]);
        }
        ok = wait_bar(S, kBarK1Mma, k1ph, p.status);
        k1ph ^= 1u;
        if (named_sync_or(kBarF, kSubThreads, !ok)) break;
        tc_fence_after();
        // ---- Q'^T = acc + Diag(2^rho1) Rq^T, columns t < 32 (the state group
        // writes t >= 32)
        {
          uint32_t acc[32];
          tmem_ld32(tScr + lane_base, acc);
          tmem_wait_ld();
          qprime_store(sm + kOffQP, row, 0, acc, rq_lo, s_e1[row]);
        }
        fence_proxy_async();
        tc_fence_before();
        ok = wait_bar(S, kBarQDone, (uint32_t)(c & 1), p.status);
        if (named_sync_or(kBarF, kSubThreads, !ok)) break;
      }
      // both groups' epilogues have read 2^rho2: from here it is the state group's
      // pre-scale 2^(rho2 - m) (the overflow guard in prep)
      const_cast<float*>(s_e2)[row] = s_e2[row] * reinterpret_cast<const float*>(sm + kOffMdown)[s];
      named_sync(kBarF, kSubThreads);
      if (leader) {
        mbar_arrive(&S.bar[kBarK1Ready]);  // chunk c's factors are ready for the state group
        mbar_arrive(&S.bar[kBarSlot0 + s]);  // every read of scratch slot s is done
      }
    }
  } else {
    // =====================================================================
    // state group: the inter-chunk recurrence.  Thread owns TMEM lane `row`
    // (value channel v).  The fp32 state S (lanes v, columns k) lives in TMEM:
    // before the state MMA it is pre-scaled to 2^rho2 S so that the MMA adds
    // Delta = U^T C2 directly, and S_next = 2^(gam63 - rho2) (2^rho2 S + Delta)
    // = Diag(2^gam63) S + Diag(2^(gam63 - rho2)) Delta.
    // =====================================================================
    const int row = tid;
    const bool leader = (tid == 0);
    const uint32_t tD1 = tbase + kTD1, tSt = tbase + kTState, tSA = tbase + kTSA,
                   tUA = tbase + kTUA, tULA = tbase + kTULA;
    // initial state -> TMEM (fp32, true scale) and its bf16 copy (MMA operand)
#pragma unroll 1
    for (int pc = 0; pc < 4; ++pc) {
      float x[32];
      const int64_t base = (int64_t)row * kHeadDim + 32 * pc;
      if (init_identity) {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = (32 * pc + i == row) ? 1.f : 0.f;
      } else if (init_ptr && init_bf16) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(init_ptr) + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 w = src[i];
          x[8 * i + 0] = bf_lo(w.x); x[8 * i + 1] = bf_hi(w.x);
          x[8 * i + 2] = bf_lo(w.y); x[8 * i + 3] = bf_hi(w.y);
          x[8 * i + 4] = bf_lo(w.z); x[8 * i + 5] = bf_hi(w.z);
          x[8 * i + 6] = bf_lo(w.w); x[8 * i + 7] = bf_hi(w.w);
        }
      } else if (init_ptr) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(init_ptr) + base);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 w = src[i];
          x[4 * i + 0] = w.x; x[4 * i + 1] = w.y; x[4 * i + 2] = w.z; x[4 * i + 3] = w.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = 0.f;
      }
      uint32_t w32[32], w16[16];
#pragma unroll
      for (int i = 0; i < 32; ++i) w32[i] = __float_as_uint(x[i]);
#pragma unroll
      for (int i = 0; i < 16; ++i) w16[i] = pack_bf2(x[2 * i], x[2 * i + 1]);
      tmem_st32(tSt + lane_base + 32 * pc, w32);
      tmem_st16(tSA + lane_base + 16 * pc, w16);
      if (ck_unit && nchunks > 0) {  // checkpoint of chunk 0: the initial state
        uint4* dst = reinterpret_cast<uint4*>(ck_unit + (int64_t)row * kHeadDim + 32 * pc);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(w16[4 * i], w16[4 * i + 1], w16[4 * i + 2], w16[4 * i + 3]);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    named_sync(kBarK2, kStateThreads);

#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      const float* s_e2 = reinterpret_cast<const float*>(sm + kOffE2) + b * 128;
      const float* s_f = reinterpret_cast<const float*>(sm + kOffF) + b * 128;
      const int64_t tok0 = bos + (int64_t)c * kChunk;

      // ---- share of chunk c's factor epilogues while the factor group writes
      // -W^T and the first half of Q'^T: the U~^T tile (operand of the O_intra
      // MMA), the second half of Q'^T, and the refill of stage b once the last MMA
      // reading it has completed
      {
        uint8_t* const stb = sm + b * kStageBytes;
        const uint32_t tScr = tbase + kTSlot + kSlotCols * (uint32_t)b;  // chunk c's scratch slot
        uint32_t rq_hi[16];
        bool ok = wait_bar(S, kBarWMma, (uint32_t)(c & 1), p.status);
        if (named_sync_or(kBarK2, kStateThreads, !ok)) break;
        tc_fence_after();
        if (write_out) {
#pragma unroll 1
          for (int hq = 0; hq < 2; ++hq) {
            uint32_t u[32];
            tmem_ld32(tD1 + lane_base + 32 * hq, u);
            tmem_wait_ld();
            store_row32_bits(stb + kOffV, row, 32 * hq, u);
          }
          // Rq of rows t >= 32 for this thread's channel, read before the refill
          load_rq_col(stb, row, 32, rq_hi);
        }
        fence_proxy_async();
        tc_fence_before();
        named_sync(kBarK2, kStateThreads);
        if (leader) mbar_arrive(&S.bar[kBarWDone]);
        if (write_out) {
          ok = wait_bar(S, kBarQMma, (uint32_t)(c & 1), p.status);
          if (named_sync_or(kBarK2, kStateThreads, !ok)) break;
          tc_fence_after();
        }
        // the last MMA reading stage b has completed (without outputs, the W / U~
        // MMAs): refill it with chunk c + 2
        if (leader && c + 2 < nchunks)
          issue_chunk_loads<kGateF32>(stb, &S.bar[kBarTma0 + b], &tq, &tk, &tv, &tg, h, hk,
                                      tok0 + 2 * kChunk, !zero_v);
        if (write_out) {
          // Q'^T columns t >= 32: acc + Diag(2^rho2) Rq^T
          uint32_t acc[32];
          tmem_ld32(tScr + lane_base + 32, acc);
          tmem_wait_ld();
          qprime_store(sm + kOffQP, row, 32, acc, rq_hi, s_e2[row]);
          fence_proxy_async();
          tc_fence_before();
          named_sync(kBarK2, kStateThreads);
          if (leader) mbar_arrive(&S.bar[kBarQDone]);
        }
      }

      // ---- output MMA: D1 += S^T [-W^T | Q'^T]   (factors of chunk c ready)
      bool ok = true;
      if (leader) {
        // the state group's leader pulls chunk c + 4 into L2 while it waits
        if (c + 4 < nchunks)
          prefetch_chunk_l2<kGateF32>(&tq, &tk, &tv, &tg, h, hk, tok0 + 4 * kChunk);
        ok = wait_bar(S, kBarK1Ready, (uint32_t)(c & 1), p.status);
        if (ok) {
          tc_fence_after();
          const uint64_t dW = sw128_desc(smem_u32(sm + kOffNW), 16384, 1024);
          // the O half (Q'^T columns) only where outputs are written
          const uint32_t id = idesc_bf16_f32(128, write_out ? 128 : 64, 0, 1);
#pragma unroll 1
          for (int j = 0; j < 8; ++j) mma_bf16_ts(tD1, tSA + j * 8, dW + 128 * j, id, 1u);
          mma_commit(&S.bar[kBarMma1]);
        }
      }
      if (named_sync_or(kBarK2, kStateThreads, !ok)) break;
      tc_fence_after();
      // ---- while it runs: pre-scale the state, S <- Diag(2^rho2) S
#pragma unroll 1
      for (int pc = 0; pc < 4; ++pc) {
        uint32_t a[32];
        tmem_ld32(tSt + lane_base + 32 * pc, a);
        tmem_wait_ld();
        const float4* e2 = reinterpret_cast<const float4*>(s_e2 + 32 * pc);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 e = e2[j4];
          const float2 x = f2mul(make_float2(e.x, e.y), make_float2(__uint_as_float(a[4 * j4 + 0]),
                                                                    __uint_as_float(a[4 * j4 + 1])));
          const float2 y = f2mul(make_float2(e.z, e.w), make_float2(__uint_as_float(a[4 * j4 + 2]),
                                                                    __uint_as_float(a[4 * j4 + 3])));
          a[4 * j4 + 0] = __float_as_uint(x.x);
          a[4 * j4 + 1] = __float_as_uint(x.y);
          a[4 * j4 + 2] = __float_as_uint(y.x);
          a[4 * j4 + 3] = __float_as_uint(y.y);
        }
        tmem_st32(tSt + lane_base + 32 * pc, a);
      }
      tmem_wait_st();
      ok = wait_bar(S, kBarMma1, (uint32_t)(c & 1), p.status);
      if (named_sync_or(kBarK2, kStateThreads, !ok)) break;
      tc_fence_after();

      // ---- 2^-m U^T -> bf16 hi/lo operands in TMEM (m: the overflow guard)
      const float md = reinterpret_cast<const float*>(sm + kOffMdown)[b];
      const float2 md2 = make_float2(md, md);
#pragma unroll 1
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t a[16], hi[8], lo[8];
        tmem_ld16(tD1 + lane_base + 16 * qq, a);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 u = f2mul(md2, make_float2(__uint_as_float(a[2 * j]), __uint_as_float(a[2 * j + 1])));
          hi[j] = pack_bf2(u.x, u.y);
          const float2 r = f2sub(u, make_float2(bf_lo(hi[j]), bf_hi(hi[j])));
          lo[j] = pack_bf2(r.x, r.y);
        }
        tmem_st8(tUA + lane_base + 8 * qq, hi);
        tmem_st8(tULA + lane_base + 8 * qq, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      named_sync(kBarK2, kStateThreads);
      if (leader) mbar_arrive(&S.bar[kBarD1UFree]);  // the U half of D1 has been read

      // ---- state MMA: S += U^T C2 (hi + lo)
      if (leader) {
        tc_fence_after();
        const uint64_t dC = sw128_desc(smem_u32(sm + kOffC2 + b * 16384), 8192, 1024);
        const uint32_t id = idesc_bf16_f32(128, 128, 0, 1);
#pragma unroll 1
        for (int j = 0; j < 8; ++j)  // U^T hi, then lo
          mma_bf16_ts(tSt, (j < 4 ? tUA : tULA) + (j & 3) * 8, dC + 128 * (j & 3), id, 1u);
        mma_commit(&S.bar[kBarMma2]);
      }
      // (O, the other half of D1, is stored by the prep group)
      ok = wait_bar(S, kBarMma2, (uint32_t)(c & 1), p.status);
      if (named_sync_or(kBarK2, kStateThreads, !ok)) break;
      tc_fence_after();

      // ---- S <- Diag(2^(gam63 - rho2)) S (true scale again) and its bf16 copy
#pragma unroll 1
      for (int pc = 0; pc < 4; ++pc) {
        uint32_t a[32], w16[16];
        tmem_ld32(tSt + lane_base + 32 * pc, a);
        tmem_wait_ld();
        const float4* f4 = reinterpret_cast<const float4*>(s_f + 32 * pc);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 e = f4[j4];
          const float2 x = f2mul(make_float2(e.x, e.y), make_float2(__uint_as_float(a[4 * j4 + 0]),
                                                                    __uint_as_float(a[4 * j4 + 1])));
          const float2 y = f2mul(make_float2(e.z, e.w), make_float2(__uint_as_float(a[4 * j4 + 2]),
                                                                    __uint_as_float(a[4 * j4 + 3])));
          a[4 * j4 + 0] = __float_as_uint(x.x);
          a[4 * j4 + 1] = __float_as_uint(x.y);
          a[4 * j4 + 2] = __float_as_uint(y.x);
          a[4 * j4 + 3] = __float_as_uint(y.y);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
          w16[j] = pack_bf2(__uint_as_float(a[2 * j]), __uint_as_float(a[2 * j + 1]));
        tmem_st32(tSt + lane_base + 32 * pc, a);
        tmem_st16(tSA + lane_base + 16 * pc, w16);
        if (ck_unit && c + 1 < nchunks) {  // checkpoint of chunk c + 1
          uint4* dst = reinterpret_cast<uint4*>(
              ck_unit + ((int64_t)(c + 1) * H * kHeadDim + row) * kHeadDim + 32 * pc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(w16[4 * i], w16[4 * i + 1], w16[4 * i + 2], w16[4 * i + 3]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      named_sync(kBarK2, kStateThreads);
      if (leader) mbar_arrive(&S.bar[kBarSlotF0 + b]);  // f[b] consumed
    }

    if (!*S.abort && fin_ptr) {
      tc_fence_after();
#pragma unroll 1
      for (int pc = 0; pc < 4; ++pc) {
        uint32_t a[32];
        tmem_ld32(tSt + lane_base + 32 * pc, a);
        tmem_wait_ld();
        const int64_t base = (int64_t)row * kHeadDim + 32 * pc;
        if (fin_bf16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(fin_ptr) + base);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf2(__uint_as_float(a[8 * i + 0]), __uint_as_float(a[8 * i + 1]));
            w.y = pack_bf2(__uint_as_float(a[8 * i + 2]), __uint_as_float(a[8 * i + 3]));
            w.z = pack_bf2(__uint_as_float(a[8 * i + 4]), __uint_as_float(a[8 * i + 5]));
            w.w = pack_bf2(__uint_as_float(a[8 * i + 6]), __uint_as_float(a[8 * i + 7]));
            dst[i] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(fin_ptr) + base);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(a[4 * i + 0]), __uint_as_float(a[4 * i + 1]),
                                 __uint_as_float(a[4 * i + 2]), __uint_as_float(a[4 * i + 3]));
        }
      }
    }
  }

  // Drain: on an abort, let copies and MMAs already in flight land (bounded).
  __syncthreads();
  if (*S.abort && tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      (void)mbar_wait(&S.bar[i], 0, kWaitNs / 16);
      (void)mbar_wait(&S.bar[i], 1, kWaitNs / 16);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// --------------------------------------------------------------- host side --
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}
}  // namespace

cudaError_t encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* ptr,
                             const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                             CUtensorMapSwizzle swizzle) {
  if (!ptr) {  // an empty tensor: no kernel reads through this map
    std::memset(map, 0, sizeof(*map));
    return cudaSuccess;
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  const CUresult r = enc(map, dtype, (cuuint32_t)rank, const_cast<void*>(ptr), d, st, bx, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_qkvg_maps(const void* q, const void* k, const void* v, const void* g,
                           int64_t T_total, int32_t H, int32_t qk_group, bool gate_f32,
                           CUtensorMap maps[4]) {
  if (qk_group < 1 || H % qk_group != 0) return cudaErrorInvalidValue;
  const uint64_t T = (uint64_t)(T_total > 0 ? T_total : 1);
  const void* ptrs[4] = {q, k, v, g};
  const int32_t heads[4] = {H / qk_group, H / qk_group, H, H};
  for (int i = 0; i < 4; ++i) {
    const bool f32 = (i == 3 && gate_f32);  // fp32 gate: prefetch-only map, no swizzle
    const uint64_t esz = f32 ? 4 : 2;
    const uint64_t dims[3] = {(uint64_t)kHeadDim, (uint64_t)heads[i], T};
    const uint64_t strides[2] = {(uint64_t)kHeadDim * esz, (uint64_t)heads[i] * kHeadDim * esz};
    const uint32_t box[3] = {f32 ? 128u : 64u, 1, (uint32_t)kChunk};
    const cudaError_t e = encode_tiled_map(
        &maps[i], f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
        ptrs[i], dims, strides, box, f32 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {
template <bool kGateF32>
cudaError_t launch_instance(const CUtensorMap maps[4], const ChunkFwdParams& p, int64_t grid,
                            cudaStream_t stream) {
  static bool attr_done[64];
  const cudaError_t e = ensure_smem_attr(
      reinterpret_cast<const void*>(kda_chunk_fwd_kernel<kGateF32>), (int)kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  kda_chunk_fwd_kernel<kGateF32><<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(
      maps[0], maps[1], maps[2], maps[3], p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_chunk_fwd(const CUtensorMap maps[4], const ChunkFwdParams& p, int64_t grid,
                             cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  return p.gate_f32 ? launch_instance<true>(maps, p, grid, stream)
                    : launch_instance<false>(maps, p, grid, stream);
}

}  // namespace kda
