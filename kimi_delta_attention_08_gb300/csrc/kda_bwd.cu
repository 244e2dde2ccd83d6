// kda_bwd.cu -- backward pass of Kimi Delta Attention: reverse mode of the
// token recurrence
//   S' = Diag(alpha) S_{t-1},  d = S'^T k,  u = beta (v - d),  S_t = S' + k u^T,
//   o_t = scale S_t^T q
// (the recurrence of the forward kernels, with the same gate, l2-norm and sigmoid
// preprocessing).  The pages' kernels are forward only ("feat(kda): SM90 FlashKDA
// prefill, intracard CP, and backend dispatch", commit notes); the reverse mode
// below is derived from the recurrence:
//   dS  += scale q do^T              dq  = scale S_t do
//   du   = dS^T k                    dk += dS u
//   dbeta = du . (v - d)             dv  = beta du              dd = -beta du
//   dS'  = dS + k dd^T               dk += S' dd
//   dalpha[k] = sum_v dS'[k][v] S_{t-1}[k][v]                   dS_{t-1} = Diag(alpha) dS'
// then back through the gate, the l2 norms and the sigmoid of beta.
//
// Persistent CTAs (one per SM, 512 threads) walk the (sequence, value head)
// units.  The state and its gradient live in registers with the layout of the
// token-by-token forward kernel: warp w holds value columns 8w .. 8w+7, lane l
// key channels 4l .. 4l+3.  Per unit: a forward sweep stores the state at every
// 16-token block start (checkpoint slots in the workspace); then, block by block
// in reverse, the block is recomputed from its checkpoint: u and v - d of every
// token to shared memory, and the decayed state S' = Diag(alpha) S_{t-1} of every
// fourth token to a per-CTA scratch of 256 KiB (each thread reads back only the
// words it wrote; the scratch of all CTAs stays in L2).  Then the block's tokens
// are stepped backward; the reverse step of token j regenerates its S' from the
// kept one before it with S'_{i+1} = Diag(alpha_{i+1}) (S'_i + k_i u_i^T), the
// same operations as the recomputation and so the same values.
// The reverse step needs S_{t-1} only through S': S_t = S' + k u^T, and
// alpha[c] dalpha[c] = sum_v dS'[c][v] S'[c][v] is the product the gate's
// reverse takes.  Per token, the per-channel sums over all value columns (q and
// k gradients, alpha dalpha) and dbeta are reduced across the 16 warps through
// double-buffered shared memory with one barrier per token; once per block, one
// warp per token takes them through the preprocessing.  Every output has a
// single writer (grouped value heads write per-value-head dq / dk, summed
// afterwards in a fixed order), so results are bitwise reproducible.  Gradients
// are fp32; the four-wide products are packed f32x2 instructions.
#include <cuda_bf16.h>

#include <cstring>

#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kBwdThreads = 512;
constexpr int kBwdMaxCtas = 160;  // scratch is sized for at most this many CTAs
constexpr int kSt = kHeadDim * kHeadDim;  // floats per state

// dynamic shared memory (byte offsets)
constexpr uint32_t kVecBytes = kBwdBlock * kHeadDim * 4;  // one [block][128] fp32 array
constexpr uint32_t kRedBytes = 16 * 3 * kHeadDim * 4;     // per-warp partials [16][3][128]
constexpr uint32_t kOffK = 0;                              // l2-normalised k
constexpr uint32_t kOffQ = kOffK + kVecBytes;              // l2-normalised q
constexpr uint32_t kOffA = kOffQ + kVecBytes;              // alpha
constexpr uint32_t kOffV = kOffA + kVecBytes;              // v
constexpr uint32_t kOffDo = kOffV + kVecBytes;             // dout
constexpr uint32_t kOffPre = kOffDo + kVecBytes;           // gate pre-activation a
constexpr uint32_t kOffU = kOffPre + kVecBytes;            // u = beta (v - d), per value column
constexpr uint32_t kOffVmd = kOffU + kVecBytes;            // v - d
constexpr uint32_t kOffScal = kOffVmd + kVecBytes;         // beta, rq, rk [3][block]
constexpr uint32_t kOffRed = kOffScal + 3 * kBwdBlock * 4; // partials, two buffers [2][16][3][128]
constexpr uint32_t kOffRedB = kOffRed + 2 * kRedBytes;     // per-warp dbeta [2][16]
constexpr uint32_t kOffRes = kOffRedB + 2 * 16 * 4;        // per-token sums [block][3][128]
constexpr uint32_t kOffResB = kOffRes + kBwdBlock * 3 * kHeadDim * 4;  // per-token dbeta [block]
constexpr uint32_t kOffAcc = kOffResB + kBwdBlock * 4;      // dt_bias grad [128], A_log grad
constexpr uint32_t kBwdSmem = kOffAcc + (kHeadDim + 4) * 4;
static_assert(kBwdSmem <= 232448, "shared memory budget");

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float4 bf4(uint2 w) {
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
}
__device__ __forceinline__ float sigm(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}
// Four-wide products as two packed f32x2 instructions (each lane rounded like the
// scalar mul / fma).
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  const float2 lo = f2mul(make_float2(a.x, a.y), make_float2(b.x, b.y));
  const float2 hi = f2mul(make_float2(a.z, a.w), make_float2(b.z, b.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {  // a * b + c
  const float2 lo = f2fma(make_float2(a.x, a.y), make_float2(b.x, b.y), make_float2(c.x, c.y));
  const float2 hi = f2fma(make_float2(a.z, a.w), make_float2(b.z, b.w), make_float2(c.z, c.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 fma4s(float4 a, float s, float4 c) {  // a * s + c
  return fma4(a, make_float4(s, s, s, s), c);
}
// a . b as (a.x b.x + a.z b.z) + (a.y b.y + a.w b.w): two packed instructions and an add.
__device__ __forceinline__ float dot4p(float4 a, float4 b) {
  const float2 t = f2fma(make_float2(a.z, a.w), make_float2(b.z, b.w),
                         f2mul(make_float2(a.x, a.y), make_float2(b.x, b.y)));
  return t.x + t.y;
}

// This thread's part of a state [128 v][128 k] at `src` (fp32 or bf16): S[c]
// holds S[k = c0 .. c0+3][v = v0 + c]; null gives zero.
__device__ __forceinline__ void load_state(float4 (&S)[8], const void* src, bool is_bf16, int v0,
                                           int c0) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    if (!src) {
      S[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (is_bf16) {
      S[c] = bf4(*reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(src) +
                                                 (v0 + c) * kHeadDim + c0));
    } else {
      S[c] = *reinterpret_cast<const float4*>(static_cast<const float*>(src) +
                                              (v0 + c) * kHeadDim + c0);
    }
  }
}
__device__ __forceinline__ void store_state(float* dst, const float4 (&S)[8], int v0, int c0) {
#pragma unroll
  for (int c = 0; c < 8; ++c) *reinterpret_cast<float4*>(dst + (v0 + c) * kHeadDim + c0) = S[c];
}

__device__ __forceinline__ bool bwd_bounds(const BwdParams& p, int n, int64_t& bos, int64_t& eos) {
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

struct Smem {
  float (*k)[kHeadDim];
  float (*q)[kHeadDim];
  float (*a)[kHeadDim];
  float (*v)[kHeadDim];
  float (*dout)[kHeadDim];
  float (*pre)[kHeadDim];
  float (*u)[kHeadDim];
  float (*vmd)[kHeadDim];
  float* beta;
  float* rq;
  float* rk;
  float (*red)[16][3][kHeadDim];  // [buffer][warp][q, k, alpha][channel]
  float (*redb)[16];              // [buffer][warp]
  float (*res)[3][kHeadDim];      // [token of the block][q, k, alpha][channel]
  float* resb;                    // [token of the block]
  float* acc;
};

// Preprocessing of the block's tokens t0 .. t0+nt-1, one warp per token, lane l
// on channels 4l .. 4l+3: l2-normalised q and k, alpha = exp(lb sigmoid(e (g +
// dt_bias))) and its pre-activation e (g + dt_bias), v, beta = sigmoid(beta_raw),
// the norm factors, and dout.
__device__ void prep_block(const BwdParams& p, const Smem& sm, int64_t t0, int nt, int h, int hk,
                           float ea, const float (&dtb)[4], bool with_dout) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, c0 = 4 * lane;
  const int H = p.H, HK = p.H / p.qk_group;
  for (int j = warp; j < nt; j += 16) {
    const int64_t t = t0 + j;
    const int64_t rk_ = (t * HK + hk) * kHeadDim + c0, rv = (t * H + h) * kHeadDim + c0;
    const float4 q = bf4(*reinterpret_cast<const uint2*>(p.q + rk_));
    const float4 k = bf4(*reinterpret_cast<const uint2*>(p.k + rk_));
    const float4 v = bf4(*reinterpret_cast<const uint2*>(p.v + rv));
    const float4 g = p.gate_f32 ? *reinterpret_cast<const float4*>(static_cast<const float*>(p.g) + rv)
                                : bf4(*reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.g) + rv));
    const float rq = 1.0f / sqrtf(warp_sum(dot4(q, q)) + 1e-6f);
    const float rk = 1.0f / sqrtf(warp_sum(dot4(k, k)) + 1e-6f);
    const float gv[4] = {g.x, g.y, g.z, g.w};
    float al[4], pa[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pa[e] = ea * (gv[e] + dtb[e]);
      al[e] = expf(p.lower_bound * sigm(pa[e]));
    }
    *reinterpret_cast<float4*>(&sm.pre[j][c0]) = make_float4(pa[0], pa[1], pa[2], pa[3]);
    *reinterpret_cast<float4*>(&sm.q[j][c0]) = make_float4(q.x * rq, q.y * rq, q.z * rq, q.w * rq);
    *reinterpret_cast<float4*>(&sm.k[j][c0]) = make_float4(k.x * rk, k.y * rk, k.z * rk, k.w * rk);
    *reinterpret_cast<float4*>(&sm.a[j][c0]) = make_float4(al[0], al[1], al[2], al[3]);
    *reinterpret_cast<float4*>(&sm.v[j][c0]) = v;
    if (with_dout)
      *reinterpret_cast<float4*>(&sm.dout[j][c0]) = bf4(*reinterpret_cast<const uint2*>(p.dout + rv));
    if (lane == 0) {
      sm.beta[j] = sigm(bf(p.beta[t * H + h]));
      sm.rq[j] = rq;
      sm.rk[j] = rk;
    }
  }
}

// One forward step of token j of the block: S <- Diag(alpha) S + k u^T.  With
// kKeep, u and v - d of the warp's columns go to shared memory (lanes 4c hold
// column v0 + c) and, when `keep` is set, the decayed state S' = Diag(alpha) S to
// `keep` (this thread's part), for the reverse step.
template <bool kKeep>
__device__ __forceinline__ void fwd_step(float4 (&S)[8], const Smem& sm, int j, int v0, int c0,
                                         int lane, float* keep = nullptr) {
  const float4 a4 = *reinterpret_cast<const float4*>(&sm.a[j][c0]);
  const float4 k4 = *reinterpret_cast<const float4*>(&sm.k[j][c0]);
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    S[c] = mul4(a4, S[c]);
    if (kKeep && keep) *reinterpret_cast<float4*>(keep + (v0 + c) * kHeadDim + c0) = S[c];
    x[c] = dot4p(S[c], k4);
  }
  const int vc = v0 + (lane >> 2);
  const float d = reduce_scatter8(x, lane);  // column vc
  const float vmd = sm.v[j][vc] - d;
  const float uu = sm.beta[j] * vmd;
  if (kKeep && (lane & 3) == 0) {
    sm.u[j][vc] = uu;
    sm.vmd[j][vc] = vmd;
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) S[c] = fma4s(k4, __shfl_sync(0xffffffffu, uu, 4 * c), S[c]);
}

// S' of token i + 1 from S' of token i: Diag(alpha_{i+1}) (S'_i + k_i u_i^T), with
// the operations of fwd_step, so bit for bit the recomputed value.
__device__ __forceinline__ void regen_step(float4 (&Sp)[8], const Smem& sm, int i, int v0, int c0) {
  const float4 k4 = *reinterpret_cast<const float4*>(&sm.k[i][c0]);
  const float4 a4 = *reinterpret_cast<const float4*>(&sm.a[i + 1][c0]);
#pragma unroll
  for (int c = 0; c < 8; ++c) Sp[c] = mul4(a4, fma4s(k4, sm.u[i][v0 + c], Sp[c]));
}

__device__ __forceinline__ void prefetch_token(const BwdParams& p, int64_t t, int h, int hk,
                                               bool with_dout, int lane) {
  const int HK = p.H / p.qk_group;
  const int64_t rk_ = (t * HK + hk) * kHeadDim, rv = (t * p.H + h) * kHeadDim;
  const char* a = nullptr;
  if (lane < 2) a = reinterpret_cast<const char*>(p.q + rk_) + 128 * lane;
  else if (lane < 4) a = reinterpret_cast<const char*>(p.k + rk_) + 128 * (lane - 2);
  else if (lane < 6) a = reinterpret_cast<const char*>(p.v + rv) + 128 * (lane - 4);
  else if (lane < 8) a = reinterpret_cast<const char*>(p.dout + rv) + 128 * (lane - 6);
  else if (p.gate_f32 ? lane < 12 : lane < 10)
    a = (p.gate_f32 ? reinterpret_cast<const char*>(static_cast<const float*>(p.g) + rv)
                    : reinterpret_cast<const char*>(static_cast<const uint16_t*>(p.g) + rv)) +
        128 * (lane - 8);
  if (a && (with_dout || lane < 6 || lane >= 8)) asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// L2 prefetch of the input rows (q, k, v, g and, with_dout, dout) of tokens
// t0 .. t0+nt-1: warp w takes tokens w, w + 16, ..., one lane per 128-byte line.
__device__ __forceinline__ void prefetch_block(const BwdParams& p, int64_t t0, int nt, int h,
                                               int hk, bool with_dout) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < nt; j += 16) prefetch_token(p, t0 + j, h, hk, with_dout, lane);
}


// One backward step of token j (token t of the sequence): dS holds dL/dS_t on
// entry and dL/dS_{t-1} on exit; Sp is S' = Diag(alpha) S_{t-1}; u and v - d come
// from the recomputation.  Writes dv; the sums over the value columns of the q
// and k gradients, of alpha dalpha (sum_v dS'[c][v] S'[c][v], which is
// alpha[c] sum_v dS'[c][v] S_{t-1}[c][v]) and of dbeta go to the block's
// per-token sums (partials through shared-memory buffer `buf`, summed over the 16
// warps in a fixed order).
__device__ __forceinline__ void bwd_step(const BwdParams& p, const Smem& sm, float4 (&dS)[8],
                                         const float4 (&Sp)[8], int j, int64_t t, int h, int buf,
                                         int v0, int c0, int warp, int lane) {
  const float4 a4 = *reinterpret_cast<const float4*>(&sm.a[j][c0]);
  const float4 k4 = *reinterpret_cast<const float4*>(&sm.k[j][c0]);
  const float4 q4 = *reinterpret_cast<const float4*>(&sm.q[j][c0]);
  const float bt = sm.beta[j];
  const int vc = v0 + (lane >> 2);  // the column this lane's reductions return
  // dS += scale q do^T; partial of S_t do over the warp's columns, S_t = S' + k u^T
  float4 xq = make_float4(0.f, 0.f, 0.f, 0.f);
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float doc = sm.dout[j][v0 + c];
    const float4 St = fma4s(k4, sm.u[j][v0 + c], Sp[c]);
    xq = fma4s(St, doc, xq);
    dS[c] = fma4s(q4, p.scale * doc, dS[c]);
    x[c] = dot4p(dS[c], k4);
  }
  // du = dS^T k
  const float du = reduce_scatter8(x, lane);
  if ((lane & 3) == 0) p.dv[(t * p.H + h) * kHeadDim + vc] = bt * du;
  // dk partial: dS u + S' dd;  dS' = dS + k dd^T;  alpha dalpha partial: dS' o S';  dS <- alpha dS'
  float4 xk = make_float4(0.f, 0.f, 0.f, 0.f), xa = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float uc = sm.u[j][v0 + c];
    const float ddc = -bt * __shfl_sync(0xffffffffu, du, 4 * c);
    xk = fma4s(dS[c], uc, xk);
    xk = fma4s(Sp[c], ddc, xk);
    const float4 dsp = fma4s(k4, ddc, dS[c]);
    xa = fma4(dsp, Sp[c], xa);
    dS[c] = mul4(a4, dsp);
  }
  // dbeta partial: du (v - d) over the warp's 8 columns (lanes 4c hold column c)
  const float db = warp_sum((lane & 3) == 0 ? du * sm.vmd[j][vc] : 0.f);
  *reinterpret_cast<float4*>(&sm.red[buf][warp][0][c0]) = xq;
  *reinterpret_cast<float4*>(&sm.red[buf][warp][1][c0]) = xk;
  *reinterpret_cast<float4*>(&sm.red[buf][warp][2][c0]) = xa;
  if (lane == 0) sm.redb[buf][warp] = db;
  // One barrier per token: buffer `buf` is written again two tokens later, after
  // the next token's barrier, which every summing thread reaches only when done.
  __syncthreads();
  if (threadIdx.x < 3 * kHeadDim) {  // sum over the 16 warps in a fixed order
    const int vi = threadIdx.x >> 7, ch = threadIdx.x & 127;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 16; ++w) s += sm.red[buf][w][vi][ch];
    sm.res[j][vi][ch] = s;
  } else if (threadIdx.x == 3 * kHeadDim) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 16; ++w) s += sm.redb[buf][w];
    sm.resb[j] = s;
  }
}

// The preprocessing's reverse for token j of the block (t = t0 + j), one warp,
// lane on channels c0 .. c0+3, from the block's per-token sums: the q and k
// gradients through the l2 norms, the gate gradient, dbeta through the sigmoid.
// The gate's contribution to the dt_bias gradient replaces the alpha sums in
// sm.res[j][2]; the A_log contribution replaces sm.resb[j].
__device__ __forceinline__ void block_tail(const BwdParams& p, const Smem& sm, int j, int64_t t,
                                           int h, int hk, float ea, int c0, int lane) {
  const int H = p.H, HK = p.H / p.qk_group;
  const int64_t rk_ = (t * HK + hk) * kHeadDim + c0, rv = (t * H + h) * kHeadDim + c0;
  const float4 q4 = *reinterpret_cast<const float4*>(&sm.q[j][c0]);
  const float4 k4 = *reinterpret_cast<const float4*>(&sm.k[j][c0]);
  const float4 dq_ = *reinterpret_cast<const float4*>(&sm.res[j][0][c0]);
  const float4 dqn = make_float4(p.scale * dq_.x, p.scale * dq_.y, p.scale * dq_.z, p.scale * dq_.w);
  const float4 dkn = *reinterpret_cast<const float4*>(&sm.res[j][1][c0]);
  const float4 adal = *reinterpret_cast<const float4*>(&sm.res[j][2][c0]);  // alpha dalpha
  const float dbs = sm.resb[j];
  // x^ = x r, r = (|x|^2 + eps)^(-1/2):  dx = r dx^ - r^3 (x . dx^) x = r (dx^ - (x^ . dx^) x^)
  const float rq = sm.rq[j], rkk = sm.rk[j], bt = sm.beta[j];
  const float qd = warp_sum(dot4(q4, dqn)), kd = warp_sum(dot4(k4, dkn));
  const float4 dq = make_float4(rq * (dqn.x - qd * q4.x), rq * (dqn.y - qd * q4.y),
                                rq * (dqn.z - qd * q4.z), rq * (dqn.w - qd * q4.w));
  const float4 dk = make_float4(rkk * (dkn.x - kd * k4.x), rkk * (dkn.y - kd * k4.y),
                                rkk * (dkn.z - kd * k4.z), rkk * (dkn.w - kd * k4.w));
  if (p.qk_group == 1) {
    *reinterpret_cast<float4*>(p.dq + rk_) = dq;
    *reinterpret_cast<float4*>(p.dk + rk_) = dk;
  } else {
    *reinterpret_cast<float4*>(p.dq_part + rv) = dq;
    *reinterpret_cast<float4*>(p.dk_part + rv) = dk;
  }
  // alpha = exp(lb s), s = sigmoid(a), a = e (g + dt_bias):  da = (alpha dalpha) lb s (1 - s).
  // 1 - sigmoid(x) is taken as sigmoid(-x): near saturation the subtraction would
  // cancel most of its digits (at x = 8, 1 - s keeps only about 4 of them in fp32).
  const float4 pre = *reinterpret_cast<const float4*>(&sm.pre[j][c0]);
  const float pv[4] = {pre.x, pre.y, pre.z, pre.w}, adv[4] = {adal.x, adal.y, adal.z, adal.w};
  float dg[4], dA = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float a = pv[e], s = sigm(a);
    const float da = adv[e] * p.lower_bound * s * sigm(-a);
    dg[e] = da * ea;
    dA = fmaf(da, a, dA);
  }
  *reinterpret_cast<float4*>(p.dg + rv) = make_float4(dg[0], dg[1], dg[2], dg[3]);
  *reinterpret_cast<float4*>(&sm.res[j][2][c0]) = make_float4(dg[0], dg[1], dg[2], dg[3]);
  dA = warp_sum(dA);
  __syncwarp();  // every lane has read sm.resb[j]
  if (lane == 0) {
    sm.resb[j] = dA;
    p.dbeta[t * H + h] = dbs * bt * sigm(-bf(p.beta[t * H + h]));
  }
}

__global__ void __launch_bounds__(kBwdThreads, 1) kda_bwd_kernel(const BwdParams p) {
  extern __shared__ __align__(16) uint8_t smb[];
  Smem sm;
  sm.k = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffK);
  sm.q = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffQ);
  sm.a = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffA);
  sm.v = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffV);
  sm.dout = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffDo);
  sm.pre = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffPre);
  sm.u = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffU);
  sm.vmd = reinterpret_cast<float (*)[kHeadDim]>(smb + kOffVmd);
  sm.beta = reinterpret_cast<float*>(smb + kOffScal);
  sm.rq = sm.beta + kBwdBlock;
  sm.rk = sm.rq + kBwdBlock;
  sm.red = reinterpret_cast<float (*)[16][3][kHeadDim]>(smb + kOffRed);
  sm.redb = reinterpret_cast<float (*)[16]>(smb + kOffRedB);
  sm.res = reinterpret_cast<float (*)[3][kHeadDim]>(smb + kOffRes);
  sm.resb = reinterpret_cast<float*>(smb + kOffResB);
  sm.acc = reinterpret_cast<float*>(smb + kOffAcc);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.H, v0 = 8 * warp, c0 = 4 * lane;
  const int units = p.N * H;
  float* const scr = p.scratch + (int64_t)blockIdx.x * (kBwdBlock / kBwdKeep) * kSt;

#pragma unroll 1
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int n = u / H, h = u % H, hk = h / p.qk_group;
    int64_t bos, eos;
    if (!bwd_bounds(p, n, bos, eos)) {
      if (tid == 0) atomicOr(p.status, kDevStatusBadSeqlens);
      if (tid <= kHeadDim) p.unit_part[(int64_t)u * (kHeadDim + 1) + tid] = 0.f;
      continue;
    }
    const int64_t nblk = (eos - bos + kBwdBlock - 1) / kBwdBlock;
    const float ea = expf(p.A_log[h]);
    float dtb[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) dtb[e] = p.dt_bias[h * kHeadDim + c0 + e];
    const int64_t st_off = (int64_t)u * kSt;

    // ---- forward sweep: checkpoint at every block start
    float4 S[8];
    load_state(S,
               p.init_state ? (p.state_bf16 ? (const void*)(static_cast<const uint16_t*>(p.init_state) + st_off)
                                            : (const void*)(static_cast<const float*>(p.init_state) + st_off))
                            : nullptr,
               p.state_bf16 != 0, v0, c0);
#pragma unroll 1
    for (int64_t m = 0; m < nblk; ++m) {
      store_state(p.ckpt + (bwd_slot(bos, n, m) * H + h) * kSt, S, v0, c0);
      const int64_t t0 = bos + m * kBwdBlock;
      const int nt = (int)((eos - t0) < kBwdBlock ? (eos - t0) : kBwdBlock);
      prep_block(p, sm, t0, nt, h, hk, ea, dtb, false);
      if (m + 1 < nblk) {
        const int64_t tn = t0 + kBwdBlock;
        prefetch_block(p, tn, (int)((eos - tn) < kBwdBlock ? (eos - tn) : kBwdBlock), h, hk, false);
      }
      __syncthreads();
#pragma unroll 1
      for (int j = 0; j < nt; ++j) fwd_step<false>(S, sm, j, v0, c0, lane);
      __syncthreads();  // the next block's prep overwrites the token vectors
    }

    // ---- backward sweep
    float4 dS[8];
    load_state(dS,
               p.dfinal ? (p.state_bf16 ? (const void*)(static_cast<const uint16_t*>(p.dfinal) + st_off)
                                        : (const void*)(static_cast<const float*>(p.dfinal) + st_off))
                        : nullptr,
               p.state_bf16 != 0, v0, c0);
    if (tid <= kHeadDim) sm.acc[tid] = 0.f;
#pragma unroll 1
    for (int64_t m = nblk - 1; m >= 0; --m) {
      load_state(S, p.ckpt + (bwd_slot(bos, n, m) * H + h) * kSt, false, v0, c0);
      const int64_t t0 = bos + m * kBwdBlock;
      const int nt = (int)((eos - t0) < kBwdBlock ? (eos - t0) : kBwdBlock);
      prep_block(p, sm, t0, nt, h, hk, ea, dtb, true);
      if (m > 0) prefetch_block(p, t0 - kBwdBlock, kBwdBlock, h, hk, true);
      __syncthreads();
#pragma unroll 1
      for (int j = 0; j < nt; ++j)  // u and v - d of every token, S' of every kBwdKeep-th
        fwd_step<true>(S, sm, j, v0, c0, lane,
                       j % kBwdKeep == 0 ? scr + (j / kBwdKeep) * kSt : nullptr);
      __syncwarp();  // u and v - d of the warp's columns are visible to all its lanes
#pragma unroll 1
      for (int j = nt - 1; j >= 0; --j) {
        float4 Sp[8];
        const int b = j - j % kBwdKeep;
        load_state(Sp, scr + (b / kBwdKeep) * kSt, false, v0, c0);  // written by this thread
#pragma unroll 1
        for (int i = b; i < j; ++i) regen_step(Sp, sm, i, v0, c0);
        bwd_step(p, sm, dS, Sp, j, t0 + j, h, j & 1, v0, c0, warp, lane);
      }
      __syncthreads();  // the block's per-token sums are complete
      for (int j = warp; j < nt; j += 16) block_tail(p, sm, j, t0 + j, h, hk, ea, c0, lane);
      __syncthreads();  // the tails are done with the block's vectors and sums
      if (tid <= kHeadDim) {  // dt_bias / A_log sums in a fixed order (last token first)
        float s = sm.acc[tid];
        for (int j = nt - 1; j >= 0; --j) s += tid < kHeadDim ? sm.res[j][2][tid] : sm.resb[j];
        sm.acc[tid] = s;
      }
    }
    if (p.dinit) store_state(p.dinit + st_off, dS, v0, c0);
    if (tid <= kHeadDim) p.unit_part[(int64_t)u * (kHeadDim + 1) + tid] = sm.acc[tid];
    __syncthreads();  // before the next unit clears them
  }
}

// Fixed-order sums: dq / dk over the value heads of each q/k head (grouped
// heads), dt_bias / A_log gradients over the sequences.
__global__ void kda_bwd_reduce_kernel(const BwdParams p, float* dA_log, float* ddt_bias) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int G = p.qk_group, HK = p.H / G;
  if (G > 1) {
    const int64_t total = p.total_tokens * HK * kHeadDim;
    for (int64_t i = i0; i < total; i += stride) {
      const int64_t c = i % kHeadDim, hk = (i / kHeadDim) % HK, t = i / ((int64_t)kHeadDim * HK);
      float sq = 0.f, sk = 0.f;
      for (int j = 0; j < G; ++j) {
        const int64_t src = (t * p.H + hk * G + j) * kHeadDim + c;
        sq += p.dq_part[src];
        sk += p.dk_part[src];
      }
      p.dq[i] = sq;
      p.dk[i] = sk;
    }
  }
  for (int64_t i = i0; i < (int64_t)p.H * (kHeadDim + 1); i += stride) {
    const int h = (int)(i / (kHeadDim + 1)), e = (int)(i % (kHeadDim + 1));
    float s = 0.f;
    for (int n = 0; n < p.N; ++n) s += p.unit_part[((int64_t)n * p.H + h) * (kHeadDim + 1) + e];
    if (e < kHeadDim)
      ddt_bias[h * kHeadDim + e] = s;
    else
      dA_log[h] = s;
  }
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& p, int num_sms, float* dA_log, float* ddt_bias,
                       cudaStream_t stream) {
  static bool attr_done[64];
  const cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kda_bwd_kernel),
                                         (int)kBwdSmem, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t units = (int64_t)p.N * p.H;
  int64_t grid = units < num_sms ? units : num_sms;
  if (grid > kBwdMaxCtas) grid = kBwdMaxCtas;
  if (grid > 0) kda_bwd_kernel<<<(unsigned)grid, kBwdThreads, kBwdSmem, stream>>>(p);
  return launch_bwd_reduce(p, dA_log, ddt_bias, stream);
}

cudaError_t launch_bwd_reduce(const BwdParams& p, float* dA_log, float* ddt_bias,
                              cudaStream_t stream) {
  kda_bwd_reduce_kernel<<<256, 256, 0, stream>>>(p, dA_log, ddt_bias);
  return cudaGetLastError();
}

int64_t bwd_scratch_ctas(int64_t units) { return units < kBwdMaxCtas ? units : kBwdMaxCtas; }

}  // namespace kda
