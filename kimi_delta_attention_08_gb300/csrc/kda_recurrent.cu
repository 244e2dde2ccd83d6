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
// One CTA owns one (sequence, head).  Its 512 threads hold the fp32 state in
// registers: thread (v, part) holds S[k][v] for the 32 channels k of its part,
// so every column v evolves in four neighbouring threads and the two dot
// products per token reduce over two shuffles.
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kRecThreads = 512;
constexpr int kPart = 32;  // state channels per thread
constexpr float kLog2eR = 1.4426950408889634f;

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Block-wide sum of one value per thread among the first 128 threads (4 warps).
__device__ __forceinline__ float sum128(float x, float* red, int tid) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if ((tid & 31) == 0) red[tid >> 5] = x;
  asm volatile("bar.sync 1, 128;" ::: "memory");
  const float s = (red[0] + red[1]) + (red[2] + red[3]);
  return s;
}

}  // namespace

__global__ void __launch_bounds__(kRecThreads, 1) kda_recurrent_kernel(const RecParams p) {
  __shared__ float s_k[2][128], s_q[2][128], s_a[2][128], s_beta[2];
  __shared__ float s_red[2][2][4];
  const int tid = threadIdx.x;
  const int n = (int)blockIdx.x / p.H, h = (int)blockIdx.x % p.H;
  const int H = p.H;
  int64_t bos, eos;
  if (p.cu_seqlens) {
    bos = p.cu_seqlens[n];
    eos = p.cu_seqlens[n + 1];
  } else {
    bos = (int64_t)n * p.seq_len;
    eos = bos + p.seq_len;
  }
  if (bos < 0 || eos < bos || eos > p.total_tokens || (p.cu_seqlens && n == 0 && bos != 0) ||
      (p.cu_seqlens && n == p.N - 1 && eos != p.total_tokens)) {
    if (tid == 0) atomicOr(p.status, kDevStatusBadSeqlens);
    return;
  }
  const int v = tid >> 2, part = tid & 3;  // state column v, channels kPart*part ..
  constexpr int64_t kSlot = (int64_t)kHeadDim * kHeadDim;
  const int64_t soff = ((int64_t)n * H + h) * kSlot + (int64_t)v * kHeadDim + kPart * part;

  // ---- state: S[k][v] for k in this part, stored at state[n][h][v][k]
  float S[kPart];
  if (p.init_state == nullptr) {
#pragma unroll
    for (int i = 0; i < kPart; ++i) S[i] = 0.f;
  } else if (p.state_bf16) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.init_state) + soff);
#pragma unroll
    for (int i = 0; i < kPart / 8; ++i) {
      const uint4 w = src[i];
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        S[8 * i + 2 * e] = __uint_as_float(u[e] << 16);
        S[8 * i + 2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
      }
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.init_state) + soff);
#pragma unroll
    for (int i = 0; i < kPart / 4; ++i) {
      const float4 w = src[i];
      S[4 * i] = w.x; S[4 * i + 1] = w.y; S[4 * i + 2] = w.z; S[4 * i + 3] = w.w;
    }
  }

  // per-channel gate constants (threads 0..127 own channel c = tid)
  const int c = tid & 127;
  const float nea = -expf(p.A_log[h]) * kLog2eR;
  const float ndb = nea * p.dt_bias[h * kHeadDim + c];
  const float lb2 = p.lower_bound * kLog2eR;
  const int64_t rstride = (int64_t)H * kHeadDim;

#pragma unroll 1
  for (int64_t t = bos; t < eos; ++t) {
    const int b = (int)(t - bos) & 1;  // double-buffered token vectors: one barrier per token
    const int64_t row = t * rstride + (int64_t)h * kHeadDim;
    if (tid < 128) {
      // gate, l2 norms and beta of token t
      const float kx = bf16_to_f(p.k[row + c]), qx = bf16_to_f(p.q[row + c]);
      const float gx = bf16_to_f(p.g[row + c]);
      const float la = lb2 * rcp_approx(1.0f + ex2_approx(fmaf(nea, gx, ndb)));
      const float kk = sum128(kx * kx, s_red[b][0], tid);
      const float qq = sum128(qx * qx, s_red[b][1], tid);
      s_k[b][c] = kx * rsqrtf(kk + 1e-6f);
      s_q[b][c] = qx * rsqrtf(qq + 1e-6f);
      s_a[b][c] = ex2_approx(la);
      if (tid == 0) {
        const float bx = bf16_to_f(p.beta[t * H + h]);
        s_beta[b] = rcp_approx(1.0f + ex2_approx(-bx * kLog2eR));
      }
    }
    __syncthreads();
    const float* kh = s_k[b] + kPart * part;
    const float* qh = s_q[b] + kPart * part;
    const float* ah = s_a[b] + kPart * part;
    // S <- Diag(alpha) S ; d = (S^T k)[v]
    float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kPart; i += 2) {
      const float2 s2 = f2mul(make_float2(ah[i], ah[i + 1]), make_float2(S[i], S[i + 1]));
      S[i] = s2.x;
      S[i + 1] = s2.y;
      d2 = f2fma(s2, make_float2(kh[i], kh[i + 1]), d2);
    }
    float d = d2.x + d2.y;
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    const float u = s_beta[b] * (bf16_to_f(p.v[row + v]) - d);
    // S <- S + k u^T ; o = (S^T q)[v]
    const float2 u2 = make_float2(u, u);
    float2 o2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kPart; i += 2) {
      const float2 s2 = f2fma(make_float2(kh[i], kh[i + 1]), u2, make_float2(S[i], S[i + 1]));
      S[i] = s2.x;
      S[i + 1] = s2.y;
      o2 = f2fma(s2, make_float2(qh[i], qh[i + 1]), o2);
    }
    float o = o2.x + o2.y;
    o += __shfl_xor_sync(0xffffffffu, o, 1);
    o += __shfl_xor_sync(0xffffffffu, o, 2);
    if (part == 0) {
      const __nv_bfloat16 ob = __float2bfloat16_rn(p.scale * o);
      p.out[row + v] = *reinterpret_cast<const uint16_t*>(&ob);
    }
  }

  if (p.final_state) {
    if (p.state_bf16) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.final_state) + soff);
#pragma unroll
      for (int i = 0; i < kPart / 8; ++i) {
        uint32_t u[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(S[8 * i + 2 * e], S[8 * i + 2 * e + 1]);
          u[e] = *reinterpret_cast<uint32_t*>(&h2);
        }
        dst[i] = make_uint4(u[0], u[1], u[2], u[3]);
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.final_state) + soff);
#pragma unroll
      for (int i = 0; i < kPart / 4; ++i)
        dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
    }
  }
}

cudaError_t launch_recurrent(const RecParams& p, int64_t grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  kda_recurrent_kernel<<<(unsigned)grid, kRecThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
