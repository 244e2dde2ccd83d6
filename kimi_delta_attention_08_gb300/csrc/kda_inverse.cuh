// kda_inverse.cuh -- the 64 x 64 unit lower triangular inverse of the chunked
// WY form, shared by the forward kernel (kda_chunk_fwd.cu) and the chunked
// backward (kda_bwd_chunk.cu) (namespace kda::inv, internal linkage in each
// translation unit); the caller provides the fp32 matrix M ([64][kLdM], 16-byte
// aligned rows) and the bf16 output tile.
//
// Named barriers: kBarF0 (64 threads, level 0) and kBarF (kSubThreads = 128
// threads, levels 1 and 2).  The caller runs level 0 on the 64 threads with
// ftid < 64 after A is in M, then all 128 threads meet at kBarF before
// lbeta_inverse.
#ifndef KDA_INVERSE_CUH_
#define KDA_INVERSE_CUH_

#include <cuda_bf16.h>

#include "kda_ptx.cuh"

namespace kda {
namespace inv {
namespace {

using namespace ptx;

constexpr uint32_t kLdM = 68;          // fp32 row stride of M
constexpr uint32_t kBarF = 3, kBarF0 = 4;
constexpr uint32_t kSubThreads = 128;

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// Lbeta = L^{-1} Diag(beta) (bf16, [t][s] rows of the 128-byte-swizzled tile
// `lbt`) for the unit lower triangular L = I + A (64 x 64), A strictly lower
// in M[i][j] (i > j, fp32).  Blocks of 16 (a, b = 0..3):
//   level 0: D_a = (I + A_aa)^{-1}, forward substitution, one column per thread;
//            stored densely and transposed: M[16a + j][16a + i] = D_a[i][j]
//   level 1: L^{-1}_10 = -D_1 A_10 D_0,  L^{-1}_32 = -D_3 A_32 D_2
//            (transposed: L^{-1}[i][j] at M[j][i])
//   level 2: the lower-left 32 x 32 block -L22^{-1} A21 L11^{-1}:
//            T = A21 L11^{-1} (into the A21 slots, row-major), then
//            L^{-1}_2b = -D_2 T_2b,  L^{-1}_3b = -(L^{-1}_32 T_2b + D_3 T_3b)
// Levels 1 and 2 run on four warps with tf32 m16n8k8 mma.sync (fp32
// accumulate); every block of Lbeta is written as soon as it is known.
// ---------------------------------------------------------------------------
// A fragment of X[i][k] (rows r0.., cols k0..k0+7) from row-major X at p = &M[r0][k0]
__device__ __forceinline__ void frag_a_rm(const float* p, int g, int t, uint32_t (&a)[4]) {
  a[0] = to_tf32(p[g * kLdM + t]);
  a[1] = to_tf32(p[(g + 8) * kLdM + t]);
  a[2] = to_tf32(p[g * kLdM + t + 4]);
  a[3] = to_tf32(p[(g + 8) * kLdM + t + 4]);
}
// A fragment of X[i][k] stored transposed (X[i][k] at p[k * ld + i]), p = &M[k0][r0]
__device__ __forceinline__ void frag_a_tr(const float* p, int g, int t, uint32_t (&a)[4]) {
  a[0] = to_tf32(p[t * kLdM + g]);
  a[1] = to_tf32(p[t * kLdM + g + 8]);
  a[2] = to_tf32(p[(t + 4) * kLdM + g]);
  a[3] = to_tf32(p[(t + 4) * kLdM + g + 8]);
}
// B fragment of Y[k][n] (k0..k0+7, n0..n0+7) stored transposed (Y[k][n] at p[n * ld + k]), p = &M[n0][k0]
__device__ __forceinline__ void frag_b_tr(const float* p, int g, int t, uint32_t (&b)[2]) {
  b[0] = to_tf32(p[g * kLdM + t]);
  b[1] = to_tf32(p[g * kLdM + t + 4]);
}
// B fragment of row-major Y[k][n], p = &M[k0][n0]
__device__ __forceinline__ void frag_b_rm(const float* p, int g, int t, uint32_t (&b)[2]) {
  b[0] = to_tf32(p[t * kLdM + g]);
  b[1] = to_tf32(p[(t + 4) * kLdM + g]);
}
// Lbeta[row][col], Lbeta[row][col + 1] <- (x0 beta_col, x1 beta_col+1)  (col even)
__device__ __forceinline__ void lbeta_pair(uint8_t* lbt, const float* beta, int row, int col,
                                           float x0, float x1) {
  *reinterpret_cast<uint32_t*>(lbt + sw128(row, col * 2)) =
      pack_bf2(x0 * beta[col], x1 * beta[col + 1]);
}

// Level 0, run by the 64 threads that wrote A (named barrier kBarF0).
__device__ __forceinline__ void inverse_level0(float* M, int ftid) {
  float x[16];
  const int a0 = ftid >> 4, j0 = ftid & 15;
  {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float r[16];
      const float4* arow = reinterpret_cast<const float4*>(M + (16 * a0 + i) * kLdM + 16 * a0);
#pragma unroll
      for (int m4 = 0; m4 < (i + 3) / 4; ++m4) {
        const float4 w = arow[m4];
        r[4 * m4 + 0] = w.x; r[4 * m4 + 1] = w.y; r[4 * m4 + 2] = w.z; r[4 * m4 + 3] = w.w;
      }
      float acc0 = (i == j0) ? 1.f : 0.f, acc1 = 0.f;
#pragma unroll
      for (int m = 0; m < i; m += 2) {
        acc0 = fmaf(-r[m], x[m], acc0);
        if (m + 1 < i) acc1 = fmaf(-r[m + 1], x[m + 1], acc1);
      }
      x[i] = acc0 + acc1;
    }
  }
  named_sync(kBarF0, 64);  // every read of A_aa is done
  {
    // row 16a + j of the diagonal block holds column j of D_a
    float4* drow = reinterpret_cast<float4*>(M + (16 * a0 + j0) * kLdM + 16 * a0);
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 4 * i4 + e;
        v[e] = i < j0 ? 0.f : (i == j0 ? 1.f : x[i]);
      }
      drow[i4] = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
}

// Levels 1 and 2 and the Lbeta tile, after level 0 (all four factor warps).
// The strictly upper blocks of Lbeta are never read: the W / U~ MMAs skip them.
__device__ void lbeta_inverse(float* M, uint8_t* lbt, const float* beta, int ftid) {
  const int warp = ftid >> 5, lane = ftid & 31, g = lane >> 2, t = lane & 3;
  {
    // diagonal blocks of Lbeta: row 16a + i, 8 columns 16a + 8h .. from column i of M
    const int rr = ftid >> 1, hh = ftid & 1, a = rr >> 4, i = rr & 15;
    const float* col = M + (16 * a + 8 * hh) * kLdM + 16 * a + i;
    const float* bt = beta + 16 * a + 8 * hh;
    uint4 w;
    w.x = pack_bf2(col[0] * bt[0], col[kLdM] * bt[1]);
    w.y = pack_bf2(col[2 * kLdM] * bt[2], col[3 * kLdM] * bt[3]);
    w.z = pack_bf2(col[4 * kLdM] * bt[4], col[5 * kLdM] * bt[5]);
    w.w = pack_bf2(col[6 * kLdM] * bt[6], col[7 * kLdM] * bt[7]);
    *reinterpret_cast<uint4*>(lbt + sw128(rr, (16 * a + 8 * hh) * 2)) = w;
  }

  // ---- level 1: warp w -> block (1,0) (w < 2) or (3,2), 8-column half nh = w & 1
  {
    const int nh = warp & 1, cb = (warp >> 1) * 32, r = cb + 16;
    float xc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) {
      uint32_t af[4], bf[2];
      frag_a_rm(M + r * kLdM + cb + k0, g, t, af);
      frag_b_tr(M + (cb + 8 * nh) * kLdM + cb + k0, g, t, bf);
      mma_tf32_16x8x8(xc, af, bf);
    }
    // X (C layout) -> B fragments: X[8kk + t][g] and X[8kk + t + 4][g]
    const int s0 = t * 4 + (g >> 1), s1 = (t + 4) * 4 + (g >> 1);
    const bool odd = (g & 1) != 0;
    float yc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const float e0 = __shfl_sync(0xffffffffu, xc[2 * kk], s0);
      const float o0 = __shfl_sync(0xffffffffu, xc[2 * kk + 1], s0);
      const float e1 = __shfl_sync(0xffffffffu, xc[2 * kk], s1);
      const float o1 = __shfl_sync(0xffffffffu, xc[2 * kk + 1], s1);
      uint32_t af[4], bf[2];
      bf[0] = to_tf32(odd ? o0 : e0);
      bf[1] = to_tf32(odd ? o1 : e1);
      frag_a_tr(M + (r + 8 * kk) * kLdM + r, g, t, af);
      mma_tf32_16x8x8(yc, af, bf);
    }
    // L^{-1}[r + i][cb + 8nh + n] = -Y[i][n]: fp32 transposed, and Lbeta
    const int n0 = cb + 8 * nh + 2 * t;
    M[n0 * kLdM + r + g] = -yc[0];
    M[(n0 + 1) * kLdM + r + g] = -yc[1];
    M[n0 * kLdM + r + g + 8] = -yc[2];
    M[(n0 + 1) * kLdM + r + g + 8] = -yc[3];
    lbeta_pair(lbt, beta, r + g, n0, -yc[0], -yc[1]);
    lbeta_pair(lbt, beta, r + g + 8, n0, -yc[2], -yc[3]);
  }
  named_sync(kBarF, kSubThreads);

  // ---- level 2a: warp w -> rows a = 2 + (w >> 1), half nh: T_a0 and T_a1 columns
  {
    const int a = 2 + (warp >> 1), nh = warp & 1;
    float t0c[4] = {0.f, 0.f, 0.f, 0.f}, t1c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 32; k0 += 8) {
      uint32_t af[4], bf[2];
      frag_a_rm(M + (16 * a) * kLdM + k0, g, t, af);
      // column block 0 of L11^{-1}: [D_0; L^{-1}_10], transposed at M[n][k]
      frag_b_tr(M + (8 * nh) * kLdM + k0, g, t, bf);
      mma_tf32_16x8x8(t0c, af, bf);
      if (k0 >= 16) {  // column block 1 of L11^{-1}: [0; D_1]
        frag_b_tr(M + (16 + 8 * nh) * kLdM + k0, g, t, bf);
        mma_tf32_16x8x8(t1c, af, bf);
      }
    }
    named_sync(kBarF, kSubThreads);  // A_a0 / A_a1 are read by both halves
    float* T0 = M + (16 * a + g) * kLdM + 8 * nh + 2 * t;
    *reinterpret_cast<float2*>(T0) = make_float2(t0c[0], t0c[1]);
    *reinterpret_cast<float2*>(T0 + 8 * kLdM) = make_float2(t0c[2], t0c[3]);
    *reinterpret_cast<float2*>(T0 + 16) = make_float2(t1c[0], t1c[1]);
    *reinterpret_cast<float2*>(T0 + 8 * kLdM + 16) = make_float2(t1c[2], t1c[3]);
  }
  named_sync(kBarF, kSubThreads);

  // ---- level 2b: warp w -> column block b = w >> 1, half nh: L^{-1}_2b and L^{-1}_3b
  {
    const int b = warp >> 1, nh = warp & 1, nc = 16 * b + 8 * nh;
    float l2c[4] = {0.f, 0.f, 0.f, 0.f}, l3c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 32; k0 += 8) {
      uint32_t af[4], bf[2];
      frag_b_rm(M + (32 + k0) * kLdM + nc, g, t, bf);       // [T_2b; T_3b]
      frag_a_tr(M + (32 + k0) * kLdM + 48, g, t, af);       // [L^{-1}_32 | D_3]
      mma_tf32_16x8x8(l3c, af, bf);
      if (k0 < 16) {
        frag_a_tr(M + (32 + k0) * kLdM + 32, g, t, af);     // D_2
        mma_tf32_16x8x8(l2c, af, bf);
      }
    }
    const int n0 = nc + 2 * t;
    lbeta_pair(lbt, beta, 32 + g, n0, -l2c[0], -l2c[1]);
    lbeta_pair(lbt, beta, 40 + g, n0, -l2c[2], -l2c[3]);
    lbeta_pair(lbt, beta, 48 + g, n0, -l3c[0], -l3c[1]);
    lbeta_pair(lbt, beta, 56 + g, n0, -l3c[2], -l3c[3]);
  }
}

}  // namespace
}  // namespace inv
}  // namespace kda

#endif  // KDA_INVERSE_CUH_
