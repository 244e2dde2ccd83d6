// kda_plan.cu -- device-side schedule for variable-length batches and the
// segment scan (intracard context parallelism) of long sequences, plus the
// merge of per-segment transitions.
//
// The segment scan follows the split the cuLA FlashKDA port describes ("feat(kda):
// SM90 FlashKDA prefill, intracard CP, and backend dispatch", commit notes:
// split long sequences into segments; K1 once -> pre_scan -> merge -> segment K2;
// `use_intracard_cp` = "auto" | True | False).  The recurrence is affine in the
// state: over a segment, S_end = M_s S_start + B_s with M_s independent of the
// values.  Here
//   pre_scan  runs each segment twice through the chunk kernel: from the
//             identity with v = 0 (its final state is M_s) and from zero (its
//             final state is B_s); segment 0 runs from the true initial state;
//   merge     composes S_{s+1} = M_s S_s + B_s serially over segments in fp32,
//             split over row blocks of the state (rows are independent);
//   rerun     runs segments 1 .. nseg - 1 again from their merged start states,
//             writing the outputs, and the last one writes the final state
//             (segment 0 ran from the true initial state in the prescan and
//             wrote its outputs there).
// All state matrices in the workspace use the [V][K] layout of the user states.
#include <cstdio>

#include "kda_internal.h"

namespace kda {

WsLayout ws_layout(int64_t total_tokens, int32_t H) {
  WsLayout L{};
  const int64_t nchunks = (total_tokens + kChunk - 1) / kChunk;
  int64_t cap = nchunks * (int64_t)H;
  if (cap > kMaxSegHeads) cap = kMaxSegHeads;
  L.seg_cap = (int32_t)cap;
  L.max_slots = 2 * L.seg_cap;
  L.nmax = total_tokens + 1;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 256;  // header
  L.seg_units = off;
  off = up(off + sizeof(Unit) * (size_t)L.seg_cap);
  L.pre_units = off;
  off = up(off + sizeof(Unit) * (size_t)(2 * L.seg_cap));
  L.merge_units = off;
  off = up(off + sizeof(Unit) * (size_t)L.seg_cap);
  L.order = off;
  off = up(off + sizeof(int32_t) * (size_t)L.nmax);
  L.seq_info = off;
  off = up(off + sizeof(int32_t) * 4 * (size_t)L.nmax);
  L.slots = off;
  off = up(off + sizeof(float) * kHeadDim * kHeadDim * (size_t)L.max_slots);
  L.total = off;
  return L;
}

namespace {

constexpr int kPlanThreads = 1024;

__device__ void seq_bounds(const PlanParams& pp, int n, int64_t& bos, int64_t& eos) {
  if (pp.cu_seqlens) {
    bos = pp.cu_seqlens[n];
    eos = pp.cu_seqlens[n + 1];
  } else {
    bos = (int64_t)n * pp.seq_len;
    eos = bos + pp.seq_len;
  }
}

// Exclusive scan of one int per thread over the block; returns the block total.
__device__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int base = warp > 0 ? s_warp[warp - 1] : 0;
  total = s_warp[31];
  __syncthreads();
  return base + x - v;
}

}  // namespace

__global__ void __launch_bounds__(kPlanThreads, 1) kda_plan_kernel(const PlanParams pp) {
  __shared__ int s_bad;
  __shared__ unsigned long long s_total;
  __shared__ int s_segheads;
  __shared__ int s_rule;
  __shared__ unsigned long long s_red[9];
  __shared__ int s_warp[32];
  __shared__ int s_bcount[33], s_boff[33];
  const int tid = threadIdx.x;
  const int N = pp.N, H = pp.H;
  int32_t* info = pp.seq_info;
  if (tid == 0) {
    s_bad = 0;
    s_total = 0ull;
  }
  if (tid < 33) s_bcount[tid] = 0;
  __syncthreads();

  // ---- validate the prefix sum and count chunks per sequence
  unsigned long long local = 0;
  int bad = 0;
  for (int n = tid; n < N; n += kPlanThreads) {
    int64_t bos, eos;
    seq_bounds(pp, n, bos, eos);
    if (bos < 0 || eos < bos || eos > pp.total_tokens || (pp.cu_seqlens && n == 0 && bos != 0) ||
        (pp.cu_seqlens && n == N - 1 && eos != pp.total_tokens))
      bad = 1;
    const int64_t ch = bad ? 0 : (eos - bos + kChunk - 1) / kChunk;
    info[4 * n + 3] = (int32_t)ch;
    local += (unsigned long long)ch;
  }
  if (bad) atomicOr(&s_bad, 1);
  atomicAdd(&s_total, local);
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      pp.hdr->plan_ok = 0;
      pp.hdr->n_seg_units = pp.hdr->n_pre_units = pp.hdr->n_merge = 0;
      atomicOr(&pp.hdr->status, kDevStatusBadSeqlens);
    }
    return;
  }

  // ---- which sequences to split, and into segments of how many chunks
  const long long work = (long long)s_total * H;
  const long long avg = (work + pp.num_sms - 1) / pp.num_sms;
  // AUTO without a given length: two candidate lengths per split sequence, an even
  // share of the SMs (rule 0: ceil(ch H / SMs)) or the length whose reruns fill one
  // wave (rule 1: ch split into floor(SMs / H) + 1 segments).  A makespan estimate in
  // chunk periods (prescan waves, the unsplit sequences in the prescan's free slots,
  // rerun waves) picks the rule for the whole batch.
  const int nseg1 = pp.num_sms / H + 1;
  if (tid == 0) s_rule = 0;
  if (pp.cp_mode == KDA_CP_AUTO && pp.seg_chunks == 0 && nseg1 >= 2) {
    if (tid < 9) s_red[tid] = 0ull;
    __syncthreads();
    unsigned long long loc[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
    for (int n = tid; n < N; n += kPlanThreads) {
      const long long ch = info[4 * n + 3];
      if (ch >= 2 * kMinSegChunks && ch > 2 * avg) {
        const long long even = (ch * H + pp.num_sms - 1) / pp.num_sms;
        const long long L0 = even > kMinSegChunks ? even : kMinSegChunks;
        const long long c1 = (ch + nseg1 - 1) / nseg1;
        const long long L1 = c1 > kMinSegChunks ? c1 : kMinSegChunks;
        const long long Ls[2] = {L0, L1};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          long long ns = (ch + Ls[r] - 1) / Ls[r];
          if (ns < 2) ns = 1;
          if (ns > 1) {
            loc[3 * r + 0] += (unsigned long long)((2 * ns - 3) * H);  // prescan units
            loc[3 * r + 1] += (unsigned long long)((ns - 1) * H);      // rerun units
            if ((unsigned long long)Ls[r] > loc[3 * r + 2]) loc[3 * r + 2] = (unsigned long long)Ls[r];
          }
        }
      } else {
        loc[6] += (unsigned long long)(ch * H);  // unsplit chunk work
        if ((unsigned long long)ch > loc[7]) loc[7] = (unsigned long long)ch;
      }
    }
    for (int i = 0; i < 8; ++i) {
      if (i == 2 || i == 5 || i == 7) atomicMax(&s_red[i], loc[i]);
      else atomicAdd(&s_red[i], loc[i]);
    }
    __syncthreads();
    if (tid == 0) {
      const long long S = pp.num_sms, U = (long long)s_red[6], Umax = (long long)s_red[7];
      long long T[2];
      for (int r = 0; r < 2; ++r) {
        const long long P = (long long)s_red[3 * r], R = (long long)s_red[3 * r + 1];
        const long long L = (long long)s_red[3 * r + 2];
        const long long waves = (P + S - 1) / S;
        const long long room = (waves * S - P) * L;  // chunk periods left in the last wave
        long long t = waves * L;
        if (U > room) t += (U - room + S - 1) / S + Umax;
        T[r] = t + ((R + S - 1) / S) * L;
      }
      s_rule = T[1] < T[0] ? 1 : 0;
    }
  }
  __syncthreads();
  const int rule = s_rule;
  for (int lscale = 1;; lscale *= 2) {
    if (tid == 0) s_segheads = 0;
    __syncthreads();
    int mine = 0;
    for (int n = tid; n < N; n += kPlanThreads) {
      const long long ch = info[4 * n + 3];
      long long Lc = ch, nseg = 1;
      const long long even = (ch * H + pp.num_sms - 1) / pp.num_sms;  // chunks per SM-wide share
      if (pp.cp_mode == KDA_CP_FORCE && ch >= 2) {
        Lc = (pp.seg_chunks > 0 ? pp.seg_chunks : (even > 1 ? even : 1)) * (long long)lscale;
      } else if (pp.cp_mode == KDA_CP_AUTO && ch >= 2 * kMinSegChunks && ch > 2 * avg) {
        const long long c1 = (ch + nseg1 - 1) / nseg1;
        const long long base = rule ? c1 : even;
        Lc = (pp.seg_chunks > 0 ? pp.seg_chunks : (base > kMinSegChunks ? base : kMinSegChunks)) *
             (long long)lscale;
      }
      if (Lc < ch) nseg = (ch + Lc - 1) / Lc;
      if (nseg < 2) {
        nseg = 1;
        Lc = ch;
      }
      info[4 * n + 0] = (int32_t)nseg;
      info[4 * n + 1] = (int32_t)Lc;
      if (nseg > 1) mine += (int)nseg * H;
    }
    atomicAdd(&s_segheads, mine);
    __syncthreads();
    const int total = s_segheads;
    __syncthreads();
    if (total <= pp.seg_cap) break;
  }

  // ---- tables for the split sequences (sequence index order)
  int seg_carry = 0, pre_carry = 0, merge_carry = 0;
  for (int base = 0; base < N; base += kPlanThreads) {
    const int n = base + tid;
    int nseg = 1, L = 0;
    if (n < N) {
      nseg = info[4 * n + 0];
      L = info[4 * n + 1];
    }
    const bool split = nseg > 1;
    const int segu = split ? (nseg - 1) * H : 0;  // segment 0 runs in the prescan
    const int preu = split ? (2 * nseg - 3) * H : 0;
    const int mrg = (split && nseg > 2) ? H : 0;
    int tot_s, tot_p, tot_m;
    const int off_s = seg_carry + block_exclusive_scan(segu, s_warp, tot_s);
    const int off_p = pre_carry + block_exclusive_scan(preu, s_warp, tot_p);
    const int off_m = merge_carry + block_exclusive_scan(mrg, s_warp, tot_m);
    if (split) {
      info[4 * n + 2] = off_p;  // slot base of (n, 0); head h adds h * (2 nseg - 3)
      for (int h = 0; h < H; ++h) {
        Unit u;
        u.n = n;
        u.h = h;
        u.nseg = nseg;
        u.L = L;
        u.slot_base = off_p + h * (2 * nseg - 3);
        u.pad = 0;
        for (int s = 1; s < nseg; ++s) {
          u.seg = s;
          u.kind = kUnitRerun;
          pp.seg_units[off_s + h * (nseg - 1) + (s - 1)] = u;
        }
        int e = off_p + h * (2 * nseg - 3);
        u.seg = 0;
        u.kind = kUnitPreS1;
        pp.pre_units[e++] = u;
        for (int s = 1; s + 1 < nseg; ++s) {
          u.seg = s;
          u.kind = kUnitPreM;
          pp.pre_units[e++] = u;
          u.kind = kUnitPreB;
          pp.pre_units[e++] = u;
        }
        if (nseg > 2) {
          u.seg = 0;
          u.kind = kUnitRerun;
          pp.merge_units[off_m + h] = u;
        }
      }
    } else if (n < N) {
      info[4 * n + 2] = 0;
    }
    seg_carry += tot_s;
    pre_carry += tot_p;
    merge_carry += tot_m;
  }

  // ---- order of whole-sequence units: longest first (log2 buckets)
  auto bucket_of = [&](int n) {
    const int ch = info[4 * n + 3];
    return ch > 0 ? 32 - __clz(ch) : 0;  // 0..32, larger = longer
  };
  for (int n = tid; n < N; n += kPlanThreads) atomicAdd(&s_bcount[bucket_of(n)], 1);
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = 32; b >= 0; --b) {
      s_boff[b] = acc;
      acc += s_bcount[b];
    }
  }
  __syncthreads();
  for (int n = tid; n < N; n += kPlanThreads) pp.order[atomicAdd(&s_boff[bucket_of(n)], 1)] = n;

  if (tid == 0) {
    pp.hdr->n_seg_units = seg_carry;
    pp.hdr->n_pre_units = pre_carry;
    pp.hdr->n_merge = merge_carry;
    pp.hdr->plan_ok = 1;
  }
}

// S_{s+1} = M_s S_s + B_s for s = 1 .. nseg-2, in the stored [V][K] layout:
// X_{s+1} = X_s M_s^stored + B_s^stored.  One CTA owns 16 rows of X for one
// (sequence, head); rows evolve independently.
__global__ void __launch_bounds__(256) kda_merge_kernel(const MergeParams mp) {
  extern __shared__ float4 merge_smem[];
  float* Ms = reinterpret_cast<float*>(merge_smem);  // [128][128]
  float* Xs = Ms + kHeadDim * kHeadDim;               // [16][128]
  const int e = blockIdx.x / kMergeRowBlocks, rb = blockIdx.x % kMergeRowBlocks;
  if (!mp.hdr->plan_ok || e >= mp.hdr->n_merge) return;
  const Unit u = mp.merge_units[e];
  const int tid = threadIdx.x, v = tid >> 4, k0 = (tid & 15) * 8;
  const int vrow = rb * 16 + v;
  constexpr int kSlot = kHeadDim * kHeadDim;
  float x[8];
  {
    const float4* src =
        reinterpret_cast<const float4*>(mp.slots + (size_t)slot_S(u, 1) * kSlot + vrow * kHeadDim + k0);
    const float4 a = src[0], b = src[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  for (int s = 1; s + 1 < u.nseg; ++s) {
    const float4* Mg = reinterpret_cast<const float4*>(mp.slots + (size_t)slot_M(u, s) * kSlot);
    for (int i = tid; i < kSlot / 4; i += 256) merge_smem[i] = Mg[i];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) Xs[v * kHeadDim + k0 + kk] = x[kk];
    __syncthreads();
    float* Bg = mp.slots + (size_t)slot_S(u, s + 1) * kSlot + vrow * kHeadDim + k0;
    float acc[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) acc[kk] = Bg[kk];
#pragma unroll 4
    for (int j = 0; j < kHeadDim; ++j) {
      const float xv = Xs[v * kHeadDim + j];
      const float4 m0 = *reinterpret_cast<const float4*>(Ms + j * kHeadDim + k0);
      const float4 m1 = *reinterpret_cast<const float4*>(Ms + j * kHeadDim + k0 + 4);
      acc[0] = fmaf(xv, m0.x, acc[0]);
      acc[1] = fmaf(xv, m0.y, acc[1]);
      acc[2] = fmaf(xv, m0.z, acc[2]);
      acc[3] = fmaf(xv, m0.w, acc[3]);
      acc[4] = fmaf(xv, m1.x, acc[4]);
      acc[5] = fmaf(xv, m1.y, acc[5]);
      acc[6] = fmaf(xv, m1.z, acc[6]);
      acc[7] = fmaf(xv, m1.w, acc[7]);
    }
    reinterpret_cast<float4*>(Bg)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    reinterpret_cast<float4*>(Bg)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) x[kk] = acc[kk];
    __syncthreads();
  }
}

// Fold of affine state maps in the stored [V][K] layout: X <- S_in (or zero), then
// X <- X Mst_r + Bst_r for r = 0 .. R-1 (Mst, Bst: the stored transition and offset
// of piece r).  One CTA owns 16 rows of X for one state; rows evolve independently.
__global__ void __launch_bounds__(256) kda_compose_kernel(const ComposeParams cp) {
  extern __shared__ float4 compose_smem[];
  float* Ms = reinterpret_cast<float*>(compose_smem);  // [128][128]
  float* Xs = Ms + kHeadDim * kHeadDim;                 // [16][128]
  const int64_t e = blockIdx.x / kMergeRowBlocks;
  const int rb = blockIdx.x % kMergeRowBlocks;
  const int tid = threadIdx.x, v = tid >> 4, k0 = (tid & 15) * 8;
  const int vrow = rb * 16 + v;
  constexpr int64_t kSlot = (int64_t)kHeadDim * kHeadDim;
  float x[8];
  if (cp.S_in) {
    const float4* src = reinterpret_cast<const float4*>(cp.S_in + e * kSlot + vrow * kHeadDim + k0);
    const float4 a = src[0], b = src[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) x[kk] = 0.f;
  }
  for (int r = 0; r < cp.R; ++r) {
    const int64_t off = ((int64_t)r * cp.num_states + e) * kSlot;
    const float4* Mg = reinterpret_cast<const float4*>(cp.M + off);
    for (int i = tid; i < kSlot / 4; i += 256) compose_smem[i] = Mg[i];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) Xs[v * kHeadDim + k0 + kk] = x[kk];
    __syncthreads();
    const float* Bg = cp.B + off + vrow * kHeadDim + k0;
    float acc[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) acc[kk] = Bg[kk];
#pragma unroll 4
    for (int j = 0; j < kHeadDim; ++j) {
      const float xv = Xs[v * kHeadDim + j];
      const float4 m0 = *reinterpret_cast<const float4*>(Ms + j * kHeadDim + k0);
      const float4 m1 = *reinterpret_cast<const float4*>(Ms + j * kHeadDim + k0 + 4);
      acc[0] = fmaf(xv, m0.x, acc[0]);
      acc[1] = fmaf(xv, m0.y, acc[1]);
      acc[2] = fmaf(xv, m0.z, acc[2]);
      acc[3] = fmaf(xv, m0.w, acc[3]);
      acc[4] = fmaf(xv, m1.x, acc[4]);
      acc[5] = fmaf(xv, m1.y, acc[5]);
      acc[6] = fmaf(xv, m1.z, acc[6]);
      acc[7] = fmaf(xv, m1.w, acc[7]);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) x[kk] = acc[kk];
    __syncthreads();
  }
  float4* dst = reinterpret_cast<float4*>(cp.S_out + e * kSlot + vrow * kHeadDim + k0);
  dst[0] = make_float4(x[0], x[1], x[2], x[3]);
  dst[1] = make_float4(x[4], x[5], x[6], x[7]);
}

cudaError_t launch_compose(const ComposeParams& cp, cudaStream_t stream) {
  if (cp.num_states <= 0) return cudaSuccess;
  static bool attr_done[64];
  const int smem = (kHeadDim * kHeadDim + 16 * kHeadDim) * (int)sizeof(float);
  const cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void*>(kda_compose_kernel), smem, attr_done);
  if (e != cudaSuccess) return e;
  kda_compose_kernel<<<(unsigned)(cp.num_states * kMergeRowBlocks), 256, smem, stream>>>(cp);
  return cudaGetLastError();
}

cudaError_t launch_plan(const PlanParams& pp, cudaStream_t stream) {
  kda_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pp);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams& mp, int32_t seg_cap, cudaStream_t stream) {
  static bool attr_done[64];
  const int smem = (kHeadDim * kHeadDim + 16 * kHeadDim) * (int)sizeof(float);
  const cudaError_t e =
      ensure_smem_attr(reinterpret_cast<const void*>(kda_merge_kernel), smem, attr_done);
  if (e != cudaSuccess) return e;
  const int grid = (seg_cap / 2 > 0 ? seg_cap / 2 : 1) * kMergeRowBlocks;
  kda_merge_kernel<<<grid, 256, smem, stream>>>(mp);
  return cudaGetLastError();
}

}  // namespace kda
