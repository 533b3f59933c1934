// Passes 1 and 2 of the Megatron distributed-optimizer flow with global-norm
// clipping ("07 · 显存模型", section 2.1 item 1: the reduce-scatter result
// lands in the rank's own slice of its grad buffer; the clipping rule itself
// is PyTorch's clip_grad_norm_, the pages being silent on it).  Pass 3, the
// clipped AdamW + cast + all-gather, is sharded_step_kernel<..., kClip> in
// fsp_kernels.cuh.
//
//  * rs_writeback_norm_kernel<N_s, N_r>: one CTA per tile; reduce-scatter into
//    the owners' slices and the tile's sum of squares.
//  * norm_block_sums_kernel, norm_finalize_kernel: the tiles' sums added in an
//    order fixed by the plan; the norm and the clip coefficient.
#pragma once

#include <cstdint>

#include "fsp_args.h"
#include "fsp_kernels.cuh"

namespace fsp {

// ---- distributed-optimizer pass 1: reduce-scatter into the owner's slice + norm ----

// A sum of squares carried as an unevaluated pair of floats, hi + lo, in about
// twice fp32's precision: the Dot2 scheme of Ogita, Rump and Oishi ("Accurate
// sum and dot product", SIAM J. Sci. Comput. 26(6), 2005).  Each square is
// split exactly into p + e (p = fl(x x), e = fma(x, x, -p)); p joins hi through
// Knuth's TwoSum, whose rounding error goes to lo together with e.  The _rn
// intrinsics keep the compiler from fusing these steps into FMAs.  GB300 runs
// fp32 far faster than fp64, so the per-element work stays off the fp64 pipe.
struct SumSq2 {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float p = __fmul_rn(x, x);
    const float e = fmaf(x, x, -p);
    const float s = __fadd_rn(hi, p);
    const float bp = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
  }
  __device__ __forceinline__ double value() const { return double(hi) + double(lo); }
};

// Every element's averaged gradient (rank-ordered fp32 fold / N_d) is written
// into its owner's slice of that rank's own grad buffer (fp32; per-parameter
// tensors: of the owner's tensor, bases from the registered table), and each CTA
// leaves the sum of squares of the elements it reduced in partials[cta]: each
// thread's in SumSq2, the CTA's threads added in fp64 in a fixed order.
// Launched with one CTA per tile: one partial per tile, a grouping fixed by the
// plan alone.  NS x NR ranks known at compile time (NS = 0: a.n_shard x a.n_rep
// at run time); NR = 1 is FSDP2 / DistOpt.  HSDP (NR > 1): each replica group's
// ranks are folded in order, then the groups' sums in group order - the
// all-reduce across groups - and the result is written to the owner in every
// group; the tiles cover the first group only, so each element's square is
// counted once.

// The grouped fold of element f over the ranks' bases gb (ns ranks in each of nr groups).
__device__ __forceinline__ float fold1(const void* const* gb, int64_t f, int ns, int nr) {
  float acc = 0.f;
  for (int r = 0; r < nr; ++r) {
    float part = 0.f;
    for (int j = 0; j < ns; ++j) part += GradIO<float>::load1(gb[r * ns + j], f);
    acc = r == 0 ? part : acc + part;
  }
  return acc;
}

// The grouped fold of N = NS x NR loaded values (rank r * NS + j at x[r * NS + j]).
template <int NS, int NR>
__device__ __forceinline__ float4 fold4(const float4* x) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NS; ++j) add4(part, x[r * NS + j]);
    if (r == 0)
      acc = part;
    else
      add4(acc, part);
  }
  return acc;
}

// One tile of pass 1 with rank bases gb.
template <int NS, int NR>
__device__ __forceinline__ void rs_writeback_tile(const StepArgs& a, const Tile& tile, const void* const* gb,
                                                  SumSq2& sq) {
  const int ns = NS > 0 ? NS : a.n_shard, nr = NS > 0 ? NR : a.n_rep;
  const int n = ns * nr;
  const int64_t f0 = tile.full_begin, len = tile.len;
  const int64_t head = min(len, (4 - (f0 & 3)) & 3);
  const int64_t groups = (len - head) >> 2;
  const int64_t tail = head + groups * 4;
  int64_t i0 = threadIdx.x;
  if constexpr (NS > 0) {
    // two groups per round: every load of both before either store (the owners'
    // slices alias rank buffers, so the compiler would not reorder)
    constexpr int N = NS * NR;
    for (; i0 + kGenericThreads < groups; i0 += 2 * kGenericThreads) {
      const int64_t fa = f0 + head + 4 * i0, fb = fa + 4 * kGenericThreads;
      float4 xa[N], xb[N];
#pragma unroll
      for (int q = 0; q < N; ++q) {
        xa[q] = GradIO<float>::load4(gb[q], fa);
        xb[q] = GradIO<float>::load4(gb[q], fb);
      }
      float4 acc = fold4<NS, NR>(xa), acb = fold4<NS, NR>(xb);
      acc.x = acc.x / float(N);
      acc.y = acc.y / float(N);
      acc.z = acc.z / float(N);
      acc.w = acc.w / float(N);
      acb.x = acb.x / float(N);
      acb.y = acb.y / float(N);
      acb.z = acb.z / float(N);
      acb.w = acb.w / float(N);
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float* own = static_cast<float*>(const_cast<void*>(gb[r * NS + tile.rank]));
        *reinterpret_cast<float4*>(own + fa) = acc;
        *reinterpret_cast<float4*>(own + fb) = acb;
      }
      sq.add(acc.x);
      sq.add(acc.y);
      sq.add(acc.z);
      sq.add(acc.w);
      sq.add(acb.x);
      sq.add(acb.y);
      sq.add(acb.z);
      sq.add(acb.w);
    }
  }
  for (int64_t i = i0; i < groups; i += kGenericThreads) {
    const int64_t f = f0 + head + 4 * i;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < nr; ++r) {
      float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < ns; ++j) add4(part, GradIO<float>::load4(gb[r * ns + j], f));
      if (r == 0)
        acc = part;
      else
        add4(acc, part);
    }
    acc.x = acc.x / float(n);
    acc.y = acc.y / float(n);
    acc.z = acc.z / float(n);
    acc.w = acc.w / float(n);
    for (int r = 0; r < nr; ++r)
      *reinterpret_cast<float4*>(static_cast<float*>(const_cast<void*>(gb[r * ns + tile.rank])) + f) = acc;
    sq.add(acc.x);
    sq.add(acc.y);
    sq.add(acc.z);
    sq.add(acc.w);
  }
  const int64_t n_scalar = head + (len - tail);
  if (threadIdx.x < n_scalar) {
    const int64_t f = f0 + (threadIdx.x < head ? int64_t(threadIdx.x) : tail + (threadIdx.x - head));
    const float acc = fold1(gb, f, ns, nr) / float(n);
    for (int r = 0; r < nr; ++r) static_cast<float*>(const_cast<void*>(gb[r * ns + tile.rank]))[f] = acc;
    sq.add(acc);
  }
}

template <int NS, int NR>
__global__ void __launch_bounds__(kGenericThreads) rs_writeback_norm_kernel(const __grid_constant__ StepArgs a,
                                                                            double* partials) {
  __shared__ const void* tile_gb[kMaxRanks];
  const bool per_param = a.vgrads != nullptr;
  SumSq2 sq;
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    if (per_param) {   // this tile's rank bases from the registered table
      __syncthreads();
      if (threadIdx.x < a.n_d) tile_gb[threadIdx.x] = a.vgrads[int64_t(tile.param) * a.n_d + threadIdx.x];
      __syncthreads();
      rs_writeback_tile<NS, NR>(a, tile, tile_gb, sq);
    } else {
      rs_writeback_tile<NS, NR>(a, tile, a.grads, sq);
    }
  }
  // CTA sum in a fixed order: warp shuffles, then warp 0 over the warp sums
  __shared__ double warp_sums[kGenericThreads / 32];
  double x = sq.value();
  for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
  if (threadIdx.x % 32 == 0) warp_sums[threadIdx.x / 32] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int w = 0; w < kGenericThreads / 32; ++w) total += warp_sums[w];
    partials[blockIdx.x] = total;
  }
}

// pass 2a: out[b] = the sum of partials[b * kNormBlock, (b + 1) * kNormBlock),
// four strided values per thread, then a tree over the threads (fixed order).
constexpr int kNormBlockThreads = 1024;
constexpr int kNormBlock = 4 * kNormBlockThreads;
__global__ void __launch_bounds__(kNormBlockThreads) norm_block_sums_kernel(const double* partials, int n_partials,
                                                                           double* out) {
  __shared__ double s[kNormBlockThreads];
  const int64_t base = int64_t(blockIdx.x) * kNormBlock;
  double x = 0.0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t i = base + threadIdx.x + k * kNormBlockThreads;
    if (i < n_partials) x += partials[i];
  }
  s[threadIdx.x] = x;
  __syncthreads();
  for (int w = kNormBlockThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) s[threadIdx.x] += s[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[blockIdx.x] = s[0];
}

// pass 2b: out = {sqrt(sum of partials), min(1, max_norm / (norm + 1e-6))};
// the partials are added in a fixed order for a given count (eight strided
// sums per thread, their pairwise sum, then a tree over the threads).
constexpr int kNormFinalizeThreads = 1024;
__global__ void __launch_bounds__(kNormFinalizeThreads) norm_finalize_kernel(const double* partials, int n_partials,
                                                                             float max_norm, float* out) {
  __shared__ double s[kNormFinalizeThreads];
  // eight independent sums per thread keep eight loads in flight
  constexpr int T = kNormFinalizeThreads;
  double acc[8] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
  int i = threadIdx.x;
  for (; i + 7 * T < n_partials; i += 8 * T) {
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] += partials[i + k * T];
  }
  for (; i < n_partials; i += T) acc[0] += partials[i];
  s[threadIdx.x] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  __syncthreads();
  for (int w = kNormFinalizeThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) s[threadIdx.x] += s[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double norm = sqrt(s[0]);
    const double c = double(max_norm) / (norm + 1e-6);
    out[0] = float(norm);
    out[1] = float(c < 1.0 ? c : 1.0);
  }
}

}  // namespace fsp
