// Device code of the fused sharded step (sm_103a): reduce-scatter (rank-
// ordered fp32 sum, divided by N_d) + AdamW on the fp32 shard + bf16 cast +
// all-gather, in one streaming pass over the plan's tiles.
//
// Stages: "Parallelism strategies: which state to shard", section 二.2 (ZeRO-1
// puts the optimizer between the two halves of an all-reduce) and 二.6 (HSDP);
// "FSDP2 Qwen3 Decoder Layer Walkthrough", sections "Step 0" (all-gather) and
// "Backward 简述" (reduce-scatter with averaging, then a communication-free
// update of the local shard); "07 · 显存模型", section 2.1 (fp32 master + Adam
// m/v, bf16 params, fp32 or bf16 main grads; the reduce-scatter result lands in
// the rank's own slice of its grad buffer).
//
// The step moves (N_d * sizeof(grad) + 24 N_r + 2 N_d) bytes per element at
// ~0.3 flop/byte: it is bound by HBM bandwidth and has no contraction for
// tensor cores.  Kernels:
//
//  * sharded_step_kernel<NS, NR, GradT, kClip> (N_d = NS x NR known at compile
//    time; NR > 1 is HSDP: NR replica groups of NS shard ranks, each group with
//    its own copy of the fp32 state): one CTA per SM, warp-specialised.  A
//    producer thread takes tiles in order from the launch's counter (or with
//    a fixed stride on small plans) and streams every chunk of up to E
//    aligned elements of the N_d gradient slices and the NR x 3 state slices
//    into a ring of S shared-memory stages with 1-D bulk asynchronous copies
//    (cp.async.bulk, completion counted on an mbarrier), each stage with a
//    header saying what it holds; eight consumer warps fold, update and cast
//    from shared memory, leaving the new master/m/v in place and one bf16
//    tile per replica group beside them; a storer thread writes the chunk back
//    with bulk stores: the state slices and the same bf16 tile to each rank of
//    the group (the all-gather is N_s bulk copies of one tile).  Segment edges
//    that are not 16-byte aligned take a scalar path from global memory.
//    Per-parameter tensors: the producer reads each tile's rank bases from
//    the registered table and passes them on beside the stage.
//    kClip: the clipped update of the distributed-optimizer flow - one slice,
//    the already-reduced gradient in its owner's grad buffer, scaled by the
//    clip coefficient.
//  * sharded_step_generic_kernel<GradT, kClip> (any N_d up to 64, any
//    grouping): the same arithmetic with vectorised per-thread loads/stores,
//    one CTA per tile.
//  (Passes 1 and 2 of the clipped flow - the reduce-scatter written back into
//  the owners' slices, the global norm - are in fsp_norm_kernels.cuh.)
//  * step_advance_kernel: t += 1 for steps whose update index is in device
//    memory (coeffs_of rebuilds the t-dependent scalars on the device).
//  * bounded_wait_selftest_kernel: the bounded wait against an mbarrier that
//    nothing completes.
//
// Every wait is bounded: an mbarrier wait gives up after ~2 s, records a bit in
// g_fsp_device_error, lets its own copies land and returns.  No trap, assert
// or unbounded loop exists.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fsp_args.h"
#include "fsp_internal.h"

namespace fsp {

constexpr int kGenericThreads = 256;
constexpr int kConsumerThreads = 256;                  // 8 consumer warps
constexpr int kBulkThreads = kConsumerThreads + 64;    // + producer warp + storer warp
constexpr int kBulkSmemBudget = 196608;                // stage ring, bytes
constexpr int kBulkStageBudget = 65536;                // one stage, bytes

// Device error bits (sticky until read by fsp_device_error).
constexpr unsigned kErrConsumerWait = 1u;
constexpr unsigned kErrProducerWait = 2u;
static __device__ unsigned int g_fsp_device_error = 0;

constexpr unsigned kErrStepIndex = 8u;   // *step_dev < 1 (treated as 1)

// ---- the t-dependent AdamW scalars, identically on host and device -----------------

// IEEE double operations that no compiler contraction can fuse (the host code
// is built with -ffp-contract=off), so host and device get the same bits.
__host__ __device__ __forceinline__ double dmul(double a, double b) {
#ifdef __CUDA_ARCH__
  return __dmul_rn(a, b);
#else
  return a * b;
#endif
}
__host__ __device__ __forceinline__ double dsub(double a, double b) {
#ifdef __CUDA_ARCH__
  return __dsub_rn(a, b);
#else
  return a - b;
#endif
}
__host__ __device__ __forceinline__ double ddiv(double a, double b) {
#ifdef __CUDA_ARCH__
  return __ddiv_rn(a, b);
#else
  return a / b;
#endif
}
__host__ __device__ __forceinline__ double dsqrt(double a) {
#ifdef __CUDA_ARCH__
  return __dsqrt_rn(a);
#else
  return std::sqrt(a);
#endif
}

// hi = fl(x), lo = fl(x - hi): a double as a float pair.
__host__ __device__ __forceinline__ void split_pair(double x, float& hi, float& lo) {
  hi = float(x);
  lo = float(dsub(x, double(hi)));
}

// b^t for t >= 1 by binary powering (square-and-multiply).
__host__ __device__ __forceinline__ double pow_int(double b, int64_t t) {
  double r = 1.0, p = b;
  for (uint64_t k = uint64_t(t); k != 0; k >>= 1) {
    if (k & 1u) r = dmul(r, p);
    p = dmul(p, p);
  }
  return r;
}

// Bias-correction scalars of update t: lr / (1 - beta1^t) and
// 1 / sqrt(1 - beta2^t), in double, as float pairs.
__host__ __device__ __forceinline__ void bias_scalars(Coeffs& c, float lr, int64_t t) {
  const double bc1 = dsub(1.0, pow_int(double(c.beta1), t));
  const double bc2 = dsub(1.0, pow_int(double(c.beta2), t));
  split_pair(ddiv(double(lr), bc1), c.step_hi, c.step_lo);
  split_pair(ddiv(1.0, dsqrt(bc2)), c.isb_hi, c.isb_lo);
}

// The AdamW scalars of this launch: from the host (c) or, when the update
// index lives in device memory, with the bias corrections of t = *step_dev
// computed here exactly as the host computes them.
__device__ __forceinline__ Coeffs coeffs_of(const StepArgs& a) {
  if (!a.step_dev) return a.c;
  int64_t t = *a.step_dev;
  if (t < 1) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&g_fsp_device_error, kErrStepIndex);
    t = 1;
  }
  Coeffs c = a.c;
  bias_scalars(c, a.lr, t);
  return c;
}

// Chunk size E and stage count S of the bulk kernel for NS x NR ranks (NR
// replica groups of NS shard ranks) with grads of type GradT.
// NG: gradient slices staged per chunk (N_d, or 1 for the clipped update,
// which reads the already-reduced gradient from its owner's slice).
template <int NS, int NR, typename GradT, int NG = NS * NR>
struct BulkCfg {
  static constexpr int N = NS * NR;
  // per element: NG grads, NR copies of master/m/v, NR bf16 tiles
  static constexpr int kBytesPerElem = NG * int(sizeof(GradT)) + NR * (12 + 2);
  static constexpr int E = 1024 * kBytesPerElem <= kBulkStageBudget  ? 1024
                           : 512 * kBytesPerElem <= kBulkStageBudget ? 512
                                                                     : 256;
  static constexpr int kStageBytes = E * kBytesPerElem;
  static constexpr int kS0 = kBulkSmemBudget / kStageBytes;
  static constexpr int S = kS0 > 8 ? 8 : (kS0 < 2 ? 2 : kS0);
  static constexpr int kGradOff = 0;                                  // [NG][E] GradT
  static constexpr int kStateOff = NG * E * int(sizeof(GradT));       // [NR][3][E] float
  static constexpr int kParamOff = kStateOff + NR * 3 * E * 4;        // [NR][E] bf16
  static constexpr int kBarrierBytes = 256;                           // full, computed, empty [S]
  static constexpr int kHeaderOff = kBarrierBytes;                    // StageHdr [S]
  // per-parameter tensors: each stage's N grad and N param bases, then the
  // producer's bases of its current tile
  static constexpr int kBaseOff = kBarrierBytes + 8 * 64;
  static constexpr int kBaseStride = 16 * N;
  static constexpr int kTileBaseOff = kBaseOff + S * kBaseStride;
  static constexpr int kMetaBytes = (kTileBaseOff + kBaseStride + 127) / 128 * 128;
  static constexpr int kSmemBytes = kMetaBytes + S * kStageBytes;
  static_assert(kStageBytes % 128 == 0, "stage alignment");
  static_assert(3 * S * 8 <= kBarrierBytes, "barrier area");
  static_assert(S <= 8, "header area");
};

// ---- element math -------------------------------------------------------------

// Float pairs: a value carried as hi + lo, |lo| <= ulp(hi) / 2 - about 48
// significant bits.  two_sum is Knuth's error-free sum (TAOCP vol. 2, 4.2.2),
// fast_two_sum Dekker's (|a| >= |b|, "A floating-point technique for extending
// the available precision", Numer. Math. 18, 1971), two_prod the exact product
// with an FMA.  Every step is an explicitly rounded intrinsic, so no compiler
// contraction changes them.
struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

__device__ __forceinline__ F2 fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ F2 two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}

// (a.hi + a.lo) + (b.hi + b.lo), renormalised.
__device__ __forceinline__ F2 add_pairs(F2 a, F2 b) {
  const F2 s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

// Approximate square root and reciprocal (one special-function-unit
// instruction each; about 2^-22 relative error).
__device__ __forceinline__ float sqrt_approx(float x) {
  float y;
  asm("sqrt.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// AdamW on one element with its intermediate values carried as float pairs
// (about 2^-44 of the terms' size), each result rounded once to fp32:
//   m' = b1 m + (1 - b1) G,   v' = b2 v + (1 - b2) G^2,
//   theta' = theta (1 - lr wd) - u,  u = lr / (1 - b1^t) * m' / (sqrt(v') / sqrt(1 - b2^t) + eps).
// The square root and the quotient are corrected once each from their fp32
// values: sqrt(h + l) ~ s + (h - s^2 + l) / (2 s) and n / d ~ q + (n - q d) / d,
// with the residuals taken with FMAs.  Taken only where theta' cancels.
__device__ __forceinline__ void adamw_pairs(float g, float& theta, float& m, float& v, const Coeffs& c) {
  // m' = b1 m + (1 - b1) G
  F2 gm = two_prod(c.one_minus_beta1_hi, g);
  gm.lo = __fmaf_rn(c.one_minus_beta1_lo, g, gm.lo);
  const F2 mp = add_pairs(two_prod(c.beta1, m), gm);
  // v' = b2 v + (1 - b2) G^2
  const F2 gg = two_prod(g, g);
  F2 gv = two_prod(c.one_minus_beta2_hi, gg.hi);
  gv.lo = __fmaf_rn(c.one_minus_beta2_hi, gg.lo, gv.lo);
  gv.lo = __fmaf_rn(c.one_minus_beta2_lo, gg.hi, gv.lo);
  const F2 vp = add_pairs(two_prod(c.beta2, v), gv);
  // sqrt(v')
  const float sh = __fsqrt_rn(vp.hi);
  const float sl = vp.hi > 0.f
                       ? __fmul_rn(__fadd_rn(__fmaf_rn(-sh, sh, vp.hi), vp.lo), __fmul_rn(0.5f, __frcp_rn(sh)))
                       : 0.f;
  // denominator sqrt(v') / sqrt(1 - b2^t) + eps
  F2 d = two_prod(sh, c.isb_hi);
  d.lo = __fmaf_rn(sh, c.isb_lo, d.lo);
  d.lo = __fmaf_rn(sl, c.isb_hi, d.lo);
  const F2 de = two_sum(d.hi, c.eps);
  d = fast_two_sum(de.hi, __fadd_rn(de.lo, d.lo));
  // quotient m' / denominator
  const float rc = __frcp_rn(d.hi);
  const float qh = __fmul_rn(mp.hi, rc);
  float rem = __fmaf_rn(-qh, d.hi, mp.hi);
  rem = __fadd_rn(rem, mp.lo);
  rem = __fmaf_rn(-qh, d.lo, rem);
  const float ql = __fmul_rn(rem, rc);
  // u = lr / (1 - b1^t) * quotient
  F2 u = two_prod(qh, c.step_hi);
  u.lo = __fmaf_rn(qh, c.step_lo, u.lo);
  u.lo = __fmaf_rn(ql, c.step_hi, u.lo);
  // theta' = theta (1 - lr wd) - u
  F2 td = two_prod(theta, c.decay_hi);
  td.lo = __fmaf_rn(theta, c.decay_lo, td.lo);
  const F2 r = two_sum(td.hi, -u.hi);
  theta = __fadd_rn(r.hi, __fadd_rn(r.lo, __fsub_rn(td.lo, u.lo)));
  m = mp.hi;
  v = vp.hi;
}

// theta' is taken from the fp32 evaluation when it is at least this fraction
// of the size of its terms.
constexpr float kRefineBelow = 0x1p-10f;

// AdamW on one element, in place (decoupled weight decay on the old theta,
// bias-corrected moments, eps outside the square root).  First in fp32: there
// theta' = theta (1 - lr wd) - u is off by a few fp32 ulps of its terms'
// size, |theta (1 - lr wd)| and |u|'s terms lr / (1 - b1^t) (|b1 m| +
// |(1 - b1) G|) / denominator.  Where theta' is at least 2^-10 of that size
// (all but a few elements in a million on the synthetic workloads), that is
// well under one bf16 ulp of theta'; where it cancels further, a fraction of
// an fp32 ulp of theta can be many bf16 ulps of the tiny result, and the
// element is evaluated again with float pairs (adamw_pairs), whose cast then
// stays within one bf16 ulp of the exact value's.  Every step is an explicitly
// rounded intrinsic, so every kernel and call site gets the same bits.
__device__ __forceinline__ void adamw(float g, float& theta, float& m, float& v, const Coeffs& c) {
  const float m1 = __fmaf_rn(c.beta1, m, __fmul_rn(c.one_minus_beta1_hi, g));
  const float v1 = __fmaf_rn(c.beta2, v, __fmul_rn(c.one_minus_beta2_hi, __fmul_rn(g, g)));
  const float r = rcp_approx(__fmaf_rn(sqrt_approx(v1), c.isb_hi, c.eps));
  const float u = __fmul_rn(c.step_hi, __fmul_rn(m1, r));
  const float td = __fmul_rn(theta, c.decay_hi);
  const float t1 = __fsub_rn(td, u);
  const float u_terms =
      __fmul_rn(c.step_hi, __fmul_rn(__fadd_rn(fabsf(__fmul_rn(c.beta1, m)), fabsf(__fmul_rn(c.one_minus_beta1_hi, g))), r));
  if (fabsf(t1) >= __fmul_rn(kRefineBelow, fmaxf(fabsf(td), u_terms))) {
    theta = t1;
    m = m1;
    v = v1;
    return;
  }
  adamw_pairs(g, theta, m, v, c);   // cancellation (or a NaN): the float-pair evaluation
}

__device__ __forceinline__ uint16_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

__device__ __forceinline__ uint2 pack_bf16x4(float4 t) {
  uint2 b;
  b.x = uint32_t(bf16_bits(t.x)) | (uint32_t(bf16_bits(t.y)) << 16);
  b.y = uint32_t(bf16_bits(t.z)) | (uint32_t(bf16_bits(t.w)) << 16);
  return b;
}

// ---- gradient element access ------------------------------------------------------

template <typename GradT>
struct GradIO;

template <>
struct GradIO<float> {
  static __device__ __forceinline__ float4 load4(const void* base, int64_t i) {
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
  }
  static __device__ __forceinline__ float load1(const void* base, int64_t i) {
    return __ldcs(static_cast<const float*>(base) + i);
  }
  static __device__ __forceinline__ float4 smem4(const unsigned char* base, int i) {
    return *reinterpret_cast<const float4*>(base + 4 * i);
  }
};

template <>
struct GradIO<__nv_bfloat16> {
  static __device__ __forceinline__ float4 widen(uint2 w) {
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
  }
  static __device__ __forceinline__ float4 load4(const void* base, int64_t i) {
    return widen(__ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i)));
  }
  static __device__ __forceinline__ float load1(const void* base, int64_t i) {
    const uint16_t h = __ldcs(static_cast<const unsigned short*>(base) + i);
    return __uint_as_float(uint32_t(h) << 16);
  }
  static __device__ __forceinline__ float4 smem4(const unsigned char* base, int i) {
    return widen(*reinterpret_cast<const uint2*>(base + 2 * i));
  }
};

// ---- one element from global memory (segment edges, generic kernel) -----------

// NS / NR > 0: fixed at compile time; 0: taken from the arguments.
// Reduce: inside replica group r the rank-ordered fold of its NS slices (the
// reduce-scatter), then the rank-ordered fold of the NR partial sums (the
// all-reduce across groups); with NR = 1 it is the plain rank-ordered fold.
// kClip: the clipped update - the gradient is already reduced and sits in
// its owner's slice, and is multiplied by the clip coefficient instead.
// gb / pb: rank q's grad and param bases (element f is gb[q] + f).
template <int NS, int NR, typename GradT, bool kClip>
__device__ __forceinline__ void step_one(const StepArgs& a, const void* const* gb, uint16_t* const* pb,
                                         const Coeffs& cf, int64_t f, int64_t s, int64_t owner, float coef) {
  const int ns = NS > 0 ? NS : a.n_shard;
  const int nr = NR > 0 ? NR : a.n_rep;
  float acc = 0.f;
  if (kClip) {
    acc = GradIO<GradT>::load1(gb[owner], f) * coef;
  } else {
#pragma unroll(NR > 0 ? NR : 1)
    for (int r = 0; r < nr; ++r) {
      float part = 0.f;
#pragma unroll(NS > 0 ? NS : 1)
      for (int j = 0; j < ns; ++j) part += GradIO<GradT>::load1(gb[r * ns + j], f);
      acc = r == 0 ? part : acc + part;
    }
    acc = acc / float(ns * nr);
    if (a.writeback) const_cast<float*>(static_cast<const float*>(gb[owner]))[f] = acc;   // fp32, one group
  }
#pragma unroll(NR > 0 ? NR : 1)
  for (int r = 0; r < nr; ++r) {
    const int64_t sr = s + r * a.rep_stride;
    float th = a.master[sr], mm = a.m[sr], vv = a.v[sr];
    adamw(acc, th, mm, vv, cf);
    a.master[sr] = th;
    a.m[sr] = mm;
    a.v[sr] = vv;
    if (a.reduced) a.reduced[sr] = acc;
    if (a.gather && a.param_f32) {
#pragma unroll(NS > 0 ? NS : 1)
      for (int j = 0; j < ns; ++j) reinterpret_cast<float*>(pb[r * ns + j])[f] = th;
    } else if (a.gather) {
      const uint16_t b = bf16_bits(th);
#pragma unroll(NS > 0 ? NS : 1)
      for (int j = 0; j < ns; ++j) pb[r * ns + j][f] = b;
    }
  }
}

// ---- generic kernel: per-thread vector loads and stores ---------------------------

__device__ __forceinline__ void add4(float4& a, float4 b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

// f: full index (multiple of 4); s: state index (same residue mod 16); gb /
// pb as for step_one.
template <typename GradT, bool kClip>
__device__ __forceinline__ void step_group(const StepArgs& a, const void* const* gb, uint16_t* const* pb,
                                           const Coeffs& cf, int64_t f, int64_t s, int64_t owner, float coef) {
  const int ns = a.n_shard, nr = a.n_rep;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (kClip) {
    acc = GradIO<GradT>::load4(gb[owner], f);
    acc.x *= coef;
    acc.y *= coef;
    acc.z *= coef;
    acc.w *= coef;
  } else {
    for (int r = 0; r < nr; ++r) {
      float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < ns; ++j) add4(part, GradIO<GradT>::load4(gb[r * ns + j], f));
      if (r == 0)
        acc = part;
      else
        add4(acc, part);
    }
    const float nd = float(ns * nr);
    acc.x = acc.x / nd;
    acc.y = acc.y / nd;
    acc.z = acc.z / nd;
    acc.w = acc.w / nd;
    if (a.writeback)   // fp32, one replica group
      __stcs(reinterpret_cast<float4*>(const_cast<float*>(static_cast<const float*>(gb[owner])) + f), acc);
  }
  for (int r = 0; r < nr; ++r) {
    const int64_t sr = s + r * a.rep_stride;
    float4 th = __ldcs(reinterpret_cast<const float4*>(a.master + sr));
    float4 mm = __ldcs(reinterpret_cast<const float4*>(a.m + sr));
    float4 vv = __ldcs(reinterpret_cast<const float4*>(a.v + sr));
    adamw(acc.x, th.x, mm.x, vv.x, cf);
    adamw(acc.y, th.y, mm.y, vv.y, cf);
    adamw(acc.z, th.z, mm.z, vv.z, cf);
    adamw(acc.w, th.w, mm.w, vv.w, cf);
    __stcs(reinterpret_cast<float4*>(a.master + sr), th);
    __stcs(reinterpret_cast<float4*>(a.m + sr), mm);
    __stcs(reinterpret_cast<float4*>(a.v + sr), vv);
    if (a.reduced) __stcs(reinterpret_cast<float4*>(a.reduced + sr), acc);
    if (a.gather && a.param_f32) {
      for (int j = 0; j < ns; ++j) __stcs(reinterpret_cast<float4*>(reinterpret_cast<float*>(pb[r * ns + j]) + f), th);
    } else if (a.gather) {
      const uint2 b = pack_bf16x4(th);
      for (int j = 0; j < ns; ++j) __stcs(reinterpret_cast<uint2*>(pb[r * ns + j] + f), b);
    }
  }
}

// One tile of the generic kernel with rank bases gb / pb.
template <typename GradT, bool kClip>
__device__ __forceinline__ void generic_tile(const StepArgs& a, const Coeffs& cf, const Tile& tile,
                                             const void* const* gb, uint16_t* const* pb, float coef) {
  const int64_t f0 = tile.full_begin;
  const int64_t delta = tile.state_begin - tile.full_begin;
  const int64_t len = tile.len;
  // [0, head): before the first multiple of 4; [head, tail): 4-element
  // groups; [tail, len): the remainder.
  const int64_t head = min(len, (4 - (f0 & 3)) & 3);
  const int64_t groups = (len - head) >> 2;
  const int64_t tail = head + groups * 4;
  for (int64_t i = threadIdx.x; i < groups; i += kGenericThreads) {
    const int64_t f = f0 + head + 4 * i;
    step_group<GradT, kClip>(a, gb, pb, cf, f, f + delta, tile.rank, coef);
  }
  const int64_t n_scalar = head + (len - tail);
  if (threadIdx.x < n_scalar) {
    const int64_t e = threadIdx.x < head ? int64_t(threadIdx.x) : tail + (threadIdx.x - head);
    step_one<0, 0, GradT, kClip>(a, gb, pb, cf, f0 + e, f0 + e + delta, tile.rank, coef);
  }
}

// Any N_d up to 64 and any replica grouping; full-size buffers or, with
// a.vgrads set, per-parameter tensors (each tile's bases from the tables).
// The two cases are separate paths, so that full-size buffers read their
// bases straight from the argument block.
template <typename GradT, bool kClip>
__global__ void __launch_bounds__(kGenericThreads) sharded_step_generic_kernel(const __grid_constant__ StepArgs a) {
  __shared__ const void* tile_gb[kMaxRanks];
  __shared__ uint16_t* tile_pb[kMaxRanks];
  const float coef = kClip ? a.clip[1] : 1.f;
  const Coeffs cf = coeffs_of(a);
  const bool per_param = a.vgrads != nullptr;
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    if (per_param) {
      __syncthreads();   // the previous tile's bases are no longer read
      if (threadIdx.x < a.n_d) {
        const int64_t e = int64_t(tile.param) * a.n_d + threadIdx.x;
        tile_gb[threadIdx.x] = a.vgrads[e];
        tile_pb[threadIdx.x] = a.vparams ? a.vparams[e] : nullptr;
      }
      __syncthreads();
      generic_tile<GradT, kClip>(a, cf, tile, tile_gb, tile_pb, coef);
    } else {
      generic_tile<GradT, kClip>(a, cf, tile, a.grads, a.params, coef);
    }
  }
}

// ---- PTX: mbarrier, bulk asynchronous copies, fences --------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Waits for the phase of parity `parity` to complete; false once `limit_ns`
// has passed (or after 2^30 polls, whichever comes first).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < (1u << 30); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// Programmatic dependent launch.  launch_dependents: the next launch on the
// stream that allows it may be scheduled (its CTAs take SMs as this grid's
// CTAs leave them and run up to their own grid_dependency_wait).
// grid_dependency_wait: returns once the launches this grid depends on have
// completed and their writes are visible (at once for a launch without the
// attribute).  A kernel launched with it must read and write nothing that an
// earlier launch may write before it waits.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// ever arrives at; the wait must give up after `limit_ns` and report through
// the device error word, exactly as the step kernel's waits do.
constexpr unsigned kErrSelfTest = 4u;
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_addr(&bar), 1);
  fence_mbar_init();
  if (!mbar_wait(smem_addr(&bar), 0, limit_ns)) atomicOr(&g_fsp_device_error, kErrSelfTest);
}

// t <- t + 1 after a step that read its update index from device memory.
__global__ void step_advance_kernel(int64_t* step_dev) { *step_dev += 1; }

// Aligned body [b0, b1) of a tile: 8-element (16-byte) boundaries in the full
// index, so every bulk copy starts and ends on 16 bytes for fp32 and bf16.
struct Body {
  int64_t b0, b1;
};
__device__ __forceinline__ Body tile_body(const Tile& t) {
  const int64_t end = t.full_begin + t.len;
  int64_t b0 = (t.full_begin + 7) & ~int64_t(7);
  int64_t b1 = end & ~int64_t(7);
  if (b1 < b0) b0 = b1 = end;   // no aligned body: everything is edge
  return {b0, b1};
}

// ---- bulk kernel --------------------------------------------------------------------

// What the producer puts in a stage besides the data: which chunk it holds and
// the unaligned edges of its tile (on the tile's first stage only).  len > 0:
// a chunk of len elements at full index c; 0: edges only; -1: no more work.
struct StageHdr {
  int64_t c;        // first element of the chunk (full index)
  int64_t delta;    // state index - full index, replica group 0
  int64_t edge_f0;  // the tile's first element (head edge starts here)
  int64_t edge_b1;  // end of the tile's aligned body (tail edge starts here)
  int32_t len;
  int32_t n_head;   // head / tail edge elements to do with this stage
  int32_t n_tail;
  int32_t rank;     // owner rank of the tile
};
static_assert(sizeof(StageHdr) == 48, "stage header layout");

// Next work tile of this CTA: from the launch's tile counter when there is one
// (tiles are handed out in order, so the CTAs' traffic stays in one compact,
// moving window of the buffers), else the static stride blockIdx.x + k * grid.
__device__ __forceinline__ int64_t next_tile(const StepArgs& a, int64_t k) {
  if (a.tile_ctr) return int64_t(atomicAdd(a.tile_ctr, 1ull));
  return int64_t(blockIdx.x) + k * int64_t(gridDim.x);
}

// Roles (warp index): 0-7 consumers, 8 producer (lane 0), 9 storer (lane 0).
// The producer alone picks tiles; every stage carries a StageHdr, so the
// consumers and the storer follow the producer's sequence.  Per stage s of the
// ring three mbarriers carry the hand-offs:
//   full[s]      producer -> consumers: header written, the chunk's N_d + 3 slices landed
//   computed[s]  consumers -> storer: all 8 warps left results in the stage
//   empty[s]     storer -> producer: the bulk stores have read the stage out
template <int NS, int NR, typename GradT, bool kClip>
__global__ void __launch_bounds__(kBulkThreads, 1) sharded_step_kernel(const __grid_constant__ StepArgs a) {
  constexpr int N = NS * NR;
  constexpr int NG = kClip ? 1 : N;   // gradient slices staged per chunk
  using Cfg = BulkCfg<NS, NR, GradT, NG>;
  constexpr int E = Cfg::E, S = Cfg::S, G = int(sizeof(GradT));
  constexpr int kConsumerWarps = kConsumerThreads / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* computed = full + S;
  uint64_t* empty = full + 2 * S;
  StageHdr* hdr = reinterpret_cast<StageHdr*>(smem + Cfg::kHeaderOff);
  unsigned char* stages = smem + Cfg::kMetaBytes;
  // per-parameter tensors (a.vgrads set): stage s's rank bases for its tile
  const bool per_param = a.vgrads != nullptr;
  auto stage_gb = [&](int s) { return reinterpret_cast<const void**>(smem + Cfg::kBaseOff + s * Cfg::kBaseStride); };
  auto stage_pb = [&](int s) {
    return reinterpret_cast<uint16_t**>(smem + Cfg::kBaseOff + s * Cfg::kBaseStride + 8 * N);
  };

  // The next step launch may start its prologue on the SMs this grid frees;
  // this grid's own reads of the step's buffers wait for the previous launch
  // below (the tile list and the per-parameter tables are written by no kernel).
  launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full[s]), 1);                  // producer's arrive (+ the copies' bytes)
      mbar_init(smem_addr(&computed[s]), kConsumerWarps); // one arrive per consumer warp
      mbar_init(smem_addr(&empty[s]), 1);                 // storer's arrive
    }
    fence_mbar_init();
    fence_async_smem();
  }
  __syncthreads();

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (warp == kConsumerWarps) {
    // ---------------- producer: one thread picks tiles and streams chunks into the ring ----------------
    if (lane != 0) return;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t used = 0;   // stages that ever received a header (bit s)
    bool ok = true;
    // Look-ahead.  By default, at a tile's start the next tile is claimed and
    // its descriptor requested (used a tile later).  Per-parameter tensors,
    // whose rank bases are read through a tile's descriptor, and the ZeRO-3
    // step on large plans (no all-gather stores, so nothing hides a stall):
    // tiles are claimed two ahead and descriptors loaded one ahead, and a
    // tile's bases are requested from its already-loaded descriptor one tile
    // ahead (kept in registers), so that no load's latency stalls the producer
    // at a tile's start.  Measured on Qwen3-0.6B: the per-parameter ZeRO-3 step
    // 4.54 instead of 4.98 ms, the ZeRO-3 step on full-size buffers 4.51
    // instead of 4.64; the step with the all-gather is 0.2-0.5 % faster with
    // the one-tile look-ahead.
    const bool deep = per_param || (a.tile_ctr != nullptr && !a.gather);
    if (a.tile_ctr) grid_dependency_wait();   // the counter is zeroed just before the launch
    int64_t k = 0;
    int64_t t_cur = next_tile(a, k++);
    Tile d_cur = t_cur < a.n_tiles ? a.tiles[t_cur] : Tile{};
    int64_t t_n1 = a.n_tiles, t_n2 = a.n_tiles;
    Tile d_n1{};
    if (deep && t_cur < a.n_tiles) {
      t_n1 = next_tile(a, k++);
      d_n1 = t_n1 < a.n_tiles ? a.tiles[t_n1] : Tile{};
      t_n2 = t_n1 < a.n_tiles ? next_tile(a, k++) : a.n_tiles;
    }
    const void* gb[N] = {};      // per-parameter tensors: the current tile's grad bases (registers)
    const void* gb_n1[N] = {};   // T + 1's, requested one tile ahead
    uint16_t* pb_n1[N] = {};
    uint16_t** pb = reinterpret_cast<uint16_t**>(smem + Cfg::kTileBaseOff + 8 * N);   // the current tile's
    auto fetch_bases = [&](const Tile& d) {
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const int64_t e = int64_t(d.param) * a.n_d + q;
        gb_n1[q] = a.vgrads[e];
        pb_n1[q] = a.vparams ? a.vparams[e] : nullptr;
      }
    };
    if (per_param && t_cur < a.n_tiles) {
      fetch_bases(d_cur);
#pragma unroll
      for (int q = 0; q < N; ++q) {
        gb[q] = gb_n1[q];
        pb[q] = pb_n1[q];
      }
    }
    if (!a.tile_ctr) grid_dependency_wait();   // first descriptors fetched: now the data
    for (;;) {
      const Tile tile = d_cur;
      const bool done = t_cur >= a.n_tiles;
      Tile d_n2{};
      int64_t t_n3 = a.n_tiles;
      if (!done && deep) {
        if (per_param && t_n1 < a.n_tiles) fetch_bases(d_n1);   // T + 1's descriptor landed a tile ago
        if (t_n2 < a.n_tiles) {
          d_n2 = a.tiles[t_n2];                    // T + 2's index was claimed a tile ago
          t_n3 = next_tile(a, k++);
        }
      } else if (!done) {
        t_n1 = next_tile(a, k++);
        d_n1 = t_n1 < a.n_tiles ? a.tiles[t_n1] : Tile{};
      }
      const Body body = done ? Body{0, 0} : tile_body(tile);
      const int64_t delta = tile.state_begin - tile.full_begin;
      int64_t c = body.b0;
      bool first = true;
      do {
        const int32_t len = done ? -1 : int32_t(min(int64_t(E), body.b1 - c));
        if (!mbar_wait(smem_addr(&empty[stage]), phase ^ 1u)) {
          atomicOr(&g_fsp_device_error, kErrProducerWait);
          ok = false;
          break;
        }
        StageHdr& h = hdr[stage];
        h.c = c;
        h.delta = delta;
        h.edge_f0 = tile.full_begin;
        h.edge_b1 = body.b1;
        h.len = len;
        h.n_head = first && !done ? int32_t(body.b0 - tile.full_begin) : 0;
        h.n_tail = first && !done ? int32_t(tile.full_begin + tile.len - body.b1) : 0;
        h.rank = int32_t(tile.rank);
        if (per_param && !done) {
#pragma unroll
          for (int q = 0; q < N; ++q) {
            stage_gb(stage)[q] = gb[q];
            stage_pb(stage)[q] = pb[q];
          }
        }
        const uint32_t bar = smem_addr(&full[stage]);
        if (len > 0) {
          unsigned char* st = stages + stage * Cfg::kStageBytes;
          mbar_arrive_expect_tx(bar, uint32_t(len) * uint32_t(NG * G + NR * 12));
          // (separate paths, so that full-size buffers read their bases straight from the arguments)
          if (kClip) {   // the reduced gradient, from its owner's slice
            const void* own = per_param ? stage_gb(stage)[tile.rank] : a.grads[tile.rank];
            bulk_load(smem_addr(st + Cfg::kGradOff), static_cast<const unsigned char*>(own) + c * G, len * G, bar);
          } else if (per_param) {
#pragma unroll
            for (int q = 0; q < N; ++q)
              bulk_load(smem_addr(st + Cfg::kGradOff + q * E * G), static_cast<const unsigned char*>(gb[q]) + c * G,
                        len * G, bar);
          } else {
#pragma unroll
            for (int q = 0; q < N; ++q)
              bulk_load(smem_addr(st + Cfg::kGradOff + q * E * G),
                        static_cast<const unsigned char*>(a.grads[q]) + c * G,
                        len * G, bar);
          }
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            const int64_t s = c + delta + r * a.rep_stride;
            unsigned char* sb = st + Cfg::kStateOff + r * 3 * E * 4;
            bulk_load(smem_addr(sb), a.master + s, len * 4, bar);
            bulk_load(smem_addr(sb + E * 4), a.m + s, len * 4, bar);
            bulk_load(smem_addr(sb + 2 * E * 4), a.v + s, len * 4, bar);
          }
        } else {
          mbar_arrive(bar);   // header only: edges, or the end of the work
        }
        used |= 1u << stage;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
        first = false;
        c += E;
      } while (!done && c < body.b1);
      if (!ok || done) break;
      // T + 1 becomes the current tile
      t_cur = t_n1;
      d_cur = d_n1;
      if (deep) {
        if (per_param) {
#pragma unroll
          for (int q = 0; q < N; ++q) {
            gb[q] = gb_n1[q];
            pb[q] = pb_n1[q];
          }
        }
        t_n1 = t_n2;
        d_n1 = d_n2;
        t_n2 = t_n3;
      }
    }
    if (!ok) {
      // Let every issued copy land before this CTA can retire: the most recent
      // phase used on stage s has parity `phase` for s < stage, else phase ^ 1.
      for (int s = 0; s < S; ++s)
        if (used & (1u << s)) mbar_wait(smem_addr(&full[s]), s < stage ? phase : phase ^ 1u);
    }
    return;
  }

  if (warp == kConsumerWarps + 1) {
    // ---------------- storer: one thread writes finished stages back ----------------
    if (lane != 0) return;
    grid_dependency_wait();
    int stage = 0;
    uint32_t phase = 0;
    for (;;) {
      if (!mbar_wait(smem_addr(&computed[stage]), phase)) {
        atomicOr(&g_fsp_device_error, kErrConsumerWait);
        break;
      }
      const StageHdr h = hdr[stage];
      if (h.len < 0) break;
      if (h.len > 0) {
        const uint32_t len = uint32_t(h.len);
        unsigned char* st = stages + stage * Cfg::kStageBytes;
        uint16_t* const* spb = stage_pb(stage);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          const uint32_t th_s = smem_addr(st + Cfg::kStateOff + r * 3 * E * 4);
          const uint32_t p_s = smem_addr(st + Cfg::kParamOff + r * E * 2);
          const int64_t s = h.c + h.delta + r * a.rep_stride;
          bulk_store(a.master + s, th_s, len * 4);
          bulk_store(a.m + s, th_s + E * 4, len * 4);
          bulk_store(a.v + s, th_s + 2 * E * 4, len * 4);
          if (a.gather && a.param_f32 && per_param) {   // the all-gather of the fp32 master itself
#pragma unroll
            for (int j = 0; j < NS; ++j) bulk_store(reinterpret_cast<float*>(spb[r * NS + j]) + h.c, th_s, len * 4);
          } else if (a.gather && a.param_f32) {
#pragma unroll
            for (int j = 0; j < NS; ++j)
              bulk_store(reinterpret_cast<float*>(a.params[r * NS + j]) + h.c, th_s, len * 4);
          } else if (a.gather && per_param) {   // the all-gather
#pragma unroll
            for (int j = 0; j < NS; ++j) bulk_store(spb[r * NS + j] + h.c, p_s, len * 2);
          } else if (a.gather) {
#pragma unroll
            for (int j = 0; j < NS; ++j) bulk_store(a.params[r * NS + j] + h.c, p_s, len * 2);
          }
        }
        if (sizeof(GradT) == 4 && NR == 1 && !kClip && a.writeback) {   // the owner's averaged slice
          const void* own = per_param ? stage_gb(stage)[h.rank] : a.grads[h.rank];
          bulk_store(static_cast<unsigned char*>(const_cast<void*>(own)) + h.c * G,
                     smem_addr(st + Cfg::kGradOff + h.rank * E * G), len * G);
        }
        bulk_commit();
        bulk_wait_read_all();   // the stage may be refilled once its bytes have been read out
      }
      mbar_arrive(smem_addr(&empty[stage]));
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
    bulk_wait_all();
    return;
  }

  // ---------------- consumers: fold, update, cast in shared memory ----------------
  const int tid = threadIdx.x;
  grid_dependency_wait();   // before the clip coefficient, t in device memory and the tile edges
  const float coef = kClip ? a.clip[1] : 1.f;
  const Coeffs cf = coeffs_of(a);
  int stage = 0;
  uint32_t phase = 0;
  for (;;) {
    // a warp-uniform decision, so that a wait running out ends the whole warp
    const bool landed = __all_sync(0xffffffffu, mbar_wait(smem_addr(&full[stage]), phase));
    if (!landed) return;   // the storer's bounded wait records the error
    const StageHdr h = hdr[stage];
    if (h.len >= 0) {
      // unaligned edges of the tile, straight from global memory (fewer than 16 elements)
      if (tid < h.n_head + h.n_tail) {
        const int64_t f = tid < h.n_head ? h.edge_f0 + tid : h.edge_b1 + (tid - h.n_head);
        step_one<NS, NR, GradT, kClip>(a, per_param ? stage_gb(stage) : a.grads,
                                       per_param ? stage_pb(stage) : a.params, cf, f, f + h.delta, h.rank, coef);
      }
      const int len = h.len;
      const int64_t c = h.c, delta = h.delta;
      unsigned char* st = stages + stage * Cfg::kStageBytes;
      for (int j = 4 * tid; j < len; j += 4 * kConsumerThreads) {
        // (1) reduce-scatter (inside each replica group) and all-reduce (across
        // groups): rank-ordered folds, then divide by N_d
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (kClip) {
          acc = GradIO<GradT>::smem4(st + Cfg::kGradOff, j);
          acc.x *= coef;
          acc.y *= coef;
          acc.z *= coef;
          acc.w *= coef;
        } else {
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NS; ++q)
              add4(part, GradIO<GradT>::smem4(st + Cfg::kGradOff + (r * NS + q) * E * G, j));
            if (r == 0)
              acc = part;
            else
              add4(acc, part);
          }
          acc.x = acc.x / float(N);
          acc.y = acc.y / float(N);
          acc.z = acc.z / float(N);
          acc.w = acc.w / float(N);
          // write-back (fp32, one replica group): the owner's slice in the stage now
          // holds the averaged gradient; this thread alone read its elements there
          if (sizeof(GradT) == 4 && NR == 1 && a.writeback)
            *reinterpret_cast<float4*>(st + Cfg::kGradOff + h.rank * E * G + j * G) = acc;
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          // (2) AdamW on replica r's copy of the shard, in place in the stage
          float* th_s = reinterpret_cast<float*>(st + Cfg::kStateOff + r * 3 * E * 4);
          float* m_s = th_s + E;
          float* v_s = th_s + 2 * E;
          uint16_t* p_s = reinterpret_cast<uint16_t*>(st + Cfg::kParamOff + r * E * 2);
          float4 th = *reinterpret_cast<float4*>(th_s + j);
          float4 mm = *reinterpret_cast<float4*>(m_s + j);
          float4 vv = *reinterpret_cast<float4*>(v_s + j);
          adamw(acc.x, th.x, mm.x, vv.x, cf);
          adamw(acc.y, th.y, mm.y, vv.y, cf);
          adamw(acc.z, th.z, mm.z, vv.z, cf);
          adamw(acc.w, th.w, mm.w, vv.w, cf);
          *reinterpret_cast<float4*>(th_s + j) = th;
          *reinterpret_cast<float4*>(m_s + j) = mm;
          *reinterpret_cast<float4*>(v_s + j) = vv;
          if (a.reduced) __stcs(reinterpret_cast<float4*>(a.reduced + c + delta + r * a.rep_stride + j), acc);
          // (3) bf16 cast, one tile for the replica group's ranks
          if (!a.param_f32) *reinterpret_cast<uint2*>(p_s + j) = pack_bf16x4(th);
        }
      }
      fence_async_smem();   // this thread's shared-memory writes -> visible to the bulk stores
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&computed[stage]));
    if (h.len < 0) return;
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

}  // namespace fsp
