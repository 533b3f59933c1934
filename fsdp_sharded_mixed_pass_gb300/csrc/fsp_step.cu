// The fused sharded step for sm_103a: reduce-scatter (rank-ordered fp32 sum,
// averaged by N_d) + AdamW on the fp32 shard + bf16 cast + all-gather, in one
// streaming pass over the plan's tiles.
//
// Stages: "Parallelism strategies: which state to shard", section 二.2 (ZeRO-1
// puts the optimizer between the two halves of an all-reduce); "FSDP2 Qwen3
// Decoder Layer Walkthrough", sections "Step 0" (all-gather) and "Backward 简述"
// (reduce-scatter with averaging, then a communication-free update of the
// local shard); "07 · 显存模型", section 2.1 (fp32 master + Adam m/v, bf16
// params, fp32 or bf16 main grads).
//
// Design: the step moves (N_d * sizeof(grad) + 24 + 2 N_d) bytes per element
// at ~0.3 flop/byte, so it is bound by HBM bandwidth and uses no tensor cores.
// A persistent grid (a multiple of the SM count) walks fixed 4096-element
// tiles round-robin; inside a tile each thread handles 4-element groups with
// 16-byte (fp32) or 8-byte (bf16) vector accesses, so a warp touches 512 or
// 256 contiguous bytes of each of the 2 N_d + 3 streams per access.  Streaming
// cache hints (.cs) keep the once-touched data from displacing anything in L2.
// Nothing waits on anything: there are no barriers, atomics or spin loops.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <string>
#include <vector>

#include "fsp_internal.h"

namespace fsp {
namespace {

constexpr int kThreads = 256;

// Scalars of one AdamW update, from the fp32 hyper-parameters and t in double.
struct Coeffs {
  float beta1, one_minus_beta1;
  float beta2, one_minus_beta2;
  float decay;          // 1 - lr * weight_decay
  float step_size;      // lr / (1 - beta1^t)
  float inv_sqrt_bc2;   // 1 / sqrt(1 - beta2^t)
  float eps;
};

struct StepArgs {
  const void* grads[kMaxRanks];
  uint16_t* params[kMaxRanks];
  float* master;
  float* m;
  float* v;
  float* reduced;   // averaged shard gradient (state layout); nullptr in production
  const Tile* tiles;
  int64_t n_tiles;
  int n_d;
  Coeffs c;
};

// ---- element math ---------------------------------------------------------

// AdamW on one element: updates m, v, theta in place (fp32).
__device__ __forceinline__ void adamw(float g, float& theta, float& m, float& v, const Coeffs& c) {
  m = fmaf(c.beta1, m, c.one_minus_beta1 * g);
  v = fmaf(c.beta2, v, c.one_minus_beta2 * (g * g));
  const float denom = fmaf(sqrtf(v), c.inv_sqrt_bc2, c.eps);
  theta = fmaf(theta, c.decay, -(c.step_size * (m / denom)));
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ---- loads / stores -------------------------------------------------------

template <typename GradT> struct GradIO;

template <> struct GradIO<float> {
  static __device__ __forceinline__ float4 load4(const void* base, int64_t i) {
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
  }
  static __device__ __forceinline__ float load1(const void* base, int64_t i) {
    return __ldcs(static_cast<const float*>(base) + i);
  }
};

template <> struct GradIO<__nv_bfloat16> {
  static __device__ __forceinline__ float4 load4(const void* base, int64_t i) {
    const uint2 w = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i));
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
  }
  static __device__ __forceinline__ float load1(const void* base, int64_t i) {
    const uint16_t h = __ldcs(static_cast<const unsigned short*>(base) + i);
    return __uint_as_float(uint32_t(h) << 16);
  }
};

// ---- one 4-element group and one scalar element ---------------------------

// f: full index (multiple of 4); s: state index (same residue mod 16).
template <int NT, typename GradT>
__device__ __forceinline__ void step_group(const StepArgs& a, int n, int64_t f, int64_t s) {
  // (1) reduce-scatter: left fold in rank order, then divide by N_d
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int q = 0; q < (NT > 0 ? NT : kMaxRanks); ++q) {
    if (NT == 0 && q >= n) break;
    const float4 g = GradIO<GradT>::load4(a.grads[q], f);
    acc.x += g.x;
    acc.y += g.y;
    acc.z += g.z;
    acc.w += g.w;
  }
  const float nd = float(NT > 0 ? NT : n);
  acc.x = acc.x / nd;
  acc.y = acc.y / nd;
  acc.z = acc.z / nd;
  acc.w = acc.w / nd;

  // (2) AdamW on the shard
  float4 th = __ldcs(reinterpret_cast<const float4*>(a.master + s));
  float4 mm = __ldcs(reinterpret_cast<const float4*>(a.m + s));
  float4 vv = __ldcs(reinterpret_cast<const float4*>(a.v + s));
  adamw(acc.x, th.x, mm.x, vv.x, a.c);
  adamw(acc.y, th.y, mm.y, vv.y, a.c);
  adamw(acc.z, th.z, mm.z, vv.z, a.c);
  adamw(acc.w, th.w, mm.w, vv.w, a.c);
  __stcs(reinterpret_cast<float4*>(a.master + s), th);
  __stcs(reinterpret_cast<float4*>(a.m + s), mm);
  __stcs(reinterpret_cast<float4*>(a.v + s), vv);
  if (a.reduced) __stcs(reinterpret_cast<float4*>(a.reduced + s), acc);

  // (3) bf16 cast + all-gather into every rank's buffer
  uint2 b;
  b.x = uint32_t(bf16_bits(th.x)) | (uint32_t(bf16_bits(th.y)) << 16);
  b.y = uint32_t(bf16_bits(th.z)) | (uint32_t(bf16_bits(th.w)) << 16);
#pragma unroll
  for (int q = 0; q < (NT > 0 ? NT : kMaxRanks); ++q) {
    if (NT == 0 && q >= n) break;
    __stcs(reinterpret_cast<uint2*>(a.params[q] + f), b);
  }
}

template <int NT, typename GradT>
__device__ __forceinline__ void step_one(const StepArgs& a, int n, int64_t f, int64_t s) {
  float acc = 0.f;
#pragma unroll
  for (int q = 0; q < (NT > 0 ? NT : kMaxRanks); ++q) {
    if (NT == 0 && q >= n) break;
    acc += GradIO<GradT>::load1(a.grads[q], f);
  }
  acc = acc / float(NT > 0 ? NT : n);
  float th = a.master[s], mm = a.m[s], vv = a.v[s];
  adamw(acc, th, mm, vv, a.c);
  a.master[s] = th;
  a.m[s] = mm;
  a.v[s] = vv;
  if (a.reduced) a.reduced[s] = acc;
  const uint16_t b = bf16_bits(th);
#pragma unroll
  for (int q = 0; q < (NT > 0 ? NT : kMaxRanks); ++q) {
    if (NT == 0 && q >= n) break;
    a.params[q][f] = b;
  }
}

// ---- the kernel -------------------------------------------------------------

// NT > 0: N_d fixed at compile time; NT == 0: N_d = a.n_d (up to 64).
template <int NT, typename GradT>
__global__ void __launch_bounds__(kThreads) sharded_step_kernel(const __grid_constant__ StepArgs a) {
  const int n = NT > 0 ? NT : a.n_d;
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    const int64_t f0 = tile.full_begin;
    const int64_t delta = tile.state_begin - tile.full_begin;
    const int64_t len = tile.len;
    // [0, head): before the first multiple of 4; [head, tail): 4-element
    // groups; [tail, len): the remainder.
    const int64_t head = min(len, (4 - (f0 & 3)) & 3);
    const int64_t groups = (len - head) >> 2;
    const int64_t tail = head + groups * 4;
    for (int64_t i = threadIdx.x; i < groups; i += kThreads) {
      const int64_t f = f0 + head + 4 * i;
      step_group<NT, GradT>(a, n, f, f + delta);
    }
    const int64_t n_scalar = head + (len - tail);
    if (threadIdx.x < n_scalar) {
      const int64_t e = threadIdx.x < head ? int64_t(threadIdx.x) : tail + (threadIdx.x - head);
      step_one<NT, GradT>(a, n, f0 + e, f0 + e + delta);
    }
  }
}

// ---- host side -------------------------------------------------------------

using KernelFn = void (*)(StepArgs);

template <typename GradT, int... Ns>
struct KernelTable {
  static KernelFn get(int n) {
    KernelFn fn = sharded_step_kernel<0, GradT>;
    ((n == Ns ? (fn = sharded_step_kernel<Ns, GradT>, 0) : 0), ...);
    return fn;
  }
};
using F32Kernels = KernelTable<float, 1, 2, 3, 4, 5, 6, 7, 8, 12, 16>;
using BF16Kernels = KernelTable<__nv_bfloat16, 1, 2, 3, 4, 5, 6, 7, 8, 12, 16>;

std::string cuda_msg(const char* what, cudaError_t e) {
  return std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
}

// Whether [ptr, ptr + bytes) lies inside one live allocation of the driver.
fsp_status check_allocation(const void* ptr, size_t bytes, const char* name) {
  static PFN_cuMemGetAddressRange_v3020 get_range = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuMemGetAddressRange_v3020>(nullptr);
    return reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(fn);
  }();
  if (!get_range) return fail(FSP_ECUDA, "cannot resolve cuMemGetAddressRange");
  CUdeviceptr base = 0;
  size_t size = 0;
  if (get_range(&base, &size, reinterpret_cast<CUdeviceptr>(ptr)) != CUDA_SUCCESS)
    return fail(FSP_EINVAL, std::string(name) + " is not a live device allocation");
  const uintptr_t p = reinterpret_cast<uintptr_t>(ptr);
  if (p + bytes > uintptr_t(base) + size)
    return fail(FSP_EINVAL, std::string(name) + " allocation is smaller than the plan requires");
  return FSP_OK;
}

fsp_status device_tiles(const fsp_plan* p, const Tile** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  std::lock_guard<std::mutex> lock(p->mu);
  auto it = p->device_tiles.find(dev);
  if (it != p->device_tiles.end()) {
    *out = it->second;
    return FSP_OK;
  }
  Tile* d = nullptr;
  const size_t bytes = p->tiles.size() * sizeof(Tile);
  e = cudaMalloc(&d, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(FSP_ENOMEM, cuda_msg("cudaMalloc (tile table)", e));
  }
  e = cudaMemcpy(d, p->tiles.data(), bytes, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(d);
    return fail(FSP_ECUDA, cuda_msg("cudaMemcpy (tile table)", e));
  }
  p->device_tiles[dev] = d;
  *out = d;
  return FSP_OK;
}

int grid_for(KernelFn fn) {
  // Cached per (kernel, device): SM count times resident CTAs per SM.
  static std::mutex mu;
  static std::map<std::pair<KernelFn, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(fn, dev);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int sms = 0, per_sm = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void*>(fn), kThreads, 0);
  const int g = std::max(1, sms) * std::max(1, per_sm);
  cache[key] = g;
  return g;
}

bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.f; }

fsp_status run_step(const fsp_plan* p, const void* const* grads, int32_t dtype, float* master, float* m,
                    float* v, void* const* params, const fsp_adamw_hparams* hp, int64_t step, bool debug,
                    float* reduced, void* stream) {
  clear_error();
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  if (!grads || !params) return fail(FSP_EINVAL, "grad_bufs or param_bufs is NULL");
  if (!hp) return fail(FSP_EINVAL, "hparams is NULL");
  if (dtype != FSP_DTYPE_F32 && dtype != FSP_DTYPE_BF16) return fail(FSP_EINVAL, "unknown grad dtype");
  if (step < 1) return fail(FSP_EINVAL, "step must be >= 1 (1-based update index)");
  if (!finite_nonneg(hp->lr) || !finite_nonneg(hp->eps) || !finite_nonneg(hp->weight_decay) ||
      !finite_nonneg(hp->beta1) || !finite_nonneg(hp->beta2) || !(hp->beta1 < 1.f) || !(hp->beta2 < 1.f))
    return fail(FSP_EINVAL, "hyper-parameters out of range");

  const int n = p->n_d;
  const size_t gsize = dtype == FSP_DTYPE_F32 ? 4 : 2;
  struct Buf {
    const void* ptr;
    size_t bytes;
    std::string name;
  };
  std::vector<Buf> bufs;
  for (int q = 0; q < n; ++q) {
    bufs.push_back({grads[q], size_t(p->full_len_padded) * gsize, "grad_bufs[" + std::to_string(q) + "]"});
    bufs.push_back({params[q], size_t(p->full_len_padded) * 2, "param_bufs[" + std::to_string(q) + "]"});
  }
  const size_t sbytes = size_t(p->state_len_total) * 4;
  bufs.push_back({master, sbytes, "master"});
  bufs.push_back({m, sbytes, "exp_avg"});
  bufs.push_back({v, sbytes, "exp_avg_sq"});
  if (debug) bufs.push_back({reduced, sbytes, "reduced_grad"});
  for (const Buf& b : bufs) {
    // NULL stands for a buffer of zero bytes (e.g. every buffer of an empty plan)
    if (!b.ptr && b.bytes) return fail(FSP_EINVAL, b.name + " is NULL");
    if (reinterpret_cast<uintptr_t>(b.ptr) % 16 != 0) return fail(FSP_EINVAL, b.name + " is not 16-byte aligned");
  }
  std::vector<size_t> order(bufs.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::sort(order.begin(), order.end(), [&](size_t x, size_t y) {
    return reinterpret_cast<uintptr_t>(bufs[x].ptr) < reinterpret_cast<uintptr_t>(bufs[y].ptr);
  });
  for (size_t i = 1; i < order.size(); ++i) {
    const Buf& lo = bufs[order[i - 1]];
    const Buf& hi = bufs[order[i]];
    if (lo.ptr && lo.bytes && hi.bytes &&
        reinterpret_cast<uintptr_t>(lo.ptr) + lo.bytes > reinterpret_cast<uintptr_t>(hi.ptr))
      return fail(FSP_EINVAL, lo.name + " overlaps " + hi.name);
  }
  if (p->tiles.empty()) return FSP_OK;
  for (const Buf& b : bufs) {
    fsp_status s = check_allocation(b.ptr, b.bytes, b.name.c_str());
    if (s != FSP_OK) return s;
  }

  const Tile* tiles = nullptr;
  fsp_status s = device_tiles(p, &tiles);
  if (s != FSP_OK) return s;

  StepArgs a{};
  for (int q = 0; q < n; ++q) {
    a.grads[q] = grads[q];
    a.params[q] = static_cast<uint16_t*>(params[q]);
  }
  a.master = master;
  a.m = m;
  a.v = v;
  a.reduced = reduced;
  a.tiles = tiles;
  a.n_tiles = int64_t(p->tiles.size());
  a.n_d = n;
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, wd = hp->weight_decay;
  const double bc1 = 1.0 - std::pow(b1, double(step));
  const double bc2 = 1.0 - std::pow(b2, double(step));
  a.c.beta1 = hp->beta1;
  a.c.one_minus_beta1 = float(1.0 - b1);
  a.c.beta2 = hp->beta2;
  a.c.one_minus_beta2 = float(1.0 - b2);
  a.c.decay = float(1.0 - lr * wd);
  a.c.step_size = float(lr / bc1);
  a.c.inv_sqrt_bc2 = float(1.0 / std::sqrt(bc2));
  a.c.eps = hp->eps;

  KernelFn fn = dtype == FSP_DTYPE_F32 ? F32Kernels::get(n) : BF16Kernels::get(n);
  const int grid = int(std::min<int64_t>(grid_for(fn), a.n_tiles));
  fn<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("sharded_step_kernel launch", e));
  return FSP_OK;
}

}  // namespace
}  // namespace fsp

extern "C" fsp_status fsp_sharded_step(const fsp_plan* plan, const void* const* grad_bufs, int32_t grad_dtype,
                                       float* master, float* exp_avg, float* exp_avg_sq,
                                       void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                                       void* cuda_stream) {
  return fsp::run_step(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step, false,
                       nullptr, cuda_stream);
}

extern "C" fsp_status fsp_sharded_step_debug(const fsp_plan* plan, const void* const* grad_bufs,
                                             int32_t grad_dtype, float* master, float* exp_avg,
                                             float* exp_avg_sq, void* const* param_bufs,
                                             const fsp_adamw_hparams* hp, int64_t step, float* reduced_grad,
                                             void* cuda_stream) {
  return fsp::run_step(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step, true,
                       reduced_grad, cuda_stream);
}

// ---- entry point that allocates nothing --------------------------------------
//
// For callers that cannot call cudaMalloc: code running while a framework's
// allocator owns all device memory, inside a memory pool that must not grow,
// or on a path that must never touch the CUDA allocator.  fsp_sharded_step
// allocates one tile table per plan and device on its first call; this entry
// point instead keeps the tile list in a fixed array of device memory that
// the library declares at file scope (kNoAllocMaxTiles tiles, 8 MiB, held on
// every device that loads the library until the process exits), rewrites it
// with a stream-ordered copy on every call, and runs the same kernel on it.

namespace fsp {
namespace {

constexpr int64_t kNoAllocMaxTiles = 262144;   // 8 MiB of 32-byte tile descriptors
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) Tile g_noalloc_tiles[kNoAllocMaxTiles];

// Device address of g_noalloc_tiles on each device (the name itself is a host
// stand-in in host code), resolved once per device with that device current.
std::mutex g_noalloc_mu;
Tile* g_noalloc_addr[kNoAllocMaxDevices] = {};

fsp_status noalloc_tiles_on_current_device(Tile** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(FSP_EUNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_tiles);
    if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetSymbolAddress(g_noalloc_tiles)", e));
    g_noalloc_addr[dev] = static_cast<Tile*>(ptr);
  }
  *out = g_noalloc_addr[dev];
  return FSP_OK;
}

fsp_status run_step_noalloc(const fsp_plan* p, const void* const* grads, int32_t dtype, float* master, float* m,
                            float* v, void* const* params, const fsp_adamw_hparams* hp, int64_t step,
                            void* stream) {
  clear_error();
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  if (!grads || !params) return fail(FSP_EINVAL, "grad_bufs or param_bufs is NULL");
  if (!hp) return fail(FSP_EINVAL, "hparams is NULL");
  if (dtype != FSP_DTYPE_F32 && dtype != FSP_DTYPE_BF16) return fail(FSP_EINVAL, "unknown grad dtype");
  if (step < 1) return fail(FSP_EINVAL, "step must be >= 1 (1-based update index)");
  if (!finite_nonneg(hp->lr) || !finite_nonneg(hp->eps) || !finite_nonneg(hp->weight_decay) ||
      !finite_nonneg(hp->beta1) || !finite_nonneg(hp->beta2) || !(hp->beta1 < 1.f) || !(hp->beta2 < 1.f))
    return fail(FSP_EINVAL, "hyper-parameters out of range");
  if (int64_t(p->tiles.size()) > kNoAllocMaxTiles)
    return fail(FSP_EUNSUPPORTED, "plan needs " + std::to_string(p->tiles.size()) +
                                      " work tiles; fsp_sharded_step_noalloc holds at most 262144");

  // The same buffer checks as fsp_sharded_step, on fixed storage.
  const int n = p->n_d;
  const size_t gsize = dtype == FSP_DTYPE_F32 ? 4 : 2;
  const size_t fbytes = size_t(p->full_len_padded), sbytes = size_t(p->state_len_total) * 4;
  const void* ptrs[2 * kMaxRanks + 3];
  size_t sizes[2 * kMaxRanks + 3];
  int nb = 0;
  for (int q = 0; q < n; ++q) {
    ptrs[nb] = grads[q];
    sizes[nb++] = fbytes * gsize;
    ptrs[nb] = params[q];
    sizes[nb++] = fbytes * 2;
  }
  ptrs[nb] = master;
  sizes[nb++] = sbytes;
  ptrs[nb] = m;
  sizes[nb++] = sbytes;
  ptrs[nb] = v;
  sizes[nb++] = sbytes;
  for (int i = 0; i < nb; ++i) {
    if (!ptrs[i] && sizes[i]) return fail(FSP_EINVAL, "a buffer is NULL");
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0) return fail(FSP_EINVAL, "a buffer is not 16-byte aligned");
  }
  for (int i = 0; i < nb; ++i) {
    for (int j = i + 1; j < nb; ++j) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(ptrs[i]), b0 = reinterpret_cast<uintptr_t>(ptrs[j]);
      if (ptrs[i] && ptrs[j] && sizes[i] && sizes[j] && a0 < b0 + sizes[j] && b0 < a0 + sizes[i])
        return fail(FSP_EINVAL, "two buffers overlap");
    }
  }
  if (p->tiles.empty()) return FSP_OK;
  for (int i = 0; i < nb; ++i) {
    fsp_status s = check_allocation(ptrs[i], sizes[i], "a buffer");
    if (s != FSP_OK) return s;
  }

  Tile* tiles = nullptr;
  fsp_status s = noalloc_tiles_on_current_device(&tiles);
  if (s != FSP_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(tiles, p->tiles.data(), p->tiles.size() * sizeof(Tile), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaMemcpyAsync (tile list)", e));

  StepArgs a{};
  for (int q = 0; q < n; ++q) {
    a.grads[q] = grads[q];
    a.params[q] = static_cast<uint16_t*>(params[q]);
  }
  a.master = master;
  a.m = m;
  a.v = v;
  a.reduced = nullptr;
  a.tiles = tiles;
  a.n_tiles = int64_t(p->tiles.size());
  a.n_d = n;
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, wd = hp->weight_decay;
  const double bc1 = 1.0 - std::pow(b1, double(step));
  const double bc2 = 1.0 - std::pow(b2, double(step));
  a.c.beta1 = hp->beta1;
  a.c.one_minus_beta1 = float(1.0 - b1);
  a.c.beta2 = hp->beta2;
  a.c.one_minus_beta2 = float(1.0 - b2);
  a.c.decay = float(1.0 - lr * wd);
  a.c.step_size = float(lr / bc1);
  a.c.inv_sqrt_bc2 = float(1.0 / std::sqrt(bc2));
  a.c.eps = hp->eps;

  KernelFn fn = dtype == FSP_DTYPE_F32 ? F32Kernels::get(n) : BF16Kernels::get(n);
  const int grid = int(std::min<int64_t>(grid_for(fn), a.n_tiles));
  fn<<<grid, kThreads, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("sharded_step_kernel launch", e));
  return FSP_OK;
}

}  // namespace
}  // namespace fsp

extern "C" fsp_status fsp_sharded_step_noalloc(const fsp_plan* plan, const void* const* grad_bufs,
                                               int32_t grad_dtype, float* master, float* exp_avg,
                                               float* exp_avg_sq, void* const* param_bufs,
                                               const fsp_adamw_hparams* hp, int64_t step, void* cuda_stream) {
  return fsp::run_step_noalloc(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step,
                               cuda_stream);
}
