// Host side of the fused sharded step: kernel selection and launch, argument
// checks, and the C entry points that take device buffers (the step, its
// debug / device-t / clipped / no-allocation variants, the device error word
// and the bounded-wait self-test).  The kernels are in fsp_kernels.cuh and
// fsp_norm_kernels.cuh; the host-buffer pipeline is in fsp_host.cu and the
// unshard in fsp_unshard.cu.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <string>
#include <vector>

#include "fsp_host.h"
#include "fsp_internal.h"
#include "fsp_kernels.cuh"
#include "fsp_norm_kernels.cuh"

namespace fsp {

// ---- host side -------------------------------------------------------------

// Which kernel runs for (N_d, grad dtype): the bulk-copy pipeline for the
// N_d it is instantiated for, the generic kernel otherwise.
struct KernelInfo {
  const void* fn;
  int threads;
  int smem;
  bool bulk;   // the bulk-copy pipeline (takes StepArgs::tile_ctr)
};

// (N_s, N_r) pairs with a bulk-copy instantiation: FSDP2 / DistOpt (N_r = 1)
// and the common HSDP meshes.
template <int NS, int NR>
struct Mesh {};

template <typename GradT, typename... Ms>
struct KernelTable;

template <typename GradT, int... NS, int... NR>
struct KernelTable<GradT, Mesh<NS, NR>...> {
  // kClip: the clipped update of the distributed-optimizer flow
  template <bool kClip>
  static KernelInfo get(int n_shard, int n_rep) {
    KernelInfo k{reinterpret_cast<const void*>(&sharded_step_generic_kernel<GradT, kClip>), kGenericThreads, 0,
                 false};
    ((n_shard == NS && n_rep == NR
          ? (k = KernelInfo{reinterpret_cast<const void*>(&sharded_step_kernel<NS, NR, GradT, kClip>), kBulkThreads,
                            BulkCfg<NS, NR, GradT, kClip ? 1 : NS * NR>::kSmemBytes, true},
             0)
          : 0),
     ...);
    return k;
  }
};

template <typename GradT>
using Kernels = KernelTable<GradT, Mesh<1, 1>, Mesh<2, 1>, Mesh<3, 1>, Mesh<4, 1>, Mesh<5, 1>, Mesh<6, 1>,
                            Mesh<7, 1>, Mesh<8, 1>, Mesh<12, 1>, Mesh<16, 1>, Mesh<2, 2>, Mesh<4, 2>, Mesh<8, 2>,
                            Mesh<2, 4>, Mesh<4, 4>>;
// the clipped update (fp32 grads): the same meshes
using ClipKernels = KernelTable<float, Mesh<1, 1>, Mesh<2, 1>, Mesh<3, 1>, Mesh<4, 1>, Mesh<5, 1>, Mesh<6, 1>,
                                Mesh<7, 1>, Mesh<8, 1>, Mesh<12, 1>, Mesh<16, 1>, Mesh<2, 2>, Mesh<4, 2>,
                                Mesh<8, 2>, Mesh<2, 4>, Mesh<4, 4>>;

// Pass 1 of the clipped flow for N_s x N_r ranks (the step kernel's meshes;
// others run the run-time instantiation <0, 0>).
template <typename... Ms>
struct NormKernelTable;

template <int... NS, int... NR>
struct NormKernelTable<Mesh<NS, NR>...> {
  static KernelInfo get(int n_shard, int n_rep) {
    KernelInfo k{reinterpret_cast<const void*>(&rs_writeback_norm_kernel<0, 0>), kGenericThreads, 0, false};
    ((n_shard == NS && n_rep == NR
          ? (k = KernelInfo{reinterpret_cast<const void*>(&rs_writeback_norm_kernel<NS, NR>), kGenericThreads, 0,
                            false},
             0)
          : 0),
     ...);
    return k;
  }
};
using NormKernels = NormKernelTable<Mesh<1, 1>, Mesh<2, 1>, Mesh<3, 1>, Mesh<4, 1>, Mesh<5, 1>, Mesh<6, 1>,
                                    Mesh<7, 1>, Mesh<8, 1>, Mesh<12, 1>, Mesh<16, 1>, Mesh<2, 2>, Mesh<4, 2>,
                                    Mesh<8, 2>, Mesh<2, 4>, Mesh<4, 4>>;

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
  // The driver call needs a current context on this thread; a thread that has
  // made no runtime call yet has none, so bind the current device's primary
  // context (cudaSetDevice does that, and nothing else, when it is current).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("binding the device context", e));
  CUdeviceptr base = 0;
  size_t size = 0;
  if (get_range(&base, &size, reinterpret_cast<CUdeviceptr>(ptr)) != CUDA_SUCCESS)
    return fail(FSP_EINVAL, std::string(name) + " is not a live device allocation");
  const uintptr_t p = reinterpret_cast<uintptr_t>(ptr);
  if (p + bytes > uintptr_t(base) + size)
    return fail(FSP_EINVAL, std::string(name) + " allocation is smaller than the plan requires");
  return FSP_OK;
}

// A synchronous cudaMemcpy from pageable host memory may return before its
// last bytes have reached the device (it is ordered on the legacy stream
// only); tables that kernels on any stream read later are complete once this
// returns.
cudaError_t upload_table(void* dst, const void* src, size_t bytes) {
  cudaError_t e = cudaMemcpy(dst, src, bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cudaStreamLegacy);
  return e;
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
  e = upload_table(d, p->tiles.data(), bytes);
  if (e != cudaSuccess) {
    cudaFree(d);
    return fail(FSP_ECUDA, cuda_msg("cudaMemcpy (tile table)", e));
  }
  p->device_tiles[dev] = d;
  *out = d;
  return FSP_OK;
}

// The step kernels run large plans (at least kOrderedMinTilesPerCta tiles per
// CTA) on full-size buffers with the all-gather on the plan's tiles split at
// multiples of this many elements: the CTAs, which take the tiles in order,
// then work in a narrower window of the buffers.  Measured against the plan's
// 4096-element tiles (same box, 50 steps, two runs): Qwen3-0.6B FSDP2 5.967 vs
// 6.008 ms, DistOpt 5.952 vs 5.997, HSDP 2 x 4 8.004 vs 8.054, ragged N_d = 6
// 11.818 vs 11.870, bf16 grads N_d = 16 13.458 vs 13.468, with write-back 6.330
// vs 6.369, fp32 gather 7.387 vs 7.424, N_d = 24 (per-thread kernel) 14.49 vs
// 14.62; 1024 and 1536 were 6-20 % slower, 8192 slower.  Kept on the plan's
// tiles, where 2048 measured slower: the ZeRO-3 step (4.89 vs 4.61 ms),
// per-parameter tensors (4.74 vs 4.53), the clipped flow (7.07 vs 6.83) and
// one-layer slices of 6-7 tiles per CTA (47.4 vs 46.7 and 75.9 vs 73.8 us).
constexpr int64_t kStepTileElems = 2048;
static_assert(kTileElems % kStepTileElems == 0, "step tiles split plan tiles");

std::vector<Tile> split_tiles(const std::vector<Tile>& tiles, int64_t unit) {
  std::vector<Tile> out;
  out.reserve(tiles.size() * size_t(std::max<int64_t>(1, kTileElems / unit)));
  for (const Tile& t : tiles) {
    const int64_t end = t.full_begin + t.len;
    for (int64_t f = t.full_begin; f < end;) {
      const int64_t stop = std::min(end, (f / unit + 1) * unit);
      Tile u = t;
      u.full_begin = f;
      u.state_begin = t.state_begin + (f - t.full_begin);
      u.len = int32_t(stop - f);
      out.push_back(u);
      f = stop;
    }
  }
  return out;
}

// The plan's step tiles on the current device (built and uploaded on first use).
fsp_status device_step_tiles(const fsp_plan* p, const Tile** out, int64_t* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  std::lock_guard<std::mutex> lock(p->mu);
  auto it = p->device_step_tiles.find(dev);
  if (it == p->device_step_tiles.end()) {
    const std::vector<Tile> host = split_tiles(p->tiles, kStepTileElems);
    Tile* d = nullptr;
    e = cudaMalloc(&d, std::max<size_t>(1, host.size()) * sizeof(Tile));
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(FSP_ENOMEM, cuda_msg("cudaMalloc (step tile table)", e));
    }
    e = upload_table(d, host.data(), host.size() * sizeof(Tile));
    if (e != cudaSuccess) {
      cudaFree(d);
      return fail(FSP_ECUDA, cuda_msg("cudaMemcpy (step tile table)", e));
    }
    it = p->device_step_tiles.emplace(dev, std::make_pair(d, int64_t(host.size()))).first;
  }
  *out = it->second.first;
  *n = it->second.second;
  return FSP_OK;
}

// Small plans run with a fixed stride: CTA b takes tiles b, b + grid, b +
// 2 grid, ...; tiles differ in length (segment ends), so some CTAs get more
// chunks than others and the launch waits for the busiest.  Balanced order:
// the tiles of every round [k grid, (k + 1) grid) are handed, longest first,
// to the CTAs with the fewest chunks so far (1024-element chunks, a partial
// chunk counting as one); every round still holds the same tiles, so the
// CTAs' window of the buffers is unchanged.  The last, partial round reaches
// CTAs 0 .. n - 1 only: the CTAs are renumbered so that the ones it feeds
// (the least loaded before it) are those.
int64_t tile_chunks(const Tile& t) { return (int64_t(t.len) + 1023) / 1024; }

// The most chunks any CTA takes when CTA b takes tiles b, b + grid, ...
int64_t busiest_cta_chunks(const std::vector<Tile>& tiles, int grid) {
  std::vector<int64_t> load(size_t(grid), 0);
  for (size_t i = 0; i < tiles.size(); ++i) load[i % size_t(grid)] += tile_chunks(tiles[i]);
  return load.empty() ? 0 : *std::max_element(load.begin(), load.end());
}

std::vector<Tile> balance_rounds(const std::vector<Tile>& tiles, int grid) {
  const size_t n_tiles = tiles.size(), g = size_t(grid);
  if (n_tiles <= g) return tiles;   // one round, one tile per CTA: nothing to balance
  auto chunks = tile_chunks;
  std::vector<int64_t> load(g, 0);
  std::vector<size_t> owner(n_tiles);   // virtual CTA of each tile
  std::vector<size_t> idx, cta(g);
  for (size_t k = 0; k < n_tiles; k += g) {
    const size_t n = std::min(n_tiles - k, g);
    idx.resize(n);
    for (size_t j = 0; j < n; ++j) idx[j] = k + j;
    std::stable_sort(idx.begin(), idx.end(),
                     [&](size_t x, size_t y) { return chunks(tiles[x]) > chunks(tiles[y]); });
    for (size_t b = 0; b < g; ++b) cta[b] = b;
    std::stable_sort(cta.begin(), cta.end(), [&](size_t x, size_t y) { return load[x] < load[y]; });
    for (size_t j = 0; j < n; ++j) {
      owner[idx[j]] = cta[j];
      load[cta[j]] += chunks(tiles[idx[j]]);
    }
  }
  // renumber: the CTAs of the last round's tiles first
  const size_t last = (n_tiles - 1) / g * g;
  std::vector<size_t> phys(g, g);
  size_t next = 0;
  for (size_t i = last; i < n_tiles; ++i) phys[owner[i]] = next++;
  for (size_t b = 0; b < g; ++b)
    if (phys[b] == g) phys[b] = next++;
  std::vector<Tile> out(n_tiles);
  for (size_t i = 0; i < n_tiles; ++i) out[i / g * g + phys[owner[i]]] = tiles[i];
  return out;
}

// The plan's tiles in balanced order for `grid` CTAs on the current device
// (built and uploaded on first use), or NULL where that order does not lower
// the busiest CTA's chunk count: there the plan's own order is kept (on
// Qwen3-layer-sized plans a reordering without that gain measured 2 % slower).
fsp_status device_round_tiles(const fsp_plan* p, int grid, const Tile** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  std::lock_guard<std::mutex> lock(p->mu);
  // one table per grid: a launch of another kernel of this plan may still read
  // the table of its own grid
  auto it = p->device_round_tiles.find({dev, grid});
  if (it == p->device_round_tiles.end()) {
    const std::vector<Tile> host = balance_rounds(p->tiles, grid);
    Tile* d = nullptr;
    if (busiest_cta_chunks(host, grid) < busiest_cta_chunks(p->tiles, grid)) {
      e = cudaMalloc(&d, std::max<size_t>(1, host.size()) * sizeof(Tile));
      if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(FSP_ENOMEM, cuda_msg("cudaMalloc (balanced tile table)", e));
      }
      e = upload_table(d, host.data(), host.size() * sizeof(Tile));
      if (e != cudaSuccess) {
        cudaFree(d);
        return fail(FSP_ECUDA, cuda_msg("cudaMemcpy (balanced tile table)", e));
      }
    }
    it = p->device_round_tiles.emplace(std::make_pair(dev, grid), d).first;
  }
  *out = it->second;
  return FSP_OK;
}

// Grid for a kernel on the current device: SM count times resident CTAs
// (one for the bulk kernel), after allowing its dynamic shared memory.
// Cached per (kernel, device).
fsp_status grid_for(const KernelInfo& k, int* grid) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(k.fn, dev);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *grid = it->second;
    return FSP_OK;
  }
  if (k.smem > 48 * 1024) {
    e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem);
    if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaFuncSetAttribute", e));
  }
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaDeviceGetAttribute", e));
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn, k.threads, k.smem);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaOccupancyMaxActiveBlocksPerMultiprocessor", e));
  if (per_sm < 1) return fail(FSP_ECUDA, "the step kernel cannot be resident on this device");
  *grid = sms * per_sm;
  cache[key] = *grid;
  return FSP_OK;
}

// Fills the AdamW scalars of update t (in double, as float pairs; the
// bias corrections through bias_scalars, as the kernels compute them when t
// is in device memory).
void set_coeffs(StepArgs& a, const fsp_adamw_hparams* hp, int64_t step) {
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, wd = hp->weight_decay;
  a.c.beta1 = hp->beta1;
  split_pair(dsub(1.0, b1), a.c.one_minus_beta1_hi, a.c.one_minus_beta1_lo);
  a.c.beta2 = hp->beta2;
  split_pair(dsub(1.0, b2), a.c.one_minus_beta2_hi, a.c.one_minus_beta2_lo);
  split_pair(dsub(1.0, dmul(lr, wd)), a.c.decay_hi, a.c.decay_lo);
  bias_scalars(a.c, hp->lr, step);
  a.c.eps = hp->eps;
  a.lr = hp->lr;
}

// Rank layout of the plan in the argument block.
void set_mesh(StepArgs& a, const fsp_plan* p) {
  a.n_d = p->n_d;
  a.n_rep = p->n_rep;
  a.n_shard = p->n_shard;
  a.rep_stride = p->n_rep > 1 ? p->rep_stride : 0;
}

// Pool of the launches' tile counters on the current device: 8-byte
// stream-ordered allocations, memory kept by the pool between launches.
fsp_status counter_pool(cudaMemPool_t* out) {
  static std::mutex mu;
  static std::map<int, cudaMemPool_t> pools;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  std::lock_guard<std::mutex> lock(mu);
  auto it = pools.find(dev);
  if (it != pools.end()) {
    *out = it->second;
    return FSP_OK;
  }
  cudaMemPoolProps props{};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  cudaMemPool_t pool = nullptr;
  e = cudaMemPoolCreate(&pool, &props);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaMemPoolCreate (tile counters)", e));
  uint64_t keep = ~uint64_t(0);
  e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
  if (e != cudaSuccess) {
    cudaMemPoolDestroy(pool);
    return fail(FSP_ECUDA, cuda_msg("cudaMemPoolSetAttribute (tile counters)", e));
  }
  pools[dev] = pool;
  *out = pool;
  return FSP_OK;
}

// Bulk-kernel plans with at least this many tiles per CTA hand their tiles out
// in order from a counter: with a fixed stride the CTAs drift apart over a long
// launch, their copies spread over the whole buffers, and HBM throughput drops
// (smaller plans finish before that matters).
constexpr int64_t kOrderedMinTilesPerCta = 16;
// The ZeRO-3 step of one replica group (no all-gather stores) keeps the fixed
// stride, in balanced order, up to this many tiles per CTA.  Measured against
// the counter (same box, two runs): one Qwen3-0.6B layer 129-131 vs 136-137 us
// (per-parameter tensors 130 vs 137), two layers 250-251 vs 255, one layer of
// the 1.5B bf16-gradient stack (73 tiles per CTA) 386-387 vs 397-398, four
// Qwen3-0.6B layers (103) 492 vs 492-493; with the all-gather, or for HSDP,
// the counter stays ahead from 16 tiles per CTA (one layer with the all-gather
// 172 vs 184 us, HSDP ZeRO-3 190 vs 192).
constexpr int64_t kOrderedMinTilesPerCtaZero3 = 128;

// Launches the step for argument block `a` (tiles already on the device);
// `clip`: the clipped update (a.clip set, fp32 grads, one replica group).
fsp_status launch(StepArgs& a, int32_t dtype, void* stream, bool clip, unsigned long long* fixed_ctr,
                  const fsp_plan* step_plan, bool early_start) {
  const KernelInfo k = clip                     ? ClipKernels::get<true>(a.n_shard, a.n_rep)
                       : dtype == FSP_DTYPE_F32 ? Kernels<float>::get<false>(a.n_shard, a.n_rep)
                                                : Kernels<__nv_bfloat16>::get<false>(a.n_shard, a.n_rep);
  int grid = 0;
  fsp_status s = grid_for(k, &grid);
  if (s != FSP_OK) return s;
  if (step_plan && !clip && !a.vgrads && a.gather && a.n_tiles >= kOrderedMinTilesPerCta * grid &&
      a.n_tiles == int64_t(step_plan->tiles.size())) {
    // a large plan on full-size buffers with the all-gather: the step tiles
    s = device_step_tiles(step_plan, &a.tiles, &a.n_tiles);
    if (s != FSP_OK) return s;
  }
  // The generic kernel runs one CTA per tile: the block scheduler hands the
  // tiles out in order.  The bulk kernel keeps one CTA per SM.
  const int64_t min_ordered = !a.gather && a.n_rep == 1 ? kOrderedMinTilesPerCtaZero3 : kOrderedMinTilesPerCta;
  const bool ordered = k.bulk && a.n_tiles >= min_ordered * grid;
  if (step_plan && k.bulk && !ordered && a.n_tiles > grid && a.n_tiles == int64_t(step_plan->tiles.size())) {
    // a small plan's own tiles over several rounds: the balanced order
    const Tile* balanced = nullptr;
    s = device_round_tiles(step_plan, grid, &balanced);
    if (s != FSP_OK) return s;
    if (balanced) a.tiles = balanced;
  }
  grid = int(std::min<int64_t>(k.bulk ? grid : int64_t(INT32_MAX), a.n_tiles));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  a.tile_ctr = nullptr;
  if (ordered && fixed_ctr) {
    cudaError_t e = cudaMemsetAsync(fixed_ctr, 0, sizeof(unsigned long long), st);
    if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaMemsetAsync (tile counter)", e));
    a.tile_ctr = fixed_ctr;
  } else if (ordered) {
    cudaMemPool_t pool = nullptr;
    s = counter_pool(&pool);
    if (s != FSP_OK) return s;
    void* ctr = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ctr, sizeof(unsigned long long), pool, st);
    if (e != cudaSuccess) return fail(FSP_ENOMEM, cuda_msg("cudaMallocFromPoolAsync (tile counter)", e));
    e = cudaMemsetAsync(ctr, 0, sizeof(unsigned long long), st);
    if (e != cudaSuccess) {
      cudaFreeAsync(ctr, st);
      return fail(FSP_ECUDA, cuda_msg("cudaMemsetAsync (tile counter)", e));
    }
    a.tile_ctr = static_cast<unsigned long long*>(ctr);
  }
  void* args[] = {&a};
  // The bulk kernel allows programmatic stream serialisation: launched right
  // after another kernel on the stream, its CTAs may start (set up their
  // barriers, fetch their first tile descriptors) while that kernel's last
  // CTAs finish, and wait for it on the device before touching its buffers.
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(k.threads);
  cfg.dynamicSmemBytes = size_t(k.smem);
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = k.bulk && early_start ? 1 : 0;
  cudaError_t e = cudaLaunchKernelExC(&cfg, k.fn, args);
  if (a.tile_ctr && a.tile_ctr != fixed_ctr) {
    const cudaError_t f = cudaFreeAsync(a.tile_ctr, st);
    if (e == cudaSuccess) e = f;
  }
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("sharded step kernel launch", e));
  return FSP_OK;
}

bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.f; }

fsp_status check_hparams(const fsp_adamw_hparams* hp, int64_t step) {
  if (!hp) return fail(FSP_EINVAL, "hparams is NULL");
  if (step < 1) return fail(FSP_EINVAL, "step must be >= 1 (1-based update index)");
  if (!finite_nonneg(hp->lr) || !finite_nonneg(hp->eps) || !finite_nonneg(hp->weight_decay) ||
      !finite_nonneg(hp->beta1) || !finite_nonneg(hp->beta2) || !(hp->beta1 < 1.f) || !(hp->beta2 < 1.f))
    return fail(FSP_EINVAL, "hyper-parameters out of range");
  return FSP_OK;
}

// Host-side checks shared by the device-buffer entry points: arguments,
// hyper-parameters, NULL / alignment / overlap of every buffer (the step's and
// `extra`), and - for a non-empty plan - that each lies in a live allocation.
fsp_status check_device_step(const fsp_plan* p, const void* const* grads, int32_t dtype, float* master, float* m,
                             float* v, void* const* params, const fsp_adamw_hparams* hp, int64_t step,
                             const std::vector<Buf>& extra, size_t param_size = 2) {
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  if (!grads) return fail(FSP_EINVAL, "grad_bufs is NULL");   // param_bufs NULL: no all-gather
  if (dtype != FSP_DTYPE_F32 && dtype != FSP_DTYPE_BF16) return fail(FSP_EINVAL, "unknown grad dtype");
  if (fsp_status hs = check_hparams(hp, step); hs != FSP_OK) return hs;

  const int n = p->n_d;
  const size_t gsize = dtype == FSP_DTYPE_F32 ? 4 : 2;
  std::vector<Buf> bufs;
  for (int q = 0; q < n; ++q) {
    bufs.push_back({grads[q], size_t(p->full_len_padded) * gsize, "grad_bufs[" + std::to_string(q) + "]"});
    if (params)
      bufs.push_back({params[q], size_t(p->full_len_padded) * param_size, "param_bufs[" + std::to_string(q) + "]"});
  }
  const size_t sbytes = size_t(p->state_len_total) * 4;
  bufs.push_back({master, sbytes, "master"});
  bufs.push_back({m, sbytes, "exp_avg"});
  bufs.push_back({v, sbytes, "exp_avg_sq"});
  for (const Buf& b : extra) bufs.push_back(b);
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
  return FSP_OK;
}

// Argument block for the plan's tiles on the current device.
fsp_status step_args(const fsp_plan* p, const void* const* grads, float* master, float* m, float* v,
                     void* const* params, const fsp_adamw_hparams* hp, int64_t step, StepArgs* a) {
  const Tile* tiles = nullptr;
  fsp_status s = device_tiles(p, &tiles);
  if (s != FSP_OK) return s;
  *a = StepArgs{};
  for (int q = 0; q < p->n_d; ++q) {
    a->grads[q] = grads[q];
    a->params[q] = params ? static_cast<uint16_t*>(params[q]) : nullptr;
  }
  a->gather = params ? 1 : 0;
  a->master = master;
  a->m = m;
  a->v = v;
  a->tiles = tiles;
  a->n_tiles = int64_t(p->tiles.size());
  set_mesh(*a, p);
  set_coeffs(*a, hp, step);
  return FSP_OK;
}

fsp_status run_step(const fsp_plan* p, const void* const* grads, int32_t dtype, float* master, float* m,
                    float* v, void* const* params, const fsp_adamw_hparams* hp, int64_t step, bool debug,
                    float* reduced, void* stream) {
  clear_error();
  std::vector<Buf> extra;
  if (debug && p) extra.push_back({reduced, size_t(p->state_len_total) * 4, "reduced_grad"});
  fsp_status s = check_device_step(p, grads, dtype, master, m, v, params, hp, step, extra);
  if (s != FSP_OK || p->tiles.empty()) return s;
  StepArgs a;
  s = step_args(p, grads, master, m, v, params, hp, step, &a);
  if (s != FSP_OK) return s;
  a.reduced = reduced;
  return launch(a, dtype, stream, false, nullptr, p);
}

// Partial sums of the clipped step's norm, one array per plan and device: one
// double per work tile, then one per block of kNormBlock tiles.
fsp_status device_partials(const fsp_plan* p, double** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  std::lock_guard<std::mutex> lock(p->mu);
  auto it = p->device_partials.find(dev);
  if (it != p->device_partials.end()) {
    *out = it->second;
    return FSP_OK;
  }
  double* d = nullptr;
  const size_t n = p->tiles.size();
  e = cudaMalloc(&d, std::max<size_t>(1, n + (n + kNormBlock - 1) / kNormBlock) * sizeof(double));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(FSP_ENOMEM, cuda_msg("cudaMalloc (norm partials)", e));
  }
  p->device_partials[dev] = d;
  *out = d;
  return FSP_OK;
}

// Passes 1-3 of the clipped flow for an argument block whose tiles, buffers
// (or per-parameter tables) and coefficients are set; the plan is non-empty.
fsp_status run_clipped_passes(const fsp_plan* p, StepArgs& a, float max_norm, float* norm_out, void* stream) {
  double* partials = nullptr;
  fsp_status s = device_partials(p, &partials);
  if (s != FSP_OK) return s;

  // pass 1: reduce-scatter into the owners' slices and each tile's sum of
  // squares, one CTA per tile (the block scheduler takes the tiles in order)
  if (a.n_tiles > INT32_MAX) return fail(FSP_EUNSUPPORTED, "the clipped step takes at most 2^31 - 1 work tiles");
  const KernelInfo k1 = NormKernels::get(p->n_shard, p->n_rep);
  const int grid = int(a.n_tiles);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* args1[] = {&a, &partials};
  cudaError_t e = cudaLaunchKernel(k1.fn, dim3(grid), dim3(k1.threads), args1, 0, st);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("reduce-scatter / norm kernel launch", e));
  // pass 2: the norm (the tiles' sums added in a fixed order) and the clip coefficient
  const int n_blocks = int((a.n_tiles + kNormBlock - 1) / kNormBlock);
  double* block_sums = partials + a.n_tiles;
  norm_block_sums_kernel<<<n_blocks, kNormBlockThreads, 0, st>>>(partials, grid, block_sums);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("norm block-sum kernel launch", e));
  norm_finalize_kernel<<<1, kNormFinalizeThreads, 0, st>>>(block_sums, n_blocks, max_norm, norm_out);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("norm kernel launch", e));
  // pass 3: AdamW on the clipped gradient read from the owners' slices
  a.clip = norm_out;
  return launch(a, FSP_DTYPE_F32, stream, true, nullptr, p);
}

fsp_status advance_step(int64_t* step_dev, void* stream) {
  step_advance_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(step_dev);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FSP_OK : fail(FSP_ECUDA, cuda_msg("step counter advance", e));
}

// norm_out = {0, 1} for a plan with nothing to reduce.
fsp_status clipped_empty(float* norm_out, void* stream) {
  const float out[2] = {0.f, 1.f};
  cudaError_t e =
      cudaMemcpyAsync(norm_out, out, sizeof(out), cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FSP_OK : fail(FSP_ECUDA, cuda_msg("writing norm_out", e));
}

fsp_status run_step_clipped(const fsp_plan* p, void* const* grads, int32_t dtype, float* master, float* m, float* v,
                            void* const* params, const fsp_adamw_hparams* hp, int64_t step, float max_norm,
                            float* norm_out, void* stream) {
  clear_error();
  if (dtype != FSP_DTYPE_F32) return fail(FSP_EUNSUPPORTED, "the clipped step writes back into fp32 grad buffers");
  if (!(std::isfinite(max_norm) && max_norm > 0.f)) return fail(FSP_EINVAL, "max_norm must be finite and > 0");
  std::vector<Buf> extra{{norm_out, 2 * sizeof(float), "norm_out"}};
  fsp_status s = check_device_step(p, reinterpret_cast<const void* const*>(grads), dtype, master, m, v, params, hp,
                                   step, extra);
  if (s != FSP_OK) return s;
  if (p->tiles.empty()) return clipped_empty(norm_out, stream);   // nothing to reduce: norm 0, coefficient 1
  StepArgs a;
  s = step_args(p, reinterpret_cast<const void* const*>(grads), master, m, v, params, hp, step, &a);
  if (s != FSP_OK) return s;
  return run_clipped_passes(p, a, max_norm, norm_out, stream);
}

}  // namespace fsp

extern "C" fsp_status fsp_sharded_step(const fsp_plan* plan, const void* const* grad_bufs, int32_t grad_dtype,
                                       float* master, float* exp_avg, float* exp_avg_sq,
                                       void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                                       void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step, false,
                         nullptr, cuda_stream);
  });
}

extern "C" fsp_status fsp_sharded_step_clipped(const fsp_plan* plan, void* const* grad_bufs, int32_t grad_dtype,
                                               float* master, float* exp_avg, float* exp_avg_sq,
                                               void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                                               float max_norm, float* norm_out, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step_clipped(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step,
                                 max_norm, norm_out, cuda_stream);
  });
}

extern "C" fsp_status fsp_sharded_step_device_t(const fsp_plan* plan, const void* const* grad_bufs,
                                                int32_t grad_dtype, float* master, float* exp_avg, float* exp_avg_sq,
                                                void* const* param_bufs, const fsp_adamw_hparams* hp,
                                                int64_t* step_dev, int32_t advance, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    using namespace fsp;
    clear_error();
    if (!step_dev) return fail(FSP_EINVAL, "step_dev is NULL");
    if (reinterpret_cast<uintptr_t>(step_dev) % 8 != 0) return fail(FSP_EINVAL, "step_dev is not 8-byte aligned");
    // t only enters the bias corrections, which the kernel recomputes from *step_dev
    fsp_status s = check_device_step(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, 1, {});
    if (s != FSP_OK) return s;
    s = check_allocation(step_dev, sizeof(int64_t), "step_dev");
    if (s != FSP_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    if (!plan->tiles.empty()) {
      StepArgs a;
      s = step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hp, 1, &a);
      if (s != FSP_OK) return s;
      a.step_dev = step_dev;
      s = launch(a, grad_dtype, cuda_stream, false, nullptr, plan);
      if (s != FSP_OK) return s;
    }
    if (advance) return advance_step(step_dev, st);
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_sharded_step_writeback(const fsp_plan* plan, void* const* grad_bufs, int32_t grad_dtype,
                                                 float* master, float* exp_avg, float* exp_avg_sq,
                                                 void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                                                 void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    using namespace fsp;
    clear_error();
    if (plan && plan->n_rep != 1) return fail(FSP_EUNSUPPORTED, "the write-back step is for FSDP2 and DistOpt plans");
    if (grad_dtype != FSP_DTYPE_F32)
      return fail(FSP_EUNSUPPORTED, "the write-back step stores the averaged gradient into fp32 grad buffers");
    const void* const* grads = reinterpret_cast<const void* const*>(grad_bufs);
    fsp_status s = check_device_step(plan, grads, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step, {});
    if (s != FSP_OK || plan->tiles.empty()) return s;
    StepArgs a;
    s = step_args(plan, grads, master, exp_avg, exp_avg_sq, param_bufs, hp, step, &a);
    if (s != FSP_OK) return s;
    a.writeback = 1;
    return launch(a, grad_dtype, cuda_stream, false, nullptr, plan);
  });
}

extern "C" fsp_status fsp_sharded_step_fp32_gather(const fsp_plan* plan, const void* const* grad_bufs,
                                                   int32_t grad_dtype, float* master, float* exp_avg,
                                                   float* exp_avg_sq, void* const* param_bufs,
                                                   const fsp_adamw_hparams* hp, int64_t step, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    using namespace fsp;
    clear_error();
    if (!param_bufs) return fail(FSP_EINVAL, "param_bufs is NULL");
    fsp_status s = check_device_step(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step,
                                     {}, 4);
    if (s != FSP_OK || plan->tiles.empty()) return s;
    StepArgs a;
    s = step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hp, step, &a);
    if (s != FSP_OK) return s;
    a.param_f32 = 1;
    return launch(a, grad_dtype, cuda_stream, false, nullptr, plan);
  });
}

extern "C" fsp_status fsp_sharded_step_debug(const fsp_plan* plan, const void* const* grad_bufs,
                                             int32_t grad_dtype, float* master, float* exp_avg,
                                             float* exp_avg_sq, void* const* param_bufs,
                                             const fsp_adamw_hparams* hp, int64_t step, float* reduced_grad,
                                             void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step, true,
                         reduced_grad, cuda_stream);
  });
}

// ---- entry point that allocates nothing --------------------------------------
//
// For callers that cannot call cudaMalloc: code running while a framework's
// allocator owns all device memory, inside a memory pool that must not grow,
// or on a path that must never touch the CUDA allocator.  fsp_sharded_step
// allocates one tile table per plan and device on its first call; this entry
// point instead keeps the tile list in a fixed array of device memory that
// the library declares at file scope (kNoAllocMaxTiles tiles, 8 MiB, held on
// every device that loads the library until the process exits), copies the
// plan's list there on the stream when the array does not already hold it,
// and runs the same kernel on it; its tile counter is a second file-scope
// variable, zeroed on the stream.

namespace fsp {
namespace {

constexpr int64_t kNoAllocMaxTiles = 262144;   // 8 MiB of 32-byte tile descriptors
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) Tile g_noalloc_tiles[kNoAllocMaxTiles];
// The kernel's tile counter for this entry (zeroed on the stream before each launch).
static __device__ __align__(8) unsigned long long g_noalloc_tile_ctr;

// Per device: the device addresses of g_noalloc_tiles and g_noalloc_tile_ctr
// (the names themselves are host stand-ins in host code), resolved once with
// that device current, and the uid of the plan whose tile list the array
// holds (0: none yet).
struct NoAllocDevice {
  Tile* tiles = nullptr;
  unsigned long long* ctr = nullptr;
  uint64_t loaded_uid = 0;
};
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices] = {};

// The arrays of the current device; copies plan p's tile list into the tile
// array on `st` unless the array already holds it (from an earlier call with
// this plan on this device: calls are ordered by the caller, so that copy has
// landed before this call's kernel runs).
fsp_status noalloc_arrays_for(const fsp_plan* p, cudaStream_t st, Tile** tiles, unsigned long long** ctr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(FSP_EUNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.tiles) {
    void* tiles_addr = nullptr;
    void* ctr_addr = nullptr;
    e = cudaGetSymbolAddress(&tiles_addr, g_noalloc_tiles);
    if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetSymbolAddress(g_noalloc_tiles)", e));
    e = cudaGetSymbolAddress(&ctr_addr, g_noalloc_tile_ctr);
    if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetSymbolAddress(g_noalloc_tile_ctr)", e));
    d.ctr = static_cast<unsigned long long*>(ctr_addr);
    d.tiles = static_cast<Tile*>(tiles_addr);
  }
  if (d.loaded_uid != p->uid) {
    d.loaded_uid = 0;   // a failed copy leaves the array's contents unknown
    e = cudaMemcpyAsync(d.tiles, p->tiles.data(), p->tiles.size() * sizeof(Tile), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaMemcpyAsync (tile list)", e));
    d.loaded_uid = p->uid;
  }
  *tiles = d.tiles;
  *ctr = d.ctr;
  return FSP_OK;
}

fsp_status run_step_noalloc(const fsp_plan* p, const void* const* grads, int32_t dtype, float* master, float* m,
                            float* v, void* const* params, const fsp_adamw_hparams* hp, int64_t step,
                            void* stream) {
  clear_error();
  if (p && int64_t(p->tiles.size()) > kNoAllocMaxTiles)
    return fail(FSP_EUNSUPPORTED, "plan needs " + std::to_string(p->tiles.size()) +
                                      " work tiles; fsp_sharded_step_noalloc holds at most 262144");
  // the checks of fsp_sharded_step (host memory only)
  fsp_status s = check_device_step(p, grads, dtype, master, m, v, params, hp, step, {});
  if (s != FSP_OK || p->tiles.empty()) return s;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Tile* tiles = nullptr;
  unsigned long long* ctr = nullptr;
  s = noalloc_arrays_for(p, st, &tiles, &ctr);
  if (s != FSP_OK) return s;

  StepArgs a{};
  for (int q = 0; q < p->n_d; ++q) {
    a.grads[q] = grads[q];
    a.params[q] = params ? static_cast<uint16_t*>(params[q]) : nullptr;
  }
  a.gather = params ? 1 : 0;   // NULL param_bufs: the ZeRO-3 step, as fsp_sharded_step
  a.master = master;
  a.m = m;
  a.v = v;
  a.reduced = nullptr;
  a.tiles = tiles;
  a.n_tiles = int64_t(p->tiles.size());
  set_mesh(a, p);
  set_coeffs(a, hp, step);
  return launch(a, dtype, st, false, ctr);   // the library's counter: nothing to allocate
}

}  // namespace
}  // namespace fsp

extern "C" fsp_status fsp_sharded_step_noalloc(const fsp_plan* plan, const void* const* grad_bufs,
                                               int32_t grad_dtype, float* master, float* exp_avg,
                                               float* exp_avg_sq, void* const* param_bufs,
                                               const fsp_adamw_hparams* hp, int64_t step, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step_noalloc(plan, grad_bufs, grad_dtype, master, exp_avg, exp_avg_sq, param_bufs, hp, step,
                                 cuda_stream);
  });
}

extern "C" fsp_status fsp_plan_tiles(const fsp_plan* plan, int32_t unit, fsp_tile* out, int64_t cap, int64_t* n) {
  return fsp::guard([&]() -> fsp_status {
    using namespace fsp;
    clear_error();
    if (!plan || !n) return fail(FSP_EINVAL, "plan or n is NULL");
    if (unit < 0 || unit % 8 != 0 || (unit > 0 && kTileElems % unit != 0))
      return fail(FSP_EINVAL, "unit must be 0 or a multiple of 8 that divides 4096");
    if (cap < 0 || (cap > 0 && !out)) return fail(FSP_EINVAL, "out is NULL or cap < 0");
    static_assert(sizeof(fsp_tile) == sizeof(Tile), "fsp_tile mirrors the internal tile");
    const std::vector<Tile> cut = unit > 0 ? split_tiles(plan->tiles, unit) : std::vector<Tile>();
    const std::vector<Tile>& tiles = unit > 0 ? cut : plan->tiles;
    *n = int64_t(tiles.size());
    const int64_t k = std::min<int64_t>(cap, int64_t(tiles.size()));
    for (int64_t i = 0; i < k; ++i)
      out[i] = fsp_tile{tiles[i].full_begin, tiles[i].state_begin, tiles[i].len, tiles[i].rank, tiles[i].param, 0};
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_plan_round_order(const fsp_plan* plan, int32_t grid, fsp_tile* out, int64_t cap,
                                           int64_t* n) {
  return fsp::guard([&]() -> fsp_status {
    using namespace fsp;
    clear_error();
    if (!plan || !n) return fail(FSP_EINVAL, "plan or n is NULL");
    if (grid < 1) return fail(FSP_EINVAL, "grid must be >= 1");
    if (cap < 0 || (cap > 0 && !out)) return fail(FSP_EINVAL, "out is NULL or cap < 0");
    std::vector<Tile> order = balance_rounds(plan->tiles, grid);
    if (plan->tiles.size() <= size_t(grid) ||
        busiest_cta_chunks(order, grid) >= busiest_cta_chunks(plan->tiles, grid))
      order = plan->tiles;
    *n = int64_t(order.size());
    const int64_t k = std::min<int64_t>(cap, int64_t(order.size()));
    for (int64_t i = 0; i < k; ++i)
      out[i] = fsp_tile{order[i].full_begin, order[i].state_begin, order[i].len, order[i].rank, order[i].param, 0};
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_device_error(uint32_t* bits) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!bits) return fsp::fail(FSP_EINVAL, "bits is NULL");
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, fsp::g_fsp_device_error, sizeof(v));
    if (e != cudaSuccess) return fsp::fail(FSP_ECUDA, fsp::cuda_msg("reading the device error word", e));
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(fsp::g_fsp_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return fsp::fail(FSP_ECUDA, fsp::cuda_msg("clearing the device error word", e));
    *bits = v;
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_selftest_bounded_wait(uint32_t limit_ms, uint32_t* bits) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!bits) return fsp::fail(FSP_EINVAL, "bits is NULL");
    if (limit_ms < 1 || limit_ms > 2000) return fsp::fail(FSP_EINVAL, "limit_ms must be in [1, 2000]");
    uint32_t before = 0;
    fsp_status s = fsp_device_error(&before);   // start from a clear word
    if (s != FSP_OK) return s;
    fsp::bounded_wait_selftest_kernel<<<1, 32>>>(uint64_t(limit_ms) * 1000000ull);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fsp::fail(FSP_ECUDA, fsp::cuda_msg("bounded-wait self-test", e));
    s = fsp_device_error(bits);
    if (s != FSP_OK) return s;
    *bits |= before;
    return FSP_OK;
  });
}
