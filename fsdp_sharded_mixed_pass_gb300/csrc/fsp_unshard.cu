// FSDP2 unshard for sm_103a: every rank's fp32 shard (its slots of the master
// buffer) is cast to bf16 and all-gathered into every rank's full param buffer
// of its group - the pre-forward / pre-backward all-gather of ZeRO-3 with a
// bf16 MixedPrecisionPolicy ("Parallelism strategies: which state to shard",
// section 二.5: copy-in, one all-gather, copy-out; "FSDP2 Qwen3 Decoder Layer
// Walkthrough", section "Step 0").  With N_d ranks as buffers on one device the
// copy-in / all-gather / copy-out collapse into one pass: each element is read
// once (4 B) and written once per rank of its group (2 B each).
//
// One CTA per tile (the loop over tiles also serves any smaller grid): the
// threads read the tile's fp32 master with 16-byte loads and cast it into
// shared memory; one thread then writes the bf16 tile to every rank's buffer
// with bulk asynchronous copies.  Unaligned segment edges are done one element
// at a time.  The only waits are the bulk-copy group waits on this CTA's own
// stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <string>
#include <vector>

#include "fsp_host.h"
#include "fsp_internal.h"

namespace fsp {
namespace {

constexpr int kUnshardThreads = 256;

// Arguments of the unshard kernel.
struct UnshardArgs {
  const float* master;
  uint16_t* params[kMaxRanks];
  // per-parameter plans: entry param * n_d + q is rank q's virtual base for
  // that parameter (element f at base + f); nullptr for full-size buffers
  uint16_t* const* vparams;
  int n_d;
  int param_f32;   // 1: the parameter buffers / tensors are fp32 (the master copied, no cast)
  const Tile* tiles;
  int64_t n_tiles;
  int n_rep;
  int n_shard;
  int64_t rep_stride;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(static_cast<uint32_t>(__cvta_generic_to_shared(src))), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Programmatic dependent launch: let the next launch on the stream that allows
// it be scheduled; wait until the launches this grid depends on have completed
// and their writes are visible (at once for a launch without the attribute).
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// At most N committed bulk groups may still be reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// A tile is at most kTileElems elements: two 8-element groups per thread.
static_assert(kTileElems == 2 * 8 * kUnshardThreads, "unshard covers a tile in one pass of the CTA");

// Per tile and replica group: the threads cast the master's aligned body to
// bf16 in shared memory (kF32: copy it as it is), then one thread writes it to
// each rank of the group with a bulk copy (one 8 KB store per rank for a full
// bf16 tile).  Two buffers alternate, so replica r + 1 is cast while r's
// stores drain.
template <bool kF32>
__global__ void __launch_bounds__(kUnshardThreads) unshard_kernel(const __grid_constant__ UnshardArgs a) {
  constexpr int kOut = kF32 ? 4 : 2;   // bytes per output element
  __shared__ __align__(128) unsigned char cast[2][kTileElems * kOut];
  __shared__ uint16_t* tile_pb[kMaxRanks];
  const int ns = a.n_shard, nr = a.n_rep;
  const int i0 = threadIdx.x, i1 = threadIdx.x + kUnshardThreads;
  const bool per_param = a.vparams != nullptr;
  // Launched with programmatic stream serialisation: nothing of the master or
  // the parameter buffers is touched before the launch before this one is done.
  launch_dependents();
  grid_dependency_wait();
  int buf = 0;
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    if (per_param) {
      __syncthreads();   // the previous tile's bases are no longer read
      if (threadIdx.x < a.n_d) tile_pb[threadIdx.x] = a.vparams[int64_t(tile.param) * a.n_d + threadIdx.x];
      __syncthreads();
    }
    uint16_t* const* pb = per_param ? tile_pb : a.params;
    const int64_t f0 = tile.full_begin, end = f0 + tile.len;
    const int64_t delta = tile.state_begin - tile.full_begin;
    // aligned body [b0, b1): 8-element (16-byte bf16) boundaries of the full index
    int64_t b0 = (f0 + 7) & ~int64_t(7), b1 = end & ~int64_t(7);
    if (b1 < b0) b0 = b1 = end;
    const int groups = int((b1 - b0) >> 3);
    if (groups > 0) {
      for (int r = 0; r < nr; ++r) {
        const float* src = a.master + b0 + delta + r * a.rep_stride;
        float4 x0, y0, x1, y1;
        if (i0 < groups) {
          x0 = __ldcs(reinterpret_cast<const float4*>(src + 8 * i0));
          y0 = __ldcs(reinterpret_cast<const float4*>(src + 8 * i0 + 4));
        }
        if (i1 < groups) {
          x1 = __ldcs(reinterpret_cast<const float4*>(src + 8 * i1));
          y1 = __ldcs(reinterpret_cast<const float4*>(src + 8 * i1 + 4));
        }
        if (threadIdx.x == 0) bulk_wait_read<1>();   // this buffer's previous stores have read it
        __syncthreads();
        if (kF32) {
          float4* d = reinterpret_cast<float4*>(cast[buf]);
          if (i0 < groups) {
            d[2 * i0] = x0;
            d[2 * i0 + 1] = y0;
          }
          if (i1 < groups) {
            d[2 * i1] = x1;
            d[2 * i1 + 1] = y1;
          }
        } else {
          uint4* d = reinterpret_cast<uint4*>(cast[buf]);
          if (i0 < groups)
            d[i0] = make_uint4(pack2(x0.x, x0.y), pack2(x0.z, x0.w), pack2(y0.x, y0.y), pack2(y0.z, y0.w));
          if (i1 < groups)
            d[i1] = make_uint4(pack2(x1.x, x1.y), pack2(x1.z, x1.w), pack2(y1.x, y1.y), pack2(y1.z, y1.w));
        }
        fence_async_smem();   // the casts -> visible to the bulk stores
        __syncthreads();
        if (threadIdx.x == 0) {
          for (int j = 0; j < ns; ++j)
            bulk_store(reinterpret_cast<unsigned char*>(pb[r * ns + j]) + b0 * kOut, cast[buf],
                       uint32_t(groups) * 8u * kOut);
          bulk_commit();
        }
        buf ^= 1;
      }
    }
    // unaligned edges (fewer than 16 elements), one element per thread
    const int64_t n_head = b0 - f0, n_scalar = n_head + (end - b1);
    if (threadIdx.x < n_scalar) {
      const int64_t f = threadIdx.x < n_head ? f0 + threadIdx.x : b1 + (threadIdx.x - n_head);
      for (int r = 0; r < nr; ++r) {
        const float x = a.master[f + delta + r * a.rep_stride];
        if (kF32) {
          for (int j = 0; j < ns; ++j) reinterpret_cast<float*>(pb[r * ns + j])[f] = x;
        } else {
          const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(x));
          for (int j = 0; j < ns; ++j) pb[r * ns + j][f] = b;
        }
      }
    }
  }
  if (threadIdx.x == 0) bulk_wait_read<0>();   // shared memory must outlive the stores' reads
}

// Launched with programmatic stream serialisation (see the kernel): right
// after another kernel on the stream, its CTAs may be scheduled while that
// kernel's last CTAs finish.
cudaError_t launch_unshard(const UnshardArgs& a, int grid, void* stream) {
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kUnshardThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return a.param_f32 ? cudaLaunchKernelEx(&cfg, unshard_kernel<true>, a)
                     : cudaLaunchKernelEx(&cfg, unshard_kernel<false>, a);
}

// ---- FSDP2 unshard: host side -----------------------------------------------------------

fsp_status run_unshard(const fsp_plan* p, const float* master, void* const* params, bool f32, void* stream) {
  clear_error();
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  if (!params) return fail(FSP_EINVAL, "param_bufs is NULL");
  std::vector<Buf> bufs;
  for (int q = 0; q < p->n_d; ++q)
    bufs.push_back({params[q], size_t(p->full_len_padded) * (f32 ? 4 : 2), "param_bufs[" + std::to_string(q) + "]"});
  bufs.push_back({master, size_t(p->state_len_total) * 4, "master"});
  for (const Buf& b : bufs) {
    if (!b.ptr && b.bytes) return fail(FSP_EINVAL, b.name + " is NULL");
    if (reinterpret_cast<uintptr_t>(b.ptr) % 16 != 0) return fail(FSP_EINVAL, b.name + " is not 16-byte aligned");
  }
  for (size_t i = 0; i < bufs.size(); ++i)
    for (size_t j = i + 1; j < bufs.size(); ++j) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(bufs[i].ptr), b0 = reinterpret_cast<uintptr_t>(bufs[j].ptr);
      if (bufs[i].bytes && bufs[j].bytes && a0 < b0 + bufs[j].bytes && b0 < a0 + bufs[i].bytes)
        return fail(FSP_EINVAL, bufs[i].name + " overlaps " + bufs[j].name);
    }
  if (p->tiles.empty()) return FSP_OK;
  for (const Buf& b : bufs) {
    fsp_status s = check_allocation(b.ptr, b.bytes, b.name.c_str());
    if (s != FSP_OK) return s;
  }
  const Tile* tiles = nullptr;
  fsp_status s = device_tiles(p, &tiles);
  if (s != FSP_OK) return s;
  UnshardArgs a{};
  a.master = master;
  a.n_d = p->n_d;
  a.param_f32 = f32 ? 1 : 0;
  for (int q = 0; q < p->n_d; ++q) a.params[q] = static_cast<uint16_t*>(params[q]);
  a.tiles = tiles;
  a.n_tiles = int64_t(p->tiles.size());
  a.n_rep = p->n_rep;
  a.n_shard = p->n_shard;
  a.rep_stride = p->n_rep > 1 ? p->rep_stride : 0;
  // one CTA per tile: the block scheduler hands the tiles out in order, which
  // keeps the writes in one compact, moving window of the param buffers
  const int grid = int(std::min<int64_t>(INT32_MAX, a.n_tiles));
  cudaError_t e = launch_unshard(a, grid, stream);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("unshard kernel launch", e));
  return FSP_OK;
}

fsp_status run_unshard_params(const fsp_plan* p, const fsp_param_table* t, const float* master, void* stream) {
  clear_error();
  if (!p || !t) return fail(FSP_EINVAL, "plan or table is NULL");
  if (t->plan != p) return fail(FSP_EINVAL, "the table was created for another plan");
  if (!t->vparams) return fail(FSP_EINVAL, "the table has no param tensors");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  if (dev != t->device) return fail(FSP_EINVAL, "the table was created on another device");
  const size_t sbytes = size_t(p->state_len_total) * 4;
  if (!master && sbytes) return fail(FSP_EINVAL, "master is NULL");
  if (reinterpret_cast<uintptr_t>(master) % 16 != 0) return fail(FSP_EINVAL, "master is not 16-byte aligned");
  if (p->tiles.empty()) return FSP_OK;
  fsp_status s = check_allocation(master, sbytes, "master");
  if (s != FSP_OK) return s;
  const Tile* tiles = nullptr;
  s = device_tiles(p, &tiles);
  if (s != FSP_OK) return s;
  UnshardArgs a{};
  a.master = master;
  a.vparams = t->vparams;
  a.n_d = p->n_d;
  a.param_f32 = t->param_dtype == FSP_DTYPE_F32 ? 1 : 0;
  a.tiles = tiles;
  a.n_tiles = int64_t(p->tiles.size());
  a.n_rep = p->n_rep;
  a.n_shard = p->n_shard;
  a.rep_stride = p->n_rep > 1 ? p->rep_stride : 0;
  e = launch_unshard(a, int(std::min<int64_t>(INT32_MAX, a.n_tiles)), stream);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("unshard kernel launch", e));
  return FSP_OK;
}

// ---- FSDP2 shard: the inverse of the unshard -------------------------------------------

// Every owned element of the full fp32 parameter buffer goes to its slot of
// every replica group's master copy ("Parallelism strategies: which state to
// shard", section 二.5: fully_shard splits each parameter on dim 0 into
// per-rank DTensor shards).  One CTA per tile; 8-element groups of the full
// index move as two 16-byte loads and stores (full and state indices share
// their residue modulo 16), the unaligned edges one element per thread.
__global__ void __launch_bounds__(kUnshardThreads) shard_kernel(const float* __restrict__ full,
                                                                float* __restrict__ master, const Tile* tiles,
                                                                int64_t n_tiles, int n_rep, int64_t rep_stride) {
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const Tile tile = tiles[t];
    const int64_t f0 = tile.full_begin, end = f0 + tile.len;
    const int64_t delta = tile.state_begin - tile.full_begin;
    int64_t b0 = (f0 + 7) & ~int64_t(7), b1 = end & ~int64_t(7);
    if (b1 < b0) b0 = b1 = end;
    const int64_t groups = (b1 - b0) >> 3;
    for (int64_t i = threadIdx.x; i < groups; i += kUnshardThreads) {
      const int64_t f = b0 + 8 * i;
      const float4 x = __ldcs(reinterpret_cast<const float4*>(full + f));
      const float4 y = __ldcs(reinterpret_cast<const float4*>(full + f + 4));
      for (int r = 0; r < n_rep; ++r) {
        float* dst = master + f + delta + r * rep_stride;
        __stcs(reinterpret_cast<float4*>(dst), x);
        __stcs(reinterpret_cast<float4*>(dst + 4), y);
      }
    }
    const int64_t n_head = b0 - f0, n_scalar = n_head + (end - b1);
    if (threadIdx.x < n_scalar) {
      const int64_t f = threadIdx.x < n_head ? f0 + threadIdx.x : b1 + (threadIdx.x - n_head);
      for (int r = 0; r < n_rep; ++r) master[f + delta + r * rep_stride] = full[f];
    }
  }
}

fsp_status run_shard(const fsp_plan* p, const float* full, float* master, float* m, float* v, void* stream) {
  clear_error();
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  const size_t fbytes = size_t(p->full_len_padded) * 4, sbytes = size_t(p->state_len_total) * 4;
  std::vector<Buf> bufs{{full, fbytes, "full"}, {master, sbytes, "master"}};
  if (m) bufs.push_back({m, sbytes, "exp_avg"});
  if (v) bufs.push_back({v, sbytes, "exp_avg_sq"});
  for (const Buf& b : bufs) {
    if (!b.ptr && b.bytes) return fail(FSP_EINVAL, b.name + " is NULL");
    if (reinterpret_cast<uintptr_t>(b.ptr) % 16 != 0) return fail(FSP_EINVAL, b.name + " is not 16-byte aligned");
  }
  for (size_t i = 0; i < bufs.size(); ++i)
    for (size_t j = i + 1; j < bufs.size(); ++j) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(bufs[i].ptr), b0 = reinterpret_cast<uintptr_t>(bufs[j].ptr);
      if (bufs[i].bytes && bufs[j].bytes && a0 < b0 + bufs[j].bytes && b0 < a0 + bufs[i].bytes)
        return fail(FSP_EINVAL, bufs[i].name + " overlaps " + bufs[j].name);
    }
  if (p->tiles.empty()) return FSP_OK;
  for (const Buf& b : bufs) {
    fsp_status s = check_allocation(b.ptr, b.bytes, b.name.c_str());
    if (s != FSP_OK) return s;
  }
  const Tile* tiles = nullptr;
  fsp_status s = device_tiles(p, &tiles);
  if (s != FSP_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (m) e = cudaMemsetAsync(m, 0, sbytes, st);
  if (e == cudaSuccess && v) e = cudaMemsetAsync(v, 0, sbytes, st);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("zeroing the Adam moments", e));
  const int64_t n_tiles = int64_t(p->tiles.size());
  shard_kernel<<<int(std::min<int64_t>(INT32_MAX, n_tiles)), kUnshardThreads, 0, st>>>(
      full, master, tiles, n_tiles, p->n_rep, p->n_rep > 1 ? p->rep_stride : 0);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("shard kernel launch", e));
  return FSP_OK;
}

}  // namespace
}  // namespace fsp

extern "C" fsp_status fsp_unshard(const fsp_plan* plan, const float* master, void* const* param_bufs,
                                  void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_unshard(plan, master, param_bufs, false, cuda_stream);
  });
}

extern "C" fsp_status fsp_unshard_fp32(const fsp_plan* plan, const float* master, void* const* param_bufs,
                                       void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_unshard(plan, master, param_bufs, true, cuda_stream);
  });
}

extern "C" fsp_status fsp_unshard_params(const fsp_plan* plan, const fsp_param_table* table, const float* master,
                                         void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_unshard_params(plan, table, master, cuda_stream);
  });
}

extern "C" fsp_status fsp_shard(const fsp_plan* plan, const float* full, float* master, float* exp_avg,
                                float* exp_avg_sq, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_shard(plan, full, master, exp_avg, exp_avg_sq, cuda_stream);
  });
}
