// FSDP2 unshard for sm_103a: every rank's fp32 shard (its slots of the master
// buffer) is cast to bf16 and all-gathered into every rank's full param buffer
// of its group - the pre-forward / pre-backward all-gather of ZeRO-3 with a
// bf16 MixedPrecisionPolicy ("Parallelism strategies: which state to shard",
// section 二.5: copy-in, one all-gather, copy-out; "FSDP2 Qwen3 Decoder Layer
// Walkthrough", section "Step 0").  With N_d ranks as buffers on one device the
// copy-in / all-gather / copy-out collapse into one pass: each element is read
// once (4 B) and written once per rank of its group (2 B each).
//
// One CTA per tile (the loop over tiles also serves any smaller grid); each
// thread takes 8-element groups (two 16-byte loads of the master, one 16-byte
// store per rank); unaligned segment edges are done one element at a time.
// No waits of any kind.
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

__global__ void __launch_bounds__(kUnshardThreads) unshard_kernel(const __grid_constant__ UnshardArgs a) {
  const int ns = a.n_shard, nr = a.n_rep;
  for (int64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tile = a.tiles[t];
    const int64_t f0 = tile.full_begin, len = tile.len;
    const int64_t delta = tile.state_begin - tile.full_begin;
    // [0, head): before the first multiple of 8; [head, tail): 8-element groups
    const int64_t head = min(len, (8 - (f0 & 7)) & 7);
    const int64_t groups = (len - head) >> 3;
    const int64_t tail = head + groups * 8;
    for (int64_t i = threadIdx.x; i < groups; i += kUnshardThreads) {
      const int64_t f = f0 + head + 8 * i;
      for (int r = 0; r < nr; ++r) {
        const float* src = a.master + f + delta + r * a.rep_stride;
        const float4 x = __ldcs(reinterpret_cast<const float4*>(src));
        const float4 y = __ldcs(reinterpret_cast<const float4*>(src + 4));
        const uint4 b = make_uint4(pack2(x.x, x.y), pack2(x.z, x.w), pack2(y.x, y.y), pack2(y.z, y.w));
        for (int j = 0; j < ns; ++j) __stcs(reinterpret_cast<uint4*>(a.params[r * ns + j] + f), b);
      }
    }
    const int64_t n_scalar = head + (len - tail);
    if (threadIdx.x < n_scalar) {
      const int64_t f = f0 + (threadIdx.x < head ? int64_t(threadIdx.x) : tail + (threadIdx.x - head));
      for (int r = 0; r < nr; ++r) {
        const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rn(a.master[f + delta + r * a.rep_stride]));
        for (int j = 0; j < ns; ++j) a.params[r * ns + j][f] = b;
      }
    }
  }
}

cudaError_t launch_unshard(const UnshardArgs& a, int grid, void* stream) {
  unshard_kernel<<<grid, kUnshardThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError();
}

// ---- FSDP2 unshard: host side -----------------------------------------------------------

fsp_status run_unshard(const fsp_plan* p, const float* master, void* const* params, void* stream) {
  clear_error();
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  if (!params) return fail(FSP_EINVAL, "param_bufs is NULL");
  std::vector<Buf> bufs;
  for (int q = 0; q < p->n_d; ++q)
    bufs.push_back({params[q], size_t(p->full_len_padded) * 2, "param_bufs[" + std::to_string(q) + "]"});
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

}  // namespace
}  // namespace fsp

extern "C" fsp_status fsp_unshard(const fsp_plan* plan, const float* master, void* const* param_bufs,
                                  void* cuda_stream) {
  return fsp::run_unshard(plan, master, param_bufs, cuda_stream);
}
