// FSDP2 unshard for sm_103a: every rank's fp32 shard (its slots of the master
// buffer) is cast to bf16 and all-gathered into every rank's full param buffer
// of its group - the pre-forward / pre-backward all-gather of ZeRO-3 with a
// bf16 MixedPrecisionPolicy ("Parallelism strategies: which state to shard",
// section 二.5: copy-in, one all-gather, copy-out; "FSDP2 Qwen3 Decoder Layer
// Walkthrough", section "Step 0").  With N_d ranks as buffers on one device the
// copy-in / all-gather / copy-out collapse into one pass: each element is read
// once (4 B) and written once per rank of its group (2 B each).
//
// Persistent grid over the plan's tiles; each thread takes 8-element groups
// (two 16-byte loads of the master, one 16-byte store per rank); unaligned
// segment edges are done one element at a time.  No waits of any kind.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "fsp_internal.h"

namespace fsp {
namespace {

constexpr int kUnshardThreads = 256;

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

}  // namespace

int unshard_threads() { return kUnshardThreads; }

cudaError_t unshard_grid(int* grid) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, unshard_kernel, kUnshardThreads, 0);
  if (e == cudaSuccess) *grid = std::max(1, sms) * std::max(1, per_sm);
  return e;
}

cudaError_t launch_unshard(const UnshardArgs& a, int grid, void* stream) {
  unshard_kernel<<<grid, kUnshardThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError();
}

}  // namespace fsp
