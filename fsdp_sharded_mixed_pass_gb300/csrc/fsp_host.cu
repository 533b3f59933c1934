// The step with the gradients and params in host memory: a chunked
// H2D / kernel / D2H pipeline behind fsp_sharded_step_host.
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "fsp_host.h"
#include "fsp_internal.h"

// The N_d gradient buffers come from host memory and the N_d bf16 param buffers
// go back to it, while master/m/v stay on the device.  The plan's tiles are cut
// into chunks of about `chunk_elems` elements (at 4096-element tile boundaries);
// chunk k's gradient slices are copied into one of two device staging slots on
// a host-to-device stream, the kernel runs on the caller's stream, and the bf16
// result is copied from a staging slot to every rank's host buffer on a
// device-to-host stream, so H2D of chunk k+1, the kernel on chunk k and D2H of
// chunk k-1 overlap (NVLink-C2C carries both directions at once).

namespace fsp {
namespace {

int64_t host_slot_elems(int64_t chunk_elems) {
  const int64_t c = chunk_elems > 0 ? chunk_elems : (int64_t(1) << 24);
  return (c + kTileElems - 1) / kTileElems * kTileElems + kTileElems;
}

size_t host_workspace_bytes(const fsp_plan* p, int32_t dtype, int64_t chunk_elems) {
  const size_t g = dtype == FSP_DTYPE_F32 ? 4 : 2;
  return 2 * size_t(host_slot_elems(chunk_elems)) * (size_t(p->n_d) * g + 2 * size_t(p->n_rep));
}

// Copies of different ranks' slices run on several streams at once so that
// several copy engines share each direction of the link.
constexpr int kCopyLanes = 4;

struct CopyStreams {
  cudaStream_t h2d[kCopyLanes] = {}, d2h[kCopyLanes] = {};
};

// 2 x kCopyLanes non-blocking copy streams per device, created on first use
// and kept for the life of the process.
fsp_status copy_streams(CopyStreams* out) {
  static std::mutex mu;
  static std::map<int, CopyStreams> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) {
    *out = it->second;
    return FSP_OK;
  }
  CopyStreams s;
  for (int j = 0; e == cudaSuccess && j < kCopyLanes; ++j) {
    e = cudaStreamCreateWithFlags(&s.h2d[j], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.d2h[j], cudaStreamNonBlocking);
  }
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaStreamCreateWithFlags", e));
  cache[dev] = s;
  *out = s;
  return FSP_OK;
}

bool is_host_pointer(const void* ptr) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeHost || attr.type == cudaMemoryTypeUnregistered;
}

fsp_status run_step_host(const fsp_plan* p, const void* const* host_grads, int32_t dtype, float* master, float* m,
                         float* v, void* const* host_params, const fsp_adamw_hparams* hp, int64_t step,
                         void* workspace, size_t workspace_bytes, int64_t chunk_elems, void* stream) {
  clear_error();
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  if (!host_grads || !host_params) return fail(FSP_EINVAL, "host_grads or host_params is NULL");
  if (dtype != FSP_DTYPE_F32 && dtype != FSP_DTYPE_BF16) return fail(FSP_EINVAL, "unknown grad dtype");
  if (chunk_elems < 0) return fail(FSP_EINVAL, "chunk_elems must be >= 0 (0: default)");
  if (fsp_status hs = check_hparams(hp, step); hs != FSP_OK) return hs;
  const int n = p->n_d;
  const size_t g = dtype == FSP_DTYPE_F32 ? 4 : 2;
  const size_t sbytes = size_t(p->state_len_total) * 4;
  const float* state[3] = {master, m, v};
  const char* names[3] = {"master", "exp_avg", "exp_avg_sq"};
  for (int i = 0; i < 3; ++i) {
    if (!state[i] && sbytes) return fail(FSP_EINVAL, std::string(names[i]) + " is NULL");
    if (reinterpret_cast<uintptr_t>(state[i]) % 16)
      return fail(FSP_EINVAL, std::string(names[i]) + " is not 16-byte aligned");
  }
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j) {
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(state[i]), b0 = reinterpret_cast<uintptr_t>(state[j]);
      if (sbytes && a0 < b0 + sbytes && b0 < a0 + sbytes) return fail(FSP_EINVAL, "state buffers overlap");
    }
  const size_t need = host_workspace_bytes(p, dtype, chunk_elems);
  if (p->tiles.empty()) return FSP_OK;
  for (int q = 0; q < n; ++q) {
    if (!host_grads[q] || !host_params[q]) return fail(FSP_EINVAL, "a host buffer is NULL");
    if (!is_host_pointer(host_grads[q]) || !is_host_pointer(host_params[q]))
      return fail(FSP_EINVAL, "host_grads / host_params must be host memory");
  }
  if (!workspace) return fail(FSP_EINVAL, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(FSP_EINVAL, "workspace is not 256-byte aligned");
  if (workspace_bytes < need)
    return fail(FSP_EINVAL, "workspace too small: " + std::to_string(need) + " bytes needed");
  for (int i = 0; i < 3; ++i) {
    fsp_status s = check_allocation(state[i], sbytes, names[i]);
    if (s != FSP_OK) return s;
  }
  fsp_status s = check_allocation(workspace, need, "workspace");
  if (s != FSP_OK) return s;

  const Tile* dtiles = nullptr;
  s = device_tiles(p, &dtiles);
  if (s != FSP_OK) return s;
  CopyStreams cs;
  s = copy_streams(&cs);
  if (s != FSP_OK) return s;

  // chunk k = tiles [cuts[k], cuts[k+1]), a contiguous full-index range
  const int64_t slot = host_slot_elems(chunk_elems);
  const int64_t target = slot - kTileElems;
  std::vector<size_t> cuts{0};
  int64_t start = p->tiles[0].full_begin;
  for (size_t i = 1; i < p->tiles.size(); ++i) {
    const Tile& t = p->tiles[i];
    if (t.full_begin % kTileElems == 0 && t.full_begin - start >= target) {
      cuts.push_back(i);
      start = t.full_begin;
    }
  }
  cuts.push_back(p->tiles.size());
  const size_t n_chunks = cuts.size() - 1;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  auto stg_grad = [&](int sl, int q) { return ws + (size_t(sl) * n + q) * size_t(slot) * g; };
  const int n_rep = p->n_rep, n_shard = p->n_shard;
  // one bf16 tile per replica group per slot
  auto stg_param = [&](int sl, int r) {
    return ws + 2 * size_t(n) * size_t(slot) * g + (size_t(sl) * n_rep + r) * size_t(slot) * 2;
  };

  cudaStream_t cs_main = static_cast<cudaStream_t>(stream);
  const int lanes = std::min(kCopyLanes, n);
  // per chunk: `lanes` H2D events, one kernel event, `lanes` D2H events
  const size_t per = size_t(2 * lanes + 1);
  std::vector<cudaEvent_t> ev(per * n_chunks + 1, nullptr);
  auto cleanup = [&]() {
    for (cudaEvent_t x : ev)
      if (x) cudaEventDestroy(x);
  };
  for (auto& x : ev) {
    cudaError_t e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      cleanup();
      return fail(FSP_ECUDA, cuda_msg("cudaEventCreateWithFlags", e));
    }
  }
  cudaEvent_t entry = ev[per * n_chunks];
  auto ev_h2d = [&](size_t k, int j) { return ev[per * k + j]; };
  auto ev_kern = [&](size_t k) { return ev[per * k + lanes]; };
  auto ev_d2h = [&](size_t k, int j) { return ev[per * k + lanes + 1 + j]; };

  StepArgs a{};
  a.master = master;
  a.m = m;
  a.v = v;
  a.reduced = nullptr;
  a.gather = 1;
  set_mesh(a, p);
  set_coeffs(a, hp, step);

  cudaError_t e = cudaEventRecord(entry, cs_main);   // copies start after earlier work on the stream
  for (int j = 0; e == cudaSuccess && j < lanes; ++j) {
    e = cudaStreamWaitEvent(cs.h2d[j], entry, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.d2h[j], entry, 0);
  }
  for (size_t k = 0; e == cudaSuccess && k < n_chunks; ++k) {
    const int sl = int(k % 2);
    const Tile& first = p->tiles[cuts[k]];
    const Tile& last = p->tiles[cuts[k + 1] - 1];
    const int64_t f0 = first.full_begin, f1 = last.full_begin + last.len;
    const size_t len = size_t(f1 - f0);
    // H2D, rank q on lane q % lanes: this slot's previous reader (the kernel of
    // chunk k-2) must be done
    for (int j = 0; e == cudaSuccess && j < lanes; ++j) {
      if (k >= 2) e = cudaStreamWaitEvent(cs.h2d[j], ev_kern(k - 2), 0);
      for (int q = j; e == cudaSuccess && q < n; q += lanes)
        e = cudaMemcpyAsync(stg_grad(sl, q), static_cast<const unsigned char*>(host_grads[q]) + size_t(f0) * g,
                            len * g, cudaMemcpyHostToDevice, cs.h2d[j]);
      if (e == cudaSuccess) e = cudaEventRecord(ev_h2d(k, j), cs.h2d[j]);
      // the kernel waits for every lane's gradients ...
      if (e == cudaSuccess) e = cudaStreamWaitEvent(cs_main, ev_h2d(k, j), 0);
      // ... and for the D2H of chunk k-2, which read this slot's bf16 tile
      if (e == cudaSuccess && k >= 2) e = cudaStreamWaitEvent(cs_main, ev_d2h(k - 2, j), 0);
    }
    if (e != cudaSuccess) break;
    for (int q = 0; q < n; ++q) {
      // staging holds full indices [f0, f1): index it with the full index
      a.grads[q] = stg_grad(sl, q) - size_t(f0) * g;
      a.params[q] = reinterpret_cast<uint16_t*>(stg_param(sl, q / n_shard)) - f0;   // one tile per group
    }
    a.tiles = dtiles + cuts[k];
    a.n_tiles = int64_t(cuts[k + 1] - cuts[k]);
    // (a plain launch: the kernel follows the copies' events, not only the previous chunk's kernel)
    s = launch(a, dtype, cs_main, false, nullptr, nullptr, false);
    if (s != FSP_OK) {
      cleanup();
      return s;
    }
    e = cudaEventRecord(ev_kern(k), cs_main);
    // D2H: the all-gather into every rank's host buffer
    for (int j = 0; e == cudaSuccess && j < lanes; ++j) {
      e = cudaStreamWaitEvent(cs.d2h[j], ev_kern(k), 0);
      for (int q = j; e == cudaSuccess && q < n; q += lanes)
        e = cudaMemcpyAsync(static_cast<unsigned char*>(host_params[q]) + size_t(f0) * 2, stg_param(sl, q / n_shard),
                            len * 2, cudaMemcpyDeviceToHost, cs.d2h[j]);
      if (e == cudaSuccess) e = cudaEventRecord(ev_d2h(k, j), cs.d2h[j]);
    }
  }
  // the caller's stream completes only after every copy back
  for (size_t k = n_chunks >= 2 ? n_chunks - 2 : 0; e == cudaSuccess && k < n_chunks; ++k)
    for (int j = 0; e == cudaSuccess && j < lanes; ++j) e = cudaStreamWaitEvent(cs_main, ev_d2h(k, j), 0);
  cleanup();
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("host-buffer step pipeline", e));
  return FSP_OK;
}

}  // namespace
}  // namespace fsp

extern "C" fsp_status fsp_host_step_workspace_bytes(const fsp_plan* plan, int32_t grad_dtype, int64_t chunk_elems,
                                                    size_t* bytes) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!plan || !bytes) return fsp::fail(FSP_EINVAL, "NULL argument");
    if (grad_dtype != FSP_DTYPE_F32 && grad_dtype != FSP_DTYPE_BF16) return fsp::fail(FSP_EINVAL, "unknown grad dtype");
    if (chunk_elems < 0) return fsp::fail(FSP_EINVAL, "chunk_elems must be >= 0 (0: default)");
    *bytes = fsp::host_workspace_bytes(plan, grad_dtype, chunk_elems);
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_sharded_step_host(const fsp_plan* plan, const void* const* host_grads, int32_t grad_dtype,
                                            float* master, float* exp_avg, float* exp_avg_sq,
                                            void* const* host_params, const fsp_adamw_hparams* hp, int64_t step,
                                            void* workspace, size_t workspace_bytes, int64_t chunk_elems,
                                            void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step_host(plan, host_grads, grad_dtype, master, exp_avg, exp_avg_sq, host_params, hp, step,
                              workspace, workspace_bytes, chunk_elems, cuda_stream);
  });
}

