// Per-parameter tensors: the table that registers them (fsp_param_table_create
// / _destroy) and the steps that read every rank's per-parameter gradients and
// write every rank's per-parameter bf16 or fp32 parameters in place
// (fsp_sharded_step_params and its _device_t, write-back and clipped
// variants) - FSDP2's copy-in before the reduce-scatter and copy-out after the
// all-gather folded into the step ("Parallelism strategies: which state to
// shard", section 二.5).  The unshard into the same tensors is
// fsp_unshard_params in fsp_unshard.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "fsp_host.h"
#include "fsp_internal.h"

namespace fsp {
namespace {

void free_table(fsp_param_table* t) {
  if (!t) return;
  if (t->vgrads || t->vparams) {
    int prev = -1;
    const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
    if (cudaSetDevice(t->device) == cudaSuccess) {
      cudaFree(const_cast<void**>(t->vgrads));
      cudaFree(t->vparams);
    }
    if (have_prev) cudaSetDevice(prev);
  }
  delete t;
}

fsp_status create_table(const fsp_plan* p, const void* const* grad_ptrs, int32_t dtype, void* const* param_ptrs,
                        int32_t param_dtype, fsp_param_table** out) {
  clear_error();
  if (!out) return fail(FSP_EINVAL, "out is NULL");
  *out = nullptr;
  if (!p) return fail(FSP_EINVAL, "plan is NULL");
  if (p->param_align != kParamAlign)
    return fail(FSP_EINVAL, "the plan is not a per-parameter plan (fsp_plan_layout_params)");
  if (dtype != FSP_DTYPE_F32 && dtype != FSP_DTYPE_BF16) return fail(FSP_EINVAL, "unknown grad dtype");
  if (param_dtype != FSP_DTYPE_F32 && param_dtype != FSP_DTYPE_BF16) return fail(FSP_EINVAL, "unknown param dtype");
  const size_t psz = param_dtype == FSP_DTYPE_F32 ? 4 : 2;
  const int n = p->n_d, np = p->n_params;
  if (np > 0 && !grad_ptrs) return fail(FSP_EINVAL, "grad_ptrs is NULL");
  const size_t g = dtype == FSP_DTYPE_F32 ? 4 : 2;

  // host-side checks first (NULL, alignment, overlap), then the driver's
  std::vector<const void*> vg(size_t(np) * n, nullptr);
  std::vector<uint16_t*> vp(param_ptrs ? size_t(np) * n : 0, nullptr);
  std::vector<std::pair<uintptr_t, uintptr_t>> spans;
  std::vector<std::string> names;
  for (int q = 0; q < n; ++q) {
    for (int i = 0; i < np; ++i) {
      const int64_t numel = p->param_numel[size_t(i)], off = p->param_off[size_t(i)];
      if (numel == 0) continue;
      for (int kind = 0; kind < (param_ptrs ? 2 : 1); ++kind) {
        const void* ptr = kind == 0 ? grad_ptrs[size_t(q) * np + i] : param_ptrs[size_t(q) * np + i];
        const size_t esz = kind == 0 ? g : psz;
        const std::string name = std::string(kind == 0 ? "grad_ptrs[" : "param_ptrs[") +
                                 std::to_string(size_t(q) * np + i) + "]";
        if (!ptr) return fail(FSP_EINVAL, name + " is NULL");
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return fail(FSP_EINVAL, name + " is not 16-byte aligned");
        const uintptr_t b = reinterpret_cast<uintptr_t>(ptr);
        spans.emplace_back(b, b + size_t(numel) * esz);
        names.push_back(name);
        // the virtual base: element f of this parameter is at base + f
        const uintptr_t base = b - uintptr_t(off) * esz;
        if (kind == 0)
          vg[size_t(i) * n + q] = reinterpret_cast<const void*>(base);
        else
          vp[size_t(i) * n + q] = reinterpret_cast<uint16_t*>(base);
      }
    }
  }
  std::vector<size_t> order(spans.size());
  for (size_t k = 0; k < order.size(); ++k) order[k] = k;
  std::sort(order.begin(), order.end(), [&](size_t x, size_t y) { return spans[x].first < spans[y].first; });
  for (size_t k = 1; k < order.size(); ++k)
    if (spans[order[k - 1]].second > spans[order[k]].first)
      return fail(FSP_EINVAL, names[order[k - 1]] + " overlaps " + names[order[k]]);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  for (size_t k = 0; k < spans.size(); ++k) {
    fsp_status s = check_allocation(reinterpret_cast<const void*>(spans[k].first), spans[k].second - spans[k].first,
                                    names[k].c_str());
    if (s != FSP_OK) return s;
  }

  fsp_param_table* t = new (std::nothrow) fsp_param_table();
  if (!t) return fail(FSP_ENOMEM, "host allocation failed");
  t->plan = p;
  t->device = dev;
  t->grad_dtype = dtype;
  t->param_dtype = param_dtype;
  try {
    t->spans.reserve(spans.size());
    for (size_t k : order) t->spans.push_back(spans[k]);
  } catch (const std::bad_alloc&) {
    delete t;
    return fail(FSP_ENOMEM, "host allocation failed");
  }
  const size_t bytes = std::max<size_t>(1, vg.size()) * sizeof(void*);
  e = cudaMalloc(reinterpret_cast<void**>(&t->vgrads), bytes);
  if (e == cudaSuccess && !vg.empty())
    e = upload_table(t->vgrads, vg.data(), vg.size() * sizeof(void*));
  if (e == cudaSuccess && param_ptrs) {
    e = cudaMalloc(reinterpret_cast<void**>(&t->vparams), bytes);
    if (e == cudaSuccess && !vp.empty())
      e = upload_table(t->vparams, vp.data(), vp.size() * sizeof(void*));
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_table(t);
    return fail(e == cudaErrorMemoryAllocation ? FSP_ENOMEM : FSP_ECUDA, cuda_msg("uploading the tensor table", e));
  }
  *out = t;
  return FSP_OK;
}

// Whether [ptr, ptr + bytes) overlaps a registered tensor.
bool overlaps_table(const fsp_param_table* t, const void* ptr, size_t bytes) {
  if (!bytes) return false;
  const uintptr_t b = reinterpret_cast<uintptr_t>(ptr), e = b + bytes;
  auto it = std::lower_bound(t->spans.begin(), t->spans.end(), std::make_pair(e, uintptr_t(0)));
  return it != t->spans.begin() && std::prev(it)->second > b;
}

// Checks shared by the per-parameter steps: plan / table / device, hp and t,
// and the state buffers (and `extra`) against each other and the tensors.
fsp_status check_params_step(const fsp_plan* p, const fsp_param_table* t, float* master, float* m, float* v,
                             const fsp_adamw_hparams* hp, int64_t step, const std::vector<Buf>& extra) {
  if (!p || !t) return fail(FSP_EINVAL, "plan or table is NULL");
  if (t->plan != p) return fail(FSP_EINVAL, "the table was created for another plan");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FSP_ECUDA, cuda_msg("cudaGetDevice", e));
  if (dev != t->device) return fail(FSP_EINVAL, "the table was created on another device");
  if (fsp_status hs = check_hparams(hp, step); hs != FSP_OK) return hs;
  const size_t sbytes = size_t(p->state_len_total) * 4;
  std::vector<Buf> bufs{{master, sbytes, "master"}, {m, sbytes, "exp_avg"}, {v, sbytes, "exp_avg_sq"}};
  for (const Buf& b : extra) bufs.push_back(b);
  for (const Buf& b : bufs) {
    if (!b.ptr && b.bytes) return fail(FSP_EINVAL, b.name + " is NULL");
    if (reinterpret_cast<uintptr_t>(b.ptr) % 16 != 0) return fail(FSP_EINVAL, b.name + " is not 16-byte aligned");
    if (overlaps_table(t, b.ptr, b.bytes)) return fail(FSP_EINVAL, b.name + " overlaps a registered tensor");
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
  return FSP_OK;
}

// The argument block of a per-parameter step on the current device.
fsp_status params_step_args(const fsp_plan* p, const fsp_param_table* t, float* master, float* m, float* v,
                            const fsp_adamw_hparams* hp, int64_t step, StepArgs* a) {
  const Tile* tiles = nullptr;
  fsp_status s = device_tiles(p, &tiles);
  if (s != FSP_OK) return s;
  *a = StepArgs{};
  a->vgrads = t->vgrads;
  a->vparams = t->vparams;
  a->gather = t->vparams ? 1 : 0;
  a->param_f32 = t->param_dtype == FSP_DTYPE_F32 ? 1 : 0;
  a->master = master;
  a->m = m;
  a->v = v;
  a->tiles = tiles;
  a->n_tiles = int64_t(p->tiles.size());
  set_mesh(*a, p);
  set_coeffs(*a, hp, step);
  return FSP_OK;
}

fsp_status run_step_params(const fsp_plan* p, const fsp_param_table* t, float* master, float* m, float* v,
                           const fsp_adamw_hparams* hp, int64_t step, void* stream) {
  clear_error();
  fsp_status s = check_params_step(p, t, master, m, v, hp, step, {});
  if (s != FSP_OK || p->tiles.empty()) return s;
  StepArgs a;
  s = params_step_args(p, t, master, m, v, hp, step, &a);
  if (s != FSP_OK) return s;
  return launch(a, t->grad_dtype, stream, false, nullptr, p);
}

fsp_status run_step_params_device_t(const fsp_plan* p, const fsp_param_table* t, float* master, float* m, float* v,
                                    const fsp_adamw_hparams* hp, int64_t* step_dev, int32_t advance, void* stream) {
  clear_error();
  if (!step_dev) return fail(FSP_EINVAL, "step_dev is NULL");
  if (reinterpret_cast<uintptr_t>(step_dev) % 8 != 0) return fail(FSP_EINVAL, "step_dev is not 8-byte aligned");
  // t only enters the bias corrections, which the kernel recomputes from *step_dev
  fsp_status s = check_params_step(p, t, master, m, v, hp, 1, {});
  if (s != FSP_OK) return s;
  if (overlaps_table(t, step_dev, sizeof(int64_t))) return fail(FSP_EINVAL, "step_dev overlaps a registered tensor");
  s = check_allocation(step_dev, sizeof(int64_t), "step_dev");
  if (s != FSP_OK) return s;
  if (!p->tiles.empty()) {
    StepArgs a;
    s = params_step_args(p, t, master, m, v, hp, 1, &a);
    if (s != FSP_OK) return s;
    a.step_dev = step_dev;
    s = launch(a, t->grad_dtype, stream, false, nullptr, p);
    if (s != FSP_OK) return s;
  }
  return advance ? advance_step(step_dev, stream) : FSP_OK;
}

fsp_status run_step_writeback_params(const fsp_plan* p, const fsp_param_table* t, float* master, float* m, float* v,
                                     const fsp_adamw_hparams* hp, int64_t step, void* stream) {
  clear_error();
  if (p && p->n_rep != 1) return fail(FSP_EUNSUPPORTED, "the write-back step is for FSDP2 plans");
  if (t && t->grad_dtype != FSP_DTYPE_F32)
    return fail(FSP_EUNSUPPORTED, "the write-back step stores the averaged gradient into fp32 gradient tensors");
  fsp_status s = check_params_step(p, t, master, m, v, hp, step, {});
  if (s != FSP_OK || p->tiles.empty()) return s;
  StepArgs a;
  s = params_step_args(p, t, master, m, v, hp, step, &a);
  if (s != FSP_OK) return s;
  a.writeback = 1;
  return launch(a, t->grad_dtype, stream, false, nullptr, p);
}

fsp_status run_step_clipped_params(const fsp_plan* p, const fsp_param_table* t, float* master, float* m, float* v,
                                   const fsp_adamw_hparams* hp, int64_t step, float max_norm, float* norm_out,
                                   void* stream) {
  clear_error();
  if (t && t->grad_dtype != FSP_DTYPE_F32)
    return fail(FSP_EUNSUPPORTED, "the clipped step writes back into fp32 gradient tensors");
  if (!(std::isfinite(max_norm) && max_norm > 0.f)) return fail(FSP_EINVAL, "max_norm must be finite and > 0");
  fsp_status s = check_params_step(p, t, master, m, v, hp, step, {{norm_out, 2 * sizeof(float), "norm_out"}});
  if (s != FSP_OK) return s;
  if (p->tiles.empty()) return clipped_empty(norm_out, stream);
  StepArgs a;
  s = params_step_args(p, t, master, m, v, hp, step, &a);
  if (s != FSP_OK) return s;
  return run_clipped_passes(p, a, max_norm, norm_out, stream);
}

}  // namespace
}  // namespace fsp

extern "C" fsp_status fsp_param_table_create(const fsp_plan* plan, const void* const* grad_ptrs, int32_t grad_dtype,
                                             void* const* param_ptrs, int32_t param_dtype,
                                             fsp_param_table** out) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::create_table(plan, grad_ptrs, grad_dtype, param_ptrs, param_dtype, out);
  });
}

extern "C" void fsp_param_table_destroy(fsp_param_table* table) { fsp::free_table(table); }

extern "C" fsp_status fsp_sharded_step_params_device_t(const fsp_plan* plan, const fsp_param_table* table,
                                                       float* master, float* exp_avg, float* exp_avg_sq,
                                                       const fsp_adamw_hparams* hp, int64_t* step_dev,
                                                       int32_t advance, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step_params_device_t(plan, table, master, exp_avg, exp_avg_sq, hp, step_dev, advance, cuda_stream);
  });
}

extern "C" fsp_status fsp_sharded_step_writeback_params(const fsp_plan* plan, const fsp_param_table* table,
                                                        float* master, float* exp_avg, float* exp_avg_sq,
                                                        const fsp_adamw_hparams* hp, int64_t step,
                                                        void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step_writeback_params(plan, table, master, exp_avg, exp_avg_sq, hp, step, cuda_stream);
  });
}

extern "C" fsp_status fsp_sharded_step_clipped_params(const fsp_plan* plan, const fsp_param_table* table,
                                                      float* master, float* exp_avg, float* exp_avg_sq,
                                                      const fsp_adamw_hparams* hp, int64_t step, float max_norm,
                                                      float* norm_out, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step_clipped_params(plan, table, master, exp_avg, exp_avg_sq, hp, step, max_norm, norm_out,
                                        cuda_stream);
  });
}

extern "C" fsp_status fsp_sharded_step_params(const fsp_plan* plan, const fsp_param_table* table, float* master,
                                              float* exp_avg, float* exp_avg_sq, const fsp_adamw_hparams* hp,
                                              int64_t step, void* cuda_stream) {
  return fsp::guard([&]() -> fsp_status {
    return fsp::run_step_params(plan, table, master, exp_avg, exp_avg_sq, hp, step, cuda_stream);
  });
}
