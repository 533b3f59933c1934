// Layout planner of the sharded step: which elements each simulated rank owns,
// where its fp32 state lives, and the tile list the kernel walks.
//
// FSDP2 Shard(0): "FSDP2 Qwen3 Decoder Layer Walkthrough", section "FSDP2 设置"
// and its per-rank shard table; "Parallelism strategies: which state to
// shard", section 二.5 (per-parameter dim-0 DTensor shards).
// DistOpt flat shards: "07 · 显存模型", section 2.1 item 1 (shards ignore
// parameter boundaries) and section 8 item 4 (lcm(DP, 128) padding).
#include <cuda_runtime_api.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <limits>
#include <new>

#include "fsp_internal.h"

namespace fsp {

namespace {
thread_local std::string g_last_error;

constexpr int64_t kMaxElems = int64_t(1) << 56;

int64_t gcd64(int64_t a, int64_t b) {
  while (b) {
    int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

int64_t round_up(int64_t x, int64_t m) { return m ? (x + m - 1) / m * m : x; }

// Cuts segment `s` into tiles at multiples of kTileElems of the full index.
void append_tiles(const fsp_segment& s, std::vector<Tile>& out) {
  int64_t f = s.full_off;
  const int64_t end = s.full_off + s.len;
  while (f < end) {
    int64_t stop = std::min(end, (f / kTileElems + 1) * kTileElems);
    out.push_back(Tile{f, s.state_off + (f - s.full_off), int32_t(stop - f), s.rank, s.param, 0});
    f = stop;
  }
}

}  // namespace

// The message buffer used when recording a message could itself fail.
thread_local const char* g_static_error = nullptr;

fsp_status fail(fsp_status s, const std::string& msg) {
  g_static_error = nullptr;
  g_last_error = msg;
  return s;
}
fsp_status fail_static(fsp_status s, const char* msg) noexcept {
  g_static_error = msg;
  return s;
}
void clear_error() {
  g_static_error = nullptr;
  g_last_error.clear();
}
const char* last_error() { return g_static_error ? g_static_error : g_last_error.c_str(); }

}  // namespace fsp

using fsp::fail;

extern "C" const char* fsp_last_error(void) { return fsp::last_error(); }

extern "C" const char* fsp_status_string(fsp_status s) {
  switch (s) {
    case FSP_OK: return "ok";
    case FSP_EINVAL: return "invalid argument";
    case FSP_ENOMEM: return "out of memory";
    case FSP_ECUDA: return "CUDA error";
    case FSP_EUNSUPPORTED: return "unsupported";
  }
  return "unknown status";
}

namespace {

// Rows (dim 0), cols (product of the other dims) and start of each param in
// the full index (rounded up to a multiple of `align`); total = elements,
// extent = end of the last parameter.
fsp_status parse_shapes(const int64_t* dims, const int32_t* ndims, int32_t n_params, int64_t align,
                        std::vector<int64_t>& rows, std::vector<int64_t>& cols, std::vector<int64_t>& start,
                        int64_t& total, int64_t& extent) {
  if (n_params < 0) return fail(FSP_EINVAL, "fsp_plan_layout: n_params < 0");
  if (n_params > 0 && (!dims || !ndims)) return fail(FSP_EINVAL, "fsp_plan_layout: dims or ndims is NULL");
  rows.assign(n_params, 0);
  cols.assign(n_params, 0);
  start.assign(n_params, 0);
  int64_t cursor = 0;
  total = 0;
  extent = 0;
  for (int32_t i = 0; i < n_params; ++i) {
    if (ndims[i] < 1 || ndims[i] > fsp::kMaxDims)
      return fail(FSP_EINVAL, "fsp_plan_layout: ndims[" + std::to_string(i) + "] must be in [1, 8]");
    int64_t c = 1;
    for (int32_t k = 0; k < ndims[i]; ++k) {
      const int64_t d = dims[cursor + k];
      if (d < 0) return fail(FSP_EINVAL, "fsp_plan_layout: negative dim in parameter " + std::to_string(i));
      if (k == 0) {
        rows[i] = d;
      } else {
        if (d != 0 && c > fsp::kMaxElems / d) return fail(FSP_EINVAL, "fsp_plan_layout: parameter too large");
        c *= d;
      }
    }
    cursor += ndims[i];
    cols[i] = c;
    if (rows[i] != 0 && c > fsp::kMaxElems / rows[i]) return fail(FSP_EINVAL, "fsp_plan_layout: parameter too large");
    start[i] = fsp::round_up(extent, align);
    total += rows[i] * c;
    extent = start[i] + rows[i] * c;
    if (extent > fsp::kMaxElems) return fail(FSP_EINVAL, "fsp_plan_layout: model too large");
  }
  return FSP_OK;
}

// FSDP2 Shard(0) over n_shard ranks, repeated for n_rep replica groups.
void build_fsdp2(fsp_plan* p, const std::vector<int64_t>& rows, const std::vector<int64_t>& cols,
                 const std::vector<int64_t>& start, int64_t extent, int32_t n_shard, int32_t n_rep) {
  const int32_t n_params = int32_t(rows.size());
  p->full_len_padded = extent;
  // each shard rank's local slot for each (param, rank)
  std::vector<int64_t> local(size_t(n_params) * n_shard);
  int64_t widest = 0;
  for (int32_t r = 0; r < n_shard; ++r) {
    int64_t at = 0;
    for (int32_t i = 0; i < n_params; ++i) {
      const int64_t c = (rows[i] + n_shard - 1) / n_shard;  // padded shard height
      const int64_t first = std::min<int64_t>(int64_t(r) * c, rows[i]);
      const int64_t full_off = start[i] + first * cols[i];
      // first slot >= at with slot == full_off (mod kStateAlign)
      const int64_t want = full_off % fsp::kStateAlign;
      const int64_t have = at % fsp::kStateAlign;
      at += (want - have + fsp::kStateAlign) % fsp::kStateAlign;
      local[size_t(r) * n_params + i] = at;
      at += c * cols[i];
    }
    widest = std::max(widest, at);
  }
  p->state_len_per_rank = fsp::round_up(widest, fsp::kStateAlign);
  p->rep_stride = p->state_len_per_rank * n_shard;
  p->state_len_total = p->rep_stride * n_rep;
  p->segments.reserve(size_t(n_params) * n_shard * n_rep);
  for (int32_t g = 0; g < n_rep; ++g) {
    for (int32_t r = 0; r < n_shard; ++r) {
      for (int32_t i = 0; i < n_params; ++i) {
        const int64_t c = (rows[i] + n_shard - 1) / n_shard;
        const int64_t first = std::min<int64_t>(int64_t(r) * c, rows[i]);
        const int64_t owned_rows = std::min<int64_t>(c, rows[i] - first);
        fsp_segment s;
        s.param = i;
        s.rank = g * n_shard + r;
        s.full_off = start[i] + first * cols[i];
        s.state_off = g * p->rep_stride + int64_t(r) * p->state_len_per_rank + local[size_t(r) * n_params + i];
        s.len = owned_rows * cols[i];
        s.padded_len = c * cols[i];
        p->segments.push_back(s);
      }
    }
  }
}

// Tiles of replica 0's segments, in full-index order so a CTA's consecutive
// tiles are neighbours in every buffer.
void build_tiles(fsp_plan* p) {
  std::vector<const fsp_segment*> order;
  order.reserve(p->segments.size());
  for (const auto& s : p->segments)
    if (s.len > 0 && s.rank < p->n_shard) order.push_back(&s);
  std::sort(order.begin(), order.end(),
            [](const fsp_segment* a, const fsp_segment* b) { return a->full_off < b->full_off; });
  p->tiles.reserve(size_t(p->valid_elems / fsp::kTileElems + 2 * order.size() + 1));
  for (const fsp_segment* s : order) fsp::append_tiles(*s, p->tiles);
}

fsp_status make_plan(const int64_t* dims, const int32_t* ndims, int32_t n_params, int32_t n_rep, int32_t n_shard,
                     int32_t mode, int32_t param_align, fsp_plan** out) {
  std::vector<int64_t> rows, cols, start;
  int64_t total = 0, extent = 0;
  fsp_status st = parse_shapes(dims, ndims, n_params, param_align, rows, cols, start, total, extent);
  if (st != FSP_OK) return st;
  fsp_plan* p = new (std::nothrow) fsp_plan();
  if (!p) return fail(FSP_ENOMEM, "fsp_plan_layout: host allocation failed");
  static std::atomic<uint64_t> next_uid{1};
  p->uid = next_uid.fetch_add(1);
  try {
    p->n_d = n_rep * n_shard;
    p->n_rep = n_rep;
    p->n_shard = n_shard;
    p->n_params = n_params;
    p->mode = mode;
    p->valid_elems = total;
    p->param_align = param_align;
    p->param_off = start;
    p->param_numel.resize(size_t(n_params));
    for (int32_t i = 0; i < n_params; ++i) p->param_numel[size_t(i)] = rows[size_t(i)] * cols[size_t(i)];
    if (mode == FSP_MODE_DISTOPT_FLAT) {
      const int32_t n_d = n_shard;
      const int64_t unit = int64_t(n_d) / fsp::gcd64(n_d, fsp::kDistOptAlign) * fsp::kDistOptAlign;
      p->full_len_padded = fsp::round_up(total, unit);
      p->state_len_per_rank = p->full_len_padded / n_d;
      p->state_len_total = p->full_len_padded;
      p->rep_stride = p->state_len_total;
      for (int32_t r = 0; r < n_d; ++r) {
        fsp_segment s;
        s.param = -1;
        s.rank = r;
        s.full_off = int64_t(r) * p->state_len_per_rank;
        s.state_off = s.full_off;
        s.len = std::max<int64_t>(0, std::min<int64_t>(p->state_len_per_rank, total - s.full_off));
        s.padded_len = p->state_len_per_rank;
        p->segments.push_back(s);
      }
    } else {
      build_fsdp2(p, rows, cols, start, extent, n_shard, n_rep);
    }
    build_tiles(p);
  } catch (const std::bad_alloc&) {
    delete p;
    return fail(FSP_ENOMEM, "fsp_plan_layout: host allocation failed");
  }
  *out = p;
  return FSP_OK;
}

}  // namespace

extern "C" fsp_status fsp_plan_layout(const int64_t* dims, const int32_t* ndims, int32_t n_params,
                                      int32_t n_d, int32_t mode, fsp_plan** out) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!out) return fail(FSP_EINVAL, "fsp_plan_layout: out is NULL");
    *out = nullptr;
    if (n_d < 1 || n_d > fsp::kMaxRanks) return fail(FSP_EINVAL, "fsp_plan_layout: n_d must be in [1, 64]");
    if (mode != FSP_MODE_FSDP2_SHARD0 && mode != FSP_MODE_DISTOPT_FLAT)
      return fail(FSP_EINVAL, "fsp_plan_layout: unknown mode");
    return make_plan(dims, ndims, n_params, 1, n_d, mode, 1, out);
  });
}

extern "C" fsp_status fsp_plan_layout_hsdp(const int64_t* dims, const int32_t* ndims, int32_t n_params,
                                           int32_t n_replicate, int32_t n_shard, fsp_plan** out) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!out) return fail(FSP_EINVAL, "fsp_plan_layout_hsdp: out is NULL");
    *out = nullptr;
    if (n_replicate < 1 || n_shard < 1 || int64_t(n_replicate) * n_shard > fsp::kMaxRanks)
      return fail(FSP_EINVAL, "fsp_plan_layout_hsdp: need n_replicate, n_shard >= 1 and their product <= 64");
    return make_plan(dims, ndims, n_params, n_replicate, n_shard, FSP_MODE_HSDP, 1, out);
  });
}

extern "C" fsp_status fsp_plan_layout_params(const int64_t* dims, const int32_t* ndims, int32_t n_params,
                                             int32_t n_replicate, int32_t n_shard, fsp_plan** out) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!out) return fail(FSP_EINVAL, "fsp_plan_layout_params: out is NULL");
    *out = nullptr;
    if (n_replicate < 1 || n_shard < 1 || int64_t(n_replicate) * n_shard > fsp::kMaxRanks)
      return fail(FSP_EINVAL, "fsp_plan_layout_params: need n_replicate, n_shard >= 1 and their product <= 64");
    return make_plan(dims, ndims, n_params, n_replicate, n_shard,
                     n_replicate == 1 ? FSP_MODE_FSDP2_SHARD0 : FSP_MODE_HSDP, int32_t(fsp::kParamAlign), out);
  });
}

extern "C" fsp_status fsp_plan_param(const fsp_plan* p, int32_t i, int64_t* full_off, int64_t* numel) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!p || !full_off || !numel) return fail(FSP_EINVAL, "fsp_plan_param: NULL argument");
    if (i < 0 || i >= p->n_params) return fail(FSP_EINVAL, "fsp_plan_param: index out of range");
    *full_off = p->param_off[size_t(i)];
    *numel = p->param_numel[size_t(i)];
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_plan_info_get(const fsp_plan* p, fsp_plan_info* out) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!p || !out) return fail(FSP_EINVAL, "fsp_plan_info_get: NULL argument");
    out->n_d = p->n_d;
    out->n_params = p->n_params;
    out->mode = p->mode;
    out->tile_elems = int32_t(fsp::kTileElems);
    out->valid_elems = p->valid_elems;
    out->full_len_padded = p->full_len_padded;
    out->state_len_per_rank = p->state_len_per_rank;
    out->state_len_total = p->state_len_total;
    out->n_segments = int64_t(p->segments.size());
    out->n_tiles = int64_t(p->tiles.size());
    out->n_replicate = p->n_rep;
    out->n_shard = p->n_shard;
    out->param_align = p->param_align;
    out->reserved = 0;
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_plan_segment(const fsp_plan* p, int64_t i, fsp_segment* out) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!p || !out) return fail(FSP_EINVAL, "fsp_plan_segment: NULL argument");
    if (i < 0 || i >= int64_t(p->segments.size())) return fail(FSP_EINVAL, "fsp_plan_segment: index out of range");
    *out = p->segments[size_t(i)];
    return FSP_OK;
  });
}

extern "C" fsp_status fsp_plan_ledger(const fsp_plan* p, int32_t grad_dtype, fsp_ledger* out) {
  return fsp::guard([&]() -> fsp_status {
    fsp::clear_error();
    if (!p || !out) return fail(FSP_EINVAL, "fsp_plan_ledger: NULL argument");
    if (grad_dtype != FSP_DTYPE_F32 && grad_dtype != FSP_DTYPE_BF16)
      return fail(FSP_EINVAL, "fsp_plan_ledger: unknown grad dtype");
    const double P = double(p->valid_elems), n = double(p->n_d);
    const double ns = double(p->n_shard), nr = double(p->n_rep);
    const double g = grad_dtype == FSP_DTYPE_F32 ? 4.0 : 2.0;
    out->resident_ddp = (2.0 + g + 12.0) * P;
    out->resident_distopt = (2.0 + g) * P + 12.0 * P / n;
    out->resident_zero2 = 2.0 * P + (g + 12.0) * P / n;
    out->resident_fsdp = (2.0 + g + 12.0) * P / n;
    // collectives of this plan's own layout (the shard group for HSDP)
    out->reduce_scatter_sent = (ns - 1.0) / ns * g * P;
    out->all_gather_sent = (ns - 1.0) / ns * 2.0 * P;
    out->step_hbm_bytes = (n * g + 24.0 * nr + 2.0 * n) * P;
    out->resident_hsdp = (2.0 + g + 12.0) * P / ns;
    out->cross_group_all_reduce_sent = nr > 1.0 ? 2.0 * (nr - 1.0) / nr * g * P / ns : 0.0;
    return FSP_OK;
  });
}

extern "C" void fsp_plan_destroy(fsp_plan* p) {
  if (!p) return;
  if (!p->device_tiles.empty() || !p->device_partials.empty() || !p->device_step_tiles.empty() ||
      !p->device_round_tiles.empty()) {
    std::lock_guard<std::mutex> lock(p->mu);
    int prev = -1;
    const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
    for (auto& kv : p->device_tiles) {
      if (cudaSetDevice(kv.first) == cudaSuccess) cudaFree(kv.second);
    }
    for (auto& kv : p->device_partials) {
      if (cudaSetDevice(kv.first) == cudaSuccess) cudaFree(kv.second);
    }
    for (auto& kv : p->device_step_tiles) {
      if (cudaSetDevice(kv.first) == cudaSuccess) cudaFree(kv.second.first);
    }
    for (auto& kv : p->device_round_tiles) {
      if (kv.second && cudaSetDevice(kv.first.first) == cudaSuccess) cudaFree(kv.second);
    }
    if (have_prev) cudaSetDevice(prev);
    p->device_tiles.clear();
    p->device_partials.clear();
    p->device_step_tiles.clear();
    p->device_round_tiles.clear();
  }
  delete p;
}
