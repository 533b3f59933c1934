// Internal declarations shared by the planner (fsp_plan.cpp) and the step
// (fsp_step.cu).  Not part of the C ABI.
#pragma once

#include <cstdint>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include <cuda_runtime_api.h>

#include "fsp.h"

namespace fsp {

constexpr int kMaxRanks = 64;
constexpr int kMaxDims = 8;
// Work tiles never cross a multiple of this many elements of the full-size
// buffers, so only a segment's first and last tile can start or end off a
// vector boundary.
constexpr int64_t kTileElems = 4096;
// State segments start at a slot congruent to their full-buffer offset modulo
// this, so grads, params and state share vector alignment.
constexpr int64_t kStateAlign = 16;
// DistOpt buffers are padded to a multiple of lcm(N_d, this).
constexpr int64_t kDistOptAlign = 128;
// Per-parameter plans start every parameter at a multiple of this many
// elements of the (virtual) full index.
constexpr int64_t kParamAlign = 16;

// One unit of work for a CTA: `len` elements starting at `full_begin` of every
// full-size buffer and at `state_begin` of the state buffers, owned by `rank`
// (the rank whose shard the elements are; replica group 0 for HSDP), all in
// parameter `param` (-1 for a DistOpt shard, which spans parameters).  32
// bytes so a descriptor is two aligned 16-byte loads.
struct Tile {
  int64_t full_begin;
  int64_t state_begin;
  int32_t len;
  int32_t rank;
  int32_t param;
  int32_t reserved;
};
static_assert(sizeof(Tile) == 32, "tile descriptor layout");

}  // namespace fsp

struct fsp_plan {
  uint64_t uid = 0;       // unique among the process's plans (never reused)
  int32_t n_d = 0;
  int32_t n_rep = 1;      // HSDP replica groups; 1 for FSDP2 and DistOpt
  int32_t n_shard = 0;    // ranks per shard group (= n_d when n_rep == 1)
  int32_t n_params = 0;
  int32_t mode = 0;
  int64_t rep_stride = 0; // state elements between two replicas' copies
  int32_t param_align = 1; // 16: per-parameter buffers (virtual offsets); 1: full-size buffers
  std::vector<int64_t> param_off;    // each parameter's first full (virtual) index
  std::vector<int64_t> param_numel;
  int64_t valid_elems = 0;
  int64_t full_len_padded = 0;
  int64_t state_len_per_rank = 0;
  int64_t state_len_total = 0;
  std::vector<fsp_segment> segments;
  std::vector<fsp::Tile> tiles;   // one replica's elements (replica 0's state offsets)

  // Device copies of `tiles`, one per device ordinal, uploaded on first use,
  // and per device the per-CTA partial sums of the clipped step's norm.
  mutable std::mutex mu;
  mutable std::map<int, fsp::Tile*> device_tiles;
  mutable std::map<int, double*> device_partials;
  // Per device: `tiles` split at multiples of kStepTileElems (the step
  // kernels' schedule on full-size buffers) and their number.
  mutable std::map<int, std::pair<fsp::Tile*, int64_t>> device_step_tiles;
  // Per (device, grid): `tiles` in the order a fixed-stride launch of `grid`
  // CTAs takes them with its rounds balanced (balance_rounds); nullptr where
  // that order gains nothing (the launch keeps the plan's own order).
  mutable std::map<std::pair<int, int>, fsp::Tile*> device_round_tiles;
};

// Per-parameter tensors registered for a per-parameter plan on one device
// (fsp_params.cu): device tables of virtual bases, entry param * n_d + q, such
// that rank q's element at full index f of that parameter is at base + f.
struct fsp_param_table {
  const fsp_plan* plan = nullptr;
  int device = -1;
  int32_t grad_dtype = 0;
  int32_t param_dtype = 1;         // fsp_dtype of the param tensors (FSP_DTYPE_BF16 or FSP_DTYPE_F32)
  const void** vgrads = nullptr;   // device, n_params * n_d entries
  uint16_t** vparams = nullptr;    // device, or nullptr: no param tensors (fp32 ones are cast back)
  // every registered tensor as [begin, end) device addresses, sorted by begin
  std::vector<std::pair<uintptr_t, uintptr_t>> spans;
};

namespace fsp {

// Records the thread-local message behind an error status and returns it.
fsp_status fail(fsp_status s, const std::string& msg);
void clear_error();
// As fail, for a message that must not allocate (a string literal).
fsp_status fail_static(fsp_status s, const char* msg) noexcept;

// Runs the body of a C entry point: a host allocation failure (or any other
// C++ exception) becomes a status instead of crossing the C boundary.
template <typename F>
fsp_status guard(F&& body) noexcept {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    return fail_static(FSP_ENOMEM, "host allocation failed");
  } catch (...) {
    return fail_static(FSP_EINVAL, "unexpected host-side error");
  }
}
}  // namespace fsp
