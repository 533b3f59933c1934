// Host-side helpers shared by the translation units that launch kernels
// (defined in fsp_step.cu).  Not part of the C ABI.
#pragma once

#include <cuda_runtime_api.h>

#include <string>

#include "fsp_args.h"
#include "fsp_internal.h"

namespace fsp {

// A buffer an entry point validates: pointer, bytes, name for messages.
struct Buf {
  const void* ptr;
  size_t bytes;
  std::string name;
};

std::string cuda_msg(const char* what, cudaError_t e);
bool finite_nonneg(float x);
// Whether [ptr, ptr + bytes) lies inside one live allocation of the driver.
fsp_status check_allocation(const void* ptr, size_t bytes, const char* name);
// Copies a host table into device memory and returns once it has landed
// (a table that kernels on any stream may read).
cudaError_t upload_table(void* dst, const void* src, size_t bytes);
// The plan's tile table on the current device (uploaded on first use).
fsp_status device_tiles(const fsp_plan* p, const Tile** out);
// AdamW scalars of update t, and the plan's rank layout, into `a`.
void set_coeffs(StepArgs& a, const fsp_adamw_hparams* hp, int64_t step);
void set_mesh(StepArgs& a, const fsp_plan* p);
// hp and t within the ranges fsp.h states.
fsp_status check_hparams(const fsp_adamw_hparams* hp, int64_t step);
// Launches the step kernel for `a` (clip: the clipped update).
// On plans with many tiles per CTA (16, or 128 for the ZeRO-3 step of one
// replica group) the bulk kernel takes its tiles in order from a counter:
// `fixed_ctr` when given (zeroed here on `stream`), else one allocated from a
// library pool on `stream` and freed after the launch.
// With `step_plan` given, a launch of a large plan (at least 16 tiles per
// resident CTA) that holds all of that plan's tiles on full-size buffers with
// the all-gather (no clip, no per-parameter tables) runs on the plan's step
// tiles instead (the tiles split at multiples of 2048 elements, uploaded once
// per plan and device); a bulk launch of a smaller plan's tiles over several
// rounds of CTAs takes them in balanced order where that lowers the busiest
// CTA's work (uploaded once per plan and device).
// `early_start`: the bulk kernel is launched with programmatic stream
// serialisation (its prologue may overlap the previous kernel on the stream;
// it waits for that kernel on the device before reading or writing buffers).
fsp_status launch(StepArgs& a, int32_t dtype, void* stream, bool clip = false,
                  unsigned long long* fixed_ctr = nullptr, const fsp_plan* step_plan = nullptr,
                  bool early_start = true);
// Passes 1-3 of the clipped flow on a prepared argument block (non-empty
// plan, fp32 grads; HSDP plans too); clipped_empty writes norm_out = {0, 1}
// for a plan with nothing to reduce.
fsp_status run_clipped_passes(const fsp_plan* p, StepArgs& a, float max_norm, float* norm_out, void* stream);
fsp_status clipped_empty(float* norm_out, void* stream);
// *step_dev += 1 on `stream` (one thread).
fsp_status advance_step(int64_t* step_dev, void* stream);

}  // namespace fsp
