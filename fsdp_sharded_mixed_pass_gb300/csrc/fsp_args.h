// Argument block of the step kernels, shared by the host code that fills it
// (fsp_step.cu, fsp_host.cu) and the device code that reads it
// (fsp_kernels.cuh).  Plain data: passed by value as a __grid_constant__.
#pragma once

#include <cstdint>

#include "fsp_internal.h"

namespace fsp {

// Scalars of one AdamW update.  The kernel evaluates the update with float
// pairs (hi + lo), so every scalar that is not an fp32 number of its own
// (1 - beta, 1 - lr wd and the two bias-correction factors) is carried as the
// pair hi = fl(x), lo = fl(x - hi) of its double value.
struct Coeffs {
  float beta1, one_minus_beta1_hi, one_minus_beta1_lo;
  float beta2, one_minus_beta2_hi, one_minus_beta2_lo;
  float decay_hi, decay_lo;   // 1 - lr * weight_decay
  float step_hi, step_lo;     // lr / (1 - beta1^t)
  float isb_hi, isb_lo;       // 1 / sqrt(1 - beta2^t)
  float eps;
};

struct StepArgs {
  const void* grads[kMaxRanks];
  uint16_t* params[kMaxRanks];
  float* master;
  float* m;
  float* v;
  float* reduced;   // averaged shard gradient (state layout); nullptr in production
  // Per-parameter plans: device tables of "virtual base" pointers, entry
  // param * n_d + q, such that rank q's element at full index f of that
  // parameter is at base + f; nullptr for full-size buffers (grads / params).
  const void* const* vgrads;
  uint16_t* const* vparams;
  const Tile* tiles;
  int64_t n_tiles;
  // Bulk kernel: tiles are taken in order from this counter (zeroed before the
  // launch, one per launch); nullptr: CTA b takes tiles b, b + grid, ...
  unsigned long long* tile_ctr;
  int n_d;             // = n_rep * n_shard
  int n_rep;           // HSDP replica groups (1: FSDP2 / DistOpt)
  int n_shard;         // ranks per shard group; rank q = r * n_shard + j
  int64_t rep_stride;  // state elements between replica r's copy and r + 1's
  const float* clip;   // clipped update: {norm, coefficient} on the device
  const int64_t* step_dev;  // update index t in device memory (nullptr: t is folded into c)
  int gather;               // 0: ZeRO-3 / FSDP2 reshard - no all-gather, params untouched
  int writeback;            // 1: the averaged gradient also goes into the owner's slice of its fp32 grad buffer
  int param_f32;            // 1: the parameter buffers / tensors are fp32 (all-gather of the master, no cast)
  float lr;                 // kept to rebuild c's t-dependent scalars from *step_dev
  Coeffs c;
};

}  // namespace fsp
