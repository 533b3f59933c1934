/*
 * fsp.h - C ABI of the GB300 sharded mixed-precision optimizer step.
 *
 * One data-parallel training step of ZeRO / FSDP with N_d ranks simulated as
 * N_d separate buffers on one GPU:
 *
 *   (1) reduce-scatter: the owner of every element receives the sum over all
 *       ranks of that element's gradient, taken as an fp32 left fold in rank
 *       order 0..N_d-1, then divided (IEEE, round to nearest) by N_d.
 *       "FSDP2 Qwen3 Decoder Layer Walkthrough", section "Backward 简述";
 *       "Parallelism strategies: which state to shard", section 二.2.
 *   (2) AdamW on the owner's fp32 master / Adam m / Adam v shard, with no
 *       communication.  "07 · 显存模型", section 2.1 (fp32 master + m/v).
 *       Each element is updated in fp32; where the new master cancels
 *       (theta (1 - lr wd) - u below 2^-10 of its terms' size) it is
 *       evaluated again with pairs of floats (about 2^-44 of the terms'
 *       size), so every stored fp32 result is close to the exactly rounded
 *       value and its bf16 cast within one ulp of the exact update's.
 *   (3) cast of the new master to bf16 (round to nearest even) and all-gather
 *       into every rank's full bf16 param buffer.
 *       "FSDP2 Qwen3 Decoder Layer Walkthrough", section "Step 0".
 *
 * Steps (1)-(3) run as one fused streaming kernel: every gradient is read
 * once, the fp32 state is read and written once, every bf16 copy is written
 * once; the reduced gradient is never stored (except by the debug entry).
 * For N_d in {1..8, 12, 16} (and the HSDP meshes 2x2, 4x2, 8x2, 2x4, 4x4) the
 * kernel stages the gradient and state slices in shared memory with bulk
 * asynchronous copies and writes the N_d bf16 copies as bulk stores of one
 * tile; other N_d (up to 64) use per-thread vector loads and stores.
 * Gradients and parameters are either one full-size buffer per rank
 * (fsp_plan_layout / fsp_plan_layout_hsdp with the *_step entries) or one
 * tensor per parameter per rank (fsp_plan_layout_params with an
 * fsp_param_table and the *_params entries).
 *
 * Conventions for every function below:
 *   - Return FSP_OK or an error status; fsp_last_error() then gives a
 *     one-line, thread-local description.  Argument errors are detected on the
 *     host before anything is launched; no function traps or asserts on the
 *     device, and the only device-side waits are the step kernel's bounded
 *     waits on its own copy pipeline (see fsp_device_error).
 *   - The caller owns every device buffer and the CUDA stream.  The library
 *     owns plans and, per device, small read-only tables of work tiles that a
 *     plan uploads on its first step on that device (the plan's tiles and, for
 *     steps with the all-gather on full-size buffers of large plans, the same
 *     tiles split at 2048 elements; one cudaMalloc and one synchronous copy
 *     each; make that first call outside any stream capture).
 *     It also owns one CUDA memory pool per device: a step whose plan has at
 *     least 16 work tiles per SM (the ZeRO-3 step of one replica group: 128)
 *     takes an 8-byte tile counter from it on the step's stream, zeroed
 *     before the kernel and freed after it
 *     (stream-ordered, so concurrent steps and CUDA-graph replays each get
 *     their own; the kernel hands its tiles out in order from it).
 *   - Steps are asynchronous on the given stream (NULL = legacy default
 *     stream) and run on the current CUDA device.  Stream order is kept: the
 *     bulk step kernel and the unshard kernel are launched with programmatic
 *     stream serialisation, so right after another kernel on the stream their
 *     CTAs may start and set up while that kernel finishes, but they read and
 *     write no buffer before it has completed.  (The host-buffer entry
 *     launches the step kernel plainly.)
 *     "One synchronous copy" above returns only once the table has landed.
 *   - A plan may be used from several threads at once; fsp_plan_destroy must
 *     not race with any call or in-flight step using the same plan.
 */
#ifndef FSP_H
#define FSP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FSP_OK = 0,
  FSP_EINVAL = 1,        /* bad argument (null, range, alignment, overlap, size) */
  FSP_ENOMEM = 2,        /* host or device allocation failed                       */
  FSP_ECUDA = 3,         /* a CUDA runtime call or kernel launch failed             */
  FSP_EUNSUPPORTED = 4   /* valid request the library does not handle              */
} fsp_status;

typedef enum {
  /* FSDP2 per-parameter Shard(0): each parameter is split on dim 0 into N_d
   * chunks of c = ceil(rows / N_d) rows; rank r owns rows [r*c, min((r+1)*c,
   * rows)) and holds a padded shard of c rows.  "FSDP2 Qwen3 Decoder Layer
   * Walkthrough", section "FSDP2 设置"; "Parallelism strategies: which state to
   * shard", section 二.5. */
  FSP_MODE_FSDP2_SHARD0 = 0,
  /* Megatron distributed optimizer (ZeRO-1): all parameters form one flat
   * buffer padded to a multiple of lcm(N_d, 128) and cut into N_d equal
   * contiguous shards that ignore parameter boundaries.  "07 · 显存模型",
   * section 2.1 item 1 and section 8 item 4. */
  FSP_MODE_DISTOPT_FLAT = 1,
  /* HSDP: the N_d = N_r * N_s ranks form a (replicate, shard) mesh, rank
   * q = r * N_s + j.  Each replica group r shards the parameters FSDP2-style
   * over its N_s ranks and keeps its own copy of the fp32 state; gradients are
   * reduce-scattered inside each group (rank-ordered fp32 fold over its N_s
   * ranks), then all-reduced across the N_r groups (fold of the partial sums in
   * group order), divided by N_d; each group all-gathers its bf16 params.
   * "Parallelism strategies: which state to shard", section 二.6.  Created by
   * fsp_plan_layout_hsdp. */
  FSP_MODE_HSDP = 2
} fsp_mode;

typedef enum {
  FSP_DTYPE_F32 = 0,     /* fp32 main grads (grad_reduce_in_fp32 on)            */
  FSP_DTYPE_BF16 = 1     /* bf16 grads, widened exactly and reduced in fp32      */
} fsp_dtype;

typedef struct fsp_plan fsp_plan;   /* opaque; created by fsp_plan_layout */

/* AdamW hyper-parameters (fp32).  Update index t is passed to the step.
 * Requires lr >= 0, 0 <= beta1 < 1, 0 <= beta2 < 1, eps >= 0, weight_decay >= 0,
 * all finite. */
typedef struct {
  float lr;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
} fsp_adamw_hparams;

/* Sizes of the buffers a step on this plan reads and writes (in elements). */
typedef struct {
  int32_t n_d;
  int32_t n_params;
  int32_t mode;                 /* fsp_mode                                          */
  int32_t tile_elems;           /* largest work tile                                 */
  int64_t valid_elems;          /* P: parameters in the model                        */
  int64_t full_len_padded;      /* length of each grad_bufs[r] and param_bufs[r]      */
  int64_t state_len_per_rank;   /* one rank's shard of master / m / v                 */
  int64_t state_len_total;      /* length of master, m and v: n_d * state_len_per_rank */
  int64_t n_segments;
  int64_t n_tiles;
  int32_t n_replicate;          /* N_r: HSDP replica groups (1 otherwise)            */
  int32_t n_shard;              /* N_s: ranks per shard group (n_d otherwise)         */
  int32_t param_align;          /* 16: per-parameter plan (fsp_plan_layout_params); 1 */
  int32_t reserved;
} fsp_plan_info;

/* One contiguous run of a rank's shard.  Elements [full_off, full_off + len)
 * of every full-size buffer live in slots [state_off, state_off + len) of
 * master / m / v; slots [state_off + len, state_off + padded_len) are shard
 * padding and are never written.  param = -1 for a DistOpt shard.  HSDP:
 * replica group r's copy of the state is the state_len_total / N_r slots
 * starting at r * state_len_total / N_r. */
typedef struct {
  int32_t param;
  int32_t rank;
  int64_t full_off;
  int64_t state_off;
  int64_t len;
  int64_t padded_len;
} fsp_segment;

/* Per-rank byte ledger of this plan's model ("07 · 显存模型", section 2.1;
 * "Parallelism strategies: which state to shard", section 九 Q1 and its
 * coll_bytes listing), for the given gradient dtype. */
typedef struct {
  double resident_ddp;        /* (2 + g + 12) P                     */
  double resident_distopt;    /* (2 + g) P + 12 P / N_d             */
  double resident_zero2;      /* 2 P + (g + 12) P / N_d             */
  double resident_fsdp;       /* (2 + g + 12) P / N_d               */
  double reduce_scatter_sent; /* (N_s - 1) / N_s * g P  (N_s = N_d unless HSDP) */
  double all_gather_sent;     /* (N_s - 1) / N_s * 2 P              */
  double step_hbm_bytes;      /* (N_d g + 24 N_r + 2 N_d) P: one fused step on one GPU */
  double resident_hsdp;       /* (2 + g + 12) P / N_s               */
  double cross_group_all_reduce_sent; /* 2 (N_r - 1) / N_r * g P / N_s (0 when N_r = 1) */
} fsp_ledger;

/* Plans the layout of n_params parameters over n_d simulated ranks.
 *   dims:    the parameters' shapes, row-major, concatenated (sum of ndims
 *            entries, each >= 0); host memory, read during the call only.
 *   ndims:   number of dims of each parameter, 1..8.
 *   n_params >= 0 (0 gives an empty plan), 1 <= n_d <= 64, mode an fsp_mode.
 * FSDP2 state placement: master/m/v are rank-major (rank r's shard starts at
 * r * state_len_per_rank); inside a rank, segments follow parameter order and
 * each starts at the first slot at or after the previous one's end that is
 * congruent to its full_off modulo 16.  DistOpt: state index = flat index.
 * On success *out owns a new plan (free with fsp_plan_destroy). */
fsp_status fsp_plan_layout(const int64_t* dims, const int32_t* ndims, int32_t n_params,
                           int32_t n_d, int32_t mode, fsp_plan** out);

/* HSDP plan (FSP_MODE_HSDP) of n_replicate groups of n_shard ranks each
 * (n_replicate, n_shard >= 1, product <= 64); dims / ndims / n_params as for
 * fsp_plan_layout.  master / m / v then hold n_replicate copies of the
 * n_shard-rank FSDP2 state (state_len_total covers all of them). */
fsp_status fsp_plan_layout_hsdp(const int64_t* dims, const int32_t* ndims, int32_t n_params,
                                int32_t n_replicate, int32_t n_shard, fsp_plan** out);

/* Per-parameter plan: FSDP2 (n_replicate == 1) or HSDP over n_replicate groups
 * of n_shard ranks, for steps that read each rank's gradient of each
 * parameter from a tensor of its own and write its bf16 parameter into a
 * tensor of its own - FSDP2's per-parameter tensors, whose copy-in before the
 * reduce-scatter and copy-out after the all-gather the step then does in
 * place ("Parallelism strategies: which state to shard", section 二.5).
 * Parameter i occupies [full_off_i, full_off_i + numel_i) of a virtual full
 * index, full_off_i being the previous parameter's end rounded up to a
 * multiple of 16 (fsp_plan_param); shards, segments, state placement and
 * tiles follow from that index exactly as for fsp_plan_layout /
 * fsp_plan_layout_hsdp (full_len_padded is the index's extent; the gaps belong
 * to no rank).  Use with fsp_param_table_create, fsp_sharded_step_params and
 * fsp_unshard_params. */
fsp_status fsp_plan_layout_params(const int64_t* dims, const int32_t* ndims, int32_t n_params,
                                  int32_t n_replicate, int32_t n_shard, fsp_plan** out);

/* Parameter i's first full (virtual, for per-parameter plans) index and its
 * number of elements (0 <= i < n_params). */
fsp_status fsp_plan_param(const fsp_plan* plan, int32_t i, int64_t* full_off, int64_t* numel);

fsp_status fsp_plan_info_get(const fsp_plan* plan, fsp_plan_info* out);

/* Segment i (0 <= i < n_segments).  FSDP2 and HSDP: ordered by rank, then
 * parameter.  DistOpt: one segment per rank. */
fsp_status fsp_plan_segment(const fsp_plan* plan, int64_t i, fsp_segment* out);

fsp_status fsp_plan_ledger(const fsp_plan* plan, int32_t grad_dtype, fsp_ledger* out);

/* One unit of work of the step kernels: `len` elements from full index
 * `full_begin` (of every rank's buffer) and state index `state_begin`, owned
 * by rank `rank`, inside parameter `param` (-1: a DistOpt shard). */
typedef struct {
  int64_t full_begin, state_begin;
  int32_t len, rank, param, reserved;
} fsp_tile;

/* The work tiles (host only, no device call).  unit == 0: the plan's tiles,
 * each non-empty segment cut at multiples of 4096 elements of the full index,
 * in full-index order - the tiles of small plans (in fsp_plan_round_order's
 * order), the ZeRO-3 step, per-parameter tensors, the clipped flow, the
 * unshard and the host-buffer step.  unit > 0 (a multiple of 8 that divides
 * 4096): those tiles split at multiples of `unit` elements, in the same
 * order; the step kernels run steps with the all-gather on full-size buffers
 * of plans with at least 16 tiles per resident CTA on unit 2048.
 * Step kernels take the tiles in order from a counter on plans with at least
 * 16 tiles per CTA (128 for the ZeRO-3 step of one replica group), else CTA
 * b takes entries b, b + grid, ... of the round order below.  The number goes to *n; up to `cap` tiles to `out` (out may be
 * NULL when cap is 0). */
fsp_status fsp_plan_tiles(const fsp_plan* plan, int32_t unit, fsp_tile* out, int64_t cap, int64_t* n);

/* The order in which the bulk step kernel, launched with `grid` (>= 1) CTAs,
 * takes the plan's tiles when it strides over them (plans with fewer than 16
 * tiles per CTA, or 128 for the ZeRO-3 step of one replica group; CTA b takes
 * entries b, b + grid, b + 2 grid, ...).  Host
 * only.  Each round of `grid` consecutive tiles is handed out longest first
 * to the CTAs with the fewest 1024-element chunks so far (a partial chunk
 * counts as one), the CTAs renumbered so that the last, partial round goes to
 * CTAs 0 .. n - 1; this order is used only where it lowers the busiest CTA's
 * chunk count, else the plan's own order is (and is what this returns).
 * Every round holds the same tiles as in the plan's order.  *n, out, cap as
 * in fsp_plan_tiles; grid < 1: FSP_EINVAL. */
fsp_status fsp_plan_round_order(const fsp_plan* plan, int32_t grid, fsp_tile* out, int64_t cap, int64_t* n);

/* Frees the plan and its device tile tables.  NULL is a no-op. */
void fsp_plan_destroy(fsp_plan* plan);

/* The fused step (1)-(3), asynchronous on `cuda_stream` (a cudaStream_t).
 *   grad_bufs:  host array of n_d device pointers, each full_len_padded
 *               elements of grad_dtype; only read.
 *   master, exp_avg, exp_avg_sq: device, fp32, state_len_total elements each;
 *               updated in place at owned slots only.
 *   param_bufs: host array of n_d device pointers, each full_len_padded bf16
 *               elements; owned elements written, padding untouched.  NULL:
 *               no all-gather - the ZeRO-3 / FSDP2 step that leaves the
 *               parameters sharded (only master/m/v change; gather them
 *               later with fsp_unshard).
 *   hp:         host pointer; step: t >= 1, the 1-based index of this update
 *               (bias corrections use beta^t).
 * Every device pointer must be 16-byte aligned and no two buffers may
 * overlap.  Each device pointer must lie in a live CUDA allocation that holds
 * the whole buffer (checked with the driver).  A pointer may be NULL only
 * where its buffer has zero elements.  An empty plan returns FSP_OK and
 * launches nothing. */
fsp_status fsp_sharded_step(const fsp_plan* plan, const void* const* grad_bufs, int32_t grad_dtype,
                            float* master, float* exp_avg, float* exp_avg_sq,
                            void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                            void* cuda_stream);

/* fsp_sharded_step with the update index t read from device memory, for
 * loops captured once in a CUDA graph and replayed: the kernel computes the
 * bias corrections of t = *step_dev (in double, as the host would) and, when
 * `advance` is non-zero, a one-thread kernel then adds 1 to *step_dev on the
 * same stream, so each replay applies the next update.  step_dev: device,
 * 8-byte aligned int64 inside a live allocation; a value below 1 is treated as
 * 1 and sets bit 8 of the device error word.  Everything else as
 * fsp_sharded_step (make the first call on a device outside any capture). */
fsp_status fsp_sharded_step_device_t(const fsp_plan* plan, const void* const* grad_bufs, int32_t grad_dtype,
                                     float* master, float* exp_avg, float* exp_avg_sq,
                                     void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t* step_dev,
                                     int32_t advance, void* cuda_stream);

/* The Megatron distributed-optimizer flow with global-norm gradient clipping,
 * for FSDP2, DistOpt and HSDP plans with fp32 grads (bf16: FSP_EUNSUPPORTED):
 *   1. reduce-scatter with write-back: every element's averaged gradient
 *      (the rank-ordered fp32 fold / N_d; HSDP: the fold inside each replica
 *      group, then across groups, as fsp_sharded_step) is stored into its
 *      owner's slice of the owner's own grad buffer ("07 · 显存模型", section
 *      2.1 item 1) - for HSDP into the owner's slice in every replica group,
 *      all of which hold the all-reduced slice; the rest of each grad buffer
 *      is left as it was;
 *   2. norm = sqrt(sum of squares of every reduced element, each counted
 *      once) to fp64 accuracy
 *      (each thread's squares summed as a pair of floats - Dot2 of Ogita,
 *      Rump and Oishi 2005 - one fp64 partial per work tile, the partials
 *      added in an order fixed by the plan), and coefficient = min(1,
 *      max_norm / (norm + 1e-6)) rounded to fp32 (the pages are silent on
 *      clipping; this is clip_grad_norm_'s rule);
 *   3. AdamW on coefficient * gradient (one fp32 multiply), bf16 cast and
 *      all-gather, as in fsp_sharded_step.
 *   max_norm: finite, > 0.  norm_out: device, 2 floats, 16-byte aligned;
 *   receives {norm, coefficient}.  Four kernels on `cuda_stream`; the plan
 *   owns a per-device array of partial sums (8 bytes per work tile,
 *   allocated on first use), so clipped steps on one plan must be ordered on
 *   the device. */
fsp_status fsp_sharded_step_clipped(const fsp_plan* plan, void* const* grad_bufs, int32_t grad_dtype,
                                    float* master, float* exp_avg, float* exp_avg_sq,
                                    void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                                    float max_norm, float* norm_out, void* cuda_stream);

/* fsp_sharded_step that also writes every element's averaged gradient into
 * its owner's slice of the owner's own grad buffer - the Megatron distributed
 * optimizer's reduce-scatter, whose result lands in the rank's 1/DP slice of
 * its full grad buffer ("07 · 显存模型", section 2.1 item 1) - in the same
 * pass: 4 more bytes per element (76 B for N_d = 8 fp32 instead of 72).  The
 * rest of each grad buffer is left as it was.  FSDP2 and DistOpt plans with
 * fp32 grads (others: FSP_EUNSUPPORTED); otherwise as fsp_sharded_step
 * (param_bufs NULL: no all-gather). */
fsp_status fsp_sharded_step_writeback(const fsp_plan* plan, void* const* grad_bufs, int32_t grad_dtype,
                                      float* master, float* exp_avg, float* exp_avg_sq, void* const* param_bufs,
                                      const fsp_adamw_hparams* hp, int64_t step, void* cuda_stream);

/* fsp_sharded_step whose all-gather writes the fp32 master itself: FSDP2
 * with a MixedPrecisionPolicy that keeps parameters in fp32 ("Parallelism
 * strategies: which state to shard", section 二.5: the policy chooses the
 * dtype the gathered parameters compute in).  param_bufs: n_d device pointers
 * to fp32 buffers of full_len_padded elements (owned elements written with the
 * new master exactly, padding untouched); 4 bytes per element and rank instead
 * of 2.  Everything else as fsp_sharded_step (param_bufs may not be NULL). */
fsp_status fsp_sharded_step_fp32_gather(const fsp_plan* plan, const void* const* grad_bufs, int32_t grad_dtype,
                                        float* master, float* exp_avg, float* exp_avg_sq, void* const* param_bufs,
                                        const fsp_adamw_hparams* hp, int64_t step, void* cuda_stream);

/* FSDP2 unshard of the plan's parameters (the all-gather before forward and
 * before backward in ZeRO-3 / FSDP2, with a bf16 MixedPrecisionPolicy): every
 * rank's fp32 shard - its owned slots of `master` - is cast to bf16 (round to
 * nearest even) and gathered into the full buffer of every rank of its group
 * (all N_d ranks; HSDP: the N_s ranks of each replica group, from that group's
 * state copy).  "Parallelism strategies: which state to shard", section 二.5
 * (copy-in, one all-gather, copy-out); "FSDP2 Qwen3 Decoder Layer
 * Walkthrough", section "Step 0".  master: device, state layout,
 * state_len_total fp32; param_bufs: host array of n_d device pointers,
 * full_len_padded bf16 each (padding untouched).  Asynchronous on
 * `cuda_stream`; one kernel reading 4 B and writing 2 N_s B per element. */
fsp_status fsp_unshard(const fsp_plan* plan, const float* master, void* const* param_bufs, void* cuda_stream);

/* FSDP2 shard, the inverse of the unshard: every owned element of `full` (the
 * unsharded fp32 parameters in the plan's full index, full_len_padded
 * elements; padding ignored) is copied to its slot of `master` - of every
 * replica group's copy for HSDP - as fully_shard splits each parameter into
 * per-rank shards ("Parallelism strategies: which state to shard", section
 * 二.5).  exp_avg / exp_avg_sq, when not NULL, are zeroed (whole buffers): the
 * state of a fresh optimizer.  Use it to start training from full
 * parameters or to load a checkpoint.  Shard padding slots of master are
 * left as they were.  Asynchronous on `cuda_stream`. */
fsp_status fsp_shard(const fsp_plan* plan, const float* full, float* master, float* exp_avg, float* exp_avg_sq,
                     void* cuda_stream);

/* fsp_unshard into fp32 param buffers (full_len_padded fp32 each): the owned
 * master values copied to every rank of the group, no cast. */
fsp_status fsp_unshard_fp32(const fsp_plan* plan, const float* master, void* const* param_bufs, void* cuda_stream);

/* As fsp_sharded_step, and also stores the averaged shard gradient of every
 * owned element into reduced_grad (device, fp32, state layout,
 * state_len_total elements; padding slots untouched).  For testing: it adds
 * a 4-byte store per element. */
fsp_status fsp_sharded_step_debug(const fsp_plan* plan, const void* const* grad_bufs, int32_t grad_dtype,
                                  float* master, float* exp_avg, float* exp_avg_sq,
                                  void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                                  float* reduced_grad, void* cuda_stream);

/* Device workspace, in bytes, that fsp_sharded_step_host needs for this plan,
 * gradient dtype and chunk size (chunk_elems >= 0; 0 selects 2^24). */
fsp_status fsp_host_step_workspace_bytes(const fsp_plan* plan, int32_t grad_dtype, int64_t chunk_elems,
                                         size_t* bytes);

/* The fused step with the N_d gradient buffers and the N_d bf16 param buffers
 * in HOST memory (pinned memory for full speed; pageable works, slower) and
 * master / exp_avg / exp_avg_sq on the device, as a pipeline over chunks of
 * about chunk_elems elements: host-to-device copies of chunk k+1's gradient
 * slices, the step kernel on chunk k and device-to-host copies of chunk k-1's
 * bf16 result to every rank's host buffer overlap, on library-owned copy
 * streams (four per direction, created once per device, kept until exit) and
 * `cuda_stream`.
 *   host_grads[r], host_params[r]: full_len_padded elements each; only the
 *               P owned elements are copied (padding is left alone).
 *   workspace:  device, 256-byte aligned, at least
 *               fsp_host_step_workspace_bytes(...) bytes; two staging slots.
 * Asynchronous: returns once everything is enqueued; `cuda_stream` completes
 * after the last copy back, and the host buffers and the workspace must stay
 * valid and untouched until then.  Same results as fsp_sharded_step. */
fsp_status fsp_sharded_step_host(const fsp_plan* plan, const void* const* host_grads, int32_t grad_dtype,
                                 float* master, float* exp_avg, float* exp_avg_sq, void* const* host_params,
                                 const fsp_adamw_hparams* hp, int64_t step, void* workspace,
                                 size_t workspace_bytes, int64_t chunk_elems, void* cuda_stream);

/* The per-parameter tensors of a per-parameter plan, registered once on the
 * current device (the library uploads a table of their addresses; steps read
 * and write the tensors through it until it is destroyed).
 *   grad_ptrs:  host array of n_d * n_params device pointers; entry
 *               q * n_params + i is rank q's gradient of parameter i
 *               (numel_i elements of grad_dtype, the unsharded gradient), only
 *               read by the step.
 *   param_ptrs: host array of n_d * n_params device pointers to tensors of
 *               numel_i elements of param_dtype (rank q's unsharded parameter
 *               i), written by the step's all-gather and by
 *               fsp_unshard_params; NULL for a table that only reduces (steps
 *               then leave the parameters sharded, as fsp_sharded_step with
 *               param_bufs = NULL).
 *   param_dtype: FSP_DTYPE_BF16 (the cast master, as fsp_sharded_step) or
 *               FSP_DTYPE_F32 (the master itself, as
 *               fsp_sharded_step_fp32_gather).
 * Every pointer must be 16-byte aligned and lie in a live allocation holding
 * its tensor (NULL only for a parameter with 0 elements); no two tensors may
 * overlap.  The plan must come from fsp_plan_layout_params and outlive the
 * table.  Synchronous (allocates and uploads); free with
 * fsp_param_table_destroy. */
typedef struct fsp_param_table fsp_param_table;
fsp_status fsp_param_table_create(const fsp_plan* plan, const void* const* grad_ptrs, int32_t grad_dtype,
                                  void* const* param_ptrs, int32_t param_dtype, fsp_param_table** out);

/* Frees the table (its device memory); NULL is a no-op.  Must not race with a
 * call or an in-flight step that uses it. */
void fsp_param_table_destroy(fsp_param_table* table);

/* fsp_sharded_step on the tensors of `table` (a table of this plan, created on
 * the current device): the reduce-scatter reads every rank's per-parameter
 * gradient tensors in place and the all-gather writes every rank's
 * per-parameter bf16 tensors (none when the table has no param tensors).
 * master / exp_avg / exp_avg_sq and every other rule as fsp_sharded_step;
 * the results are those of fsp_sharded_step on full-size buffers holding the
 * same values at the plan's full indices (the same kernels: the rank bases of
 * each tile come from the table). */
fsp_status fsp_sharded_step_params(const fsp_plan* plan, const fsp_param_table* table, float* master,
                                   float* exp_avg, float* exp_avg_sq, const fsp_adamw_hparams* hp, int64_t step,
                                   void* cuda_stream);

/* fsp_sharded_step_params with the update index in device memory, as
 * fsp_sharded_step_device_t (for a step captured once in a CUDA graph and
 * replayed: t = *step_dev, then *step_dev += 1 when `advance` is non-zero). */
fsp_status fsp_sharded_step_params_device_t(const fsp_plan* plan, const fsp_param_table* table, float* master,
                                            float* exp_avg, float* exp_avg_sq, const fsp_adamw_hparams* hp,
                                            int64_t* step_dev, int32_t advance, void* cuda_stream);

/* fsp_sharded_step_writeback on the tensors of `table` (an FSDP2
 * per-parameter plan, fp32 gradients; others: FSP_EUNSUPPORTED): every
 * element's averaged gradient also lands in its owner's slice of the owner's
 * gradient tensor, in the same pass. */
fsp_status fsp_sharded_step_writeback_params(const fsp_plan* plan, const fsp_param_table* table, float* master,
                                             float* exp_avg, float* exp_avg_sq, const fsp_adamw_hparams* hp,
                                             int64_t step, void* cuda_stream);

/* fsp_sharded_step_clipped on the tensors of `table` (an FSDP2 or HSDP
 * per-parameter plan, fp32 gradients; bf16: FSP_EUNSUPPORTED): every
 * element's averaged gradient is written back into its owner's slice of the
 * owner's gradient tensor (HSDP: in every replica group), then the norm, the
 * coefficient and the clipped update as there.  norm_out: device, 2 floats,
 * 16-byte aligned. */
fsp_status fsp_sharded_step_clipped_params(const fsp_plan* plan, const fsp_param_table* table, float* master,
                                           float* exp_avg, float* exp_avg_sq, const fsp_adamw_hparams* hp,
                                           int64_t step, float max_norm, float* norm_out, void* cuda_stream);

/* fsp_unshard into the per-parameter tensors of `table`: the bf16 cast of the
 * owned master values (an fp32 table: the values themselves) into every rank
 * of the group.  A table created without param tensors: FSP_EINVAL; a table
 * of another plan or device: FSP_EINVAL. */
fsp_status fsp_unshard_params(const fsp_plan* plan, const fsp_param_table* table, const float* master,
                              void* cuda_stream);

/* fsp_sharded_step for callers that cannot allocate device memory (a
 * framework's allocator owns the device, a fixed memory pool must not grow,
 * or the call sits on a path that must never reach cudaMalloc).  The pages
 * have no counterpart: this is a property of the library, not of the step.
 *   Same arguments, results and checks as fsp_sharded_step (param_bufs NULL:
 *   the ZeRO-3 step, no all-gather); it allocates no device memory (the
 *   kernel's tile counter is a library variable too, zeroed on `cuda_stream`).
 *   The plan's work-tile list lives in a fixed array of device memory declared
 *   by the library (262144 tiles, 8 MiB, present on every device that loads
 *   the library until the process exits).  A call copies the list there, on
 *   `cuda_stream`, only when the array does not already hold this plan's list
 *   on this device (the first call with the plan, or the first after a call
 *   with another plan); that copy is from pageable host memory, so such a call
 *   may wait on the host for earlier work on the stream.  Plans with more
 *   tiles (roughly more than 1.07e9 elements) return FSP_EUNSUPPORTED.
 *   The first call on a device looks up that array's device address (with the
 *   device current) and keeps it for later calls.
 *   Every call shares the one array, which keeps the last list copied into it:
 *   calls that can overlap on the GPU (other streams, other threads) race and
 *   must be ordered by the caller.  Nothing in the array needs clearing
 *   between calls: the kernel reads only the tiles of the plan it runs. */
fsp_status fsp_sharded_step_noalloc(const fsp_plan* plan, const void* const* grad_bufs, int32_t grad_dtype,
                                    float* master, float* exp_avg, float* exp_avg_sq,
                                    void* const* param_bufs, const fsp_adamw_hparams* hp, int64_t step,
                                    void* cuda_stream);

/* Reads and clears the device error word of the current device (synchronous:
 * waits for the device).  The step kernel's waits on its own copy pipeline
 * are bounded (about 2 s); one that runs out sets a bit here (1: the storer
 * waited for the consumers' results, 2: the producer waited for a free
 * stage; 4: the self-test below; 8: a device-resident update index below 1),
 * lets its copies land and ends the kernel,
 * leaving that step's results incomplete.  0 means every step since the last
 * read completed normally. */
fsp_status fsp_device_error(uint32_t* bits);

/* Self-test of the step kernel's bounded waits: runs one thread that waits
 * on an mbarrier nothing ever arrives at, with the step kernel's wait routine
 * and a limit of limit_ms (1..2000) milliseconds, synchronises the device and
 * returns the device error word in *bits (cleared afterwards).  A working
 * bound gives bit 4 after about limit_ms; the device stays usable. */
fsp_status fsp_selftest_bounded_wait(uint32_t limit_ms, uint32_t* bits);

/* Message for a status code (static storage). */
const char* fsp_status_string(fsp_status status);

/* Description of the last error returned on the calling thread ("" if none). */
const char* fsp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FSP_H */
