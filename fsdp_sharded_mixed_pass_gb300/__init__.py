"""GB300 (sm_103a) sharded mixed-precision optimizer step.

One data-parallel ZeRO / FSDP step with N_d ranks simulated as N_d buffers on
one GPU: rank-ordered fp32 reduce-scatter averaged by N_d, AdamW on the fp32
master / m / v shard, bf16 cast and all-gather into every rank's param buffer,
fused into one streaming CUDA kernel behind the C ABI in ``include/fsp.h``.

    from fsdp_sharded_mixed_pass_gb300 import plan_layout, sharded_step
"""
from .fsp import (  # noqa: F401
    EXPORTS,
    FspError,
    ParamTable,
    Plan,
    Segment,
    device_error,
    lib,
    plan_layout,
    plan_layout_params,
    selftest_bounded_wait,
    shard,
    sharded_step,
    sharded_step_clipped,
    sharded_step_clipped_params,
    sharded_step_debug,
    sharded_step_device_t,
    sharded_step_host,
    host_step_workspace_bytes,
    sharded_step_noalloc,
    sharded_step_params,
    sharded_step_params_device_t,
    sharded_step_writeback,
    sharded_step_writeback_params,
    sharded_step_fp32_gather,
    unshard,
    unshard_params,
)
from .optim import ShardedAdamW  # noqa: F401,E402
