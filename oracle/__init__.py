"""Oracle for the sharded mixed-precision step - TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU statement of what the step computes,
written from the pages, for checking the CUDA path.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may import it.  The product (``fsdp_sharded_mixed_pass_gb300``)
never imports it, and it imports nothing from the product: the two share no
code.  Its only shared dependency is the seeded input generator
(``synth_inputs``), which holds none of the step's arithmetic.

Modules
-------
``oracle.plan``    layout rules: FSDP2 per-parameter Shard(0) with padding,
                   Megatron DistOpt flat shards with lcm(N_d, 128) padding, and
                   the rank-major state placement.
``oracle.step``    the step itself, one function per stage: rank-ordered
                   reduce-scatter averaged by N_d, AdamW on the fp32 shard
                   (computed in fp64, stored in fp32), bf16 round-to-nearest-even
                   cast, all-gather into every rank's buffer; plus the unsharded
                   all-reduce definition it must equal.
``oracle.ledger``  the pages' per-parameter byte ledger, per-rank collective
                   volumes and the dense-model parameter-count formula.

Pins (``tests/test_oracle_*.py``, ``-m "not gpu"``) tie every function to
something other than itself: the pages' worked numbers (``tests/golden/``),
hand-worked AdamW cases, brute force on tiny inputs, and library routines for
special cases.  The AdamW update rule is a reading, not a page's: the pages
name "Adam m/v" as state but never print the rule.  The oracle's statement of
the reading (PyTorch's decoupled, bias-corrected AdamW) is pinned by
hand-worked closed forms and against torch.optim.AdamW run in fp64; which rule
the pages' systems use is beyond what the pages fix.
"""
from . import plan, step, ledger  # noqa: F401
