"""Byte ledger and collective volumes of the pages (test infrastructure only).

* Resident bytes per parameter ("07 · 显存模型", section 2.1 "每参数字节", and
  "Parallelism strategies: which state to shard", section 九 Q1): bf16 param
  (2 B), main grad (4 B fp32, or 2 B when grad_reduce_in_fp32 is off), fp32
  master + Adam m + Adam v (12 B).  DDP keeps all of it; the distributed
  optimizer (ZeRO-1) shards only the 12 B; ZeRO-2 also shards the grad; ZeRO-3 /
  FSDP shards everything.
* Per-rank send volume of a collective on n ranks with payload S bytes
  ("Parallelism strategies: which state to shard", section 一.1 and the volume
  formulas of its ledger appendix): all-reduce 2(n-1)/n S; all-gather,
  reduce-scatter and all-to-all (n-1)/n S; send/recv S; nothing when n <= 1.
* Dense GQA/SwiGLU/RMSNorm parameter count with a tied embedding ("07 · 显存模型",
  section 2.2 "参数量估算"):
  L [2 h q (1 + g/a) + 3 h ffn + 2 h] + V h, plus one final norm of h.
"""
from __future__ import annotations

from fractions import Fraction

PARAM_BYTES = 2          # bf16 param
MASTER_ADAM_BYTES = 12   # fp32 master + m + v


def bytes_per_param(scheme: str, n_d: int, grad_bytes: int = 4) -> Fraction:
    """Resident bytes per parameter on one rank, as an exact fraction."""
    n = Fraction(n_d)
    p, g, k = PARAM_BYTES, grad_bytes, MASTER_ADAM_BYTES
    if scheme == "ddp":
        return Fraction(p + g + k)
    if scheme in ("distopt", "zero1"):
        return p + g + k / n
    if scheme == "zero2":
        return p + (g + k) / n
    if scheme in ("fsdp", "zero3"):
        return (p + g + k) / n
    raise ValueError(scheme)


def hsdp_bytes_per_param(n_shard: int, grad_bytes: int = 4) -> Fraction:
    """HSDP: ZeRO-3 inside an N_s-rank shard group, plain replication across
    groups, so a rank keeps (2 + g + 12) / N_s bytes per parameter
    ("Parallelism strategies: which state to shard", section 二.6)."""
    return Fraction(PARAM_BYTES + grad_bytes + MASTER_ADAM_BYTES, n_shard)


def hsdp_step_sent(n_rep: int, n_shard: int, grad_payload: float, param_payload: float) -> dict:
    """Bytes one rank sends for the optimizer-side collectives of an HSDP step:
    reduce-scatter and all-gather inside the shard group, all-reduce of its
    1/N_s gradient shard across the N_r replica groups (the pages' ledger
    listing, the HSDP branch of its DP section)."""
    return {
        "reduce_scatter": coll_bytes("reduce_scatter", n_shard, grad_payload),
        "all_gather": coll_bytes("all_gather", n_shard, param_payload),
        "cross_group_all_reduce": coll_bytes("all_reduce", n_rep, Fraction(grad_payload) / n_shard),
    }


def resident_bytes(scheme: str, n_params: int, n_d: int, grad_bytes: int = 4) -> Fraction:
    return bytes_per_param(scheme, n_d, grad_bytes) * n_params


def resident_breakdown_distopt(p_shard: int, dp: int, grad_bytes: int = 4) -> dict:
    """(param, grad, optimizer) bytes of a DistOpt rank holding ``p_shard`` params."""
    return {
        "param": Fraction(PARAM_BYTES * p_shard),
        "grad": Fraction(grad_bytes * p_shard),
        "optimizer": Fraction(MASTER_ADAM_BYTES * p_shard, dp),
    }


# Ring collectives move the payload in phases.  In one phase the payload is
# cut into n equal pieces and every rank sends n - 1 of them, so a rank sends
# (n - 1)/n of the payload per phase.  Reduce-scatter, all-gather and
# all-to-all take one phase; all-reduce is a reduce-scatter and then an
# all-gather ("Parallelism strategies: which state to shard", section 一.1),
# so it takes two.
RING_PHASES = {"reduce_scatter": 1, "all_gather": 1, "all_to_all": 1, "all_reduce": 2}
# A point-to-point transfer sends the whole payload once, whatever n is.
POINT_TO_POINT = ("send_recv",)


def coll_bytes(kind: str, n: int, size: float) -> Fraction:
    """Bytes one rank sends in collective ``kind`` over ``n`` ranks with
    payload ``size`` bytes (a group of one rank sends nothing)."""
    payload = Fraction(size)
    if kind in POINT_TO_POINT:
        return payload
    if kind not in RING_PHASES:
        raise ValueError(f"unknown collective {kind!r}")
    ranks = max(n, 1)
    return RING_PHASES[kind] * Fraction(ranks - 1, ranks) * payload


def dense_param_count(h: int, layers: int, heads: int, kv_heads: int, head_dim: int, ffn: int,
                      vocab: int, final_norm: bool = True, qk_norm: bool = False) -> int:
    """Parameter count of a dense GQA / SwiGLU / RMSNorm stack with tied embedding.

    ``qk_norm`` adds Qwen3's two head-dim RMSNorm weights per layer.
    """
    q = heads * head_dim
    attn = Fraction(2 * h * q) * (1 + Fraction(kv_heads, heads))
    per_layer = attn + 3 * h * ffn + 2 * h + (2 * head_dim if qk_norm else 0)
    total = layers * per_layer + vocab * h + (h if final_norm else 0)
    assert total.denominator == 1
    return int(total)


def sharded_step_bytes(n_d: int, grad_bytes: int, n_rep: int = 1) -> int:
    """Minimum HBM bytes the fused step moves per valid element when N_d ranks
    are buffers on one device: each rank's grad read once, each of the N_r
    copies of fp32 master/m/v read and written once, one bf16 param written per
    rank."""
    return n_d * grad_bytes + 2 * MASTER_ADAM_BYTES * n_rep + n_d * PARAM_BYTES
