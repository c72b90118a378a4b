"""Algorithmic bytes and FLOPs of a round, for roofline fractions.

Counting rules: every weight matrix is read once per sequential pass that uses
it; the prefix K/V of a request is read once per pass; token-embedding rows,
features and activations are counted at their size; no logits are written (the
heads reduce them on chip).  Padding, split-K partials and re-reads are not
algorithmic work and are not counted.
"""
from __future__ import annotations

from .configs import RoundConfig


def _esz(cfg: RoundConfig) -> int:
    return 2 if cfg.dtype == "bf16" else 4


def layer_params(cfg: RoundConfig) -> int:
    d, qd, kvd = cfg.d, cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    return 2 * d * (qd + 2 * kvd) + qd * d + 3 * cfg.ffn * d


def head_bytes(cfg: RoundConfig, rows: int, weights: str = "lm") -> int:
    """One launch of a vocabulary head on `rows` rows: the weight once plus the rows."""
    e = _esz(cfg)
    if cfg.lr_rank and weights == "lm":
        return e * (cfg.vocab * cfg.lr_rank + cfg.lr_rank * cfg.d + rows * cfg.d)
    return e * (cfg.vocab * cfg.d + rows * cfg.d)


def head_flops(cfg: RoundConfig, rows: int) -> int:
    return 2 * rows * cfg.vocab * cfg.d


def round_bytes(cfg: RoundConfig, prefix_mean: float | None = None, n_new: int = 1,
                verify: bool = True) -> dict:
    """Algorithmic HBM bytes of one draft round (and its verify stand-in)."""
    e = _esz(cfg)
    B, d, k, D, M = cfg.batch, cfg.d, cfg.topk, cfg.depth, cfg.n_verify
    kvd = cfg.n_kv_heads * cfg.head_dim
    P = prefix_mean if prefix_mean is not None else cfg.prefix
    kv_read = 2 * B * P * kvd * e                      # K and V of the prefix, once per pass
    layer = layer_params(cfg) * e
    head = head_bytes(cfg, 0)
    draft = 0
    # pass 0: fusion of the new rows, then the root rows
    draft += d * 3 * d * e + B * n_new * 3 * d * e + B * n_new * d * e
    draft += layer + kv_read + B * n_new * 2 * kvd * e + head + B * d * e
    # passes 1..D-1: k frontier rows per request
    rows = B * k
    draft += (D - 1) * (layer + kv_read + rows * d * e + head + rows * 2 * kvd * e + rows * d * e)
    out = {"draft": int(draft)}
    if verify:
        rv = B * M
        out["verify"] = int(layer + kv_read + rv * d * e + head_bytes(cfg, B * (M + 1), "target")
                            + rv * 2 * kvd * e)
    out["step"] = out["draft"] + out.get("verify", 0)
    return out
