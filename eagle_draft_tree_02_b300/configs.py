"""The five workloads of one EAGLE-3 draft-and-verify round, as plain shapes.

Each workload is named by what it is.  The model shapes follow the draft
decoders the pages talk about: a Llama-3.1-8B-shaped and a Llama-3.3-70B-shaped
one-layer drafter ("EAGLE-3 精读", §4 结果与消融), the serving set-up with a
length-3 chain at batch 64 (same section, SGLang/H100 paragraph), and the
two-stage "Efficient LM Head" of the EAGLE-4 blog (section 关于 Efficient LM
Head).  No arithmetic of the method lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class RoundConfig:
    name: str
    dtype: str              # "fp32" or "bf16": storage type of weights/features/KV
    batch: int              # requests per round (B)
    d: int                  # model width
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int                # SwiGLU inner width (F)
    vocab: int              # V
    prefix: int             # rows in the cache after the round's new row(s) (root = prefix-1)
    depth: int              # D: tree depth (= sequential decoder passes per round)
    topk: int               # k: children per expanded node, frontier width
    n_verify: int           # M: nodes kept for verification
    lm_std: float = 0.02    # std of the draft LM head
    eps_target: float = 0.3 # target head = W_lm + eps_target * G
    rope_theta: float = 5e5
    rms_eps: float = 1e-5
    page_size: int = 0      # 0 = contiguous per-request cache, else paged
    prefix_range: tuple | None = None  # (lo, hi): per-request prefix ~ U{lo..hi}
    lr_rank: int = 0        # two-stage head rank r (0 = single-stage head)
    lr_cand: int = 0        # two-stage head candidate count
    temperatures: tuple = (0.0,)  # verify modes: 0.0 = greedy, >0 = sampling at T
    fc_norm: bool = False   # drafter variant: RMSNorm (gain g_fc) on the fused feature
    post_norm: bool = False # drafter variant: norms after the residual adds
    gain_std: float = 0.0   # RMSNorm gains ~ 1 + N(0, gain_std^2) (0: all gains 1)
    sampled_draft: bool = False  # children drawn from q; T > 0 verification by the q-ratio test

    @property
    def pool_size(self) -> int:
        """Nodes created per request: k at depth 1, k*k at each deeper level."""
        return self.topk + (self.depth - 1) * self.topk * self.topk

    @property
    def qkv_dim(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def scaled(self, **kw) -> "RoundConfig":
        return replace(self, **kw)


CONFIGS = [
    RoundConfig(
        name="tiny_fp32_b1", dtype="fp32", batch=1, d=256, n_q_heads=4, n_kv_heads=4,
        head_dim=64, ffn=688, vocab=1024, prefix=64, depth=5, topk=4, n_verify=16,
        lm_std=0.08, temperatures=(0.0, 1.0)),
    RoundConfig(
        name="llama31_8b_b1_tree", dtype="bf16", batch=1, d=4096, n_q_heads=32, n_kv_heads=8,
        head_dim=128, ffn=14336, vocab=128256, prefix=2048, depth=6, topk=10, n_verify=60,
        temperatures=(0.0, 1.0)),
    RoundConfig(
        name="llama31_8b_b64_chain3_paged", dtype="bf16", batch=64, d=4096, n_q_heads=32,
        n_kv_heads=8, head_dim=128, ffn=14336, vocab=128256, prefix=4096, depth=3, topk=1,
        n_verify=3, page_size=64, prefix_range=(512, 4096), temperatures=(0.0,)),
    RoundConfig(
        name="llama33_70b_b4_tree", dtype="bf16", batch=4, d=8192, n_q_heads=64, n_kv_heads=8,
        head_dim=128, ffn=28672, vocab=128256, prefix=8192, depth=8, topk=8, n_verify=64,
        temperatures=(1.0,)),
    RoundConfig(
        name="two_stage_head_b16_tree", dtype="bf16", batch=16, d=5120, n_q_heads=40,
        n_kv_heads=8, head_dim=128, ffn=17408, vocab=151936, prefix=4096, depth=6, topk=8,
        n_verify=48, lr_rank=256, lr_cand=64, temperatures=(0.0, 1.0)),
]


def by_name(name: str) -> RoundConfig:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


# Small cases for the oracle's own CPU tests: same structure, tiny sizes.
TINY_V8 = RoundConfig(
    name="chi2_v8", dtype="fp32", batch=1, d=16, n_q_heads=2, n_kv_heads=1, head_dim=8,
    ffn=24, vocab=8, prefix=6, depth=3, topk=2, n_verify=6, lm_std=0.3,
    temperatures=(1.0,))
