"""GPU parity at the workloads' full sizes (the launch configuration bench.py times).

Every request of every workload is checked.  The oracle runs each request's
round on the GPU's own prefix K/V (read back from the cache, through the
page table for the paged serving batch), after sampled rows of that cache
have been checked against the oracle's own K/V at their true positions; this
keeps the CPU work to the round itself.  Near-ties (decisions whose oracle
margin is under the tie tolerance, which the parity rule counts instead of
failing) are reported in every assertion message and bounded per workload.

* 8B-shaped tree, batch 1, prefix 2048, greedy and T=1.
* 8B-shaped serving batch 64, chain of 3, paged cache with 64-token pages.
* 70B-shaped tree, batch 4, prefix 8192, T=1.
* two-stage head tree, batch 16, prefix 4096, vocabulary 151936, greedy and
  T=1; the GPU's candidate sets must be valid top-64 sets of the oracle's
  low-rank scores.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs
from oracle import layers as L
from oracle import round as R
from parity import TOL, Report, compare_request, gpu_round

# largest near-tie count accepted per workload (all requests, all temperatures),
# not counting the two-stage head's candidate sets: the 64th and 65th best of
# 151936 low-rank scores are nearly always within the bf16 tolerance, so the
# GPU's set is adopted whenever it is a valid top-64 of the oracle's scores
# (counted apart, at most one per expanded node)
NEAR_TIE_LIMIT = {"llama31_8b_b1_tree": 4, "llama31_8b_b64_chain3_paged": 8,
                  "llama33_70b_b4_tree": 8, "two_stage_head_b16_tree": 16}


def _cache_rows(eng, b, P):
    """Request b's prefix K/V rows 0..P-1 from the GPU cache, as float64."""
    cfg = eng.cfg
    if cfg.page_size:
        ps = cfg.page_size
        pages = eng.page_table[b, :(P + ps - 1) // ps].long()
        k = eng.k_cache[pages].reshape(-1, cfg.n_kv_heads, cfg.head_dim)[:P]
        v = eng.v_cache[pages].reshape(-1, cfg.n_kv_heads, cfg.head_dim)[:P]
    else:
        k, v = eng.k_cache[b, :P], eng.v_cache[b, :P]
    return (k.float().cpu().numpy().astype(np.float64), v.float().cpu().numpy().astype(np.float64))


def _run(cfg, kv_rows_checked):
    import torch
    from eagle_draft_tree_02_b300.runner import Engine
    inp = make_inputs(cfg)
    eng = Engine(inp)
    eng.prefill()
    torch.cuda.synchronize()
    eng.check()
    temps = cfg.temperatures
    gpu = gpu_round(eng, temps, seed=0, round_id=7)
    # float64 copies of the weights, made once: the oracle's products then read them directly
    w = {k: np.asarray(v, dtype=np.float64) if k != "embed" else v
         for k, v in R.weights_f32(inp).items()}
    f = inp.feats_f32()
    rng = np.random.default_rng(0)
    tol = TOL[cfg.dtype]
    rep = Report()
    kv_err = 0.0
    for b in range(cfg.batch):
        lo, hi = int(inp.cu_rows[b]), int(inp.cu_rows[b + 1])
        P = hi - lo
        K, V = _cache_rows(eng, b, P)
        rows = np.sort(rng.choice(P, size=min(P, kv_rows_checked), replace=False))
        g = L.fused_feature(w, cfg, f[lo:hi][rows])
        x = L.decoder_input(w, cfg, inp.tokens[lo:hi][rows], g)
        _, k, v = L.qkv(w, cfg, x, rows)
        kv_err = max(kv_err, np.abs(K[rows] - k).max(), np.abs(V[rows] - v).max())
        compare_request(cfg, w, K, V, f[hi - 1], inp.tokens[hi - 1], P, gpu, b, temps, rep,
                        seed=0, round_id=7)
    cand_ties = sum(1 for t in rep.near_ties if t[0] == "candidates")
    n_ties = len(rep.near_ties) - cand_ties
    n_expanded = cfg.batch * (1 + (cfg.depth - 1) * cfg.topk)
    msg = (f"{cfg.name}: near-ties {n_ties} (limit {NEAR_TIE_LIMIT[cfg.name]}), candidate-set "
           f"near-ties {cand_ties} of {n_expanded} expanded nodes, {rep}, kv_err {kv_err:.3g}")
    print(msg)
    assert kv_err < tol["logit"], msg
    assert not rep.failures, msg
    assert rep.max_err["logq"] <= tol["logit"], msg
    assert rep.max_err["score/depth"] <= tol["logit"], msg
    assert rep.max_err["z_max"] <= tol["logit"] and rep.max_err["lse"] <= tol["logit"], msg
    assert n_ties <= NEAR_TIE_LIMIT[cfg.name], msg
    assert cand_ties <= n_expanded, msg
    eng.close()
    return rep


@pytest.mark.gpu
def test_full_8b_batch1_tree(cuda, lib_built):
    _run(by_name("llama31_8b_b1_tree"), kv_rows_checked=32)


@pytest.mark.gpu
def test_full_8b_batch64_chain_paged(cuda, lib_built):
    _run(by_name("llama31_8b_b64_chain3_paged"), kv_rows_checked=4)


@pytest.mark.gpu
def test_full_70b_batch4_tree(cuda, lib_built):
    _run(by_name("llama33_70b_b4_tree"), kv_rows_checked=16)


@pytest.mark.gpu
def test_full_two_stage_b16_tree(cuda, lib_built):
    _run(by_name("two_stage_head_b16_tree"), kv_rows_checked=8)
