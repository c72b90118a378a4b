"""GPU parity at the workloads' full sizes (the launch configuration bench.py times).

* 8B-shaped tree, batch 1, prefix 2048: the oracle recomputes everything
  (prefix K/V included) and checks the whole round, greedy and T=1.
* 8B-shaped serving batch 64, chain of 3, paged cache with 64-token pages:
  sampled requests, each recomputed by the oracle from its own features.
* 70B-shaped tree, batch 4, prefix 8192: sampled K/V rows of the cache are
  checked against the oracle, then the oracle's round for a sampled request
  runs on the GPU's cache (conditioned on the shared prefix K/V).
* two-stage head tree, batch 16, prefix 4096, vocabulary 151936: as the 70B
  case, for two sampled requests; the GPU's candidate sets must be valid
  top-64 sets of the oracle's low-rank scores.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import CONFIGS
from eagle_draft_tree_02_b300.synth import make_inputs
from oracle import round as R
from parity import TOL, compare, gpu_round


def _run(cfg, requests=None, conditioned_kv=False, kv_rows_checked=0):
    import torch
    from eagle_draft_tree_02_b300.runner import Engine
    inp = make_inputs(cfg)
    eng = Engine(inp)
    eng.prefill()
    torch.cuda.synchronize()
    eng.check()
    temps = cfg.temperatures
    gpu = gpu_round(eng, temps, seed=0, round_id=7)
    prefix_kv = None
    if conditioned_kv:
        w = R.weights_f32(inp)
        f = inp.feats_f32()
        rng = np.random.default_rng(0)
        cache = {}
        for b in requests:
            lo, hi = int(inp.cu_rows[b]), int(inp.cu_rows[b + 1])
            P = hi - lo
            gk = eng.k_cache[b, :P].float().cpu().numpy().astype(np.float64)
            gv = eng.v_cache[b, :P].float().cpu().numpy().astype(np.float64)
            rows = np.sort(rng.choice(P, size=min(P, kv_rows_checked), replace=False))
            # sampled rows at their true positions
            from oracle import layers as L
            g = L.fused_feature(w, cfg, f[lo:hi][rows])
            x = L.decoder_input(w, cfg, inp.tokens[lo:hi][rows], g)
            _, k, v = L.qkv(w, cfg, x, rows)
            tol = TOL[cfg.dtype]["logit"]
            assert np.abs(gk[rows] - k).max() < tol and np.abs(gv[rows] - v).max() < tol
            cache[b] = (gk, gv)
        prefix_kv = lambda b: cache[b]
    rep = compare(cfg, inp, gpu, temps, seed=0, round_id=7, prefix_kv=prefix_kv, requests=requests)
    tol = TOL[cfg.dtype]
    print(cfg.name, rep)
    assert not rep.failures, rep
    assert rep.max_err["logq"] <= tol["logit"], rep
    assert rep.max_err["score/depth"] <= tol["logit"], rep
    assert rep.max_err["z_max"] <= tol["logit"] and rep.max_err["lse"] <= tol["logit"], rep
    eng.close()
    return rep


@pytest.mark.gpu
def test_full_8b_batch1_tree(cuda, lib_built):
    _run(CONFIGS[1])


@pytest.mark.gpu
def test_full_8b_batch64_chain_paged(cuda, lib_built):
    _run(CONFIGS[2], requests=[0, 17, 63])


@pytest.mark.gpu
def test_full_70b_batch4_tree(cuda, lib_built):
    _run(CONFIGS[3], requests=[2], conditioned_kv=True, kv_rows_checked=24)


@pytest.mark.gpu
def test_full_two_stage_b16_tree(cuda, lib_built):
    _run(CONFIGS[4], requests=[0, 11], conditioned_kv=True, kv_rows_checked=24)
