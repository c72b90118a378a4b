"""Per-request caps and the cost-aware rules through the C ABI (eagle3_set_control).

One batch mixes requests of different depth, branch and verify caps, and the
three rules (another draft layer, how many nodes to verify, how many branches
a node expands) run on the device from a cost table; every pool slot, tree
slot, accepted path and emitted token is compared with the oracle given the
same control, in conditioned mode (parity.py).  A batch whose requests all stop
after the root pass skips the heavy kernels of the later passes and must give
the same result as the oracle.  Graph replay keeps the captured control.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs
from oracle import round as R
from parity import TOL, compare, gpu_round

C0 = by_name("tiny_fp32_b1")
SMALL_BF16 = C0.scaled(name="ctl_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2,
                       head_dim=64, ffn=512, vocab=2048, prefix=100, batch=3, depth=4, topk=4,
                       n_verify=12, lm_std=0.08, temperatures=(0.0, 1.0))
B3 = C0.scaled(name="ctl_fp32", batch=3, prefix=64, prefix_range=(30, 64), depth=5, topk=4,
               n_verify=16, temperatures=(0.0, 1.0))

CASES = {
    "caps_fp32": (B3, dict(depth_cap=[5, 2, 1], topk_cap=[4, 2, 3], verify_cap=[16, 5, 2])),
    "caps_bf16": (SMALL_BF16, dict(depth_cap=[1, 4, 3], topk_cap=[1, 4, 2], verify_cap=[12, 7, 3])),
    "rules_fp32": (B3, dict(tau_depth=0.0005, depth_growth=1.2, pass_us=[120.0, 100.0, 100.0, 100.0, 100.0],
                            tau_verify=0.0005, verify_us=[10.0 * m for m in range(17)],
                            light_batch=2, k_light=4, k_heavy=3)),
    "rules_bf16": (SMALL_BF16, dict(tau_depth=0.00025, depth_growth=1.2, pass_us=[100.0] * 4,
                                    tau_verify=0.0005, verify_us=[10.0 * m for m in range(13)],
                                    light_batch=4, k_light=3, k_heavy=2)),
    "all_stop_after_root": (SMALL_BF16, dict(depth_cap=[1, 1, 1])),
}


def _oracle_control(kw):
    k = {n: v for n, v in kw.items()}
    return R.Control(**k)


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_control_parity(cuda, lib_built, name):
    from eagle_draft_tree_02_b300.runner import Engine
    cfg, kw = CASES[name]
    inp = make_inputs(cfg, seed=17)
    eng = Engine(inp)
    eng.prefill()
    eng.set_control(**kw)
    temps = cfg.temperatures
    gpu = gpu_round(eng, temps, seed=13, round_id=4)
    rep = compare(cfg, inp, gpu, temps, seed=13, round_id=4, ctl=_oracle_control(kw))
    tol = TOL[cfg.dtype]
    assert not rep.failures, rep
    assert rep.max_err.get("logq", 0.0) <= tol["logit"], rep
    assert rep.max_err.get("score/depth", 0.0) <= tol["logit"], rep
    assert rep.max_err["z_max"] <= tol["logit"], rep
    # the caps hold on the device
    kept = (gpu.tree["tokens"][:, 1:] >= 0).sum(axis=1)
    if "verify_cap" in kw:
        assert (kept <= np.asarray(kw["verify_cap"])).all(), kept
    if "depth_cap" in kw:
        made = gpu.pool["tok"] >= 0
        depth = np.where(made, gpu.pool["depth"], 0).max(axis=1)
        assert (depth <= np.asarray(kw["depth_cap"])).all(), depth
    print(name, rep, "kept", kept)
    eng.close()


@pytest.mark.gpu
def test_control_survives_graph_replay(cuda, lib_built):
    import torch
    from eagle_draft_tree_02_b300.runner import Engine
    cfg, kw = CASES["caps_bf16"]
    inp = make_inputs(cfg, seed=19)
    eng = Engine(inp)
    eng.prefill()
    eng.set_control(**kw)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eng.draft_round(with_pool=False)
        a, p, o = eng.verify(0.0, seed=5, round_id=2, with_stats=False)
        want = (eng.tree.tokens.clone(), a.clone(), o.clone())
        eng.capture(temperature=0.0, seed=5)
        eng.replay(2)
        torch.cuda.current_stream().synchronize()
        eng.check()
        assert torch.equal(eng.tree.tokens, want[0])
        assert torch.equal(eng.accept_len, want[1])
        assert torch.equal(eng.out_tokens, want[2])
    eng.set_control()
    eng.close()


@pytest.mark.gpu
def test_warmup_table_feeds_the_depth_rule(cuda, lib_built):
    """The warm-up measures the passes on the device; its table, looked up for the
    engine's shape, gives the depth rule positive pass costs, and a threshold far
    above any frontier mass stops every request after the root pass."""
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine
    cfg = SMALL_BF16
    inp = make_inputs(cfg, seed=23)
    eng = Engine(inp)
    eng.prefill()
    batch, prefix, tokens, draft_us, verify_us = eng.warmup_latency_table(reps=2)
    # the root pass and verification cost time; a later pass may cost nothing
    # measurable on a shape this small (every kernel is launch-bound)
    assert draft_us[0, 0, 0] > 0 and (draft_us >= 0).all() and (verify_us > 0).all()
    s, pu, vu = E.eagle3_latency_costs(batch, prefix, tokens, draft_us, verify_us, eng.B,
                                       int(eng.max_prefix), cfg.depth, cfg.topk, cfg.n_verify)
    assert s == E.OK and vu[0] == 0.0
    assert pu[0] == pytest.approx(float(draft_us[0, 0, 0]))
    assert vu[cfg.n_verify] == pytest.approx(float(verify_us[0, 0, tokens.index(cfg.n_verify)]))
    eng.set_control(tau_depth=1e6, pass_us=[max(x, 1.0) for x in pu])
    gpu = gpu_round(eng, (0.0,), seed=1, round_id=1)
    made = gpu.pool["tok"] >= 0
    assert (np.where(made, gpu.pool["depth"], 0).max(axis=1) == 1).all()
    eng.set_control()
    eng.close()
