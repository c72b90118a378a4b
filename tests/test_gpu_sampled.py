"""Sampled drafting with q-ratio verification through the C ABI.

The children of every expanded node are drawn from the draft distribution by
Gumbel-top-k on Philox stream 2 (eagle3_draft_noise), and T > 0 verification is
the q-ratio test over the draws (eagle3_verify mode 2).  Every pool slot, tree
slot, accepted path and emitted token is compared with the oracle given the
same seeds, in conditioned mode (parity.py): near-ties of the draw keys, the
acceptance tests and the residual draw are counted, not failed.  A graph
replay draws its noise with the replay's round id and must equal the eager
calls made with that round id.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs
from parity import TOL, compare, gpu_round

C0 = by_name("tiny_fp32_b1")
CASES = {
    "sampled_fp32": (C0.scaled(name="samp_fp32", sampled_draft=True, temperatures=(0.0, 1.0)), 3),
    "sampled_fp32_b3": (C0.scaled(name="samp_fp32_b3", sampled_draft=True, batch=3, prefix=64,
                                  prefix_range=(30, 64), depth=4, topk=3, n_verify=10,
                                  temperatures=(1.0,)), 4),
    "sampled_bf16": (C0.scaled(name="samp_bf16", sampled_draft=True, dtype="bf16", d=256,
                               n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512, vocab=2048,
                               prefix=100, batch=2, depth=4, topk=4, n_verify=12, lm_std=0.08,
                               temperatures=(0.0, 1.0)), 5),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_sampled_draft_parity(cuda, lib_built, name):
    from eagle_draft_tree_02_b300.runner import Engine
    cfg, seed = CASES[name]
    inp = make_inputs(cfg, seed=seed)
    eng = Engine(inp)
    eng.prefill()
    eng.draft_noise(21, 5)
    temps = cfg.temperatures
    gpu = gpu_round(eng, temps, seed=13, round_id=6)
    rep = compare(cfg, inp, gpu, temps, seed=13, round_id=6, samp=(21, 5))
    tol = TOL[cfg.dtype]
    assert not rep.failures, rep
    assert rep.max_err["logq"] <= tol["logit"], rep
    assert rep.max_err["score/depth"] <= tol["logit"], rep
    # siblings: scores non-increasing in draw order, kept ones the first draws
    for b in range(cfg.batch):
        par, sc, tok = gpu.pool["parent"][b], gpu.pool["score"][b], gpu.pool["tok"][b]
        kept = set(int(i) for i in gpu.tree["pool_index"][b, 1:] if i >= 0)
        for p in set(int(x) for x in par[tok >= 0]):
            sib = [i for i in range(len(par)) if tok[i] >= 0 and par[i] == p]
            assert all(sc[i] >= sc[j] for i, j in zip(sib, sib[1:]))
            inn = [i in kept for i in sib]
            assert inn == sorted(inn, reverse=True)
    print(name, rep)
    eng.close()


@pytest.mark.gpu
def test_sampled_draft_graph_replay_uses_the_replay_round(cuda, lib_built):
    import torch
    from eagle_draft_tree_02_b300.runner import Engine
    cfg, seed = CASES["sampled_bf16"]
    inp = make_inputs(cfg, seed=seed)
    eng = Engine(inp)
    eng.prefill()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eager = {}
        for rid in (2, 7):
            eng.draft_noise(31, rid)
            eng.draft_round(with_pool=False)
            a, p, o = eng.verify(1.0, seed=9, round_id=rid, with_stats=False)
            eager[rid] = (eng.tree.tokens.clone(), a.clone(), o.clone())
        eng.capture(temperature=1.0, seed=9)
        for rid in (7, 2):
            eng.replay(rid)
            torch.cuda.current_stream().synchronize()
            eng.check()
            tt, a, o = eager[rid]
            assert torch.equal(eng.tree.tokens, tt)
            assert torch.equal(eng.accept_len, a)
            assert torch.equal(eng.out_tokens, o)
        assert not torch.equal(eager[2][0], eager[7][0])  # the draws depend on the round
    eng.close()
