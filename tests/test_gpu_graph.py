"""CUDA-graph replay of a whole step (draft round + verify) through the C ABI.

eagle3_graph_capture records the step once; eagle3_graph_launch replays it
with a new round id.  The replay runs the same kernels on the same inputs, so
its tree, accepted lengths and emitted tokens must equal the eager calls' bit
for bit, for every round id (the sampling draws depend on it).
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs

C0 = by_name("tiny_fp32_b1")
SMALL_BF16 = C0.scaled(name="graph_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2,
                       head_dim=64, ffn=512, vocab=2048, prefix=100, batch=2, depth=4, topk=4,
                       n_verify=12, lm_std=0.08, temperatures=(0.0, 1.0))


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [C0, SMALL_BF16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("T", [0.0, 1.0])
def test_graph_replay_equals_eager(cuda, lib_built, cfg, T):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine
    inp = make_inputs(cfg, seed=41)
    eng = Engine(inp)
    eng.prefill()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eager = {}
        for rid in (0, 3, 9):
            eng.draft_round(with_pool=False)
            a, p, o = eng.verify(T, seed=5, round_id=rid, with_stats=False)
            eager[rid] = (eng.tree.tokens.clone(), a.clone(), o.clone())
        eng.capture(temperature=T, seed=5)
        for rid in (9, 0, 3):
            eng.replay(rid)
            torch.cuda.current_stream().synchronize()
            eng.check()
            assert E.eagle3_last_launch_count(eng.ctx) > 10
            tt, a, o = eager[rid]
            assert torch.equal(eng.tree.tokens, tt)
            assert torch.equal(eng.accept_len, a), (rid, eng.accept_len, a)
            assert torch.equal(eng.out_tokens, o), (rid, eng.out_tokens, o)
    eng.close()
