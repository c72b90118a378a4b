"""The allocation-free LM-head entry point against the context-based one.

eagle3_lm_head_topk_noalloc serves callers that must not allocate device
memory (a runtime that owns all of HBM, a plugin bound to its host's
allocator, a latency-critical path): it keeps its scratch in a fixed array in
the library's device memory instead of a context workspace.  Here it must give
the same (token, log q, log-sum-exp) rows as eagle3_lm_head_topk on the same
weights and inputs, on two calls in a row with different inputs (the shared
array keeps the previous call's contents), and the second call must not change
the device's free memory.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import CONFIGS
from eagle_draft_tree_02_b300.synth import make_inputs
from parity import TOL

C0 = CONFIGS[0]
SMALL_BF16 = C0.scaled(name="noalloc_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2,
                       head_dim=64, ffn=512, vocab=5000, prefix=40, batch=3, depth=3, topk=5,
                       n_verify=8, lm_std=0.08)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [C0, SMALL_BF16], ids=["fp32", "bf16"])
def test_noalloc_head_matches_context_head(cuda, lib_built, cfg):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine

    inp = make_inputs(cfg, seed=31)
    eng = Engine(inp)
    R, k = cfg.batch * cfg.topk, cfg.topk
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    code = E.BF16 if cfg.dtype == "bf16" else E.FP32
    tol = TOL[cfg.dtype]["logit"]
    i32 = dict(dtype=torch.int32, device=cuda)
    f32 = dict(dtype=torch.float32, device=cuda)
    w_lm = eng.w["w_lm"]
    st = eng.stream()
    free = []
    for call in range(2):
        h = torch.from_numpy(np.random.default_rng(100 + call).standard_normal((R, cfg.d))
                             .astype(np.float32)).to(cuda).to(dt)
        tok_a, lq_a, lse_a = torch.empty((R, k), **i32), torch.empty((R, k), **f32), torch.empty(R, **f32)
        s = E.eagle3_lm_head_topk(eng.ctx, R, h.data_ptr(), tok_a.data_ptr(), lq_a.data_ptr(),
                                  lse_a.data_ptr(), st)
        assert s == E.OK, E.eagle3_last_error(eng.ctx)
        tok_b = torch.full((R, k), -7, **i32)
        lq_b, lse_b = torch.full((R, k), 9.0, **f32), torch.full((R,), 9.0, **f32)
        status = torch.full((1,), -1, **i32)
        s = E.eagle3_lm_head_topk_noalloc(code, cfg.vocab, cfg.d, k, w_lm.data_ptr(), R, h.data_ptr(),
                                          tok_b.data_ptr(), lq_b.data_ptr(), lse_b.data_ptr(),
                                          status.data_ptr(), st)
        assert s == E.OK
        torch.cuda.synchronize()
        eng.check()
        free.append(torch.cuda.mem_get_info()[0])
        assert int(status.item()) == 0
        assert torch.equal(tok_a, tok_b), (call, tok_a, tok_b)
        assert (lq_a - lq_b).abs().max().item() <= tol
        assert (lse_a - lse_b).abs().max().item() <= tol
    # the second call allocated nothing
    assert free[1] == free[0]
    eng.close()
