"""The allocation-free LM-head entry point against the context-based one and
against the oracle.

eagle3_lm_head_topk_noalloc serves callers that must not allocate device
memory (a runtime that owns all of HBM, a plugin bound to its host's
allocator, a latency-critical path): it keeps its scratch in a fixed array in
the library's device memory instead of a context workspace.  Here it must give
the same (token, log q, log-sum-exp) rows as eagle3_lm_head_topk on the same
weights and inputs, on two calls in a row with different inputs (the shared
array keeps the previous call's contents), agree with the oracle's draft head,
and the second call must not change the device's free memory.  Requests whose
partials exceed the fixed array, and bf16 requests of more than 256 rows, are
refused with EAGLE3_ERR_SHAPE and leave the outputs untouched.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import bf16_bits_to_f32, make_inputs
from oracle import layers as L
from parity import TOL, _valid_choice

C0 = by_name("tiny_fp32_b1")
SMALL_BF16 = C0.scaled(name="noalloc_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2,
                       head_dim=64, ffn=512, vocab=5000, prefix=40, batch=3, depth=3, topk=5,
                       n_verify=8, lm_std=0.08)
# 256 rows with k = 16: the persistent head's running state does not fit in
# shared memory, so the head falls back to the tiled kernel with more partials
WIDE_BF16 = SMALL_BF16.scaled(name="noalloc_bf16_wide", batch=16, topk=16, depth=2, n_verify=8)


def _host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.float().cpu().numpy()


def _against_oracle(cfg, w_lm_host, h, tok, lq, lse):
    """GPU rows vs the oracle's draft head (fp64): tokens a valid top-k up to
    the tie tolerance, log q and log-sum-exp within the logit tolerance."""
    tol = TOL[cfg.dtype]
    hv = _host(h).astype(np.float64)
    ell = L.linear(hv, w_lm_host)
    _, logq, _ = L.draft_logq({"w_lm": w_lm_host}, cfg, hv)
    tok, lq, lse = tok.cpu().numpy(), lq.cpu().numpy(), lse.cpu().numpy()
    for r in range(hv.shape[0]):
        assert _valid_choice(logq[r], tok[r].tolist(), tol["tie"]), r
        assert np.abs(logq[r][tok[r]] - lq[r]).max() <= tol["logit"], r
    assert np.abs(L.logsumexp(ell) - lse).max() <= tol["logit"]


def _run_pair(cuda, cfg, seed, rows=None):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine

    inp = make_inputs(cfg, seed=seed)
    eng = Engine(inp, with_target=False)
    R, k = rows or cfg.batch * cfg.topk, cfg.topk
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    code = E.BF16 if cfg.dtype == "bf16" else E.FP32
    tol = TOL[cfg.dtype]["logit"]
    i32 = dict(dtype=torch.int32, device=cuda)
    f32 = dict(dtype=torch.float32, device=cuda)
    w_lm = eng.w["w_lm"]
    w_host = inp.f32("w_lm")
    st = eng.stream()
    free = []  # (before, after) the allocation-free call, per call
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
        # every tensor of the call exists before the first reading, so the two
        # readings bracket the entry point alone (not the test's own tensors)
        torch.cuda.synchronize()
        before = torch.cuda.mem_get_info()[0]
        s = E.eagle3_lm_head_topk_noalloc(code, cfg.vocab, cfg.d, k, w_lm.data_ptr(), R, h.data_ptr(),
                                          tok_b.data_ptr(), lq_b.data_ptr(), lse_b.data_ptr(),
                                          status.data_ptr(), st)
        assert s == E.OK
        torch.cuda.synchronize()
        free.append((before, torch.cuda.mem_get_info()[0]))
        eng.check()
        assert int(status.item()) == 0
        assert torch.equal(tok_a, tok_b), (call, tok_a, tok_b)
        assert (lq_a - lq_b).abs().max().item() <= tol
        assert (lse_a - lse_b).abs().max().item() <= tol
        _against_oracle(cfg, w_host, h, tok_b, lq_b, lse_b)
    # the first call on a device may load the module that holds the fixed
    # array (lazy loading); the second call allocated nothing
    print(f"{cfg.name}: free memory (before, after) call 1, call 2: {free}")
    assert free[1][1] == free[1][0]
    eng.close()


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [C0, SMALL_BF16], ids=["fp32", "bf16"])
def test_noalloc_head_matches_context_head(cuda, lib_built, cfg):
    _run_pair(cuda, cfg, 31)


@pytest.mark.gpu
def test_noalloc_head_wide_fallback_matches_context_head(cuda, lib_built):
    """R = 256, k = 16: the tiled fallback writes 4 partials per 128 tokens."""
    _run_pair(cuda, WIDE_BF16, 37, rows=256)


@pytest.mark.gpu
def test_noalloc_head_refuses_what_does_not_fit(cuda, lib_built):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E

    i32 = dict(dtype=torch.int32, device=cuda)
    f32 = dict(dtype=torch.float32, device=cuda)
    st = torch.cuda.current_stream().cuda_stream
    d, V, k = 64, 131072, 16
    w = torch.zeros((V, d), dtype=torch.bfloat16, device=cuda)
    for R, why in ((256, "partials exceed the fixed array"), (257, "more than 256 bf16 rows")):
        h = torch.zeros((R, d), dtype=torch.bfloat16, device=cuda)
        tok = torch.full((R, k), -7, **i32)
        lq, lse = torch.full((R, k), 9.0, **f32), torch.full((R,), 9.0, **f32)
        status = torch.full((1,), -1, **i32)
        torch.cuda.synchronize()
        s = E.eagle3_lm_head_topk_noalloc(E.BF16, V, d, k, w.data_ptr(), R, h.data_ptr(),
                                          tok.data_ptr(), lq.data_ptr(), lse.data_ptr(),
                                          status.data_ptr(), st)
        torch.cuda.synchronize()
        assert s == E.ERR_SHAPE, (why, s)
        # nothing ran: the outputs and the status word are untouched
        assert (tok == -7).all() and (lq == 9.0).all() and (lse == 9.0).all(), why
        assert int(status.item()) == -1, why
