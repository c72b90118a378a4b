"""Steady-state decoding: rounds chained on the device, checked round by round.

After each round's verification, eagle3_next_rows turns the accepted tokens
and the bonus token of every request into the next round's new rows (a
different count per request), the caller adds their target features (seeded
synthetic rows stand in for the target's) and advances seq_lens by the rows
just committed, and eagle3_draft_round_ragged drafts from the new roots.  The
oracle sees the same committed rows: each round it recomputes the prefix K/V
of all of a request's rows and runs the round from the last one.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs
from oracle import round as R
from parity import TOL

C0 = by_name("tiny_fp32_b1")
CASES = {
    "fp32_b3": C0.scaled(batch=3, prefix=40, prefix_range=(20, 40), depth=4, topk=3, n_verify=10,
                         lm_std=0.3),
    "bf16_b2": C0.scaled(name="steady_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                         ffn=512, vocab=2048, prefix=60, batch=2, depth=4, topk=4, n_verify=12,
                         lm_std=0.3),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_steady_state_rounds_match_oracle(cuda, lib_built, name):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine, to_device
    from eagle_draft_tree_02_b300.synth import bf16_bits_from_f64
    cfg = CASES[name]
    inp = make_inputs(cfg, seed=51)
    D, B = cfg.depth, cfg.batch
    rounds = 3
    eng = Engine(inp, max_new=D + 1, max_prefix_extra=rounds * (D + 1))
    eng.prefill()
    w = R.weights_f32(inp)
    f32 = inp.feats_f32()
    # committed rows per request (oracle's view): features and tokens
    rows_f = [list(f32[inp.cu_rows[b]:inp.cu_rows[b + 1]]) for b in range(B)]
    rows_t = [list(inp.tokens[inp.cu_rows[b]:inp.cu_rows[b + 1]]) for b in range(B)]
    rng = np.random.default_rng(77)
    st = eng.stream()
    cu = torch.empty(B + 1, dtype=torch.int32, device=cuda)
    toks = torch.empty(B * (D + 1), dtype=torch.int32, device=cuda)
    tol = TOL[cfg.dtype]
    accepted_total = 0
    for rnd in range(rounds):
        if rnd == 0:
            eng.draft_round(with_pool=False)          # one new row per request: the root
            counts = [1] * B
        else:
            s = E.eagle3_next_rows(eng.ctx, B, eng.accept_len.data_ptr(), eng.out_tokens.data_ptr(),
                                   cu.data_ptr(), toks.data_ptr(), st)
            assert s == E.OK
            cu_h = cu.cpu().numpy()
            counts = list(np.diff(cu_h))
            total = int(cu_h[-1])
            new_t = toks[:total].cpu().numpy()
            feats = rng.standard_normal((total, 3 * cfg.d))
            fbits = bf16_bits_from_f64(feats) if cfg.dtype == "bf16" else feats.astype(np.float32)
            fd = to_device(fbits, cuda)
            f_rows = fd.float().cpu().numpy() if cfg.dtype == "bf16" else fbits
            for b in range(B):
                lo, hi = int(cu_h[b]), int(cu_h[b + 1])
                rows_f[b] += list(f_rows[lo:hi])
                rows_t[b] += list(new_t[lo:hi])
            s = E.eagle3_draft_round_ragged(eng.ctx, B, total, cu.data_ptr(), fd.data_ptr(),
                                            toks.data_ptr(), eng.kv, eng._tree_s, None, st)
            assert s == E.OK, E.eagle3_last_error(eng.ctx)
        eng.verify(0.0, with_stats=False)
        torch.cuda.synchronize()
        eng.check()
        acc = eng.accept_len.cpu().numpy()
        outs = eng.out_tokens.cpu().numpy()
        for b in range(B):
            F = np.stack(rows_f[b])
            T = np.array(rows_t[b], dtype=np.int64)
            P = len(T)
            K, V = R.prefix_kv(w, cfg, F, T)
            rr = R.round_request(w, cfg, K, V, F[-1], T[-1], P - 1, temperatures=(0.0,))
            assert np.array_equal(rr.tree.tok, eng.tree.tokens[b].cpu().numpy()), (rnd, b)
            res = rr.verify[0.0]
            assert int(acc[b]) == res.accept_len, (rnd, b)
            assert [int(x) for x in outs[b] if x >= 0] == res.out_tokens, (rnd, b)
            # the new rows' K/V in the cache
            L0 = P - counts[b]
            gk = eng.k_cache[b, L0:P].float().cpu().numpy()
            assert np.abs(gk - K[L0:P]).max() < max(tol["logit"], 1e-3)
        accepted_total += int(acc.sum())
        # commit this round's rows
        eng.seq_lens += torch.tensor(counts, dtype=torch.int32, device=cuda)
    assert accepted_total > 0   # the loop did carry accepted tokens into later rounds
