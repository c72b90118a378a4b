"""Verification against caller-supplied target logits (eagle3_verify_logits)
compared with the oracle's verification on the same logits.

"EAGLE-3 精读" §5 (正确性、复现与风险): greedy verification keeps the target's
greedy sequence and sampling keeps its distribution with the residual
correction.  The oracle's verify_greedy / verify_sample take the logits as
given (they are pinned by brute force over all paths and by the chi-square
test of the output marginals), so they are the reference here: the kernels
must emit the same accepted lengths, paths and tokens, bit for bit, up to the
counted near-ties of the parity rule, and the same per-node argmax,
log-sum-exp and largest logit within the logit tolerance.

Trees come from real GPU draft rounds (including padded trees under a verify
cap); the logits are seeded normals with planted agreement so that long
paths are accepted, in fp32 and bf16, with padded rows (ld > vocab) and a
vocabulary that is not a multiple of the vector width.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import bf16_bits_to_f32, draw_logits, make_inputs
from oracle import layers as L
from oracle import round as R
from parity import TOL, Follow, GpuRound, Report

C0 = by_name("tiny_fp32_b1")
CASES = {
    # fp32 context, ragged vocabulary (1003 is not a multiple of 4), B = 2
    "fp32_b2_v1003": (C0.scaled(name="vl_fp32", batch=2, vocab=1003, prefix=40), "fp32", 1004, {}),
    # fp32 context, bf16 logits with padded rows, a verify cap that pads the tree
    "fp32_bf16logits_capped": (C0.scaled(name="vl_cap", batch=3, prefix=48), "bf16", 1040,
                               dict(verify_cap=[16, 5, 1])),
    # bf16 context (tcgen05 round), bf16 logits, k = 6
    "bf16_b3": (C0.scaled(name="vl_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2,
                          head_dim=64, ffn=512, vocab=4000, prefix=64, batch=3, depth=4, topk=6,
                          n_verify=20), "bf16", 4000, {}),
    # Llama-3.1-8B vocabulary and tree shape (d reduced: the logits path never reads weights)
    "vocab128256_tree": (C0.scaled(name="vl_8b_vocab", dtype="bf16", d=256, n_q_heads=4,
                                   n_kv_heads=2, head_dim=64, ffn=512, vocab=128256, prefix=64,
                                   batch=1, depth=6, topk=10, n_verify=60), "bf16", 128256, {}),
    # the serving batch shape: 64 chains of 3
    "vocab128256_b64_chain": (C0.scaled(name="vl_b64", dtype="bf16", d=256, n_q_heads=4,
                                        n_kv_heads=2, head_dim=64, ffn=512, vocab=128256,
                                        prefix=32, batch=64, depth=3, topk=1, n_verify=3),
                              "fp32", 128256, {}),
}


def _plant(z, tree_tok, tree_par, rng, V):
    """Make the target agree with the draft often: at most nodes, one child's
    token gets the row's largest logit (plus a margin), so long paths exist."""
    for b in range(tree_tok.shape[0]):
        M1 = tree_tok.shape[1]
        for u in range(M1):
            if u > 0 and tree_tok[b, u] < 0:
                continue
            kids = [c for c in range(M1) if tree_par[b, c] == u and tree_tok[b, c] >= 0]
            if kids and rng.random() < 0.8:
                c = kids[int(rng.integers(len(kids)))]
                row = b * M1 + u
                z[row, tree_tok[b, c]] = z[row, :V].max() + 2.0 + rng.random()
    return z


def _host_tree(tr, b):
    n = tr["tokens"].shape[1]
    return R.Tree(tr["tokens"][b].astype(np.int64), tr["parent"][b].astype(np.int64),
                  tr["depth"][b].astype(np.int64), tr["pos"][b].astype(np.int64),
                  tr["score"][b].astype(np.float64), tr["pool_index"][b].astype(np.int64),
                  np.zeros((n, n), dtype=bool))


def _run_case(cuda, name, temps=(0.0, 1.0, 0.7), seed=3, round_id=11):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine

    cfg, ldt, ld, caps = CASES[name]
    inp = make_inputs(cfg, seed=seed, with_target=False)
    eng = Engine(inp, with_target=False)
    eng.prefill()
    if caps:
        eng.set_control(**caps)
    eng.draft_round(with_pool=False)
    torch.cuda.synchronize()
    eng.check()
    tr = {k: getattr(eng.tree, k).cpu().numpy() for k in
          ("tokens", "parent", "depth", "pos", "pool_index", "score")}
    B, M1, V = cfg.batch, cfg.n_verify + 1, cfg.vocab
    rng = np.random.default_rng(seed)
    raw = draw_logits(seed, B * M1, V, ld, 2.0, ldt)
    zf = bf16_bits_to_f32(raw) if ldt == "bf16" else raw.copy()
    zf = _plant(zf.astype(np.float64), tr["tokens"], tr["parent"], rng, V)
    # round the planted values to the storage type too (exactly representable)
    if ldt == "bf16":
        from eagle_draft_tree_02_b300.synth import bf16_bits_from_f64
        raw = bf16_bits_from_f64(zf.reshape(-1)).reshape(zf.shape)
        zf = bf16_bits_to_f32(raw).astype(np.float64)
        dev = torch.from_numpy(raw.view(np.int16)).to(cuda).view(torch.bfloat16)
        code = E.BF16
    else:
        zf = zf.astype(np.float32).astype(np.float64)
        dev = torch.from_numpy(zf.astype(np.float32)).to(cuda)
        code = E.FP32
    # the logits are given exactly to both sides, so only the kernels' fp32
    # arithmetic separates them: the fp32 tolerances apply for either dtype
    tol = TOL["fp32"]
    st = eng.stream()
    for T in temps:
        mode = 0 if T == 0 else 1
        s = E.eagle3_verify_logits(eng.ctx, B, eng._tree_s, dev.data_ptr(), code, ld, mode,
                                   float(T or 1.0), 5, round_id, eng.accept_len.data_ptr(),
                                   eng.path.data_ptr(), eng.out_tokens.data_ptr(), eng.stats, st)
        assert s == E.OK, E.eagle3_last_error(eng.ctx)
        torch.cuda.synchronize()
        eng.check()
        v = dict(accept_len=eng.accept_len.cpu().numpy(), path=eng.path.cpu().numpy(),
                 out_tokens=eng.out_tokens.cpu().numpy(),
                 stats={k: t.cpu().numpy() for k, t in eng.stats_t.items()})
        gpu = GpuRound(tree=tr, pool={}, verify={T: v})
        rep = Report()
        for b in range(B):
            tree = _host_tree(tr, b)
            n = tree.n_real
            z = zf[b * M1:(b + 1) * M1, :V]
            real = [0] + [u for u in range(1, M1) if tree.tok[u] >= 0]
            zt = z[real] / (T if T else 1.0)
            rep.err("z_max", np.abs(z[real].max(axis=1) - v["stats"]["z_max"][b][real]).max())
            rep.err("lse", np.abs(L.logsumexp(zt) - v["stats"]["lse"][b][real]).max())
            dec = Follow(cfg, gpu, rep, tol["tie"], T)
            res = (R.verify_greedy(tree, z, dec, b) if T == 0 else
                   R.verify_sample(tree, z, T, 5, round_id, dec, b))
            if int(v["accept_len"][b]) != res.accept_len:
                rep.failures.append(("accept_len", T, b))
            if [int(x) for x in v["path"][b] if x >= 0] != res.path:
                rep.failures.append(("path", T, b))
            if [int(x) for x in v["out_tokens"][b] if x >= 0] != res.out_tokens:
                rep.failures.append(("out_tokens", T, b))
            assert n >= 1
        print(name, T, rep, "accept", v["accept_len"].tolist()[:8])
        assert not rep.failures, rep
        assert rep.max_err["z_max"] <= tol["logit"] and rep.max_err["lse"] <= tol["logit"], rep
        assert len(rep.near_ties) <= 2, rep
    eng.close()


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_verify_logits_matches_oracle(cuda, lib_built, name):
    _run_case(cuda, name)


@pytest.mark.gpu
def test_verify_logits_rejects_bad_layouts(cuda, lib_built):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine

    cfg = CASES["fp32_b2_v1003"][0]
    eng = Engine(make_inputs(cfg, seed=1, with_target=False), with_target=False)
    eng.prefill()
    eng.draft_round(with_pool=False)
    B, M1 = cfg.batch, cfg.n_verify + 1
    buf = torch.zeros(B * M1 * 1008 + 8, dtype=torch.float32, device=cuda)
    st = eng.stream()
    args = lambda ptr, code, ld, mode=0: E.eagle3_verify_logits(
        eng.ctx, B, eng._tree_s, ptr, code, ld, mode, 1.0, 0, 0, eng.accept_len.data_ptr(),
        eng.path.data_ptr(), eng.out_tokens.data_ptr(), None, st)
    assert args(buf.data_ptr(), E.FP32, 1002) == E.ERR_SHAPE          # ld < vocab
    assert args(buf.data_ptr(), E.FP32, 1005) == E.ERR_INVALID_ARG    # rows not 16-byte aligned
    assert args(buf.data_ptr() + 4, E.FP32, 1004) == E.ERR_INVALID_ARG  # base not aligned
    assert args(buf.data_ptr(), 7, 1004) == E.ERR_INVALID_ARG         # unknown dtype
    assert args(buf.data_ptr(), E.FP32, 1004, mode=2) == E.ERR_UNSUPPORTED
    assert args(0, E.FP32, 1004) == E.ERR_INVALID_ARG
    assert args(buf.data_ptr(), E.FP32, 1008) == E.OK
    torch.cuda.synchronize()
    eng.check()
    eng.close()
