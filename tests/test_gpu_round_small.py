"""GPU parity of whole rounds on small shapes (the oracle finishes in seconds).

Each case runs prefill, one draft round and verification (greedy and/or T=1)
through the C ABI and compares every index, token and value with the oracle
(see parity.py for the tolerances and the near-tie rule).
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs
from parity import TOL, compare, gpu_round
from oracle import round as R

C0 = by_name("tiny_fp32_b1")
SMALL_BF16 = C0.scaled(name="small_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2,
                       head_dim=64, ffn=512, vocab=2048, prefix=100, batch=2, depth=4, topk=4,
                       n_verify=12, lm_std=0.02 * 4, temperatures=(0.0, 1.0))

TWO_STAGE_FP32 = C0.scaled(name="two_stage_fp32", lr_rank=16, lr_cand=32, depth=4, topk=4,
                           n_verify=12, temperatures=(0.0, 1.0))
TWO_STAGE_BF16 = SMALL_BF16.scaled(name="two_stage_bf16", vocab=40000, lr_rank=64, lr_cand=64,
                                   depth=4, topk=5, n_verify=14)

CASES = {
    "tiny_fp32": (C0, 0),
    "tiny_fp32_seed7": (C0, 7),
    "ragged_b3": (C0.scaled(batch=3, prefix=64, prefix_range=(20, 64), depth=4, topk=3, n_verify=10), 1),
    "chain_paged_b4": (C0.scaled(batch=4, prefix=60, prefix_range=(10, 60), depth=3, topk=1,
                                 n_verify=3, page_size=16), 2),
    "depth1": (C0.scaled(depth=1, topk=4, n_verify=4), 3),
    "keep_all": (C0.scaled(depth=3, topk=3, n_verify=3 + 2 * 9), 4),
    "wide_k16": (C0.scaled(depth=2, topk=16, n_verify=40, prefix=70), 5),
    "small_bf16": (SMALL_BF16, 6),
    "two_stage_fp32": (TWO_STAGE_FP32, 8),
    "two_stage_bf16_v40k": (TWO_STAGE_BF16, 9),
    # drafter variants (FC norm, post-norm) with non-unit gains
    "variant_fc_norm_fp32": (C0.scaled(name="fc_norm_fp32", fc_norm=True, gain_std=0.1), 10),
    "variant_post_norm_fp32": (C0.scaled(name="post_norm_fp32", post_norm=True, gain_std=0.1), 11),
    "variant_fc_post_bf16": (SMALL_BF16.scaled(name="fc_post_bf16", fc_norm=True, post_norm=True,
                                               gain_std=0.1), 12),
    # 16 query heads on one KV head: the verify pass's 208 queries per KV head
    # take the tcgen05 attention (two groups of up to 128), the draft passes'
    # 64 the queries-as-M kernel, the root's 16 the keys-as-M kernel
    "wide_groups_bf16": (SMALL_BF16.scaled(name="wide_groups_bf16", d=1024, n_q_heads=16, n_kv_heads=1,
                                           head_dim=64, ffn=1024), 13),
    # sampling at T != 1: 1/T scales the target logits in the head, the walk and the bonus draw
    "small_bf16_t07": (SMALL_BF16.scaled(name="small_bf16_t07", temperatures=(0.7,)), 14),
}


def _engine(cfg, seed):
    from eagle_draft_tree_02_b300.runner import Engine
    inp = make_inputs(cfg, seed=seed)
    eng = Engine(inp)
    eng.prefill()
    return inp, eng


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_round_parity(cuda, lib_built, name):
    cfg, seed = CASES[name]
    inp, eng = _engine(cfg, seed)
    temps = cfg.temperatures
    gpu = gpu_round(eng, temps, seed=11, round_id=3)
    rep = compare(cfg, inp, gpu, temps, seed=11, round_id=3)
    tol = TOL[cfg.dtype]
    assert not rep.failures, rep
    assert rep.max_err["logq"] <= tol["logit"], rep
    assert rep.max_err["score/depth"] <= tol["logit"], rep
    if temps:
        assert rep.max_err["z_max"] <= tol["logit"], rep
        assert rep.max_err["lse"] <= tol["logit"], rep
    print(name, rep)


@pytest.mark.gpu
def test_prefix_cache_matches_oracle(cuda, lib_built):
    cfg = CASES["ragged_b3"][0]
    inp, eng = _engine(cfg, 1)
    import torch
    torch.cuda.synchronize()
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    for b in range(cfg.batch):
        lo, hi = int(inp.cu_rows[b]), int(inp.cu_rows[b + 1])
        K, V = R.prefix_kv(w, cfg, f[lo:hi], inp.tokens[lo:hi])
        gk = eng.k_cache[b, : hi - lo].float().cpu().numpy()
        gv = eng.v_cache[b, : hi - lo].float().cpu().numpy()
        assert np.max(np.abs(gk - K)) < 1e-4
        assert np.max(np.abs(gv - V)) < 1e-4


@pytest.mark.gpu
def test_sampling_many_round_ids(cuda, lib_built):
    cfg = C0
    inp, eng = _engine(cfg, 0)
    gpu = gpu_round(eng, (), seed=0)
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    rr = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1, with_verify=False)
    z, _ = R.verify_logits(w, cfg, K, V, P - 1, rr.tree, rr.draft)
    assert np.array_equal(rr.tree.tok, gpu.tree["tokens"][0])
    mism = 0
    for rid in range(40):
        a, p, o = eng.verify(1.0, 5, rid)
        res = R.verify_sample(rr.tree, z, 1.0, 5, rid)
        go = [int(x) for x in o[0].cpu().numpy() if x >= 0]
        mism += go != res.out_tokens
    assert mism == 0


@pytest.mark.gpu
def test_build_tree_entry_point_random_pools(cuda, lib_built):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine, TreeOut
    cfg = C0.scaled(batch=4, depth=4, topk=3, n_verify=12)
    eng = Engine(make_inputs(cfg, seed=2))
    rng = np.random.default_rng(0)
    B, k, D = cfg.batch, cfg.topk, cfg.depth
    pool_n = cfg.pool_size
    tok = np.zeros((B, pool_n), np.int32); par = np.zeros((B, pool_n), np.int32)
    sc = np.zeros((B, pool_n), np.float32); dep = np.zeros((B, pool_n), np.int32)
    for b in range(B):
        n = 0
        for j in range(k):
            tok[b, n], par[b, n], sc[b, n], dep[b, n] = j, -1, -rng.exponential(), 1; n += 1
        front = list(range(k))
        for t in range(2, D + 1):
            base = n
            for p in front:
                for j in range(k):
                    q = 0.0 if rng.random() < 0.2 else -rng.exponential()
                    tok[b, n], par[b, n], sc[b, n], dep[b, n] = j + 10 * t, p, np.float32(sc[b, p] + q), t
                    n += 1
            front = sorted(range(base, n), key=lambda i: (-sc[b, i], i))[:k]
    dev = torch.device("cuda")
    # keep every device tensor alive until the kernel has run
    d_tok, d_par, d_sc, d_dep = (torch.from_numpy(a).to(dev) for a in (tok, par, sc, dep))
    rt = torch.from_numpy(np.arange(B, dtype=np.int32) + 100).to(dev)
    rpos = torch.from_numpy(np.full(B, 50, np.int32)).to(dev)
    s = E.eagle3_build_tree(eng.ctx, B, pool_n, d_tok.data_ptr(), d_par.data_ptr(), d_sc.data_ptr(),
                            d_dep.data_ptr(), rt.data_ptr(), rpos.data_ptr(), eng._tree_s, eng.stream())
    assert s == E.OK
    torch.cuda.synchronize()
    eng.check()
    for b in range(B):
        tr = R.build_tree(tok[b], par[b], sc[b].astype(np.float64), dep[b], 100 + b, 50, cfg.n_verify)
        assert np.array_equal(eng.tree.tokens[b].cpu().numpy(), tr.tok)
        assert np.array_equal(eng.tree.parent[b].cpu().numpy(), tr.parent)
        assert np.array_equal(eng.tree.pool_index[b].cpu().numpy(), tr.pool_index)
        assert np.array_equal(eng.tree.pos[b].cpu().numpy(), tr.pos)


@pytest.mark.gpu
def test_build_tree_flags_unclosed_pool(cuda, lib_built):
    """A pool whose kept set is not ancestor-closed raises the device flag (no fault)."""
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine
    cfg = C0.scaled(batch=1, depth=2, topk=2, n_verify=2)
    eng = Engine(make_inputs(cfg, seed=2))
    dev = torch.device("cuda")
    tok = torch.tensor([[1, 2, 3, 4, 5, 6]], dtype=torch.int32, device=dev)
    par = torch.tensor([[-1, -1, 0, 0, 1, 1]], dtype=torch.int32, device=dev)
    sc = torch.tensor([[-5.0, -6.0, -0.1, -0.2, -7, -8]], dtype=torch.float32, device=dev)  # children beat parents
    dep = torch.tensor([[1, 1, 2, 2, 2, 2]], dtype=torch.int32, device=dev)
    rt = torch.tensor([9], dtype=torch.int32, device=dev)
    rp = torch.tensor([10], dtype=torch.int32, device=dev)
    s = E.eagle3_build_tree(eng.ctx, 1, 6, tok.data_ptr(), par.data_ptr(), sc.data_ptr(), dep.data_ptr(),
                            rt.data_ptr(), rp.data_ptr(), eng._tree_s, eng.stream())
    assert s == E.OK
    assert E.eagle3_check(eng.ctx) == E.ERR_DEVICE_ASSERT
    assert "ancestor" in E.eagle3_last_error(eng.ctx)
    assert E.eagle3_check(eng.ctx) == E.OK   # the flag is cleared once reported


@pytest.mark.gpu
def test_lm_head_topk_planted_ties(cuda, lib_built):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine
    cfg = C0
    inp = make_inputs(cfg, seed=4)
    eng = Engine(inp)
    rng = np.random.default_rng(1)
    Rr = cfg.topk
    h = rng.standard_normal((Rr, cfg.d)).astype(np.float32)
    # plant exact ties: duplicate LM-head rows so that several tokens share a logit
    W = inp.w["w_lm"].copy()
    W[17] = W[900]; W[901] = W[900]; W[5] = W[3]
    eng.w["w_lm"].copy_(torch.from_numpy(W))
    dev = torch.device("cuda")
    hd = torch.from_numpy(h).to(dev)
    tok = torch.empty((Rr, cfg.topk), dtype=torch.int32, device=dev)
    lq = torch.empty((Rr, cfg.topk), dtype=torch.float32, device=dev)
    lse = torch.empty(Rr, dtype=torch.float32, device=dev)
    # make row 0 prefer the tied tokens
    h[0] = W[900] / np.linalg.norm(W[900]) * 30
    hd.copy_(torch.from_numpy(h))
    s = E.eagle3_lm_head_topk(eng.ctx, Rr, hd.data_ptr(), tok.data_ptr(), lq.data_ptr(), lse.data_ptr(),
                              eng.stream())
    assert s == E.OK
    torch.cuda.synchronize()
    from oracle import layers as L
    ell = h.astype(np.float64) @ W.astype(np.float64).T
    for r in range(Rr):
        order = sorted(range(cfg.vocab), key=lambda j: (-ell[r, j], j))[: cfg.topk]
        got = tok[r].cpu().numpy().tolist()
        # exact ties must come out in ascending token order
        assert got == order, (r, got, order)
        np.testing.assert_allclose(lq[r].cpu().numpy(), ell[r, order] - L.logsumexp(ell[r]), atol=1e-4)
    assert tok[0].cpu().numpy().tolist()[:3] == [17, 900, 901]


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [TWO_STAGE_FP32.scaled(vocab=6000), TWO_STAGE_BF16.scaled(vocab=6000)],
                         ids=["fp32", "bf16"])
def test_two_stage_head_all_tied_lowrank_scores(cuda, lib_built, cfg):
    """Identical low-rank rows tie every token's low-rank score: the candidate
    buffer overflows (6000 tokens > 4096 entries) and the exact radix select
    must return the lr_cand lowest token ids, as the oracle's order does."""
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine
    from oracle import layers as L
    inp = make_inputs(cfg, seed=12)
    U = inp.w["lr_u"].copy()
    U[:] = U[7]
    inp.w["lr_u"] = U
    eng = Engine(inp)
    R, k = 3, cfg.topk
    rng = np.random.default_rng(3)
    h = rng.standard_normal((R, cfg.d)).astype(np.float32)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    hd = torch.from_numpy(h).to(cuda).to(dt)
    h64 = hd.float().cpu().numpy().astype(np.float64)
    tok = torch.empty((R, k), dtype=torch.int32, device=cuda)
    lq = torch.empty((R, k), dtype=torch.float32, device=cuda)
    lse = torch.empty(R, dtype=torch.float32, device=cuda)
    s = E.eagle3_lm_head_topk(eng.ctx, R, hd.data_ptr(), tok.data_ptr(), lq.data_ptr(), lse.data_ptr(),
                              eng.stream())
    assert s == E.OK, E.eagle3_last_error(eng.ctx)
    torch.cuda.synchronize()
    eng.check()
    w = {n: inp.f32(n) for n in ("lr_u", "lr_v", "w_lm")}
    cand, logq, _ = L.draft_logq(w, cfg, h64)
    tol = TOL[cfg.dtype]["logit"]
    for r in range(R):
        assert list(cand[r]) == list(range(cfg.lr_cand))     # all tied: lowest ids
        order = np.lexsort((cand[r], -logq[r]))[:k]
        assert tok[r].cpu().numpy().tolist() == [int(cand[r][j]) for j in order]
        np.testing.assert_allclose(lq[r].cpu().numpy(), logq[r][order], atol=tol)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg,T", [(SMALL_BF16, 1.0), (TWO_STAGE_BF16, 1.0), (SMALL_BF16, 0.7)],
                         ids=["bf16", "two_stage_bf16", "bf16_t07"])
def test_deferred_bonus_matches_the_head_draw(cuda, lib_built, cfg, T):
    """Sampling without the per-node Gumbel-argmax: the tensor-core head stores
    the target logits and the bonus is drawn only at each request's stop node.
    The walk's outputs equal those of the draw made inside the head (stats with
    g_argmax) over many round ids, and the bonus is that draw's Gumbel-argmax
    at the stop node."""
    import torch
    inp, eng = _engine(cfg, 6)
    eng.draft_round()
    for rid in range(48):
        a1, p1, o1 = [t.clone() for t in eng.verify(T, 5, rid, g_argmax=True)]
        g = eng.stats_t["g_argmax"].clone()
        a2, p2, o2 = [t.clone() for t in eng.verify(T, 5, rid)]
        assert torch.equal(a1, a2) and torch.equal(p1, p2) and torch.equal(o1, o2), rid
        for b in range(cfg.batch):
            n = int(a1[b])
            u = 0 if n == 0 else int(p1[b, n - 1])
            assert int(o1[b, n]) == int(g[b, u]) >= 0, (rid, b)
