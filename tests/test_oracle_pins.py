"""Pins of the CPU oracle against things other than itself.

The pages print no worked example, so each part of the oracle is pinned by an
independent library routine, a closed form, an invariant or brute force:

* primitives vs torch CPU float64 functional ops;
* RoPE: identity at position 0, norm preservation, the 2-D closed form and the
  relative-position invariant <R(m)q, R(n)k> = f(m - n);
* tree attention + positions + own-state feedback vs a sequential causal
  forward over every root-to-node path ("EAGLE-3 精读" §2, Training-Time Test);
* children / frontier / kept set vs brute-force sorts on the stated keys, and
  the tree invariants (ancestor closure, |kept| = M, monotone scores, mask =
  transitive closure of parent, k = 1 gives a chain);
* greedy verification vs brute force over all root-to-node paths ("EAGLE-3
  精读" §5: greedy keeps the target's sequence);
* sampling verification: output marginals vs the target distribution at V = 8
  (chi-square; "EAGLE-3 精读" §5: sampling keeps the target distribution when
  the residual correction is done), and a planted mistake (no residual
  correction) that the same test rejects;
* Philox4x64-10 vs numpy.random.Philox (an independent implementation);
* two-stage head: with all tokens as candidates it equals the single-stage
  head; with an exactly low-rank head the candidates are the true top-c;
* drafter variants (EAGLE-4 blog, 在EAGLE4中: FC Norm and Post-norm): the
  scale invariances that only a norm in the stated place gives (a post-norm
  layer is unchanged when hid and the attention output are scaled together; an
  FC-normed round is unchanged when every target feature is scaled), unit RMS
  of the normalised rows, and the tree/path equivalence with the variants on.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy import stats

from eagle_draft_tree_02_b300.configs import by_name, TINY_V8
from eagle_draft_tree_02_b300.synth import bf16_bits_from_f64, bf16_bits_to_f32, make_inputs
from oracle import layers as L
from oracle import philox
from oracle import round as R

T64 = torch.float64


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


# ----------------------------------------------------------------------------- primitives
def test_linear_rmsnorm_silu_match_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 37))
    W = rng.standard_normal((70000 // 1000 * 300, 37)).astype(np.float32)  # > one row chunk
    np.testing.assert_allclose(L.linear(x, W), F.linear(_t(x), _t(W)).numpy(), rtol=1e-12, atol=1e-12)
    g = rng.standard_normal(37)
    np.testing.assert_allclose(L.rmsnorm(x, g, 1e-5),
                               F.rms_norm(_t(x), (37,), _t(g), eps=1e-5).numpy(), rtol=1e-12)
    np.testing.assert_allclose(L.silu(x), F.silu(_t(x)).numpy(), rtol=1e-12)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (6, 3)])
def test_attend_matches_torch_sdpa_gqa(hq, hkv):
    rng = np.random.default_rng(hq * 10 + hkv)
    dh, n = 16, 23
    cfg = by_name("tiny_fp32_b1").scaled(n_q_heads=hq, n_kv_heads=hkv, head_dim=dh)
    q = rng.standard_normal((hq, dh))
    K = rng.standard_normal((n, hkv, dh))
    V = rng.standard_normal((n, hkv, dh))
    ours = L.attend(q, K, V, cfg).reshape(hq, dh)
    Kr = _t(K).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    Vr = _t(V).permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    ref = F.scaled_dot_product_attention(_t(q)[:, None, :], Kr, Vr)[:, 0, :]
    np.testing.assert_allclose(ours, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_rope_closed_form_and_invariants():
    rng = np.random.default_rng(2)
    # dh = 2: one pair, inv_freq = 1, so R(p) is the plane rotation by p radians.
    x = rng.standard_normal((4, 1, 2))
    pos = np.array([0, 1, 5, 1000])
    y = L.rope(x, pos, 5e5)
    c, s = np.cos(pos), np.sin(pos)
    np.testing.assert_allclose(y[:, 0, 0], c * x[:, 0, 0] - s * x[:, 0, 1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[:, 0, 1], s * x[:, 0, 0] + c * x[:, 0, 1], rtol=1e-12, atol=1e-12)
    # general dh: identity at 0, norms kept, and dot products depend only on m - n
    dh = 64
    q = rng.standard_normal((1, 3, dh))
    k = rng.standard_normal((1, 3, dh))
    np.testing.assert_allclose(L.rope(q, np.array([0]), 5e5), q, rtol=0, atol=0)
    qm = L.rope(q, np.array([1234]), 5e5)
    np.testing.assert_allclose(np.linalg.norm(qm, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-12)
    d1 = (L.rope(q, np.array([10]), 5e5) * L.rope(k, np.array([3]), 5e5)).sum(-1)
    d2 = (L.rope(q, np.array([2007]), 5e5) * L.rope(k, np.array([2000]), 5e5)).sum(-1)
    np.testing.assert_allclose(d1, d2, rtol=1e-9, atol=1e-10)
    # rotate-half pairing: perturbing element j moves only outputs j and j + dh/2
    e = np.zeros((1, 1, dh)); e[0, 0, 5] = 1.0
    out = L.rope(e, np.array([7]), 5e5)[0, 0]
    assert set(np.nonzero(np.abs(out) > 1e-15)[0]) <= {5, 5 + dh // 2}


# ----------------------------------------------------------------------------- Philox
def test_philox_matches_numpy_philox():
    rng = np.random.default_rng(3)
    for _ in range(50):
        ctr = [int(x) for x in rng.integers(0, 2 ** 63, size=4, dtype=np.int64)]
        ctr = [c * 2 + int(rng.integers(0, 2)) for c in ctr]
        key = [int(x) for x in rng.integers(0, 2 ** 63, size=2, dtype=np.int64)]
        # numpy's Philox increments its counter before producing a block.
        prev = ctr.copy()
        i = 0
        while True:
            prev[i] = (prev[i] - 1) % 2 ** 64
            if prev[i] != 2 ** 64 - 1:
                break
            i += 1
        # explicit uint64 arrays: a list of Python ints would pass through float64
        ref = np.random.Philox(counter=np.array(prev, dtype=np.uint64),
                               key=np.array(key, dtype=np.uint64)).random_raw(4)
        assert tuple(int(v) for v in ref) == philox.philox4x64_scalar(ctr, key)
        vec = philox.philox4x64(*[np.uint64(c) for c in ctr], key[0], key[1])
        assert tuple(int(v) for v in vec) == philox.philox4x64_scalar(ctr, key)


def test_gumbel_stream_layout_against_the_scalar_definition():
    """Token x reads word x % 4 of the block at counter index x // 4 (stream 1);
    checked against the word-by-word definition, not the vectorised code."""
    seed, rid, b, node = 11, 5, 3, 17
    xs = np.array([0, 1, 2, 3, 4, 7, 8, 1001, 128255], dtype=np.int64)
    g = philox.gumbel(seed, rid, b, node, xs)
    for x, gx in zip(xs, g):
        w = philox.philox4x64_scalar((rid, (b << 32) + node, int(x) // 4, 1), (seed, 0))[int(x) % 4]
        u = ((w >> 40) + 0.5) * 2.0 ** -24
        assert gx == -np.log(-np.log(u))


def test_philox_uniform_and_gumbel_ranges():
    u = philox.uniform(7, 3, 0, np.arange(1000), 2)
    assert u.min() >= 0 and u.max() < 1
    assert abs(u.mean() - 0.5) < 0.05
    g = philox.gumbel(7, 3, 0, 1, np.arange(200000))
    assert abs(g.mean() - np.euler_gamma) < 0.01          # Gumbel mean
    assert abs(g.var() - np.pi ** 2 / 6) < 0.03            # Gumbel variance


# ----------------------------------------------------------------------------- tree forward
def _brute_path_states(w, cfg, f, tok, P, pool, node):
    """Plain causal forward, one row at a time with a growing KV list, over
    prefix rows 0..P-1 and then the root-to-node path; returns (s, h) of the last row."""
    Ks, Vs = [], []
    path = pool.ancestors_or_self(node) if node is not None else []
    rows = [(tok[i], L.fused_feature(w, cfg, f[i][None])[0]) for i in range(P)]
    for t, i in enumerate(path):
        rows.append((pool.tok[i], None))
    s = h = None
    for pos, (y, g) in enumerate(rows):
        hid = g if g is not None else s
        x = L.decoder_input(w, cfg, np.array([y]), hid[None])
        q, k, v = L.qkv(w, cfg, x, np.array([pos]))
        Ks.append(k[0]); Vs.append(v[0])
        o = L.attend(q[0], np.stack(Ks), np.stack(Vs), cfg)
        s, h = L.layer_tail(w, cfg, hid[None], o[None])
        s, h = s[0], h[0]
    return s, h


@pytest.fixture(scope="module")
def tiny_round():
    cfg = by_name("tiny_fp32_b1").scaled(prefix=24, depth=4, topk=3, n_verify=10)
    inp = make_inputs(cfg, seed=11)
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    rr = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1, temperatures=(0.0, 1.0))
    return cfg, inp, w, f, P, K, V, rr


def test_tree_states_equal_sequential_path_forward(tiny_round):
    cfg, inp, w, f, P, K, V, rr = tiny_round
    s, h = _brute_path_states(w, cfg, f, inp.tokens, P, rr.draft.pool, None)
    np.testing.assert_allclose(rr.draft.s_root, s, rtol=1e-10, atol=1e-10)
    assert rr.draft.states, "no expanded node"
    for i, st in rr.draft.states.items():
        s, h = _brute_path_states(w, cfg, f, inp.tokens, P, rr.draft.pool, i)
        np.testing.assert_allclose(st, s, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(rr.draft.h[i], h, rtol=1e-10, atol=1e-10)


def test_verify_pass_equals_sequential_path_forward(tiny_round):
    cfg, inp, w, f, P, K, V, rr = tiny_round
    z, hv = R.verify_logits(w, cfg, K, V, P - 1, rr.tree, rr.draft)
    for u in range(1, len(rr.tree.tok)):
        _, h = _brute_path_states(w, cfg, f, inp.tokens, P, rr.draft.pool, int(rr.tree.pool_index[u]))
        np.testing.assert_allclose(hv[u], h, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(z, L.linear(hv, w["w_target"]), rtol=1e-12)


def test_prefix_kv_matches_sequential_forward(tiny_round):
    cfg, inp, w, f, P, K, V, rr = tiny_round
    # rows computed one at a time (position = row index) equal the batched prefix
    for i in (0, 5, P - 1):
        k1, v1 = R.prefix_kv(w, cfg, f[i:i + 1], inp.tokens[i:i + 1], rows=None)
        k1 = L.rope(L.linear(L.decoder_input(w, cfg, inp.tokens[i:i + 1],
                                             L.fuse(f[i:i + 1], w["w_fc"])), w["w_k"])
                    .reshape(1, cfg.n_kv_heads, cfg.head_dim), np.array([i]), cfg.rope_theta)
        np.testing.assert_allclose(K[i], k1[0], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- orderings
def test_children_frontier_and_kept_set_by_brute_force(tiny_round):
    cfg, inp, w, f, P, K, V, rr = tiny_round
    pool, k = rr.draft.pool, cfg.topk
    # children: the k best (log q desc, token asc) of each expanded node
    for (depth, rank), (cand, logq) in rr.draft.node_logq.items():
        best = sorted(range(len(cand)), key=lambda j: (-logq[j], cand[j]))[:k]
        base = 0 if depth == 0 else k + (depth - 1) * k * k + rank * k
        assert [pool.tok[base + j] for j in range(k)] == [int(cand[j]) for j in best]
        for j, c in enumerate(best):
            assert pool.logq[base + j] == logq[c]
    # frontier: k best of the depth's k*k candidates by (score desc, creation id asc)
    for t, fr in enumerate(rr.draft.frontiers[1:], start=2):
        base = k + (t - 2) * k * k
        cands = list(range(base, base + k * k))
        assert fr == sorted(cands, key=lambda i: (-pool.score[i], i))[:k]
    # kept set: global top-M by (score desc, depth asc, creation id asc)
    n = len(pool.tok)
    kept = sorted(range(n), key=lambda i: (-pool.score[i], pool.depth[i], i))[:cfg.n_verify]
    assert sorted(int(p) for p in rr.tree.pool_index[1:]) == sorted(kept)


def _check_tree_invariants(tr, m):
    n = len(tr.tok)
    assert n == m + 1 and tr.parent[0] == -1 and tr.depth[0] == 0
    for u in range(1, n):
        p = tr.parent[u]
        assert 0 <= p < u                           # ancestor-closed, parents come first
        assert tr.depth[u] == tr.depth[p] + 1
        assert tr.score[u] <= tr.score[p]           # confidence never rises along a path
        assert tr.pos[u] == tr.pos[0] + tr.depth[u]
    assert list(tr.depth) == sorted(tr.depth)       # depth-major order
    # mask = reflexive transitive closure of parent
    anc = np.eye(n, dtype=bool)
    for u in range(n):
        j = tr.parent[u]
        while j >= 0:
            anc[u, j] = True
            j = tr.parent[j]
    assert (tr.mask == anc).all()


@pytest.mark.parametrize("seed", range(6))
def test_build_tree_random_pools(seed):
    rng = np.random.default_rng(100 + seed)
    k, D = int(rng.integers(1, 5)), int(rng.integers(1, 6))
    # a synthetic pool with the draft's structure: log q <= 0 per edge
    tok, par, sc, dep = [], [], [], []
    for j in range(k):
        tok.append(j); par.append(-1); sc.append(-float(rng.exponential())); dep.append(1)
    front = list(range(k))
    for t in range(2, D + 1):
        base = len(tok)
        for r, p in enumerate(front):
            for j in range(k):
                q = -float(rng.exponential()) if rng.random() > 0.2 else 0.0  # planted ties
                tok.append(j); par.append(p); sc.append(sc[p] + q); dep.append(t)
        front = sorted(range(base, len(tok)), key=lambda i: (-sc[i], i))[:k]
    m = int(rng.integers(1, len(tok) + 1))
    tr = R.build_tree(tok, par, np.array(sc), dep, 7, 99, m)
    _check_tree_invariants(tr, m)
    kept = sorted(range(len(tok)), key=lambda i: (-sc[i], dep[i], i))[:m]
    assert sorted(tr.pool_index[1:].tolist()) == sorted(kept)
    if k == 1:   # a chain: every node has at most one child
        assert all(len(tr.children(u)) <= 1 for u in range(len(tr.tok)))


def test_chain_k1_is_a_chain():
    cfg = by_name("tiny_fp32_b1").scaled(prefix=8, depth=3, topk=1, n_verify=3)
    inp = make_inputs(cfg, seed=5)
    w = R.weights_f32(inp); f = inp.feats_f32(); P = 8
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    rr = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1)
    assert list(rr.tree.parent) == [-1, 0, 1, 2] and list(rr.tree.depth) == [0, 1, 2, 3]


# ----------------------------------------------------------------------------- verification
def _all_paths(tr):
    paths = [[]]
    stack = [[]]
    while stack:
        p = stack.pop()
        u = p[-1] if p else 0
        for c in tr.children(u):
            paths.append(p + [c]); stack.append(p + [c])
    return paths


@pytest.mark.parametrize("seed", range(8))
def test_greedy_is_longest_matching_path(seed, tiny_round):
    cfg, inp, w, f, P, K, V, rr = tiny_round
    tr = rr.tree
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((len(tr.tok), 40))
    # plant agreement so that long paths exist: make the target prefer some children
    for u in range(len(tr.tok)):
        kids = tr.children(u)
        if kids and rng.random() < 0.7:
            c = kids[int(rng.integers(len(kids)))]
            z[u, tr.tok[c] % 40] = 10.0
    tr2 = R.Tree(tr.tok % 40, tr.parent, tr.depth, tr.pos, tr.score, tr.pool_index, tr.mask)
    # sibling tokens must stay distinct for the path to be unique
    if any(len(set(tr2.tok[tr2.children(u)])) != len(tr2.children(u)) for u in range(len(tr2.tok))):
        pytest.skip("token folding made siblings collide")
    res = R.verify_greedy(tr2, z)
    best = max((p for p in _all_paths(tr2)
                if all(tr2.tok[c] == np.argmax(z[0 if i == 0 else p[i - 1]]) for i, c in enumerate(p))),
               key=len)
    assert res.path == best
    last = best[-1] if best else 0
    assert res.out_tokens == [int(tr2.tok[c]) for c in best] + [int(np.argmax(z[last]))]


def _v8_round():
    cfg = TINY_V8
    inp = make_inputs(cfg, seed=3)
    w = R.weights_f32(inp); f = inp.feats_f32(); P = cfg.prefix
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    rr = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1, with_verify=False)
    z, _ = R.verify_logits(w, cfg, K, V, P - 1, rr.tree, rr.draft)
    return rr.tree, z


class _NoResidual(R.Decisions):
    """Planted mistake: accept each child with probability p(c), ignoring the
    mass already rejected (no residual renormalisation)."""

    def accept(self, b, node, i, u, rejected_mass, p_child):
        return u < p_child


def _chi2_marginals(tree, z, n, dec=None):
    V = z.shape[1]
    p_root = np.exp(z[0] - L.logsumexp(z[0]))
    first = np.zeros(V)
    second = {c: np.zeros(V) for c in tree.children(0)}
    for rid in range(n):
        res = R.verify_sample(tree, z, 1.0, 0, rid, dec)
        first[res.out_tokens[0]] += 1
        if res.accept_len >= 1:
            second[res.path[0]][res.out_tokens[1]] += 1
    pvals = [stats.chisquare(first, p_root * n).pvalue]
    for c, cnt in second.items():
        if cnt.sum() > 500:
            pc = np.exp(z[c] - L.logsumexp(z[c]))
            pvals.append(stats.chisquare(cnt, pc * cnt.sum()).pvalue)
    return pvals


@pytest.mark.slow
def test_sampling_marginals_chi_square_v8():
    tree, z = _v8_round()
    assert len(tree.children(0)) == 2
    pvals = _chi2_marginals(tree, z, 30000)
    assert len(pvals) >= 2
    assert min(pvals) > 1e-3, pvals


@pytest.mark.slow
def test_sampling_chi_square_rejects_missing_residual():
    tree, z = _v8_round()
    pvals = _chi2_marginals(tree, z, 30000, _NoResidual())
    assert min(pvals) < 1e-6, pvals


def test_sampling_deterministic_in_seed_and_round():
    tree, z = _v8_round()
    a = [R.verify_sample(tree, z, 1.0, 5, rid).out_tokens for rid in range(50)]
    b = [R.verify_sample(tree, z, 1.0, 5, rid).out_tokens for rid in range(50)]
    c = [R.verify_sample(tree, z, 1.0, 6, rid).out_tokens for rid in range(50)]
    assert a == b and a != c


# ----------------------------------------------------------------------------- two-stage head
def test_two_stage_head_reduces_to_single_stage():
    rng = np.random.default_rng(9)
    V, d, r = 300, 24, 8
    cfg1 = by_name("tiny_fp32_b1").scaled(d=d, vocab=V)
    w = {"w_lm": rng.standard_normal((V, d)).astype(np.float32),
         "lr_u": rng.standard_normal((V, r)).astype(np.float32),
         "lr_v": rng.standard_normal((r, d)).astype(np.float32)}
    h = rng.standard_normal((3, d))
    _, lq1, _ = L.draft_logq(w, cfg1, h)
    cand, lq2, _ = L.draft_logq(w, cfg1.scaled(lr_rank=r, lr_cand=V), h)
    for i in range(3):   # all tokens are candidates: the same distribution
        np.testing.assert_allclose(lq2[i], lq1[i][cand[i]], rtol=1e-12, atol=1e-12)
    # exactly low-rank head: the candidates are the true top-c of the exact logits
    w2 = dict(w, w_lm=(w["lr_u"].astype(np.float64) @ w["lr_v"]).astype(np.float32))
    w2["lr_u"] = w["lr_u"]; w2["lr_v"] = w["lr_v"]
    cfg2 = cfg1.scaled(lr_rank=r, lr_cand=16)
    cand, _, _ = L.draft_logq(w2, cfg2, h)
    exact = h @ w2["w_lm"].astype(np.float64).T
    for i in range(3):
        assert set(cand[i].tolist()) == set(np.argsort(-exact[i])[:16].tolist())


# ----------------------------------------------------------------------------- inputs
def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1e-3, 3.14159, 1.0 + 2 ** -8 + 2 ** -30])
    b = bf16_bits_to_f32(bf16_bits_from_f64(x)).astype(np.float64)
    assert b[1] == 1.0                 # tie -> even (down)
    assert b[2] == 1.0 + 2 ** -6       # tie -> even (up)
    assert b[6] == 1.0 + 2 ** -7       # just above the tie -> up
    rng = np.random.default_rng(0)
    y = rng.standard_normal(100000) * 0.02
    yb = bf16_bits_to_f32(bf16_bits_from_f64(y)).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(y))) - 7)
    assert (np.abs(yb - y) <= ulp / 2 + 1e-300).all()


def test_inputs_are_deterministic():
    cfg = by_name("tiny_fp32_b1")
    a, b = make_inputs(cfg, threads=1), make_inputs(cfg, threads=4)
    for k in a.w:
        assert np.array_equal(a.w[k], b.w[k]), k
    assert np.array_equal(a.feats, b.feats) and np.array_equal(a.tokens, b.tokens)


# ----------------------------------------------------------------------------- drafter variants
def _variant_cfg(**kw):
    return by_name("tiny_fp32_b1").scaled(name="variant_pin", prefix=24, depth=3, topk=3, n_verify=8,
                             gain_std=0.1, **kw)


def test_post_norm_layer_is_scale_invariant_and_unit_rms():
    cfg = _variant_cfg(post_norm=True, rms_eps=0.0)
    w = R.weights_f32(make_inputs(cfg, seed=21))
    rng = np.random.default_rng(5)
    hid = rng.standard_normal((3, cfg.d))
    o = rng.standard_normal((3, cfg.n_q_heads * cfg.head_dim))
    s1, h1 = L.layer_tail(w, cfg, hid, o)
    s2, h2 = L.layer_tail(w, cfg, 3.7 * hid, 3.7 * o)
    np.testing.assert_allclose(s2, s1, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(s1, h1)  # the state fed to children is the head's input
    ms = np.mean((s1 / w["g_final"].astype(np.float64)) ** 2, axis=-1)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-12)
    # the pre-norm layer has neither property
    pre = _variant_cfg(rms_eps=0.0)
    p1, q1 = L.layer_tail(w, pre, hid, o)
    p2, _ = L.layer_tail(w, pre, 3.7 * hid, 3.7 * o)
    assert np.abs(p2 - p1).max() > 1e-3 and np.abs(p1 - q1).max() > 1e-3


def test_fc_norm_feature_is_scale_invariant_with_unit_rms():
    cfg = _variant_cfg(fc_norm=True, rms_eps=0.0)
    w = R.weights_f32(make_inputs(cfg, seed=22))
    f = np.random.default_rng(6).standard_normal((4, 3 * cfg.d))
    g = L.fused_feature(w, cfg, f)
    np.testing.assert_allclose(L.fused_feature(w, cfg, 0.25 * f), g, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(np.mean((g / w["g_fc"].astype(np.float64)) ** 2, axis=-1), 1.0,
                               rtol=1e-12)
    plain = L.fused_feature(w, _variant_cfg(), f)
    np.testing.assert_allclose(plain, L.fuse(f, w["w_fc"]), rtol=0, atol=0)


def test_fc_norm_round_is_invariant_to_feature_scale():
    """With the FC norm every use of g (prefix rows, root) sees a normalised
    feature, so scaling all target features leaves the whole round unchanged;
    without it the round changes."""
    for fc, expect_same in ((True, True), (False, False)):
        cfg = _variant_cfg(fc_norm=fc, post_norm=True, rms_eps=0.0)
        inp = make_inputs(cfg, seed=23)
        w = R.weights_f32(inp)
        f = inp.feats_f32().astype(np.float64)
        P = int(inp.prefix_lens[0])
        outs = []
        for a in (1.0, 2.5):
            K, V = R.prefix_kv(w, cfg, a * f[:P], inp.tokens[:P])
            rr = R.round_request(w, cfg, K, V, a * f[P - 1], inp.tokens[P - 1], P - 1,
                                 temperatures=(0.0,))
            outs.append(rr)
        same = (np.array_equal(outs[0].tree.tok, outs[1].tree.tok)
                and np.allclose(outs[0].draft.pool.logq, outs[1].draft.pool.logq, rtol=0,
                                atol=1e-9))
        assert same == expect_same, (fc, same)


@pytest.fixture(scope="module")
def variant_round():
    cfg = _variant_cfg(fc_norm=True, post_norm=True)
    inp = make_inputs(cfg, seed=24)
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    rr = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1, temperatures=(0.0,))
    return cfg, inp, w, f, P, K, V, rr


def test_variant_tree_states_equal_sequential_path_forward(variant_round):
    test_tree_states_equal_sequential_path_forward(variant_round)


# ----------------------------------------------------------------------------- per-request control
def _ctl_setup(seed=31, **kw):
    cfg = by_name("tiny_fp32_b1").scaled(name="ctl_pin", prefix=24, depth=4, topk=3, n_verify=10, **kw)
    inp = make_inputs(cfg, seed=seed)
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])

    def run(ctl=None, B=1):
        return R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1, temperatures=(0.0,),
                               ctl=ctl, B=B)
    return cfg, run


def test_control_with_full_caps_and_no_rules_is_the_plain_round():
    cfg, run = _ctl_setup()
    a = run()
    b = run(R.Control(depth_cap=[cfg.depth], topk_cap=[cfg.topk], verify_cap=[cfg.n_verify]))
    assert a.draft.pool.tok == b.draft.pool.tok and a.draft.pool.fwd == b.draft.pool.fwd
    np.testing.assert_array_equal(a.tree.tok, b.tree.tok)
    np.testing.assert_array_equal(a.tree.mask, b.tree.mask)
    assert a.verify[0.0].out_tokens == b.verify[0.0].out_tokens


def test_depth_and_branch_caps_prune_the_pool():
    cfg, run = _ctl_setup()
    full = run()
    d1 = run(R.Control(depth_cap=[1]))
    made = [i for i, t in enumerate(d1.draft.pool.tok) if t >= 0]
    assert made == list(range(cfg.topk))                  # only the root's children
    assert all(np.isneginf(d1.draft.pool.score[i]) for i in range(cfg.topk, len(d1.draft.pool.tok)))
    assert set(d1.tree.depth[1:d1.tree.n_real]) == {1} and d1.tree.n_real == 1 + cfg.topk
    k2 = run(R.Control(topk_cap=[2]))
    p = k2.draft.pool
    kids = {}
    for i, (t, par) in enumerate(zip(p.tok, p.parent)):
        if t >= 0:
            kids.setdefault(par, []).append(i)
    assert all(len(v) <= 2 for v in kids.values())
    # each node keeps its two best children of the uncapped round (same tokens, same order)
    assert [p.tok[i] for i in kids[-1]] == full.draft.pool.tok[:2]


def test_verify_cap_and_rule_keep_a_prefix_of_the_selection_order():
    cfg, run = _ctl_setup()
    full = run()
    p = full.draft.pool
    order = R.Decisions().select(0, np.asarray(p.score), np.asarray(p.depth), cfg.n_verify)
    for m in (1, 4, 7):
        t = run(R.Control(verify_cap=[m])).tree
        assert t.n_real == m + 1 and len(t.tok) == cfg.n_verify + 1
        assert sorted(t.pool_index[1:m + 1]) == sorted(int(i) for i in order[:m])
        assert (t.tok[m + 1:] == -1).all() and (t.parent[m + 1:] == -1).all()
        assert all(t.mask[u].sum() == 1 and t.mask[u, u] for u in range(m + 1, len(t.tok)))
    vu = list(np.arange(cfg.n_verify + 1, dtype=np.float64))   # one unit per node
    assert run(R.Control(tau_verify=1e9, verify_us=vu)).tree.n_real == 2
    assert run(R.Control(tau_verify=1e-30, verify_us=vu)).tree.n_real == cfg.n_verify + 1
    # a mid threshold keeps exactly the nodes whose exp(score) clears it, as a prefix
    sc = np.exp(np.asarray(p.score)[order])
    thr = float(np.sqrt(sc[3] * sc[4]))
    if sc[3] > sc[4]:
        assert run(R.Control(tau_verify=thr, verify_us=vu)).tree.n_real == 1 + 4


def test_depth_rule_stops_where_the_frontier_mass_falls_short():
    cfg, run = _ctl_setup()
    full = run()
    p = full.draft.pool
    masses = [float(np.exp([p.score[i] for i in fr]).sum()) for fr in full.draft.frontiers]
    pu = [100.0] * cfg.depth
    assert len(run(R.Control(tau_depth=1e9, pass_us=pu)).draft.frontiers[0]) == 0
    r = run(R.Control(tau_depth=1e-30, pass_us=pu))
    assert r.draft.pool.tok == p.tok
    # threshold between the masses of the frontiers of depth 1 and 2 (growth 1): pass 1 runs, pass 2 not
    if masses[0] > masses[1]:
        tau = float(np.sqrt(masses[0] * masses[1])) / 100.0
        r = run(R.Control(tau_depth=tau, pass_us=pu))
        assert r.draft.frontiers[0] == full.draft.frontiers[0] and r.draft.frontiers[1] == []
        assert max(d for d, t in zip(r.draft.pool.depth, r.draft.pool.tok) if t >= 0) == 2


def test_branch_rule_uses_the_light_and_heavy_caps():
    cfg, run = _ctl_setup()
    ctl = R.Control(light_batch=1, k_light=2, k_heavy=1)
    for B, k in ((1, 2), (2, 1)):
        p = run(ctl, B=B).draft.pool
        assert sum(1 for t in p.tok[:cfg.topk] if t >= 0) == k


def test_greedy_on_a_capped_tree_is_the_longest_matching_path():
    cfg, run = _ctl_setup()
    tr = run(R.Control(verify_cap=[6], topk_cap=[2])).tree
    rng = np.random.default_rng(9)
    z = rng.standard_normal((tr.n_real, cfg.vocab))
    for u in range(tr.n_real):
        kids = tr.children(u)
        if kids:
            z[u, tr.tok[kids[0]]] = 50.0
    res = R.verify_greedy(tr, z)
    best = max((q for q in _all_paths(tr)
                if all(tr.tok[c] == np.argmax(z[0 if i == 0 else q[i - 1]]) for i, c in enumerate(q))),
               key=len)
    assert res.path == best


# ----------------------------------------------------------------------------- sampled drafting, q-ratio verify
def _single_node_emissions(p, q, k, n, scheme, seed=5, sampled=True):
    """Emitted token of a root with k children (drawn from q by Gumbel-top-k, or
    the top-k of q), over n round ids, verified by the q-ratio or point-mass scheme."""
    V = len(p)
    out = np.empty(n, dtype=np.int64)
    zrow, erow = np.log(p), np.log(q)
    for rid in range(n):
        keys = erow + philox.gumbel(seed, rid, 0, 0, np.arange(V), stream=2) if sampled else erow
        kids = L.topk_order(keys, k)
        tok = np.concatenate([[0], kids])
        tr = R.Tree(tok, np.array([-1] + [0] * k), np.array([0] + [1] * k), np.zeros(k + 1),
                    np.zeros(k + 1), np.array([-1] + list(range(k))), np.eye(k + 1, dtype=bool))
        z = np.tile(zrow, (k + 1, 1))
        if scheme == "qratio":
            r = R.verify_qratio(tr, z, np.tile(erow, (k + 1, 1)), 1.0, seed, rid)
        else:
            r = R.verify_sample(tr, z, 1.0, seed, rid)
        out[rid] = r.out_tokens[0]
    return out


def _chi2_p(samples, probs):
    counts = np.bincount(samples, minlength=len(probs))
    return stats.chisquare(counts, len(samples) * probs).pvalue


def test_sampled_children_first_draw_follows_q():
    """Gumbel-top-k over Philox stream 2: the first draw of a node is distributed as q."""
    rng = np.random.default_rng(2)
    q = rng.dirichlet(np.ones(8))
    first = np.array([int(np.argmax(np.log(q) + philox.gumbel(7, rid, 0, 3, np.arange(8), stream=2)))
                      for rid in range(20000)])
    assert _chi2_p(first, q) > 1e-3


def test_qratio_verification_emits_the_target_distribution():
    """Exactness of recursive rejection over draws without replacement (R-17):
    the emitted token is distributed as p for any draft q (chi-square, 7 dof)."""
    rng = np.random.default_rng(4)
    p = rng.dirichlet(np.ones(8))
    q = rng.dirichlet(0.5 * np.ones(8))
    assert _chi2_p(_single_node_emissions(p, q, 3, 20000, "qratio"), p) > 1e-3


def test_qratio_on_top_k_children_is_biased_but_point_masses_are_not():
    """Planted mistake: the q-ratio scheme on deterministic top-k children (not
    draws from q) does not emit p, and the same chi-square sees it; the
    point-mass scheme of the plain round is exact for any candidate set."""
    p = np.array([0.30, 0.25, 0.15, 0.10, 0.08, 0.06, 0.04, 0.02])
    q = np.array([0.02, 0.04, 0.06, 0.08, 0.10, 0.15, 0.25, 0.30])
    assert _chi2_p(_single_node_emissions(p, q, 3, 20000, "qratio", sampled=False), p) < 1e-3
    assert _chi2_p(_single_node_emissions(p, q, 3, 20000, "point", sampled=True), p) > 1e-3


def test_sampled_round_keeps_sibling_prefixes_in_draw_order():
    cfg = by_name("tiny_fp32_b1").scaled(name="samp_pin", prefix=24, depth=4, topk=3, n_verify=7)
    inp = make_inputs(cfg, seed=33)
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    rr = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1, temperatures=(0.0, 1.0),
                         samp=(9, 2))
    p = rr.draft.pool
    kept = set(int(i) for i in rr.tree.pool_index[1:] if i >= 0)
    by_parent = {}
    for i, par in enumerate(p.parent):
        if p.tok[i] >= 0:
            by_parent.setdefault(par, []).append(i)
    for par, sib in by_parent.items():
        sc = [p.score[i] for i in sib]
        assert all(a >= b for a, b in zip(sc, sc[1:]))          # non-increasing in draw order
        mine = [i in kept for i in sib]
        assert mine == sorted(mine, reverse=True)              # kept siblings: first draws
    # the sampled children differ from the top-k ones somewhere, yet every token is a valid index
    plain = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1, with_verify=False)
    assert p.tok != plain.draft.pool.tok
    assert all(0 <= t < cfg.vocab for t in p.tok if t >= 0)


# whole sampled round at V = 8 (d = 32 so the draft and target heads differ)
_V8_ROUND = by_name("tiny_fp32_b1").scaled(name="samp_round_v8", d=32, n_q_heads=2, n_kv_heads=2, head_dim=16,
                              ffn=32, vocab=8, prefix=6, depth=3, topk=2, n_verify=6, lm_std=0.3,
                              sampled_draft=True)


class _OwnDrawScore(R.Decisions):
    """Planted mistake: a draw's score uses its own log q (the running minimum
    including the draw), so whether a draw is kept depends on the draw itself."""

    def draw_score(self, cap, logq_draw):
        return min(cap, logq_draw)


def _sampled_round_marginals(n, dec=None):
    """Emitted tokens of the whole sampled round (draft + q-ratio verification)
    over n round ids, and the target distributions at the root and at the
    depth-1 node of each token."""
    cfg = _V8_ROUND
    inp = make_inputs(cfg, seed=3)
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    acc, out = np.zeros(n, dtype=np.int64), np.full((n, cfg.depth + 1), -1)
    for rid in range(n):
        rr = R.round_request(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1,
                             temperatures=(1.0,), seed=17, round_id=rid, samp=(11, rid), dec=dec)
        r = rr.verify[1.0]
        acc[rid] = r.accept_len
        out[rid, :len(r.out_tokens)] = r.out_tokens
    s_root, h_root = R.root_forward(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1)
    z1 = {}
    for c in range(cfg.vocab):   # a depth-1 node's target logits depend on its token only
        pool = R.Pool()
        pool.add(c, -1, 0.0, 1, 0.0)
        tr = R.build_tree([c], [-1], np.array([0.0]), [1], int(inp.tokens[P - 1]), P - 1, 1)
        z, _ = R.verify_logits(w, cfg, K, V, P - 1, tr, R.DraftResult(pool, s_root, h_root, {}, {},
                                                                      {}, []))
        z1[c] = z[1]
    soft = lambda v: np.exp(v - L.logsumexp(v))
    pv = [_chi2_p(out[:, 0], soft(z[0]))]
    for c in range(cfg.vocab):
        sel = (acc >= 1) & (out[:, 0] == c)
        if sel.sum() > 1000:
            pv.append(_chi2_p(out[sel, 1], soft(z1[c])))
    return pv


@pytest.mark.slow
def test_sampled_round_second_token_follows_the_target():
    """Whole sampled round (R-17): the first emitted token follows p at the root,
    and given the accepted depth-1 child c the second follows p at c, because a
    draw's score never looks at the draw itself; the planted own-draw score,
    which lets the draws decide how many siblings are verified, is rejected."""
    pv = _sampled_round_marginals(6000)
    assert len(pv) >= 2 and min(pv) > 1e-3, pv
    bad = _sampled_round_marginals(6000, _OwnDrawScore())
    assert min(bad) < 1e-4, bad
