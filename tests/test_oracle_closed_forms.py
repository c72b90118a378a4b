"""Closed-form and library pins of the oracle functions that the brute-force
pins leave open: each case is one where the mathematics fixes the answer, so a
plausible slip in the oracle (a dropped residual, the FFN fed the wrong vector,
a swapped gain, halves in the wrong order, a mis-normalised log-sum-exp, a
rescoring on the wrong rows) fails here.

* the pre-norm layer tail (the decoder layer of "EAGLE-3 精读" §1 paragraph 2):
  with the output projections zeroed the state is the input; with the FFN's
  down projection zeroed it is the attention residual; with single-coordinate
  FFN weights every output coordinate follows by hand from torch's RMSNorm and
  SiLU;
* the decoder input [rms(E[y]); rms(hid)]: one-hot embedding rows and constant
  hidden rows have RMS values known in closed form;
* logsumexp against scipy.special.logsumexp;
* the two-stage head inside a whole draft round (EAGLE-4 blog, 关于 Efficient
  LM Head: low-rank recall, exact rerank): with every token a candidate the
  round's pool equals the single-stage round's pool;
* Philox4x64-10 against the published known-answer vectors.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp as sp_logsumexp

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs
from oracle import layers as L
from oracle import philox
from oracle import round as R

HERE = os.path.dirname(os.path.abspath(__file__))


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


def _rms(v, g, eps):
    """Reference RMSNorm: torch's own routine (pinned separately)."""
    return F.rms_norm(_t(v), (v.shape[-1],), _t(g), eps=eps).numpy()


def _layer_setup(seed, d=16, ffn=12, heads=2, dh=8, eps=1e-5):
    cfg = by_name("tiny_fp32_b1").scaled(d=d, ffn=ffn, n_q_heads=heads, n_kv_heads=heads, head_dim=dh,
                            rms_eps=eps)
    rng = np.random.default_rng(seed)
    od = heads * dh
    w = {"w_o": rng.standard_normal((d, od)) * 0.3,
         "w_gate": rng.standard_normal((ffn, d)) * 0.3,
         "w_up": rng.standard_normal((ffn, d)) * 0.3,
         "w_down": rng.standard_normal((d, ffn)) * 0.3,
         # distinct, non-unit gains so that a swapped or dropped gain shows
         "g_post": 1.0 + 0.5 * rng.standard_normal(d),
         "g_final": 1.0 + 0.5 * rng.standard_normal(d)}
    hid = rng.standard_normal((3, d)) * 2.0
    o = rng.standard_normal((3, od))
    return cfg, w, hid, o


# ----------------------------------------------------------------------------- layer tail
def test_layer_tail_with_zero_projections_passes_hid_through():
    cfg, w, hid, o = _layer_setup(1)
    w["w_o"][:] = 0.0
    w["w_down"][:] = 0.0
    s, h = L.layer_tail(w, cfg, hid, o)
    np.testing.assert_array_equal(s, hid)                       # s = hid
    np.testing.assert_allclose(h, _rms(hid, w["g_final"], cfg.rms_eps), rtol=1e-12, atol=1e-12)


def test_layer_tail_with_zero_down_projection_is_the_attention_residual():
    cfg, w, hid, o = _layer_setup(2)
    w["w_down"][:] = 0.0
    s, h = L.layer_tail(w, cfg, hid, o)
    r = hid + F.linear(_t(o), _t(w["w_o"])).numpy()
    np.testing.assert_allclose(s, r, rtol=1e-12, atol=1e-12)   # s = hid + W_o o
    np.testing.assert_allclose(h, _rms(r, w["g_final"], cfg.rms_eps), rtol=1e-12, atol=1e-12)


def test_layer_tail_single_coordinate_ffn_by_hand():
    """W_gate, W_up and W_down pick single coordinates: FFN channel j reads
    gate input a_j and up input b_j of z = rms(r; g_post) and writes output
    coordinate i_j, so s_i = r_i + sum_j c_j silu(al_j z[a_j]) be_j z[b_j]."""
    cfg, w, hid, o = _layer_setup(3)
    d, ffn = cfg.d, cfg.ffn
    w["w_gate"][:] = 0.0
    w["w_up"][:] = 0.0
    w["w_down"][:] = 0.0
    chans = [(0, 3, 7, 5, 1.3, -0.7, 0.9), (1, 11, 2, 5, -0.4, 1.1, -1.7), (4, 9, 9, 14, 2.0, 0.6, 0.5)]
    for j, a, b, i, al, be, c in chans:
        w["w_gate"][j, a] = al
        w["w_up"][j, b] = be
        w["w_down"][i, j] = c
    s, h = L.layer_tail(w, cfg, hid, o)
    r = hid + F.linear(_t(o), _t(w["w_o"])).numpy()
    z = _rms(r, w["g_post"], cfg.rms_eps)
    want = r.copy()
    for j, a, b, i, al, be, c in chans:
        want[:, i] += c * F.silu(_t(al * z[:, a])).numpy() * (be * z[:, b])
    np.testing.assert_allclose(s, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h, _rms(want, w["g_final"], cfg.rms_eps), rtol=1e-12, atol=1e-12)
    # untouched coordinates carry the attention residual only
    rest = [x for x in range(d) if x not in {ch[3] for ch in chans}]
    np.testing.assert_allclose(s[:, rest], r[:, rest], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- decoder input
def test_decoder_input_halves_and_gains_in_closed_form():
    """Embedding rows c_y e_{y} (one-hot) have RMS |c_y| / sqrt(d), so with eps = 0
    rms(E[y]; g_emb) = sign(c_y) sqrt(d) g_emb[y] e_y; a constant hidden row kappa 1
    has RMS |kappa|, so rms(hid; g_hid) = sign(kappa) g_hid.  The first half is the
    embedding's, the second the hidden state's."""
    d, V = 8, 8
    cfg = by_name("tiny_fp32_b1").scaled(d=d, vocab=V, rms_eps=0.0)
    rng = np.random.default_rng(4)
    c = np.array([2.0, -0.5, 3.0, 1.0, -4.0, 0.25, 7.0, -1.5])
    w = {"embed": np.diag(c), "g_emb": 1.0 + rng.standard_normal(d), "g_hid": 1.0 + rng.standard_normal(d)}
    toks = np.array([3, 0, 6, 1])
    kappa = np.array([0.7, -2.0, 5.0, 1e-3])
    hid = kappa[:, None] * np.ones((4, d))
    x = L.decoder_input(w, cfg, toks, hid)
    assert x.shape == (4, 2 * d)
    for r, (y, kp) in enumerate(zip(toks, kappa)):
        e = np.zeros(d)
        e[y] = np.sign(c[y]) * np.sqrt(d) * w["g_emb"][y]
        np.testing.assert_allclose(x[r, :d], e, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(x[r, d:], np.sign(kp) * w["g_hid"], rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- logsumexp
def test_logsumexp_matches_scipy():
    rng = np.random.default_rng(5)
    for shape, scale, shift in (((7, 300), 1.0, 0.0), ((3, 5), 40.0, 1e4), ((2, 128256), 3.0, -7e3),
                                ((1, 1), 1.0, 0.0)):
        v = rng.standard_normal(shape) * scale + shift
        np.testing.assert_allclose(L.logsumexp(v), sp_logsumexp(v, axis=-1), rtol=1e-13, atol=1e-11)
    v = rng.standard_normal((4, 9))
    v[:, [1, 4]] = -np.inf          # excluded entries contribute nothing
    np.testing.assert_allclose(L.logsumexp(v), sp_logsumexp(v, axis=-1), rtol=1e-13)
    np.testing.assert_allclose(L.logsumexp(v.T, axis=0), sp_logsumexp(v.T, axis=0), rtol=1e-13)


def test_draft_logq_single_stage_is_a_log_softmax():
    cfg = by_name("tiny_fp32_b1").scaled(d=24, vocab=50)
    rng = np.random.default_rng(6)
    w = {"w_lm": rng.standard_normal((50, 24)).astype(np.float32)}
    h = rng.standard_normal((3, 24))
    tok, lq, lr = L.draft_logq(w, cfg, h)
    ref = torch.log_softmax(F.linear(_t(h), _t(w["w_lm"])), dim=-1).numpy()
    np.testing.assert_allclose(lq, ref, rtol=1e-12, atol=1e-12)
    assert lr is None and (tok == np.arange(50)).all()


# ----------------------------------------------------------------------------- two-stage round
def test_two_stage_round_with_every_token_a_candidate_is_the_single_stage_round():
    """The rescoring inside draft_request (exact logits on the candidates, log q
    over the candidates, children from them) must give the single-stage pool
    when the candidate set is the whole vocabulary."""
    V = 96
    cfg2 = by_name("tiny_fp32_b1").scaled(name="two_stage_pin", d=32, n_q_heads=2, n_kv_heads=2, head_dim=16,
                             ffn=48, vocab=V, prefix=20, depth=4, topk=3, n_verify=10,
                             lr_rank=8, lr_cand=V, lm_std=0.3)
    cfg1 = cfg2.scaled(lr_rank=0, lr_cand=0)
    inp = make_inputs(cfg2, seed=8)
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, Vc = R.prefix_kv(w, cfg2, f[:P], inp.tokens[:P])
    d2 = R.draft_request(w, cfg2, K, Vc, f[P - 1], inp.tokens[P - 1], P - 1, R.Decisions())
    d1 = R.draft_request(w, cfg1, K, Vc, f[P - 1], inp.tokens[P - 1], P - 1, R.Decisions())
    for name in ("tok", "parent", "depth", "fwd"):
        assert getattr(d2.pool, name) == getattr(d1.pool, name), name
    np.testing.assert_allclose(d2.pool.logq, d1.pool.logq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(d2.pool.score, d1.pool.score, rtol=0, atol=1e-12)
    # and with fewer candidates the round differs (the test can see the head)
    d3 = R.draft_request(w, cfg2.scaled(lr_cand=8), K, Vc, f[P - 1], inp.tokens[P - 1], P - 1,
                         R.Decisions())
    assert not np.allclose(d3.pool.logq, d1.pool.logq)


# ----------------------------------------------------------------------------- Philox
def _kat_rows():
    rows = []
    with open(os.path.join(HERE, "golden", "philox4x64_10_kat.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    return rows


def test_philox_known_answer_vectors():
    rows = _kat_rows()
    assert len(rows) == 3
    for r in rows:
        ctr, key, want = r[:4], r[4:6], tuple(r[6:])
        assert philox.philox4x64_scalar(ctr, key) == want
        vec = philox.philox4x64(*[np.uint64(c) for c in ctr], key[0], key[1])
        assert tuple(int(v) for v in vec) == want
