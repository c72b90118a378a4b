"""The CUDA sampling walk keeps the target distribution: a chi-square test of
its output marginals over many round ids.

"EAGLE-3 精读" §5 (正确性、复现与风险): speculative sampling keeps the target's
distribution only when the residual correction is done.  At a vocabulary of
8 the marginals are checked directly against the target distribution p (from
the oracle's float64 target logits): the first emitted token must follow
p_root, and, given that the depth-1 child c was accepted, the second emitted
token must follow p_c.  Each round id is one CUDA-graph replay of the whole
step (draft round + verification) with that round id, so every replay draws
fresh Philox numbers:
  * point-mass verification of the deterministic top-k tree (mode 1);
  * the sampled draft (children drawn from q by Gumbel-top-k, whose noise also
    follows the replay's round id) with q-ratio verification (mode 2).
"""
import numpy as np
import pytest
from scipy import stats

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs
from oracle import layers as L
from oracle import round as R

V8 = by_name("tiny_fp32_b1").scaled(name="chi2_v8_gpu", d=32, n_q_heads=2, n_kv_heads=2, head_dim=16, ffn=32,
                       vocab=8, prefix=6, depth=3, topk=2, n_verify=6, lm_std=0.3,
                       temperatures=(1.0,))
N = 24000


def _target_rows(cfg, inp):
    """Oracle target logits at the root and at a depth-1 node of each token."""
    w = R.weights_f32(inp)
    f = inp.feats_f32()
    P = int(inp.prefix_lens[0])
    K, V = R.prefix_kv(w, cfg, f[:P], inp.tokens[:P])
    s_root, h_root = R.root_forward(w, cfg, K, V, f[P - 1], inp.tokens[P - 1], P - 1)
    z1 = {}
    for c in range(cfg.vocab):
        pool = R.Pool()
        pool.add(c, -1, 0.0, 1, 0.0)
        tree = R.build_tree([c], [-1], np.array([0.0]), [1], int(inp.tokens[P - 1]), P - 1, 1)
        dr = R.DraftResult(pool, s_root, h_root, {}, {}, {}, [])
        z, _ = R.verify_logits(w, cfg, K, V, P - 1, tree, dr)
        z1[c] = z[1]
    return z[0], z1


def _softmax(z):
    return np.exp(z - L.logsumexp(z))


def _replays(cfg, seed):
    import torch
    from eagle_draft_tree_02_b300.runner import Engine
    inp = make_inputs(cfg, seed=seed)
    eng = Engine(inp)
    eng.prefill()
    D = cfg.depth
    s = torch.cuda.Stream()
    acc = torch.empty(N, dtype=torch.int32, device="cuda")
    out = torch.empty((N, D + 1), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        if cfg.sampled_draft:
            eng.draft_noise(11, 0)
        eng.draft_round(with_pool=False)
        eng.verify(1.0, seed=17, round_id=0, with_stats=False)
        eng.capture(temperature=1.0, seed=17)
        for rid in range(N):
            eng.replay(rid)
            acc[rid] = eng.accept_len[0]
            out[rid].copy_(eng.out_tokens[0])
        torch.cuda.current_stream().synchronize()
        eng.check()
    eng.close()
    return inp, acc.cpu().numpy(), out.cpu().numpy()


def _chi2(counts, p):
    keep = p * counts.sum() >= 5          # cells too rare for the test are pooled
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(p[keep], p[~keep].sum()) * counts.sum()
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    return stats.chisquare(obs, exp).pvalue


@pytest.mark.gpu
@pytest.mark.parametrize("sampled", [False, True], ids=["point_mass", "q_ratio"])
def test_gpu_sampling_marginals_chi_square(cuda, lib_built, sampled):
    cfg = V8.scaled(sampled_draft=sampled)
    inp, acc, out = _replays(cfg, seed=3)
    z0, z1 = _target_rows(cfg, inp)
    first = np.bincount(out[:, 0], minlength=cfg.vocab)
    pvals = [_chi2(first, _softmax(z0))]
    tested = 0
    for c in range(cfg.vocab):
        sel = (acc >= 1) & (out[:, 0] == c)
        if sel.sum() > 500:
            second = np.bincount(out[sel, 1], minlength=cfg.vocab)
            pvals.append(_chi2(second, _softmax(z1[c])))
            tested += 1
    print("sampled" if sampled else "point-mass", "accept mean", acc.mean(), "p-values", pvals)
    assert tested >= 1 and (acc >= 1).mean() > 0.2
    assert min(pvals) > 1e-3, pvals
    # the draws differ between replays (fresh round ids)
    assert len(set(map(tuple, out[:200].tolist()))) > 5
