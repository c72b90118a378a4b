"""Parity harness: run a round on the GPU through the C ABI and compare it with
the CPU oracle, element by element, in free-running and conditioned modes.

Tolerances (the round's contract): logits, log q and log-sum-exp within 1e-4
(fp32 storage) or 0.05 (bf16); cumulative scores within that times the depth.
A decision (a top-k, the frontier, the kept set, an argmax, an acceptance test)
whose oracle margin is under 1e-3 (fp32) or 0.05 (bf16) is a near-tie: if the
GPU chose differently there, the choice is counted, not failed, and in
conditioned mode the oracle adopts the GPU's choice and carries on.  Every
other decision, every index and every token must agree exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from oracle import layers as L
from oracle import round as R

TOL = {"fp32": dict(logit=1e-4, tie=1e-3), "bf16": dict(logit=0.05, tie=0.05)}


@dataclass
class GpuRound:
    """Host copies of one GPU round's outputs (request-major arrays)."""
    tree: dict
    pool: dict
    verify: dict = field(default_factory=dict)   # T -> dict(accept_len, path, out_tokens, stats)


def gpu_round(eng, temps=(0.0,), seed=0, round_id=0) -> GpuRound:
    eng.draft_round(with_pool=True)
    return gpu_outputs(eng, temps, lambda T: eng.verify(T, seed, round_id))


class Report:
    def __init__(self):
        self.near_ties = []
        self.failures = []
        self.max_err = {}

    def err(self, name, value):
        self.max_err[name] = max(self.max_err.get(name, 0.0), float(value))

    def __repr__(self):
        return f"Report(near_ties={len(self.near_ties)}, failures={self.failures[:5]}, max_err={self.max_err})"


def _valid_choice(values, chosen, tol):
    """Is the ordered list `chosen` a correct top-len(chosen) of `values` up to tol?"""
    chosen = list(chosen)
    if len(set(chosen)) != len(chosen):
        return False
    v = np.asarray(values, dtype=np.float64)
    rest = np.ones(len(v), dtype=bool)
    rest[chosen] = False
    worst = min(v[c] for c in chosen)
    if rest.any() and v[rest].max() > worst + tol:
        return False
    return all(v[chosen[i]] >= v[chosen[i + 1]] - tol for i in range(len(chosen) - 1))


class Follow(R.Decisions):
    """Oracle decisions conditioned on the GPU's choices at near-ties."""

    def __init__(self, cfg, gpu: GpuRound, rep: Report, tol_tie, T=None):
        self.cfg, self.g, self.rep, self.tol = cfg, gpu, rep, tol_tie
        self.T = T

    def _adopt(self, what, own, gpu_choice, values, tol):
        own = [int(x) for x in own]
        gpu_choice = [int(x) for x in gpu_choice]
        if own == gpu_choice:
            return own
        if _valid_choice(values, gpu_choice, tol):
            self.rep.near_ties.append(what)
            return gpu_choice
        self.rep.failures.append(what)
        return own

    def candidates(self, b, depth, rank, lowrank_row, c):
        """Two-stage head: the GPU's candidate set of this node, if it is a valid top-c."""
        own = super().candidates(b, depth, rank, lowrank_row, c)
        slot = 0 if depth == 0 else 1 + (depth - 1) * self.cfg.topk + rank
        gpu = self.g.pool["cand"][b, slot]
        return np.asarray(self._adopt(("candidates", b, depth, rank), own, gpu, lowrank_row, self.tol))

    def children(self, b, depth, rank, cand_tokens, logq_row, k):
        own = super().children(b, depth, rank, cand_tokens, logq_row, k)
        base = 0 if depth == 0 else k + (depth - 1) * k * k + rank * k
        gtok = [int(t) for t in self.g.pool["tok"][b, base:base + k] if t >= 0]  # created ones
        pos = {int(t): i for i, t in enumerate(np.asarray(cand_tokens))}
        if any(t not in pos for t in gtok):
            self.rep.failures.append(("children-token", b, depth, rank))
            return own
        n = len(gtok)
        got = self._adopt(("children", b, depth, rank), [int(x) for x in own[:n]],
                          [pos[t] for t in gtok], logq_row, self.tol)
        return list(got) + [int(x) for x in own[n:] if int(x) not in got][:k - n]

    def frontier(self, b, depth, scores, k):
        own = super().frontier(b, depth, scores, k)
        base = k + (depth - 2) * k * k
        fwd = self.g.pool["fwd"][b, base:base + k * k]
        chosen = [i for _, i in sorted((int(f), i) for i, f in enumerate(fwd) if f >= 0)]
        if not chosen:  # the GPU expanded none of them (the request stopped drafting)
            return own
        own_real = [int(i) for i in own if np.isfinite(scores[i])]
        got = self._adopt(("frontier", b, depth), own_real, chosen, scores, self.tol * depth)
        return got + [int(i) for i in own if not np.isfinite(scores[i])]

    def keep_drafting(self, b, t, mass, threshold):
        own = super().keep_drafting(b, t, mass, threshold)
        k = self.cfg.topk
        lo, hi = (0, k) if t == 1 else (k + (t - 2) * k * k, k + (t - 1) * k * k)
        gpu = bool((self.g.pool["fwd"][b, lo:hi] >= 0).any())
        if gpu == own:
            return own
        if abs(np.log(max(mass, 1e-300)) - np.log(max(threshold, 1e-300))) < self.tol * t:
            self.rep.near_ties.append(("keep_drafting", b, t))
            return gpu
        self.rep.failures.append(("keep_drafting", b, t, float(mass), float(threshold)))
        return own

    def verify_count(self, b, gains, costs, m_cap):
        own = super().verify_count(b, gains, costs, m_cap)
        gpu = int((self.g.tree["tokens"][b, 1:] >= 0).sum())
        if gpu == own:
            return own
        i = min(own, gpu)  # the comparison where the two part
        tol = self.tol * self.cfg.depth
        if i < len(gains) and abs(np.log(max(gains[i], 1e-300)) - np.log(max(costs[i], 1e-300))) < tol:
            self.rep.near_ties.append(("verify_count", b))
            return gpu
        self.rep.failures.append(("verify_count", b, own, gpu))
        return own

    def select(self, b, scores, depths, m):
        own = [int(x) for x in super().select(b, scores, depths, m)]
        rank = {p: r for r, p in enumerate(own)}
        own_tree_order = sorted(own, key=lambda p: (depths[p], rank[p]))
        gsel = [int(p) for p in self.g.tree["pool_index"][b, 1:] if p >= 0]
        if gsel == own_tree_order:
            return own
        tol = self.tol * self.cfg.depth
        # the GPU's kept set must be a top-M up to tol, and inside each depth its
        # order (selection rank) must be by score up to tol
        set_ok = _valid_choice(scores, sorted(gsel, key=lambda p: -scores[p]), tol)
        order_ok = all(scores[p] >= scores[q] - tol for p, q in zip(gsel, gsel[1:])
                       if depths[p] == depths[q])
        if set_ok and order_ok and len(set(gsel)) == len(gsel):
            self.rep.near_ties.append(("select", b))
            return gsel
        self.rep.failures.append(("select", b))
        return own

    def greedy(self, b, node, z_row):
        own = super().greedy(b, node, z_row)
        g = int(self.g.verify[self.T]["stats"]["z_argmax"][b, node])
        return self._adopt(("greedy", b, node), [own], [g], z_row, self.tol)[0]

    def accept(self, b, node, i, u, rejected_mass, p_child):
        own = super().accept(b, node, i, u, rejected_mass, p_child)
        v = self.g.verify[self.T]
        # the GPU's choice at (node, i): accepted iff its path leaves `node` through child i
        path = [0] + [int(x) for x in v["path"][b] if x >= 0]
        gpu_acc = None
        if node in path:
            j = path.index(node)
            if j + 1 < len(path):
                nxt = path[j + 1]
                kids = [c for c in range(len(self.g.tree["parent"][b])) if self.g.tree["parent"][b, c] == node]
                gpu_acc = (kids.index(nxt) == i) if nxt in kids else None
            else:
                gpu_acc = False
        if gpu_acc is None or gpu_acc == own:
            return own
        margin = abs(u * (1.0 - rejected_mass) - p_child)
        if margin < max(p_child, 1e-30) * self.tol + 1e-7:
            self.rep.near_ties.append(("accept", b, node, i))
            return gpu_acc
        self.rep.failures.append(("accept", b, node, i, float(margin)))
        return own

    def accept_q(self, b, node, i, u, q_child, p_child):
        own = super().accept_q(b, node, i, u, q_child, p_child)
        gpu_acc = self._gpu_acceptance(b, node, i)
        if gpu_acc is None or gpu_acc == own:
            return own
        margin = abs(u * q_child - p_child)
        if margin < max(p_child, 1e-30) * self.tol + 1e-7:
            self.rep.near_ties.append(("accept_q", b, node, i))
            return gpu_acc
        self.rep.failures.append(("accept_q", b, node, i, float(margin)))
        return own

    def _gpu_acceptance(self, b, node, i):
        """The GPU's choice at (node, i): accepted iff its path leaves `node` through
        its i-th draw (children in pool order); None where the GPU never got there."""
        v = self.g.verify[self.T]
        path = [0] + [int(x) for x in v["path"][b] if x >= 0]
        if node not in path:
            return None
        j = path.index(node)
        if j + 1 >= len(path):
            return False
        nxt = path[j + 1]
        par = self.g.tree["parent"][b]
        kids = sorted((c for c in range(len(par)) if par[c] == node),
                      key=lambda c: int(self.g.tree["pool_index"][b, c]))
        return (kids.index(nxt) == i) if nxt in kids else None

    def bonus(self, b, node, scores):
        own = super().bonus(b, node, scores)
        v = self.g.verify[self.T]
        n = int(v["accept_len"][b])
        g = int(v["out_tokens"][b, n])
        return self._adopt(("bonus", b, node), [own], [g], scores, self.tol)[0]


def gpu_outputs(eng, temps, verify_fn) -> GpuRound:
    """Host copies of the round just drafted on `eng` (its tree and pool buffers)
    and of verify_fn(T) -> (accept_len, path, out_tokens) for each T."""
    import torch
    torch.cuda.synchronize()
    eng.check()
    tree = {k: getattr(eng.tree, k).cpu().numpy() for k in
            ("tokens", "parent", "depth", "pos", "pool_index", "score", "mask")}
    pool = {k: getattr(eng.pool, k).cpu().numpy() for k in ("tok", "parent", "depth", "fwd", "score", "logq")}
    if eng.pool.cand is not None:
        pool["cand"] = eng.pool.cand.cpu().numpy()
    out = GpuRound(tree, pool)
    for T in temps:
        a, p, o = verify_fn(T)
        torch.cuda.synchronize()
        eng.check()
        out.verify[T] = dict(accept_len=a.cpu().numpy().copy(), path=p.cpu().numpy().copy(),
                             out_tokens=o.cpu().numpy().copy(),
                             stats={k: v.cpu().numpy().copy() for k, v in eng.stats_t.items()})
    return out


def compare(cfg, inp, gpu: GpuRound, temps, seed=0, round_id=0, prefix_kv=None, requests=None,
            ctl=None, samp=None):
    """Conditioned oracle run and element-wise comparison.  Returns a Report."""
    rep = Report()
    w = R.weights_f32(inp)
    feats = inp.feats_f32()
    for b in (requests if requests is not None else range(cfg.batch)):
        lo, hi = int(inp.cu_rows[b]), int(inp.cu_rows[b + 1])
        if prefix_kv is None:
            K, V = R.prefix_kv(w, cfg, feats[lo:hi], inp.tokens[lo:hi])
        else:
            K, V = prefix_kv(b)
        compare_request(cfg, w, K, V, feats[hi - 1], inp.tokens[hi - 1], hi - lo, gpu, b, temps,
                        rep, seed, round_id, ctl, samp)
    return rep


def compare_request(cfg, w, K, V, feat_root, tok_root, P, gpu: GpuRound, b, temps, rep: Report,
                    seed=0, round_id=0, ctl=None, samp=None, B=None):
    """Request b of a GPU round against the oracle's round from its committed
    rows: K, V the prefix cache of rows 0..P-1 (the root, row P-1, included),
    feat_root / tok_root the root row.  Adds failures, errors and near-ties to rep."""
    tol = TOL[cfg.dtype]
    B = cfg.batch if B is None else B
    dec = Follow(cfg, gpu, rep, tol["tie"])
    dr = R.draft_request(w, cfg, K, V, feat_root, tok_root, P - 1, dec, b, ctl, B, samp)
    pool = dr.pool
    n = len(pool.tok)
    # pool: tokens / parents / depth exact; log q and scores within tolerance
    for name, mine in (("tok", pool.tok), ("parent", pool.parent), ("depth", pool.depth)):
        if not np.array_equal(np.asarray(mine), gpu.pool[name][b, :n]):
            rep.failures.append(("pool-" + name, b))
    made = np.asarray(pool.tok) >= 0  # created nodes (the rest hold -inf)
    if not (np.isneginf(gpu.pool["score"][b, :n][~made]).all()
            and np.isneginf(gpu.pool["logq"][b, :n][~made]).all()):
        rep.failures.append(("pool-uncreated", b))
    if made.any():
        rep.err("logq", np.max(np.abs(np.asarray(pool.logq)[made] - gpu.pool["logq"][b, :n][made])))
        dsc = (np.abs(np.asarray(pool.score)[made] - gpu.pool["score"][b, :n][made])
               / np.maximum(1, np.asarray(pool.depth)[made]))
        rep.err("score/depth", np.max(dsc))
    tree = R.build_tree(pool.tok, pool.parent, pool.score, pool.depth, tok_root, P - 1,
                        cfg.n_verify, dec, b, ctl)
    for name, mine in (("tokens", tree.tok), ("parent", tree.parent), ("depth", tree.depth),
                       ("pos", tree.pos), ("pool_index", tree.pool_index)):
        if not np.array_equal(np.asarray(mine), gpu.tree[name][b]):
            rep.failures.append(("tree-" + name, b))
    mask_bits = np.zeros_like(tree.mask)
    words = gpu.tree["mask"][b]
    for i in range(tree.mask.shape[0]):
        for j in range(tree.mask.shape[1]):
            mask_bits[i, j] = (int(words[i, j >> 5]) >> (j & 31)) & 1
    if not np.array_equal(mask_bits, tree.mask):
        rep.failures.append(("tree-mask", b))
    if not temps:
        return rep
    z, hv = R.verify_logits(w, cfg, K, V, P - 1, tree, dr)
    for T in temps:
        st = gpu.verify[T]["stats"]
        nr = z.shape[0]  # the root and the kept nodes (padding slots are not verified)
        rep.err("z_max", np.max(np.abs(z.max(axis=1) - st["z_max"][b][:nr])))
        zt = z / (T if T else 1.0)
        rep.err("lse", np.max(np.abs(L.logsumexp(zt) - st["lse"][b][:nr])))
        dec.T = T
        if T == 0:
            res = R.verify_greedy(tree, z, dec, b)
        elif samp is None:
            res = R.verify_sample(tree, z, T, seed, round_id, dec, b)
        else:
            res = R.verify_qratio(tree, z, L.linear(hv, w["w_lm"]), T, seed, round_id, dec, b)
        v = gpu.verify[T]
        if int(v["accept_len"][b]) != res.accept_len:
            rep.failures.append(("accept_len", T, b))
        gp = [int(x) for x in v["path"][b] if x >= 0]
        if gp != res.path:
            rep.failures.append(("path", T, b))
        go = [int(x) for x in v["out_tokens"][b] if x >= 0]
        if go != res.out_tokens:
            rep.failures.append(("out_tokens", T, b))
    return rep
