"""One EAGLE-3 draft-and-verify round, plain and slow, in float64 (oracle).

Steps, in the pages' order:

1. prefix rows: fused feature g_i and the token emitted after position i give
   the decoder input of row i; its K/V go to the draft cache ("EAGLE-3 精读"
   §1 paragraph 2).  The newest row is the root of the round's tree (R-2).
2. draft passes ("each added tree depth still costs one more sequential drafter
   round", scholarfeed EAGLE-3 quotes): pass 0 runs the root; pass t runs the
   frontier nodes of depth t with their parent's own state as hidden input
   ("EAGLE-3 精读" §2, Training-Time Test: the draft is fed its own
   trajectory).  Tree nodes attend to the prefix plus their ancestors-or-self
   (the tree mask; "EAGLE-3 精读" §2 and §5 — rollout nodes never see what is
   not on their path).
3. children: per expanded node the k most likely draft tokens; a node's
   confidence is the product of draft probabilities along its path (EAGLE-4
   blog, 几条技术路线正在收敛, second trend), kept as a sum of log q.
4. EAGLE-2 confidence dynamic tree ("EAGLE-3 精读" 核心变化 and §2 last
   paragraph): R-7 — depth 1 is the root's k children; each deeper level
   expands the k best-scoring nodes of the level above (k*k candidates); the
   tree kept for verification is the global top-M of all created nodes.
5. strict verification ("EAGLE-3 精读" §5 正确性、复现与风险): greedy keeps
   the target's greedy sequence; sampling keeps the target distribution when
   the residual correction is done.  The target here is a synthetic head
   W_t = W_lm + 0.3 G applied to a tree-masked decoder pass over the kept
   nodes (R-8).

Orderings (R-7): children by (log q desc, token asc); frontier by (score desc,
creation id asc); kept set by (score desc, depth asc, creation id asc); the
creation id is the pool index (depth-major, then parent's frontier rank, then
child rank).  Output tree order: root, then depth asc, then selection rank.

Sampling (R-9): the tree's children are deterministic top-k picks, so each is a
point-mass proposal: child c_i is accepted iff U (1 - R) < p(c_i), with R the
target mass of the children already rejected at that node; if none is accepted
(or the node is a leaf) the bonus token is the Gumbel-argmax of z/T over the
tokens that are not children of the node, an exact draw from the residual.

Per-request control (R-16; EAGLE-4 blog, EAGLE-Harness paragraph, and
几条技术路线正在收敛, second trend): a request b may carry caps -- depth D_b,
branch count k_b, verify count M_b -- and three cost-aware rules, each of the
form "expected extra accepted tokens / extra time >= threshold":
  * another draft layer (pass t+1) runs only while the confidence mass of the
    next frontier, sum of exp(score), is at least tau_depth * growth**(t+1) *
    pass_us[t+1] (a threshold that rises with depth);
  * the kept set is the longest prefix of the score order whose i-th node has
    exp(score_i) >= tau_verify * (verify_us[i] - verify_us[i-1]) (at least one
    node);
  * a node expands at most k_light children when B <= light_batch, else
    k_heavy.
A node that a cap or rule leaves out is not created: its pool slot holds token
-1, parent -1, score and log q -inf.  Tree slots past the kept count hold
token -1, parent -1, depth 0, score -inf and only their own mask bit.

Sampled drafting with q-ratio verification (R-17; "EAGLE-3 精读" §5: the
draft's sampling verification keeps the target distribution with the residual
correction, which with the min(1, p/q) rule needs children drawn from q): a
node's k children are drawn from q without replacement by Gumbel-top-k
(Philox stream 2 at the node's slot), in draw order.  The i-th draw's score
is its parent's plus min(log max q, log q of draws 1..i-1): it never depends
on the draw itself, only on what was drawn before it, and it is
non-increasing in draw order.  So a kept sibling set is always the first
draws, and whether the i-th draw is kept is decided without looking at it --
a stopping rule, under which recursive rejection over the kept draws keeps
the target distribution (a score that used the draw's own log q made the
number of verified siblings depend on the draws and biased the emitted
tokens).  Verification walks the draws:
the i-th is accepted when U q_i(c) < p_i(c); on rejection p_{i+1} =
norm(max(0, p_i - q_i)) and q_{i+1} = q_i without c; with no acceptance the
bonus is the Gumbel-argmax of log p over its support (stream 1).

Every decision goes through a ``Decisions`` object.  The plain class takes the
oracle's own choice; tests may pass a subclass that, where the oracle's margin
is inside a stated tolerance, adopts another valid choice (conditioned mode).

ORACLE / TEST INFRASTRUCTURE ONLY.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import layers as L
from . import philox


# --------------------------------------------------------------------------- decisions
class Decisions:
    """The oracle's own choices.  Subclasses may override (conditioned mode)."""

    def children(self, b, depth, rank, cand_tokens, logq_row, k):
        """Ordered indices into cand_tokens of a node's k children (log q desc, token asc)."""
        return np.lexsort((np.asarray(cand_tokens), -np.asarray(logq_row)))[:k]

    def candidates(self, b, depth, rank, lowrank_row, c):
        """Two-stage head: ordered indices of the c candidates of the low-rank head."""
        return L.topk_order(lowrank_row, c)

    def frontier(self, b, depth, scores, k):
        """Ordered indices (into this depth's k*k candidates) of the next frontier."""
        return L.topk_order(scores, k)

    def select(self, b, scores, depths, m):
        """Pool indices of the kept nodes, in selection order."""
        idx = np.arange(len(scores))
        return np.lexsort((idx, depths, -scores))[:m]

    def greedy(self, b, node, z_row):
        """Target argmax at a node (ties: lowest token)."""
        return int(np.argmax(z_row))

    def accept(self, b, node, i, u, rejected_mass, p_child):
        return u * (1.0 - rejected_mass) < p_child

    def bonus(self, b, node, scores):
        """Gumbel-argmax (scores already hold -inf at excluded tokens)."""
        return int(np.argmax(scores))

    def accept_q(self, b, node, i, u, q_child, p_child):
        """q-ratio test of the i-th draw: accept when U q_i(c) < p_i(c)."""
        return u * q_child < p_child

    def draw_score(self, cap, logq_draw):
        """Score increment of a sampled draw (R-17): `cap`, the node's largest
        log q capped by the log q of its earlier draws; the draw's own log q
        (logq_draw) is deliberately not used."""
        return cap

    def keep_drafting(self, b, t, mass, threshold):
        """Cost-aware depth rule: run pass t (mass = the frontier's sum of exp(score))."""
        return mass >= threshold

    def verify_count(self, b, gains, costs, m_cap):
        """Kept-set size: the longest prefix (at least 1) with gains[i] >= costs[i]."""
        m = 1
        while m < m_cap and gains[m] >= costs[m]:
            m += 1
        return m


@dataclass
class Control:
    """Per-request caps and the cost-aware rules of one round (R-16).

    Caps are lists over requests (None = the config's value).  A rule is off
    while its threshold is 0 (light_batch 0 turns the branch rule off).
    pass_us[t] is the cost of draft pass t, verify_us[m] that of verifying m
    nodes (verify_us[0] = 0), both from the latency table at the call's shape.
    """
    depth_cap: list | None = None
    topk_cap: list | None = None
    verify_cap: list | None = None
    tau_depth: float = 0.0
    depth_growth: float = 1.0
    tau_verify: float = 0.0
    light_batch: int = 0
    k_light: int = 8
    k_heavy: int = 4
    pass_us: list | None = None
    verify_us: list | None = None

    def k_for(self, b, B, k):
        """Branch cap of request b (caps below 1 count as 1)."""
        if self.light_batch > 0:
            k = max(1, min(k, self.k_light if B <= self.light_batch else self.k_heavy))
        return k if self.topk_cap is None else max(1, min(k, int(self.topk_cap[b])))

    def d_for(self, b, D):
        return D if self.depth_cap is None else max(1, min(D, int(self.depth_cap[b])))

    def m_for(self, b, M):
        return M if self.verify_cap is None else max(1, min(M, int(self.verify_cap[b])))


# --------------------------------------------------------------------------- prefix
def prefix_kv(w, cfg, feats, tokens, rows=None):
    """Post-RoPE K and V of prefix rows (all rows, or the listed ones).

    feats [P, 3d], tokens [P].  Row i has position i, hid = g_i (R-2, R-4).
    """
    rows = np.arange(feats.shape[0]) if rows is None else np.asarray(rows)
    g = L.fused_feature(w, cfg, feats[rows])
    x = L.decoder_input(w, cfg, tokens[rows], g)
    _, k, v = L.qkv(w, cfg, x, rows)
    return k, v


def root_forward(w, cfg, K, V, feat_root, tok_root, root_pos):
    """Pass 0: the root row attends to prefix rows 0..root_pos (its own K/V included)."""
    g = L.fused_feature(w, cfg, feat_root[None])
    x = L.decoder_input(w, cfg, np.array([tok_root]), g)
    q, _, _ = L.qkv(w, cfg, x, np.array([root_pos]))
    o = L.attend(q[0], K[:root_pos + 1], V[:root_pos + 1], cfg)
    s, h = L.layer_tail(w, cfg, g, o[None])
    return s[0], h[0]


# --------------------------------------------------------------------------- draft
@dataclass
class Pool:
    tok: list = field(default_factory=list)
    parent: list = field(default_factory=list)   # pool index, -1 = root
    score: list = field(default_factory=list)
    depth: list = field(default_factory=list)
    logq: list = field(default_factory=list)
    fwd: list = field(default_factory=list)      # frontier slot if expanded, else -1

    def add(self, tok, parent, score, depth, logq):
        self.tok.append(int(tok)); self.parent.append(int(parent)); self.score.append(float(score))
        self.depth.append(int(depth)); self.logq.append(float(logq)); self.fwd.append(-1)

    def ancestors_or_self(self, i):
        out = []
        while i >= 0:
            out.append(i)
            i = self.parent[i]
        return out[::-1]


@dataclass
class DraftResult:
    pool: Pool
    s_root: np.ndarray
    h_root: np.ndarray
    states: dict          # pool index -> s (pre-final-norm state) of expanded nodes
    h: dict               # pool index -> h of expanded nodes
    node_logq: dict       # key (depth, rank) -> (cand tokens, logq) of each expanded node
    frontiers: list       # per pass t>=1: pool indices forwarded, in rank order


def _tree_pass(w, cfg, K, V, root_pos, pool, nodes, states, s_root, tree_kv):
    """One draft pass over frontier nodes: hid = parent's state, keys = prefix + path."""
    tok = np.array([pool.tok[i] for i in nodes])
    hid = np.stack([s_root if pool.parent[i] < 0 else states[pool.parent[i]] for i in nodes])
    pos = np.array([root_pos + pool.depth[i] for i in nodes])
    x = L.decoder_input(w, cfg, tok, hid)
    q, k, v = L.qkv(w, cfg, x, pos)
    for j, i in enumerate(nodes):
        tree_kv[i] = (k[j], v[j])
    o = np.empty((len(nodes), cfg.n_q_heads * cfg.head_dim))
    for j, i in enumerate(nodes):
        path = pool.ancestors_or_self(i)
        Kt = np.concatenate([K[:root_pos + 1], np.stack([tree_kv[a][0] for a in path])])
        Vt = np.concatenate([V[:root_pos + 1], np.stack([tree_kv[a][1] for a in path])])
        o[j] = L.attend(q[j], Kt, Vt, cfg)
    return L.layer_tail(w, cfg, hid, o)


def draft_request(w, cfg, K, V, feat_root, tok_root, root_pos, dec: Decisions, b=0,
                  ctl: Control | None = None, B=1, samp=None):
    """Draft passes and pool of one request (steps 2-4 up to the kept set).

    With ``ctl`` the request's branch and depth caps and the depth rule apply
    (R-16); the pool keeps its layout, with uncreated nodes as -inf slots.
    With ``samp = (seed, round_id)`` the children are sampled (R-17)."""
    k_, D = cfg.topk, cfg.depth
    kb = ctl.k_for(b, B, k_) if ctl else k_
    db = ctl.d_for(b, D) if ctl else D
    s_root, h_root = root_forward(w, cfg, K, V, feat_root, tok_root, root_pos)
    pool = Pool()
    states, hs, node_logq, frontiers, tree_kv = {}, {}, {}, [], {}
    ninf = -np.inf

    def expand(depth, nodes, h_rows):
        """LM head on a pass's rows (one call), then each node's k children."""
        cands, logqs, lowrank = L.draft_logq(w, cfg, h_rows)
        for rank, parent in enumerate(nodes):
            cand, logq = cands[rank], logqs[rank]
            if lowrank is not None:  # candidate choice of the low-rank stage may be conditioned
                order = dec.candidates(b, depth, rank, lowrank[rank], cfg.lr_cand)
                ell = np.array([L.f64(w["w_lm"][c]) @ L.f64(h_rows[rank]) for c in order])
                cand, logq = order, ell - L.logsumexp(ell)
            node_logq[(depth, rank)] = (np.asarray(cand), logq)
            base = 0.0 if parent < 0 else pool.score[parent]
            if samp is None:
                order = dec.children(b, depth, rank, cand, logq, k_)
            else:  # Gumbel-top-k: k draws without replacement, in draw order
                slot = 0 if depth == 0 else 1 + (depth - 1) * k_ + rank
                keys = logq + philox.gumbel(samp[0], samp[1], b, slot, np.asarray(cand), stream=2)
                order = dec.children(b, depth, rank, cand, keys, k_)
            # sampled draft: the i-th draw's score uses only what was drawn before it
            # (the node's largest log q, capped by the earlier draws' log q)
            cap = float(np.max(logq))
            for jr, j in enumerate(order):
                if jr < kb:
                    inc = logq[j] if samp is None else dec.draw_score(cap, float(logq[j]))
                    pool.add(cand[j], parent, base + inc, depth + 1, logq[j])
                    cap = min(cap, float(logq[j]))
                else:
                    pool.add(-1, -1, ninf, depth + 1, ninf)

    def empty_level(depth, n):
        for _ in range(n):
            pool.add(-1, -1, ninf, depth + 1, ninf)

    expand(0, [-1], h_root[None])
    frontier = [i for i in range(k_) if np.isfinite(pool.score[i])] if D >= 2 else []
    for t in range(1, D):
        if ctl is not None and t < db and ctl.tau_depth > 0 and frontier:
            mass = float(np.sum(np.exp([pool.score[i] for i in frontier])))
            thr = ctl.tau_depth * ctl.depth_growth ** t * float(ctl.pass_us[t])
            if not dec.keep_drafting(b, t, mass, thr):
                db = t
        if t >= db or not frontier:
            frontiers.append([])
            empty_level(t, k_ * k_)
            continue
        for r, i in enumerate(frontier):
            pool.fwd[i] = (t - 1) * k_ + r
        frontiers.append(list(frontier))
        s, h = _tree_pass(w, cfg, K, V, root_pos, pool, frontier, states, s_root, tree_kv)
        base = len(pool.tok)
        for r, i in enumerate(frontier):
            states[i], hs[i] = s[r], h[r]
        expand(t, frontier, h)
        empty_level(t, (k_ - len(frontier)) * k_)   # frontier slots with no node
        if t + 1 < D:
            sc = np.array(pool.score[base:])
            fin = int(np.isfinite(sc).sum())
            frontier = [base + int(j) for j in dec.frontier(b, t + 1, sc, k_)][:fin]
    return DraftResult(pool, s_root, h_root, states, hs, node_logq, frontiers)


# --------------------------------------------------------------------------- tree
@dataclass
class Tree:
    """Kept nodes: index 0 is the root, 1..M the kept pool nodes."""
    tok: np.ndarray
    parent: np.ndarray     # tree index of the parent (-1 for the root)
    depth: np.ndarray
    pos: np.ndarray
    score: np.ndarray
    pool_index: np.ndarray  # pool index (-1 for the root)
    mask: np.ndarray       # [M+1, M+1] bool: j is an ancestor-or-self of i

    def children(self, u):
        return [int(c) for c in np.nonzero(self.parent == u)[0]]

    @property
    def n_real(self) -> int:
        """Root plus kept nodes (the slots after them are padding)."""
        return int(np.sum(self.tok >= 0))


def build_tree(pool_tok, pool_parent, pool_score, pool_depth, tok_root, root_pos, m,
               dec: Decisions | None = None, b=0, ctl: Control | None = None) -> Tree:
    """Global top-M of the pool, ancestor-closed, in canonical order, with its mask.

    With ``ctl``: at most the request's verify cap, never an uncreated node, and
    the verify rule of R-16; the tree is padded to M + 1 slots."""
    dec = dec or Decisions()
    score = np.asarray(pool_score, dtype=np.float64)
    depth = np.asarray(pool_depth)
    m_slots = m
    if ctl is not None:
        m = min(ctl.m_for(b, m), int(np.isfinite(score).sum()))
    sel = [int(i) for i in dec.select(b, score, depth, m)]
    if ctl is not None and ctl.tau_verify > 0 and len(sel) > 1:
        gains = np.exp(score[sel])
        vu = np.asarray(ctl.verify_us, dtype=np.float64)
        costs = ctl.tau_verify * (vu[1:len(sel) + 1] - vu[:len(sel)])
        sel = sel[:dec.verify_count(b, gains, costs, len(sel))]
    rank = {p: r for r, p in enumerate(sel)}
    order = sorted(sel, key=lambda p: (depth[p], rank[p]))
    tidx = {p: t + 1 for t, p in enumerate(order)}
    n = len(order) + 1
    tok = np.empty(n, dtype=np.int64); par = np.empty(n, dtype=np.int64)
    dep = np.empty(n, dtype=np.int64); sc = np.empty(n); pidx = np.empty(n, dtype=np.int64)
    tok[0], par[0], dep[0], sc[0], pidx[0] = tok_root, -1, 0, 0.0, -1
    for p in order:
        t = tidx[p]
        pp = int(pool_parent[p])
        if pp >= 0 and pp not in tidx:
            raise ValueError("kept set is not ancestor-closed")
        tok[t], par[t], dep[t], sc[t], pidx[t] = pool_tok[p], (0 if pp < 0 else tidx[pp]), depth[p], score[p], p
    if ctl is not None and n < m_slots + 1:  # padding slots
        pad = m_slots + 1 - n
        tok = np.concatenate([tok, np.full(pad, -1)]); par = np.concatenate([par, np.full(pad, -1)])
        dep = np.concatenate([dep, np.zeros(pad, dtype=np.int64)])
        sc = np.concatenate([sc, np.full(pad, -np.inf)]); pidx = np.concatenate([pidx, np.full(pad, -1)])
        n = m_slots + 1
    mask = np.zeros((n, n), dtype=bool)
    for i in range(n):
        j = i
        while j >= 0:
            mask[i, j] = True
            j = par[j] if (i == 0 or tok[i] >= 0) else -1
    return Tree(tok, par, dep, root_pos + dep, sc, pidx, mask)


# --------------------------------------------------------------------------- verify
def verify_logits(w, cfg, K, V, root_pos, tree: Tree, draft: DraftResult):
    """Target logits z [n, V] of the synthetic target over the root and the kept
    nodes (R-8); padding slots are not evaluated."""
    n = tree.n_real
    h = np.empty((n, cfg.d))
    h[0] = draft.h_root
    if n > 1:
        nodes = np.arange(1, n)
        hid = np.stack([draft.s_root if tree.parent[u] == 0 else
                        draft.states[int(tree.pool_index[tree.parent[u]])] for u in nodes])
        x = L.decoder_input(w, cfg, tree.tok[1:n], hid)
        q, k, v = L.qkv(w, cfg, x, tree.pos[1:n])
        o = np.empty((n - 1, cfg.n_q_heads * cfg.head_dim))
        for j, u in enumerate(nodes):
            anc = [a - 1 for a in np.nonzero(tree.mask[u])[0] if a > 0]
            o[j] = L.attend(q[j], np.concatenate([K[:root_pos + 1], k[anc]]),
                            np.concatenate([V[:root_pos + 1], v[anc]]), cfg)
        _, h[1:] = L.layer_tail(w, cfg, hid, o)
    return L.linear(h, w["w_target"]), h


@dataclass
class VerifyResult:
    accept_len: int
    path: list            # tree indices of accepted nodes
    out_tokens: list      # accepted tokens then the bonus token


def verify_greedy(tree: Tree, z, dec: Decisions | None = None, b=0) -> VerifyResult:
    """Walk from the root while the target's argmax is one of the node's children."""
    dec = dec or Decisions()
    u, path = 0, []
    while True:
        a = dec.greedy(b, u, z[u])
        nxt = [c for c in tree.children(u) if tree.tok[c] == a]
        if not nxt:
            return VerifyResult(len(path), path, [int(tree.tok[p]) for p in path] + [a])
        u = nxt[0]
        path.append(u)


def verify_sample(tree: Tree, z, temperature, seed, round_id, dec: Decisions | None = None,
                  b=0) -> VerifyResult:
    """Sequential point-mass acceptance with residual resampling (R-9, R-10)."""
    dec = dec or Decisions()
    zt = np.asarray(z, dtype=np.float64) / temperature
    u, path = 0, []
    while True:
        p = np.exp(zt[u] - L.logsumexp(zt[u]))
        kids = tree.children(u)
        rejected, taken = 0.0, None
        for i, c in enumerate(kids):
            U = float(philox.uniform(seed, round_id, b, u, i))
            if dec.accept(b, u, i, U, rejected, p[tree.tok[c]]):
                taken = c
                break
            rejected += p[tree.tok[c]]
        if taken is None:
            g = philox.gumbel(seed, round_id, b, u, np.arange(zt.shape[1]))
            sc = zt[u] + g
            sc[[int(tree.tok[c]) for c in kids]] = -np.inf
            x = dec.bonus(b, u, sc)
            return VerifyResult(len(path), path, [int(tree.tok[q]) for q in path] + [x])
        u = taken
        path.append(u)


def verify_qratio(tree: Tree, z, ell, temperature, seed, round_id, dec: Decisions | None = None,
                  b=0) -> VerifyResult:
    """Recursive rejection of sampled children against the draft q (R-17): the
    draws of a node in draw order (pool index), p_i and q_i updated on each
    rejection, the bonus drawn from the last residual."""
    dec = dec or Decisions()
    zt = np.asarray(z, dtype=np.float64) / temperature
    ell = np.asarray(ell, dtype=np.float64)
    u, path = 0, []
    while True:
        p = np.exp(zt[u] - L.logsumexp(zt[u]))
        q = np.exp(ell[u] - L.logsumexp(ell[u]))
        kids = sorted(tree.children(u), key=lambda c: int(tree.pool_index[c]))
        taken = None
        for i, c in enumerate(kids):
            x = int(tree.tok[c])
            U = float(philox.uniform(seed, round_id, b, u, i))
            if dec.accept_q(b, u, i, U, q[x], p[x]):
                taken = c
                break
            r = np.maximum(p - q, 0.0)
            if r.sum() > 0:
                p = r / r.sum()
            q[x] = 0.0
            if q.sum() > 0:
                q = q / q.sum()
        if taken is None:
            g = philox.gumbel(seed, round_id, b, u, np.arange(zt.shape[1]))
            with np.errstate(divide="ignore"):
                sc = np.where(p > 0, np.log(p) + g, -np.inf)
            x = dec.bonus(b, u, sc)
            return VerifyResult(len(path), path, [int(tree.tok[q_]) for q_ in path] + [x])
        u = taken
        path.append(u)


# --------------------------------------------------------------------------- whole round
@dataclass
class RequestRound:
    draft: DraftResult
    tree: Tree
    z: np.ndarray | None
    verify: dict          # temperature -> VerifyResult


def round_request(w, cfg, K, V, feat_root, tok_root, root_pos, temperatures=(0.0,), seed=0,
                  round_id=0, dec: Decisions | None = None, b=0, with_verify=True,
                  ctl: Control | None = None, B=1, samp=None):
    """One request's round.  With ``samp = (draft_seed, draft_round)`` the children
    are sampled and T > 0 verification is the q-ratio scheme (R-17)."""
    dec = dec or Decisions()
    dr = draft_request(w, cfg, K, V, feat_root, tok_root, root_pos, dec, b, ctl, B, samp)
    p = dr.pool
    tree = build_tree(p.tok, p.parent, p.score, p.depth, tok_root, root_pos, cfg.n_verify, dec, b,
                      ctl)
    z, out = None, {}
    if with_verify:
        z, hv = verify_logits(w, cfg, K, V, root_pos, tree, dr)
        ell = L.linear(hv, w["w_lm"]) if samp is not None else None
        for T in temperatures:
            if T == 0:
                out[T] = verify_greedy(tree, z, dec, b)
            elif samp is None:
                out[T] = verify_sample(tree, z, T, seed, round_id, dec, b)
            else:
                out[T] = verify_qratio(tree, z, ell, T, seed, round_id, dec, b)
    return RequestRound(dr, tree, z, out)


def weights_f32(inputs) -> dict:
    """Upcast every stored tensor to float32 (exact for bf16) for the oracle."""
    return {k: inputs.f32(k) for k in inputs.w}
