"""fp64 building blocks of the one-layer EAGLE-3 draft decoder (oracle).

Every function takes the exact stored values (fp32 or bf16 upcast) and computes
in float64.  Page citations:

* fusion of the target's low/mid/high features into g by one linear map:
  "EAGLE-3 精读" §1 (为什么推翻 feature regression), paragraph 2; abstract of
  "EAGLE-3: Scaling up Inference Acceleration of LLMs via Training-Time Test"
  (multi-layer feature fusion);
* the decoder combines g (or its own state), and the token embedding, in one
  Transformer layer: "EAGLE-3 精读" §1 paragraph 2 and §2 (Training-Time
  Test: the draft feeds back its own trajectory); the EAGLE-4 blog (the drafter
  is still a single Transformer layer);
* the draft distribution is the softmax of the LM head's logits: the EAGLE-4
  blog, section 关于 Efficient LM Head.

Readings where the pages are silent (listed again in the design notes):
  R-1 fusion has no bias and no norm on g;
  R-3 RMSNorm eps = 1e-5, gains as given (1 in the synthetic inputs);
  R-4 decoder input x = [rms(E[y]); rms(hid)], hid = g for a prefix row and the
      parent's pre-final-norm state s for a tree node;
  R-5 rotate-half RoPE, inv_freq_j = theta^(-2j/dh), angle = pos * inv_freq in
      float64, no frequency scaling;
  R-6 pre-norm layer: r = hid + W_o attn(x); s = r + W_down(silu(W_g z) * W_u z)
      with z = rms(r); h = rms(s) feeds the LM head.
  R-15 drafter variants named by the EAGLE-4 blog (section 在EAGLE4中: the
      drafter keeps EAGLE-3.1's FC Norm and Post-norm), with no formula there:
      FC norm g = rms(W_fc f; g_fc); post-norm r = rms(hid + W_o attn(x); g_post),
      s = rms(r + W_down(silu(W_g r) * W_u r); g_final), and s is both the LM
      head's input and the state fed to children.

ORACLE / TEST INFRASTRUCTURE ONLY.
"""
from __future__ import annotations

import numpy as np

_ROW_CHUNK = 16384


def f64(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x W^T in float64.  W is [out, in] (fp32 storage is upcast block by block)."""
    x = f64(x)
    out = np.empty(x.shape[:-1] + (W.shape[0],), dtype=np.float64)
    for i in range(0, W.shape[0], _ROW_CHUNK):
        j = min(W.shape[0], i + _ROW_CHUNK)
        out[..., i:j] = x @ f64(W[i:j]).T
    return out


def rmsnorm(v: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    v = f64(v)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps) * f64(gamma)


def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE: pairs (j, j + dh/2) turn by pos * theta^(-2j/dh).

    x: [n, H, dh], pos: [n] integer positions.
    """
    x = f64(x)
    dh = x.shape[-1]
    half = dh // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / dh)
    ang = f64(pos)[:, None] * inv[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def fuse(feats: np.ndarray, w_fc: np.ndarray) -> np.ndarray:
    """g = W_fc [low; mid; high] (R-1: no bias, no norm)."""
    return linear(feats, w_fc)


def fused_feature(w: dict, cfg, feats: np.ndarray) -> np.ndarray:
    """The decoder's hid for prefix rows: g = W_fc f, or rms(W_fc f; g_fc) with the
    FC-norm variant (R-15)."""
    g = fuse(feats, w["w_fc"])
    if getattr(cfg, "fc_norm", False):
        g = rmsnorm(g, w["g_fc"], cfg.rms_eps)
    return g


def decoder_input(w: dict, cfg, tokens: np.ndarray, hid: np.ndarray) -> np.ndarray:
    """x = [rms(E[y]; g_emb); rms(hid; g_hid)]  -> [n, 2d]."""
    e = f64(w["embed"][np.asarray(tokens)])
    return np.concatenate([rmsnorm(e, w["g_emb"], cfg.rms_eps),
                           rmsnorm(hid, w["g_hid"], cfg.rms_eps)], axis=-1)


def qkv(w: dict, cfg, x: np.ndarray, pos: np.ndarray):
    """Projections and RoPE: q [n,Hq,dh], k [n,Hkv,dh], v [n,Hkv,dh]."""
    n, dh = x.shape[0], cfg.head_dim
    q = linear(x, w["w_q"]).reshape(n, cfg.n_q_heads, dh)
    k = linear(x, w["w_k"]).reshape(n, cfg.n_kv_heads, dh)
    v = linear(x, w["w_v"]).reshape(n, cfg.n_kv_heads, dh)
    return rope(q, pos, cfg.rope_theta), rope(k, pos, cfg.rope_theta), v


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, cfg) -> np.ndarray:
    """Softmax attention of one query row over an explicit key list.

    q: [Hq, dh]; K, V: [n_keys, Hkv, dh].  Query head h reads KV head
    floor(h * Hkv / Hq) (grouped-query attention).  Returns [Hq * dh].
    """
    Hq, dh = q.shape
    out = np.empty((Hq, dh), dtype=np.float64)
    scale = 1.0 / np.sqrt(dh)
    for h in range(Hq):
        kv = h * cfg.n_kv_heads // Hq
        s = K[:, kv, :] @ q[h] * scale
        s = np.exp(s - s.max())
        out[h] = (s / s.sum()) @ V[:, kv, :]
    return out.reshape(-1)


def layer_tail(w: dict, cfg, hid: np.ndarray, o: np.ndarray):
    """O-projection, residual, SwiGLU FFN and the final norm.

    Returns (s, h): s is the pre-final-norm state fed to children, h = rms(s).
    With the post-norm variant (R-15) both sums are normalised after the add and
    s = h.
    """
    if getattr(cfg, "post_norm", False):
        r = rmsnorm(f64(hid) + linear(o, w["w_o"]), w["g_post"], cfg.rms_eps)
        s = rmsnorm(r + linear(silu(linear(r, w["w_gate"])) * linear(r, w["w_up"]), w["w_down"]),
                    w["g_final"], cfg.rms_eps)
        return s, s
    r = f64(hid) + linear(o, w["w_o"])
    z = rmsnorm(r, w["g_post"], cfg.rms_eps)
    s = r + linear(silu(linear(z, w["w_gate"])) * linear(z, w["w_up"]), w["w_down"])
    return s, rmsnorm(s, w["g_final"], cfg.rms_eps)


def logsumexp(v: np.ndarray, axis=-1) -> np.ndarray:
    m = v.max(axis=axis, keepdims=True)
    return (m + np.log(np.exp(v - m).sum(axis=axis, keepdims=True))).squeeze(axis)


def draft_logq(w: dict, cfg, h: np.ndarray):
    """Draft log-probabilities.  Single-stage: log softmax of W_lm h over the vocab.

    Two-stage head (EAGLE-4 blog, sections on the Efficient LM Head): a low-rank
    head U (V_lr h) scores the whole vocabulary, its top-`lr_cand` tokens are
    rescored with the exact head rows, and (R-11) log q is normalised over that
    candidate set only.  Returns (tokens [n, c], logq [n, c], lowrank_scores or
    None); tokens is arange(V) broadcast for the single-stage head.
    """
    h = f64(h)
    n = h.shape[0]
    if not cfg.lr_rank:
        ell = linear(h, w["w_lm"])
        logq = ell - logsumexp(ell)[:, None]
        return np.broadcast_to(np.arange(cfg.vocab), (n, cfg.vocab)), logq, None
    t = linear(h, w["lr_v"])
    ell_lr = linear(t, w["lr_u"])
    cand = np.stack([topk_order(ell_lr[i], cfg.lr_cand) for i in range(n)])
    ell = np.stack([f64(w["w_lm"][cand[i]]) @ h[i] for i in range(n)])
    logq = ell - logsumexp(ell)[:, None]
    return cand, logq, ell_lr


def topk_order(values: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values, ordered by (value desc, index asc)."""
    idx = np.arange(values.shape[0])
    return np.lexsort((idx, -values))[:k]
