"""Seeded synthetic inputs for one EAGLE-3 round (weights, target features, tokens).

This module is the only code that the CUDA path and the CPU oracle both use.  It
draws random numbers and rounds them to the storage type; it holds none of the
method's arithmetic.

Recipe (every config):
  * one PCG64 stream per (config seed, tensor id, chunk id), built from
    ``numpy.random.SeedSequence(seed, spawn_key=(tensor, chunk))`` so chunks can
    be drawn on several threads and still give the same numbers;
  * normals drawn in float64 and rounded once (round-to-nearest-even) to the
    storage type (fp32, or bf16 kept as raw uint16 bits);
  * weights ~ N(0, 0.02); the draft LM head ~ N(0, lm_std) (0.08 for the tiny
    fp32 case so its logits are peaked, 0.02 elsewhere, which gives the same
    logit spread 1.28 at both widths); RMSNorm gains are 1;
  * target head ``W_t = round(W_lm + eps * G)``, G ~ N(0, 0.02), eps = 0.3;
  * target features ~ N(0, 1); tokens ~ U[0, V);
  * two-stage head: U ~ N(0, (1/16)^2) [V, r], V_lr ~ N(0, 0.02^2) [r, d],
    ``W_lm = round(U V_lr + 0.5 * N(0, 0.02^2))`` (the low-rank part carries 80%
    of the variance, total std about 0.022);
  * RMSNorm gains are 1, except in the drafter-variant cases, which draw them
    as 1 + N(0, gain_std^2) so that a dropped or misplaced gain shows;
  * ragged prefixes: P_b ~ U{lo..hi}; a paged cache gets its physical pages in a
    random permutation so the page table is exercised.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

from .configs import CONFIGS, RoundConfig

_CHUNK = 1 << 23

# tensor ids (fixed: they are part of the recipe)
T_WFC, T_EMB, T_WQ, T_WK, T_WV, T_WO, T_WG, T_WU, T_WD, T_WLM, T_G, T_FEAT, T_TOK, T_PLEN, \
    T_PAGES, T_LRU, T_LRV, T_LRN, T_GAIN = range(19)


def bf16_bits_from_f64(x: np.ndarray) -> np.ndarray:
    """Round float64 values once, to nearest even, to bfloat16; return raw uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    # bf16 keeps 7 explicit mantissa bits; float64 has 52, so drop 45 bits.
    lsb = (u >> np.uint64(45)) & np.uint64(1)
    u = (u + (np.uint64((1 << 44) - 1) + lsb)) & ~np.uint64((1 << 45) - 1)
    f32 = u.view(np.float64).astype(np.float32)  # exact: value has <= 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw(seed: int, tensor: int, n: int, std: float, dtype: str, threads: int) -> np.ndarray:
    """n normals N(0, std^2), rounded once to the storage type."""
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    chunks = [(i, min(_CHUNK, n - i * _CHUNK)) for i in range((n + _CHUNK - 1) // _CHUNK)]

    def work(c):
        ci, cn = c
        ss = np.random.SeedSequence(seed, spawn_key=(tensor, ci))
        v = np.random.Generator(np.random.PCG64(ss)).standard_normal(cn) * std
        sl = slice(ci * _CHUNK, ci * _CHUNK + cn)
        out[sl] = bf16_bits_from_f64(v) if dtype == "bf16" else v.astype(np.float32)

    if threads > 1 and len(chunks) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, chunks))
    else:
        for c in chunks:
            work(c)
    return out


def _rng(seed: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(tensor, 0))))


@dataclass
class RoundInputs:
    """Everything one round consumes.  bf16 tensors are raw uint16 bits."""
    cfg: RoundConfig
    seed: int
    w: dict                 # name -> array (storage dtype), row-major [out, in]
    prefix_lens: np.ndarray  # [B] int32: rows in the cache after the round's new row
    feats: np.ndarray       # [sum P_b, 3d] storage dtype, packed by request
    tokens: np.ndarray      # [sum P_b] int32
    cu_rows: np.ndarray     # [B+1] int64 offsets into feats/tokens
    page_table: np.ndarray | None = None  # [B, pages_per_req] int32 (paged cache)
    n_pages: int = 0

    def f32(self, name: str) -> np.ndarray:
        a = self.w[name]
        return bf16_bits_to_f32(a) if a.dtype == np.uint16 else a

    def feats_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.feats) if self.feats.dtype == np.uint16 else self.feats


def make_inputs(cfg: RoundConfig, seed: int | None = None, threads: int | None = None,
                with_target: bool = True) -> RoundInputs:
    """Draw the inputs of one round for ``cfg`` (seed defaults to the config's index)."""
    if seed is None:
        seed = next((i for i, c in enumerate(CONFIGS) if c.name == cfg.name), 0)
    if threads is None:
        threads = min(16, len(os.sched_getaffinity(0)))
    d, V, dt = cfg.d, cfg.vocab, cfg.dtype
    qd, kvd = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim

    def W(tid, rows, cols, std=0.02):
        return _draw(seed, tid, rows * cols, std, dt, threads).reshape(rows, cols)

    w = {
        "w_fc": W(T_WFC, d, 3 * d),
        "embed": W(T_EMB, V, d),
        "w_q": W(T_WQ, qd, 2 * d),
        "w_k": W(T_WK, kvd, 2 * d),
        "w_v": W(T_WV, kvd, 2 * d),
        "w_o": W(T_WO, d, qd),
        "w_gate": W(T_WG, cfg.ffn, d),
        "w_up": W(T_WU, cfg.ffn, d),
        "w_down": W(T_WD, d, cfg.ffn),
    }
    gains = ("g_emb", "g_hid", "g_post", "g_final") + (("g_fc",) if cfg.fc_norm else ())
    for i, g in enumerate(gains):
        v = np.ones(d, dtype=np.float64)
        if cfg.gain_std > 0:
            v = v + cfg.gain_std * _rng(seed, T_GAIN * 1000 + i).standard_normal(d)
        w[g] = bf16_bits_from_f64(v) if dt == "bf16" else v.astype(np.float32)

    if cfg.lr_rank:
        r = cfg.lr_rank
        w["lr_u"] = W(T_LRU, V, r, 1.0 / 16.0)
        w["lr_v"] = W(T_LRV, r, d, 0.02)
        u32 = bf16_bits_to_f32(w["lr_u"]) if dt == "bf16" else w["lr_u"]
        v32 = bf16_bits_to_f32(w["lr_v"]) if dt == "bf16" else w["lr_v"]
        lm = np.empty((V, d), dtype=np.uint16 if dt == "bf16" else np.float32)
        step = 8192

        def lm_block(i):
            j = min(V, i + step)
            noise = _draw(seed, T_LRN * 1000 + i // step, (j - i) * d, 1.0, "fp32", 1)
            blk = (u32[i:j] @ v32).astype(np.float64) + 0.5 * 0.02 * noise.reshape(j - i, d)
            lm[i:j] = bf16_bits_from_f64(blk).reshape(j - i, d) if dt == "bf16" else blk

        with ThreadPoolExecutor(max(1, threads)) as ex:
            list(ex.map(lm_block, range(0, V, step)))
        w["w_lm"] = lm
    else:
        w["w_lm"] = W(T_WLM, V, d, cfg.lm_std)

    if with_target:
        lm_bits = w["w_lm"]
        wt = np.empty((V, d), dtype=lm_bits.dtype)
        step = 8192

        def target_block(i):
            j = min(V, i + step)
            g = _draw(seed, T_G * 1000 + i // step, (j - i) * d, 0.02, "fp32", 1)
            lm = bf16_bits_to_f32(lm_bits[i:j]) if dt == "bf16" else lm_bits[i:j]
            blk = lm.astype(np.float64) + cfg.eps_target * g.reshape(j - i, d).astype(np.float64)
            wt[i:j] = bf16_bits_from_f64(blk).reshape(j - i, d) if dt == "bf16" else blk

        with ThreadPoolExecutor(max(1, threads)) as ex:
            list(ex.map(target_block, range(0, V, step)))
        w["w_target"] = wt

    B = cfg.batch
    if cfg.prefix_range is not None:
        lo, hi = cfg.prefix_range
        plen = _rng(seed, T_PLEN).integers(lo, hi + 1, size=B).astype(np.int32)
    else:
        plen = np.full(B, cfg.prefix, dtype=np.int32)
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(plen)
    rows = int(cu[-1])
    feats = _draw(seed, T_FEAT, rows * 3 * d, 1.0, dt, threads).reshape(rows, 3 * d)
    tokens = _rng(seed, T_TOK).integers(0, V, size=rows).astype(np.int32)

    page_table, n_pages = None, 0
    if cfg.page_size:
        ps = cfg.page_size
        per = (int(plen.max()) + ps - 1) // ps
        n_pages = B * per
        perm = _rng(seed, T_PAGES).permutation(n_pages).astype(np.int32)
        page_table = perm.reshape(B, per)
    return RoundInputs(cfg=cfg, seed=seed, w=w, prefix_lens=plen, feats=feats, tokens=tokens,
                       cu_rows=cu, page_table=page_table, n_pages=n_pages)


T_LOGITS = 40  # tensor id of caller-supplied target logits (test inputs)


def draw_logits(seed: int, rows: int, V: int, ld: int, std: float, dtype: str) -> np.ndarray:
    """Stand-in target logits [rows, ld]: N(0, std^2) in the first V columns,
    zeros in the row padding, rounded once to the storage type (bf16 as raw
    uint16 bits)."""
    z = _rng(seed, T_LOGITS).standard_normal((rows, V)) * std
    out = np.zeros((rows, ld), dtype=np.float64)
    out[:, :V] = z
    if dtype == "bf16":
        return bf16_bits_from_f64(out.reshape(-1)).reshape(rows, ld)
    return out.astype(np.float32)
