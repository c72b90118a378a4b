"""ctypes binding of ``libeagle3.so``: the C ABI of ``include/eagle3.h``, same names.

Argument marshalling only — every step of the round runs in the library's
CUDA kernels.  Pointers are passed as Python ints (e.g. ``tensor.data_ptr()``),
streams as ``torch.cuda.Stream.cuda_stream`` ints.  Importing this module loads
the library and fails loudly if it is missing.
"""
from __future__ import annotations

import ctypes as C
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libeagle3.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "eagle3.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m eagle_draft_tree_02_b300.build`")
lib = C.CDLL(LIB_PATH)

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_UNSUPPORTED, ERR_OOM, ERR_CUDA, ERR_TIMEOUT, \
    ERR_DEVICE_ASSERT, ERR_STATE = range(9)
FP32, BF16 = 0, 1


class eagle3_config(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("d", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                                       "lr_rank", "lr_cand")] + \
               [("rope_theta", C.c_float), ("rms_eps", C.c_float)] + \
               [(n, C.c_int) for n in ("dtype", "depth", "topk", "n_verify", "page_size",
                                       "max_batch", "max_prefix", "max_new", "variant")]


WEIGHT_NAMES = ("w_fc", "embed", "w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down",
                "g_emb", "g_hid", "g_post", "g_final", "w_lm", "w_target", "lr_u", "lr_v", "g_fc")
FC_NORM, POST_NORM, SAMPLED_DRAFT = 1, 2, 4  # eagle3_config.variant bits


class eagle3_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_NAMES]


class eagle3_kv(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("page_table", C.c_void_p),
                ("seq_lens", C.c_void_p), ("max_pages", C.c_int), ("n_pages", C.c_int)]


class eagle3_tree(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("tokens", "parent", "depth", "pos", "pool_index",
                                          "score", "mask")]


class eagle3_pool(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("tok", "parent", "depth", "fwd", "score", "logq", "cand")]


class eagle3_control(C.Structure):
    _fields_ = [("depth_cap", C.c_void_p), ("topk_cap", C.c_void_p), ("verify_cap", C.c_void_p),
                ("tau_depth", C.c_float), ("depth_growth", C.c_float), ("tau_verify", C.c_float),
                ("light_batch", C.c_int), ("k_light", C.c_int), ("k_heavy", C.c_int),
                ("pass_us", C.POINTER(C.c_float)), ("verify_us", C.POINTER(C.c_float))]


class eagle3_latency_table(C.Structure):
    _fields_ = [("n_batch", C.c_int), ("n_prefix", C.c_int), ("n_tokens", C.c_int),
                ("batch", C.POINTER(C.c_int)), ("prefix", C.POINTER(C.c_int)),
                ("tokens", C.POINTER(C.c_int)), ("draft_us", C.POINTER(C.c_float)),
                ("verify_us", C.POINTER(C.c_float))]


class eagle3_verify_stats(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("z_max", "lse", "z_argmax", "g_argmax")]


_P = C.c_void_p
_sig = {
    "eagle3_create": (C.c_int, [C.POINTER(eagle3_config), C.POINTER(eagle3_weights), C.POINTER(_P)]),
    "eagle3_destroy": (None, [_P]),
    "eagle3_prefill": (C.c_int, [_P, C.c_int, C.c_int, _P, _P, _P, C.POINTER(eagle3_kv), _P]),
    "eagle3_draft_round": (C.c_int, [_P, C.c_int, C.c_int, _P, _P, C.POINTER(eagle3_kv),
                                     C.POINTER(eagle3_tree), C.POINTER(eagle3_pool), _P]),
    "eagle3_draft_round_ragged": (C.c_int, [_P, C.c_int, C.c_int, _P, _P, _P, C.POINTER(eagle3_kv),
                                            C.POINTER(eagle3_tree), C.POINTER(eagle3_pool), _P]),
    "eagle3_next_rows": (C.c_int, [_P, C.c_int, _P, _P, _P, _P, _P]),
    "eagle3_build_tree": (C.c_int, [_P, C.c_int, C.c_int, _P, _P, _P, _P, _P, _P,
                                    C.POINTER(eagle3_tree), _P]),
    "eagle3_verify": (C.c_int, [_P, C.c_int, C.POINTER(eagle3_tree), C.POINTER(eagle3_kv), C.c_int,
                                C.c_float, C.c_ulonglong, C.c_ulonglong, _P, _P, _P,
                                C.POINTER(eagle3_verify_stats), _P]),
    "eagle3_verify_logits": (C.c_int, [_P, C.c_int, C.POINTER(eagle3_tree), _P, C.c_int,
                                       C.c_longlong, C.c_int, C.c_float, C.c_ulonglong,
                                       C.c_ulonglong, _P, _P, _P, C.POINTER(eagle3_verify_stats),
                                       _P]),
    "eagle3_graph_capture": (C.c_int, [_P, C.c_int, C.c_int, _P, _P, C.POINTER(eagle3_kv),
                                       C.POINTER(eagle3_tree), C.c_int, C.c_int, C.c_float,
                                       C.c_ulonglong, _P, _P, _P, _P]),
    "eagle3_graph_launch": (C.c_int, [_P, C.c_ulonglong, _P]),
    "eagle3_lm_head_topk": (C.c_int, [_P, C.c_int, _P, _P, _P, _P, _P]),
    "eagle3_lm_head_topk_noalloc": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, _P, C.c_int, _P,
                                              _P, _P, _P, _P, _P]),
    "eagle3_linear": (C.c_int, [_P, C.c_int, C.c_int, _P, _P, _P]),
    "eagle3_check": (C.c_int, [_P]),
    "eagle3_last_error": (C.c_char_p, [_P]),
    "eagle3_workspace_bytes": (C.c_size_t, [_P]),
    "eagle3_last_launch_count": (C.c_int, [_P]),
    "eagle3_set_control": (C.c_int, [_P, C.POINTER(eagle3_control)]),
    "eagle3_draft_noise": (C.c_int, [_P, C.c_ulonglong, C.c_ulonglong, _P]),
    "eagle3_latency_costs": (C.c_int, [C.POINTER(eagle3_latency_table), C.c_int, C.c_int, C.c_int,
                                       C.c_int, C.c_int, C.POINTER(C.c_float),
                                       C.POINTER(C.c_float)]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def declared_functions() -> list[str]:
    """Names of the entry points declared in include/eagle3.h."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(eagle3_[a-z_]+)\s*\(", txt)))


class Eagle3Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"eagle3 status {status}: {msg}")
        self.status = status


def _ref(x):
    return None if x is None else C.byref(x)


# -------------------------------------------------------------- same-name wrappers
def eagle3_create(cfg: eagle3_config, w: eagle3_weights) -> tuple[int, int]:
    out = _P()
    s = lib.eagle3_create(C.byref(cfg), C.byref(w), C.byref(out))
    return s, (out.value or 0)


def eagle3_destroy(ctx: int) -> None:
    lib.eagle3_destroy(ctx)


def eagle3_prefill(ctx, B, total_rows, cu_rows, feats, tokens, kv: eagle3_kv, stream=0) -> int:
    return lib.eagle3_prefill(ctx, B, total_rows, cu_rows, feats, tokens, C.byref(kv), stream)


def eagle3_draft_round(ctx, B, n_new, feats_new, tokens_new, kv: eagle3_kv, tree: eagle3_tree,
                       pool: eagle3_pool | None = None, stream=0) -> int:
    return lib.eagle3_draft_round(ctx, B, n_new, feats_new, tokens_new, C.byref(kv), C.byref(tree),
                                  _ref(pool), stream)


def eagle3_draft_round_ragged(ctx, B, total_new, cu_new, feats_new, tokens_new, kv: eagle3_kv,
                              tree: eagle3_tree, pool: eagle3_pool | None = None, stream=0) -> int:
    return lib.eagle3_draft_round_ragged(ctx, B, total_new, cu_new, feats_new, tokens_new, C.byref(kv),
                                         C.byref(tree), _ref(pool), stream)


def eagle3_next_rows(ctx, B, accept_len, out_tokens, cu_new, tokens_new, stream=0) -> int:
    return lib.eagle3_next_rows(ctx, B, accept_len, out_tokens, cu_new, tokens_new, stream)


def eagle3_build_tree(ctx, B, pool_n, pool_tok, pool_parent, pool_score, pool_depth, root_tok,
                      root_pos, tree: eagle3_tree, stream=0) -> int:
    return lib.eagle3_build_tree(ctx, B, pool_n, pool_tok, pool_parent, pool_score, pool_depth,
                                 root_tok, root_pos, C.byref(tree), stream)


def eagle3_verify(ctx, B, tree: eagle3_tree, kv: eagle3_kv, mode, temperature, seed, round_id,
                  accept_len, path, out_tokens, stats: eagle3_verify_stats | None = None,
                  stream=0) -> int:
    return lib.eagle3_verify(ctx, B, C.byref(tree), C.byref(kv), mode, temperature, seed, round_id,
                             accept_len, path, out_tokens, _ref(stats), stream)


def eagle3_verify_logits(ctx, B, tree: eagle3_tree, logits, logits_dtype, ld, mode, temperature,
                         seed, round_id, accept_len, path, out_tokens,
                         stats: eagle3_verify_stats | None = None, stream=0) -> int:
    return lib.eagle3_verify_logits(ctx, B, C.byref(tree), logits, logits_dtype, ld, mode,
                                    temperature, seed, round_id, accept_len, path, out_tokens,
                                    _ref(stats), stream)


def eagle3_graph_capture(ctx, B, n_new, feats_new, tokens_new, kv: eagle3_kv, tree: eagle3_tree,
                         with_verify, mode, temperature, seed, accept_len, path, out_tokens,
                         stream) -> int:
    return lib.eagle3_graph_capture(ctx, B, n_new, feats_new, tokens_new, C.byref(kv), C.byref(tree),
                                    with_verify, mode, temperature, seed, accept_len, path,
                                    out_tokens, stream)


def eagle3_graph_launch(ctx, round_id, stream) -> int:
    return lib.eagle3_graph_launch(ctx, round_id, stream)


def eagle3_lm_head_topk(ctx, R, h, tok, logq, lse=None, stream=0) -> int:
    return lib.eagle3_lm_head_topk(ctx, R, h, tok, logq, lse, stream)


def eagle3_lm_head_topk_noalloc(dtype, vocab, d, topk, w_lm, R, h, tok, logq, lse=None,
                                dev_status=None, stream=0) -> int:
    return lib.eagle3_lm_head_topk_noalloc(dtype, vocab, d, topk, w_lm, R, h, tok, logq, lse,
                                           dev_status, stream)


def eagle3_linear(ctx, which, R, X, Y, stream=0) -> int:
    return lib.eagle3_linear(ctx, which, R, X, Y, stream)


def eagle3_check(ctx) -> int:
    return lib.eagle3_check(ctx)


def eagle3_last_error(ctx) -> str:
    v = lib.eagle3_last_error(ctx)
    return v.decode() if v else ""


def eagle3_workspace_bytes(ctx) -> int:
    return lib.eagle3_workspace_bytes(ctx)


def eagle3_last_launch_count(ctx) -> int:
    return lib.eagle3_last_launch_count(ctx)


def eagle3_draft_noise(ctx, seed, round_id, stream=0) -> int:
    return lib.eagle3_draft_noise(_P(ctx), seed, round_id, _P(stream))


def eagle3_set_control(ctx, ctl: eagle3_control | None) -> int:
    return lib.eagle3_set_control(_P(ctx), C.byref(ctl) if ctl is not None else None)


def make_control(depth_cap=None, topk_cap=None, verify_cap=None, tau_depth=0.0, depth_growth=1.0,
                 tau_verify=0.0, light_batch=0, k_light=8, k_heavy=4, pass_us=None,
                 verify_us=None) -> eagle3_control:
    """Marshal the control: caps are device pointers (int or None), costs host sequences."""
    c = eagle3_control()
    c.depth_cap, c.topk_cap, c.verify_cap = depth_cap, topk_cap, verify_cap
    c.tau_depth, c.depth_growth, c.tau_verify = tau_depth, depth_growth, tau_verify
    c.light_batch, c.k_light, c.k_heavy = light_batch, k_light, k_heavy
    if pass_us is not None:
        c._pass = (C.c_float * len(pass_us))(*pass_us)
        c.pass_us = C.cast(c._pass, C.POINTER(C.c_float))
    if verify_us is not None:
        c._verify = (C.c_float * len(verify_us))(*verify_us)
        c.verify_us = C.cast(c._verify, C.POINTER(C.c_float))
    return c


def eagle3_latency_costs(batch, prefix, tokens, draft_us, verify_us, B, P, depth, topk, n_verify):
    """Host lookup of one round's costs from a latency table (grids and [nb][np][nt] arrays)."""
    import numpy as _np
    t = eagle3_latency_table()
    g = [(_np.ascontiguousarray(x, dtype=_np.int32)) for x in (batch, prefix, tokens)]
    v = [(_np.ascontiguousarray(x, dtype=_np.float32)) for x in (draft_us, verify_us)]
    t.n_batch, t.n_prefix, t.n_tokens = (len(x) for x in g)
    ip, fp = C.POINTER(C.c_int), C.POINTER(C.c_float)
    t.batch, t.prefix, t.tokens = (x.ctypes.data_as(ip) for x in g)
    t.draft_us, t.verify_us = (x.ctypes.data_as(fp) for x in v)
    pu = (C.c_float * depth)()
    vu = (C.c_float * (n_verify + 1))()
    s = lib.eagle3_latency_costs(C.byref(t), B, P, depth, topk, n_verify, pu, vu)
    return s, list(pu), list(vu)


def check(ctx, status: int) -> None:
    """Raise Eagle3Error for a non-OK status."""
    if status != OK:
        raise Eagle3Error(status, eagle3_last_error(ctx) if ctx else "")
