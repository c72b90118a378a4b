"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point that include/eagle3.h declares, and rejects bad arguments
before touching the device."""
import ctypes as C

import pytest


@pytest.fixture(scope="module")
def E(lib_built):
    from eagle_draft_tree_02_b300 import eagle3
    return eagle3


def test_library_exports_every_declared_symbol(E):
    names = E.declared_functions()
    assert "eagle3_draft_round" in names and "eagle3_build_tree" in names and "eagle3_verify" in names
    for n in names:
        assert hasattr(E.lib, n), n


def _cfg(E, **kw):
    from eagle_draft_tree_02_b300.configs import by_name
    from eagle_draft_tree_02_b300.runner import make_config
    c = make_config(by_name("tiny_fp32_b1"), max_prefix=64)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _weights(E, missing=()):
    w = E.eagle3_weights()
    for i, n in enumerate(E.WEIGHT_NAMES):
        if n not in missing and n not in ("lr_u", "lr_v"):
            setattr(w, n, 0x1000 * (i + 1))
    return w


@pytest.mark.parametrize("field,value,status", [
    ("d", 0, 1), ("d", 100, 1), ("head_dim", 200, 1), ("n_kv_heads", 3, 1), ("dtype", 5, 1),
    ("depth", 0, 3), ("depth", 17, 3), ("topk", 17, 3), ("n_verify", 129, 3),
    ("n_verify", 1000, 3), ("max_batch", 0, 1), ("max_new", 0, 1),
])
def test_create_rejects_bad_config(E, field, value, status):
    s, ctx = E.eagle3_create(_cfg(E, **{field: value}), _weights(E))
    assert s == status and ctx == 0


def test_create_rejects_pool_smaller_than_m(E):
    s, ctx = E.eagle3_create(_cfg(E, depth=1, topk=4, n_verify=5), _weights(E))
    assert s == E.ERR_SHAPE and ctx == 0


def test_create_rejects_missing_weight(E):
    s, ctx = E.eagle3_create(_cfg(E), _weights(E, missing=("w_lm",)))
    assert s == E.ERR_INVALID_ARG and ctx == 0


def test_null_context_calls_fail_cleanly(E):
    kv, tree = E.eagle3_kv(), E.eagle3_tree()
    assert E.eagle3_draft_round(0, 1, 1, 1, 1, kv, tree) == E.ERR_INVALID_ARG
    assert E.eagle3_verify(0, 1, tree, kv, 0, 1.0, 0, 0, 1, 1, 1) == E.ERR_INVALID_ARG
    assert E.eagle3_build_tree(0, 1, 4, 1, 1, 1, 1, 1, 1, tree) == E.ERR_INVALID_ARG
    assert E.eagle3_prefill(0, 1, 1, 1, 1, 1, kv) == E.ERR_INVALID_ARG
    assert E.eagle3_lm_head_topk(0, 1, 1, 1, 1) == E.ERR_INVALID_ARG
    assert E.eagle3_check(0) == E.ERR_INVALID_ARG
    assert E.eagle3_last_error(0) == "null context"
    assert E.eagle3_workspace_bytes(0) == 0


def test_noalloc_head_rejects_bad_requests_before_launch(E):
    """Argument checks of the allocation-free head run on the host, before any CUDA call."""
    ok_args = dict(dtype=E.BF16, vocab=128256, d=4096, topk=10, w_lm=0x10000, R=10, h=0x20000,
                   tok=0x30000, logq=0x40000)

    def call(**kw):
        a = dict(ok_args, **kw)
        return E.eagle3_lm_head_topk_noalloc(a["dtype"], a["vocab"], a["d"], a["topk"], a["w_lm"],
                                             a["R"], a["h"], a["tok"], a["logq"])
    assert call(dtype=7) == E.ERR_INVALID_ARG
    assert call(topk=17) == E.ERR_INVALID_ARG
    assert call(R=0) == E.ERR_INVALID_ARG
    assert call(w_lm=None) == E.ERR_INVALID_ARG
    assert call(w_lm=0x10008) == E.ERR_INVALID_ARG      # TMA needs 16-byte aligned bases
    assert call(d=4100) == E.ERR_INVALID_ARG            # ... and 16-byte rows
    assert call(R=257) == E.ERR_SHAPE                   # tensor-core head: <= 256 rows
    assert call(R=200) == E.ERR_SHAPE                   # partials beyond the 16 MiB scratch


def test_graph_calls_need_a_context(E):
    kv, tree = E.eagle3_kv(), E.eagle3_tree()
    assert E.eagle3_graph_launch(0, 0, 0) == E.ERR_INVALID_ARG
    assert E.eagle3_graph_capture(0, 1, 1, 1, 1, kv, tree, 1, 0, 1.0, 0, 1, 1, 1, 0) == E.ERR_INVALID_ARG


def test_latency_costs_match_scipy_grid_interpolation(E):
    """The warm-up table's lookup is trilinear interpolation clamped at the grid's
    ends: checked against scipy's RegularGridInterpolator (an independent routine)."""
    import numpy as np
    from scipy.interpolate import RegularGridInterpolator
    rng = np.random.default_rng(3)
    batch, prefix, tokens = [1, 4, 16, 64], [256, 1024, 4096], [1, 2, 4, 8, 16, 32, 64]
    shape = (len(batch), len(prefix), len(tokens))
    draft = rng.uniform(50, 500, shape).astype(np.float32)
    verify = rng.uniform(100, 900, shape).astype(np.float32)
    fd = RegularGridInterpolator((batch, prefix, tokens), draft.astype(np.float64))
    fv = RegularGridInterpolator((batch, prefix, tokens), verify.astype(np.float64))

    def at(f, b, p, n):
        pt = [min(max(b, batch[0]), batch[-1]), min(max(p, prefix[0]), prefix[-1]),
              min(max(n, tokens[0]), tokens[-1])]
        return float(f([pt])[0])
    for B, P in ((1, 256), (3, 700), (64, 4096), (100, 9000), (7, 100), (16, 2048)):
        depth, topk, M = 6, 10, 60
        s, pu, vu = E.eagle3_latency_costs(batch, prefix, tokens, draft, verify, B, P, depth, topk, M)
        assert s == E.OK
        np.testing.assert_allclose(pu[0], at(fd, B, P, 1), rtol=1e-5)
        np.testing.assert_allclose(pu[1:], [at(fd, B, P, topk)] * (depth - 1), rtol=1e-5)
        assert vu[0] == 0.0
        np.testing.assert_allclose(vu[1:], [at(fv, B, P, m) for m in range(1, M + 1)], rtol=1e-5)


def test_latency_costs_and_control_reject_bad_arguments(E):
    import numpy as np
    g = np.ones((2, 1, 1), dtype=np.float32)
    assert E.eagle3_latency_costs([4, 1], [8], [1], g, g, 1, 8, 2, 1, 1)[0] == E.ERR_INVALID_ARG
    assert E.eagle3_latency_costs([1, 4], [8], [1], g, g, 1, 8, 0, 1, 1)[0] == E.ERR_INVALID_ARG
    assert E.eagle3_latency_costs([1, 4], [8], [1], g, g, 1, 8, 2, 1, 1)[0] == E.OK
    assert E.eagle3_set_control(0, None) == E.ERR_INVALID_ARG
    assert E.eagle3_set_control(0, E.make_control(tau_depth=1.0)) == E.ERR_INVALID_ARG


def test_draft_noise_needs_a_context(E):
    assert E.eagle3_draft_noise(0, 1, 2, 0) == E.ERR_INVALID_ARG
