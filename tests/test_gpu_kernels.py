"""Kernel-level GPU tests through the C ABI (no whole round).

* eagle3_linear runs the context's GEMM kernel (tcgen05 for bf16 storage, the
  CUDA-core fp32 kernel for fp32) on every weight matrix; compared with a
  float64 product of the same stored values.  Row counts cover one column of
  MMA (R=1), ragged tails, the 256-row tile limit and two column tiles.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import make_inputs

C0 = by_name("tiny_fp32_b1")
LIN_BF16 = C0.scaled(name="lin_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                     ffn=512, vocab=1000, prefix=400, batch=2, depth=3, topk=4, n_verify=8,
                     lm_std=0.08)
# the fp32 context needs a prefix long enough for 300 rows of row capacity
LIN_FP32 = C0.scaled(name="lin_fp32", prefix=400)
NAMES = ["w_fc", "w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down", "w_lm", "w_target"]


@pytest.fixture(scope="module")
def lin_engines(cuda, lib_built):
    from eagle_draft_tree_02_b300.runner import Engine
    out = {}
    for cfg in (LIN_BF16, LIN_FP32):
        inp = make_inputs(cfg, seed=21)
        out[cfg.dtype] = (inp, Engine(inp))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("R", [1, 10, 16, 17, 61, 200, 256, 300])
def test_linear_matches_fp64(lin_engines, dtype, R):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    inp, eng = lin_engines[dtype]
    if R > min(eng.cstruct.max_batch * eng.cstruct.max_prefix, 2048):
        pytest.skip("beyond this context's row capacity")
    rng = np.random.default_rng(R)
    for which, name in enumerate(NAMES):
        W = inp.f32(name).astype(np.float64)
        N, K = W.shape
        x = rng.standard_normal((R, K)).astype(np.float32)
        if dtype == "bf16":
            xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
            x64 = xd.float().cpu().numpy().astype(np.float64)
        else:
            xd = torch.from_numpy(x).cuda()
            x64 = x.astype(np.float64)
        y = torch.empty((R, N), dtype=torch.float32, device="cuda")
        s = E.eagle3_linear(eng.ctx, which, R, xd.data_ptr(), y.data_ptr(), eng.stream())
        assert s == E.OK, (name, E.eagle3_last_error(eng.ctx))
        torch.cuda.synchronize()
        eng.check()
        ref = x64 @ W.T
        err = np.abs(y.cpu().numpy() - ref).max()
        scale = np.abs(ref).max()
        assert err <= 1e-5 * max(1.0, scale) * np.sqrt(K), (name, R, err, scale)
