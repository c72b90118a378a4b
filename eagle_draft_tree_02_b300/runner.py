"""Python driver for the C ABI: puts a round's inputs in device memory (torch is
used only to allocate and copy), creates a context, runs prefill, draft rounds
and verification through ``eagle3`` and returns the outputs as torch tensors.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import eagle3 as E
from .configs import RoundConfig
from .synth import RoundInputs


def to_device(a: np.ndarray, device) -> torch.Tensor:
    """numpy array (bf16 kept as uint16 bits) -> torch tensor on `device`."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def make_config(cfg: RoundConfig, max_prefix: int, max_new: int = 1, max_batch: int | None = None):
    c = E.eagle3_config()
    c.d, c.n_q_heads, c.n_kv_heads, c.head_dim = cfg.d, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    c.ffn, c.vocab, c.lr_rank, c.lr_cand = cfg.ffn, cfg.vocab, cfg.lr_rank, cfg.lr_cand
    c.rope_theta, c.rms_eps = cfg.rope_theta, cfg.rms_eps
    c.dtype = E.BF16 if cfg.dtype == "bf16" else E.FP32
    c.depth, c.topk, c.n_verify, c.page_size = cfg.depth, cfg.topk, cfg.n_verify, cfg.page_size
    c.max_batch = max_batch or cfg.batch
    c.max_prefix, c.max_new = max_prefix, max_new
    c.variant = ((E.FC_NORM if cfg.fc_norm else 0) | (E.POST_NORM if cfg.post_norm else 0) |
                 (E.SAMPLED_DRAFT if cfg.sampled_draft else 0))
    return c


@dataclass
class TreeOut:
    tokens: torch.Tensor
    parent: torch.Tensor
    depth: torch.Tensor
    pos: torch.Tensor
    pool_index: torch.Tensor
    score: torch.Tensor
    mask: torch.Tensor

    def struct(self) -> E.eagle3_tree:
        t = E.eagle3_tree()
        for n in ("tokens", "parent", "depth", "pos", "pool_index", "score", "mask"):
            setattr(t, n, getattr(self, n).data_ptr())
        return t


@dataclass
class PoolOut:
    tok: torch.Tensor
    parent: torch.Tensor
    depth: torch.Tensor
    fwd: torch.Tensor
    score: torch.Tensor
    logq: torch.Tensor
    cand: torch.Tensor | None = None   # two-stage head: [B, 1 + (D-1)k, lr_cand]

    def struct(self) -> E.eagle3_pool:
        p = E.eagle3_pool()
        for n in ("tok", "parent", "depth", "fwd", "score", "logq", "cand"):
            t = getattr(self, n)
            setattr(p, n, t.data_ptr() if t is not None else None)
        return p


class Engine:
    """One context plus the device copies of one round's inputs and its KV cache."""

    def __init__(self, inputs: RoundInputs, device="cuda", max_new: int = 1, with_target=True,
                 max_prefix_extra: int = 0, page_capacity: tuple | None = None):
        """page_capacity = (logical pages per request, physical pages) sizes a
        paged cache for requests that join and leave the batch; the inputs'
        page table fills the first columns of each request's row."""
        self.inp = inputs
        cfg = self.cfg = inputs.cfg
        self.device = torch.device(device)
        dev = self.device
        self.B = cfg.batch
        self.w = {k: to_device(v, dev) for k, v in inputs.w.items()
                  if with_target or k != "w_target"}
        # contiguous cache: room for the prefix plus rows later rounds commit
        self.max_prefix = int(inputs.prefix_lens.max()) + max_prefix_extra
        if cfg.page_size:
            pt = inputs.page_table.astype(np.int32)
            pages_per_req, n_pages = (pt.shape[1], inputs.n_pages) if page_capacity is None \
                else page_capacity
            table = np.zeros((self.B, pages_per_req), dtype=np.int32)
            table[:, :pt.shape[1]] = pt
            self.max_prefix = pages_per_req * cfg.page_size
        ws = E.eagle3_weights()
        for n in E.WEIGHT_NAMES:
            setattr(ws, n, self.w[n].data_ptr() if n in self.w else None)
        self.cstruct = make_config(cfg, self.max_prefix, max_new)
        s, self.ctx = E.eagle3_create(self.cstruct, ws)
        if s != E.OK:
            raise E.Eagle3Error(s, "eagle3_create")
        self._ws = ws
        # KV cache
        dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        kvd = (cfg.n_kv_heads, cfg.head_dim)
        self.kv = E.eagle3_kv()
        if cfg.page_size:
            self.k_cache = torch.zeros((n_pages, cfg.page_size) + kvd, dtype=dt, device=dev)
            self.v_cache = torch.zeros_like(self.k_cache)
            self.page_table = to_device(table, dev)
            self.kv.page_table = self.page_table.data_ptr()
            self.kv.max_pages = pages_per_req
            self.kv.n_pages = n_pages
        else:
            self.k_cache = torch.zeros((self.B, self.max_prefix) + kvd, dtype=dt, device=dev)
            self.v_cache = torch.zeros_like(self.k_cache)
        self.kv.k, self.kv.v = self.k_cache.data_ptr(), self.v_cache.data_ptr()
        self.seq_lens = torch.zeros(self.B, dtype=torch.int32, device=dev)
        self.kv.seq_lens = self.seq_lens.data_ptr()
        # the round's new row per request: the last prefix row (the root)
        cu = inputs.cu_rows
        last = cu[1:] - 1
        self.feats_all = to_device(inputs.feats, dev)
        self.tokens_all = to_device(inputs.tokens, dev)
        self.cu_rows = to_device(cu.astype(np.int32), dev)
        self.feats_new = self.feats_all[torch.from_numpy(last).to(dev)].unsqueeze(1).contiguous()
        self.tokens_new = self.tokens_all[torch.from_numpy(last).to(dev)].unsqueeze(1).contiguous()
        M1 = cfg.n_verify + 1
        W = (M1 + 31) // 32
        i32 = dict(dtype=torch.int32, device=dev)
        self.tree = TreeOut(*(torch.empty((self.B, M1), **i32) for _ in range(5)),
                            torch.empty((self.B, M1), dtype=torch.float32, device=dev),
                            torch.empty((self.B, M1, W), **i32))
        pn = cfg.pool_size
        cand = (torch.empty((self.B, 1 + (cfg.depth - 1) * cfg.topk, cfg.lr_cand), **i32)
                if cfg.lr_rank else None)
        self.pool = PoolOut(*(torch.empty((self.B, pn), **i32) for _ in range(4)),
                            torch.empty((self.B, pn), dtype=torch.float32, device=dev),
                            torch.empty((self.B, pn), dtype=torch.float32, device=dev), cand)
        D = cfg.depth
        self.accept_len = torch.empty(self.B, **i32)
        self.path = torch.empty((self.B, D), **i32)
        self.out_tokens = torch.empty((self.B, D + 1), **i32)
        f32 = dict(dtype=torch.float32, device=dev)
        self.stats_t = dict(z_max=torch.empty((self.B, M1), **f32), lse=torch.empty((self.B, M1), **f32),
                            z_argmax=torch.empty((self.B, M1), **i32),
                            g_argmax=torch.empty((self.B, M1), **i32))
        # the per-node Gumbel-argmax makes the head draw noise at every node;
        # without it a sampling pass draws only where each walk stops
        self.stats = E.eagle3_verify_stats(*(self.stats_t[n].data_ptr()
                                             for n in ("z_max", "lse", "z_argmax")), None)
        self.stats_g = E.eagle3_verify_stats(*(self.stats_t[n].data_ptr()
                                               for n in ("z_max", "lse", "z_argmax", "g_argmax")))
        self._tree_s = self.tree.struct()
        self._pool_s = self.pool.struct()

    def stream(self) -> int:
        return torch.cuda.current_stream(self.device).cuda_stream

    def close(self):
        if self.ctx:
            E.eagle3_destroy(self.ctx)
            self.ctx = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self):
        """K/V of every prefix row (the root row included; the round rewrites it)."""
        self.seq_lens.zero_()
        rows = int(self.inp.cu_rows[-1])
        s = E.eagle3_prefill(self.ctx, self.B, rows, self.cu_rows.data_ptr(), self.feats_all.data_ptr(),
                             self.tokens_all.data_ptr(), self.kv, self.stream())
        E.check(self.ctx, s)
        self.seq_lens.copy_(torch.from_numpy(self.inp.prefix_lens - 1).to(self.device))

    def set_control(self, depth_cap=None, topk_cap=None, verify_cap=None, **rules):
        """Per-request caps (host int sequences, copied to the device) and the
        cost-aware rules (keyword arguments of eagle3_control); no arguments: off."""
        if depth_cap is None and topk_cap is None and verify_cap is None and not rules:
            E.check(self.ctx, E.eagle3_set_control(self.ctx, None))
            return
        caps = {}
        for name, v in (("depth_cap", depth_cap), ("topk_cap", topk_cap), ("verify_cap", verify_cap)):
            if v is not None:
                caps[name] = torch.tensor(list(v), dtype=torch.int32, device=self.device)
        self._caps = caps  # kept alive while the control is set
        ctl = E.make_control(**{k: t.data_ptr() for k, t in caps.items()}, **rules)
        E.check(self.ctx, E.eagle3_set_control(self.ctx, ctl))

    def draft_round(self, with_pool=True, feats_new=None, tokens_new=None):
        f = self.feats_new if feats_new is None else feats_new
        t = self.tokens_new if tokens_new is None else tokens_new
        s = E.eagle3_draft_round(self.ctx, self.B, 1, f.data_ptr(), t.data_ptr(), self.kv,
                                 self._tree_s, self._pool_s if with_pool else None, self.stream())
        E.check(self.ctx, s)
        return self.tree

    def draft_noise(self, seed, round_id):
        """Seed and round id of the sampled draft's noise for the next rounds."""
        E.check(self.ctx, E.eagle3_draft_noise(self.ctx, seed, round_id, self.stream()))

    def verify(self, temperature=0.0, seed=0, round_id=0, with_stats=True, g_argmax=False):
        """g_argmax: also fill stats_t["g_argmax"] at every node (the head then
        draws the Gumbel noise of every node instead of deferring it)."""
        mode = 0 if temperature == 0 else (2 if self.cfg.sampled_draft else 1)
        stats = (self.stats_g if g_argmax else self.stats) if with_stats else None
        s = E.eagle3_verify(self.ctx, self.B, self._tree_s, self.kv, mode, float(temperature or 1.0),
                            seed, round_id, self.accept_len.data_ptr(), self.path.data_ptr(),
                            self.out_tokens.data_ptr(), stats, self.stream())
        E.check(self.ctx, s)
        return self.accept_len, self.path, self.out_tokens

    def capture(self, temperature=0.0, seed=0, stream=None, with_verify=True):
        """Capture one step (draft round, + verify) into the context's CUDA graph.

        Needs an eager draft round first and a non-default stream; replays read
        the same input and output buffers (self.feats_new, self.tokens_new,
        self.tree, self.accept_len, ...)."""
        mode = 0 if temperature == 0 else (2 if self.cfg.sampled_draft else 1)
        st = stream if stream is not None else self.stream()
        s = E.eagle3_graph_capture(self.ctx, self.B, 1, self.feats_new.data_ptr(),
                                   self.tokens_new.data_ptr(), self.kv, self._tree_s,
                                   1 if with_verify else 0, mode,
                                   float(temperature or 1.0), seed, self.accept_len.data_ptr(),
                                   self.path.data_ptr(), self.out_tokens.data_ptr(), st)
        E.check(self.ctx, s)

    def replay(self, round_id=0, stream=None):
        st = stream if stream is not None else self.stream()
        E.check(self.ctx, E.eagle3_graph_launch(self.ctx, round_id, st))

    def warmup_latency_table(self, reps=3):
        """The EAGLE-Harness warm-up at this engine's batch size and prefix: draft
        rounds under depth caps 1..D give the root pass and the later passes'
        cost (by difference), verification under verify caps 1 and M the verify
        cost.  Returns (batch, prefix, tokens, draft_us, verify_us) for
        eagle3_latency_costs; tokens = [1, k, M] (k and M merged if equal)."""
        cfg, dev = self.cfg, self.device
        st = torch.cuda.current_stream(dev)

        def timed(fn):
            fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            for _ in range(reps):
                fn()
            b.record(st)
            b.synchronize()
            return a.elapsed_time(b) * 1e3 / reps  # microseconds

        t_round = []
        for d in range(1, cfg.depth + 1):
            self.set_control(depth_cap=[d] * self.B)
            t_round.append(timed(lambda: self.draft_round(with_pool=False)))
        self.set_control()
        root = t_round[0]
        # on launch-bound shapes a pass costs nothing measurable: the difference is noise
        later = max(0.0, (t_round[-1] - t_round[0]) / max(1, cfg.depth - 1))
        t_ver = {}
        for m in sorted({1, cfg.n_verify}):
            self.set_control(verify_cap=[m] * self.B)
            self.draft_round(with_pool=False)
            t_ver[m] = timed(lambda: self.verify(0.0, with_stats=False))
        self.set_control()
        tokens = sorted({1, cfg.topk, cfg.n_verify})
        draft = [root if n == 1 else later for n in tokens]
        verify = [t_ver[1] if n == 1 else t_ver[cfg.n_verify] if n >= cfg.n_verify else
                  t_ver[1] + (t_ver[cfg.n_verify] - t_ver[1]) * (n - 1) / max(1, cfg.n_verify - 1)
                  for n in tokens]
        shape = (1, 1, len(tokens))
        return ([self.B], [int(self.max_prefix)], tokens,
                np.asarray(draft, dtype=np.float32).reshape(shape),
                np.asarray(verify, dtype=np.float32).reshape(shape))

    def check(self):
        E.check(self.ctx, E.eagle3_check(self.ctx))

    def launches(self) -> int:
        return E.eagle3_last_launch_count(self.ctx)
