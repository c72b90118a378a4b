#!/usr/bin/env python
"""Throughput of one EAGLE-3 draft-and-verify round on B300, as one JSON line.

A step is the whole hot path on one batch: the draft round (fusion, D decoder
passes with tree attention, fused LM-head top-k, frontier expansion, global
top-M tree) followed by verification (the tree-masked verify pass, the target
head and the accept/sample walk).  Inputs are seeded synthetic tensors with the
shapes of the named workload, resident in HBM before timing; the prefix is
prefilled once, outside the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU as an
independent replica (disjoint requests, no collective on the data path); the
timed region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "llama31_8b_b1_tree"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload summary of the other full-size workloads")
    ap.add_argument("--variant", default="none", choices=["none", "fc_post", "sampled"],
                    help="drafter variant: FC norm + post-norm, or sampled drafting with q-ratio "
                         "verification (the headline is 'none')")
    ap.add_argument("--control", default="none", choices=["none", "caps"],
                    help="per-request control: 'caps' halves every request's depth and verify count")
    ap.add_argument("--prefix-scale", type=float, default=1.0,
                    help="scale the prefix lengths (a small case of the same kernels for profiling; "
                         "the bench line is only valid at 1.0)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [ln.split(",") for ln in open(self.f.name).read().splitlines() if ln.strip()]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows if len(r) >= 9 for n, v in zip(names, r[5:9])
                          if v.strip() == "Active"})
        busy = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def job_rate(local_ms: float, steps: int, world: int, dist=None, device=None):
    """Whole-job rate of independent replicas: the slowest rank's time bounds the job.

    Returns (max_ms over ranks, rounds/s of all ranks together).  Every rank
    runs `steps` rounds of its own requests; no data crosses ranks.
    """
    ms = float(local_ms)
    if world > 1:
        import torch
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * steps / (ms / 1e3)


def step_temperature(cfg):
    hot = [t for t in cfg.temperatures if t > 0]
    return hot[0] if hot else 0.0


class OracleRound:
    """One oracle round (draft + verify) of request 0 on the host cores.

    The prefix K/V (setup, like the GPU's prefill) is computed once, outside
    the timed calls; each call times the round itself.
    """

    def __init__(self, cfg, inp):
        from oracle import round as R
        self.R, self.cfg = R, cfg
        self.w = R.weights_f32(inp)
        f = inp.feats_f32()
        lo, hi = int(inp.cu_rows[0]), int(inp.cu_rows[1])
        self.K, self.V = R.prefix_kv(self.w, cfg, f[lo:hi], inp.tokens[lo:hi])
        self.feat_root, self.tok_root, self.root_pos = f[hi - 1], inp.tokens[hi - 1], hi - lo - 1
        self.T = step_temperature(cfg)

    def __call__(self, round_id=0) -> float:
        t0 = time.perf_counter()
        self.R.round_request(self.w, self.cfg, self.K, self.V, self.feat_root, self.tok_root,
                             self.root_pos, temperatures=(self.T,), seed=0, round_id=round_id)
        return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return len(os.sched_getaffinity(0))


def run_reference(args, cfg):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from eagle_draft_tree_02_b300.synth import make_inputs
    inp = make_inputs(cfg)
    oracle = OracleRound(cfg, inp)
    budget = 120.0
    warm = min(args.warmup, 1)
    for i in range(warm):
        oracle(i)
    times = []
    for i in range(args.steps):
        times.append(oracle(warm + i))
        if sum(times) > budget:
            break
    # B requests per round on the GPU; the oracle sample is request 0, so scale to the batch
    per_round = sum(times) / len(times) * cfg.batch
    value = 1.0 / per_round
    cores = blas_threads()
    sample = (f"{len(times)} oracle round(s) of request 0 (draft D={cfg.depth} passes + verify at "
              f"T={oracle.T}), scaled by B={cfg.batch}; prefix K/V computed once, untimed; "
              f"{warm} warm-up")
    print(json.dumps({
        "impl": "reference", "metric": "draft-tree rounds/s", "value": value, "unit": "rounds/s",
        "n_gpus": args.gpus, "steps": len(times), "warmup": warm, "ms_per_step": per_round * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": cfg.name},
        "cpu_baseline": {"value": value, "unit": "rounds/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def prefill_flops(cfg, rows: int) -> int:
    """Tensor-core FLOPs of prefilling `rows` prefix rows: the fusion GEMM (3d -> d)
    and the K/V projections (2d -> 2 Hkv dh); a prefix row needs no query."""
    kvd = cfg.n_kv_heads * cfg.head_dim
    return 2 * rows * (3 * cfg.d * cfg.d + 2 * cfg.d * 2 * kvd)


def timed(fn, n):
    """CUDA-event milliseconds of n calls on the current stream."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        fn(i)
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1)


def measure_workload(cfg, args, dev, side, world=1, dist=None, barrier=lambda: None,
                     full=True, steps=None, warmup=None):
    """Graph-replay step rate of one workload (inputs resident in HBM), the
    draft-only rate and their HBM fractions; with `full`, also the roofline
    of the draft head, the prefill, the caller-logits verification and the
    end-to-end rate through the ABI with host buffers."""
    import numpy as np
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.roofline import head_bytes, round_bytes
    from eagle_draft_tree_02_b300.runner import Engine
    from eagle_draft_tree_02_b300.synth import make_inputs

    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    inp = make_inputs(cfg, seed=None)
    eng = Engine(inp, device=dev)
    torch.cuda.synchronize()   # the inputs' copies are complete before the side stream reads them
    torch.cuda.set_stream(side)
    eng.prefill()
    if cfg.sampled_draft:
        eng.draft_noise(0, 0)
    if args.control == "caps":
        eng.set_control(depth_cap=[max(1, cfg.depth // 2)] * cfg.batch,
                        verify_cap=[max(1, cfg.n_verify // 2)] * cfg.batch)
    torch.cuda.synchronize()
    eng.check()
    T = step_temperature(cfg)
    hbm, tflops, src = peaks()

    def step_eager(i):
        eng.draft_round(with_pool=False)
        eng.verify(T, seed=0, round_id=i, with_stats=False)

    for i in range(warmup):
        step_eager(i)
    # the draft round alone as a CUDA graph, for the draft-only rate
    nd = max(10, steps // 2)
    eng.capture(temperature=T, seed=0, with_verify=False)
    for i in range(3):
        eng.replay(round_id=i)
    draft_ms = timed(lambda i: eng.replay(round_id=i), nd) / nd
    # the step as one CUDA graph (eagle3_graph_capture / eagle3_graph_launch)
    eng.capture(temperature=T, seed=0)
    for i in range(3):
        eng.replay(round_id=i)
    torch.cuda.synchronize()
    eng.check()
    barrier()
    torch.cuda.synchronize()
    launches = {"n": 0}

    def step_graph(i):
        eng.replay(round_id=warmup + i)
        launches["n"] += eng.launches()

    ms = timed(step_graph, steps)
    barrier()
    torch.cuda.synchronize()
    eng.check()
    ms, value = job_rate(ms, steps, world, dist, dev)
    ms_per_step = ms / steps
    rb = round_bytes(cfg, prefix_mean=float(np.mean(inp.prefix_lens)))
    out = {
        "value": value, "ms_per_step": ms_per_step, "launches": launches["n"], "T": T, "rb": rb,
        "draft_ms": draft_ms,
        "summary": {
            "rounds_per_s": round(value, 2), "ms_per_step": round(ms_per_step, 4),
            "draft_rounds_per_s_draft_only": round(world * 1e3 / draft_ms, 2),
            "draft_tokens_per_s": round(value * cfg.batch * cfg.n_verify, 1),
            "step_hbm_frac": round(rb["step"] / (ms_per_step / 1e3) / 1e9 / hbm, 4),
            "draft_hbm_frac": round(rb["draft"] / (draft_ms / 1e3) / 1e9 / hbm, 4),
            "verify": f"T={T}" if T else "greedy", "batch": cfg.batch, "dtype": cfg.dtype},
    }
    if not full:
        eng.close()
        return out
    stream = side.cuda_stream
    # the same step as eager calls, for reference
    out["eager_ms"] = timed(lambda i: step_eager(10 ** 5 + i), nd) / nd

    # dominant kernel: the draft LM head with its fused softmax/top-k, on B*k rows
    Rh = cfg.batch * cfg.topk
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    h = torch.randn(Rh, cfg.d, device=dev).to(dt)
    tok = torch.empty((Rh, cfg.topk), dtype=torch.int32, device=dev)
    lq = torch.empty((Rh, cfg.topk), dtype=torch.float32, device=dev)
    for _ in range(5):
        E.check(eng.ctx, E.eagle3_lm_head_topk(eng.ctx, Rh, h.data_ptr(), tok.data_ptr(), lq.data_ptr(),
                                               None, stream))
    nh = 50
    head_s = timed(lambda i: E.eagle3_lm_head_topk(eng.ctx, Rh, h.data_ptr(), tok.data_ptr(),
                                                   lq.data_ptr(), None, stream), nh) / nh / 1e3
    hb = head_bytes(cfg, Rh)
    achieved = hb / head_s / 1e9
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        try:
            import hashlib
            j = json.load(open(tp))
            src_hash = hashlib.sha256(open(os.path.join(ROOT, "eagle_draft_tree_02_b300", "csrc",
                                                        "gemm_tc.cu"), "rb").read()).hexdigest()[:16]
            e = j.get("lm_head", {})
            if e.get("source_sha256_16") == src_hash and e.get("config") == cfg.name:
                traffic = e.get("dram_bytes_per_launch")
        except Exception:
            traffic = None
    head_kernel = ("tc_head_kernel<1> + topk_merge_kernel (draft LM head, fused softmax/top-k)"
                   if cfg.dtype == "bf16" and not cfg.lr_rank else
                   "two-stage head (low-rank sample/append + select/rescore)" if cfg.lr_rank else
                   "lm_head_simt_kernel + topk_merge_kernel")
    # the head's share of the timed step: its launches per step at the isolated launch time
    head_per_step = cfg.depth
    out["roofline"] = {
        "bound": "hbm", "kernel": head_kernel, "achieved": round(achieved, 1), "peak": hbm,
        "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": src,
        "algorithmic_bytes_per_launch": hb, "launch_us": round(head_s * 1e6, 2),
        "launches_per_step": head_per_step,
        "share_of_step": round(head_per_step * head_s * 1e3 / ms_per_step, 4)}

    # prefill: every prefix row's K/V through the tensor-core GEMMs (untimed set-up of
    # the round, timed here on its own against the bf16 tensor peak)
    rows = int(inp.cu_rows[-1])
    committed = eng.seq_lens.clone()
    eng.seq_lens.zero_()

    def prefill(i):
        E.check(eng.ctx, E.eagle3_prefill(eng.ctx, cfg.batch, rows, eng.cu_rows.data_ptr(),
                                          eng.feats_all.data_ptr(), eng.tokens_all.data_ptr(),
                                          eng.kv, stream))
    prefill(0)
    pf_ms = timed(prefill, 3) / 3
    eng.seq_lens.copy_(committed)
    fl = prefill_flops(cfg, rows)
    out["prefill"] = {"rows": rows, "ms": round(pf_ms, 4), "tflop": round(fl / 1e12, 4),
                      "tflops": round(fl / (pf_ms / 1e3) / 1e12, 1), "bound": "tensor",
                      "peak_tflops": tflops,
                      "frac_of_bf16_peak": round(fl / (pf_ms / 1e3) / 1e12 / tflops, 4)}
    # the prefill rewrote the same K/V rows with the same values
    torch.cuda.synchronize()
    eng.check()

    # verification against caller-supplied target logits [B, M+1, V] (bf16): the tree of
    # the last step, greedy and at the step's temperature
    M1 = cfg.n_verify + 1
    logits = torch.randn(cfg.batch * M1, cfg.vocab, device=dev).to(torch.bfloat16)
    vl = {}
    for Tv in sorted({0.0, T}):
        mode = 0 if Tv == 0 else 1

        def call(i, mode=mode, Tv=Tv):
            E.check(eng.ctx, E.eagle3_verify_logits(
                eng.ctx, cfg.batch, eng._tree_s, logits.data_ptr(), E.BF16, cfg.vocab, mode,
                float(Tv or 1.0), 0, i, eng.accept_len.data_ptr(), eng.path.data_ptr(),
                eng.out_tokens.data_ptr(), None, stream))
        for i in range(3):
            call(i)
        # GPU time of the call: its four kernels captured once and replayed
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            call(7)
        for i in range(3):
            graph.replay()
        us = timed(lambda i: graph.replay(), 20) / 20 * 1e3
        del graph
        lb = logits.numel() * 2
        vl["greedy" if mode == 0 else f"T={Tv}"] = {
            "us": round(us, 2), "logits_bytes": lb, "gbs": round(lb / (us / 1e6) / 1e9, 1),
            "hbm_frac": round(lb / (us / 1e6) / 1e9 / hbm, 4)}
    out["verify_logits"] = vl

    # end to end through the ABI with host buffers: each step copies its new rows
    # from pinned host memory into the captured input buffers, replays the graph
    # and reads the accepted lengths and tokens back
    fh = eng.feats_new.cpu().pin_memory()
    th = eng.tokens_new.cpu().pin_memory()
    out_h = torch.empty((cfg.batch, cfg.depth + 2), dtype=torch.int32).pin_memory()
    ne = max(10, steps // 2)
    for i in range(3 + ne):
        if i == 3:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        eng.feats_new.copy_(fh, non_blocking=True)
        eng.tokens_new.copy_(th, non_blocking=True)
        eng.replay(round_id=10 ** 6 + i)
        out_h[:, 0].copy_(eng.accept_len, non_blocking=True)
        out_h[:, 1:].copy_(eng.out_tokens, non_blocking=True)
        side.synchronize()
    e2e_s = (time.perf_counter() - t0) / ne
    out["e2e"] = {"value": round(world / e2e_s, 3), "unit": "rounds/s",
                  "h2d_bytes_per_step": fh.numel() * fh.element_size() + th.numel() * th.element_size(),
                  "d2h_bytes_per_step": out_h.numel() * out_h.element_size()}
    out["inp"] = inp
    eng.close()
    return out


def main():
    args = parse()
    from eagle_draft_tree_02_b300.configs import CONFIGS, by_name
    cfg = by_name(args.config)
    if args.prefix_scale != 1.0:
        sc = args.prefix_scale
        rng = cfg.prefix_range
        cfg = cfg.scaled(prefix=max(2, int(cfg.prefix * sc)),
                         prefix_range=None if rng is None else (max(2, int(rng[0] * sc)),
                                                                max(2, int(rng[1] * sc))))
    if args.variant == "fc_post":
        cfg = cfg.scaled(fc_norm=True, post_norm=True)
    elif args.variant == "sampled":
        cfg = cfg.scaled(sampled_draft=True)
    if args.impl == "reference":
        run_reference(args, cfg)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    # every launch goes to one non-default stream: a CUDA graph is captured on it
    side = torch.cuda.Stream(dev)
    sampler = ClockSampler(local)
    sampler.start()
    r = measure_workload(cfg, args, dev, side, world, dist, barrier)
    clocks = sampler.stop()
    hbm, tflops, src = peaks()
    rb, T = r["rb"], r["T"]
    line = {
        "metric": "draft-tree rounds/s", "value": round(r["value"], 3), "unit": "rounds/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(r["ms_per_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic (seeded weights, features, tokens; no trained model)",
        "config": {"workload": cfg.name, "batch": cfg.batch, "prefix": cfg.prefix, "d": cfg.d,
                   "prefix_scale": args.prefix_scale,
                   "variant": args.variant, "control": args.control,
                   "vocab": cfg.vocab, "depth": cfg.depth, "topk": cfg.topk, "n_verify": cfg.n_verify,
                   "verify": f"T={T}" if T else "greedy",
                   "l2": f"inputs larger than L2: {rb['step'] / 1e9:.2f} GB of weights/KV streamed per step"},
        "draft_tokens_per_s": r["summary"]["draft_tokens_per_s"],
        "step": "eagle3_graph_launch: one CUDA graph of eagle3_draft_round + eagle3_verify",
        "eager_ms_per_step": round(r["eager_ms"], 4),
        "draft_rounds_per_s_draft_only": r["summary"]["draft_rounds_per_s_draft_only"],
        "step_algorithmic_bytes": rb["step"],
        "step_hbm_frac": r["summary"]["step_hbm_frac"],
        "draft_hbm_frac": r["summary"]["draft_hbm_frac"],
        "roofline": r["roofline"],
        "prefill": r["prefill"],
        "verify_logits": r["verify_logits"],
        "e2e": r["e2e"],
        "gpu_launches": r["launches"],
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t = OracleRound(cfg, r["inp"])()
        line["cpu_baseline"] = {"value": round(1.0 / (t * cfg.batch), 6), "unit": "rounds/s",
                                "cores": blas_threads(), "kind": "oracle",
                                "sample": f"1 oracle round of request 0 (draft + verify at T={T}), "
                                          f"scaled by B={cfg.batch}; prefix K/V precomputed"}
    del r
    if world == 1 and not args.no_workloads and args.prefix_scale == 1.0 and args.variant == "none" \
            and args.control == "none":
        # the other workloads, each as a graph-replayed step on the same GPU (own clock record)
        others = {}
        for c in CONFIGS:
            if c.name == cfg.name or c.dtype != "bf16":  # the fp32 tiny case is a test shape
                continue
            sampler = ClockSampler(local)
            sampler.start()
            o = measure_workload(c, args, dev, side, full=False, steps=min(args.steps, 20),
                                 warmup=min(args.warmup, 3))
            others[c.name] = dict(o["summary"], clocks=sampler.stop())
            del o
            torch.cuda.empty_cache()
        line["workloads"] = others
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
