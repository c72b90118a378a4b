"""Continuous batching of draft trees in one paged batch.

"EAGLE-3 精读" §6 names tree drafting under continuous batching as an open
problem, and §4 reports the serving set-up (SGLang, batch 64).  Here a batch
of request slots shares one paged KV cache; between rounds some requests
leave and new ones join their slots.  A join rewrites the slot's row of the
page table with fresh physical pages, resets its committed length, prefills
the new prefix through eagle3_prefill (every other slot contributes zero
rows) and starts drafting from its root, while the other slots continue from
their accepted tokens.  Every slot carries its own depth, branch and verify
caps (read from device arrays when the round runs), so trees of different
shapes share the batch.  After every round each slot's pool, tree, accepted
path and emitted tokens are compared with the oracle's round on that
request's committed rows (conditioned mode, parity.py).

The graph case captures one step (draft round + verification) once and keeps
replaying it while requests are swapped in between replays: the graph reads
the page table, the committed lengths, the caps and the new rows from device
memory, so it stays valid without a new capture.
"""
import numpy as np
import pytest

from eagle_draft_tree_02_b300.configs import by_name
from eagle_draft_tree_02_b300.synth import bf16_bits_from_f64, bf16_bits_to_f32, make_inputs
from oracle import round as R
from parity import TOL, compare_request, gpu_outputs, Report

C0 = by_name("tiny_fp32_b1")
CASES = {
    "fp32": C0.scaled(name="cb_fp32", batch=4, prefix=48, prefix_range=(20, 48), depth=4, topk=3,
                      n_verify=10, page_size=16, lm_std=0.3),
    "bf16": C0.scaled(name="cb_bf16", dtype="bf16", d=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                      ffn=512, vocab=2048, prefix=60, prefix_range=(30, 60), batch=4, depth=4,
                      topk=4, n_verify=12, page_size=16, lm_std=0.3),
}
ROUNDS = 4
LEAVE_AFTER = {0: [1], 1: [0, 3], 2: [2]}   # round -> slots whose request leaves; a new one joins


class Batch:
    """Host bookkeeping of the slots: committed rows, caps and pages of each."""

    def __init__(self, cfg, eng, inp, rng, pages_per_req):
        import torch
        self.cfg, self.eng, self.rng = cfg, eng, rng
        B, ps = cfg.batch, cfg.page_size
        self.pages_per_req = pages_per_req
        table = eng.page_table.cpu().numpy()
        used = set(table[:, :inp.page_table.shape[1]].reshape(-1).tolist())
        self.free = [p for p in rng.permutation(eng.kv.n_pages).tolist() if p not in used]
        for b in range(B):   # room for the rows later rounds commit
            for j in range(inp.page_table.shape[1], pages_per_req):
                table[b, j] = self.free.pop()
        eng.page_table.copy_(torch.from_numpy(table))
        self.table = table
        f32 = inp.feats_f32()
        self.rows_f = [list(f32[inp.cu_rows[b]:inp.cu_rows[b + 1]]) for b in range(B)]
        self.rows_t = [list(inp.tokens[inp.cu_rows[b]:inp.cu_rows[b + 1]]) for b in range(B)]
        k = cfg.topk
        self.caps = dict(depth_cap=[cfg.depth, 2, 3, 1][:B], topk_cap=[k, 1, max(1, k - 1), k][:B],
                         verify_cap=[cfg.n_verify, 4, cfg.n_verify - 3, 2][:B])
        self.request_id = list(range(B))
        self.next_id = B

    def rounded(self, x):
        if self.cfg.dtype == "bf16":
            bits = bf16_bits_from_f64(x)
            return bits, bf16_bits_to_f32(bits)
        return x.astype(np.float32), x.astype(np.float32)

    def control(self):
        return R.Control(**{n: list(v) for n, v in self.caps.items()})

    def write_caps(self):
        import torch
        for n, v in self.caps.items():
            self.eng._caps[n].copy_(torch.tensor(v, dtype=torch.int32))

    def admit(self, b, st):
        """A new request takes slot b: new pages, committed length 0, its prefix
        prefilled except the root row, which the next round appends."""
        import torch
        from eagle_draft_tree_02_b300 import eagle3 as E
        from eagle_draft_tree_02_b300.runner import to_device
        cfg, eng = self.cfg, self.eng
        old = self.table[b].tolist()
        self.free = old + self.free
        self.rng.shuffle(self.free)
        self.table[b] = [self.free.pop() for _ in range(self.pages_per_req)]
        eng.page_table[b].copy_(torch.from_numpy(self.table[b].copy()))
        lo, hi = cfg.prefix_range
        P = int(self.rng.integers(lo, hi + 1))
        bits, f = self.rounded(self.rng.standard_normal((P, 3 * cfg.d)))
        toks = self.rng.integers(0, cfg.vocab, size=P).astype(np.int32)
        self.rows_f[b], self.rows_t[b] = list(f), list(toks)
        eng.seq_lens[b] = 0
        cu = np.zeros(cfg.batch + 1, dtype=np.int32)
        cu[b + 1:] = P - 1
        # device inputs stay referenced until the stream has read them
        ins = [to_device(cu, eng.device), to_device(bits[:P - 1], eng.device),
               to_device(toks[:P - 1], eng.device)]
        s = E.eagle3_prefill(eng.ctx, cfg.batch, P - 1, ins[0].data_ptr(), ins[1].data_ptr(),
                             ins[2].data_ptr(), eng.kv, st)
        assert s == E.OK, E.eagle3_last_error(eng.ctx)
        eng.seq_lens[b] = P - 1
        # the joining request's own caps (the slot's device entries, read at run time)
        k = cfg.topk
        self.caps["depth_cap"][b] = int(self.rng.integers(1, cfg.depth + 1))
        self.caps["topk_cap"][b] = int(self.rng.integers(1, k + 1))
        self.caps["verify_cap"][b] = int(self.rng.integers(1, cfg.n_verify + 1))
        self.write_caps()
        self.request_id[b] = self.next_id
        self.next_id += 1
        torch.cuda.synchronize()
        eng.check()

    def compare(self, gpu, temps, seed, round_id):
        cfg = self.cfg
        w = self.w
        rep = Report()
        ctl = self.control()
        for b in range(cfg.batch):
            F = np.stack(self.rows_f[b]).astype(np.float64)
            T = np.array(self.rows_t[b], dtype=np.int64)
            K, V = R.prefix_kv(w, cfg, F, T)
            compare_request(cfg, w, K, V, F[-1], T[-1], len(T), gpu, b, temps, rep, seed, round_id,
                            ctl=ctl)
        return rep


def _check(rep, cfg, what):
    tol = TOL[cfg.dtype]
    print(what, rep)
    assert not rep.failures, (what, rep)
    assert rep.max_err.get("logq", 0.0) <= tol["logit"], (what, rep)
    assert rep.max_err.get("z_max", 0.0) <= tol["logit"], (what, rep)
    assert len(rep.near_ties) <= 4, (what, rep)


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_requests_join_and_leave_between_rounds(cuda, lib_built, name):
    import torch
    from eagle_draft_tree_02_b300 import eagle3 as E
    from eagle_draft_tree_02_b300.runner import Engine, to_device
    cfg = CASES[name]
    D, B, ps = cfg.depth, cfg.batch, cfg.page_size
    inp = make_inputs(cfg, seed=61)
    pages_per_req = -(-(cfg.prefix_range[1] + ROUNDS * (D + 1)) // ps)
    eng = Engine(inp, max_new=D + 1, page_capacity=(pages_per_req, 4 * B * pages_per_req))
    eng.prefill()
    rng = np.random.default_rng(5)
    bt = Batch(cfg, eng, inp, rng, pages_per_req)
    bt.w = R.weights_f32(inp)
    eng.set_control(**bt.caps)
    st = eng.stream()
    temps = (1.0, 0.0)   # greedy last: its outputs feed the next round
    counts = [1] * B
    new_f = [[bt.rows_f[b][-1]] for b in range(B)]
    new_bits = [None] * B
    joined = set()
    for rnd in range(ROUNDS):
        # the round's new rows (already appended to each request's history)
        total = sum(counts)
        cu = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        fb = np.concatenate([np.asarray(new_bits[b]) if new_bits[b] is not None else
                             bt.rounded(np.asarray(new_f[b], dtype=np.float64))[0] for b in range(B)])
        tk = np.concatenate([np.array(bt.rows_t[b][-counts[b]:], dtype=np.int32) for b in range(B)])
        ins = [to_device(cu, cuda), to_device(fb, cuda), to_device(tk, cuda)]  # kept alive
        s = E.eagle3_draft_round_ragged(eng.ctx, B, total, ins[0].data_ptr(), ins[1].data_ptr(),
                                        ins[2].data_ptr(), eng.kv, eng._tree_s, eng._pool_s, st)
        assert s == E.OK, E.eagle3_last_error(eng.ctx)
        gpu = gpu_outputs(eng, temps, lambda T: eng.verify(T, 9, rnd))
        del ins
        _check(bt.compare(gpu, temps, 9, rnd), cfg, f"round {rnd} ids {bt.request_id}")
        # the caps held on the device
        kept = (gpu.tree["tokens"][:, 1:] >= 0).sum(axis=1)
        assert (kept <= np.asarray(bt.caps["verify_cap"])).all()
        # commit the round's rows
        eng.seq_lens += torch.tensor(counts, dtype=torch.int32, device=cuda)
        acc = gpu.verify[0.0]["accept_len"]
        outs = gpu.verify[0.0]["out_tokens"]
        leaving = LEAVE_AFTER.get(rnd, [])
        for b in leaving:
            bt.admit(b, st)
            joined.add(bt.request_id[b])
        for b in range(B):
            if b in leaving:
                counts[b] = 1
                new_bits[b] = None
                new_f[b] = [bt.rows_f[b][-1]]
                continue
            n = int(acc[b]) + 1
            toks = [int(x) for x in outs[b][:n]]
            bits, f = bt.rounded(rng.standard_normal((n, 3 * cfg.d)))
            bt.rows_f[b] += list(f)
            bt.rows_t[b] += toks
            counts[b] = n
            new_bits[b] = bits
    assert len(joined) == 4
    eng.set_control()
    eng.close()


@pytest.mark.gpu
def test_graph_replays_across_joins(cuda, lib_built):
    """One captured step serves requests that join between replays."""
    import torch
    from eagle_draft_tree_02_b300.runner import Engine, to_device
    cfg = CASES["bf16"]
    D, B, ps = cfg.depth, cfg.batch, cfg.page_size
    inp = make_inputs(cfg, seed=67)
    pages_per_req = -(-cfg.prefix_range[1] // ps) + 1
    eng = Engine(inp, page_capacity=(pages_per_req, 3 * B * pages_per_req))
    eng.prefill()
    rng = np.random.default_rng(8)
    bt = Batch(cfg, eng, inp, rng, pages_per_req)
    bt.w = R.weights_f32(inp)
    eng.set_control(**bt.caps)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        st = eng.stream()
        eng.draft_round(with_pool=False)
        eng.verify(0.0, seed=3, round_id=0, with_stats=False)
        eng.capture(temperature=0.0, seed=3)
        for rep_i, joins in enumerate(([], [2], [0, 1], [3])):
            for b in joins:
                bt.admit(b, st)
                # the slot's new row in the captured input buffers: its root row
                f = np.asarray(bt.rows_f[b][-1], dtype=np.float64)
                bits, _ = bt.rounded(f[None])
                eng.feats_new[b].copy_(to_device(bits, cuda))
                eng.tokens_new[b, 0] = int(bt.rows_t[b][-1])
            eng.replay(rep_i)
            torch.cuda.current_stream().synchronize()
            eng.check()
            gpu_t = {k: getattr(eng.tree, k).cpu().numpy() for k in
                     ("tokens", "parent", "depth", "pos", "pool_index", "score", "mask")}
            rep = Report()
            ctl = bt.control()
            w = bt.w
            for b in range(B):
                F = np.stack(bt.rows_f[b]).astype(np.float64)
                T = np.array(bt.rows_t[b], dtype=np.int64)
                K, V = R.prefix_kv(w, cfg, F, T)
                rr = R.round_request(w, cfg, K, V, F[-1], T[-1], len(T) - 1, temperatures=(0.0,),
                                     b=b, ctl=ctl, B=B)
                if not np.array_equal(rr.tree.tok, gpu_t["tokens"][b]):
                    rep.failures.append(("tree", rep_i, b))
                res = rr.verify[0.0]
                if int(eng.accept_len[b]) != res.accept_len:
                    rep.failures.append(("accept_len", rep_i, b))
                if [int(x) for x in eng.out_tokens[b].cpu().numpy() if x >= 0] != res.out_tokens:
                    rep.failures.append(("out_tokens", rep_i, b))
            print("replay", rep_i, "ids", bt.request_id, rep)
            assert not rep.failures, rep
    eng.set_control()
    eng.close()
