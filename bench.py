"""Benchmark of one Medusa decode step on GB300.

Workload: the Vicuna-7B-shaped batch-1 step (hidden 4096, vocab 32000, 5 heads,
top-8 per head, 64-node sparse tree, 32 query heads x 128 head dim, KV length
2048, bf16 storage, greedy acceptance with planted alpha = 0.8, then KV
compaction), with seeded synthetic inputs and random-init weights of that shape.

A step is one pass of the whole hot path through the C ABI:
  medusa_heads_topk -> medusa_build_tree -> medusa_tree_attention (one layer)
  -> medusa_verify_accept_tree -> medusa_kv_compact
with every input resident in HBM.  The step reads ~1.52 GB, more than L2, so
consecutive steps start cold.  kv_len is restored before each step (compaction
grows it) so every step sees the same workload.

Beside the step, the JSON line carries:
  step_graph_32_layers  the step as one CUDA graph with tree attention over 32
                        layers' caches, and the per-layer attention time
  chained_rounds        16 chained rounds as one CUDA graph (root = the last
                        next token, heads on h_next, kv_len growing), with 1 and
                        32 attention layers: tokens per wall-second
  tree_sizes            the step with the sparse 64-node and the dense 341-node
                        tree at equal planted acceptance
  workload_steps        whole steps of the 13B-shaped ragged batch-8 workload and
                        of the batch-4 KV-8192 workload (sparse and dense tree,
                        typical acceptance): steps/s and tree tokens/s
  verify_projection     the fused verification projection (lm_head x tree
                        hidden states on the tensor cores, reduced to acceptance)
  attention_workloads   tree attention alone at the batched shapes
  chain_sweep           speculative-sampling acceptance at batch 64, vocab
                        128256, sigma 0.1/0.5/1.0 x gamma 0..32, 64 rounds each:
                        measured alpha and tokens per round against E
  chain_acceptance      that call's HBM roofline at gamma 1/4/8/32
  heads_batches         the heads alone at batch 1-64
  cpu_baseline          the float64 C oracle on the host cores

Prints one JSON line (rank 0).  --impl reference runs the oracle's full step
instead: --warmup then --steps steps, spread over the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

CFG = W.WORKLOADS["h4096_b1_sparse64"]
METRIC = "Medusa decode steps/s (tree tokens verified/s = steps/s x 64 nodes)"
WORKLOAD = ("vicuna7b-shaped medusa step, batch 1: hidden 4096, vocab 32000, 5 heads, top-8, "
            "sparse 64-node tree, 32x128 attention over KV 2048 (one layer), greedy acceptance, "
            "KV compaction; bf16 storage, fp32 accumulate")

# DRAM bytes per launch of the heads call, from the ncu capture summarised in
# profiles/ (dram__bytes_read.sum + dram__bytes_write.sum summed over its three
# kernels), with the sha1 of heads.cu it was taken on; null once that file changes.
HEADS_TRAFFIC = {"sha1": "0767f4c9c673445c393a5d345066140df4f30dee", "bytes": 1478950826}


def _sha1(path):
    with open(path, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tpeak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def _tree_tables():
    import medusa_speculative_decoding_gb300 as M
    paths = M.sparse_tree_paths(64, 5, 8, 0.6, 0.5)
    return M.tree_layout(paths, 5)


def make_inputs(seed=None):
    seed = CFG["seed"] if seed is None else seed
    c = CFG
    t = _tree_tables()
    N = t["N"]
    heads = W.heads_inputs(seed, c["B"], c["H"], c["V"], c["K"], c["dtype"])
    kv_len = W.kv_lengths(seed, c["B"], c["L_lo"], c["L_hi"])
    Lmax = c["L_hi"] + N
    att = W.attention_inputs(seed, c["B"], N, c["Hq"], c["Hkv"], c["D"], Lmax, c["dtype"])
    ht = W.hidden_tree(seed, c["B"], N, c["H"], c["dtype"])
    root = W.root_tokens(seed, c["B"], c["V"])
    return dict(tree=t, heads=heads, kv_len=kv_len, Lmax=Lmax, att=att, ht=ht, root=root)


def algorithmic_bytes(c, N, Lmax_used):
    K, H, V, B = c["K"], c["H"], c["V"], c["B"]
    heads = K * (H * H + H + V * H) * 2 + B * H * 2 + B * K * c["topk"] * 8
    att = 2 * c["Hkv"] * Lmax_used * c["D"] * 2 * B + B * N * c["Hq"] * c["D"] * (2 + 4)
    verify = B * N * c["V"] * 4 + B * N * 4
    return heads, att, verify


# ----------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
class Step:
    """Device buffers and the five C-ABI calls of one decode step."""

    def __init__(self, inp, device):
        import torch
        import medusa_speculative_decoding_gb300 as M
        self.M, self.torch = M, torch
        c = CFG
        t = inp["tree"]
        self.t = t
        self.N, self.Dmax = t["N"], t["max_depth"]
        dev = device

        def td(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
            if a.dtype == np.uint64:
                return torch.from_numpy(a.view(np.int64)).to(dev)
            return torch.from_numpy(a).to(dev)

        self.td = td
        hd = inp["heads"]
        self.h, self.w1, self.b1, self.w2 = (td(hd[k]) for k in ("h", "w1", "b1", "w2"))
        self.root = td(inp["root"])
        self.depth, self.rank, self.parent = td(t["depth"]), td(t["rank"]), td(t["parent"])
        self.mask = td(t["mask"])
        self.scale = 1.0 / float(np.sqrt(c["D"]))  # the softmax scale of the attention layer
        self.q = td(inp["att"]["q"])
        self.kc, self.vc = td(inp["att"]["k_cache"]), td(inp["att"]["v_cache"])
        self.kv_len0 = td(inp["kv_len"])
        self.kv_len = self.kv_len0.clone()
        self.ht = td(inp["ht"])
        B, K, topk, V = c["B"], c["K"], c["topk"], c["V"]
        i32 = torch.int32
        self.idx = torch.empty((B, K, topk), dtype=i32, device=dev)
        self.val = torch.empty((B, K, topk), dtype=torch.float32, device=dev)
        self.cand = torch.empty((B, self.N), dtype=i32, device=dev)
        self.att_out = torch.empty((B, self.N, c["Hq"], c["D"]), dtype=torch.float32, device=dev)
        self.acc = dict(accept_len=torch.empty(B, dtype=i32, device=dev),
                        best_node=torch.empty(B, dtype=i32, device=dev),
                        path_nodes=torch.empty((B, self.Dmax + 1), dtype=i32, device=dev),
                        next_tok=torch.empty(B, dtype=i32, device=dev))
        self.h_next = torch.empty((B, c["H"]), dtype=torch.bfloat16, device=dev)
        self.src = torch.empty((B, self.Dmax + 1), dtype=i32, device=dev)
        u8 = torch.uint8
        self.ws_heads = torch.empty(max(16, M.heads_topk_workspace(B, K, c["H"], V, topk)), dtype=u8, device=dev)
        self.ws_att_n = M.tree_attention_workspace(B, self.N, c["Hq"], c["Hkv"], c["D"], inp["Lmax"])
        self.ws_att = torch.empty(max(16, self.ws_att_n), dtype=u8, device=dev)
        self.ws_ver = torch.empty(max(16, M.verify_accept_workspace(B, self.N, V)), dtype=u8, device=dev)
        # verifier logits planted around this step's own candidates (setup, untimed)
        self.heads()
        self.M.build_tree(self.idx, self.root, self.depth, self.rank, out=self.cand)
        cand = self.cand.cpu().numpy()
        self.vlogits = td(W.planted_logits(CFG["seed"], cand, t["parent"], V, c["alpha"]))
        # heads 2 (W1, W2 with the merge) + tree 1 + attention 1-2 + verify 2 + compaction 1
        self.launches = 2 + 1 + (2 if self.ws_att_n > 0 else 1) + 2 + 1

    def with_tree(self, t, seed=3):
        """A copy of this step that verifies tree `t` instead (same weights, batch,
        KV length and planted acceptance): tree tables, queries, caches with
        room for the tree, tree hidden states and verifier logits planted around
        the new tree's candidates.  Set-up only; nothing here is timed."""
        import copy
        torch, M, c = self.torch, self.M, CFG
        s = copy.copy(self)
        dev = self.h.device
        B, V = c["B"], c["V"]
        s.t = t
        s.N, s.Dmax = t["N"], t["max_depth"]
        s.depth, s.rank, s.parent = self.td(t["depth"]), self.td(t["rank"]), self.td(t["parent"])
        s.mask = self.td(t["mask"])
        Lmax = int(self.kv_len0.max().item()) + s.N
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        s.q = torch.randn((B, s.N, c["Hq"], c["D"]), device=dev, generator=g).to(self.q.dtype)
        s.kc = torch.randn((B, c["Hkv"], Lmax, c["D"]), device=dev, generator=g).to(self.kc.dtype)
        s.vc = torch.randn((B, c["Hkv"], Lmax, c["D"]), device=dev, generator=g).to(self.vc.dtype)
        s.ht = torch.randn((B, s.N, c["H"]), device=dev, generator=g).to(self.ht.dtype)
        s.kv_len = self.kv_len0.clone()
        i32 = torch.int32
        s.cand = torch.empty((B, s.N), dtype=i32, device=dev)
        s.att_out = torch.empty((B, s.N, c["Hq"], c["D"]), dtype=torch.float32, device=dev)
        s.acc = dict(accept_len=torch.empty(B, dtype=i32, device=dev), best_node=torch.empty(B, dtype=i32, device=dev),
                     path_nodes=torch.empty((B, s.Dmax + 1), dtype=i32, device=dev),
                     next_tok=torch.empty(B, dtype=i32, device=dev))
        s.h_next = torch.empty_like(self.h_next)
        s.src = torch.empty((B, s.Dmax + 1), dtype=i32, device=dev)
        s.ws_att_n = M.tree_attention_workspace(B, s.N, c["Hq"], c["Hkv"], c["D"], Lmax)
        s.ws_att = torch.empty(max(16, s.ws_att_n), dtype=torch.uint8, device=dev)
        s.ws_ver = torch.empty(max(16, M.verify_accept_workspace(B, s.N, V)), dtype=torch.uint8, device=dev)
        s.heads()
        M.build_tree(s.idx, s.root, s.depth, s.rank, out=s.cand)
        s.vlogits = self.td(W.planted_logits(CFG["seed"], s.cand.cpu().numpy(), t["parent"], V, c["alpha"]))
        s.launches = 2 + 1 + (2 if s.ws_att_n > 0 else 1) + 2 + 1
        return s

    def heads(self):
        c = CFG
        self.M.heads_topk(self.h, self.w1, self.b1, self.w2, c["topk"], out=(self.idx, self.val, None),
                          ws=self.ws_heads)

    CALLS = ("heads_topk", "build_tree", "tree_attention", "verify_accept_tree", "kv_compact")

    def run(self, ev=None):
        """One step; ev (6 events) brackets the five calls when given."""
        M = self.M
        self.kv_len.copy_(self.kv_len0)
        rec = (lambda i: ev[i].record()) if ev is not None else (lambda i: None)
        rec(0)
        self.heads()
        rec(1)
        M.build_tree(self.idx, self.root, self.depth, self.rank, out=self.cand)
        rec(2)
        M.tree_attention(self.q, self.kc, self.vc, self.kv_len, self.mask, self.scale, out=self.att_out,
                         ws=self.ws_att)
        rec(3)
        M.verify_accept_tree(self.vlogits, self.cand, self.parent, self.depth, self.Dmax, out=self.acc,
                             ws=self.ws_ver)
        rec(4)
        M.kv_compact(self.kc, self.vc, self.kv_len, self.acc["path_nodes"], self.acc["accept_len"],
                     self.acc["best_node"], self.N, self.Dmax, hidden_tree=self.ht, h_next=self.h_next,
                     src_idx=self.src)
        rec(5)


def _pack(tensors, device, pinned=False):
    """One buffer holding `tensors` at 256-byte aligned offsets; returns the
    buffer and views of it shaped like the inputs (contents copied in)."""
    import torch
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off = (off + t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = []
    for t, o in zip(tensors, offs):
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


def run_e2e(step, steps, warmup, pipelined=True, host_results=False):
    """Same step through the C ABI with host buffers: per-step inputs copied from
    pinned host memory, results read back, all inside the timed region.  Every
    input (h, q, verifier logits, tree hidden states, the tree's K/V rows)
    travels in one packed host-to-device copy and the results in one packed
    read; the tree's K/V rows then move from the staging buffer into their
    cache slots on the device.  The input copy, the step (its K/V placement and
    five calls) and the result read are CUDA graphs on three streams.

    pipelined: two staging and two result buffers; step k + 1's inputs are
    copied while step k computes, step k's results are read back while step
    k + 1 computes, and the host waits for step k's results right after
    enqueuing step k + 1 (two steps in flight, as a serving loop with a
    prefetching input queue runs).  Otherwise every step copies, computes, is
    read back and waited for before the next starts.

    host_results: also return, per result buffer, the read-back results as host
    tensors (accept_len, best_node, path_nodes, next_tok, h_next)."""
    torch = step.torch
    L = int(step.kv_len0[0].item())
    N = step.N
    dev = step.h.device
    nbuf = 2 if pipelined else 1
    names_in = ("h", "q", "vlogits", "ht")
    tree_kv = [step.kc[:, :, L:L + N].contiguous(), step.vc[:, :, L:L + N].contiguous()]
    src = [getattr(step, n) for n in names_in] + tree_kv
    staged = [_pack(src, dev) for _ in range(nbuf)]  # (device buffer, views) per slot
    hbuf_in, _ = _pack([t.cpu() for t in src], "cpu", pinned=True)
    names_out = ("accept_len", "best_node", "path_nodes", "next_tok")
    results = [_pack([step.acc[n] for n in names_out] + [step.h_next], dev) for _ in range(nbuf)]
    hbuf_out = [torch.empty(results[0][0].numel(), dtype=torch.uint8).pin_memory() for _ in range(nbuf)]
    h2d = hbuf_in.numel()
    d2h = results[0][0].numel()

    def enqueue_copy(p):
        staged[p][0].copy_(hbuf_in, non_blocking=True)

    def enqueue_step(p):
        views = staged[p][1]
        for n, v in zip(names_in, views):
            setattr(step, n, v)
        outs = results[p][1]
        for n, v in zip(names_out, outs[:4]):
            step.acc[n] = v
        step.h_next = outs[4]
        step.kc[:, :, L:L + N].copy_(views[4])
        step.vc[:, :, L:L + N].copy_(views[5])
        step.run()

    def enqueue_read(p):
        hbuf_out[p].copy_(results[p][0], non_blocking=True)

    cs, ss, rs = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for x in (cs, ss, rs):
        x.wait_stream(torch.cuda.current_stream())
    for p in range(nbuf):  # warm-up before capture
        with torch.cuda.stream(cs):
            enqueue_copy(p)
        ss.wait_stream(cs)
        with torch.cuda.stream(ss):
            enqueue_step(p)
        rs.wait_stream(ss)
        with torch.cuda.stream(rs):
            enqueue_read(p)
    torch.cuda.synchronize()
    gc, gs, gr = [], [], []
    for p in range(nbuf):
        for lst, strm, fn in ((gc, cs, enqueue_copy), (gs, ss, enqueue_step), (gr, rs, enqueue_read)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=strm):
                fn(p)
            lst.append(g)
    copied = [torch.cuda.Event() for _ in range(nbuf)]
    computed = [torch.cuda.Event() for _ in range(nbuf)]
    done = [torch.cuda.Event() for _ in range(nbuf)]

    def launch(k):
        p = k % nbuf
        with torch.cuda.stream(cs):
            if k >= nbuf:
                cs.wait_event(computed[p])  # slot p's inputs were read by step k - nbuf
            gc[p].replay()
            copied[p].record(cs)
        with torch.cuda.stream(ss):
            ss.wait_event(copied[p])
            if k >= nbuf:
                ss.wait_event(done[p])  # slot p's results of step k - nbuf are on the host
            gs[p].replay()
            computed[p].record(ss)
        with torch.cuda.stream(rs):
            rs.wait_event(computed[p])
            gr[p].replay()
            done[p].record(rs)

    def run(n):
        for k in range(n):
            launch(k)
            if pipelined:
                if k >= 1:
                    done[(k - 1) % nbuf].synchronize()  # step k - 1's results are on the host
            else:
                done[0].synchronize()
        done[(n - 1) % nbuf].synchronize()

    run(max(warmup, 2))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    if host_results:
        got = []
        for p in range(nbuf):
            base = results[p][0].data_ptr()
            segs = []
            for v in results[p][1]:
                off, nb = v.data_ptr() - base, v.numel() * v.element_size()
                segs.append(hbuf_out[p][off:off + nb].view(v.dtype).view(v.shape).clone())
            got.append(segs)
        return dt, h2d, d2h, got
    return dt, h2d, d2h


def measure_projection(dev, iters=50, warmup=5):
    """medusa_verify_project_tree (lm_head x tree hidden states on the tensor
    cores, reduced to acceptance without writing logits) at two shapes: the
    Vicuna-7B-shaped batch-1 sparse tree (greedy; HBM-bound: lm_head is read
    once) and batch 4 of the dense 341-node tree (typical; tensor-bound).
    Each is timed over `iters` back-to-back calls with events at both ends."""
    import torch
    import medusa_speculative_decoding_gb300 as M
    c = CFG
    H, V = c["H"], c["V"]
    td = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    lm = td(W.normal(2, "LMHEAD", (V, H), 0.02, "bf16"))
    dense_paths = np.array([[a, b, x, y] for a in range(4) for b in range(4) for x in range(4)
                            for y in range(4)], np.int32)
    cases = (("vicuna7b_b1_sparse64_greedy", M.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5, 1, 5, 8,
              "greedy", "hbm"),
             ("dense341_b4_typical", dense_paths, 4, 4, 4, 4, "typical", "tensor"))
    out = {}
    for name, paths, maxd, B, K, k, mode, bound in cases:
        t = M.tree_layout(paths, maxd)
        N = t["N"]
        hid = td(W.hidden_tree(4, B, N, H, "bf16"))
        par, dep, rnk = (torch.from_numpy(t[x]).to(dev) for x in ("parent", "depth", "rank"))
        lists = torch.from_numpy(W.random_topk_lists(4, B, K, k, V)).to(dev)
        cand = M.build_tree(lists, torch.from_numpy(W.root_tokens(4, B, V)).to(dev), dep, rnk)
        ws = torch.empty(max(16, M.verify_project_workspace(B, N, H, V)), dtype=torch.uint8, device=dev)
        res = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   best_node=torch.empty(B, dtype=torch.int32, device=dev),
                   path_nodes=torch.empty((B, t["max_depth"] + 1), dtype=torch.int32, device=dev),
                   next_tok=torch.empty(B, dtype=torch.int32, device=dev))
        call = lambda: M.verify_project_tree(hid, lm, cand, par, dep, t["max_depth"], mode, out=res, ws=ws)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            call()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / iters
        rows = B * N
        if bound == "hbm":
            by = V * H * 2 + rows * H * 2
            peak, kind = _peaks()
            ach = by / (us * 1e-6) / 1e9
            out[name] = {"us": us, "bound": "hbm", "achieved": ach, "unit": "GB/s", "peak": peak,
                         "peak_kind": kind, "frac": ach / peak, "algorithmic_bytes": by, "rows": rows}
        else:
            fl = 2.0 * rows * V * H
            peak, kind = _tpeak()
            ach = fl / (us * 1e-6) / 1e12
            out[name] = {"us": us, "bound": "tensor", "achieved": ach, "unit": "TFLOP/s", "peak": peak,
                         "peak_kind": kind, "frac": ach / peak, "algorithmic_flops": fl, "rows": rows}
        del hid, ws
    return out


def measure_attention_workloads(dev, iters=20, warmup=3, names=None):
    """medusa_tree_attention alone at the other workloads' shapes: batch 8 of
    the 13B shape (40 heads, ragged KV lengths 1024..4096, sparse tree) and
    batch 4 at KV 8192 with the sparse 64-node and the dense 341-node trees.
    Each is timed over `iters` back-to-back calls with events at both ends (the
    KV cache of each exceeds L2)."""
    import torch
    import medusa_speculative_decoding_gb300 as M
    dense_paths = np.array([[a, b, x, y] for a in range(4) for b in range(4) for x in range(4)
                            for y in range(4)], np.int32)
    cases = (("13b_b8_ragged_sparse64", M.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5, 8, 40,
              W.kv_lengths(3, 8, 1024, 4096)),
             ("b4_kv8192_sparse64", M.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5, 4, 32,
              np.full(4, 8192, np.int32)),
             ("b4_kv8192_dense341", dense_paths, 4, 4, 32, np.full(4, 8192, np.int32)))
    hbm, _ = _peaks()
    tpk, _ = _tpeak()
    D = 128
    out = {}
    for name, paths, maxd, B, Hq, lens in cases:
        if names is not None and name not in names:
            continue
        t = M.tree_layout(paths, maxd)
        N = t["N"]
        Lmax = int(lens.max()) + N
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        q = torch.randn(B, N, Hq, D, device=dev, generator=g).bfloat16()
        kc = torch.randn(B, Hq, Lmax, D, device=dev, generator=g).bfloat16()
        vc = torch.randn(B, Hq, Lmax, D, device=dev, generator=g).bfloat16()
        kl = torch.from_numpy(lens.astype(np.int32)).to(dev)
        mask = torch.from_numpy(t["mask"].view(np.int64)).to(dev)
        o = torch.empty(B, N, Hq, D, device=dev)
        ws = torch.empty(max(16, M.tree_attention_workspace(B, N, Hq, Hq, D, Lmax)), dtype=torch.uint8,
                         device=dev)
        call = lambda: M.tree_attention(q, kc, vc, kl, mask, 1.0 / np.sqrt(D), out=o, ws=ws)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            call()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / iters
        by = sum(2 * Hq * (int(L) + N) * D * 2 for L in lens) + B * N * Hq * D * (2 + 4)
        fl = sum(4.0 * N * Hq * D * (int(L) + N) for L in lens)
        out[name] = {"us": us, "gbs": by / (us * 1e-6) / 1e9, "frac_hbm": by / (us * 1e-6) / 1e9 / hbm,
                     "tflops": fl / (us * 1e-6) / 1e12, "frac_bf16": fl / (us * 1e-6) / 1e12 / tpk,
                     "algorithmic_bytes": by, "flops_upper_bound": fl}
        del q, kc, vc, o
    return out


def measure_step_graph(step, layers=32, iters=200, warmup=5):
    """The decode step as one CUDA graph with tree attention over `layers`
    layers (each with its own KV cache; a stand-in for the backbone's attention
    layers, whose other work is not part of this path): heads -> build_tree ->
    layers x tree_attention -> verify -> one compaction of every layer's cache.
    The caches are one tensor [B, layers * Hkv, Lmax, D], so layer l is heads
    l*Hkv .. (l+1)*Hkv and one compaction call moves all layers' rows.  Reports
    graph replays per second and accepted tokens per second (accept_len + 1
    tokens per round)."""
    import torch
    M, c = step.M, CFG
    dev = step.kc.device
    B, Hkv, D = c["B"], c["Hkv"], c["D"]
    Lmax = step.kc.shape[2]
    if B != 1:
        return None
    kc = torch.empty((B, layers * Hkv, Lmax, D), dtype=step.kc.dtype, device=dev)
    vc = torch.empty_like(kc)
    for l in range(layers):  # every layer starts from the step's own cache
        kc[:, l * Hkv:(l + 1) * Hkv].copy_(step.kc)
        vc[:, l * Hkv:(l + 1) * Hkv].copy_(step.vc)
    kls = [kc[:, l * Hkv:(l + 1) * Hkv] for l in range(layers)]
    vls = [vc[:, l * Hkv:(l + 1) * Hkv] for l in range(layers)]

    def one():
        step.kv_len.copy_(step.kv_len0)
        step.heads()
        M.build_tree(step.idx, step.root, step.depth, step.rank, out=step.cand)
        for l in range(layers):
            M.tree_attention(step.q, kls[l], vls[l], step.kv_len, step.mask, step.scale, out=step.att_out,
                             ws=step.ws_att)
        M.verify_accept_tree(step.vlogits, step.cand, step.parent, step.depth, step.Dmax, out=step.acc,
                             ws=step.ws_ver)
        M.kv_compact(kc, vc, step.kv_len, step.acc["path_nodes"], step.acc["accept_len"], step.acc["best_node"],
                     step.N, step.Dmax, hidden_tree=step.ht, h_next=step.h_next, src_idx=step.src)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warmup):
            one()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        one()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / iters
    tokens = float(step.acc["accept_len"].float().mean().item()) + 1.0
    # the layers' tree attention alone: one graph of `layers` back-to-back
    # calls, each on its own layer's cache (1.1 GB in all, more than L2, so
    # every call reads its keys and values from HBM)
    def att():
        for l in range(layers):
            M.tree_attention(step.q, kls[l], vls[l], step.kv_len, step.mask, step.scale, out=step.att_out,
                             ws=step.ws_att)
    step.kv_len.copy_(step.kv_len0)
    with torch.cuda.stream(s):
        att()
    torch.cuda.synchronize()
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga, stream=s):
        att()
    for _ in range(warmup):
        ga.replay()
    torch.cuda.synchronize()
    reps = max(1, iters // 4)
    a.record()
    for _ in range(reps):
        ga.replay()
    b.record()
    torch.cuda.synchronize()
    us_att = a.elapsed_time(b) * 1e3 / (reps * layers)
    hbm, _ = _peaks()
    abytes = algorithmic_bytes(CFG, step.N, int(step.kv_len0.max().item()) + step.N)[1]
    del kc, vc
    return {"layers": layers, "us_per_step": us, "steps_per_s": 1e6 / us, "tokens_per_step": tokens,
            "tokens_per_s": tokens * 1e6 / us, "launches_per_step": 2 + 1 + layers + 2 + 1,
            "attention_per_layer": {"us": us_att, "algorithmic_bytes": abytes,
                                    "gbs": abytes / (us_att * 1e-6) / 1e9,
                                    "frac_hbm": abytes / (us_att * 1e-6) / 1e9 / hbm,
                                    "method": f"graph of {layers} back-to-back calls, one cache per layer"}}


def measure_tree_sizes(step, iters=200, warmup=10):
    """The step verifying the sparse 64-node tree and, at the same batch, KV
    length and planted acceptance, the dense 341-node tree (top-4 of heads 1-4,
    Cartesian product), each timed over `iters` back-to-back steps with events at
    the two ends.  Acceptance is planted along the rank-0 chain in both (alpha
    0.8), so both accept the same expected number of tokens: the comparison is
    the cost side of choosing the smaller tree."""
    import torch
    M = step.M
    dense_paths = np.array([[a, b, x, y] for a in range(4) for b in range(4) for x in range(4)
                            for y in range(4)], np.int32)
    out = {}
    for name, make in (("sparse64", lambda: step), ("dense341", lambda: step.with_tree(M.tree_layout(dense_paths, 4)))):
        s = make()
        for _ in range(warmup):
            s.run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            s.run()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / iters
        # expected tokens per step of the planted acceptance: sum of alpha^i up to
        # the tree's depth (the same 3.36 for both depth-4 trees)
        depth = int(np.max(s.t["depth"]))  # the deepest node (the layout's cap may be larger)
        tokens = sum(CFG["alpha"] ** i for i in range(depth + 1))
        out[name] = {"nodes": s.N, "us_per_step": us, "steps_per_s": 1e6 / us,
                     "tree_tokens_verified_per_s": s.N * 1e6 / us, "expected_tokens_per_step": tokens,
                     "expected_tokens_per_s": tokens * 1e6 / us}
        del s
    return out


def measure_heads_batches(dev, iters=10, warmup=2):
    """Batch sweep of medusa_heads_topk: hidden 4096 at batch 1, 2, 4, 8, 16, 32
    and 64, and hidden 5120 at batch 8; 5 heads, vocab 32000, top-8, bf16
    (random-init weights of those shapes, allocated once per hidden size; they
    exceed L2), each point timed over `iters` back-to-back calls.  Batches 1-2
    run on CUDA cores, 3-64 on the tensor cores."""
    import torch
    import medusa_speculative_decoding_gb300 as M
    hbm, _ = _peaks()
    out = {}
    K, V, topk = 5, 32000, 8
    for H, batches in ((4096, (1, 2, 4, 8, 16, 32, 64)), (5120, (8,))):
        g = torch.Generator(device=dev)
        g.manual_seed(11)
        w1 = (torch.randn(K, H, H, device=dev, generator=g) * 0.02).bfloat16()
        b1 = torch.zeros(K, H, device=dev).bfloat16()
        w2 = (torch.randn(K, V, H, device=dev, generator=g) * 0.02).bfloat16()
        for B in batches:
            h = torch.randn(B, H, device=dev, generator=g).bfloat16()
            ws = torch.empty(M.heads_topk_workspace(B, K, H, V, topk), dtype=torch.uint8, device=dev)
            res = (torch.empty(B, K, topk, dtype=torch.int32, device=dev),
                   torch.empty(B, K, topk, device=dev), None)
            call = lambda: M.heads_topk(h, w1, b1, w2, topk, out=res, ws=ws)
            for _ in range(warmup):
                call()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(iters):
                call()
            b.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / iters
            by = K * (H * H + H + V * H) * 2 + B * H * 2 + B * K * topk * 8
            fl = 2.0 * B * K * (H * H + V * H)
            out[f"b{B}_h{H}"] = {"us": us, "gbs": by / (us * 1e-6) / 1e9,
                                 "frac_hbm": by / (us * 1e-6) / 1e9 / hbm, "algorithmic_bytes": by,
                                 "tflops": fl / (us * 1e-6) / 1e12, "sequences_per_s": B * 1e6 / us,
                                 "path": "tcgen05" if B >= 3 else "cuda cores"}
            del h, ws
        del w1, b1, w2
    return out


# ----------------------------------------------------------------------------
# whole decode steps of the batched workloads
# ----------------------------------------------------------------------------
DENSE_PATHS = np.array([[a, b, x, y] for a in range(4) for b in range(4) for x in range(4) for y in range(4)],
                       np.int32)


class WorkloadStep:
    """The five C-ABI calls of one decode step of a batched workload, with
    random-init weights of its shape drawn on the GPU (seeded), the workload's
    KV lengths, and verifier logits planted around the step's own candidates
    (greedy, alpha = 0.8) or drawn N(0, 3) (typical acceptance)."""

    def __init__(self, name, tree_kind, dev, seed=21):
        import torch
        import medusa_speculative_decoding_gb300 as M
        self.M, self.torch, self.name = M, torch, name
        c = self.c = W.WORKLOADS[name]
        paths, md = ((M.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5) if tree_kind == "sparse64" else (DENSE_PATHS, 4))
        t = self.t = M.tree_layout(paths, md)
        self.N, self.Dmax = t["N"], t["max_depth"]
        B, H, V, K, topk = c["B"], c["H"], c["V"], c["K"], c["topk"]
        Hq, Hkv, D = c["Hq"], c["Hkv"], c["D"]
        self.mode = "typical" if c["accept"] == "typical" else "greedy"
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        rn = lambda *shape, std=1.0: (torch.randn(*shape, device=dev, generator=g) * std).to(bf)
        self.h = rn(B, H)
        self.w1 = rn(K, H, H, std=c["w_std"])
        self.b1 = torch.zeros(K, H, device=dev, dtype=bf)
        self.w2 = rn(K, V, H, std=c["w_std"])
        self.kv_len0 = torch.from_numpy(W.kv_lengths(c["seed"], B, c["L_lo"], c["L_hi"])).to(dev)
        self.kv_len = self.kv_len0.clone()
        Lmax = c["L_hi"] + self.N
        self.q = rn(B, self.N, Hq, D)
        self.kc, self.vc = rn(B, Hkv, Lmax, D), rn(B, Hkv, Lmax, D)
        self.ht = rn(B, self.N, H)
        self.scale = 1.0 / float(np.sqrt(D))
        td = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.root = td(W.root_tokens(c["seed"], B, V))
        self.depth, self.rank, self.parent = td(t["depth"]), td(t["rank"]), td(t["parent"])
        self.mask = torch.from_numpy(t["mask"].view(np.int64)).to(dev)
        i32 = torch.int32
        self.idx = torch.empty(B, K, topk, dtype=i32, device=dev)
        self.val = torch.empty(B, K, topk, device=dev)
        self.cand = torch.empty(B, self.N, dtype=i32, device=dev)
        self.att_out = torch.empty(B, self.N, Hq, D, device=dev)
        self.acc = dict(accept_len=torch.empty(B, dtype=i32, device=dev), best_node=torch.empty(B, dtype=i32, device=dev),
                        path_nodes=torch.empty(B, self.Dmax + 1, dtype=i32, device=dev),
                        next_tok=torch.empty(B, dtype=i32, device=dev))
        self.h_next = torch.empty(B, H, dtype=bf, device=dev)
        self.src = torch.empty(B, self.Dmax + 1, dtype=i32, device=dev)
        u8 = torch.uint8
        self.ws_heads = torch.empty(max(16, M.heads_topk_workspace(B, K, H, V, topk)), dtype=u8, device=dev)
        self.ws_att = torch.empty(max(16, M.tree_attention_workspace(B, self.N, Hq, Hkv, D, Lmax)), dtype=u8,
                                  device=dev)
        self.ws_ver = torch.empty(max(16, M.verify_accept_workspace(B, self.N, V)), dtype=u8, device=dev)
        self.heads()
        M.build_tree(self.idx, self.root, self.depth, self.rank, out=self.cand)
        if self.mode == "greedy":
            self.vlogits = td(W.planted_logits(c["seed"], self.cand.cpu().numpy(), t["parent"], V, c["alpha"]))
        else:
            self.vlogits = torch.randn(B, self.N, V, device=dev, generator=g) * float(c["logit_std"])
        lens = self.kv_len0.cpu().numpy()
        self.bytes = {
            "heads": K * (H * H + H + V * H) * 2 + B * H * 2 + B * K * topk * 8,
            "attention": sum(2 * Hkv * (int(L) + self.N) * D * 2 for L in lens) + B * self.N * Hq * D * (2 + 4),
            "verify": B * self.N * V * 4 + B * self.N * 4}

    def heads(self):
        self.M.heads_topk(self.h, self.w1, self.b1, self.w2, self.c["topk"], out=(self.idx, self.val, None),
                          ws=self.ws_heads)

    def run(self, ev=None):
        M = self.M
        rec = (lambda i: ev[i].record()) if ev is not None else (lambda i: None)
        self.kv_len.copy_(self.kv_len0)
        rec(0)
        self.heads()
        rec(1)
        M.build_tree(self.idx, self.root, self.depth, self.rank, out=self.cand)
        rec(2)
        M.tree_attention(self.q, self.kc, self.vc, self.kv_len, self.mask, self.scale, out=self.att_out,
                         ws=self.ws_att)
        rec(3)
        M.verify_accept_tree(self.vlogits, self.cand, self.parent, self.depth, self.Dmax, self.mode,
                             out=self.acc, ws=self.ws_ver)
        rec(4)
        M.kv_compact(self.kc, self.vc, self.kv_len, self.acc["path_nodes"], self.acc["accept_len"],
                     self.acc["best_node"], self.N, self.Dmax, hidden_tree=self.ht, h_next=self.h_next,
                     src_idx=self.src)
        rec(5)


def measure_workload_steps(dev, iters=100, warmup=10):
    """Whole decode steps (heads -> tree -> tree attention, one layer ->
    acceptance -> compaction) of the 13B-shaped ragged batch-8 workload (sparse
    64-node tree, greedy) and the batch-4 KV-8192 workload with the sparse
    64-node and the dense 341-node tree (typical acceptance): steps/s, tree
    tokens verified/s, per-call times, and the step's algorithmic bytes against
    the HBM ceiling.  `iters` back-to-back steps with events at the two ends
    (each step streams 1.9-2.3 GB, more than L2); a second pass with events
    around every call gives the per-call times."""
    import torch
    hbm, kind = _peaks()
    out = {}
    for key, name, tree in (("h5120_b8_ragged_sparse64_greedy", "h5120_b8_ragged", "sparse64"),
                            ("h4096_b4_kv8192_sparse64_typical", "h4096_b4_kv8192", "sparse64"),
                            ("h4096_b4_kv8192_dense341_typical", "h4096_b4_kv8192", "dense341")):
        s = WorkloadStep(name, tree, dev)
        for _ in range(warmup):
            s.run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(iters):
            s.run()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / iters
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(20)]
        for e in evs:
            s.run(e)
        torch.cuda.synchronize()
        calls = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) * 1e3 for e in evs) for i, n in enumerate(Step.CALLS)}
        total = sum(s.bytes.values())
        B = s.c["B"]
        out[key] = {"batch": B, "nodes": s.N, "acceptance": s.mode, "us_per_step": us, "steps_per_s": 1e6 / us,
                    "tree_tokens_verified_per_s": B * s.N * 1e6 / us,
                    "tokens_per_step": float((s.acc["accept_len"].float() + 1).sum().item()),
                    "call_us": {k: round(v, 2) for k, v in calls.items()},
                    "algorithmic_bytes": s.bytes, "step_gbs": total / (us * 1e-6) / 1e9,
                    "frac_of_step_ceiling": total / (us * 1e-6) / 1e9 / hbm, "peak_kind": kind}
        del s
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------
# chained decode rounds as one CUDA graph
# ----------------------------------------------------------------------------
def measure_rounds(step, rounds=16, layers=32, iters=20, warmup=3, seed=31):
    """`rounds` chained decode rounds of the Vicuna-7B-shaped batch-1 workload
    captured as one CUDA graph: round r + 1's root token is round r's next
    token, its heads read round r's h_next, and its KV prefix is round r's
    compacted cache (kv_len grows by accept_len + 1 per round).  Per round:
    heads -> build_tree -> the round's tree K/V rows written into every
    layer's cache at slots [kv_len, kv_len + N) (the backbone's part, from a
    pool drawn ahead) -> tree attention over `layers` layers -> verifier logits
    planted around the round's own candidates (the lowest-index child of a node
    carries its row's argmax with probability 0.8, drawn ahead) -> greedy
    acceptance -> one compaction of every layer's cache.  Reports graph time per
    round, rounds/s and accepted tokens per wall-second (sum of accept_len + 1
    over the rounds, read after the timed replays)."""
    import torch
    M, c = step.M, CFG
    dev = step.h.device
    B, N, Dmax, Hkv, D, H, V = c["B"], step.N, step.Dmax, c["Hkv"], c["D"], c["H"], c["V"]
    if B != 1:
        return None
    L0 = int(step.kv_len0[0].item())
    Lmax = L0 + N + rounds * (Dmax + 1)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    bf = torch.bfloat16
    kc = torch.randn(B, layers * Hkv, Lmax, D, device=dev, generator=g).to(bf)
    vc = torch.randn(B, layers * Hkv, Lmax, D, device=dev, generator=g).to(bf)
    kls = [kc[:, l * Hkv:(l + 1) * Hkv] for l in range(layers)]
    vls = [vc[:, l * Hkv:(l + 1) * Hkv] for l in range(layers)]
    tk = torch.randn(rounds, B, layers * Hkv, N, D, device=dev, generator=g).to(bf)  # tree K/V rows per round
    tv = torch.randn(rounds, B, layers * Hkv, N, D, device=dev, generator=g).to(bf)
    qs = torch.randn(rounds, B, N, c["Hq"], D, device=dev, generator=g).to(bf)
    hts = torch.randn(rounds, B, N, H, device=dev, generator=g).to(bf)
    base = torch.randn(B, N, V, device=dev, generator=g)  # N(0, 1) verifier rows
    parent = step.t["parent"]
    first_child = np.zeros(N, np.int64)
    has_child = np.zeros(N, bool)
    for j in range(N - 1, 0, -1):
        first_child[parent[j]] = j
        has_child[parent[j]] = True
    fc = torch.from_numpy(first_child).to(dev)
    plant = (torch.rand(rounds, B, N, device=dev, generator=g) < c["alpha"]) & torch.from_numpy(has_child).to(dev)
    plant_val = plant.float() * 100.0  # far above any N(0, 1) draw
    vwork = torch.empty_like(base)
    ar = torch.arange(N, device=dev)
    h0, root0 = step.h.clone(), step.root.clone()
    h_cur, root_cur = torch.empty_like(h0), torch.empty_like(root0)
    kv_len = torch.empty_like(step.kv_len0)
    tokens = torch.zeros(1, dtype=torch.int64, device=dev)
    i32 = torch.int32
    idx = torch.empty(B, c["K"], c["topk"], dtype=i32, device=dev)
    val = torch.empty(B, c["K"], c["topk"], device=dev)
    cand = torch.empty(B, N, dtype=i32, device=dev)
    att_out = torch.empty(B, N, c["Hq"], D, device=dev)
    acc = dict(accept_len=torch.empty(B, dtype=i32, device=dev), best_node=torch.empty(B, dtype=i32, device=dev),
               path_nodes=torch.empty(B, Dmax + 1, dtype=i32, device=dev), next_tok=torch.empty(B, dtype=i32, device=dev))
    h_next = torch.empty_like(h0)
    src = torch.empty(B, Dmax + 1, dtype=i32, device=dev)
    ws_att = torch.empty(max(16, M.tree_attention_workspace(B, N, c["Hq"], Hkv, D, Lmax)), dtype=torch.uint8,
                         device=dev)

    def one():
        kv_len.copy_(step.kv_len0)
        h_cur.copy_(h0)
        root_cur.copy_(root0)
        tokens.zero_()
        for r in range(rounds):
            M.heads_topk(h_cur, step.w1, step.b1, step.w2, c["topk"], out=(idx, val, None), ws=step.ws_heads)
            M.build_tree(idx, root_cur, step.depth, step.rank, out=cand)
            slots = kv_len[0].long() + ar  # batch 1: one set of slots
            kc.index_copy_(2, slots, tk[r])
            vc.index_copy_(2, slots, tv[r])
            for l in range(layers):
                M.tree_attention(qs[r], kls[l], vls[l], kv_len, step.mask, step.scale, out=att_out, ws=ws_att)
            vwork.copy_(base)
            vwork.view(B * N, V).scatter_add_(1, cand[:, fc].reshape(B * N, 1).long(),
                                              plant_val[r].reshape(B * N, 1))
            M.verify_accept_tree(vwork, cand, step.parent, step.depth, Dmax, out=acc, ws=step.ws_ver)
            M.kv_compact(kc, vc, kv_len, acc["path_nodes"], acc["accept_len"], acc["best_node"], N, Dmax,
                         hidden_tree=hts[r], h_next=h_next, src_idx=src)
            tokens.add_(acc["accept_len"].sum() + B)
            h_cur.copy_(h_next)
            root_cur.copy_(acc["next_tok"])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            one()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        one()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    us_round = a.elapsed_time(b) * 1e3 / (iters * rounds)
    tok = int(tokens.item())  # of the last replay (every replay starts from the same state)
    grown = int(kv_len[0].item()) - L0
    out = {"rounds": rounds, "layers": layers, "us_per_round": us_round, "rounds_per_s": 1e6 / us_round,
           "tokens_per_round": tok / rounds, "tokens_per_s": tok / rounds * 1e6 / us_round,
           "kv_len_growth": grown, "graph_replays": iters}
    del kc, vc, tk, tv, qs, hts
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------
# speculative-sampling acceptance sweep
# ----------------------------------------------------------------------------
def expected_tokens(alpha, gamma):
    """Expected tokens per round, (1 - alpha^(gamma+1)) / (1 - alpha), gamma + 1
    at alpha = 1 (speculative-decoding e-book page, "Expected tokens per round")."""
    if alpha >= 1.0:
        return gamma + 1.0
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def measure_chain_sweep(dev, rounds=64, sigmas=(0.1, 0.5, 1.0), gmax=32, B=64, V=128256):
    """medusa_verify_accept_chain over sigma x gamma = 0..gmax, `rounds` rounds
    each, batch 64, vocab 128256.  Every round draws, on the GPU and untimed,
    ql ~ N(0, 2) for gmax + 1 positions, q = softmax(ql), p = softmax(ql +
    N(0, sigma)) and drafts x_i ~ q_i; the call at gamma reads the first gamma
    + 1 rows of p and gamma rows of q (copied into buffers of their own, then L2
    flushed by a 256 MB write, so each timed call reads HBM).  Reported per
    (sigma, gamma): measured alpha = accepted / drafts examined, alpha =
    mean over positions of sum_v min(p, q) (1 - total variation), mean tokens
    per round next to E(alpha_hat, gamma) and E(alpha, gamma), the median call
    time, rounds/s and tokens/s; plus the HBM roofline of the call at
    gamma = 1, 4, 8, 32 (sigma 0.5)."""
    import torch
    import medusa_speculative_decoding_gb300 as M
    hbm, kind = _peaks()
    g = torch.Generator(device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ws = torch.empty(max(16, M.verify_chain_workspace(B, gmax, V)), dtype=torch.uint8, device=dev)
    n_acc = torch.empty(B, dtype=torch.int32, device=dev)
    toks = torch.empty(B, gmax + 1, dtype=torch.int32, device=dev)
    res = {}
    roof = {}
    for si, sigma in enumerate(sigmas):
        acc = torch.zeros(gmax + 1, dtype=torch.float64, device=dev)
        exam = torch.zeros_like(acc)
        tok = torch.zeros_like(acc)
        by = torch.zeros_like(acc)
        asum = torch.zeros_like(acc)
        times = [[] for _ in range(gmax + 1)]
        for r in range(rounds):
            g.manual_seed(5_000_000 + 1000 * si + r)
            ql = torch.randn(B, gmax + 1, V, device=dev, generator=g) * 2.0
            p = torch.softmax(ql + sigma * torch.randn(B, gmax + 1, V, device=dev, generator=g), -1)
            q = torch.softmax(ql[:, :gmax], -1)
            del ql
            draft = torch.multinomial(q.reshape(-1, V), 1, generator=g).reshape(B, gmax).to(torch.int32)
            amin = torch.minimum(p[:, :gmax], q).sum(-1, dtype=torch.float64)  # [B, gmax]
            evs = []
            for gam in range(gmax + 1):
                P = p[:, :gam + 1].contiguous()
                Q = q[:, :gam].contiguous() if gam else None
                Dr = draft[:, :gam].contiguous() if gam else None
                flush.fill_(r & 255)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                M.verify_accept_chain(P, Q, Dr, 1234 + si, r, out=(n_acc, toks), ws=ws)
                e1.record()
                evs.append((e0, e1))
                n = n_acc.to(torch.float64)
                acc[gam] += n.sum()
                if gam:
                    exam[gam] += torch.minimum(n + 1, torch.full_like(n, gam)).sum()
                    asum[gam] += amin[:, :gam].mean(1).sum()
                tok[gam] += (n + 1).sum()
                by[gam] += (8 * torch.minimum(n + 1, torch.full_like(n, gam))
                            + torch.where(n == gam, 4.0 * V, 8.0 * V)).sum()
                del P, Q, Dr
            torch.cuda.synchronize()
            for gam, (e0, e1) in enumerate(evs):
                times[gam].append(e0.elapsed_time(e1) * 1e3)
            del p, q, draft, amin
        acc, exam, tok, by, asum = (x.cpu().numpy() for x in (acc, exam, tok, by, asum))
        rows = {}
        for gam in range(gmax + 1):
            us = statistics.median(times[gam])
            a_hat = float(acc[gam] / exam[gam]) if gam else None
            a_th = float(asum[gam] / (rounds * B)) if gam else None
            mean_tok = float(tok[gam] / (rounds * B))
            rows[str(gam)] = {
                "alpha_hat": None if a_hat is None else round(a_hat, 5),
                "alpha": None if a_th is None else round(a_th, 5),
                "tokens_per_round": round(mean_tok, 5),
                "E_alpha_hat": round(expected_tokens(a_hat, gam), 5) if gam else 1.0,
                "E_alpha": round(expected_tokens(a_th, gam), 5) if gam else 1.0,
                "us": round(us, 2), "rounds_per_s": round(1e6 / us, 1),
                "tokens_per_s": round(mean_tok * B * 1e6 / us, 1)}
            if sigma == 0.5 and gam in (1, 4, 8, 32):
                bb = float(by[gam] / rounds)
                roof[f"gamma{gam}"] = {"us": us, "algorithmic_bytes": bb, "gbs": bb / (us * 1e-6) / 1e9,
                                       "frac_hbm": bb / (us * 1e-6) / 1e9 / hbm, "peak_kind": kind}
        res[f"sigma{sigma}"] = rows
    del flush, ws
    torch.cuda.empty_cache()
    return {"rounds": rounds, "batch": B, "vocab": V, "sweep": res}, roof


# ----------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------
def host_cores():
    """Threads this process may run on (its CPU affinity mask)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (model name on x86; implementer
    and part numbers on Arm, e.g. 0x41/0xd4f for Neoverse V2)."""
    import platform
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model"):
        for ln in info.splitlines():
            if ln.startswith(key):
                return ln.split(":", 1)[1].strip()
    imp = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU implementer")]
    part = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU part")]
    return f"{platform.machine()} implementer {imp[0] if imp else '?'} part {part[0] if part else '?'}"


class OracleStep:
    """The whole decode step in the oracle (float64 C): every head and vocab
    row, the top-k and candidates, every attention row, greedy acceptance of
    the planted verifier logits, compaction.  Steps share only read-only
    inputs, so independent steps run concurrently on host threads (the C
    oracle releases the interpreter lock)."""

    def __init__(self, inp):
        from oracle import oracle as O
        self.O, self.inp, c = O, inp, CFG
        self.t = t = O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
        hd = inp["heads"]
        lg = O.heads_logits(hd["h"], hd["w1"], hd["b1"], hd["w2"], c["dtype"])
        idx, _ = O.topk(lg, c["topk"])
        cand = O.build_tree(idx, inp["root"], t["depth"], t["rank"])
        self.vlogits = W.planted_logits(c["seed"], cand, t["parent"], c["V"], c["alpha"])

    def step(self, _=None):
        O, c, t, inp = self.O, CFG, self.t, self.inp
        hd = inp["heads"]
        t0 = time.perf_counter()
        lg = O.heads_logits(hd["h"], hd["w1"], hd["b1"], hd["w2"], c["dtype"])
        idx, _ = O.topk(lg, c["topk"])
        cand = O.build_tree(idx, inp["root"], t["depth"], t["rank"])
        O.tree_attention(inp["att"]["q"], inp["att"]["k_cache"], inp["att"]["v_cache"], inp["kv_len"], t["mask"],
                         c["dtype"], 1 / np.sqrt(c["D"]))
        r = O.verify_tree(self.vlogits, cand, t["parent"], t["depth"], t["max_depth"])
        O.kv_compact(inp["att"]["k_cache"], inp["att"]["v_cache"], inp["kv_len"], r["path_nodes"], r["accept_len"],
                     r["best_node"], inp["ht"], t["N"], t["max_depth"])
        return time.perf_counter() - t0


def oracle_throughput(inp, steps, warmup):
    """Runs `warmup` then `steps` full oracle steps, spread over every host core
    (one step per thread at a time); returns (steps/s of the timed steps, wall
    seconds, mean seconds of one step, threads)."""
    import concurrent.futures as cf
    s = OracleStep(inp)
    n = host_cores()
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        if warmup:
            list(ex.map(s.step, range(warmup)))
        t0 = time.perf_counter()
        per = list(ex.map(s.step, range(steps)))
        wall = time.perf_counter() - t0
    return steps / wall, wall, statistics.mean(per), min(n, steps)


def cpu_baseline(inp):
    """The oracle on the host: one full step per host thread, all at once
    (about one step's time of wall clock)."""
    n = host_cores()
    val, wall, per, used = oracle_throughput(inp, steps=n, warmup=0)
    return {"value": val, "unit": "steps/s", "cores": used, "kind": "oracle", "cpu_model": cpu_model(),
            "single_step_s": per,
            "sample": f"{n} full oracle steps of the workload (every head and vocab row, every attention row, "
                      f"full verify and compaction; float64 C), one per host thread, run together in "
                      f"{wall:.1f} s"}


# ----------------------------------------------------------------------------
# replicas: every rank runs its own batch; the job's time is the slowest rank's
def max_over_ranks(ms, world, device):
    """The largest of the ranks' timed-region milliseconds (ms itself at world 1)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(steps, ms_total, world):
    """Whole-job steps/s: every one of `world` replicas ran `steps` steps within
    the slowest rank's `ms_total` milliseconds."""
    return world * steps / (ms_total / 1e3)


def only_heads(B, H, calls):
    """medusa_heads_topk alone at batch B, `calls` back-to-back calls (a short
    command for ncu captures of the heads kernels at one batch size)."""
    import torch
    import medusa_speculative_decoding_gb300 as M
    dev = torch.device("cuda", 0)
    K, V, topk = 5, 32000, 8
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    h = torch.randn(B, H, device=dev, generator=g).bfloat16()
    w1 = (torch.randn(K, H, H, device=dev, generator=g) * 0.02).bfloat16()
    b1 = torch.zeros(K, H, device=dev).bfloat16()
    w2 = (torch.randn(K, V, H, device=dev, generator=g) * 0.02).bfloat16()
    ws = torch.empty(M.heads_topk_workspace(B, K, H, V, topk), dtype=torch.uint8, device=dev)
    res = (torch.empty(B, K, topk, dtype=torch.int32, device=dev), torch.empty(B, K, topk, device=dev), None)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(max(1, calls)):
        a.record()
        M.heads_topk(h, w1, b1, w2, topk, out=res, ws=ws)
        b.record()
    torch.cuda.synchronize()
    print(json.dumps({"heads_batch": B, "hidden": H, "calls": calls, "last_call_us": a.elapsed_time(b) * 1e3}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-heads", type=int, default=0, metavar="B",
                    help="profiling aid: run medusa_heads_topk at batch B (hidden --hidden, vocab 32000, "
                         "5 heads, top-8, bf16, random-init weights) --steps times, print the last "
                         "call's time, and exit")
    ap.add_argument("--hidden", type=int, default=4096)
    ap.add_argument("--only-attention", default="", metavar="NAME",
                    choices=["", "13b_b8_ragged_sparse64", "b4_kv8192_sparse64", "b4_kv8192_dense341"],
                    help="profiling aid: run medusa_tree_attention at one of the attention workloads' "
                         "shapes, --warmup then --steps calls, print the time per call, and exit")
    ap.add_argument("--only-step", action="store_true",
                    help="profiling aid: run --warmup then --steps steps of --workload, print their time, and exit")
    ap.add_argument("--workload", default="h4096_b1_sparse64",
                    choices=["h4096_b1_sparse64", "h5120_b8_ragged", "h4096_b4_kv8192_sparse64",
                             "h4096_b4_kv8192_dense341"],
                    help="with --only-step: the headline batch-1 step or one of the batched steps")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only_heads:
        return only_heads(args.only_heads, args.hidden, args.steps)
    if args.only_attention:
        import torch
        res = measure_attention_workloads(torch.device("cuda", 0), iters=args.steps, warmup=args.warmup,
                                          names=[args.only_attention])
        print(json.dumps({"only_attention": args.only_attention, "calls": args.steps,
                          **{k: res[args.only_attention][k] for k in ("us", "frac_hbm", "frac_bf16")}}))
        return 0

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        inp = make_inputs_host_only()
        val, wall, per, used = oracle_throughput(inp, args.steps, args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "steps/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": WORKLOAD, "timed_wall_s": wall, "single_step_s": per,
                           "extrapolated": False},
                "cpu_baseline": {"value": val, "unit": "steps/s", "cores": used, "kind": "oracle",
                                 "cpu_model": cpu_model(),
                                 "sample": f"{args.steps} full oracle steps (every head and vocab row, every "
                                           f"attention row, full verify and compaction; float64 C) after "
                                           f"{args.warmup} warm-up steps, spread over {used} host threads, "
                                           f"one step per thread at a time"},
                "e2e": {"value": val, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from medusa_speculative_decoding_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()

    if args.only_step and args.workload != "h4096_b1_sparse64":
        name, tree = {"h5120_b8_ragged": ("h5120_b8_ragged", "sparse64"),
                      "h4096_b4_kv8192_sparse64": ("h4096_b4_kv8192", "sparse64"),
                      "h4096_b4_kv8192_dense341": ("h4096_b4_kv8192", "dense341")}[args.workload]
        s = WorkloadStep(name, tree, dev)
        for _ in range(args.warmup):
            s.run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            s.run()
        b.record()
        torch.cuda.synchronize()
        print(json.dumps({"only_step": True, "workload": args.workload, "steps": args.steps,
                          "us_per_step": a.elapsed_time(b) * 1e3 / args.steps}))
        return 0
    inp = make_inputs()
    step = Step(inp, dev)
    c = CFG
    N = step.N
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if args.only_step:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            step.run()
        b.record()
        torch.cuda.synchronize()
        print(json.dumps({"only_step": True, "steps": args.steps, "us_per_step": a.elapsed_time(b) * 1e3 / args.steps}))
        return 0

    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # headline: K steps back to back, events only at the two ends (an event between
    # two calls would stop the next kernel from being scheduled early)
    start.record(stream)
    for i in range(K):
        step.run()
    end.record(stream)
    torch.cuda.synchronize()
    # per-call durations: the same K steps with an event around every call
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for i in range(K):
        step.run(evs[i])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(start.elapsed_time(end), world, dev)
    call_ms = {name: statistics.mean(evs[i][c].elapsed_time(evs[i][c + 1]) for i in range(K))
               for c, name in enumerate(Step.CALLS)}
    # per-step distribution from the event pass (events between the calls
    # lengthen each step a little, so these run slightly above ms_per_step)
    per_step = sorted(evs[i][0].elapsed_time(evs[i][5]) for i in range(K))
    pct = lambda f: per_step[min(K - 1, int(f * K))]
    step_dist = {"p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9), "with_call_events": True}
    heads_ms = call_ms["heads_topk"]
    att_ms = call_ms["tree_attention"]
    ms_step = ms_total / K
    value = replica_throughput(K, ms_total, world)

    ke = max(20, K // 4)
    e2e_serial_s, _, _ = run_e2e(step, ke, args.warmup, pipelined=False)
    e2e_s, h2d, d2h = run_e2e(step, ke, args.warmup, pipelined=True)
    e2e_val = world * ke / e2e_s

    lead = world == 1 or rank == 0
    graph = measure_step_graph(step) if lead else None
    rounds = {"layers1": measure_rounds(step, layers=1), "layers32": measure_rounds(step, layers=32)} if lead else None
    trees = measure_tree_sizes(step) if lead else None
    steps_w = measure_workload_steps(dev) if lead else None
    proj = measure_projection(dev) if lead else None
    att_w = measure_attention_workloads(dev) if lead else None
    sweep, chain = measure_chain_sweep(dev) if lead else (None, None)
    heads_b = measure_heads_batches(dev) if lead else None

    peak, peak_kind = _peaks()
    hb, ab, vb = algorithmic_bytes(c, N, int(inp["kv_len"][0]) + N)
    heads_gbs = hb / (heads_ms * 1e-3) / 1e9
    att_gbs = ab / (att_ms * 1e-3) / 1e9
    cur = _sha1(os.path.join(ROOT, "medusa_speculative_decoding_gb300", "csrc", "heads.cu"))
    traffic = HEADS_TRAFFIC["bytes"] if HEADS_TRAFFIC["sha1"] == cur else None

    line = {"metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": c["B"] * world, "tree_nodes": N,
                       "kv_len": int(inp["kv_len"][0]), "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: each step streams 1.52 GB",
                       "tree_tokens_verified_per_s": value * N * c["B"]},
            "roofline": {"bound": "hbm", "kernel": "medusa_heads_topk (W1+SiLU, W2+top-k, merge)",
                         "achieved": heads_gbs, "peak": peak, "unit": "GB/s", "frac": heads_gbs / peak,
                         "traffic": traffic, "peak_kind": peak_kind, "algorithmic_bytes": hb,
                         "ms": heads_ms},
            "attention": {"achieved": att_gbs, "unit": "GB/s", "frac": att_gbs / peak,
                          "algorithmic_bytes": ab, "ms": att_ms},
            "call_ms": {k: round(v, 5) for k, v in call_ms.items()},
            "step_ms_distribution": step_dist,
            "step_graph_32_layers": graph,
            "chained_rounds": rounds,
            "tree_sizes": trees,
            "workload_steps": steps_w,
            "verify_projection": proj,
            "attention_workloads": att_w,
            "chain_acceptance": chain,
            "chain_sweep": sweep,
            "heads_batches": heads_b,
            "clocks": clocks,
            "e2e": {"value": e2e_val, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "pipeline": "two steps in flight: the next step's inputs are copied from pinned host "
                                "memory and the previous step's results read back on streams of their own "
                                "while the current step computes; the host waits for every step's results"},
            "e2e_serial": {"value": world * ke / e2e_serial_s, "unit": "steps/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": step.launches * K}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def make_inputs_host_only(seed=None):
    """Inputs of the reference arm: the same generator, tree from the oracle."""
    seed = CFG["seed"] if seed is None else seed
    from oracle import oracle as O
    c = CFG
    t = O.tree_layout(O.sparse_tree_paths(64, 5, 8, 0.6, 0.5), 5)
    N = t["N"]
    heads = W.heads_inputs(seed, c["B"], c["H"], c["V"], c["K"], c["dtype"])
    kv_len = W.kv_lengths(seed, c["B"], c["L_lo"], c["L_hi"])
    Lmax = c["L_hi"] + N
    att = W.attention_inputs(seed, c["B"], N, c["Hq"], c["Hkv"], c["D"], Lmax, c["dtype"])
    ht = W.hidden_tree(seed, c["B"], N, c["H"], c["dtype"])
    root = W.root_tokens(seed, c["B"], c["V"])
    return dict(tree=t, heads=heads, kv_len=kv_len, Lmax=Lmax, att=att, ht=ht, root=root)


if __name__ == "__main__":
    sys.exit(main())
