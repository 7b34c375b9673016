#!/usr/bin/env python
"""Benchmark: one MagicDec-style speculative round per step on one GB300 per rank.

A step is one pass of the whole hot path over one batch (the MagicDec long-context workload:
B=32, 32/8 heads x 128, bf16 KV, 64K context, gamma=4, a 512-slot draft ring, vocab 128256):
  4 x spec_draft_window_attn (draft single-query attention over the ring, appending one token)
  1 x spec_verify_attn       (gamma+1 causal queries over the full 64K cache)
  1 x spec_sample            (softmax, accept/reject, residual/bonus draw over the vocabulary)

Printed JSON line (rank 0): metric/value = verify-attention KV GB/s (algorithmic K+V bytes of
the cache / event-timed duration of the spec_verify_attn call), summed over ranks; plus
spec_sample rounds/s, tokens verified/s, draft-window GB/s, the roofline of the verify kernel
against the measured HBM copy peak, the CPU oracle timed on a bounded sample (cpu_baseline), and
an end-to-end figure through the public API with per-step host<->device copies (e2e).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads.configs import get_config  # noqa: E402

METRIC = "verify-attn KV GB/s (% HBM peak); spec_sample rounds/s; at 1 GB300"
DEFAULT_WORKLOAD = "magicdec-64k"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 126 << 20
# the bench line's sub-records: every workload that has verify attention at full size
SUB_WORKLOADS = ("llama3-70b-layer", "llama3-8b-layer", "medusa-tree-8k", "magicdec-64k")


class L2Flush:
    """Evicts L2 between timed replays: a 512 MB write replaces every line, then a 512 MB read
    replaces the written lines with clean ones.  Without the read the timed kernel would also pay
    for writing back the flush's own ~126 MB of dirty lines, a cost no kernel of the round leaves
    behind (the steps before a verify or sampling call read caches and weights)."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        self.r = torch.zeros(128 << 20, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self, k: int = 1):
        self.w.fill_(k & 0xFF)
        self.sink.copy_(self.r.sum())


L2_NOTE = "L2 flushed (512 MB write, then a 512 MB read so the lines left are clean) before every"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling a small case)")
    ap.add_argument("--context", type=int, default=0,
                    help="override the verify context length (profiling the draft-window and sampling kernels at "
                         "full size beside a small verify cache)")
    ap.add_argument("--clocks-csv", default=None, help="write the raw nvidia-smi clock samples of the timed region here")
    ap.add_argument("--no-graphs", action="store_true", help="issue every call eagerly instead of graph replays")
    ap.add_argument("--sinks", type=int, default=0, help="attention-sink slots at the front of the draft ring")
    ap.add_argument("--no-sub-configs", action="store_true",
                    help="time only --workload, not the other full-size workloads' sub-records")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: copy, read+write bytes)"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s (burst: a kernel timed alone) and where it comes from."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        if d.get("bf16_tflops"):
            return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops: cuBLAS burst)"
    return FALLBACK_BF16_TFLOPS, "fallback 1.9 PFLOP/s bf16 burst (no MEASURED_PEAKS.json)"


def profile_counters(cfg):
    """ncu counters committed for a workload's verify kernel (profiles/roofline_counters.json),
    or None when absent, taken on another kernel revision than the one built now, or when this
    run's sizes are not the workload's own (a --batch or --context override)."""
    path = os.path.join(ROOT, "profiles", "roofline_counters.json")
    if not os.path.exists(path) or cfg != get_config(cfg.name):
        return None
    d = json.load(open(path)).get(cfg.name)
    if not d or d.get("kernel_rev") != KERNEL_REVS.get(cfg.name):
        return None
    return d


# ---------------------------------------------------------------------------- distributed plumbing
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def max_over_ranks(pg, x: float, device=None) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, x: float, device=None) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, csv_path=None):
        self.proc = None
        self.gpu = gpu_index
        self.path = csv_path      # optional: keep the raw samples of the timed region

    def start(self):
        try:
            self.out = open(self.path, "w") if self.path else subprocess.DEVNULL
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            txt, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            txt, _ = self.proc.communicate()
        if self.path:
            with open(self.path, "w") as f:
                f.write(txt)
        rows = [r.split(",") for r in txt.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------- workload
def make_inputs(cfg, device, seed):
    """Seeded synthetic inputs generated on the device (torch Philox generator)."""
    import torch
    from workloads import gen
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, Hq, Hkv, D, nq, V, gamma = cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.nq, cfg.vocab, cfg.gamma
    lo, hi = cfg.ctx
    kv_len_h = np.random.default_rng([seed, 4]).integers(lo, hi + 1, size=B).astype(np.int32) if lo != hi \
        else np.full(B, lo, np.int32)
    Lmax = int(kv_len_h.max())
    dt = torch.bfloat16 if cfg.kv_dtype == "bf16" else torch.float32
    k = torch.empty((B, Hkv, Lmax, D), dtype=dt, device=device)
    v = torch.empty((B, Hkv, Lmax, D), dtype=dt, device=device)
    for b in range(B):
        k[b] = torch.randn((Hkv, Lmax, D), generator=g, device=device).to(dt)
        v[b] = torch.randn((Hkv, Lmax, D), generator=g, device=device).to(dt)
    inp = dict(k=k, v=v, kv_len_h=kv_len_h, kv_len=torch.from_numpy(kv_len_h).to(device))
    inp["q"] = torch.randn((B, nq, Hq, D), generator=g, device=device).to(dt)
    inp["o"] = torch.empty((B, nq, Hq, D), dtype=torch.float32, device=device)
    inp["tree"] = None
    W = cfg.window
    if W:
        inp["k_ring"] = torch.randn((B, Hkv, W, D), generator=g, device=device).to(dt)
        inp["v_ring"] = torch.randn((B, Hkv, W, D), generator=g, device=device).to(dt)
        inp["pos0"] = kv_len_h.copy()      # the draft has written as many tokens as the target cache holds
        inp["dq"] = torch.randn((cfg.draft_steps, B, Hq, D), generator=g, device=device).to(dt)
        inp["dk"] = torch.randn((cfg.draft_steps, B, Hkv, D), generator=g, device=device).to(dt)
        inp["dv"] = torch.randn((cfg.draft_steps, B, Hkv, D), generator=g, device=device).to(dt)
        inp["dpos"] = torch.from_numpy(np.stack([kv_len_h + s for s in range(cfg.draft_steps)])).to(device)
        inp["do"] = torch.empty((B, Hq, D), dtype=torch.float32, device=device)
    if cfg.tree_nodes:
        N = cfg.tree_nodes
        inp["tree"] = gen.random_tree(N, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
        tl = cfg.target_sigma * torch.randn((B, N, V), generator=g, device=device)
        # each node's first child carries its parent's planted argmax with probability 0.6
        tok = torch.randint(0, V, (B, N), generator=g, device=device, dtype=torch.int32)
        first = {}
        for i in range(1, N):
            first.setdefault(int(inp["tree"][i]), i)
        for p_, c_ in first.items():
            hit = torch.rand((B,), generator=g, device=device) < 0.6
            tl[hit, p_, tok[hit, c_].long()] = 30.0
        depth = int(gen_depths(inp["tree"]).max())
        inp.update(tl=tl.contiguous(), x=tok, out=torch.empty((B, depth + 1), dtype=torch.int32, device=device),
                   nodes=torch.empty((B, depth + 1), dtype=torch.int32, device=device),
                   nacc=torch.empty((B,), dtype=torch.int32, device=device))
        return inp
    z = torch.randn((B, gamma + 1, V), generator=g, device=device)
    tl = cfg.target_sigma * z
    eps = torch.randn((B, gamma, V), generator=g, device=device)
    if cfg.draft_corr > 0:
        dl = cfg.target_sigma * (cfg.draft_corr * z[:, :gamma] + float(np.sqrt(1 - cfg.draft_corr ** 2)) * eps)
    else:
        dl = tl[:, :gamma] + cfg.draft_noise_sigma * eps
    # draft tokens x_i ~ softmax(draft row i) by Gumbel-max
    gum = -torch.log(-torch.log(torch.rand((B, gamma, V), generator=g, device=device).clamp_min(1e-30)))
    x = torch.argmax(dl + gum, dim=-1).to(torch.int32)
    del gum, z, eps
    inp.update(tl=tl.contiguous(), dl=dl.contiguous(), x=x.contiguous(),
               u=torch.rand((B, gamma + 1), generator=g, device=device),
               out=torch.empty((B, gamma + 1), dtype=torch.int32, device=device),
               nacc=torch.empty((B,), dtype=torch.int32, device=device))
    return inp


def gen_depths(parent):
    d = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        d[i] = d[int(parent[i])] + 1
    return d


def step_bytes(cfg, inp):
    kvb = 2 if cfg.kv_dtype == "bf16" else 4
    kv = int(inp["kv_len_h"].sum()) * cfg.Hkv * cfg.D * 2 * kvb
    qo = cfg.B * cfg.nq * cfg.Hq * cfg.D * (kvb + 4)
    win = 0
    if cfg.window:
        valid = np.minimum(inp["pos0"] + 1, cfg.window)   # tokens visible at the first draft step
        win = int(valid.sum()) * cfg.Hkv * cfg.D * 2 * kvb + cfg.B * cfg.Hq * cfg.D * (kvb + 4)
    if cfg.tree_nodes:
        samp = cfg.B * cfg.tree_nodes * cfg.vocab * 4
    else:
        samp = cfg.B * (2 * cfg.gamma + 1) * cfg.vocab * 4 + cfg.B * 2 * cfg.vocab * 4
    return dict(verify_kv=kv, verify_total=kv + qo, window=win, sample=samp)


class Runner:
    """Holds workspaces and issues one step through the public binding."""

    def __init__(self, sv, cfg, inp, device):
        import torch
        self.sv, self.cfg, self.inp, self.torch = sv, cfg, inp, torch
        u8 = torch.uint8
        self.mode = sv.SPEC_SAMPLE_TREE_GREEDY if cfg.tree_nodes else sv.SPEC_SAMPLE_CHAIN
        self.n_sinks = 0
        self.ws_v = torch.empty(sv.spec_verify_attn_workspace(inp["q"], inp["k"], inp["o"]), dtype=u8, device=device)
        self.ws_s = torch.empty(sv.spec_sample_workspace(self.mode, inp["tl"]), dtype=u8, device=device)
        self.ws_w = None
        if cfg.window:
            self.ws_w = torch.empty(sv.spec_draft_window_attn_workspace(inp["dq"][0], inp["k_ring"], inp["do"]),
                                    dtype=u8, device=device)

    def draft(self, s):
        i = self.inp
        self.sv.spec_draft_window_attn(i["dq"][s], i["k_ring"], i["v_ring"], i["dpos"][s], i["do"],
                                       k_new=i["dk"][s], v_new=i["dv"][s], workspace=self.ws_w,
                                       n_sinks=self.n_sinks)

    def verify(self):
        i = self.inp
        self.sv.spec_verify_attn(i["q"], i["k"], i["v"], i["kv_len"], i["o"], tree_parent=i["tree"],
                                 workspace=self.ws_v)

    def sample(self):
        i = self.inp
        if self.cfg.tree_nodes:
            self.sv.spec_sample(self.mode, i["tl"], i["out"], i["nacc"], draft_tokens=i["x"], tree_parent=i["tree"],
                                out_path_nodes=i["nodes"], workspace=self.ws_s)
        else:
            self.sv.spec_sample(self.mode, i["tl"], i["out"], i["nacc"], draft_logits=i["dl"],
                                draft_tokens=i["x"], uniforms=i["u"], workspace=self.ws_s)

    def launches_per_step(self):
        """Our kernels per step by the library's launch rules (status memsets are not counted);
        used only when the captured graphs cannot be inspected.  Verify: partial + merge.  Window:
        one per-segment kernel for bf16 rings with <= 16 query rows per KV head and D 64/128, else
        see below.  Sampling: one warp-per-sequence kernel for V <= 2048, else statistics + the
        finishing kernel (cluster finish or greedy finalize)."""
        import torch
        cfg = self.cfg
        win = 0
        if cfg.window:
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            S, seg_tiles = cfg.B * cfg.Hkv, -(-cfg.window // 128)
            spc, even = -(-S // sms), -(-S * seg_tiles // sms)
            if cfg.kv_dtype == "bf16" and cfg.G <= 16 and cfg.D in (64, 128):
                per_call = 1                     # attn_window_bf16: one CTA per segment
            elif cfg.kv_dtype == "bf16" and cfg.D == 128 and cfg.G > 32:
                per_call = 3                     # append + tensor-core partial + merge
            elif cfg.kv_dtype == "bf16" and cfg.G <= 64 and spc * seg_tiles <= max(2 * even, 16):
                per_call = 1                     # whole segments per CTA: partial writes o itself
            else:
                per_call = 2                     # partial + merge (append fused into the merge)
            win = cfg.draft_steps * per_call
        samp = 1 if cfg.vocab <= 2048 else 2
        return win + 2 + samp


def count_kernel_nodes(graph):
    """Kernel nodes in a captured CUDA graph (driver API on the raw cudaGraph_t), or None."""
    import ctypes
    try:
        raw = ctypes.c_void_p(graph.raw_cuda_graph())
        cu = ctypes.CDLL("libcuda.so.1")
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(raw, None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * max(1, n.value))()
        if cu.cuGraphGetNodes(raw, nodes, ctypes.byref(n)) != 0:
            return None
        kernels = 0
        for i in range(n.value):
            t = ctypes.c_int(-1)
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) != 0:
                return None
            kernels += int(t.value == 0)   # CU_GRAPH_NODE_TYPE_KERNEL
        return kernels
    except Exception:
        return None


class GraphOps:
    """Each op of a step (the draft-window calls, verify, sample) captured once into a CUDA graph
    through the public binding and replayed, so that host launch overhead stays out of the device
    timings.  Per-op CUDA events are recorded between replays, outside the graphs."""

    def __init__(self, runner, stream):
        import torch
        self.g = {}
        self.kernels_per_step = 0          # kernel nodes over the captured ops, None if not countable
        cfg = runner.cfg
        ops = {"verify": runner.verify, "sample": runner.sample}
        if cfg.window:
            ops["draft"] = lambda: [runner.draft(s) for s in range(cfg.draft_steps)]
        with torch.cuda.stream(stream):
            for name, fn in ops.items():
                fn()                       # eager first call (module load, attributes)
                stream.synchronize()
                try:
                    g, kept = torch.cuda.CUDAGraph(keep_graph=True), True
                except TypeError:
                    g, kept = torch.cuda.CUDAGraph(), False
                with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                    fn()
                k = count_kernel_nodes(g) if kept else None
                self.kernels_per_step = None if (k is None or self.kernels_per_step is None) \
                    else self.kernels_per_step + k
                if kept:
                    g.instantiate()
                self.g[name] = g
        torch.cuda.synchronize()

    def draft(self):
        if "draft" in self.g:
            self.g["draft"].replay()

    def verify(self):
        self.g["verify"].replay()

    def sample(self):
        self.g["sample"].replay()


def time_steps(runner, K, W, pg, device, use_graphs=True, clocks_csv=None):
    """K timed steps bracketed by barrier + synchronize; per-op CUDA events on the launching stream."""
    import torch
    cfg = runner.cfg
    stream = torch.cuda.Stream(device=device) if use_graphs else torch.cuda.current_stream()
    if use_graphs:
        gops = GraphOps(runner, stream)
        do_draft, do_verify, do_sample = gops.draft, gops.verify, gops.sample
    else:
        def do_draft():
            for s in range(cfg.draft_steps if cfg.window else 0):
                runner.draft(s)
        do_verify, do_sample = runner.verify, runner.sample
    ctx = torch.cuda.stream(stream)
    ctx.__enter__()
    for _ in range(W):
        do_draft()
        do_verify()
        do_sample()
    torch.cuda.synchronize()
    n_ev = 4
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # working sets that L2 (~126 MB) could hold between steps are flushed (L2Flush)
    nb = step_bytes(cfg, runner.inp)
    flush = None
    if nb["verify_total"] + nb["sample"] < 4 * L2_BYTES:
        flush = L2Flush(device)
    barrier(pg, device)
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index, clocks_csv)
    clocks.start()
    t0 = time.perf_counter()
    start.record(stream)
    for k in range(K):
        e = evs[k]
        if flush is not None:
            flush(k)
        e[0].record(stream)
        do_draft()
        e[1].record(stream)
        do_verify()
        e[2].record(stream)
        do_sample()
        e[3].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ctx.__exit__(None, None, None)
    barrier(pg, device)
    ck = clocks.stop()
    total_ms = start.elapsed_time(end)
    if flush is not None:   # exclude the flushes: sum of the steps themselves
        total_ms = float(sum(e[0].elapsed_time(e[3]) for e in evs))
    win = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    ver = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    smp = float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    return dict(total_ms=total_ms, wall_s=wall, window_ms=win, verify_ms=ver, sample_ms=smp, clocks=ck,
                l2_flush=flush is not None, graphs=use_graphs,
                kernels_per_step=gops.kernels_per_step if use_graphs else None)


def time_commit(runner, K, device):
    """spec_commit after the step, timed alone (CUDA graph replays, events on the stream).  Chain:
    every draft accepted, so kv_len is unchanged and the op can be replayed as it is.  Tree: the
    accepted paths of the last sampling call are gathered; each replay first restores kv_len from
    a copy (a 4-byte-per-sequence device copy, included in the time)."""
    import torch
    sv, cfg, inp = runner.sv, runner.cfg, runner.inp
    stream = torch.cuda.Stream(device=device)
    kv_len = inp["kv_len"]
    backup = kv_len.clone()
    ws = torch.empty(256, dtype=torch.uint8, device=device)
    if cfg.tree_nodes:
        mode, nacc = sv.SPEC_COMMIT_TREE, inp["nacc"]

        def op():
            kv_len.copy_(backup)
            sv.spec_commit(mode, kv_len, nacc, cfg.nq, k=inp["k"], v=inp["v"], path_nodes=inp["nodes"],
                           workspace=ws, stream=stream)
    else:
        mode = sv.SPEC_COMMIT_CHAIN
        nacc = torch.full((cfg.B,), cfg.gamma, dtype=torch.int32, device=device)

        def op():
            sv.spec_commit(mode, kv_len, nacc, cfg.nq, workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        op()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            op()
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
        stream.synchronize()
        kv_len.copy_(backup)
        stream.synchronize()
    moved = 0
    if cfg.tree_nodes:
        elem = 2 if cfg.kv_dtype == "bf16" else 4
        moved = int(inp["nacc"].clamp_min(0).sum().item()) * cfg.Hkv * cfg.D * elem * 2 * 2
    return {"mode": "tree" if cfg.tree_nodes else "chain", "us": 1000 * e0.elapsed_time(e1) / K,
            "bytes_moved": moved, "includes_kv_len_restore": bool(cfg.tree_nodes)}


def time_verify_append(runner, K, device):
    """spec_verify_attn with the fused append of the nq new tokens' K/V, timed like the verify of
    the step (CUDA graph replays, L2 flushed before each, events on the stream).  k_new, v_new are
    the rows already at those cache positions, so every replay leaves the cache as it was."""
    import torch
    sv, cfg, inp = runner.sv, runner.cfg, runner.inp
    stream = torch.cuda.Stream(device=device)
    lens = inp["kv_len"].cpu().tolist()
    nq = cfg.nq
    k_new = torch.stack([inp["k"][b, :, L - nq:L].transpose(0, 1) for b, L in enumerate(lens)]).contiguous()
    v_new = torch.stack([inp["v"][b, :, L - nq:L].transpose(0, 1) for b, L in enumerate(lens)]).contiguous()

    def op():
        sv.spec_verify_attn(inp["q"], inp["k"], inp["v"], inp["kv_len"], inp["o"], tree_parent=inp["tree"],
                            workspace=runner.ws_v, stream=stream, k_new=k_new, v_new=v_new)
    flush = L2Flush(device)
    with torch.cuda.stream(stream):
        op()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            op()
        for _ in range(3):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for e0, e1 in evs:
            flush(1)
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
    elem = 2 if cfg.kv_dtype == "bf16" else 4
    return {"us": 1000 * float(np.mean([a.elapsed_time(b) for a, b in evs])),
            "bytes_appended": int(2 * cfg.B * nq * cfg.Hkv * cfg.D * elem),
            "launch": "append kernel + attention in one spec_verify_attn call (one graph)"}


def time_tree_stochastic(runner, K, device):
    """spec_sample(SPEC_SAMPLE_TREE) -- stochastic tree acceptance -- on the tree workload's shape
    (same B, N, V and tree; draft rows correlated 0.8 with the target, children drawn from their
    parent's draft row), CUDA graph replays with L2 flushed before each, events on the stream."""
    import torch
    from workloads import gen
    sv, cfg, inp = runner.sv, runner.cfg, runner.inp
    parent = inp["tree"]
    host = gen.tree_stochastic_inputs(cfg.B, parent, cfg.vocab, cfg.seed + 11)
    tl = torch.from_numpy(host["target_logits"]).to(device)
    dl = torch.from_numpy(host["draft_logits"]).to(device)
    tok = torch.from_numpy(host["node_tokens"]).to(device)
    u = torch.from_numpy(host["uniforms"]).to(device)
    cols = int(inp["out"].shape[1])
    out = torch.empty((cfg.B, cols), dtype=torch.int32, device=device)
    nodes = torch.empty_like(out)
    nacc = torch.empty((cfg.B,), dtype=torch.int32, device=device)
    ws = torch.empty(256, dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)

    def op():
        sv.spec_sample(sv.SPEC_SAMPLE_TREE, tl, out, nacc, draft_logits=dl, draft_tokens=tok, uniforms=u,
                       tree_parent=parent, out_path_nodes=nodes, workspace=ws, stream=stream)
    flush = L2Flush(device)
    with torch.cuda.stream(stream):
        op()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            op()
        for _ in range(3):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for e0, e1 in evs:
            flush(1)
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
    us = 1000 * float(np.mean([a.elapsed_time(b) for a, b in evs]))
    return {"us": us, "rounds_per_s": cfg.B / (us * 1e-6), "mean_accepted": float(nacc.float().mean().item()),
            "draft_corr": 0.8}


LM_HIDDEN = 4096   # hidden size of the LLaMA-3-8B / Vicuna-7B targets whose LM heads the workloads use


def time_lmhead(runner, K, device, plant=0.6):
    """spec_lmhead_sample -- the LM-head GEMM reduced to per-row argmaxes and the greedy rule in
    one call -- on the workload's verify rows (B x nq hidden states of width 4096) against its
    vocabulary, chain or tree as the workload is; beside it, for context, the unfused pipeline of
    the same result (cuBLAS bf16 logits, an fp32 copy, spec_sample greedy).  Inputs follow the
    LM-head recipe of the input generator (hidden N(0, 1), weight N(0, 1/d), a fraction `plant`
    of the drafts made their row's argmax) but are drawn on the device from a seeded torch
    generator, the 1 GB weight being too slow to draw on the host.  CUDA graph replays; the weight
    is larger than L2 and L2 is also flushed before each replay.  The record's "stochastic" part
    times the stochastic mode of the same call (SPEC_SAMPLE_CHAIN / SPEC_SAMPLE_TREE: logits
    written to the workspace, sampled in the same call) beside cuBLAS + spec_sample."""
    import torch
    sv, cfg = runner.sv, runner.cfg
    tree = bool(cfg.tree_nodes)
    parent = runner.inp["tree"] if tree else None
    B, R, d, V = cfg.B, cfg.nq, LM_HIDDEN, cfg.vocab
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed + 404)
    h = torch.randn((B, R, d), generator=g, device=device).to(torch.bfloat16)
    w = (torch.randn((V, d), generator=g, device=device) / (d ** 0.5)).to(torch.bfloat16)
    rng = np.random.default_rng(cfg.seed + 405)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    if tree:
        first = {}
        for c in range(1, R):
            first.setdefault(int(parent[c]), c)
        pairs = sorted(first.items())
    else:
        pairs = [(i, i + 1) for i in range(R - 1)]
    used = set()
    for b in range(B):
        for src, dst in pairs:
            t = int(rng.integers(V))
            if rng.random() < plant and t not in used:
                used.add(t)
                w[t] = (h[b, src].float() * (3.0 / d ** 0.5)).to(torch.bfloat16)
                tok[b, dst] = t
    tok_d = torch.from_numpy(tok if tree else np.ascontiguousarray(tok[:, 1:])).to(device)
    mode = sv.SPEC_SAMPLE_TREE_GREEDY if tree else sv.SPEC_SAMPLE_CHAIN_GREEDY
    cols = int(runner.inp["out"].shape[1]) if tree else R
    out = torch.empty((B, cols), dtype=torch.int32, device=device)
    nodes = torch.empty_like(out) if tree else None
    nacc = torch.empty((B,), dtype=torch.int32, device=device)
    ws = torch.empty(sv.spec_lmhead_sample_workspace(mode, h, w), dtype=torch.uint8, device=device)
    out_u, nacc_u = torch.empty_like(out), torch.empty_like(nacc)
    nodes_u = torch.empty_like(out) if tree else None
    ws_u = torch.empty(sv.spec_sample_workspace(mode, torch.empty((B, R, V), device="meta"), parent),
                       dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)

    def fused():
        sv.spec_lmhead_sample(mode, h, w, out, nacc, draft_tokens=tok_d, tree_parent=parent, out_path_nodes=nodes,
                              workspace=ws, stream=stream)

    h2 = h.view(B * R, d)
    try:   # cuBLAS with fp32 output (the fused kernel's accumulator precision), where PyTorch has it
        torch.mm(h2[:1], w[:16].t(), out_dtype=torch.float32)
        fp32_out = True
    except (TypeError, RuntimeError, NotImplementedError):
        fp32_out = False

    def unfused():
        if fp32_out:
            logits = torch.mm(h2, w.t(), out_dtype=torch.float32).view(B, R, V)
        else:
            logits = torch.matmul(h2, w.t()).float().view(B, R, V)
        sv.spec_sample(mode, logits, out_u, nacc_u, draft_tokens=tok_d, tree_parent=parent, out_path_nodes=nodes_u,
                       workspace=ws_u, stream=stream)

    flush = L2Flush(device)

    def timed(op):
        with torch.cuda.stream(stream):
            op()
            stream.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream, capture_error_mode="thread_local"):
                op()
            for _ in range(3):
                gr.replay()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
            for e0, e1 in evs:
                flush(1)
                e0.record(stream)
                gr.replay()
                e1.record(stream)
            stream.synchronize()
        return 1000 * float(np.mean([a.elapsed_time(b) for a, b in evs]))

    us = timed(fused)
    us_u = timed(unfused)
    agree = bool(torch.equal(nacc, nacc_u) and torch.equal(out, out_u))
    rows = B * R
    nbytes = V * d * 2 + rows * d * 2 + 2 * rows * ((V + 127) // 128) * 8 + B * (R + cols + 1) * 4
    peak, _ = peaks()

    # the stochastic mode of the same call: the GEMM writes the fp32 logits into the workspace
    # (L2-sized at these shapes) and spec_sample's kernels read them back within the call; draft
    # logits N(0, 4) fp32 and uniforms drawn on the device
    smode = sv.SPEC_SAMPLE_TREE if tree else sv.SPEC_SAMPLE_CHAIN
    nd = R if tree else R - 1
    dl = 2.0 * torch.randn((B, nd, V), generator=g, device=device)
    uni = torch.rand((B, R), generator=g, device=device)
    out_s, nacc_s = torch.empty_like(out), torch.empty_like(nacc)
    nodes_s = torch.empty_like(out) if tree else None
    ws_s = torch.empty(sv.spec_lmhead_sample_workspace(smode, h, w), dtype=torch.uint8, device=device)
    out_su, nacc_su = torch.empty_like(out), torch.empty_like(nacc)
    nodes_su = torch.empty_like(out) if tree else None
    ws_su = torch.empty(sv.spec_sample_workspace(smode, torch.empty((B, R, V), device="meta"), parent),
                        dtype=torch.uint8, device=device)

    def fused_s():
        sv.spec_lmhead_sample(smode, h, w, out_s, nacc_s, draft_tokens=tok_d, tree_parent=parent,
                              out_path_nodes=nodes_s, workspace=ws_s, stream=stream, draft_logits=dl, uniforms=uni)

    def unfused_s():
        if fp32_out:
            logits = torch.mm(h2, w.t(), out_dtype=torch.float32).view(B, R, V)
        else:
            logits = torch.matmul(h2, w.t()).float().view(B, R, V)
        sv.spec_sample(smode, logits, out_su, nacc_su, draft_logits=dl, draft_tokens=tok_d, uniforms=uni,
                       tree_parent=parent, out_path_nodes=nodes_su, workspace=ws_su, stream=stream)

    us_s = timed(fused_s)
    us_su = timed(unfused_s)
    # HBM bytes of the stochastic call: the weight once, the hidden rows, the draft logits and
    # uniforms (the target logits stay in L2 between the GEMM and the sampler)
    nbytes_s = V * d * 2 + rows * d * 2 + B * nd * V * 4 + B * R * 4 + B * (R + cols + 1) * 4
    stochastic = {"us": us_s, "gbs": nbytes_s / (us_s * 1e-6) / 1e9,
                  "hbm_frac": nbytes_s / (us_s * 1e-6) / 1e9 / peak, "algorithmic_bytes": int(nbytes_s),
                  "mode": "tree" if tree else "chain", "mean_accepted": float(nacc_s.float().mean().item()),
                  "unfused_us": us_su,
                  "unfused": ("cuBLAS bf16 GEMM with fp32 output -> spec_sample" if fp32_out
                              else "cuBLAS bf16 GEMM (bf16 output) -> fp32 copy -> spec_sample"),
                  "logits_bytes": rows * V * 4}
    return {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9, "hbm_frac": nbytes / (us * 1e-6) / 1e9 / peak,
            "algorithmic_bytes": int(nbytes), "rows": rows, "hidden": d, "vocab": V,
            "mode": "tree_greedy" if tree else "chain_greedy",
            "mean_accepted": float(nacc.float().mean().item()),
            "unfused_us": us_u,
            "unfused": ("cuBLAS bf16 GEMM with fp32 output -> spec_sample greedy" if fp32_out
                        else "cuBLAS bf16 GEMM (bf16 output) -> fp32 copy -> spec_sample greedy"),
            "unfused_same_tokens": agree,
            "stochastic": stochastic}


def time_e2e(runner, K, W, device):
    """The same round through the public API with host buffers.  Per step: pinned host -> device
    copies of the round's inputs (verify queries and the gamma+1 new K/V rows, the draft queries
    and new K/V rows, target and draft logits, draft tokens, uniforms), the calls, and a
    device -> host read of the emitted tokens and accepted counts, which the host waits for before
    it issues the step's successor.  The copies of step k + 1 run on a second stream into the
    other of two device input buffers while step k computes, as a serving loop overlaps its input
    transfers with compute; the verify call appends the new K/V rows to the cache itself (k_new,
    v_new, the fused append).  As a serving loop's decode step would be, the step's calls (draft
    window x4, verify with append, spec_sample) are captured once per input buffer through the
    binding into a CUDA graph and replayed each step (eager calls if capture is unavailable); the
    copies, the waits and the read-back stay outside the graphs, every step.  Returns (seconds
    per step, H2D bytes, D2H bytes, how the calls were issued)."""
    import torch
    cfg, inp, sv = runner.cfg, runner.inp, runner.sv
    B, nq = cfg.B, cfg.nq
    names = [n for n in ("q", "tl", "dl", "x", "u", "dq", "dk", "dv") if inp.get(n) is not None]
    saved = {n: inp[n] for n in names}
    host = {n: inp[n].cpu().pin_memory() for n in names}
    L = inp["kv_len_h"]
    # the verified positions' K/V rows, [B, nq, Hkv, D] as the append takes them
    host["k_new"] = torch.stack([inp["k"][b, :, L[b] - nq:L[b]].transpose(0, 1) for b in range(B)]).cpu().pin_memory()
    host["v_new"] = torch.stack([inp["v"][b, :, L[b] - nq:L[b]].transpose(0, 1) for b in range(B)]).cpu().pin_memory()
    bufs = [{n: torch.empty(t.shape, dtype=t.dtype, device=device) for n, t in host.items()} for _ in range(2)]
    out_h = torch.empty(tuple(inp["out"].shape), dtype=torch.int32).pin_memory()
    nacc_h = torch.empty((B,), dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 4 + nacc_h.numel() * 4
    comp = torch.cuda.Stream(device=device)
    copy_s = torch.cuda.Stream(device=device)
    ready = [torch.cuda.Event() for _ in range(2)]   # buffer i holds its step's inputs
    free = [torch.cuda.Event() for _ in range(2)]    # the step that read buffer i is done
    done = torch.cuda.Event()                        # the step's results are on the host

    def copy_in(k):
        i = k % 2
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(free[i])
            for n, t in host.items():
                bufs[i][n].copy_(t, non_blocking=True)
            ready[i].record(copy_s)

    def calls(i):
        b = bufs[i]
        for n in names:
            inp[n] = b[n]
        for s_ in range(cfg.draft_steps if cfg.window else 0):
            runner.draft(s_)
        sv.spec_verify_attn(inp["q"], inp["k"], inp["v"], inp["kv_len"], inp["o"], tree_parent=inp["tree"],
                            workspace=runner.ws_v, k_new=b["k_new"], v_new=b["v_new"])
        runner.sample()

    graphs = None
    try:
        with torch.cuda.stream(comp):
            for i in range(2):
                calls(i)
            comp.synchronize()
            graphs = []
            for i in range(2):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=comp, capture_error_mode="thread_local"):
                    calls(i)
                graphs.append(g)
    except Exception:
        graphs = None
        torch.cuda.synchronize()

    def compute(k):
        i = k % 2
        with torch.cuda.stream(comp):
            comp.wait_event(ready[i])
            if graphs is not None:
                graphs[i].replay()
            else:
                calls(i)
            free[i].record(comp)
            out_h.copy_(inp["out"], non_blocking=True)
            nacc_h.copy_(inp["nacc"], non_blocking=True)
            done.record(comp)

    def run(n):
        copy_in(0)
        compute(0)
        for k in range(n):
            if k + 1 < n:
                copy_in(k + 1)    # overlaps step k
            done.synchronize()    # step k's tokens and counts are on the host
            if k + 1 < n:
                compute(k + 1)

    run(W)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(K)
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / K
    inp.update(saved)
    how = ("one CUDA graph per input buffer (the step's API calls captured once), replayed each step"
           if graphs is not None else "eager calls through the binding")
    return sec, h2d, d2h, how


# ---------------------------------------------------------------------------- CPU oracle timing
def oracle_sample_run(cfg, seed, budget_s=12.0):
    """Time the CPU oracle on a bounded sample of the same workload: verify attention for whole
    (sequence, kv head) segments (all nq * G rows) and spec_sample for whole sequences."""
    from oracle import attn as oa
    from oracle import sample as osm
    from workloads import gen
    r = np.random.default_rng(seed)
    L = int(cfg.ctx[1])
    parent = None
    if cfg.tree_nodes:
        parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    nbytes = 0
    t_attn = 0.0
    segs = 0
    while t_attn < budget_s * 0.6 and segs < 16:
        q = gen.store(r.standard_normal((1, cfg.nq, cfg.G, cfg.D)).astype(np.float32), cfg.kv_dtype)
        k = gen.store(r.standard_normal((1, 1, L, cfg.D)).astype(np.float32), cfg.kv_dtype)
        v = gen.store(r.standard_normal((1, 1, L, cfg.D)).astype(np.float32), cfg.kv_dtype)
        t0 = time.perf_counter()
        oa.verify_attn(q, k, v, np.array([L]), tree_parent=parent)
        t_attn += time.perf_counter() - t0
        nbytes += L * cfg.D * 2 * cfg.kv_bytes
        segs += 1
    t_s = 0.0
    rounds = 0
    while t_s < budget_s * 0.4 and rounds < 64:
        if parent is not None:
            s = gen.tree_sample_inputs(1, parent, cfg.vocab, int(r.integers(1 << 30)))
            t0 = time.perf_counter()
            osm.tree_greedy(s["target_logits"], s["node_tokens"], parent)
        else:
            s = gen.chain_sample_inputs(1, cfg.gamma, cfg.vocab, int(r.integers(1 << 30)), cfg.target_sigma,
                                        cfg.draft_noise_sigma, cfg.draft_corr)
            t0 = time.perf_counter()
            osm.spec_sample_chain(s["target_logits"], s["draft_logits"], s["draft_tokens"], s["uniforms"])
        t_s += time.perf_counter() - t0
        rounds += 1
    return dict(kv_gbs=nbytes / t_attn / 1e9, rounds_per_s=rounds / t_s, segments=segs, rounds=rounds,
                seconds=t_attn + t_s, seg_len=L)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------------------- main
def run_reference(args, cfg):
    world, rank, local, pg = dist_setup(args)
    if rank != 0:
        return 0
    budget = 6.0
    for _ in range(args.warmup):
        oracle_sample_run(cfg, 7, budget_s=0.5)
    vals, rps, secs = [], [], 0.0
    for k in range(args.steps):
        r = oracle_sample_run(cfg, 100 + k, budget_s=budget)
        vals.append(r["kv_gbs"])
        rps.append(r["rounds_per_s"])
        secs += r["seconds"]
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "sample": "per step: whole (sequence, kv head) verify segments of "
                   f"{cfg.ctx[1]} keys and whole spec_sample sequences, ~{budget:.0f} s of CPU oracle work"},
        "spec_sample_rounds_per_s": float(np.mean(rps)),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": "NumPy float64 oracle on whole verify segments and whole sampling rounds"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def verify_flops(cfg, inp):
    """Dense-over-context flops of one verify call: 4 * sum_b L_b * Hq * nq * D (QK^T and PV)."""
    return 4 * int(inp["kv_len_h"].sum()) * cfg.Hq * cfg.nq * cfg.D


def time_draft_cold(runner, K, device):
    """One draft-window call (one appended token) with L2 flushed before every replay: the
    cold-cache figure of the draft step, beside the in-round figure where steps 2-4 re-read a
    ring that the step before left in L2."""
    import torch
    cfg, inp = runner.cfg, runner.inp
    stream = torch.cuda.Stream(device=device)
    flush = L2Flush(device)
    with torch.cuda.stream(stream):
        runner.draft(0)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            runner.draft(0)
        for _ in range(3):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for e0, e1 in evs:
            flush(1)
            e0.record(stream)
            g.replay()
            e1.record(stream)
        stream.synchronize()
        # the same measurement of a one-node graph holding a 16-byte fill: the part of the figure
        # any single-call graph pays (launch of the graph and its node), for context
        tiny = torch.empty(4, dtype=torch.int32, device=device)
        gt = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gt, stream=stream, capture_error_mode="thread_local"):
            tiny.fill_(1)
        for _ in range(3):
            gt.replay()
        evt = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for e0, e1 in evt:
            flush(1)
            e0.record(stream)
            gt.replay()
            e1.record(stream)
        stream.synchronize()
    us = 1000 * float(np.mean([a.elapsed_time(b) for a, b in evs]))
    floor = 1000 * float(np.mean([a.elapsed_time(b) for a, b in evt]))
    nb = step_bytes(cfg, inp)["window"]
    return {"us": us, "gbs": nb / (us * 1e-6) / 1e9, "bytes": nb,
            "l2": L2_NOTE.replace("L2 flushed", "flushed") + " call",
            "one_node_graph_floor_us": floor}


def time_draft_rotating(runner, K, device, copies=4, calls=16):
    """Draft-window calls back to back in one graph, each on a different copy of the rings
    (`copies` of them, together several times the size of L2), so that every call streams a ring
    the previous calls have evicted: the cold per-call figure of a run of draft steps, without the
    launch of a graph per call.  Beside it, the same run on one ring (L2-resident after the first
    call).  Returns both per-call times."""
    import torch
    cfg, inp = runner.cfg, runner.inp
    ring_bytes = inp["k_ring"].numel() * inp["k_ring"].element_size() * 2
    copies = max(copies, int(-(-3 * (126 << 20) // ring_bytes)) + 1)
    rings = [(inp["k_ring"].clone(), inp["v_ring"].clone()) for _ in range(copies)]
    i = inp
    stream = torch.cuda.Stream(device=device)
    flush = L2Flush(device)

    def run(rotate):
        for c in range(calls):
            kr, vr = rings[c % copies] if rotate else rings[0]
            s = c % cfg.draft_steps
            runner.sv.spec_draft_window_attn(i["dq"][s], kr, vr, i["dpos"][s], i["do"], k_new=i["dk"][s],
                                             v_new=i["dv"][s], workspace=runner.ws_w, n_sinks=runner.n_sinks)

    out = {}
    with torch.cuda.stream(stream):
        for rotate in (True, False):
            run(rotate)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                run(rotate)
            for _ in range(3):
                g.replay()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
            for e0, e1 in evs:
                flush(1)
                e0.record(stream)
                g.replay()
                e1.record(stream)
            stream.synchronize()
            out["rotating" if rotate else "same_ring"] = 1000 * float(np.mean([a.elapsed_time(b) for a, b in evs])) / calls
    del rings
    nb = step_bytes(cfg, inp)["window"]
    return {"us": out["rotating"], "gbs": nb / (out["rotating"] * 1e-6) / 1e9, "bytes": nb,
            "l2": f"{calls} calls back to back in one graph over {copies} copies of the rings "
                  f"({copies * ring_bytes / 1e6:.0f} MB): every call streams a ring evicted by the calls before it",
            "l2_resident": {"us": out["same_ring"], "gbs": nb / (out["same_ring"] * 1e-6) / 1e9,
                            "l2": f"the same {calls} calls on one ring, L2-resident after the first call"}}


def oracle_check_sampling(cfg, runner):
    """CPU-oracle leg: the oracle's spec_sample on the bench's own sampling inputs (copied back
    from the device), against the GPU's outputs of the last timed call.  Returns the counts the
    near-threshold rule reports separately: sequences with a decision within 1e-6 of its threshold,
    how many of them are valid outcomes and how many identical; and the mismatches elsewhere (0)."""
    from oracle import sample as osm
    inp = runner.inp
    if cfg.tree_nodes:
        parent = inp["tree"]
        out, nodes, nacc = osm.tree_greedy(inp["tl"].cpu().numpy(), inp["x"].cpu().numpy(), parent,
                                           int(inp["out"].shape[1]))
        same = bool(np.array_equal(out, inp["out"].cpu().numpy()) and np.array_equal(nacc, inp["nacc"].cpu().numpy()))
        return {"mode": "tree_greedy", "sequences": cfg.B, "near": 0, "mismatch": 0 if same else cfg.B,
                "note": "greedy argmax decisions are exact; no near-threshold band"}
    tl, dl = inp["tl"].cpu().numpy(), inp["dl"].cpu().numpy()
    x, u = inp["x"].cpu().numpy(), inp["u"].cpu().numpy()
    g_out, g_k = inp["out"].cpu().numpy(), inp["nacc"].cpu().numpy()
    r_out, r_k, near = osm.spec_sample_chain(tl, dl, x, u)
    far = ~near
    mism = int(np.sum(far & ((g_k != r_k) | np.any(g_out != r_out, axis=1))))
    idx = np.nonzero(near)[0]
    valid = int(np.sum(osm.chain_outcome_valid(tl[idx], dl[idx], x[idx], u[idx], g_out[idx], g_k[idx]))) if len(idx) else 0
    ident = int(np.sum(near & (g_k == r_k) & np.all(g_out == r_out, axis=1)))
    return {"mode": "chain", "sequences": int(cfg.B), "near": int(near.sum()), "near_valid": valid,
            "near_identical": ident, "far_mismatch": mism, "band": osm.NEAR_BAND}


def measure(cfg, args, pg, device, rank, world, full):
    """Times one workload's step (graph replays) and returns its record; with `full` also the
    extra legs (commit, verify with append, stochastic tree, LM-head, cold draft, e2e)."""
    import torch
    import speculative_decoding_verify_attn_gb300 as sv
    inp = make_inputs(cfg, device, seed=cfg.seed + 7919 * rank)
    runner = Runner(sv, cfg, inp, device)
    runner.n_sinks = args.sinks if full else 0
    nb = step_bytes(cfg, inp)
    t = time_steps(runner, args.steps, args.warmup, pg, device, use_graphs=not args.no_graphs,
                   clocks_csv=args.clocks_csv if full else None)
    total_ms = max_over_ranks(pg, t["total_ms"], device)
    ver_ms = max_over_ranks(pg, t["verify_ms"], device)
    smp_ms = max_over_ranks(pg, t["sample_ms"], device)
    win_ms = max_over_ranks(pg, t["window_ms"], device)
    kv_all = sum_over_ranks(pg, float(nb["verify_kv"]), device)
    value = kv_all / (ver_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    tpeak, tpeak_kind = tensor_peak()
    achieved = nb["verify_total"] / (t["verify_ms"] * 1e-3) / 1e9
    tflops = verify_flops(cfg, inp) / (t["verify_ms"] * 1e-3) / 1e12
    counters = profile_counters(cfg)
    rec = {
        "workload": cfg.name,
        "config": {"batch": cfg.B, "q_heads": cfg.Hq, "kv_heads": cfg.Hkv, "head_dim": cfg.D,
                   "context": list(cfg.ctx), "gamma": cfg.gamma, "tree_nodes": cfg.tree_nodes,
                   "query_rows_per_kv_head": cfg.nq * cfg.G, "window": cfg.window, "vocab": cfg.vocab,
                   "kv_dtype": cfg.kv_dtype},
        "verify_kv_gbs": value,
        "hbm_frac_verify": value / world / peak,
        "verify_ms": ver_ms,
        "verify_tflops": tflops,
        "tensor_frac_verify": tflops / tpeak,
        "tokens_verified_per_s": world * cfg.B * cfg.nq / (ver_ms * 1e-3),
        "spec_sample_rounds_per_s": world * cfg.B / (smp_ms * 1e-3),
        "sample_gbs": world * nb["sample"] / (smp_ms * 1e-3) / 1e9,
        "sample_hbm_frac": nb["sample"] / (smp_ms * 1e-3) / 1e9 / peak,
        "draft_window_gbs": (world * nb["window"] * (cfg.draft_steps or 1) / (win_ms * 1e-3) / 1e9) if cfg.window else None,
        "step_breakdown_ms": {"draft_window_x%d" % cfg.draft_steps: win_ms, "verify": ver_ms, "sample": smp_ms},
        "ms_per_step": total_ms / args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": counters.get("dram_bytes_per_launch") if counters else None,
                     "kernel": "spec_verify_attn (partial + merge, one call)", "peak_source": peak_kind},
        "tensor_roofline": {"achieved": tflops, "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
                            "flops": "4 * sum(kv_len) * Hq * nq * D (dense over the context)",
                            "peak_source": tpeak_kind,
                            "ncu_tensor_pipe_active_pct": counters.get("tensor_pipe_active_pct") if counters else None},
        "l2": (L2_NOTE + " timed step; flush time excluded" if t["l2_flush"] else
               f"inputs larger than L2: the {nb['verify_kv'] / 1e9:.2f} GB verify cache streamed each step evicts L2"
               + ("; draft steps 2-4 of a round re-read the ring (may be L2-resident)" if cfg.window else "")),
        "clocks": t["clocks"],
    }
    extra = {"t": t, "nb": nb, "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "value": value,
             "total_ms": total_ms, "ver_ms": ver_ms, "smp_ms": smp_ms, "win_ms": win_ms, "counters": counters,
             "launches_per_step": t["kernels_per_step"] if t["kernels_per_step"] is not None
                                  else runner.launches_per_step()}
    if full:
        rec["commit"] = time_commit(runner, 200, device)
        rec["verify_with_append"] = time_verify_append(runner, max(5, min(args.steps, 50)), device)
        rec["tree_stochastic_sample"] = time_tree_stochastic(runner, max(5, min(args.steps, 100)), device) \
            if cfg.tree_nodes else None
        rec["lmhead_greedy_sample"] = time_lmhead(runner, max(5, min(args.steps, 50)), device)
        if cfg.window:
            cold = time_draft_cold(runner, max(5, min(args.steps, 50)), device)
            cold["gbs"] = sum_over_ranks(pg, cold["gbs"], device)
            rec["draft_window_cold"] = cold
            rot = time_draft_rotating(runner, max(5, min(args.steps, 30)), device)
            rot["gbs"] = sum_over_ranks(pg, rot["gbs"], device)
            rot["l2_resident"]["gbs"] = sum_over_ranks(pg, rot["l2_resident"]["gbs"], device)
            rec["draft_window_cold_run"] = rot
        e2e = None
        if not args.no_e2e:
            sec, h2d, d2h, how = time_e2e(runner, max(3, args.steps // 2), 3, device)
            sec = max_over_ranks(pg, sec, device)
            e2e = {"value": sum_over_ranks(pg, float(nb["verify_kv"]), device) / sec / 1e9, "unit": "GB/s",
                   "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                   "ms_per_step": 1000 * sec, "rounds_per_s": world * cfg.B / sec, "launch": how}
        extra["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        rec["sample_near_threshold"] = oracle_check_sampling(cfg, runner)
    del runner, inp
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec, extra


def main():
    args = parse()
    cfg = get_config(args.workload)
    if args.batch or args.context:
        from workloads.configs import scaled
        cfg = scaled(cfg, B=args.batch or None, ctx=(args.context, args.context) if args.context else None)
    if args.impl == "reference":
        return run_reference(args, cfg)
    import torch
    world, rank, local, pg = dist_setup(args)
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}), flush=True)
        return 1
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from speculative_decoding_verify_attn_gb300 import build as _build
    _build.build()

    main_rec, x = measure(cfg, args, pg, device, rank, world, full=True)
    subs = {}
    if not args.no_sub_configs and not args.batch and not args.context:
        for name in SUB_WORKLOADS:
            if name != cfg.name:
                subs[name], _ = measure(get_config(name), args, pg, device, rank, world, full=False)
    t = x["t"]
    traffic = main_rec["roofline"]["traffic"]
    line = {
        "metric": METRIC, "value": x["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": x["total_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.kv_dtype, "data": "synthetic",
        "config": {"workload": cfg.name, "batch": cfg.B, "q_heads": cfg.Hq, "kv_heads": cfg.Hkv,
                   "head_dim": cfg.D, "context": list(cfg.ctx), "gamma": cfg.gamma, "window": cfg.window,
                   "draft_steps": cfg.draft_steps, "draft_sinks": args.sinks, "vocab": cfg.vocab, "kv_dtype": cfg.kv_dtype,
                   "parallelism": f"replicas x{world}",
                   "launch": "one CUDA graph per op (captured through the binding), replayed" if t["graphs"]
                             else "eager calls through the binding",
                   "l2": main_rec["l2"]},
        "hbm_frac_verify": main_rec["hbm_frac_verify"],
        "spec_sample_rounds_per_s": main_rec["spec_sample_rounds_per_s"],
        "tokens_verified_per_s": main_rec["tokens_verified_per_s"],
        "draft_window_gbs": main_rec["draft_window_gbs"],
        "draft_window_gbs_note": "in-round figure: steps 2-4 re-read a ring the step before left in L2 "
                                 "(see draft_window_cold for the L2-flushed call)" if cfg.window else None,
        "draft_window_cold": main_rec.get("draft_window_cold"),
        "draft_window_cold_run": main_rec.get("draft_window_cold_run"),
        "sample_gbs": main_rec["sample_gbs"],
        "sample_hbm_frac": main_rec["sample_hbm_frac"],
        "sample_near_threshold": main_rec.get("sample_near_threshold"),
        "step_breakdown_ms": main_rec["step_breakdown_ms"],
        "commit": main_rec["commit"],
        "verify_with_append": main_rec["verify_with_append"],
        "tree_stochastic_sample": main_rec["tree_stochastic_sample"],
        "lmhead_greedy_sample": main_rec["lmhead_greedy_sample"],
        "roofline": {"bound": "hbm", "achieved": x["achieved"], "peak": x["peak"], "unit": "GB/s",
                     "frac": x["achieved"] / x["peak"], "traffic": traffic,
                     "kernel": "spec_verify_attn (split-KV partial + merge, one call)", "peak_source": x["peak_kind"]},
        "tensor_roofline": main_rec["tensor_roofline"],
        "workloads": subs,
        "gpu_launches": x["launches_per_step"] * args.steps,
        "gpu_launches_source": "kernel nodes of the captured step graphs" if t["kernels_per_step"] is not None
                               else "launch rule of the library",
        "clocks": t["clocks"],
        "wall_s_timed": t["wall_s"],
        "e2e": x.get("e2e"),
    }
    if rank == 0 and not args.no_cpu_baseline:
        r = oracle_sample_run(cfg, 11, budget_s=15.0)
        line["cpu_baseline"] = {"value": r["kv_gbs"], "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"{r['segments']} whole verify segments ({r['seg_len']} keys x "
                                          f"{cfg.nq * cfg.G} rows) and {r['rounds']} spec_sample rounds; "
                                          f"{r['seconds']:.1f} s",
                                "spec_sample_rounds_per_s": r["rounds_per_s"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


# Revision tag of each verify kernel that profiles/roofline_counters.json was measured on; a
# counter taken on another revision is not reported.
KERNEL_REVS = {"magicdec-64k": "mma8w-kt128-v4", "llama3-70b-layer": "tc2wg-kt128-v3",
               "llama3-8b-layer": "mma8w-kt128-v4", "medusa-tree-8k": "pair-kt64-v8"}

if __name__ == "__main__":
    sys.exit(main())
