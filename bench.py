"""Benchmark of the EAGLE draft-tree verify round on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one full round over one batch: eagle_build_tree -> eagle_tree_attention (all layers)
-> eagle_tree_verify, through the C ABI, inputs resident in HBM.  Consecutive steps rotate over
several independent input sets whose combined size is far above the 129 MB L2, so no step reads
what the previous one left in L2.  Timing: CUDA events on the launching stream around exactly K
steps, a barrier and a device synchronize on both sides, max over ranks; rank 0 prints one JSON
line.  With N > 1 (torchrun) every rank runs its own replica of the workload (weak scaling; the
round has no cross-sequence exchange).

--impl reference times the fp64 CPU oracle on this machine's host cores on the same workload,
metric and unit (each step a bounded sample of the round, extrapolated to rounds/s).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
ATTN_EVERY = 16  # timed steps per attention launch bracketed by CUDA events (at most)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import datagen  # noqa: E402

METRIC = "tree-verify rounds/s (build+attn+sample) at 8B shape; tree-attn HBM GB/s vs peak"
L2_BYTES = 129e6
UNIT = "rounds/s"


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


def _peaks() -> dict:
    """Roofline denominators: the measured copy bandwidth and bf16 GEMM rates of this machine's
    GB300s (burst: a kernel timed alone; sustained: seconds of back-to-back work), else the
    fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", 1700.0)), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _side_roofline(nbytes: float, us: float, what: str) -> dict:
    """HBM roofline of a separately timed call: its algorithmic bytes over its event time."""
    pk = _peaks()
    achieved = nbytes / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes": nbytes, "timed": what,
            "peak_source": f"{pk['source']} hbm_gbs (MEASURED_PEAKS.json)"}


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: a job of N replicas is done when its last replica is."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(steps_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job rounds/s: every rank's rounds over the slowest rank's time (weak scaling)."""
    return world * steps_per_rank / (ms_max * 1e-3)


def _workload_desc(wl) -> str:
    ctx = f"ctx={wl.ctx}" if wl.ctx_min == wl.ctx else f"ctx=U[{wl.ctx_min},{wl.ctx}]"
    return (f"{wl.name}: B={wl.batch} V={wl.vocab} D={wl.depth} k={wl.topk} m={wl.keep} L={wl.layers} "
            f"Hq={wl.heads_q} Hkv={wl.heads_kv} d={wl.head_dim} {ctx} {wl.kv_dtype} KV, T={wl.temperature}")


# ---------------------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------- our arm

class Round:
    """Device buffers and pre-marshalled C-ABI arguments of one input set."""

    def __init__(self, eg, wl, seed, dev, ws, outs, temperature):
        self.wl = wl
        B, R, V, n = wl.batch, wl.rows, wl.vocab, wl.nodes
        self.draft = datagen.draft_logits(B, R, V, seed, dev)
        self.root = datagen.root_tokens(B, V, seed, dev)
        self.attn = datagen.attention_inputs(wl, seed, dev)
        self.u = datagen.uniforms(B, n, seed, dev)
        # the target logits follow the tree of this round (built once here, outside timing)
        tree = eg.build_tree(self.draft, self.root, depth=wl.depth, topk=wl.topk, keep=wl.keep, ws=ws)
        self.target = datagen.target_logits(self.draft, tree["node_row"], datagen.noise_sigmas(wl, seed), seed)
        torch.cuda.synchronize()
        P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
        self.tcfg = eg.TreeCfg(B, V, wl.depth, wl.topk, wl.keep, 1.0)
        dt = eg.EAGLE_DTYPE_F32 if wl.kv_dtype == "f32" else eg.EAGLE_DTYPE_BF16
        self.acfg = eg.AttnCfg(B, wl.layers, n, wl.heads_q, wl.heads_kv, wl.head_dim, wl.max_seq, dt, 0.0)
        self.vcfg = eg.VerifyCfg(B, V, wl.depth, wl.topk, wl.keep, float(temperature))
        a = self.attn
        self.build_args = (ctypes.byref(self.tcfg), P(self.draft), P(self.root), P(outs["tokens"]),
                           P(outs["parents"]), P(outs["depths"]), P(outs["node_row"]), P(outs["mask"]),
                           P(outs["node_logv"]))
        self.attn_args = (ctypes.byref(self.acfg), P(a["q"]), P(a["k_cache"]), P(a["v_cache"]), P(a["ctx_len"]),
                          P(a["k_tree"]), P(a["v_tree"]), P(outs["mask"]), P(outs["attn_out"]))
        self.verify_args = (ctypes.byref(self.vcfg), P(self.target), P(self.draft), P(outs["tokens"]),
                            P(outs["parents"]), P(outs["node_row"]), P(self.u), P(outs["out_tokens"]),
                            P(outs["out_len"]), P(outs["out_path"]), None)

    def bytes_per_set(self) -> int:
        ts = [self.draft, self.root, self.u, self.target] + [v for v in self.attn.values()]
        return sum(t.numel() * t.element_size() for t in ts)


def run_ours(args, rank, world, dev) -> dict | None:
    import eagle_draft_tree_gb300 as eg

    lib = eg.load()
    wl = datagen.WORKLOADS[args.workload]
    T = wl.temperature if args.temperature is None else args.temperature
    B, n, D = wl.batch, wl.nodes, wl.depth
    ws = eg.Workspace(device=dev)
    need = max(lib.eagle_build_tree_workspace_size(ctypes.byref(eg.TreeCfg(B, wl.vocab, D, wl.topk, wl.keep, 1.0))),
               lib.eagle_tree_attention_workspace_size(ctypes.byref(eg.AttnCfg(
                   B, wl.layers, n, wl.heads_q, wl.heads_kv, wl.head_dim, wl.max_seq,
                   0 if wl.kv_dtype == "f32" else 1, 0.0))),
               lib.eagle_tree_verify_workspace_size(ctypes.byref(eg.VerifyCfg(B, wl.vocab, D, wl.topk, wl.keep, T))))
    ws.reserve(need)
    outs = {k: torch.empty((B, n), dtype=torch.int32, device=dev) for k in ("tokens", "parents", "depths", "node_row")}
    outs["mask"] = torch.empty((B, n), dtype=torch.int64, device=dev)
    outs["node_logv"] = torch.empty((B, n), dtype=torch.float32, device=dev)
    outs["out_tokens"] = torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    outs["out_len"] = torch.empty((B,), dtype=torch.int32, device=dev)
    outs["out_path"] = torch.empty((B, D), dtype=torch.int32, device=dev)
    kvdt = torch.float32 if wl.kv_dtype == "f32" else torch.bfloat16
    outs["attn_out"] = torch.empty((wl.layers, B, n, wl.heads_q, wl.head_dim), dtype=kvdt, device=dev)

    sets = [Round(eg, wl, 1000 * rank + 17 * s + args.seed, dev, ws, outs, T) for s in range(args.sets)]
    set_bytes = sets[0].bytes_per_set()
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    wsp, wsn = ws.ptr, ctypes.c_size_t(ws.nbytes)
    launches = [0]

    def step(rd: Round, ev: tuple | None = None, sp=None):
        sp = sp or sptr
        st = lib.eagle_build_tree(*rd.build_args, wsp, wsn, sp)
        c = lib.eagle_last_launch_count()
        if ev is not None:
            ev[0].record(stream)
        st |= lib.eagle_tree_attention(*rd.attn_args, wsp, wsn, sp)
        c += lib.eagle_last_launch_count()
        if ev is not None:
            ev[1].record(stream)
        st |= lib.eagle_tree_verify(*rd.verify_args, wsp, wsn, sp)
        c += lib.eagle_last_launch_count()
        if st != 0:
            raise RuntimeError(f"C-ABI call failed with status {st}")
        launches[0] += c
        return c

    for i in range(args.warmup):
        step(sets[i % len(sets)])
    torch.cuda.synchronize(dev)
    if ws.status(stream) != 0:
        raise RuntimeError("device status not OK after warm-up")

    # --graph: each input set's round captured once as a CUDA graph (the library allocates nothing
    # and never synchronises the host, so its calls capture whole) and replayed by the timed
    # rounds, the rounds that bracket the attention launch with events running the calls
    # directly.  Measured slower than direct launches (127.7 against 134.5 us a round at the 8B
    # shape): a graph boundary ends the programmatic overlap of one round's last launch with the
    # next round's first, so by default every round's calls are launched directly.
    graphs = []
    if args.graph:
        for rd in sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                n_cap = step(rd, sp=ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
            launches[0] -= n_cap  # captured, not run
            graphs.append((g, n_cap))
        for g, _ in graphs:
            g.replay()
        torch.cuda.synchronize(dev)
        if ws.status(stream) != 0:
            raise RuntimeError("device status not OK after the graph warm-up")

    K = args.steps
    attn_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches[0] = 0
    e0.record(stream)
    # The attention launch is bracketed by events on every `every`-th step only: an event recorded
    # between two launches ends the programmatic overlap of the round's kernels, which costs about
    # 7 us on every bracketed round.  Short runs bracket every 4th step (5 launches at K = 20).
    every = max(4, min(ATTN_EVERY, K // 8))
    sampled = [i for i in range(K) if i % every == 0]
    for i in range(K):
        if i % every == 0 or not graphs:
            step(sets[i % len(sets)], attn_ev[i] if i % every == 0 else None)
        else:
            g, n_cap = graphs[i % len(sets)]
            g.replay()
            launches[0] += n_cap
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    attn_ms = statistics.mean(attn_ev[i][0].elapsed_time(attn_ev[i][1]) for i in sampled)
    gpu_launches = launches[0]
    ms = max_over_ranks(ms, world, dev)
    if ws.status(stream) != 0:
        raise RuntimeError("device status not OK after the timed steps")

    # mean committed length (synthetic inputs; not comparable to the pages' acceptance lengths)
    lens = []
    for rd in sets:
        step(rd)
        lens.append(outs["out_len"].double().mean().item())
    mean_len = statistics.mean(lens)

    # end to end: per-round inputs from pinned host memory, the three calls, results back to host
    e2e = run_e2e(eg, lib, wl, sets[0], outs, ws, stream, dev, min(K, args.e2e_steps), world)
    commit = run_kv_commit(eg, lib, wl, sets[0], outs, ws, stream, dev)
    draft_attn = run_draft_attention(eg, lib, wl, ws, stream, dev)
    static = run_static_tree(eg, lib, wl, ws, stream, dev)
    sampled_build = run_sampled_build(eg, lib, wl, ws, stream, dev)
    attn_workloads = run_attention_workloads(eg, lib, ws, stream, dev, args.attn_launches) if args.attn_launches > 0 else {}

    bytes_ = datagen.bytes_of(wl, ctx_total=float(sets[0].attn["ctx_len"].sum().item()))
    peaks = _peaks()
    attn_bytes = bytes_["attention"]
    achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
    value = job_rate(K, world, ms)
    metric_bytes = bytes_["metric"]
    bf16 = wl.kv_dtype == "bf16"
    l2_note = (f"{len(sets)} rotating input sets of {set_bytes / 1e6:.0f} MB each (> 129 MB L2)"
               if set_bytes > L2_BYTES else
               f"{len(sets)} rotating input sets of {set_bytes / 1e6:.3g} MB each (L2-resident: a parity-size workload)")
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if bf16 else "f32", "data": "synthetic",
        "config": {"workload": _workload_desc(wl), "temperature": T, "parallelism": f"replicas x{world}",
                   "l2": l2_note,
                   "launch": ("each input set's round captured as a CUDA graph and replayed; the rounds that "
                              "bracket the attention launch with events call the library directly")
                             if graphs else "every round's calls launched directly",
                   "dtype_detail": ("bf16 K/V/Q/O with fp32 softmax and accumulation; fp32 logits" if bf16 else
                                    "fp32 K/V/Q/O, softmax and accumulation; fp32 logits")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": _traffic(attn_bytes) if wl.name == "llama31_8b" else None,
                     "kernel": "tree_attn_tc_kernel" if wl.kv_dtype == "bf16" else "tree_attn_f32_kernel",
                     "algorithmic_bytes": attn_bytes, "avg_launch_ms": attn_ms,
                     "launch_samples": f"CUDA events around the attention launch of every {every}th timed "
                                       f"step ({len(sampled)} launches)",
                     "frac_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                     "loop_check": _loop_check(attn_workloads, wl.name),
                     "peak_source": f"{peaks['source']} hbm_gbs (MEASURED_PEAKS.json)"},
        "end_to_end_hbm": {"metric_bytes": metric_bytes, "exact_bytes": bytes_["exact"],
                           "gbs": metric_bytes / (ms / K * 1e-3) / 1e9,
                           "frac": metric_bytes / (ms / K * 1e-3) / 1e9 / peaks["hbm_gbs"],
                           "frac_nominal": metric_bytes / (ms / K * 1e-3) / 1e9 / NOMINAL_HBM_GBS},
        "e2e": e2e, "gpu_launches": gpu_launches, "clocks": clocks, "mean_committed": mean_len,
        "kv_commit": commit, "draft_attention": draft_attn, "static_tree": static, "sampled_build": sampled_build,
        "attention_workloads": attn_workloads,
    }
    return res


def run_e2e(eg, lib, wl, rd: Round, outs, ws, stream, dev, steps, world) -> dict:
    """The same round through the public calls with host inputs: every step copies the round's
    inputs (logits, uniforms, root tokens, q and the tree's K/V, context lengths) from pinned host
    memory and reads the committed tokens back.  The KV cache is decoder state resident on the
    device, as in any serving stack.

    The copies run on their own stream, in the order the calls need them (the draft rows and
    root tokens for the build, then the attention's inputs, then the target rows and uniforms
    for the verification), and each call waits only for its own inputs, so a round's later
    copies overlap its earlier kernels.  Two device sets of inputs alternate between rounds: a
    round's copies wait only until the round before the previous one has finished with its set."""
    names = [("draft", rd.draft), ("root", rd.root), ("q", rd.attn["q"]), ("k_tree", rd.attn["k_tree"]),
             ("v_tree", rd.attn["v_tree"]), ("ctx_len", rd.attn["ctx_len"]), ("target", rd.target), ("u", rd.u)]
    stages = [("draft", "root"), ("q", "k_tree", "v_tree", "ctx_len"), ("target", "u")]
    host = {k: t.detach().cpu().pin_memory() for k, t in names}
    dsets = [dict(names), {k: torch.empty_like(t) for k, t in names}]
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    a = rd.attn

    def call_args(d):
        return ((ctypes.byref(rd.tcfg), P(d["draft"]), P(d["root"]), P(outs["tokens"]), P(outs["parents"]),
                 P(outs["depths"]), P(outs["node_row"]), P(outs["mask"]), P(outs["node_logv"])),
                (ctypes.byref(rd.acfg), P(d["q"]), P(a["k_cache"]), P(a["v_cache"]), P(d["ctx_len"]),
                 P(d["k_tree"]), P(d["v_tree"]), P(outs["mask"]), P(outs["attn_out"])),
                (ctypes.byref(rd.vcfg), P(d["target"]), P(d["draft"]), P(outs["tokens"]), P(outs["parents"]),
                 P(outs["node_row"]), P(d["u"]), P(outs["out_tokens"]), P(outs["out_len"]), P(outs["out_path"]),
                 None))
    args = [call_args(d) for d in dsets]
    out_h = torch.empty(outs["out_tokens"].shape, dtype=torch.int32).pin_memory()
    len_h = torch.empty(outs["out_len"].shape, dtype=torch.int32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 4 + len_h.numel() * 4
    sptr = ctypes.c_void_p(stream.cuda_stream)
    wsp, wsn = ws.ptr, ctypes.c_size_t(ws.nbytes)
    cs = torch.cuda.Stream(dev)
    ev_in = [[torch.cuda.Event() for _ in stages] for _ in dsets]
    ev_done = [torch.cuda.Event() for _ in dsets]
    calls = (lib.eagle_build_tree, lib.eagle_tree_attention, lib.eagle_tree_verify)
    rounds = [0]

    def one():
        k = rounds[0] % 2
        rounds[0] += 1
        d = dsets[k]
        cs.wait_event(ev_done[k])  # the round two before this one is done with set k
        with torch.cuda.stream(cs):
            for si, stage in enumerate(stages):
                for name in stage:
                    d[name].copy_(host[name], non_blocking=True)
                ev_in[k][si].record(cs)
        st = 0
        for si, call in enumerate(calls):
            stream.wait_event(ev_in[k][si])
            st |= call(*args[k][si], wsp, wsn, sptr)
        if st:
            raise RuntimeError(f"C-ABI call failed with status {st}")
        ev_done[k].record(stream)
        out_h.copy_(outs["out_tokens"], non_blocking=True)
        len_h.copy_(outs["out_len"], non_blocking=True)

    for _ in range(3):
        one()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs.wait_event(e0)  # no copy of the timed rounds starts before the timed region
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # the host -> device ceiling: one copy of a round's input bytes from pinned memory, alone
    hb = torch.empty(h2d // 4, dtype=torch.float32).pin_memory()
    db = torch.empty(h2d // 4, dtype=torch.float32, device=dev)
    for _ in range(3):
        db.copy_(hb, non_blocking=True)
    torch.cuda.synchronize(dev)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(10):
        db.copy_(hb, non_blocking=True)
    c1.record()
    torch.cuda.synchronize(dev)
    peak = hb.numel() * 4 / (c0.elapsed_time(c1) / 10) / 1e6
    achieved = h2d * steps / ms / 1e6
    del hb, db
    return {"value": job_rate(steps, world, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "pipeline": "inputs copied on a second stream in the order the calls need them; two device "
                        "input sets alternate between rounds",
            "roofline": {"bound": "h2d", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": "one pinned host -> device copy of a round's input bytes, timed alone"}}


def run_kv_commit(eg, lib, wl, rd: Round, outs, ws, stream, dev, calls: int = 200) -> dict:
    """eagle_kv_commit after the round (not part of the round's metric): the committed nodes' keys
    and values appended to a cache with room for them (the round's own cache is full).  Timed
    with CUDA events over `calls` launches of the same commit."""
    a = rd.attn
    L, B, n, Hkv, d = a["k_tree"].shape
    ctx = a["ctx_len"]
    S = int(ctx.max().item()) + wl.depth + 8
    kc = torch.zeros((L, B, S, Hkv, d), dtype=a["k_tree"].dtype, device=dev)
    vc = torch.zeros_like(kc)
    new_ctx = torch.empty_like(ctx)
    cfg = eg.AttnCfg(B, L, n, Hkv, Hkv, d, S, eg.EAGLE_DTYPE_BF16 if kc.dtype == torch.bfloat16 else eg.EAGLE_DTYPE_F32,
                     0.0)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    cargs = (ctypes.byref(cfg), wl.depth, P(a["k_tree"]), P(a["v_tree"]), P(outs["out_path"]), P(outs["out_len"]),
             P(ctx), P(kc), P(vc), P(new_ctx), ws.ptr, ctypes.c_size_t(ws.nbytes), ctypes.c_void_p(stream.cuda_stream))
    for _ in range(3):
        if lib.eagle_kv_commit(*cargs) != 0:
            raise RuntimeError("eagle_kv_commit failed")
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(calls):
        lib.eagle_kv_commit(*cargs)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ws.status(stream) != 0:
        raise RuntimeError("device status not OK after the KV commits")
    us = e0.elapsed_time(e1) / calls * 1e3
    rows = int(outs["out_len"].sum().item())
    moved = 2 * 2 * L * rows * Hkv * d * kc.element_size()  # K and V, read and written
    return {"us": us, "rows_per_sequence": rows / B, "bytes_moved": moved, "gbs": moved / (us * 1e-6) / 1e9,
            "roofline": _side_roofline(moved, us, "kv_commit_kernel"),
            "note": "not in the round's metric; latency-bound (a few KB per layer and sequence)"}


def run_draft_attention(eg, lib, wl, ws, stream, dev, calls: int = 200) -> dict:
    """Tree attention at the draft model's shape (not part of the round's metric): one decoder
    layer with the workload's heads, one sequence at its context length, the tree as a draft step
    sees it (n = 1 + k, 1 + 3k, 1 + 6k nodes).  Timed with CUDA events over `calls` launches."""
    res = {}
    g = torch.Generator(device=dev).manual_seed(5)
    ctx = int(wl.ctx)
    S = ctx + 64
    kc = torch.randn((1, 1, S, wl.heads_kv, wl.head_dim), generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn_like(kc)
    ctx_t = torch.tensor([ctx], dtype=torch.int32, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    for n in (1 + wl.topk, 1 + 3 * wl.topk, 1 + 6 * wl.topk):
        if n > 64:
            continue
        q = torch.randn((1, 1, n, wl.heads_q, wl.head_dim), generator=g, device=dev).to(torch.bfloat16)
        kt = torch.randn((1, 1, n, wl.heads_kv, wl.head_dim), generator=g, device=dev).to(torch.bfloat16)
        vt = torch.randn_like(kt)
        mask = torch.tensor([[(1 << (i + 1)) - 1 for i in range(n)]], dtype=torch.int64, device=dev)
        out = torch.empty_like(q)
        cfg = eg.AttnCfg(1, 1, n, wl.heads_q, wl.heads_kv, wl.head_dim, S, eg.EAGLE_DTYPE_BF16, 0.0)
        need = lib.eagle_tree_attention_workspace_size(ctypes.byref(cfg))
        ws.reserve(need)
        args = (ctypes.byref(cfg), P(q), P(kc), P(vc), P(ctx_t), P(kt), P(vt), P(mask), P(out), ws.ptr,
                ctypes.c_size_t(ws.nbytes), ctypes.c_void_p(stream.cuda_stream))
        for _ in range(5):
            if lib.eagle_tree_attention(*args) != 0:
                raise RuntimeError("eagle_tree_attention failed")
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(calls):
            lib.eagle_tree_attention(*args)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[f"n{n}_us"] = e0.elapsed_time(e1) / calls * 1e3
        es = 2  # bf16
        nbytes = (2 * ctx * wl.heads_kv * wl.head_dim * es + 2 * n * wl.heads_q * wl.head_dim * es
                  + 2 * n * wl.heads_kv * wl.head_dim * es + n * 8)  # K/V context, q and out, tree K/V, masks
        res["roofline"] = _side_roofline(nbytes, res[f"n{n}_us"], f"tree attention at n={n} (split + merge)")
    if ws.status(stream) != 0:
        raise RuntimeError("device status not OK after the draft-shape attention")
    res["shape"] = f"L=1 B=1 Hq={wl.heads_q} Hkv={wl.heads_kv} d={wl.head_dim} ctx={ctx}"
    res["note"] = "not in the round's metric; the unit's context is split over several CTAs and merged"
    return res


def run_static_tree(eg, lib, wl, ws, stream, dev, calls: int = 200) -> dict:
    """eagle_build_static_tree (not part of the round's metric): the chain of the workload's depth
    and a 21-node template (the root with 4 children, each with 4), at the workload's batch and
    vocabulary.  Timed with CUDA events over `calls` launches."""
    res = {}
    B, V = wl.batch, wl.vocab
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    for name, tmpl in (("chain", eg.chain_template(wl.depth)), ("tree_4x4", [-1] + [0] * 4 + [i for i in (1, 2, 3, 4) for _ in range(4)])):
        R = len(set(tmpl[1:]))
        draft = datagen.draft_logits(B, R, V, 3, dev)
        root = datagen.root_tokens(B, V, 3, dev)
        n = len(tmpl)
        o = {k: torch.empty((B, n), dtype=torch.int32, device=dev) for k in ("tokens", "parents", "depths", "node_row")}
        mask = torch.empty((B, n), dtype=torch.int64, device=dev)
        logv = torch.empty((B, n), dtype=torch.float32, device=dev)
        cfg = eg.static_tree_cfg(B, V, tmpl, 1.0)
        ws.reserve(lib.eagle_build_static_tree_workspace_size(ctypes.byref(cfg)))
        args = (ctypes.byref(cfg), P(draft), P(root), P(o["tokens"]), P(o["parents"]), P(o["depths"]),
                P(o["node_row"]), P(mask), P(logv), ws.ptr, ctypes.c_size_t(ws.nbytes),
                ctypes.c_void_p(stream.cuda_stream))
        for _ in range(5):
            if lib.eagle_build_static_tree(*args) != 0:
                raise RuntimeError("eagle_build_static_tree failed")
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(calls):
            lib.eagle_build_static_tree(*args)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[f"{name}_n{n}_us"] = e0.elapsed_time(e1) / calls * 1e3
        if name == "chain":
            res["roofline"] = _side_roofline(B * R * V * 4, res[f"{name}_n{n}_us"],
                                             f"chain of {wl.depth}: row top-k + static tree kernel")
    if ws.status(stream) != 0:
        raise RuntimeError("device status not OK after the static builds")
    res["note"] = f"not in the round's metric; B={B} V={V}, draft rows L2-warm across calls"
    return res


def _loop_check(sweep: dict, name: str):
    """The same kernel's time from the attention-only loop of the sweep (many launches), beside the
    in-round samples of the headline roofline."""
    r = sweep.get(name)
    if not r:
        return None
    return {"us_per_launch": r["us_per_launch"], "launches": r["launches"], "frac": r["roofline"]["frac"]}


def run_attention_workloads(eg, lib, ws, stream, dev, launches: int = 100) -> dict:
    """Tree attention alone on every bf16 workload's shape (the round's dominant kernel), each
    timed with CUDA events over `launches` back-to-back launches of the whole-model call (all
    layers, the batch, the workload's tree from eagle_build_tree), HBM-cold: the KV cache of a
    launch is far larger than the L2, and the 8B shape alternates two input sets.  Reported per
    workload: the time per launch, the HBM roofline (algorithmic bytes: KV cache, tree K/V, Q and
    O) against the measured copy peak and the nominal HBM rate, and the tensor roofline (QK^T and
    PV flops) against the measured bf16 rates.  At the 8B shape the same attention also runs as
    one launch per layer (a target model interleaves its layers with other work), 32 launches."""
    pk = _peaks()
    out = {}
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    sptr = ctypes.c_void_p(stream.cuda_stream)
    for name in ("llama31_8b", "vicuna_13b", "llama2_70b_b4", "serving_b64"):
        wl = datagen.WORKLOADS[name]
        B, n, L = wl.batch, wl.nodes, wl.layers
        nsets = 2 if name == "llama31_8b" else 1
        sets = []
        for s in range(nsets):
            seed = 40 + s
            inp = datagen.attention_inputs(wl, seed, dev)
            draft = datagen.draft_logits(B, wl.rows, wl.vocab, seed, dev)
            tree = eg.build_tree(draft, datagen.root_tokens(B, wl.vocab, seed, dev), depth=wl.depth, topk=wl.topk,
                                 keep=wl.keep, ws=ws)
            del draft
            inp["mask"] = tree["mask"]
            inp["out"] = torch.empty_like(inp["q"])
            sets.append(inp)
        cfg = eg.AttnCfg(B, L, n, wl.heads_q, wl.heads_kv, wl.head_dim, wl.max_seq, eg.EAGLE_DTYPE_BF16, 0.0)
        ws.reserve(lib.eagle_tree_attention_workspace_size(ctypes.byref(cfg)))
        wsp, wsn = ws.ptr, ctypes.c_size_t(ws.nbytes)
        args = [(ctypes.byref(cfg), P(a["q"]), P(a["k_cache"]), P(a["v_cache"]), P(a["ctx_len"]), P(a["k_tree"]),
                 P(a["v_tree"]), P(a["mask"]), P(a["out"]), wsp, wsn, sptr) for a in sets]
        for i in range(3):
            if lib.eagle_tree_attention(*args[i % nsets]) != 0:
                raise RuntimeError(f"eagle_tree_attention failed ({name})")
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(launches):
            lib.eagle_tree_attention(*args[i % nsets])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) / launches * 1e3
        ctx_total = float(sets[0]["ctx_len"].sum().item())
        nbytes = datagen.bytes_of(wl, ctx_total=ctx_total)["attention"]
        flops = datagen.attention_flops(wl, ctx_total=ctx_total)
        gbs = nbytes / (us * 1e-6) / 1e9
        tfs = flops / (us * 1e-6) / 1e12
        res = {"us_per_launch": us, "launches": launches, "algorithmic_bytes": nbytes, "flops": flops,
               "flop_per_byte": flops / nbytes,
               "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                            "frac": gbs / pk["hbm_gbs"], "frac_nominal": gbs / NOMINAL_HBM_GBS,
                            "nominal_peak": NOMINAL_HBM_GBS,
                            "peak_source": f"{pk['source']} hbm_gbs (MEASURED_PEAKS.json)"},
               "tensor": {"achieved": tfs, "unit": "TFLOP/s", "frac_sustained": tfs / pk["bf16_tflops_sustained"],
                          "frac_burst": tfs / pk["bf16_tflops"], "peak_sustained": pk["bf16_tflops_sustained"],
                          "peak_burst": pk["bf16_tflops"]},
               "shape": _workload_desc(wl), "l2": f"{nsets} input set(s), KV cache {datagen.bytes_of(wl, ctx_total)['kv'] / 1e6:.0f} MB"}
        if name == "llama31_8b":
            # one launch per layer: the layer's slices of q, the caches, the tree K/V and the output
            a = sets[0]
            cfg1 = eg.AttnCfg(B, 1, n, wl.heads_q, wl.heads_kv, wl.head_dim, wl.max_seq, eg.EAGLE_DTYPE_BF16, 0.0)
            ws.reserve(lib.eagle_tree_attention_workspace_size(ctypes.byref(cfg1)))  # the context split's partials
            wsp, wsn = ws.ptr, ctypes.c_size_t(ws.nbytes)
            largs = [(ctypes.byref(cfg1), P(a["q"][l]), P(a["k_cache"][l]), P(a["v_cache"][l]), P(a["ctx_len"]),
                      P(a["k_tree"][l]), P(a["v_tree"][l]), P(a["mask"]), P(a["out"][l]), wsp, wsn, sptr)
                     for l in range(L)]
            reps = max(4, launches // L)
            for la in largs:
                lib.eagle_tree_attention(*la)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for _ in range(reps):
                for la in largs:
                    lib.eagle_tree_attention(*la)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            us_l = e0.elapsed_time(e1) / reps * 1e3
            gbs_l = nbytes / (us_l * 1e-6) / 1e9
            res["per_layer_launches"] = {"us_all_layers": us_l, "us_per_layer": us_l / L, "rounds": reps,
                                         "achieved_gbs": gbs_l, "frac": gbs_l / pk["hbm_gbs"],
                                         "note": f"{L} launches of one layer each; a layer's KV is read again only "
                                                 f"after the other {L - 1} layers', so every launch is HBM-cold"}
        if ws.status(stream) != 0:
            raise RuntimeError(f"device status not OK after the attention sweep ({name})")
        out[name] = res
        del sets, args
        torch.cuda.empty_cache()
    return out


def run_sampled_build(eg, lib, wl, ws, stream, dev, calls: int = 100) -> dict:
    """The dynamic build with sampled children (eagle_build_tree_sampled) and as a stepwise build
    (eagle_build_begin, D - 1 eagle_build_expand, eagle_build_finalize), beside the greedy
    one-call build, on the workload's rows (not part of the round's metric).  CUDA events over
    `calls` builds each."""
    B, V, D, k, m = wl.batch, wl.vocab, wl.depth, wl.topk, wl.keep
    R = 1 + (D - 1) * k
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    draft = datagen.draft_logits(B, R, V, 5, dev)
    cu = datagen.child_uniforms(B, R, k, 5, dev)
    root = datagen.root_tokens(B, V, 5, dev)
    rows = [draft[:, :1].contiguous()] + [draft[:, 1 + (f - 1) * k:1 + f * k].contiguous() for f in range(1, D)]
    us = [cu[:, :1].contiguous()] + [cu[:, 1 + (f - 1) * k:1 + f * k].contiguous() for f in range(1, D)]
    n = m + 1
    o = {key: torch.empty((B, n), dtype=torch.int32, device=dev) for key in ("tokens", "parents", "depths", "node_row")}
    mask = torch.empty((B, n), dtype=torch.int64, device=dev)
    logv = torch.empty((B, n), dtype=torch.float32, device=dev)
    ft = torch.empty((B, k), dtype=torch.int32, device=dev)
    fp = torch.empty((B, k), dtype=torch.int32, device=dev)
    cfg = eg.tree_cfg(B, V, D, k, m, 1.0)
    ws.reserve(lib.eagle_build_tree_workspace_size(ctypes.byref(cfg)))
    s = ctypes.c_void_p(stream.cuda_stream)
    wsz = ctypes.c_size_t(ws.nbytes)
    outs = (P(o["tokens"]), P(o["parents"]), P(o["depths"]), P(o["node_row"]), P(mask), P(logv))

    def greedy():
        return lib.eagle_build_tree(ctypes.byref(cfg), P(draft), P(root), *outs, ws.ptr, wsz, s)

    def sampled():
        return lib.eagle_build_tree_sampled(ctypes.byref(cfg), P(draft), P(cu), P(root), *outs, ws.ptr, wsz, s)

    def stepwise():
        st = lib.eagle_build_begin(ctypes.byref(cfg), P(rows[0]), P(us[0]), ws.ptr, wsz, P(ft), P(fp), s)
        for f in range(1, D):
            st = st or lib.eagle_build_expand(ctypes.byref(cfg), f, P(rows[f]), P(us[f]), ws.ptr, wsz, P(ft), P(fp), s)
        return st or lib.eagle_build_finalize(ctypes.byref(cfg), P(root), ws.ptr, wsz, *outs, s)

    res = {}
    for name, fn in (("greedy_us", greedy), ("sampled_us", sampled), ("stepwise_sampled_us", stepwise)):
        for _ in range(5):
            if fn() != 0:
                raise RuntimeError(f"{name}: build call failed")
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(calls):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = e0.elapsed_time(e1) / calls * 1e3
    if ws.status(stream) != 0:
        raise RuntimeError("device status not OK after the sampled builds")
    res["roofline"] = _side_roofline(B * R * V * 4, res["sampled_us"], "row_sample_kernel + tree_select_kernel")
    res["note"] = (f"not in the round's metric; B={B} V={V} D={D} k={k} m={m}; the stepwise build is "
                   f"{2 * D} launches with no draft model between them; draft rows L2-warm across calls")
    return res


def attention_source_hash() -> str:
    """sha256[:16] of the tensor-core attention kernel's source file."""
    src = os.path.join(ROOT, "eagle_draft_tree_gb300", "csrc", "tree_attention_tc.cu")
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def _traffic(attn_bytes: float):
    """DRAM bytes per attention launch from the committed ncu summary, if it was taken on the
    current attention kernel source (else null)."""
    path = os.path.join(ROOT, "profiles", "tree_attention_llama31_8b.md")
    if not os.path.exists(path):
        return None
    h = attention_source_hash()
    fields = {}
    for line in open(path):
        if line.startswith("- ") and ": " in line:
            k, v = line[2:].split(": ", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source sha256[:16]") != h:
        return None
    try:
        return float(fields["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------------- CPU oracle

def side_cpu_baselines(wl, seed: int) -> dict:
    """The fp64 oracle on the separately timed calls' shapes (one call each, on the host cores),
    beside their GPU timings: the KV commit, tree attention at the draft shape (the largest n),
    the static chain and the sampled-children build."""
    import numpy as np

    import oracle

    nthreads = os.cpu_count() or 1
    out = {}
    oracle.build()  # compiled outside the timings

    def timed(fn):  # the second of two calls (the first touches fresh pages and caches)
        fn()
        t0 = time.perf_counter()
        fn()
        return (time.perf_counter() - t0) * 1e6

    def entry(us, sample):
        return {"us": us, "unit": "us per call", "cores": nthreads, "kind": "oracle", "sample": sample}

    # KV commit: L layers, one sequence, the round's tree, three committed rows
    L, n, Hkv, d, D = wl.layers, wl.nodes, wl.heads_kv, wl.head_dim, wl.depth
    S = wl.ctx + D + 8
    g = np.random.default_rng(seed)
    kt = g.integers(0, 1 << 16, (L, 1, n, Hkv, d), dtype=np.uint16)
    vt = g.integers(0, 1 << 16, (L, 1, n, Hkv, d), dtype=np.uint16)
    kc = np.zeros((L, 1, S, Hkv, d), np.uint16)
    path = np.full((1, D), -1, np.int32)
    path[0, :2] = [1, 2]
    us = timed(lambda: oracle.kv_commit(kt, vt, path, np.array([3], np.int32), np.array([wl.ctx], np.int32), kc, kc))
    out["kv_commit"] = entry(us, f"L={L} B=1 n={n} rows=3, bf16 bytes copied")
    # tree attention at the draft shape, the largest tree a draft step sees
    nd = max(x for x in (1 + wl.topk, 1 + 3 * wl.topk, 1 + 6 * wl.topk) if x <= 64)
    one = wl.with_(layers=1, batch=1, keep=nd - 1)
    inp = datagen.attention_inputs(one, seed)
    mask = np.array([[[(1 << (i + 1)) - 1] for i in range(nd)]], np.uint64)
    arrs = [datagen.to_numpy(inp[k]) for k in ("q", "k_cache", "v_cache")]
    ctx = np.array([wl.ctx], np.int32)
    kt2, vt2 = datagen.to_numpy(inp["k_tree"]), datagen.to_numpy(inp["v_tree"])
    us = timed(lambda: oracle.tree_attention(*arrs, ctx, kt2, vt2, mask, nthreads=nthreads))
    out["draft_attention"] = entry(us, f"L=1 B=1 n={nd} Hq={wl.heads_q} Hkv={wl.heads_kv} d={wl.head_dim} "
                                       f"ctx={wl.ctx}, fp64 literal softmax")
    # static chain of the workload's depth
    x = datagen.draft_logits(1, D, wl.vocab, seed).numpy()
    us = timed(lambda: oracle.build_static_tree(x, np.zeros(1, np.int32), [-1] + list(range(D))))
    out["static_tree"] = entry(us, f"chain of {D}, B=1 V={wl.vocab}")
    # sampled-children build at the workload's shape (one sequence)
    R = 1 + (D - 1) * wl.topk
    x = datagen.draft_logits(1, R, wl.vocab, seed).numpy()
    cu = datagen.child_uniforms(1, R, wl.topk, seed).numpy()
    us = timed(lambda: oracle.build_tree(x, np.zeros(1, np.int32), D, wl.topk, wl.keep, child_u=cu))
    out["sampled_build"] = entry(us, f"B=1 V={wl.vocab} D={D} k={wl.topk} m={wl.keep}, one sequence")
    return out


class OracleRound:
    """The fp64 oracle on one round of a workload, split into timeable items: the build of every
    sequence's tree, the verification of every sequence, and the L*B*Hkv attention units (one
    unit = all query heads of one KV head, every node, the sequence's full context)."""

    def __init__(self, wl, seed, nthreads):
        import oracle

        self.oracle = oracle
        self.wl, self.nthreads = wl, nthreads
        B, R, V, n = wl.batch, wl.rows, wl.vocab, wl.nodes
        draft = datagen.draft_logits(B, R, V, seed)
        self.draft_np, self.root_np = draft.numpy(), datagen.root_tokens(B, V, seed).numpy()
        self.tree = oracle.build_tree(self.draft_np, self.root_np, wl.depth, wl.topk, wl.keep, nthreads=nthreads)
        target = datagen.target_logits(draft, torch.from_numpy(self.tree["node_row"]),
                                       datagen.noise_sigmas(wl, seed), seed)
        self.tgt_np = target.numpy()
        self.u_np = datagen.uniforms(B, n, seed).numpy()
        one = wl.with_(layers=1, batch=1, heads_q=wl.group, heads_kv=1)
        inp = datagen.attention_inputs(one, seed)
        ctx = int(datagen.ctx_lens(wl, seed)[0])
        inp["ctx_len"] = torch.tensor([ctx], dtype=torch.int32)
        self.attn = [datagen.to_numpy(inp[k]) for k in ("q", "k_cache", "v_cache", "ctx_len", "k_tree", "v_tree")]
        self.mask = self.tree["mask"][:1]
        self.units = wl.layers * wl.batch * wl.heads_kv
        # mean context of the workload over the one timed unit's context
        self.ctx_scale = ((wl.ctx + wl.ctx_min) / 2 / ctx) if wl.ctx_min != wl.ctx else 1.0
        self.times = {"build": [], "verify": [], "attn": []}

    def item(self, i: int) -> None:
        """Run and time item i of the rotation build, verify, attention unit, attention unit ..."""
        kind = "build" if i % (self.units + 2) == 0 else ("verify" if i % (self.units + 2) == 1 else "attn")
        wl, o = self.wl, self.oracle
        t0 = time.perf_counter()
        if kind == "build":
            o.build_tree(self.draft_np, self.root_np, wl.depth, wl.topk, wl.keep, nthreads=self.nthreads)
        elif kind == "verify":
            o.tree_verify(self.tgt_np, self.draft_np, self.tree["tokens"], self.tree["parents"],
                          self.tree["node_row"], self.u_np, wl.temperature, wl.depth + 1, nthreads=self.nthreads)
        else:
            o.tree_attention(*self.attn, self.mask, nthreads=self.nthreads)
        self.times[kind].append(time.perf_counter() - t0)

    def round_seconds(self) -> float:
        t = {k: statistics.mean(v) for k, v in self.times.items()}
        return t["build"] + t["verify"] + t["attn"] * self.units * self.ctx_scale

    def summary(self) -> dict:
        t = {k: statistics.mean(v) for k, v in self.times.items()}
        return {"build_s": round(t["build"], 4), "verify_s": round(t["verify"], 4),
                "attn_unit_s": round(t["attn"], 5), "attn_units_per_round": self.units,
                "attn_units_timed": len(self.times["attn"]), "round_s": round(self.round_seconds(), 3)}


def _oracle_rate(wl, seed, nthreads: int, budget_s: float) -> tuple:
    """The oracle's rounds/s on `nthreads` host threads over a bounded sample of one round (its build,
    its verify and as many attention units as the budget allows, extrapolated in units)."""
    orc = OracleRound(wl, seed, nthreads)
    t0 = time.perf_counter()
    i = 0
    while i < 3 or (time.perf_counter() - t0 < budget_s and i < orc.units + 2):
        orc.item(i)
        i += 1
    return 1.0 / orc.round_seconds(), orc


def cpu_baseline(wl, seed, budget_s: float = 20.0, single_budget_s: float = 12.0) -> dict:
    nthreads = os.cpu_count() or 1
    value, orc = _oracle_rate(wl, seed, nthreads, budget_s)
    v1, orc1 = _oracle_rate(wl, seed, 1, single_budget_s)
    return {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": (f"one round's build and verify of every sequence plus {len(orc.times['attn'])} of "
                       f"{orc.units} attention units (layer x KV head; all nodes and query heads of the group; "
                       f"full context), attention extrapolated linearly in units; fp64 C oracle, OpenMP on "
                       f"{nthreads} threads"),
            "seconds": orc.summary(),
            "single_core": {"value": v1, "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": (f"the same round on one thread: build, verify and {len(orc1.times['attn'])} "
                                       f"of {orc1.units} attention units, extrapolated in units"),
                            "seconds": orc1.summary()}}


def run_reference(args, rank, world) -> dict | None:
    """Reference arm: the fp64 CPU oracle as it stands, on the host cores, same workload/metric.
    Each step is one item of the round (build, verify, or one attention unit) in rotation; the
    round time is the sum of the item means scaled by their counts per round."""
    if rank != 0:
        return None
    wl = datagen.WORKLOADS[args.workload]
    nthreads = os.cpu_count() or 1
    orc = OracleRound(wl, args.seed, nthreads)
    for i in range(args.warmup):
        orc.item(i)
    warm = {k: list(v) for k, v in orc.times.items()}
    orc.times = {k: [] for k in orc.times}
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        orc.item(i)
    wall = time.perf_counter() - t0
    for k in orc.times:  # an item kind the timed steps did not reach keeps its warm-up timing
        if not orc.times[k]:
            orc.times[k] = warm[k]
    value = 1.0 / orc.round_seconds()
    sample = (f"each step one item of a round in rotation (build of all trees, verify of all sequences, or one of "
              f"{orc.units} attention units); round time = item means x counts; fp64 C oracle, OpenMP {nthreads} "
              f"threads")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": _workload_desc(wl), "temperature": wl.temperature},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle", "sample": sample,
                             "seconds": orc.summary()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama31_8b", choices=list(datagen.WORKLOADS))
    ap.add_argument("--temperature", type=float, default=None)
    ap.add_argument("--sets", type=int, default=4)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="replay each input set's round as a CUDA graph (slower: the overlap between consecutive "
                         "rounds' launches is lost at graph boundaries)")
    ap.add_argument("--attn-launches", type=int, default=100,
                    help="launches per workload in the attention-only sweep (0: no sweep)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    res = run_ours(args, rank, world, dev)
    if rank == 0:
        wl = datagen.WORKLOADS[args.workload]
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(wl, args.seed)
            for key, val in side_cpu_baselines(wl, args.seed).items():
                if isinstance(res.get(key), dict):
                    res[key]["cpu_baseline"] = val
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
