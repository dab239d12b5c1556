"""Benchmark of the Medusa tree-verification step on one GB300 (or N replicas).

One step = tree_attn_paged + tree_accept_commit (greedy acceptance and the KV
commit in one launch; ``--accept separate`` runs tree_accept_greedy then
kv_commit instead, ``--accept typical`` tree_accept_typical then kv_commit)
over one batch of
the serving workload (batch 16, 32 q / 8 kv heads, D 128, bf16, prefixes
uniform in [512, 8192], 64-node trees, bf16 logits over a 32000 vocab), inputs
resident in HBM.  Between steps (outside the timed events) the block tables and
sequence lengths are restored and L2 is flushed by writing a 256 MiB buffer.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tree tokens/s & tree-attn KV GB/s (% of GB300 HBM roofline), 1 GPU"
UNIT = "tree tokens/s"
DEFAULT_WORKLOAD = "serve_b16_gqa_bf16"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernel", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--no-graph", action="store_true", help="launch the step's kernels one by one")
    ap.add_argument("--cache", default="act", choices=["act", "e4m3"],
                    help="KV cache elements: the act dtype, or FP8 E4M3 codes of value / scale")
    ap.add_argument("--sustain-s", type=float, default=1.0,
                    help="seconds of back-to-back replayed steps after the timed ones (0: skip)")
    ap.add_argument("--accept", default="fused", choices=["fused", "separate", "typical"],
                    help="greedy acceptance and commit in one launch, as the two calls, or "
                         "typical acceptance then the commit")
    ap.add_argument("--temperature", type=float, default=1.0, help="typical acceptance")
    ap.add_argument("--epsilon", type=float, default=0.09, help="typical acceptance")
    ap.add_argument("--delta", type=float, default=0.3, help="typical acceptance")
    return ap.parse_args()


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling, no data exchange)."""
    return seed + 1000 * rank


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The slowest rank's time (identity for one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Units processed by all ranks per second of the slowest rank."""
    return world * units_per_rank / (ms_max * 1e-3)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, keep_samples: bool = False):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        res = {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
               "reasons": sorted(reasons), "samples": len(sm)}
        if keep_samples:
            res["sm_mhz_samples"] = sm
        return res


def kernel_code_fingerprint() -> str:
    """sha256 (16 hex digits) of the tensor-core attention kernel's sources
    with comments and blank lines removed: a comment edit keeps it, any code
    change alters it."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "medusa_tree_speculative_attn_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("attn_tc.cu", "tc_ptx.cuh", "common.cuh"):
        with open(os.path.join(csrc, f)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        for line in text.splitlines():
            code = re.sub(r"//.*", "", line).rstrip()
            if code.strip():
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str, cache: str = "act"):
    """DRAM bytes per launch of the tensor-core attention kernel from the
    committed ncu summary, or None when that capture does not describe the
    kernel as it is now (different workload, cache format, kernel or code)."""
    name = f"attn_tc_e4m3_{workload}.md" if cache == "e4m3" else f"attn_tc_{workload}.md"
    path = os.path.join(ROOT, "profiles", name)
    if kernel == "simt" or not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith(("|", "#", "`")):
            k, _, v = line.partition(":")
            fields[k.strip()] = v.strip()
    if fields.get("kernel_code_sha256_16") != kernel_code_fingerprint():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measure_candidates(w: dict, K: int, flush, stream, peak: float) -> dict:
    """The step before verification (candidate tree tokens from the base logits and
    the Medusa heads' logits), timed on its own with the workload's trees and
    max_depth heads: seeded random logits in the workload's logits dtype, L2
    flushed before every call (outside the events)."""
    import torch
    import medusa_tree_speculative_attn_gb300 as mt
    dev = w["logits"].device
    B, T, V = w["B"], w["T"], w["vocab"]
    heads = w["max_depth"] if w["max_depth"] > 0 else 1
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    dt = w["logits"].dtype
    root = torch.randn((B, V), generator=gen, device=dev, dtype=torch.float32).to(dt)
    hl = torch.randn((B, heads, V), generator=gen, device=dev, dtype=torch.float32).to(dt)
    tok = torch.empty((B, T), dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    call = lambda: mt.tree_candidates(root, hl, w["tree_parents"], tok, status_ws=ws)
    # replayed as a CUDA graph, like the step, so that host overhead stays out
    # of the events
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        for _ in range(3):
            call()
    torch.cuda.current_stream().wait_stream(gs)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        call()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(K)]
    for k in range(K):
        flush.fill_((k + 7) & 0xFF)
        ev[k][0].record(stream)
        graph.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    st = mt.read_status(ws)
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    nbytes = B * (heads + 1) * V * root.element_size() + 2 * B * T * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms_per_call": ms, "alg_bytes": nbytes, "achieved_gbs": gbs, "frac_of_hbm_peak": gbs / peak,
            "heads": heads, "status": st, "l2": "flushed before each call", "launch": "CUDA graph replay"}


def algorithmic_bytes(w_host: dict, cache_bytes=None) -> dict:
    """Bytes the path must move at least once (per step); cache_bytes is the
    size of a cached element (the act dtype's unless the cache is FP8)."""
    es = {"f32": 4, "f16": 2, "bf16": 2}[w_host["dtype"]]
    cs = es if cache_bytes is None else cache_bytes
    B, T, Hq, Hkv, D = w_host["B"], w_host["T"], w_host["Hq"], w_host["Hkv"], w_host["head_dim"]
    L = np.asarray(w_host["seq_lens_host"] if "seq_lens_host" in w_host else w_host["seq_lens"], np.int64)
    prefix_kv = int(L.sum()) * Hkv * D * 2 * cs
    tree_qo = B * T * Hq * D * 2 * es              # q read, out written
    tree_kv = B * T * Hkv * D * 2 * cs             # the tree's own K/V, as cached
    attn = prefix_kv + tree_qo + tree_kv
    logits = 0
    if "vocab" in w_host:
        les = {"f32": 4, "f16": 2, "bf16": 2}[w_host["logits_dtype"]]
        logits = B * T * w_host["vocab"] * les
    return dict(prefix_kv=prefix_kv, tree_qo=tree_qo, tree_kv=tree_kv, attn=attn, logits=logits)


def run_ours(args, rank, world, local_rank):
    import torch
    import medusa_tree_speculative_attn_gb300 as mt
    import workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = workloads.generate(args.workload, seed=rank_seed(args.seed, rank), backend="torch", device=str(dev))
    spec = w["spec"]
    k_scale = v_scale = 1.0
    if args.cache == "e4m3":
        # E4M3 codes of the N(0,1) caches / an amax-style scale (the largest
        # |value| of the draws maps near 448); unused slots stay NaN codes
        k_scale = float(w["k_cache"].float().nan_to_num(0.0).abs().max()) / 448.0
        v_scale = float(w["v_cache"].float().nan_to_num(0.0).abs().max()) / 448.0
        w["k_cache"] = (w["k_cache"].float() / k_scale).to(torch.float8_e4m3fn)
        w["v_cache"] = (w["v_cache"].float() / v_scale).to(torch.float8_e4m3fn)
    B, T, md = w["B"], w["T"], w["max_depth"]
    stream = torch.cuda.current_stream()
    rope = mt.Rope(w["rope_base"], w["head_dim"], int(w["seq_lens_host"].max()) + T + 1)
    desc = mt.make_desc(w["q"], w["k_cache"], w["block_tables"], args.splits, args.kernel,
                        k_scale=k_scale, v_scale=v_scale)
    ws = mt.alloc_attn_workspace(desc, dev)
    aws = mt.alloc_accept_workspace(B, T, dev)
    out = torch.empty_like(w["q"])
    am = torch.empty((B, T), dtype=torch.int32, device=dev)
    alen = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, md + 1), dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    node_ok = torch.empty((B, T), dtype=torch.int32, device=dev)
    rel = torch.empty((B, mt.released_width(T, w["page_size"])), dtype=torch.int32, device=dev)
    typical = dict(temperature=args.temperature, epsilon=args.epsilon, delta=args.delta)
    bt0, sl0 = w["block_tables"].clone(), w["seq_lens"].clone()
    has_accept = "logits" in w
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def restore():
        w["block_tables"].copy_(bt0)
        w["seq_lens"].copy_(sl0)

    def step(src=None):
        s = src or w
        mt.tree_attn_paged(s["q"], w["k_cache"], w["v_cache"], w["block_tables"], w["seq_lens"],
                           s["tree_parents"], s["tree_depths"], out, k_new=s["k_new"], v_new=s["v_new"],
                           rope=rope, workspace=ws, num_splits=args.splits, kernel=args.kernel,
                           k_scale=k_scale, v_scale=v_scale)
        if has_accept and args.accept == "fused":
            mt.tree_accept_commit(s["tree_tokens"], s["logits"], s["tree_parents"], alen, path,
                                  w["k_cache"], w["v_cache"], w["block_tables"], w["seq_lens"], rel,
                                  argmax_out=am, next_token=nxt, workspace=aws)
        elif has_accept:
            if args.accept == "typical":
                mt.tree_accept_typical(s["tree_tokens"], s["logits"], s["tree_parents"], alen, path,
                                       node_accept=node_ok, next_token=nxt, workspace=aws, **typical)
            else:
                mt.tree_accept_greedy(s["tree_tokens"], s["logits"], s["tree_parents"], alen, path,
                                      argmax_out=am, next_token=nxt, workspace=aws)
            mt.kv_commit(path, alen, w["k_cache"], w["v_cache"], w["block_tables"], w["seq_lens"], rel,
                         tree_size=T, status_ws=ws)

    for _ in range(args.warmup):
        restore()
        step()
    torch.cuda.synchronize()
    st = mt.read_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    K = args.steps
    # (1) kernel-level: per-call events and the main attention kernel's own
    # duration (library profiling hook), kernels launched one by one
    mk = lambda: torch.cuda.Event(enable_timing=True)
    evb = [(mk(), mk(), mk(), mk(), mk(), mk()) for _ in range(K)]
    evt = [(mk(), mk()) for _ in range(K)] if has_accept and args.accept == "typical" else []
    mt.profile_enable(K)
    for k in range(K):
        restore()
        flush.fill_(k & 0xFF)
        e0, e1, e2, e3, e4, e5 = evb[k]
        e0.record(stream)
        mt.tree_attn_paged(w["q"], w["k_cache"], w["v_cache"], w["block_tables"], w["seq_lens"],
                           w["tree_parents"], w["tree_depths"], out, k_new=w["k_new"], v_new=w["v_new"],
                           rope=rope, workspace=ws, num_splits=args.splits, kernel=args.kernel,
                           k_scale=k_scale, v_scale=v_scale)
        e1.record(stream)
        if has_accept:
            mt.tree_accept_greedy(w["tree_tokens"], w["logits"], w["tree_parents"], alen, path,
                                  argmax_out=am, next_token=nxt, workspace=aws)
            e2.record(stream)
            mt.kv_commit(path, alen, w["k_cache"], w["v_cache"], w["block_tables"], w["seq_lens"], rel,
                         tree_size=T, status_ws=ws)
            e3.record(stream)
            restore()
            flush.fill_(k & 0xFF)
            e4.record(stream)
            mt.tree_accept_commit(w["tree_tokens"], w["logits"], w["tree_parents"], alen, path,
                                  w["k_cache"], w["v_cache"], w["block_tables"], w["seq_lens"], rel,
                                  argmax_out=am, next_token=nxt, workspace=aws)
            e5.record(stream)
            if evt:
                flush.fill_(k & 0xFF)
                evt[k][0].record(stream)
                mt.tree_accept_typical(w["tree_tokens"], w["logits"], w["tree_parents"], alen, path,
                                       node_accept=node_ok, next_token=nxt, workspace=aws, **typical)
                evt[k][1].record(stream)
        else:
            for e in (e2, e3, e4, e5):
                e.record(stream)
    torch.cuda.synchronize()
    main_ms = mt.profile_read(K)
    mt.profile_enable(0)
    avg = lambda i, j: float(np.mean([e[i].elapsed_time(e[j]) for e in evb]))
    breakdown = {"tree_attn_paged_ms": avg(0, 1),
                 "attention_main_kernel_ms": float(np.mean(main_ms)) if main_ms else None,
                 "tree_accept_greedy_ms": avg(1, 2), "kv_commit_ms": avg(2, 3),
                 "tree_accept_commit_ms": avg(4, 5),
                 "note": "each call timed alone, L2 flushed before the attention and before the "
                         "fused call" + (" and the typical call" if evt else "") + "; the step uses " + {
                             "fused": "tree_accept_commit", "separate": "tree_accept_greedy + kv_commit",
                             "typical": "tree_accept_typical + kv_commit"}[args.accept]}
    if evt:
        breakdown["tree_accept_typical_ms"] = float(np.mean([a.elapsed_time(b) for a, b in evt]))
        breakdown["typical"] = typical

    # The per-call times above bracket eager calls, so for small workloads they
    # include the GPU idling while the host runs the binding's checks.  Each
    # call is also replayed alone as a CUDA graph (L2 flushed and tables
    # restored before each replay, outside the events); with graphs on, these
    # are the breakdown's times.
    if not args.no_graph:
        def attn_call():
            mt.tree_attn_paged(w["q"], w["k_cache"], w["v_cache"], w["block_tables"], w["seq_lens"],
                               w["tree_parents"], w["tree_depths"], out, k_new=w["k_new"], v_new=w["v_new"],
                               rope=rope, workspace=ws, num_splits=args.splits, kernel=args.kernel,
                               k_scale=k_scale, v_scale=v_scale)

        calls = {"tree_attn_paged_ms": attn_call}
        if has_accept:
            calls["tree_accept_greedy_ms"] = lambda: mt.tree_accept_greedy(
                w["tree_tokens"], w["logits"], w["tree_parents"], alen, path, argmax_out=am, next_token=nxt,
                workspace=aws)
            calls["kv_commit_ms"] = lambda: mt.kv_commit(path, alen, w["k_cache"], w["v_cache"],
                                                         w["block_tables"], w["seq_lens"], rel, tree_size=T,
                                                         status_ws=ws)
            calls["tree_accept_commit_ms"] = lambda: mt.tree_accept_commit(
                w["tree_tokens"], w["logits"], w["tree_parents"], alen, path, w["k_cache"], w["v_cache"],
                w["block_tables"], w["seq_lens"], rel, argmax_out=am, next_token=nxt, workspace=aws)
            if evt:
                calls["tree_accept_typical_ms"] = lambda: mt.tree_accept_typical(
                    w["tree_tokens"], w["logits"], w["tree_parents"], alen, path, node_accept=node_ok,
                    next_token=nxt, workspace=aws, **typical)
        cs_g = torch.cuda.Stream(device=dev)
        for key, fn in calls.items():
            restore()
            cs_g.wait_stream(stream)
            with torch.cuda.stream(cs_g):
                fn()                         # warm the capture stream
                cs_g.synchronize()
                restore()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cs_g):
                    fn()
            stream.wait_stream(cs_g)
            torch.cuda.synchronize()
            pairs = []
            for k in range(K):
                restore()
                flush.fill_(k & 0xFF)
                e_a, e_b = mk(), mk()
                e_a.record(stream)
                g.replay()
                e_b.record(stream)
                pairs.append((e_a, e_b))
            torch.cuda.synchronize()
            breakdown[key] = float(np.mean([x.elapsed_time(y) for x, y in pairs]))
            del g
        breakdown["note"] = ("each call replayed alone as a CUDA graph, L2 flushed and tables restored before "
                             "each replay (outside the events); the step uses " + {
                                 "fused": "tree_accept_commit", "separate": "tree_accept_greedy + kv_commit",
                                 "typical": "tree_accept_typical + kv_commit"}[args.accept])
    restore()

    # (2) the timed steps: the whole step replayed as one CUDA graph (or
    # launched kernel by kernel with --no-graph)
    graph = None
    if not args.no_graph:
        restore()
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            step()                       # warm the capture stream
            gs.synchronize()
            restore()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                step()
        stream.wait_stream(gs)
        torch.cuda.synchronize()
    run_step = graph.replay if graph is not None else step
    for _ in range(2):
        restore()
        run_step()
    torch.cuda.synchronize()
    ev = [(mk(), mk()) for _ in range(K)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    accepted = 0
    for k in range(K):
        restore()
        flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        run_step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if has_accept:
        accepted = int(alen.sum().item()) + B
    st = mt.read_status(ws)
    if st != 0 or (has_accept and mt.read_status(aws) != 0):
        raise RuntimeError(f"device status {st} after timed steps")
    ms = float(np.mean(step_ms))
    t_max = max_over_ranks(ms, world, dev)

    # (3) a sustained pass: the same replayed step back to back for at least
    # args.sustain_s seconds (restore and L2 flush between steps, outside the
    # events), with the clock samples of that stretch binned by SM clock
    sustained = None
    if args.sustain_s > 0:
        # steps for the requested seconds at the timed loop's wall rate (step,
        # restore and flush included)
        n_s = max(K, int(args.sustain_s / max(wall / K, 1e-6)) + 1)
        evs = [(mk(), mk()) for _ in range(n_s)]
        sampler_s = ClockSampler(local_rank)
        sampler_s.start()
        time.sleep(0.3)
        torch.cuda.synchronize()
        t_s = time.perf_counter()
        for k in range(n_s):
            restore()
            flush.fill_(k & 0xFF)
            evs[k][0].record(stream)
            run_step()
            evs[k][1].record(stream)
        torch.cuda.synchronize()
        wall_s = time.perf_counter() - t_s
        clk = sampler_s.stop(keep_samples=True)
        st_ms = np.array([a.elapsed_time(b) for a, b in evs])
        bins = {}
        for mhz in clk.pop("sm_mhz_samples", []):
            key = f"{int(mhz // 100) * 100}-{int(mhz // 100) * 100 + 99}"
            bins[key] = bins.get(key, 0) + 1
        sustained = {"steps": n_s, "wall_s": wall_s, "ms_per_step": float(np.mean(st_ms)),
                     "ms_per_step_median": float(np.median(st_ms)), "ms_per_step_p90": float(np.percentile(st_ms, 90)),
                     "clocks": clk, "sm_mhz_bins": bins}

    # end to end through the public API with host buffers: pinned H2D of the
    # step's inputs, the step's calls, D2H of the step's results
    e2e = e2e_overlapped = None
    if not args.no_e2e:
        keys_in = ["q", "k_new", "v_new", "tree_parents", "tree_depths"]
        if has_accept:
            keys_in += ["tree_tokens", "logits"]
        host = {k: w[k].cpu().pin_memory() for k in keys_in}
        dsrc = {k: torch.empty_like(w[k]) for k in keys_in}
        per_node = node_ok if args.accept == "typical" else am
        outs = [out, per_node, alen, path, nxt, rel] if has_accept else [out]
        houts = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        h2d = sum(host[k].numel() * host[k].element_size() for k in keys_in)
        d2h = sum(o.numel() * o.element_size() for o in outs)
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for k in range(K + 2):
            restore()
            flush.fill_(k & 0xFF)
            if k >= 2:
                eev[k - 2][0].record(stream)
            for key in keys_in:
                dsrc[key].copy_(host[key], non_blocking=True)
            step(dsrc)
            for o, ho in zip(outs, houts):
                ho.copy_(o, non_blocking=True)
            if k >= 2:
                eev[k - 2][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in eev])), world, dev)
        e2e = {"value": whole_job_rate(B * T, world, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

        # the same end-to-end steps, overlapped as a serving loop would run
        # them: step k + 1's inputs go host -> device (into the other of two
        # device input sets) while step k runs, and step k's results are read
        # back right after it.  Each iteration is one CUDA graph (a fork for
        # the next step's input copies, the step and its read-back, a join),
        # two graphs alternating over the input sets, so that the host issue
        # rate does not bound small steps.  Every step still copies its own
        # inputs in and its results out inside the timed region.  No L2 flush.
        cs = torch.cuda.Stream(device=dev)
        dsets = [dsrc, {k: torch.empty_like(w[k]) for k in keys_in}]
        n_ov = max(K, 20)

        def copy_into(d):
            for key in keys_in:
                d[key].copy_(host[key], non_blocking=True)

        def iteration(cur):
            cs.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(cs):
                copy_into(dsets[1 - cur])     # the next step's inputs
            restore()
            step(dsets[cur])
            for o, ho in zip(outs, houts):
                ho.copy_(o, non_blocking=True)
            torch.cuda.current_stream().wait_stream(cs)

        ov_graphs = []
        if not args.no_graph:
            gs2 = torch.cuda.Stream(device=dev)
            gs2.wait_stream(stream)
            with torch.cuda.stream(gs2):
                iteration(0)                  # warm the capture stream
                gs2.synchronize()
                for cur in (0, 1):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=gs2):
                        iteration(cur)
                    ov_graphs.append(g)
            stream.wait_stream(gs2)
            torch.cuda.synchronize()

        def overlapped(n, t0=None, t1=None):
            if t0 is not None:
                t0.record(stream)
            copy_into(dsets[0])               # the first step's inputs
            for i in range(n):
                if ov_graphs:
                    ov_graphs[i % 2].replay()
                else:
                    iteration(i % 2)
            if t1 is not None:
                t1.record(stream)

        overlapped(3)  # warm-up
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        overlapped(n_ov, t0, t1)
        torch.cuda.synchronize()
        ov_ms = max_over_ranks(t0.elapsed_time(t1) / n_ov, world, dev)
        e2e_overlapped = {"value": whole_job_rate(B * T, world, ov_ms), "unit": UNIT, "ms_per_step": ov_ms,
                          "steps": n_ov, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                          "launch": "one CUDA graph per iteration" if ov_graphs else "eager",
                          "note": "step k+1's inputs copied on a second stream while step k runs; "
                                  "results read back after each step; no L2 flush"}

    ab = algorithmic_bytes(w, 1 if args.cache == "e4m3" else None)
    peak, peak_src = measured_peaks()
    cand = measure_candidates(w, K, flush, stream, peak) if has_accept else None
    main_avg = float(np.mean(main_ms)) if main_ms else None
    roofline = None
    if main_avg:
        achieved = ab["attn"] / (main_avg * 1e-3) / 1e9
        roofline = {"kernel": "tree attention main kernel", "bound": "hbm", "achieved": achieved,
                    "peak": peak, "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": ncu_traffic(args.workload, args.kernel, args.cache), "ms_per_launch": main_avg,
                    "alg_bytes_per_launch": ab["attn"]}
    # the whole tree_attn_paged call (prep, main kernel, combine) against the
    # same bytes
    call_ms = breakdown["tree_attn_paged_ms"]
    roofline_call = {"call": "tree_attn_paged (prep + main kernel + combine)", "bound": "hbm",
                     "achieved": ab["attn"] / (call_ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": ab["attn"] / (call_ms * 1e-3) / 1e9 / peak, "ms_per_call": call_ms,
                     "call_over_main": call_ms / main_avg if main_avg else None}
    res = {
        "metric": METRIC, "value": whole_job_rate(B * T, world, t_max), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": t_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "batch": B, "tree_nodes": T, "q_heads": w["Hq"],
                   "kv_heads": w["Hkv"], "head_dim": w["head_dim"], "page_size": w["page_size"],
                   "prefix": list(spec.prefix), "logits": (f"{w['logits_dtype']} vocab {w['vocab']}"
                                                           if has_accept else None),
                   "kernel": args.kernel, "num_splits": args.splits, "accept": args.accept,
                   "kv_cache": "act dtype" if args.cache == "act" else
                   f"fp8 e4m3 codes (k_scale {k_scale:.5g}, v_scale {v_scale:.5g})",
                   "launch": "one CUDA graph per step" if graph is not None else "kernel by kernel",
                   "l2": "flushed between steps (256 MiB write)", "parallelism": f"replicas x{world}"},
        "kv_gbs": ab["prefix_kv"] / (main_avg * 1e-3) / 1e9 if main_avg else None,
        "accepted_tokens_per_s": whole_job_rate(accepted, world, t_max) if has_accept else None,
        "alg_bytes": ab, "roofline": roofline, "roofline_call": roofline_call, "breakdown": breakdown,
        "e2e": e2e, "e2e_overlapped": e2e_overlapped, "clocks": clocks, "sustained": sustained,
        "tree_candidates": cand,
        "gpu_launches": K * (3 + (0 if not has_accept else 1 if args.accept == "fused" else 2)),
        "wall_s_timed_region": wall,
    }
    if rank == 0 and not args.no_cpu_baseline and args.cache == "act":
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_budget_s)
    if world > 1:
        torch.distributed.destroy_process_group()
    return res


def oracle_sample_step(w_np: dict, seqs):
    """The oracle on the given sequences: attention of every (node, head) and
    greedy acceptance.  The KV commit is left out: it moves a few KB per
    sequence, next to the attention's float64 work.  Returns tree tokens
    processed."""
    import oracle
    sub = {k: w_np[k] for k in w_np}
    q_rot, k_rot = oracle.rotate_inputs(w_np)
    sel = np.array([(b, h, i) for b in seqs for i in range(w_np["T"]) for h in range(w_np["Hq"])],
                   np.int32)
    oracle.tree_attn(w_np, sel=sel, q_rot=q_rot, k_rot=k_rot)
    if "logits" in w_np:
        idx = np.asarray(seqs)
        am, alen, path, nxt = oracle.accept_greedy(w_np["tree_tokens"][idx], w_np["logits"][idx],
                                                   w_np["logits_dtype"], w_np["tree_parents"][idx],
                                                   w_np["max_depth"])
    del sub
    return len(seqs) * w_np["T"]


def cpu_baseline(w, budget_s: float):
    import oracle
    import workloads
    w_np = workloads.to_numpy(w)
    t0 = time.perf_counter()
    n = oracle_sample_step(w_np, [0])
    t1 = time.perf_counter() - t0
    seqs = list(range(1, min(w_np["B"], 1 + max(0, int(budget_s / max(t1, 1e-3)) - 1))))
    t0 = time.perf_counter()
    if seqs:
        n = oracle_sample_step(w_np, seqs)
        dt = time.perf_counter() - t0
    else:
        dt = t1
        seqs = [0]
    return {"value": n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(seqs)} of {w_np['B']} sequences of {w_np['name']}: attention of every "
                      f"(node, q head) in float64 plus greedy acceptance (no commit), {dt:.1f} s"}


def run_reference(args, rank, world):
    import oracle
    import workloads
    if rank != 0:
        return None
    w_np = workloads.generate(args.workload, seed=args.seed)
    spec = w_np["spec"]
    # one step = one sequence of the workload (a bounded sample)
    times = []
    for k in range(args.warmup + args.steps):
        b = k % w_np["B"]
        t0 = time.perf_counter()
        n = oracle_sample_step(w_np, [b])
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append(dt)
    ms = 1e3 * float(np.mean(times))
    value = w_np["T"] / (ms * 1e-3)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "batch": w_np["B"], "tree_nodes": w_np["T"],
                   "q_heads": w_np["Hq"], "kv_heads": w_np["Hkv"], "head_dim": w_np["head_dim"],
                   "step_sample": "one sequence per step (CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": "one sequence of the workload per step: attention of every "
                                   "(node, q head) in float64 plus greedy acceptance (no commit)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
