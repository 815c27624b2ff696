"""Benchmark of one paged-decode step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one pass of the whole decode path over one batch of synthetic input
(for the paged workloads: one pd_decode_attn call, i.e. the unit pass plus the
merge when the launch splits; for the tiled workload: begin, every step_tile
call and finalize; for the mixed tiled workload: one pd_tiled_run, i.e. begin,
the step_tile calls over the paged cache and then the scratch pool, finalize).
The default workload is the large-batch one: 256 sequences with lognormal
lengths (median 2048, clipped to [16, 16384]), 32 query heads over 8 KV heads,
head dim 128, block 16, Auto split count at 148 SMs (10 splits) plus the merge.

Metric: KV bytes read per second (live tokens x num_kv_heads x head_dim x 2
bytes x K and V), whole job; also microseconds per step and the fraction of the
measured HBM copy peak.  Rank 0 prints one JSON line.

Under torchrun with N > 1 every rank runs an independent replica of the same
step on its own GPU (the path has no exchange step); the timing is the max
over ranks and the value is the sum of the ranks' bytes over that time.

`--impl reference` times the FP64 CPU oracle on the same workload on this
machine's host cores (rank 0 only), each step a bounded sample of sequences.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
METRIC = "paged-decode KV-read GB/s (% of GB300 HBM peak) and us per decode step"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _workload(name):
    from paged_kv_decode_splitk_gb300 import workloads as W
    return W.WORKLOADS[name]()


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in (self.out or "").splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device) -> float:
    """The largest of the ranks' values (every rank gets it); the identity when
    the job runs alone."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(kv_bytes_per_rank: int, steps: int, total_ms: float, world_size: int) -> float:
    """Whole-job KV GB/s: every rank's bytes over the slowest rank's time (the
    ranks run independent replicas of the same step)."""
    return world_size * kv_bytes_per_rank * steps / (total_ms / 1e3) / 1e9


def source_digest() -> str:
    """Hash of the kernel sources (paged_kv_decode_splitk_gb300/csrc) with their
    comments and blank space removed: it changes when the code does."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_splitk_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"\s+", " ", text)
        h.update(f.encode() + b"\0" + text.encode())
    return h.hexdigest()[:16]


def _traffic_from_profiles(kernel_tag: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    kernel code as it is now (the summary records source_digest())."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}__{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    tag = None
    traffic = None
    for ln in text.splitlines():
        if ln.startswith("source_sha256:"):
            tag = ln.split(":", 1)[1].strip()
        if ln.startswith("dram_bytes_per_launch:"):
            traffic = float(ln.split(":", 1)[1].strip())
    if tag != source_digest():
        return None
    return traffic


def step_config(w, num_splits: int, world_size: int) -> dict:
    """The workload a step runs, as both arms report it (same keys, same values)."""
    tiled = not hasattr(w, "context_lens")
    return {
        "workload": w.name,
        "num_seqs": w.num_seqs,
        "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim,
        "block_size": w.block_size,
        "num_splits": int(num_splits),
        "gqa_pack": int(w.__dict__.get("gqa_pack", 0)),
        "kv_dtype": w.__dict__.get("kv_dtype", "bf16"),
        "kv_bytes_per_step": int(w.kv_bytes),
        "tokens": int(w.kv_tokens) if tiled else int(w.context_lens.sum()),
        "parallelism": f"replicas x{world_size}" if world_size > 1 else "single GPU",
    }


def _workload_splits(w) -> int:
    """The step's split count from the oracle's own copy of the policy rules
    (the reference arm does not load the CUDA library)."""
    if not hasattr(w, "context_lens"):
        return 1
    from oracle import policy as P
    return P.num_splits(w.policy, w.pin, w.sm_count, w.num_q_heads, w.num_seqs, w.max_decode_seqs)


def end_to_end(stream, steps, kv_bytes, world_size, small, kv, launch, out, kv_note):
    """The step through the public call with host buffers: every step copies the
    `small` inputs (q, tables) from pinned host memory, runs `launch(small_dev,
    kv_dev)` and reads the output back; the first form also uploads the K/V
    pools (`kv`) every step, the second keeps them resident in HBM."""
    import torch

    def pinned(t):
        return t.detach().cpu().pin_memory()
    h_small = [pinned(t) for t in small]
    d_small = [torch.empty_like(t) for t in small]
    h_kv = [pinned(t) for t in kv]
    d_kv = [torch.empty_like(t) for t in kv]
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step(upload_kv):
        for h, d in zip(h_small, d_small):
            d.copy_(h, non_blocking=True)
        if upload_kv:
            for h, d in zip(h_kv, d_kv):
                d.copy_(h, non_blocking=True)
        launch(d_small, d_kv if upload_kv else kv)
        hout.copy_(out, non_blocking=True)

    def timed(upload_kv, k):
        for _ in range(3):
            e2e_step(upload_kv)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k):
            e2e_step(upload_kv)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / k

    small_in = sum(t.numel() * t.element_size() for t in h_small)
    kv_in = sum(t.numel() * t.element_size() for t in h_kv)
    out_b = hout.numel() * hout.element_size()
    ms_kv = timed(True, max(3, min(steps, 20)))
    ms_res = timed(False, max(3, min(steps, 2000)))
    e2e = {"value": round(world_size * kv_bytes / (ms_kv / 1e3) / 1e9, 2), "unit": "GB/s",
           "ms_per_step": round(ms_kv, 5), "h2d_bytes_per_step": int(small_in + kv_in),
           "d2h_bytes_per_step": int(out_b),
           "note": f"host buffers: q, the tables and {kv_note} copied from pinned host memory every "
                   f"step, output read back"}
    resident = {"value": round(world_size * kv_bytes / (ms_res / 1e3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(ms_res, 5), "h2d_bytes_per_step": int(small_in),
                "d2h_bytes_per_step": int(out_b),
                "note": "KV resident in HBM (decode-serving form): only q, the tables and the output "
                        "cross the host link"}
    return e2e, resident


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from paged_kv_decode_splitk_gb300 import api, pd

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)

    w = _workload(args.workload)
    if args.seqs:
        from paged_kv_decode_splitk_gb300 import workloads as W
        if not hasattr(w, "context_lens"):
            raise SystemExit("--seqs applies to the paged workloads only")
        w = W.first_seqs(w, args.seqs)
    mixed = args.workload == "tiled_mixed"
    tiled = args.workload == "tiled" or mixed
    kv_bytes = w.kv_bytes
    stream = torch.cuda.current_stream()

    if not tiled:
        base = api.PagedInputs(w, dev)
        n = base.splits()
        pool_bytes = base.k.numel() * base.k.element_size() * 2
        copies = max(2, -(-3 * L2_BYTES // pool_bytes))
        ks = [base.k] + [base.k.clone() for _ in range(copies - 1)]
        vs = [base.v] + [base.v.clone() for _ in range(copies - 1)]
        out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
        wsp = api.workspace(w.num_seqs, w.num_q_heads, w.head_dim, n, dev)
        launches_per_step = 1 + (1 if n > 1 else 0)

        def step(i):
            api.decode_attn(base.q, ks[i % copies], vs[i % copies], base.block_table, base.context_lens,
                            w.inv_sqrt_d, n, w.gqa_pack, out, wsp, None, w.k_scale, w.v_scale)
        l2_note = f"rotating {copies} KV-cache copies ({copies * pool_bytes / 1e6:.0f} MB > 129 MB L2)"
    elif mixed:
        # one pd_tiled_run per step: begin, the paged-cache calls, the scratch-pool
        # calls, finalize
        base = api.MixedTiledInputs(w, dev)
        n = 1
        pool_bytes = (base.paged_k.numel() + base.paged_v.numel() + base.scratch.numel()) * 2
        copies = max(2, -(-3 * L2_BYTES // pool_bytes))
        t = pd.Tiled(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.tile_capacity)
        stripe = w.num_kv_heads * w.block_size * w.head_dim
        srcs = []
        for i in range(copies):
            pk = base.paged_k if i == 0 else base.paged_k.clone()
            pv = base.paged_v if i == 0 else base.paged_v.clone()
            sc = (base.scratch if i == 0 else base.scratch.clone()).view(-1)
            lst = []
            for ci, (kind, _, _, lb) in enumerate(w.calls):
                if kind == "paged":
                    lst.append((pk, pv, base.tile_blocks[ci], base.tile_counts[ci], t.paged_strides(), lb))
                else:
                    lst.append((sc, sc[stripe:], base.tile_blocks[ci], base.tile_counts[ci],
                                t.scratch_pool_strides(), lb))
            srcs.append(lst)
        out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
        launches_per_step = 2 if len(w.calls) <= 8 else 2 + len(w.calls)

        def step(i):
            t.run(base.q, srcs[i % copies], out, w.num_seqs)
        l2_note = (f"rotating {copies} copies of the paged cache and scratch pool "
                   f"({copies * pool_bytes / 1e6:.0f} MB > 129 MB L2)")
    else:
        base = api.TiledInputs(w, dev)
        n = 1
        pool_bytes = base.pool.numel() * 2
        copies = max(2, -(-3 * L2_BYTES // pool_bytes))
        pools = [base.pool] + [base.pool.clone() for _ in range(copies - 1)]
        stripe = w.num_kv_heads * w.block_size * w.head_dim
        t = pd.Tiled(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.tile_capacity)
        strides = t.scratch_pool_strides()
        out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
        launches_per_step = 2 + w.num_calls

        # the step through the library's driver, pd_tiled_run (begin, the calls,
        # finalize in one call; same bits as the calls made one by one), or,
        # with --tiled-separate, through begin / step_tile x T / finalize
        srcs = []
        for i in range(copies):
            p = pools[i].view(-1)
            srcs.append([(p, p[stripe:], base.tile_blocks[c], base.tile_counts[c], strides,
                          int(w.last_block_valid_slots[c])) for c in range(w.num_calls)])
        if args.tiled_separate:
            def step(i):
                t.begin(w.num_seqs)
                for src in srcs[i % copies]:
                    t.step(base.q, src[0], src[1], src[2], src[3], w.num_seqs, src[4], src[5])
                t.finalize(out, w.num_seqs)
        else:
            launches_per_step = 2

            def step(i):
                t.run(base.q, srcs[i % copies], out, w.num_seqs)
        l2_note = f"rotating {copies} scratch-pool copies ({copies * pool_bytes / 1e6:.0f} MB > 129 MB L2)"

    warmup = max(3, args.warmup)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if pd.pd_device_status() != 0:
        raise RuntimeError("device status flags set during warm-up")

    # CUDA graphs of whole steps: one graph of `copies` consecutive steps (one
    # per input copy, so consecutive steps read different memory) replayed back
    # to back, plus single-step graphs for a remainder, so that exactly K steps
    # run and the device, not the Python launch path, sets the pace.  Launches
    # inside a graph keep their programmatic (PDL) edges.
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        for i in range(copies):
            step(i)
    torch.cuda.synchronize()
    g_multi = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_multi, stream=cap):
        for i in range(copies):
            step(i)
    g_single = []
    for i in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            step(i)
        g_single.append(g)
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    for _ in range(3):
        g_multi.replay()
    e_b.record(stream)
    torch.cuda.synchronize()
    ms_multi = max(e_a.elapsed_time(e_b) / 3, 1e-3)
    n_multi, n_rem = divmod(args.steps, copies)

    # ---- timed region: K steps back to back, events on the launching stream ----
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_multi + n_rem + 1)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # Untimed replays of the same graphs keep the GPU under this load for about
    # a second before the timed region (which can be a few milliseconds long),
    # so that the clock samples taken meanwhile describe the clocks it ran at.
    soak_reps = max(1, int(1000.0 / ms_multi))
    soak_s = soak_reps * ms_multi / 1e3
    with ClockSampler(local) as clk:
        for _ in range(soak_reps):
            g_multi.replay()
        evs[0].record(stream)
        for j in range(n_multi):
            g_multi.replay()
            evs[j + 1].record(stream)
        for j in range(n_rem):
            g_single[j].replay()
            evs[n_multi + j + 1].record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    total_ms = max_over_ranks(evs[0].elapsed_time(evs[-1]), dev)
    ms_per_step = total_ms / args.steps
    value = job_value(kv_bytes, args.steps, total_ms, ws)
    del g_multi, g_single

    # dominant kernel: the unit pass (the only launch of a packed / non-split step;
    # with a merge the step time bounds the unit pass from above)
    unit_ms = ms_per_step
    peak, peak_kind = _peaks()
    achieved = kv_bytes / (unit_ms / 1e3) / 1e9
    kernel_tag = "unit_packed" if w.__dict__.get("gqa_pack") else ("unit_tiled" if tiled else "unit_splitk")
    if tiled and not mixed and args.tiled_separate:
        kernel_tag = "unit_tiledstep"  # one launch per step_tile call: not the fused run's kernel
    traffic = _traffic_from_profiles(kernel_tag, args.workload)

    # ---- end to end: host buffers through the public API ----
    if not tiled:
        def launch_e2e(sm, kv):
            api.decode_attn(sm[0], kv[0], kv[1], sm[1], sm[2], w.inv_sqrt_d, n, w.gqa_pack, out, wsp, None,
                            w.k_scale, w.v_scale)
        e2e, e2e_resident = end_to_end(stream, args.steps, kv_bytes, ws,
                                       [base.q, base.block_table, base.context_lens], [base.k, base.v],
                                       launch_e2e, out, "the whole K/V cache")
    elif mixed:
        T = len(w.calls)

        def launch_e2e(sm, kv):
            pk, pv, sc = kv[0], kv[1], kv[2].view(-1)
            lst = []
            for ci, (kind, _, _, lb) in enumerate(w.calls):
                if kind == "paged":
                    lst.append((pk, pv, sm[1 + ci], sm[1 + T + ci], t.paged_strides(), lb))
                else:
                    lst.append((sc, sc[stripe:], sm[1 + ci], sm[1 + T + ci], t.scratch_pool_strides(), lb))
            t.run(sm[0], lst, out, w.num_seqs)
        e2e, e2e_resident = end_to_end(stream, args.steps, kv_bytes, ws,
                                       [base.q] + list(base.tile_blocks) + list(base.tile_counts),
                                       [base.paged_k, base.paged_v, base.scratch], launch_e2e, out,
                                       "the paged cache and the scratch pool")
    else:
        T = w.num_calls

        def launch_e2e(sm, kv):
            p = kv[0].view(-1)
            t.run(sm[0], [(p, p[stripe:], sm[1 + c], sm[1 + T + c], strides, int(w.last_block_valid_slots[c]))
                          for c in range(T)], out, w.num_seqs)
        e2e, e2e_resident = end_to_end(stream, args.steps, kv_bytes, ws,
                                       [base.q] + list(base.tile_blocks) + list(base.tile_counts), [base.pool],
                                       launch_e2e, out, "the whole scratch pool")
    if pd.pd_device_status() != 0:
        raise RuntimeError("device status flags set during the timed region")

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.workload, budget_s=args.cpu_seconds)
        cpu_all = cpu_baseline_all_cores(w, args.workload, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": warmup,
            "ms_per_step": round(ms_per_step, 6),
            "us_per_step": round(ms_per_step * 1e3, 3),
            "hbm_frac": round(value / ws / peak, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            # the products' operand type: BF16, or f16 for an FP8 cache (converted exactly)
            "dtype": "f16" if w.__dict__.get("kv_dtype") == "e4m3" else "bf16",
            "data": "synthetic (seeded N(0,1) BF16 q/K/V, seeded lengths and block tables)",
            "config": step_config(w, n, ws),
            "method": {
                "l2": l2_note,
                "timing": f"CUDA events around back-to-back replays of a {copies}-step CUDA graph",
                "clocks": f"nvidia-smi every 100 ms over {soak_s:.2f} s of untimed replays of the same "
                          f"graphs right before the timed region, and over the timed region",
            },
            "roofline": {
                "bound": "hbm",
                "kernel": kernel_tag,
                "achieved": round(achieved, 2),
                "peak": peak,
                "peak_kind": peak_kind,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": traffic,
                "per_launch_us": round(unit_ms * 1e3, 3),
            },
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "e2e": e2e,
            "e2e_resident_kv": e2e_resident,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
        }
        print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()


def _oracle_step(w, seqs):
    import oracle
    if getattr(w, "kv_dtype", "bf16") == "e4m3":
        return oracle.decode_attn_fp8(w.q[seqs], w.k_cache, w.v_cache, w.k_scale, w.v_scale,
                                      w.block_table[seqs], w.context_lens[seqs], w.inv_sqrt_d)
    if hasattr(w, "context_lens"):
        return oracle.decode_attn(w.q[seqs], w.k_cache, w.v_cache, w.block_table[seqs],
                                  w.context_lens[seqs], w.inv_sqrt_d)
    from paged_kv_decode_splitk_gb300 import workloads as W
    if hasattr(w, "calls"):
        kf, vf = W.scratch_pool_views(w.scratch)
        Hkv, D, bs = w.num_kv_heads, w.head_dim, w.block_size
        calls = []
        for kind, tb, tc, lb in w.calls:
            paged = kind == "paged"
            calls.append(dict(k_pool=w.paged_k if paged else kf, v_pool=w.paged_v if paged else vf,
                              tile_blocks=tb[seqs], tile_block_counts=tc[seqs], last_block_valid_slots=lb,
                              strides=(oracle.paged_strides if paged else oracle.scratch_pool_strides)(
                                  Hkv, D, bs)))
        return oracle.tiled_attn_multi(w.q[seqs], calls, Hkv, bs)
    kf, vf = W.scratch_pool_views(w.pool)
    return oracle.tiled_attn(w.q[seqs], kf, vf, w.tile_blocks[:, seqs], w.tile_block_counts[:, seqs],
                             w.last_block_valid_slots, w.num_kv_heads, w.block_size,
                             oracle.scratch_pool_strides(w.num_kv_heads, w.head_dim, w.block_size))


def _seq_bytes(w, seqs):
    if hasattr(w, "context_lens"):
        return (int(w.context_lens[seqs].astype("int64").sum()) * w.num_kv_heads * w.head_dim * 2
                * w.kv_elem_bytes)
    bs = w.block_size
    tok = 0
    if hasattr(w, "calls"):
        for _, _, tc, lb in w.calls:
            for s in seqs:
                cnt = int(tc[s])
                if cnt:
                    tok += (cnt - 1) * bs + (lb if 1 <= lb < bs else bs)
        return tok * w.num_kv_heads * w.head_dim * 4
    for c in range(w.num_calls):
        lb = int(w.last_block_valid_slots[c])
        for s in seqs:
            cnt = int(w.tile_block_counts[c, s])
            if cnt:
                tok += (cnt - 1) * bs + (lb if 1 <= lb < bs else bs)
    return tok * w.num_kv_heads * w.head_dim * 4


def _sample_seqs(w, budget_s):
    """Sequences (in a fixed seeded order) whose oracle time fits the budget, estimated
    from a first timed sequence."""
    import numpy as np
    order = np.random.default_rng(123).permutation(w.num_seqs)
    t0 = time.perf_counter()
    _oracle_step(w, order[:1])
    dt = max(time.perf_counter() - t0, 1e-4)
    rate = _seq_bytes(w, order[:1]) / dt
    target = rate * budget_s
    acc, chosen = 0, []
    for s in order:
        b = _seq_bytes(w, [s])
        if chosen and acc + b > target:
            break
        chosen.append(int(s))
        acc += b
    return sorted(chosen)


def cpu_baseline(w, workload, budget_s=10.0):
    seqs = _sample_seqs(w, budget_s)
    # whole passes over the sample until the budget is spent (a workload that
    # the oracle finishes quickly is timed over several passes)
    passes = 0
    t0 = time.perf_counter()
    while True:
        _oracle_step(w, seqs)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= 0.9 * budget_s:
            break
    b = _seq_bytes(w, seqs)
    return {"value": round(b * passes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(seqs)} of {w.num_seqs} sequences of {workload} ({b / 1e6:.1f} MB of K/V) "
                      f"x {passes} pass(es), FP64 C oracle, single thread, {dt:.1f} s"}


def cpu_baseline_all_cores(w, workload, budget_s=10.0):
    """The same oracle on every host core: the sample's sequences dealt round-robin
    to one thread per core (the C oracle runs outside the GIL and keeps no state),
    whole passes until the budget is spent.  A workload with fewer sequences than
    cores uses as many threads as it has sequences."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle._load()  # build / load once, before the threads
    ncpu = os.cpu_count() or 1
    seqs = _sample_seqs(w, budget_s * ncpu)
    nthr = max(1, min(ncpu, len(seqs)))
    chunks = [seqs[i::nthr] for i in range(nthr)]
    passes = 0
    with ThreadPoolExecutor(nthr) as ex:
        t0 = time.perf_counter()
        while True:
            list(ex.map(lambda c: _oracle_step(w, c), chunks))
            passes += 1
            dt = time.perf_counter() - t0
            if dt >= 0.9 * budget_s:
                break
    b = _seq_bytes(w, seqs)
    return {"value": round(b * passes / dt / 1e9, 4), "unit": "GB/s", "cores": nthr, "kind": "oracle",
            "sample": f"{len(seqs)} of {w.num_seqs} sequences of {workload} ({b / 1e6:.1f} MB of K/V) "
                      f"x {passes} pass(es), FP64 C oracle, {nthr} threads of {ncpu} host cores, "
                      f"sequences dealt round-robin, {dt:.1f} s"}


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return
    import os
    from concurrent.futures import ThreadPoolExecutor
    w = _workload(args.workload)
    # the oracle on the host's cores: a step's sequences dealt round-robin to
    # one thread per core (the C oracle runs outside the GIL)
    ncpu = os.cpu_count() or 1
    budget = min(args.cpu_seconds, 150.0 / max(1, args.steps + max(3, args.warmup)))
    seqs = _sample_seqs(w, budget * ncpu)
    b = _seq_bytes(w, seqs)
    nthr = max(1, min(ncpu, len(seqs)))
    chunks = [seqs[i::nthr] for i in range(nthr)]
    pool = ThreadPoolExecutor(nthr)

    def oracle_step():
        list(pool.map(lambda c: _oracle_step(w, c), chunks))

    warm = max(3, args.warmup)
    t0 = time.perf_counter()
    oracle_step()
    t_one = max(time.perf_counter() - t0, 1e-6)
    # keep the whole run to a few minutes: the warm-up and at least 3 timed
    # steps, at most the requested count
    warm = max(3, min(warm, int(30.0 / t_one)))
    steps = max(3, min(args.steps, int(120.0 / t_one)))
    for _ in range(warm - 1):
        oracle_step()
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step()
    dt = time.perf_counter() - t0
    pool.shutdown()
    value = b * steps / dt / 1e9
    ms = dt / steps * 1e3
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": steps,
        "steps_requested": args.steps,
        "warmup": warm,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) BF16 q/K/V, seeded lengths and block tables)",
        "config": step_config(w, _workload_splits(w), ws),
        "sample": {"seqs": len(seqs), "of": w.num_seqs, "kv_bytes_per_step": b},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthr, "kind": "oracle",
                         "sample": f"{len(seqs)} of {w.num_seqs} sequences per step, dealt round-robin "
                                   f"to {nthr} threads of {ncpu} host cores"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large_batch",
                    choices=["tiny", "gqa_packed", "gqa_packed_splitk", "gqa_packed_long", "gqa_packed_long_splitk",
                             "long_context", "large_batch", "tiled", "tiled_mixed", "gqa_packed_fp8",
                             "long_context_fp8", "large_batch_fp8"])
    ap.add_argument("--seqs", type=int, default=0,
                    help="paged workloads: run only the first N sequences (a smaller case of the same "
                         "recipe, for profiler captures); not a bench line")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tiled-separate", action="store_true",
                    help="tiled workload: time begin / step_tile x T / finalize as separate calls")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
