#!/usr/bin/env python3
"""Throughput of SpecMamba-style tree verification on one GB300 (or N, one process each).

One step = one speculative round of the target's SSM side over one batch, for
every layer of every sequence: the commit of the previous round's accepted
path (selective recompute, conv ring advance) folded into the verify of this
round's tree (tree conv + SiLU, Δ, state update, y for every node) by
ssm_commit_verify, then ssm_accept_path.  The same round through the separate
calls (ssm_tree_verify -> ssm_accept_path -> ssm_commit) is timed as well and
reported under "separate_calls".  Metric: verified tree-node SSM updates per
second = nodes x layers x sequences / step time.

Default workload: batched target verify on the Mamba2-2.7B layer shape
(80 heads x 64, d_state 128), 64 layers, batch 16, one seed-generated 16-node
tree per sequence (<= 3 children, depth <= 4).  Inputs (8.9 GB per step) are
larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload on the host cores.  Under
torchrun each rank runs its own 16 sequences (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "verified tree-node SSM updates/s (all layers, 2.7B shape)"
UNIT = "updates/s"
DEFAULT_WORKLOAD = 3
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# byte counts (algorithmic: every tensor the step must touch, once)
# ---------------------------------------------------------------------------
def verify_bytes_per_instance(H, P, N, n):
    d_inner, conv_dim = H * P, H * P + 2 * N
    return H * P * N * 4 + n * conv_dim * 2 + n * H * 2 + 3 * conv_dim * 2 + n * d_inner * 4 + 4


def params_bytes_per_layer(H, P, N):
    conv_dim = H * P + 2 * N
    return conv_dim * 4 * 4 + conv_dim * 4 + 3 * H * 4


def commit_verify_bytes_per_instance(H, P, N, n, path_len):
    """Fused call: state read + write, the tree's inputs and y, the previous path's rows
    (with the three ring rows before them) and dt, the ring rows written."""
    d_inner, conv_dim = H * P, H * P + 2 * N
    return (2 * H * P * N * 4 + n * conv_dim * 2 + n * H * 2 + n * d_inner * 4
            + (path_len + 3) * conv_dim * 2 + path_len * H * 2 + min(path_len, 3) * conv_dim * 2 + 8)


def commit_bytes_per_instance(H, P, N, path_len):
    conv_dim = H * P + 2 * N
    return (2 * H * P * N * 4 + (path_len + 3) * conv_dim * 2 + path_len * H * 2
            + min(path_len, 3) * conv_dim * 2 + 8)


# ---------------------------------------------------------------------------
# distributed plumbing (host side; no collective touches the data path)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_sequences(batch: int, rank: int):
    """Weak scaling: rank r owns sequences [r*batch, (r+1)*batch) of the seed space."""
    return list(range(rank * batch, (rank + 1) * batch))


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        self.t0 = time.time()

    def mark(self):
        self.t_begin = time.time()

    def stop(self):
        self.t_end = time.time()
        time.sleep(0.12)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        # samples are ~50 ms apart; keep those from the second half (under load)
        load = rows[len(rows) // 3:] or rows
        sm = [float(r[1]) for r in load if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(load)}


# ---------------------------------------------------------------------------
# fp64 oracle as the CPU baseline / reference arm (host cores, spawn pool)
# ---------------------------------------------------------------------------
def _oracle_task(args):
    """One instance of the step on the CPU oracle: verify + accept + commit."""
    import numpy as np

    import oracle
    prm, parent, xBC, dt, h0, ring, head, tok, tgt = args
    oracle.verify(prm, parent, xBC, dt, h0, ring, head)
    path, _ = oracle.accept(parent, tok, tgt)
    oracle.commit(prm, parent, path, xBC, dt, h0, ring, head)
    return len(parent)


def _oracle_inputs(w, seq, layer, tree=0):
    import numpy as np

    from synth import batch
    from tests.helpers import f64, params_at
    b = batch(w, seqs=[seq], layers=[layer], tree=tree)
    return (params_at(b["params"], 0), b["parent"][0], f64(b["xBC"][0, 0]), f64(b["dt"][0, 0]),
            b["h0"][0, 0].astype(np.float64), f64(b["ring"][0, 0]), int(b["ring_head"][0, 0]), b["tok"][0],
            b["tgt"][0])


class OracleRunner:
    """Spawn pool of single-threaded numpy workers over sampled instances."""

    def __init__(self, w, n_inputs=None, tree=0):
        import multiprocessing as mp
        self.cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        self.pool = mp.get_context("spawn").Pool(self.cores)
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k)
            else:
                os.environ[k] = v
        import random
        rnd = random.Random(0x5EED)
        insts = [(0, 0), (w.batch - 1, w.n_layers - 1)]
        while len(insts) < (n_inputs or self.cores):
            insts.append((rnd.randrange(w.batch), rnd.randrange(w.n_layers)))
        self.insts = insts
        self.inputs = [_oracle_inputs(w, s, l, tree) for s, l in insts]
        self.cursor = 0

    def step(self):
        """One bounded sample: `cores` instances in parallel; returns (units, seconds)."""
        batch = [self.inputs[(self.cursor + i) % len(self.inputs)] for i in range(self.cores)]
        self.cursor += self.cores
        t0 = time.perf_counter()
        units = sum(self.pool.map(_oracle_task, batch, chunksize=1))
        return units, time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(w, steps=64, tree=0):
    r = OracleRunner(w, tree=tree)
    r.step()  # warm the workers (imports)
    units = secs = 0.0
    for _ in range(steps):
        u, s = r.step()
        units += u
        secs += s
    r.close()
    return {"value": units / secs, "unit": UNIT, "cores": r.cores, "kind": "oracle",
            "sample": f"{steps} x {r.cores} instances (seq, layer) of the same workload, each verify+accept+commit "
                      f"of one {w.n_nodes(tree)}-node tree in fp64 numpy, one instance per core; "
                      f"{int(units)} node updates in {secs:.1f} s"}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    r = OracleRunner(w)
    for _ in range(args.warmup):
        r.step()
    units = secs = 0.0
    for _ in range(args.steps):
        u, s = r.step()
        units += u
        secs += s
    r.close()
    value = units / secs
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "sample": f"{r.cores} instances per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": r.cores, "kind": "oracle",
                             "sample": f"{args.steps} steps x {r.cores} instances (seq, layer), fp64 numpy "
                                       "oracle, one instance per core"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # GB300 FP32 CUDA-core peak at the 2070 MHz maximum SM clock


def source_digest(paths):
    """sha256 prefix of the concatenated kernel sources a capture was taken on."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(call, units):
    """DRAM bytes of one call (all its launches) from a committed ncu summary
    (profiles/dram_traffic.txt), scaled to `units` instances; None if absent or
    taken on other kernel source (`source=` lists the files, joined by '+')."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if kv.get("call") != call:
            continue
        srcs = [os.path.join(ROOT, "speculative_decoding_mamba2_gb300", "csrc", f)
                for f in kv.get("source", "").split("+") if f]
        if not srcs or not all(os.path.exists(s) for s in srcs) or source_digest(srcs) != kv.get("sha"):
            return None
        return float(kv["bytes_per_unit"]) * units
    return None


def _timed(steps, fn, world, stream, n_events):
    """Run fn(events) `steps` times between a barrier + synchronize on both sides;
    returns (ms per step over the whole region, per-step event lists)."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(steps):
        fn(k, evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    return start.elapsed_time(end) / steps, evs


def run_ours(args, w):
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (Dims, ssm_accept_path, ssm_commit, ssm_commit_verify,
                                                   ssm_commit_verify_workspace_size, ssm_tree_layout_build,
                                                   ssm_tree_verify, ssm_tree_verify_workspace_size)
    from speculative_decoding_mamba2_gb300 import build as _build
    from synth import batch, workload

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    dev = torch.device("cuda", local)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)  # spawn pool before any CUDA work is queued

    # ---- inputs: this rank's sequences, all layers, resident in HBM ----
    seqs = shard_sequences(w.batch, rank)
    b = batch(w, seqs=seqs)
    S, L, n = len(seqs), w.n_layers, w.n_nodes()
    H, P, N = w.shape.H, w.shape.P, w.shape.N
    I = S * L
    dims = Dims(n_heads=H, n_layers=L, ring_cap=w.ring_cap)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    layout_h, depth = ssm_tree_layout_build(b["parent"], max_branches=3, max_depth=4)
    max_path = depth + 1
    prm = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev) for k, v in b["params"].items()}
    layout = torch.from_numpy(layout_h).to(dev)
    # two input buffers: a round commits the previous round's path (its tree's rows) and
    # verifies its own tree
    xBC = [bf16(b["xBC"]), bf16(b["xBC"])]
    dt = [bf16(b["dt"]), bf16(b["dt"])]
    h = torch.from_numpy(b["h0"]).to(dev)
    ring = bf16(b["ring"])
    head = torch.from_numpy(b["ring_head"]).to(dev)
    tok, tgt = torch.from_numpy(b["tok"]).to(dev), torch.from_numpy(b["tgt"]).to(dev)
    y = torch.empty((I, n, H * P), device=dev)
    path = torch.empty((S, max_path), dtype=torch.int32, device=dev)
    plen = torch.empty(S, dtype=torch.int32, device=dev)
    bonus = torch.empty(S, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, depth), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(ssm_commit_verify_workspace_size(dims, S, n, depth, max_path), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def separate(k, ev=None):
        if ev is not None:
            ev[0].record(stream)
        ssm_tree_verify(dims, prm, S, n, depth, layout, xBC[0], dt[0], h, ring, head, y, ws, status)
        if ev is not None:
            ev[1].record(stream)
        ssm_accept_path(S, n, max_path, layout, tok, tgt, path, plen, bonus, status)
        if ev is not None:
            ev[2].record(stream)
        ssm_commit(dims, prm, S, n, layout, max_path, path, plen, xBC[0], dt[0], h, ring, head, status)
        if ev is not None:
            ev[3].record(stream)

    rounds = [0]  # fused rounds so far: round r verifies buffer (r+1)%2, commits the path of r%2

    def fused(k, ev=None):
        cur, prev = (rounds[0] + 1) % 2, rounds[0] % 2
        rounds[0] += 1
        if ev is not None:
            ev[0].record(stream)
        ssm_commit_verify(dims, prm, S, n, layout, max_path, path, plen, xBC[prev], dt[prev], n, depth, layout,
                          xBC[cur], dt[cur], h, ring, head, y, ws_f, status)
        if ev is not None:
            ev[1].record(stream)
        ssm_accept_path(S, n, max_path, layout, tok, tgt, path, plen, bonus, status)
        if ev is not None:
            ev[2].record(stream)

    for k in range(args.warmup):
        separate(k)
    # the fused rounds start from a verified and accepted tree whose commit is pending
    ssm_tree_verify(dims, prm, S, n, depth, layout, xBC[0], dt[0], h, ring, head, y, ws, status)
    ssm_accept_path(S, n, max_path, layout, tok, tgt, path, plen, bonus, status)
    for k in range(args.warmup):
        fused(k)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} after warm-up")
    path_lens = plen.cpu().numpy()

    clocks = ClockSampler(local)
    clocks.start()
    clocks.mark()
    ms, evs = _timed(args.steps, fused, world, stream, 3)
    clk = clocks.stop()
    ms = max_over_ranks(ms, world, dev)
    cv_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    acc_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    units_per_step = n * L * S * world
    value = units_per_step / (ms / 1e3)

    # the same rounds through the separate calls (the pending commit first)
    last = rounds[0] % 2
    ssm_commit(dims, prm, S, n, layout, max_path, path, plen, xBC[last], dt[last], h, ring, head, status)
    for k in range(3):
        separate(k)
    ms_sep, evs_sep = _timed(args.steps, separate, world, stream, 4)
    ms_sep = max_over_ranks(ms_sep, world, dev)
    verify_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs_sep)
    accept_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs_sep)
    commit_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs_sep)

    # ---- roofline of the dominant call ----
    peak, peak_kind = measured_peaks()
    pb = L * params_bytes_per_layer(H, P, N)
    fb = sum(L * commit_verify_bytes_per_instance(H, P, N, n, int(pl)) for pl in path_lens) + pb
    vb = I * verify_bytes_per_instance(H, P, N, n) + pb
    cb = sum(L * commit_bytes_per_instance(H, P, N, int(pl)) for pl in path_lens) + pb
    kernels = {
        "ssm_commit_verify": {"ms": cv_ms, "bytes": fb, "GB/s": fb / cv_ms / 1e6, "launches_per_step": 2,
                              "frac_of_hbm_peak": fb / cv_ms / 1e6 / peak},
        "ssm_accept_path": {"ms": acc_ms, "launches_per_step": 1},
    }
    separate_calls = {
        "ms_per_step": ms_sep, "value": units_per_step / (ms_sep / 1e3),
        "ssm_tree_verify": {"ms": verify_ms, "bytes": vb, "GB/s": vb / verify_ms / 1e6, "launches_per_step": 2,
                            "frac_of_hbm_peak": vb / verify_ms / 1e6 / peak,
                            "traffic": ncu_traffic("ssm_tree_verify", I)},
        "ssm_accept_path": {"ms": accept_ms, "launches_per_step": 1},
        "ssm_commit": {"ms": commit_ms, "bytes": cb, "GB/s": cb / commit_ms / 1e6, "launches_per_step": 2,
                       "frac_of_hbm_peak": cb / commit_ms / 1e6 / peak,
                       "traffic": ncu_traffic("ssm_commit", I)},
    }
    ach = kernels["ssm_commit_verify"]["GB/s"]
    roofline = {"bound": "hbm", "kernel": "ssm_commit_verify (tree_prep_kernel + tree_verify_kernel<4,true>)",
                "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                "traffic": ncu_traffic("ssm_commit_verify", I), "algorithmic_bytes": fb}

    # ---- end to end through the public API, host buffers ----
    e2e = None
    if not args.no_e2e:
        del ws
        e2e = run_e2e(args, w, b, dims, prm, h, ring, head, ws_f, dev, stream, world)

    # ---- draft side (the draft model's own rounds) ----
    draft = None
    if not args.no_draft:
        del y, ws_f, xBC, dt
        draft = run_draft(args, dev, stream, peak, world, rank)

    # ---- draft-side tree drafting (branch states from the log) ----
    draft_tree = None
    if not args.no_draft:
        draft_tree = run_draft_tree(args, dev, stream, peak, world, rank)

    # ---- the target tree verify at batch 1 ----
    config2 = None
    if not args.no_config2:
        config2 = run_config2(args, dev, stream, world, rank, peak, peak_kind)
        if rank == 0 and cpu is not None:
            config2["cpu_baseline"] = cpu_baseline(workload(2), steps=4)

    # ---- the stress workload: ternary tree, 256-node chain, 16-step replay ----
    config4 = None
    chain = None
    if not args.no_config4:
        config4 = run_config4(args, dev, stream, world, rank, peak, peak_kind)
        c = config4["chain"]
        chain = {"workload": config4["workload"] + " (chain tree)", "nodes": c["nodes"],
                 "instances_per_gpu": config4["instances_per_gpu"], "ms": c["ssm_tree_verify"]["ms"],
                 "value": c["nodes"] * config4["instances_per_gpu"] * world / (c["ssm_tree_verify"]["ms"] / 1e3),
                 "unit": "verified tree-node SSM updates/s (ssm_tree_verify alone)",
                 "roofline": {"bound": "hbm", "achieved": c["ssm_tree_verify"]["GB/s"], "peak": peak, "unit": "GB/s",
                              "frac": c["ssm_tree_verify"]["frac_of_hbm_peak"], "peak_source": peak_kind,
                              "traffic": c["ssm_tree_verify"]["traffic"]},
                 "bytes": c["ssm_tree_verify"]["bytes"], "state_TFLOP/s": c["state_TFLOP/s"], "fp32_alu": c["fp32_alu"]}
        if rank == 0 and cpu is not None:
            config4["cpu_baseline"] = cpu_baseline(workload(4), steps=2)
            config4["cpu_baseline"]["sample"] += ("; the 40-node ternary tree only: the oracle walks every node's "
                                                  "path, about 46 s per 256-node chain instance on one core")
    elif not args.no_chain:
        chain = run_chain(args, dev, stream, world, rank)

    # ---- whole blocks: the dense steps either side of the SSM ----
    block = None
    if not args.no_block:
        block = run_block(args, dev, stream, world, rank, peak)

    if status.item() != 0:
        raise RuntimeError(f"device status {int(status.item())} after the timed steps")
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": w.name, "sequences_per_gpu": S, "layers": L, "nodes_per_tree": n,
                           "heads": H, "head_dim": P, "d_state": N, "mean_accepted_path": float(path_lens.mean()),
                           "l2": f"inputs exceed L2 ({fb / 1e9:.2f} GB touched per step); no flush"},
                "roofline": roofline, "kernels": kernels, "separate_calls": separate_calls,
                "e2e": e2e, "gpu_launches": 3 * args.steps, "clocks": clk}
        if draft is not None:
            line["draft"] = draft
        if draft_tree is not None:
            line["draft_tree"] = draft_tree
        if config2 is not None:
            line["config2"] = config2
        if config4 is not None:
            line["config4"] = config4
        if chain is not None:
            line["chain"] = chain
        if block is not None:
            line["block"] = block
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def folded_rounds(w, b, dev, stream, world, steps, warmup, flush=None, tree=0):
    """Speculative rounds of one tree workload through the folded call: round r runs
    ssm_commit_verify (commit of round r-1's accepted path, verify of round r's tree; two
    input buffers alternate) and ssm_accept_path.  CUDA events around each call of each
    timed round; `flush` (a device buffer larger than L2) is rewritten before every round,
    outside the events, when the round's working set would otherwise stay in L2.
    Returns the mean event times, the path lengths and the device state."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (Dims, ssm_accept_path, ssm_commit_verify,
                                                   ssm_commit_verify_workspace_size, ssm_tree_layout_build,
                                                   ssm_tree_verify, ssm_tree_verify_workspace_size)
    S, L, n = len(b["seqs"]), w.n_layers, b["n_nodes"]
    H, P, N = w.shape.H, w.shape.P, w.shape.N
    I = S * L
    dims = Dims(n_heads=H, n_layers=L, ring_cap=w.ring_cap)
    bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    spec = w.trees[tree]
    layout_h, depth = ssm_tree_layout_build(b["parent"], max_branches=3, max_depth=depth_cap(spec))
    max_path = depth + 1
    prm = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev) for k, v in b["params"].items()}
    layout = torch.from_numpy(layout_h).to(dev)
    xBC = [bf16(b["xBC"]), bf16(b["xBC"])]
    dt = [bf16(b["dt"]), bf16(b["dt"])]
    h = torch.from_numpy(b["h0"]).to(dev)
    ring = bf16(b["ring"])
    head = torch.from_numpy(b["ring_head"]).to(dev)
    tok, tgt = torch.from_numpy(b["tok"]).to(dev), torch.from_numpy(b["tgt"]).to(dev)
    y = torch.empty((I, n, H * P), device=dev)
    path = torch.empty((S, max_path), dtype=torch.int32, device=dev)
    plen = torch.empty(S, dtype=torch.int32, device=dev)
    bonus = torch.empty(S, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, depth), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(ssm_commit_verify_workspace_size(dims, S, n, depth, max_path), dtype=torch.uint8, device=dev)
    # the rounds start from a verified and accepted tree whose commit is pending
    ssm_tree_verify(dims, prm, S, n, depth, layout, xBC[0], dt[0], h, ring, head, y, ws, status)
    ssm_accept_path(S, n, max_path, layout, tok, tgt, path, plen, bonus, status)
    del ws
    rounds = [0]

    def one(ev=None):
        cur, prev = (rounds[0] + 1) % 2, rounds[0] % 2
        rounds[0] += 1
        if flush is not None:
            flush.fill_(1)
        if ev is not None:
            ev[0].record(stream)
        ssm_commit_verify(dims, prm, S, n, layout, max_path, path, plen, xBC[prev], dt[prev], n, depth, layout,
                          xBC[cur], dt[cur], h, ring, head, y, ws_f, status)
        if ev is not None:
            ev[1].record(stream)
        ssm_accept_path(S, n, max_path, layout, tok, tgt, path, plen, bonus, status)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    path_lens = plen.cpu().numpy()
    _, evs = _timed(steps, lambda k, ev: one(ev), world, stream, 3)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the rounds of {w.name}")
    cv_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in evs), world, dev)
    acc_ms = max_over_ranks(statistics.mean(e[1].elapsed_time(e[2]) for e in evs), world, dev)
    round_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[2]) for e in evs), world, dev)
    return {"cv_ms": cv_ms, "acc_ms": acc_ms, "round_ms": round_ms, "path_lens": path_lens, "h": h, "ring": ring,
            "head": head, "prm": prm, "dims": dims, "S": S, "L": L, "n": n, "depth": depth}


def depth_cap(spec):
    """max_depth cap passed to the layout build for a tree spec (the tree_config of the workload)."""
    if spec[0] == "random":
        return spec[3]
    if spec[0] == "full":
        return spec[2]
    return spec[1] - 1


def tree_roofline(w, r, peak, peak_kind, n_units, world, traffic_call=None):
    """Roofline of one folded round (ssm_commit_verify) and the round's throughput; the DRAM
    traffic of the call when profiles/dram_traffic.txt holds a capture `traffic_call` on the
    current kernel sources (per instance, scaled to the call's instances)."""
    import numpy as np
    H, P, N = w.shape.H, w.shape.P, w.shape.N
    pb = r["L"] * params_bytes_per_layer(H, P, N)
    fb = sum(r["L"] * commit_verify_bytes_per_instance(H, P, N, r["n"], int(pl)) for pl in r["path_lens"]) + pb
    ach = fb / r["cv_ms"] / 1e6
    return {"value": n_units * world / (r["round_ms"] / 1e3), "unit": UNIT, "ms_per_round": r["round_ms"],
            "ssm_commit_verify": {"ms": r["cv_ms"], "launches_per_round": 2},
            "ssm_accept_path": {"ms": r["acc_ms"], "launches_per_round": 1},
            "mean_accepted_path": float(np.mean(r["path_lens"])),
            "roofline": {"bound": "hbm", "kernel": "ssm_commit_verify (tree_prep_kernel + tree_verify_kernel)",
                         "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback", "algorithmic_bytes": fb,
                         "traffic": ncu_traffic(traffic_call, r["L"] * r["S"]) if traffic_call else None}}


def run_config2(args, dev, stream, world, rank, peak, peak_kind):
    """The target tree verify at batch 1 (Mamba2-2.7B shape, 64 layers, one 16-node random
    tree per rank): folded rounds (ssm_commit_verify + ssm_accept_path).  The round touches
    about 0.33 GB, a little more than L2, so a 256 MB buffer is rewritten before every
    round (outside the events): every round reads the state from HBM."""
    import torch

    from synth import batch, workload
    w = workload(2)
    b = batch(w, seqs=shard_sequences(w.batch, rank))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    steps = max(20, min(args.steps, 200))
    r = folded_rounds(w, b, dev, stream, world, steps, args.warmup, flush=flush)
    out = {"workload": w.name, "sequences_per_gpu": r["S"], "layers": r["L"], "nodes_per_tree": r["n"],
           "steps": steps, "l2": "256 MB written before every round (outside the timed events)"}
    # the traffic capture of ssm_commit_verify is taken on this workload (64 instances)
    out.update(tree_roofline(w, r, peak, peak_kind, r["n"] * r["L"] * r["S"], world, traffic_call="ssm_commit_verify"))
    return out


def run_config4(args, dev, stream, world, rank, peak, peak_kind):
    """The stress workload (Mamba2-780M shape, 48 layers, batch 64 per rank), each round:
      * ternary: the 40-node full ternary tree of depth 3 through the folded call
        (ssm_commit_verify: commit of the previous round's accepted path, verify) +
        ssm_accept_path;
      * chain: the 256-node chain tree verified from the same committed state
        (ssm_tree_verify, which takes the chain kernels), ssm_accept_path, and ssm_commit
        of its accepted path into a state buffer of its own (set up as a copy of the
        committed state; the per-round copy is not part of the timed work);
      * replay: the draft's ssm_replay of 16 logged steps for every instance (the logs
        written by 16 ssm_draft_step calls before the timed rounds).
    Every part touches far more than L2.  Inputs come from the seeded generator on a pool
    of host processes (synth.batch_parallel, identical to synth.batch)."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (ssm_accept_path, ssm_commit, ssm_draft_step, ssm_replay,
                                                   ssm_tree_layout_build, ssm_tree_verify,
                                                   ssm_tree_verify_workspace_size)
    from synth import batch_parallel, draft_inputs, workload
    w = workload(4)
    seqs = shard_sequences(w.batch, rank)
    t_gen = time.perf_counter()
    b = batch_parallel(w, seqs=seqs)
    bc = batch_parallel(w, seqs=seqs, tree=1, with_state=False)
    t_gen = time.perf_counter() - t_gen
    H, P, N = w.shape.H, w.shape.P, w.shape.N
    steps = max(5, min(args.steps, 10))
    r = folded_rounds(w, b, dev, stream, world, steps, args.warmup)
    tern = tree_roofline(w, r, peak, peak_kind, r["n"] * r["L"] * r["S"], world)
    dims, prm, S, L = r["dims"], r["prm"], r["S"], r["L"]
    I = S * L
    del b

    # ---- the chain tree, from the committed state ----
    bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    nc = bc["n_nodes"]
    lay_c, depth_c = ssm_tree_layout_build(bc["parent"])
    lay_c = torch.from_numpy(lay_c).to(dev)
    xc, dc = bf16(bc["xBC"]), bf16(bc["dt"])
    tok_c, tgt_c = torch.from_numpy(bc["tok"]).to(dev), torch.from_numpy(bc["tgt"]).to(dev)
    del bc
    h, ring, head = r["h"], r["ring"], r["head"]
    h_c, ring_c, head_c = h.clone(), ring.clone(), head.clone()
    yc = torch.empty((I, nc, dims.d_inner), device=dev)
    ws_c = torch.empty(ssm_tree_verify_workspace_size(dims, S, nc, depth_c), dtype=torch.uint8, device=dev)
    mp_c = nc
    path_c = torch.empty((S, mp_c), dtype=torch.int32, device=dev)
    plen_c = torch.empty(S, dtype=torch.int32, device=dev)
    bonus_c = torch.empty(S, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def chain_round(ev=None):
        if ev is not None:
            ev[0].record(stream)
        ssm_tree_verify(dims, prm, S, nc, depth_c, lay_c, xc, dc, h, ring, head, yc, ws_c, status)
        if ev is not None:
            ev[1].record(stream)
        ssm_accept_path(S, nc, mp_c, lay_c, tok_c, tgt_c, path_c, plen_c, bonus_c, status)
        if ev is not None:
            ev[2].record(stream)
        ssm_commit(dims, prm, S, nc, lay_c, mp_c, path_c, plen_c, xc, dc, h_c, ring_c, head_c, status)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(2):
        chain_round()
    torch.cuda.synchronize()
    _, evs = _timed(steps, lambda k, ev: chain_round(ev), world, stream, 4)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the chain rounds")
    cvm = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in evs), world, dev)
    cam = max_over_ranks(statistics.mean(e[1].elapsed_time(e[2]) for e in evs), world, dev)
    ccm = max_over_ranks(statistics.mean(e[2].elapsed_time(e[3]) for e in evs), world, dev)
    plc = plen_c.cpu().numpy()
    del yc, ws_c, xc, dc, h_c, ring_c
    d_inner, conv_dim = H * P, H * P + 2 * N
    cby = I * (H * P * N * 4 + nc * conv_dim * 2 + nc * H * 2 + 3 * conv_dim * 2 + nc * d_inner * 4)
    ccb = sum(L * commit_bytes_per_instance(H, P, N, int(pl)) for pl in plc) + L * params_bytes_per_layer(H, P, N)
    chain = {"nodes": nc, "ms_per_round": cvm + cam + ccm, "mean_accepted_path": float(plc.mean()),
             "value": nc * I * world / ((cvm + cam + ccm) / 1e3), "unit": UNIT,
             "ssm_tree_verify": {"ms": cvm, "bytes": cby, "GB/s": cby / cvm / 1e6,
                                 "frac_of_hbm_peak": cby / cvm / 1e6 / peak,
                                 "traffic": ncu_traffic("ssm_tree_verify_chain", I)},
             "ssm_accept_path": {"ms": cam},
             "ssm_commit": {"ms": ccm, "bytes": ccb, "GB/s": ccb / ccm / 1e6, "frac_of_hbm_peak": ccb / ccm / 1e6 / peak}}
    flops = 4.0 * nc * H * P * N * I
    tf = flops / (cvm / 1e3) / 1e12
    chain["state_TFLOP/s"] = tf
    chain["fp32_alu"] = {"achieved": tf, "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": tf / FP32_ALU_TFLOPS,
                         "note": "context only: the CUDA-core bound of a plain recurrence; the chain kernels "
                                 "run their products on the tensor cores"}

    # ---- the draft's replay of 16 logged steps (780M shape, every instance) ----
    T = w.draft_steps
    xs = torch.empty((T, I, conv_dim), dtype=torch.int16)
    dts = torch.empty((T, I, H), dtype=torch.int16)
    for i, q in enumerate(seqs):
        for l in range(L):
            xb, db = draft_inputs(w, q, l)
            xs[:, i * L + l] = torch.from_numpy(xb.view(np.int16))
            dts[:, i * L + l] = torch.from_numpy(db.view(np.int16))
    xs = xs.to(dev).view(torch.bfloat16)
    dts = dts.to(dev).view(torch.bfloat16)
    h_ck = h.clone()
    h_work = torch.empty_like(h_ck)
    log_d = torch.zeros(I, T, H, device=dev)
    log_b = torch.zeros(I, T, N, device=dev)
    log_x = torch.zeros(I, T, d_inner, device=dev)
    log_len = torch.zeros(I, dtype=torch.int32, device=dev)
    yd = torch.empty(I, d_inner, device=dev)
    for t in range(T):
        ssm_draft_step(dims, prm, S, t, T, xs[t], dts[t], h_ck if t == 0 else h_work, h_work, ring, head,
                       log_d, log_b, log_x, log_len, yd, status)
    del h_work, xs, dts
    kk = torch.full((S,), T, dtype=torch.int32, device=dev)
    head_d = head.clone()

    def replay(ev=None):
        log_len.fill_(T)  # the logs stay valid; replay consumed the count
        if ev is not None:
            ev[0].record(stream)
        ssm_replay(dims, prm, S, T, kk, log_d, log_b, log_x, log_len, h_ck, head_d, status)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(2):
        replay()
    torch.cuda.synchronize()
    _, evs = _timed(steps, lambda k, ev: replay(ev), world, stream, 2)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the replays")
    rpm = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in evs), world, dev)
    rb = replay_bytes(H, P, N, I, T)
    rep = {"steps_replayed": T, "ms": rpm, "bytes": rb, "GB/s": rb / rpm / 1e6, "frac_of_hbm_peak": rb / rpm / 1e6 / peak}
    round_ms = tern["ms_per_round"] + chain["ms_per_round"] + rpm
    out = {"workload": w.name, "sequences_per_gpu": S, "layers": L, "instances_per_gpu": I, "steps": steps,
           "ms_per_round": round_ms, "value": (r["n"] + nc) * I * world / (round_ms / 1e3), "unit": UNIT,
           "note": "one round = ternary (ssm_commit_verify + ssm_accept_path) + chain (ssm_tree_verify + "
                   "ssm_accept_path + ssm_commit) + ssm_replay of 16 steps; every part exceeds L2",
           "input_generation_s": t_gen, "ternary": tern, "chain": chain, "replay": rep}
    return out


def run_chain(args, dev, stream, world, rank, seqs_per_rank=8):
    """The stress workload's 256-node chain tree (Mamba2-780M shape, 48 layers) through
    ssm_tree_verify, which takes the chain kernel: 16-node chunks, each a tree verify
    from the chunk's entry state plus the commit of the whole chunk, all on the tensor
    cores with the state in registers.  Roofline: HBM (h0 read once, the inputs, y),
    which binds before the tensor pipe.  A bounded sample of the batch-64 workload:
    `seqs_per_rank` sequences x 48 layers."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (Dims, ssm_tree_layout_build, ssm_tree_verify,
                                                   ssm_tree_verify_workspace_size)
    from synth import batch, workload
    w = workload(4)
    seqs = list(range(rank * seqs_per_rank, (rank + 1) * seqs_per_rank))
    b = batch(w, seqs=seqs, tree=1)
    S, L, n = len(seqs), w.n_layers, b["n_nodes"]
    H, P, N = w.shape.H, w.shape.P, w.shape.N
    I = S * L
    dims = Dims(n_heads=H, n_layers=L, ring_cap=w.ring_cap)
    bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    lay, depth = ssm_tree_layout_build(b["parent"])
    prm = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev) for k, v in b["params"].items()}
    layout = torch.from_numpy(lay).to(dev)
    xBC, dt = bf16(b["xBC"]), bf16(b["dt"])
    h0 = torch.from_numpy(b["h0"]).to(dev)
    ring = bf16(b["ring"])
    head = torch.from_numpy(b["ring_head"]).to(dev)
    y = torch.empty((I, n, H * P), device=dev)
    ws = torch.empty(ssm_tree_verify_workspace_size(dims, S, n, depth), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    del b

    def call(k, ev=None):
        if ev is not None:
            ev[0].record(stream)
        ssm_tree_verify(dims, prm, S, n, depth, layout, xBC, dt, h0, ring, head, y, ws, status)
        if ev is not None:
            ev[1].record(stream)

    for k in range(3):
        call(k)
    torch.cuda.synchronize()
    steps = max(5, min(args.steps, 20))
    ms, evs = _timed(steps, call, world, stream, 2)
    ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in evs), world, dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the chain verify")
    peak, peak_kind = measured_peaks()
    d_inner, conv_dim = H * P, H * P + 2 * N
    by = I * (H * P * N * 4 + n * conv_dim * 2 + n * H * 2 + 3 * conv_dim * 2 + n * d_inner * 4)
    flops = 4.0 * n * H * P * N * I  # C·h and u·B over the state, 2 FLOP each per element and node
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": w.name + f" (chain tree; a sample of {S} sequences x {L} layers per GPU)",
            "nodes": n, "instances_per_gpu": I, "ms": ms,
            "value": n * I * world / (ms / 1e3), "unit": "verified tree-node SSM updates/s",
            "roofline": {"bound": "hbm", "achieved": by / ms / 1e6, "peak": peak, "unit": "GB/s",
                         "frac": by / ms / 1e6 / peak, "peak_source": peak_kind,
                         "traffic": ncu_traffic("ssm_tree_verify_chain", I)},
            "bytes": by, "state_TFLOP/s": tf,
            # the same state FLOPs against the FP32 CUDA-core peak (152 SMs x 128 lanes x 2 FLOP
            # x 2.07 GHz): the bound of a plain recurrence, which these tensor-core products lift
            "fp32_alu": {"achieved": tf, "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": tf / FP32_ALU_TFLOPS}}


def run_block(args, dev, stream, world, rank, peak):
    """Whole-model tree verify: the batched-verify trees (16 sequences x 16-node trees)
    through all 64 blocks of the Mamba2-2.7B shape (d_model 2560) with synthetic weights.
    Per block: RMSNorm -> input projection (tcgen05; z, x|B|C and dt written where the
    next steps read them) -> ssm_commit_verify (the previous round's accepted path
    committed, this round's tree verified) -> gated RMSNorm -> output projection added
    to the residual stream; then the accept walk.  Each round is one CUDA graph of
    those API calls.  The projections are also timed alone, 64 layers back to back."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (Dims, ssm_accept_path, ssm_commit_verify,
                                                   ssm_commit_verify_workspace_size, ssm_gated_rmsnorm,
                                                   ssm_linear, ssm_rmsnorm, ssm_tree_layout_build)
    from synth import batch, layer_params, workload
    w = workload(3)
    S, L, n = w.batch, w.n_layers, w.n_nodes()
    H, P, N, R = w.shape.H, w.shape.P, w.shape.N, w.ring_cap
    d_inner, conv_dim = H * P, H * P + 2 * N
    d_model = d_inner // 2
    n_in = d_inner + conv_dim + H
    T, eps = S * n, 1e-5
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242 + rank)

    def bf16_randn(*shape, scale=1.0):
        return (torch.randn(*shape, device=dev, generator=gen) * scale).to(torch.bfloat16)

    W_in = [bf16_randn(n_in, d_model, scale=d_model ** -0.5) for _ in range(L)]
    W_out = [bf16_randn(d_model, d_inner, scale=d_inner ** -0.5) for _ in range(L)]
    norm_w = [1 + 0.1 * torch.randn(d_model, device=dev, generator=gen) for _ in range(L)]
    gnorm_w = [1 + 0.1 * torch.randn(d_inner, device=dev, generator=gen) for _ in range(L)]
    b = batch(w, layers=[0])  # the trees and tokens (the tree inputs come from the projections)
    prm_all = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev) for k, v in layer_params(w).items()}
    prm = [{k: v[l:l + 1] for k, v in prm_all.items()} for l in range(L)]
    h = [torch.randn(S, H, P, N, device=dev, generator=gen) * 0.1 for _ in range(L)]
    ring = [bf16_randn(S, R, conv_dim) for _ in range(L)]
    head = [torch.full((S,), 3, dtype=torch.int32, device=dev) for _ in range(L)]
    xbc = [[torch.empty(T, conv_dim, dtype=torch.bfloat16, device=dev) for _ in range(L)] for _ in range(2)]
    dtb = [[torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(L)] for _ in range(2)]
    x0 = torch.randn(T, d_model, device=dev, generator=gen)
    x = torch.empty_like(x0)
    u = torch.empty(T, d_model, dtype=torch.bfloat16, device=dev)
    z = torch.empty(T, d_inner, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T, d_inner, device=dev)
    gb = torch.empty(T, d_inner, dtype=torch.bfloat16, device=dev)
    lay, depth = ssm_tree_layout_build(b["parent"], max_branches=3, max_depth=4)
    layout = torch.from_numpy(lay).to(dev)
    max_path = depth + 1
    tok, tgt = torch.from_numpy(b["tok"]).to(dev), torch.from_numpy(b["tgt"]).to(dev)
    path = torch.empty((S, max_path), dtype=torch.int32, device=dev)
    plen = torch.empty(S, dtype=torch.int32, device=dev)
    bonus = torch.empty(S, dtype=torch.int32, device=dev)
    dims1 = Dims(n_heads=H, n_layers=1, ring_cap=R)
    ws = torch.empty(ssm_commit_verify_workspace_size(dims1, S, n, depth, max_path), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def project_in(l, buf, cs):
        ssm_rmsnorm(x, norm_w[l], eps, u, cs)
        ssm_linear(u, W_in[l], [(0, z), (d_inner, xbc[buf][l]), (d_inner + conv_dim, dtb[buf][l])], status=status,
                   stream=cs)

    side_b = torch.cuda.Stream(dev)

    def one_round(cur, cs, reorder):
        """reorder: the B | C | dt rows of the input projection first, the SSM's prep on them
        while the z | x rows are projected on a second stream, then the SSM's main kernel."""
        prev = 1 - cur
        x.copy_(x0)
        for l in range(L):
            cv = (dims1, prm[l], S, n, layout, max_path, path, plen, xbc[prev][l], dtb[prev][l], n, depth, layout,
                  xbc[cur][l], dtb[cur][l], h[l], ring[l], head[l], y, ws, status, cs)
            if not reorder:
                project_in(l, cur, cs)
                ssm_commit_verify(*cv)
            else:
                ssm_rmsnorm(x, norm_w[l], eps, u, cs)
                side_b.wait_stream(cs)
                with torch.cuda.stream(side_b):
                    ssm_linear(u, W_in[l][:2 * d_inner], [(0, z), (d_inner, xbc[cur][l][:, :d_inner])],
                               status=status, stream=side_b)
                ssm_linear(u, W_in[l][2 * d_inner:], [(0, xbc[cur][l][:, d_inner:]), (2 * N, dtb[cur][l])],
                           status=status, stream=cs)
                ssm_commit_verify(*cv, part="prep")
                cs.wait_stream(side_b)
                ssm_commit_verify(*cv, part="main")
            ssm_gated_rmsnorm(y, z, gnorm_w[l], eps, gb, cs)
            ssm_linear(gb, W_out[l], [(0, x)], residual=x, status=status, stream=cs)
        ssm_accept_path(S, n, max_path, layout, tok, tgt, path, plen, bonus, status, cs)

    with torch.cuda.stream(stream):  # a first round's projections and accept, so every round has a path to commit
        x.copy_(x0)
        for l in range(L):
            project_in(l, 1, stream)
        ssm_accept_path(S, n, max_path, layout, tok, tgt, path, plen, bonus, status, stream)
    torch.cuda.synchronize()
    def time_rounds(reorder):
        graphs = []
        for cur in (0, 1):
            gph = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            torch.cuda.synchronize()
            with torch.cuda.graph(gph, stream=side):
                one_round(cur, torch.cuda.current_stream(), reorder)
            graphs.append(gph)
        r = [0]

        def replay(ev=None):
            with torch.cuda.stream(stream):
                graphs[r[0] % 2].replay()
            r[0] += 1

        for _ in range(max(4, args.warmup + args.warmup % 2)):  # even: leaves the state where it started
            replay()
        torch.cuda.synchronize()
        steps = max(6, min(args.steps, 20)) // 2 * 2
        t, _ = _timed(steps, lambda k, ev=None: replay(), world, stream, 0)
        return max_over_ranks(t, world, dev)

    ms_in_order = time_rounds(False)
    ms = time_rounds(True)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the block rounds")

    # the projections alone, 64 layers back to back (weights stream from HBM: 3.5 + 1.7 GB)
    def proj_loop(which):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for l in range(L):
                if which == "in":
                    ssm_linear(u, W_in[l], [(0, z), (d_inner, xbc[0][l]), (d_inner + conv_dim, dtb[0][l])],
                               stream=stream)
                else:
                    ssm_linear(gb, W_out[l], [(0, x)], residual=x, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / L
    proj = {}
    for which, (NN, KK) in (("in", (n_in, d_model)), ("out", (d_model, d_inner))):
        proj_loop(which)
        us = proj_loop(which) * 1e3
        by = NN * KK * 2 + T * KK * 2 + T * NN * (2 if which == "in" else 8)
        fl = 2.0 * T * NN * KK
        proj[which] = {"shape_MNK": [T, NN, KK], "us": us, "GB/s": by / us / 1e3, "TFLOP/s": fl / us / 1e6,
                       "frac_of_hbm_peak": by / us / 1e3 / peak}
    weights = L * (n_in * d_model + d_model * d_inner) * 2
    ssm_bytes = commit_verify_bytes_per_instance(H, P, N, n, float(plen.float().mean())) * S * L
    total = weights + ssm_bytes
    return {"workload": f"whole-model tree verify: {L} Mamba2-2.7B blocks (d_model {d_model}, synthetic weights), "
                        f"batch {S}, {n}-node random trees",
            "ms_per_round": ms, "value": n * S * L * world / (ms / 1e3), "unit": UNIT,
            "tree_tokens_per_s": n * S * world / (ms / 1e3),
            "bytes_per_round": total, "weights_bytes": weights,
            "roofline": {"bound": "hbm", "achieved": total / ms / 1e6, "peak": peak, "unit": "GB/s",
                         "frac": total / ms / 1e6 / peak},
            "launches_per_round": L * 7 + 1, "projections": proj,
            "order": "per block: the B|C|dt rows of the input projection first; the SSM's prep on them while "
                     "the z|x rows are projected on a second stream; then the SSM's main kernel",
            "ms_per_round_in_order": ms_in_order}


def run_draft_only(args):
    """The draft side alone (one GPU): the one-token draft steps with replay, and tree
    drafting level by level with the commit of the accepted path."""
    import torch
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    peak, _ = measured_peaks()
    out = {"draft": run_draft(args, dev, stream, peak, 1, 0),
           "draft_tree": run_draft_tree(args, dev, stream, peak, 1, 0)}
    print(json.dumps({"metric": "draft-side rounds", "unit": "see entries", "higher_is_better": True,
                      "data": "synthetic", "hbm_peak_gbs": peak, **out}), flush=True)
    return 0


def run_ternary_only(args):
    """The stress workload's 40-node ternary tree alone (Mamba2-780M shape, 48 layers):
    the folded rounds of config4.ternary on the first `--seqs` sequences (all 64 by
    default), with the same timing and roofline; a smaller --seqs gives a case small
    enough for a profiler capture."""
    import torch

    from synth import batch_parallel, workload
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peaks()
    w = workload(4)
    seqs = list(range(min(max(args.seqs, 1), w.batch)))
    b = batch_parallel(w, seqs=seqs)
    r = folded_rounds(w, b, dev, stream, 1, max(5, min(args.steps, 10)), args.warmup)
    out = {"workload": w.name + f" (40-node ternary tree, {len(seqs)} sequences)",
           "instances": r["L"] * r["S"], "mean_accepted_path": float(r["path_lens"].mean())}
    out.update(tree_roofline(w, r, peak, peak_kind, r["n"] * r["L"] * r["S"], 1))
    print(json.dumps({"metric": "ternary-tree folded rounds", "higher_is_better": True, "data": "synthetic",
                      **out}), flush=True)
    return 0


def run_block_steps(args):
    """One Mamba2-2.7B block's steps at the batched-verify shape (16 sequences x 16 nodes,
    256 tree tokens), each timed alone as a CUDA graph of 8 consecutive layers' launches
    (device time per launch): RMSNorm, the input projection, ssm_commit_verify (and its prep
    and main halves), the gated RMSNorm, the output projection; then the five steps in one
    graph.  Synthetic weights; the state and inputs of each layer are its own."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (Dims, ssm_accept_path, ssm_commit_verify,
                                                   ssm_commit_verify_workspace_size, ssm_gated_rmsnorm, ssm_linear,
                                                   ssm_rmsnorm, ssm_tree_layout_build)
    from synth import batch, layer_params, workload
    dev = torch.device("cuda")
    w = workload(3)
    S, n = w.batch, w.n_nodes()
    H, P, N, R = w.shape.H, w.shape.P, w.shape.N, w.ring_cap
    d_inner, conv_dim = H * P, H * P + 2 * N
    d_model = d_inner // 2
    n_in = d_inner + conv_dim + H
    T, L = S * n, 8
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    W_in = [(torch.randn(n_in, d_model, device=dev, generator=gen) * 0.02).to(torch.bfloat16) for _ in range(L)]
    W_out = [(torch.randn(d_model, d_inner, device=dev, generator=gen) * 0.02).to(torch.bfloat16) for _ in range(L)]
    nw, gw = torch.ones(d_model, device=dev), torch.ones(d_inner, device=dev)
    b = batch(w, layers=[0])
    prm_all = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev)
               for k, v in layer_params(w, range(L)).items()}
    prm = [{k: v[l:l + 1] for k, v in prm_all.items()} for l in range(L)]
    h = [torch.randn(S, H, P, N, device=dev, generator=gen) * 0.1 for _ in range(L)]
    ring = [torch.randn(S, R, conv_dim, device=dev, generator=gen).to(torch.bfloat16) for _ in range(L)]
    head = [torch.full((S,), 3, dtype=torch.int32, device=dev) for _ in range(L)]
    x = torch.randn(T, d_model, device=dev, generator=gen)
    u = torch.empty(T, d_model, dtype=torch.bfloat16, device=dev)
    z = torch.empty(T, d_inner, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T, d_inner, device=dev)
    gb = torch.empty(T, d_inner, dtype=torch.bfloat16, device=dev)
    xbc = [torch.randn(T, conv_dim, device=dev, generator=gen).to(torch.bfloat16) for _ in range(2)]
    dtb = [(torch.randn(T, H, device=dev, generator=gen) * 0.5).to(torch.bfloat16) for _ in range(2)]
    lay, depth = ssm_tree_layout_build(b["parent"])
    layout = torch.from_numpy(lay).to(dev)
    mp = depth + 1
    path = torch.empty((S, mp), dtype=torch.int32, device=dev)
    plen = torch.empty(S, dtype=torch.int32, device=dev)
    bonus = torch.empty(S, dtype=torch.int32, device=dev)
    dims1 = Dims(n_heads=H, n_layers=1, ring_cap=R)
    ws = torch.empty(ssm_commit_verify_workspace_size(dims1, S, n, depth, mp), dtype=torch.uint8, device=dev)
    ssm_accept_path(S, n, mp, layout, torch.from_numpy(b["tok"]).to(dev), torch.from_numpy(b["tgt"]).to(dev),
                    path, plen, bonus)
    torch.cuda.synchronize()

    def cv(l, s, part="all"):
        ssm_commit_verify(dims1, prm[l], S, n, layout, mp, path, plen, xbc[1], dtb[1], n, depth, layout, xbc[0],
                          dtb[0], h[l], ring[l], head[l], y, ws, None, s, part=part)

    steps = {
        "rmsnorm": lambda l, s: ssm_rmsnorm(x, nw, 1e-5, u, s),
        "input projection": lambda l, s: ssm_linear(u, W_in[l], [(0, z), (d_inner, xbc[0]),
                                                                  (d_inner + conv_dim, dtb[0])], stream=s),
        "ssm_commit_verify": lambda l, s: cv(l, s),
        "gated rmsnorm": lambda l, s: ssm_gated_rmsnorm(y, z, gw, 1e-5, gb, s),
        "output projection": lambda l, s: ssm_linear(gb, W_out[l], [(0, x)], residual=x, stream=s),
    }
    halves = {"ssm_commit_verify prep": lambda l, s: cv(l, s, "prep"),
              "ssm_commit_verify main": lambda l, s: cv(l, s, "main")}

    def graph_us(fn):
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn(0, side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for l in range(L):
                fn(l, torch.cuda.current_stream(dev))
        for _ in range(max(3, args.warmup)):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / L * 1e3

    out = {k: graph_us(f) for k, f in {**steps, **halves}.items()}

    def block(l, s):
        for f in steps.values():
            f(l, s)

    out["block (the five steps in one graph)"] = graph_us(block)
    print(json.dumps({"metric": "block step time (Mamba2-2.7B, 16 sequences x 16 nodes)", "unit": "us",
                      "higher_is_better": False, "data": "synthetic", "steps_us": out}), flush=True)
    return 0


def run_linear_only(args):
    """The block's two projections alone at the Mamba2-2.7B shape (256 tree tokens: 16
    sequences x 16 nodes): the input projection [256 x 2560] x [10576 x 2560]^T with its
    z | x B C | dt segments, and the output projection [256 x 5120] x [2560 x 5120]^T added
    into the fp32 residual stream.  Launches are captured in a CUDA graph (device time
    only), the weights rotate over copies larger than L2 (and, for `us_weights_in_l2`, one
    copy stays in L2).  torch.matmul (cuBLAS) on the same product is timed beside it as
    context."""
    import torch

    from speculative_decoding_mamba2_gb300 import ssm_linear
    dev = torch.device("cuda")
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": None}
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    T, d_model, d_inner, H = 256, 2560, 5120, 80
    conv_dim = d_inner + 256
    n_in = d_inner + conv_dim + H

    def graph_us(fn, reps=20):
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            fn(0, side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(reps):
                fn(i, torch.cuda.current_stream(dev))
        for _ in range(max(3, args.warmup)):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3

    out = {}
    A = (torch.randn(T, d_model, device=dev, generator=gen)).to(torch.bfloat16)
    W = [(torch.randn(n_in, d_model, device=dev, generator=gen) * d_model ** -0.5).to(torch.bfloat16) for _ in range(4)]
    z = torch.empty(T, d_inner, device=dev, dtype=torch.bfloat16)
    xbc = torch.empty(T, conv_dim, device=dev, dtype=torch.bfloat16)
    dt = torch.empty(T, H, device=dev, dtype=torch.bfloat16)
    full = torch.empty(T, n_in, device=dev, dtype=torch.bfloat16)
    us = graph_us(lambda i, s: ssm_linear(A, W[i % 4], [(0, z), (d_inner, xbc), (d_inner + conv_dim, dt)], stream=s))
    warm = graph_us(lambda i, s: ssm_linear(A, W[0], [(0, z), (d_inner, xbc), (d_inner + conv_dim, dt)], stream=s))
    ref = graph_us(lambda i, s: torch.matmul(A, W[i % 4].t(), out=full))
    by, fl = n_in * d_model * 2 + T * d_model * 2 + T * n_in * 2, 2.0 * T * n_in * d_model
    out["in"] = {"shape_MNK": [T, n_in, d_model], "us": us, "GB/s": by / us / 1e3, "TFLOP/s": fl / us / 1e6,
                 "frac_of_hbm_peak": by / us / 1e3 / peaks["hbm_gbs"], "us_weights_in_l2": warm,
                 "cublas_matmul_us": ref}
    G = torch.randn(T, d_inner, device=dev, generator=gen).to(torch.bfloat16)
    Wo = [(torch.randn(d_model, d_inner, device=dev, generator=gen) * d_inner ** -0.5).to(torch.bfloat16)
          for _ in range(8)]
    x = torch.randn(T, d_model, device=dev, generator=gen)
    xo = torch.empty(T, d_model, device=dev, dtype=torch.bfloat16)
    us = graph_us(lambda i, s: ssm_linear(G, Wo[i % 8], [(0, x)], residual=x, stream=s))
    warm = graph_us(lambda i, s: ssm_linear(G, Wo[0], [(0, x)], residual=x, stream=s))
    ref = graph_us(lambda i, s: torch.matmul(G, Wo[i % 8].t(), out=xo))
    by, fl = d_model * d_inner * 2 + T * d_inner * 2 + T * d_model * 8, 2.0 * T * d_model * d_inner
    out["out"] = {"shape_MNK": [T, d_model, d_inner], "us": us, "GB/s": by / us / 1e3, "TFLOP/s": fl / us / 1e6,
                  "frac_of_hbm_peak": by / us / 1e3 / peaks["hbm_gbs"], "us_weights_in_l2": warm,
                  "cublas_matmul_us": ref}
    print(json.dumps({"metric": "projection time (Mamba2-2.7B block, 256 tokens)", "unit": "us",
                      "higher_is_better": False, "data": "synthetic", "projections": out}), flush=True)
    return 0


def draft_step_bytes(H, P, N, n_inst, n_layers):
    """Algorithmic bytes of one ssm_draft_step call: state read + write, the conv window
    (3 ring rows) and the new row, dt, the ring write, the log row, y; params once per layer."""
    d_inner, conv_dim = H * P, H * P + 2 * N
    per = (2 * H * P * N * 4 + 3 * conv_dim * 2 + conv_dim * 2 + H * 2 + conv_dim * 2 + (H + N + d_inner) * 4
           + d_inner * 4 + 8)
    return n_inst * per + n_layers * params_bytes_per_layer(H, P, N)


def replay_bytes(H, P, N, n_inst, k_mean):
    d_inner = H * P
    return n_inst * (2 * H * P * N * 4 + k_mean * (H + N + d_inner) * 4 + 12)


def graph_ms(dev, stream, fn, inner=8, reps=6):
    """Device time of one fn() call: fn is captured `inner` times into one CUDA graph, which
    is replayed `reps` times back to back between two events (launch overhead of the small
    kernels inside is gone, as in a captured decode loop)."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=side):
        for _ in range(inner):
            fn()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * inner)


def run_draft(args, dev, stream, peak, world, rank):
    """Draft rounds on the Mamba2-370M draft workload (48 layers, batch 1 per rank):
    16 chained ssm_draft_step calls (one launch each, all layers batched), then
    ssm_replay of all 16 logged steps.  Device time from CUDA-graph replays (graph_ms):
    "warm" back to back (the 50 MB draft state stays in L2), "cold" with a 256 MB write
    before every call (the state comes from HBM, as after the draft model's other layers),
    the write's own time subtracted."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import Dims, ssm_draft_step, ssm_replay
    from synth import draft_batch, workload
    wd = workload(1)
    seqs = shard_sequences(wd.batch, rank)
    b = draft_batch(wd, seqs=seqs)
    S, L, T = len(seqs), wd.n_layers, wd.draft_steps
    H, P, N = wd.shape.H, wd.shape.P, wd.shape.N
    I = S * L
    dims = Dims(n_heads=H, n_layers=L, ring_cap=wd.ring_cap)
    prm = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev) for k, v in b["params"].items()}
    bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    xs = bf16(b["xBC"]).view(T, I, dims.conv_dim)
    dts = bf16(b["dt"]).view(T, I, H)
    h_ckpt = torch.from_numpy(b["h0"]).to(dev).view(I, H, P, N)
    h_work = torch.empty_like(h_ckpt)
    ring = bf16(b["ring"]).view(I, wd.ring_cap, dims.conv_dim)
    head = torch.from_numpy(b["ring_head"]).to(dev).view(I)
    log_d = torch.zeros(I, T, H, device=dev)
    log_b = torch.zeros(I, T, N, device=dev)
    log_x = torch.zeros(I, T, dims.d_inner, device=dev)
    log_len = torch.zeros(I, dtype=torch.int32, device=dev)
    y = torch.empty(I, dims.d_inner, device=dev)
    # replay every logged step (k = draft_steps): the synthetic accepted position can be 0,
    # which would time bookkeeping only
    k = torch.full((S,), T, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def steps(cold=False):
        for t in range(T):
            if cold:
                flush.fill_(1)
            ssm_draft_step(dims, prm, S, t, T, xs[t], dts[t], h_ckpt if t == 0 else h_work, h_work, ring, head,
                           log_d, log_b, log_x, log_len, y, status)

    def round_(cold=False):
        steps(cold)
        if cold:
            flush.fill_(1)
        ssm_replay(dims, prm, S, T, k, log_d, log_b, log_x, log_len, h_ckpt, head, status)

    for _ in range(args.warmup):
        round_()
    torch.cuda.synchronize()
    res = {}
    t_flush = graph_ms(dev, stream, lambda: flush.fill_(1), inner=8)
    for mode in ("warm", "cold"):
        cold = mode == "cold"
        t_steps = graph_ms(dev, stream, lambda: steps(cold), inner=2) - (t_flush * T if cold else 0.0)
        t_round = graph_ms(dev, stream, lambda: round_(cold), inner=2) - (t_flush * (T + 1) if cold else 0.0)
        res[mode] = (max_over_ranks(t_steps / T, world, dev), max_over_ranks(t_round - t_steps, world, dev))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the draft rounds")
    sb = draft_step_bytes(H, P, N, I, L)
    rb = replay_bytes(H, P, N, I, T)
    out = {"workload": wd.name, "sequences_per_gpu": S, "layers": L, "draft_steps": T, "replay_k": T,
           "unit": "draft token-layer updates/s (value)", "timing": "CUDA-graph replays (device time)"}
    for mode, (step_ms, replay_ms) in res.items():
        out[mode] = {"value": S * L * world / (step_ms / 1e3), "ms_per_draft_step": step_ms, "ms_replay": replay_ms,
                     "draft_step": {"bytes": sb, "GB/s": sb / step_ms / 1e6, "frac_of_hbm_peak": sb / step_ms / 1e6 / peak},
                     "replay": {"bytes": rb, "GB/s": rb / replay_ms / 1e6, "frac_of_hbm_peak": rb / replay_ms / 1e6 / peak}}
    out["note"] = ("warm: calls back to back, the 50 MB draft state in L2 (a fraction above 1 of the HBM peak is "
                   "possible); cold: a 256 MB write before every call, its own time subtracted")
    out.update({"value": out["warm"]["value"], "ms_per_draft_step": out["warm"]["ms_per_draft_step"],
                "ms_replay": out["warm"]["ms_replay"], "draft_step": out["warm"]["draft_step"],
                "replay": out["warm"]["replay"]})
    return out


def draft_tree_level_bytes(H, P, N, n_inst, n_layers, frontier, ancestors):
    """Algorithmic bytes of one ssm_draft_tree_level call: the committed state read once;
    per frontier node its pre-conv row, three tap rows and dt, its log row and y written;
    the log rows (Δ, B, x) of the distinct ancestors on the frontier's paths read; params
    once per layer."""
    d_inner, conv_dim = H * P, H * P + 2 * N
    log_row = (H + N + d_inner) * 4
    per = (H * P * N * 4 + frontier * (4 * conv_dim * 2 + H * 2 + log_row + d_inner * 4) + ancestors * log_row)
    return n_inst * per + n_layers * params_bytes_per_layer(H, P, N)


def draft_tree_commit_bytes(H, P, N, n_inst, path_len):
    """State read + write, the path's log rows, its last three pre-conv rows into the ring."""
    d_inner, conv_dim = H * P, H * P + 2 * N
    rows = min(3, path_len)
    return n_inst * (2 * H * P * N * 4 + path_len * (H + N + d_inner) * 4 + rows * conv_dim * 2 * 2 + 8)


def run_draft_tree(args, dev, stream, peak, world, rank):
    """Draft-side tree drafting on the Mamba2-370M draft shape (48 layers, batch 1 per rank):
    the 16-node random tree (3 branches, depth 4) drafted one depth level per
    ssm_draft_tree_level call, every branch from the one committed state and the log, then
    ssm_draft_tree_commit of the accepted path; and a 16-node chain the same way (one level
    per token: the state is read, never written, until the commit).  Device time from
    CUDA-graph replays: "warm" back to back (the 50 MB draft state stays in L2), "cold" with
    a 256 MB write before every call (between two levels the draft model's other layers
    run), the write's own time subtracted; "cold" is the figure against the HBM roofline."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (Dims, ssm_accept_path, ssm_draft_tree_commit,
                                                   ssm_draft_tree_level, ssm_draft_tree_workspace_size,
                                                   ssm_tree_layout_build)
    from synth import Workload, batch, workload
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    w5 = workload(5)
    chain = Workload(w5.index, "draft chain drafted level by level, Mamba2-370M shape, 48 layers, batch 1, "
                     "16 tokens", w5.shape, n_layers=w5.n_layers, batch=w5.batch, trees=(("chain", 16),))
    t_flush = graph_ms(dev, stream, lambda: flush.fill_(1), inner=8)
    for key, w in (("tree", w5), ("chain", chain)):
        seqs = shard_sequences(w.batch, rank)
        b = batch(w, seqs=seqs)
        S, L, n = len(seqs), w.n_layers, b["n_nodes"]
        H, P, N = w.shape.H, w.shape.P, w.shape.N
        I = S * L
        dims = Dims(n_heads=H, n_layers=L, ring_cap=w.ring_cap)
        layout_h, depth = ssm_tree_layout_build(b["parent"])
        layout = torch.from_numpy(layout_h).to(dev)
        prm = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev) for k, v in b["params"].items()}
        bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
        xBC = bf16(b["xBC"]).view(I, n, dims.conv_dim)
        dt = bf16(b["dt"]).view(I, n, H)
        h = torch.from_numpy(b["h0"]).to(dev).view(I, H, P, N)
        ring = bf16(b["ring"]).view(I, w.ring_cap, dims.conv_dim)
        head = torch.from_numpy(b["ring_head"]).to(dev).view(I)
        log_d = torch.zeros(I, n, H, device=dev)
        log_b = torch.zeros(I, n, N, device=dev)
        log_x = torch.zeros(I, n, dims.d_inner, device=dev)
        y = torch.empty(I, n, dims.d_inner, device=dev)
        ws = torch.empty(ssm_draft_tree_workspace_size(dims, S, n), dtype=torch.uint8, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        max_path = depth + 1
        path = torch.empty(S, max_path, dtype=torch.int32, device=dev)
        plen = torch.empty(S, dtype=torch.int32, device=dev)
        bonus = torch.empty(S, dtype=torch.int32, device=dev)
        if key == "tree":
            ssm_accept_path(S, n, max_path, layout, torch.from_numpy(b["tok"]).to(dev),
                            torch.from_numpy(b["tgt"]).to(dev), path, plen, bonus, status)
        else:  # the whole chain is accepted
            path.copy_(torch.arange(n, dtype=torch.int32, device=dev).expand(S, n))
            plen.fill_(n)
        levels = list(range(depth + 1))

        def level(lv, cold=False):
            if cold:
                flush.fill_(1)
            ssm_draft_tree_level(dims, prm, S, n, lv, layout, xBC, dt, h, ring, head, log_d, log_b, log_x, y, ws,
                                 status)

        def commit(cold=False):
            if cold:
                flush.fill_(1)
            ssm_draft_tree_commit(dims, prm, S, n, layout, max_path, path, plen, log_d, log_b, log_x, xBC, h, ring,
                                  head, status)

        for _ in range(args.warmup):
            for lv in levels:
                level(lv)
        torch.cuda.synchronize()
        res = {}
        for mode in ("warm", "cold"):
            cold = mode == "cold"
            sub = t_flush if cold else 0.0
            lv_ms = [max_over_ranks(graph_ms(dev, stream, lambda lv=lv: level(lv, cold)) - sub, world, dev)
                     for lv in levels]
            # each replayed commit moves the state along the path (the next round's start)
            cm_ms = max_over_ranks(graph_ms(dev, stream, lambda: commit(cold)) - sub, world, dev)
            res[mode] = (lv_ms, cm_ms)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the draft-tree rounds")
        lay = [oracle_free_depths(b["parent"][i]) for i in range(S)]
        plens = plen.cpu().numpy()
        entry = {"workload": w.name, "sequences_per_gpu": S, "layers": L, "nodes": n, "levels": len(levels),
                 "mean_accepted_path": float(plens.mean()), "timing": "CUDA-graph replays (device time)"}
        for mode, (lv_ms, cm_ms) in res.items():
            per_level = []
            tot_b = 0
            for i, lv in enumerate(levels):
                fr = int(np.mean([sum(1 for d in dep if d == lv) for dep in lay]))
                anc = int(np.mean([len(ancestors_at(b["parent"][q], dep, lv)) for q, dep in enumerate(lay)]))
                lb = draft_tree_level_bytes(H, P, N, I, L, fr, anc)
                tot_b += lb
                per_level.append({"level": lv, "nodes": fr, "ms": lv_ms[i], "GB/s": lb / lv_ms[i] / 1e6,
                                  "frac_of_hbm_peak": lb / lv_ms[i] / 1e6 / peak})
            cb = draft_tree_commit_bytes(H, P, N, I, int(round(float(plens.mean()))))
            tree_ms = sum(lv_ms) + cm_ms
            entry[mode] = {"ms_per_tree": tree_ms, "ms_levels": sum(lv_ms), "ms_commit": cm_ms,
                           "levels": per_level,
                           "level_GB/s": tot_b / sum(lv_ms) / 1e6,
                           "level_frac_of_hbm_peak": tot_b / sum(lv_ms) / 1e6 / peak,
                           "commit": {"bytes": cb, "GB/s": cb / cm_ms / 1e6, "frac_of_hbm_peak": cb / cm_ms / 1e6 / peak},
                           "value": S * L * n * world / (tree_ms / 1e3)}
        entry["unit"] = "drafted node-layer updates/s (value)"
        out[key] = entry
        del xBC, dt, h, ring, log_d, log_b, log_x, y, ws
    out["note"] = ("cold: a 256 MB write before every call, its own time subtracted, so the state comes from HBM; "
                   "warm: calls back to back with the 50 MB state in L2")
    return out


def oracle_free_depths(parent):
    """Depth of every node of a breadth-first parent[] (host bookkeeping for the byte counts)."""
    dep = [0] * len(parent)
    for v in range(1, len(parent)):
        dep[v] = dep[int(parent[v])] + 1
    return dep


def ancestors_at(parent, dep, level):
    """Distinct proper ancestors of the nodes of depth `level`."""
    out = set()
    for v in range(len(parent)):
        if dep[v] == level:
            u = int(parent[v])
            while u >= 0:
                out.add(u)
                u = int(parent[u])
    return out


def e2e_chunk_sizes(split, S, chunks=4):
    """Sequences per chunk of an e2e round (S sequences in all).
    'pairs': 1, 1, then 2 at a time: the first chunk lands early, and two compute streams
    fill each other's tails (measured at batch 16: 1.26 ms per round, against 1.26-1.29 for
    2 x 8 or 1 x 8 + 2 x 4, 1.33-1.35 for the ramp or 16 x 1, 1.38 for 4 x 4).
    'ramp': 1, 1, 2, 3, ...: the first chunk lands early, later ones keep up (a small tail
    chunk is folded into the one before).
    A list such as '2,2,4,8': those sizes (positive, summing to S).
    '': `chunks` equal chunks (one chunk when S is not a multiple)."""
    if split == "pairs":
        sizes = [1] * min(S, 2)
        while sum(sizes) < S:
            sizes.append(min(2, S - sum(sizes)))
    elif split == "ramp":
        sizes, nxt = [1], 1
        while sum(sizes) < S:
            sizes.append(min(nxt, S - sum(sizes)))
            nxt += 1
        if len(sizes) > 2 and 2 * sizes[-1] < sizes[-2]:
            tail = sizes.pop()
            sizes[-1] += tail
    elif split:
        sizes = [int(v) for v in split.split(",")]
        if sum(sizes) != S or min(sizes) < 1:
            raise SystemExit(f"--e2e-split must be positive sizes summing to {S}")
    else:
        k = chunks if chunks >= 1 and S % chunks == 0 else 1
        sizes = [S // k] * k
    return sizes


def run_e2e(args, w, b, dims, prm, h, ring, head, ws_f, dev, stream, world):
    """Same rounds through the public API with each round's inputs in pinned host
    memory.  Per round, inside the timed region: the host layout build; the H2D of
    xBC/dt/layout/tokens into one of two device buffers, in four chunks of sequences on
    a copy stream; per chunk, as soon as it has landed, ssm_commit_verify (the previous
    round's path, this round's tree) and ssm_accept_path on the compute stream; then the
    D2H of the accepted paths and bonus tokens and a synchronize."""
    import numpy as np
    import torch

    from speculative_decoding_mamba2_gb300 import (ssm_accept_path, ssm_commit, ssm_commit_verify,
                                                   ssm_tree_layout_build)
    S, L, n = len(b["seqs"]), w.n_layers, w.n_nodes()
    I = S * L
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    xBC_h = pin(b["xBC"].view(np.int16)).view(S, L * n * dims.conv_dim)
    dt_h = pin(b["dt"].view(np.int16)).view(S, L * n * dims.n_heads)
    par_h = np.ascontiguousarray(b["parent"])
    tok_h, tgt_h = pin(b["tok"]), pin(b["tgt"])
    xBC_d = [torch.empty(xBC_h.shape, dtype=torch.int16, device=dev) for _ in range(2)]
    dt_d = [torch.empty(dt_h.shape, dtype=torch.int16, device=dev) for _ in range(2)]
    lay_d = [torch.empty((S, n, 8), dtype=torch.int32, device=dev) for _ in range(2)]
    tok_d = torch.empty(tok_h.shape, dtype=torch.int32, device=dev)
    tgt_d = torch.empty(tgt_h.shape, dtype=torch.int32, device=dev)
    y = torch.empty((S, L * n * dims.d_inner), device=dev)
    hv = h.view(S, -1)
    ringv = ring.view(S, -1)
    headv = head.view(S, L)
    wsv = ws_f.view(S, -1)  # the workspace is per instance, sequence-major
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    steps = max(3, min(args.steps, args.e2e_steps))
    lay0, depth = ssm_tree_layout_build(par_h, max_branches=3, max_depth=4)
    max_path = depth + 1
    path = torch.empty((S, max_path), dtype=torch.int32, device=dev)
    plen = torch.empty(S, dtype=torch.int32, device=dev)
    bonus = torch.empty(S, dtype=torch.int32, device=dev)
    out_path = torch.empty((S, max_path), dtype=torch.int32).pin_memory()  # contiguous: graph-capturable D2H
    out_len = torch.empty(S, dtype=torch.int32).pin_memory()
    out_bonus = torch.empty(S, dtype=torch.int32).pin_memory()
    lay_pin = torch.empty((S, n, 8), dtype=torch.int32).pin_memory()
    copy_stream = torch.cuda.Stream(dev)
    sizes = e2e_chunk_sizes(args.e2e_split, S, args.e2e_chunks)
    bounds = [sum(sizes[:i]) for i in range(len(sizes) + 1)]
    n_chunks = len(sizes)
    state = {"r": 0, "depth": depth}

    computes = [torch.cuda.Stream(dev) for _ in range(max(0, args.e2e_streams - 1))]

    def enqueue(cur, prev, dp, cs):
        """One round's copies and calls: copies on copy_stream, chunk calls alternating between
        compute stream `cs` and a second one (chunks touch disjoint sequences), so one
        chunk's prep kernel overlaps the previous chunk's main kernel."""
        copy_stream.wait_stream(cs)  # the previous round is finished with both buffers
        streams = [cs] + computes
        for x in computes:
            x.wait_stream(cs)
        with torch.cuda.stream(copy_stream):  # the small per-sequence inputs of all chunks first
            lay_d[cur].copy_(lay_pin, non_blocking=True)
            tok_d.copy_(tok_h, non_blocking=True)
            tgt_d.copy_(tgt_h, non_blocking=True)
        for c in range(n_chunks):
            q = slice(bounds[c], bounds[c + 1])
            per = sizes[c]
            ccs = streams[c % len(streams)]
            with torch.cuda.stream(copy_stream):
                xBC_d[cur][q].copy_(xBC_h[q], non_blocking=True)
                dt_d[cur][q].copy_(dt_h[q], non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(copy_stream)
            ccs.wait_event(landed)
            ssm_commit_verify(dims, prm, per, n, lay_d[prev][q], state["depth"] + 1, path[q], plen[q],
                              xBC_d[prev][q].view(torch.bfloat16), dt_d[prev][q].view(torch.bfloat16), n, dp,
                              lay_d[cur][q], xBC_d[cur][q].view(torch.bfloat16), dt_d[cur][q].view(torch.bfloat16),
                              hv[q], ringv[q], headv[q], y[q], wsv[q], status, ccs)
            ssm_accept_path(per, n, dp + 1, lay_d[cur][q], tok_d[q], tgt_d[q], path[q], plen[q], bonus[q], status,
                            ccs)
        cs.wait_stream(copy_stream)
        for x in computes:
            cs.wait_stream(x)
        with torch.cuda.stream(cs):
            out_path.copy_(path, non_blocking=True)
            out_len.copy_(plen, non_blocking=True)
            out_bonus.copy_(bonus, non_blocking=True)

    # With --e2e-graph each round's copies and calls are captured once per buffer parity into a
    # CUDA graph (the tree shape, hence every size and depth, is the same each round) and
    # replayed: the host then only builds the layout, fills the pinned layout buffer and
    # launches one graph per round.
    graphs = {}

    def one():
        cur, prev = (state["r"] + 1) % 2, state["r"] % 2
        state["r"] += 1
        lay, dp = ssm_tree_layout_build(par_h, max_branches=3, max_depth=4)
        lay_pin.numpy()[...] = lay
        if args.e2e_graph:
            if dp != state["depth"]:
                raise RuntimeError("the e2e graph replays one tree shape")
            if cur not in graphs:
                g = torch.cuda.CUDAGraph()
                side = torch.cuda.Stream(dev)
                side.wait_stream(stream)
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=side):
                    enqueue(cur, prev, dp, torch.cuda.current_stream())
                graphs[cur] = g
            with torch.cuda.stream(stream):
                graphs[cur].replay()
        else:
            enqueue(cur, prev, dp, stream)
        state["depth"] = dp
        torch.cuda.synchronize()
        return out_path, out_len, out_bonus

    # the first round needs an accepted path to commit: accept the tree of buffer 0 (the
    # state it would be verified from is the one the device holds)
    lay_d[0].copy_(torch.from_numpy(lay0))
    xBC_d[0].copy_(xBC_h)
    dt_d[0].copy_(dt_h)
    tok_d.copy_(tok_h)
    tgt_d.copy_(tgt_h)
    ssm_accept_path(S, n, max_path, lay_d[0], tok_d, tgt_d, path, plen, bonus, status)
    for _ in range(2):
        one()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    secs = (time.perf_counter() - t0) / steps
    secs = max_over_ranks(secs, world, dev)
    # leave the state committed
    last = state["r"] % 2
    ssm_commit(dims, prm, S, n, lay_d[last], max_path, path, plen, xBC_d[last].view(torch.bfloat16),
               dt_d[last].view(torch.bfloat16), h, ring, head, status)
    torch.cuda.synchronize()
    h2d = xBC_h.numel() * 2 + dt_h.numel() * 2 + S * n * 32 + 2 * S * n * 4
    d2h = S * (max_path + 2) * 4
    return {"value": n * L * S * world / secs, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, "ms_per_step": secs * 1e3,
            "calls": "ssm_tree_layout_build, ssm_commit_verify, ssm_accept_path",
            "overlap": f"H2D in {n_chunks} chunks of {sizes} sequences on a copy stream; each chunk's calls start when "
                       f"its inputs have landed, alternating over {args.e2e_streams} compute stream(s)"
                       + ("; each round replayed as one CUDA graph" if args.e2e_graph else "")}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=[2, 3])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-chunks", type=int, default=4, help="equal sequence chunks of the e2e round (with --e2e-split '')")
    ap.add_argument("--e2e-graph", type=int, default=1, help="replay each e2e round as a CUDA graph (1) or enqueue it (0)")
    ap.add_argument("--e2e-streams", type=int, default=2, help="compute streams the e2e chunk calls alternate over")
    ap.add_argument("--e2e-split", default="pairs",
                    help="e2e chunk sizes in sequences: 'pairs' (1, 1, 2, 2, ...), 'ramp' (1, 1, 2, 3, ...), "
                         "a list such as '4,4,4,4', "
                         "or '' for --e2e-chunks equal chunks")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-draft", action="store_true")
    ap.add_argument("--no-chain", action="store_true", help="with --no-config4: skip the chain sample too")
    ap.add_argument("--no-config2", action="store_true", help="skip the batch-1 target verify workload")
    ap.add_argument("--no-config4", action="store_true", help="skip the stress workload (batch 64)")
    ap.add_argument("--no-block", action="store_true")
    ap.add_argument("--only", choices=["linear", "draft", "block-steps", "ternary"], default=None,
                    help="run one measurement alone: 'linear' = the block's projections, "
                         "'draft' = the draft side (one-token steps + replay, tree drafting), "
                         "'block-steps' = one block's steps timed one by one, "
                         "'ternary' = the stress workload's ternary tree (see --seqs)")
    ap.add_argument("--seqs", type=int, default=64, help="with --only ternary: sequences of the stress workload")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from synth import workload
    w = workload(args.workload)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.only == "linear":
        return run_linear_only(args)
    if args.only == "draft":
        return run_draft_only(args)
    if args.only == "block-steps":
        return run_block_steps(args)
    if args.only == "ternary":
        return run_ternary_only(args)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
