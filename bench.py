#!/usr/bin/env python
"""DSA layer benchmark on GB300: tokens/s of one layer step (indexer + top-k,
sparse attention forward and backward) at S = 131072, with the indexer's
TFLOP/s and the attention kernels' GB/s against the measured peaks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path over one synthetic sequence:
dsa_index_topk (32 indexer heads x 64, top 512 pools, query chunk 256; one
persistent kernel),
dsa_sparse_attn_fwd and dsa_sparse_attn_bwd (16 query heads sharing one KV
head of dim 128).  Inputs are seeded bf16 N(0,1) (indexer queries x 1/8,
head weights U(0,1)), resident in HBM before timing.  L2 is flushed (512 MiB
write) between timed steps, outside the timed events.  Under torchrun each
rank runs its own sequence (weak scaling, no collective on the data path).

`--impl reference` times the CPU oracle on the host cores on bounded samples
of the same workload (there is no other reference implementation).
"""
from __future__ import annotations

import argparse
import ctypes
import gc
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA layer fwd+bwd tokens/s at S=128k; indexer TFLOP/s & attn GB/s vs peak"
UNIT = "tokens/s"


def metric_for(wl):
    """The headline metric for the fwd+bwd workloads; the forward-only workloads
    (planted-cluster keys at S = 262144 and 1048576, S = 16384) report the
    forward pass: indexer + top-k + sparse attention forward."""
    if wl.backward:
        return METRIC
    return (f"DSA layer fwd tokens/s at S={wl.S} (indexer+top-k+sparse attn fwd); "
            "indexer TFLOP/s & attn GB/s vs peak")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="s128k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="backward through dsa_sparse_attn_bwd_deterministic (bit-reproducible dK/dV)")
    ap.add_argument("--varlen", type=int, default=0, metavar="N",
                    help="time the S tokens as N packed sequences of a seeded length mix (varlen calls)")
    ap.add_argument("--zigzag", type=int, default=0, metavar="N",
                    help="time the N zig-zag query shards of the sequence one after another (range calls)")
    ap.add_argument("--trace", action="store_true",
                    help="indexer item trace: one dsa_index_topk call through the DSA_ITEM_TRACE build, "
                         "time per work-item kind (fold, dependency wait, rest) and per-CTA idle time")
    ap.add_argument("--trace-stamps", action="store_true",
                    help="the same item trace through the stamps-only build (no SM-cycle counters in the "
                         "indexer's fold), whose per-item times are the default build's")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-tc-alt", action="store_true",
                    help="skip timing the tcgen05 forward alternative after the step")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target oracle time for the CPU baseline sample")
    return ap.parse_args()


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x: the slowest rank sets the job's time."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- workload accounting

def workload_counts(wl):
    """Exact per-step unit counts: indexer (query, pool) pairs and attended (query, key) pairs."""
    i = np.arange(wl.S, dtype=np.int64)
    n = i // 4
    pairs = int(n.sum())
    keys = int((4 * np.minimum(n, wl.topk) + (i % 4) + 1).sum())
    return pairs, keys


def algorithmic_work(wl):
    """Algorithmic flops / bytes per step of each kernel (see the design notes)."""
    pairs, keys = workload_counts(wl)
    S, Hq, D, k = wl.S, wl.Hq, wl.D, wl.topk
    row_kv = 2 * D * 2                     # one K row + one V row, bf16
    q_bytes = Hq * D * 2                   # one query's q (or o, dO, dq)
    return {
        # the fused indexer + top-k kernel: the indexer contraction's flops
        # (its scores also cross L2 once more for the top-k: 4 B per pair)
        "index_topk": {"flops": 2 * wl.Hi * wl.Di * pairs, "topk_bytes": 4 * pairs + 4 * S * k},
        "attn_fwd": {"bytes": keys * row_kv + S * (2 * q_bytes + 4 * Hq + 4 * k)},
        # gather K,V + read q, dO, lse, Delta, idx + write dq + fp32 dK/dV reductions (2 x 512 B per key)
        "attn_bwd": {"bytes": keys * row_kv + S * (3 * q_bytes + 8 * Hq + 4 * k) + keys * 2 * D * 4},
        # deterministic backward's span kernel: q and dO per (query, pool) pair, own partial pool included
        "det_span": {"bytes": (int(np.minimum(np.arange(S, dtype=np.int64) // 4, k).sum()) + S) * 2 * q_bytes},
        "pairs": pairs, "keys": keys,
    }


# the files holding each kernel's device code (a capture goes stale when any changes)
KERNEL_SOURCE = {"index_topk": ("index_topk.cu", "topk_row.cuh", "topk_warp.cuh", "topk_cand.cuh", "dsa_kernels.h"),
                 "attn_fwd": ("attn_fwd.cu", "dsa_kernels.h"), "attn_bwd": ("attn_bwd.cu", "dsa_kernels.h"),
                 "det_span": ("attn_bwd_det.cu",)}
# profile summary file stem of a timed launcher whose kernel has another name
PROFILE_STEM = {"det_span": "det_item"}


def profiled_traffic(kernel, S):
    """DRAM bytes per launch from the committed ncu summary under profiles/, only
    while the kernel source still hashes to the one that was captured."""
    srcs = KERNEL_SOURCE.get(kernel)
    if srcs is None:
        return None, "no capture for this kernel"
    sha = hashlib.sha256()
    for name in srcs:
        with open(os.path.join(ROOT, "long_context_sparse_index_gb300", "csrc", name), "rb") as f:
            sha.update(f.read())
    h = sha.hexdigest()[:16]
    src = " + ".join(srcs)
    stem = PROFILE_STEM.get(kernel, kernel)
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", f"{stem}_kernel_*.md"))):
        with open(path) as f:
            text = f.read()
        m = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
        t = re.search(rf"traffic_bytes_per_launch_S{S}:\s*(\d+)", text)
        if m and t:
            if m.group(1) == h:
                return int(t.group(1)), os.path.basename(path)
            return None, f"{os.path.basename(path)} was captured on an older {src}"
        if m:
            return None, f"{os.path.basename(path)} gives no DRAM traffic for S={S}"
    return None, "no capture for this kernel"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self.gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for_smi(torch, dev_index):
    try:
        uuid = str(torch.cuda.get_device_properties(dev_index).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[dev_index]
        return str(dev_index)


# ----------------------------------------------------------------------------- CPU baseline (oracle)

def oracle_sample_step(wl, host, rows):
    """Oracle work for a sample of query rows: indexer + top-k, forward, backward."""
    import oracle
    q_idx, k_idx, w, q, k, v, dO = host
    sel, _ = oracle.index_topk(q_idx, k_idx, w, wl.topk, rows=rows)
    full = np.full((wl.S, wl.topk), -1, np.int32)
    full[rows] = sel
    oracle.attn_fwd(q, k, v, full, scale=wl.scale, rows=rows)
    if wl.backward:
        oracle.attn_bwd_rows(dO, q, k, v, full, scale=wl.scale, rows=rows)


def cpu_baseline(wl, host, seconds, seed=12345):
    import oracle
    rs = np.random.RandomState(seed)
    probe = np.sort(rs.randint(0, wl.S, 16))
    t0 = time.perf_counter()
    oracle_sample_step(wl, host, probe)
    per_row = (time.perf_counter() - t0) / probe.size
    n = int(max(16, min(4096, seconds / max(per_row, 1e-6))))
    rows = np.sort(rs.randint(0, wl.S, n))
    t0 = time.perf_counter()
    oracle_sample_step(wl, host, rows)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} query rows drawn uniformly from the S={wl.S} sequence (seed {seed}); each row: indexer "
                      f"scores over its floor(i/4) pools + top-{wl.topk} by full sort, "
                      f"{'forward and backward' if wl.backward else 'forward'} over its "
                      f"key set; tokens/s = rows / oracle seconds ({dt:.1f} s)"}


def host_inputs(wl):
    import synth
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    q, k, v = synth.attention_inputs(wl)
    dO = synth.grad_output(wl) if wl.backward else None
    return q_idx, k_idx, w, q, k, v, dO


def workload_config(wl, l2_note):
    name = f"dsa_layer_fwd_bwd_S{wl.S}" if wl.backward else f"dsa_layer_fwd_S{wl.S}_{wl.values}"
    return {"workload": name, "S": wl.S, "batch": 1, "indexer_heads": wl.Hi,
            "indexer_dim": wl.Di, "pool_size": 4, "topk_pools": wl.topk, "query_chunk": wl.chunk,
            "q_heads": wl.Hq, "kv_heads": 1, "head_dim": wl.D, "max_keys_per_query": 4 * wl.topk + 4,
            "inputs": ("seeded bf16 N(0,1); indexer queries x %g; head weights U(0,1) fp32" % wl.q_idx_scale) +
                      ("; indexer keys with 8 planted clusters (1/16 of pools)" if wl.values == "cluster" else "") +
                      ("; Zipf-ranked pool magnitudes" if wl.values == "zipf" else ""),
            "l2": l2_note}


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    wl = synth.WORKLOADS[args.workload]
    host = host_inputs(wl)
    rs = np.random.RandomState(777)
    rows_per_step = 24
    for _ in range(args.warmup):
        oracle_sample_step(wl, host, np.sort(rs.randint(0, wl.S, rows_per_step)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(wl, host, np.sort(rs.randint(0, wl.S, rows_per_step)))
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps / dt
    sample = (f"{rows_per_step} query rows per step drawn uniformly from the S={wl.S} sequence; each row: indexer + "
              f"top-{wl.topk}, {'forward and backward' if wl.backward else 'forward'} over its key set; "
              f"tokens/s = rows / oracle seconds")
    line = {"impl": "reference", "metric": metric_for(wl), "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, "n/a (CPU)"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm

def measure_l2_peaks(dsa, torch, dev):
    """L2 rates of the attention kernels' access shapes, on a 64 MiB buffer
    (L2-resident): streaming reads, random 1 KB pool gathers, 16-byte fp32
    vector reductions four rows x 128 B per warp instruction (the backward's
    shape; also 2 x 256 B, 8 x 64 B and 16 x 32 B), bulk fp32 reductions from
    shared memory (2 KB and 512 B operations), and vector and bulk
    reductions issued together."""
    buf = torch.zeros(64 << 20, dtype=torch.uint8, device=dev)
    out = {"buffer_mib": 64}
    for kind, name in ((0, "stream_read_gbs"), (1, "gather_1kb_gbs"), (2, "red_v4_gbs"), (3, "bulk_red_2kb_gbs"),
                       (4, "bulk_red_512b_gbs"), (5, "red_v4_2x256b_gbs"), (6, "red_v4_8x64b_gbs"),
                       (7, "red_v4_16x32b_gbs"), (8, "red_v4_with_bulk_gbs")):
        out[name] = max(dsa.measure_l2(kind, buf, iters=20) for _ in range(3))
    del buf
    return out


def measure_umma_costs(dsa):
    """Cycles per tcgen05.mma (M 128, K 16, bf16) seen by the issuing thread:
    N = 16 is the attention's product shape (one column per query head)."""
    out = {}
    for n, issuers in ((16, 1), (16, 3), (64, 1), (128, 1), (256, 1)):
        out[f"n{n}_issuers{issuers}"] = round(dsa.measure_umma(n, issuers, groups=2000), 1)
    out["nominal_cycles_n16"] = 128 * 16 * 16 / 4096  # dense bf16: 8192 flop per SM per clock
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import synth
    import long_context_sparse_index_gb300 as dsa
    from long_context_sparse_index_gb300 import build as libbuild

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    libbuild.build()
    wl = synth.WORKLOADS[args.workload]
    backward = wl.backward
    peaks = load_peaks()
    l2 = measure_l2_peaks(dsa, torch, dev)

    host = host_inputs(wl)
    q_idx_h, k_idx_h, w_h, q_h, k_h, v_h, dO_h = host

    def pinned_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()

    pin = {"q_idx": pinned_bf16(q_idx_h), "k_idx": pinned_bf16(k_idx_h), "w": torch.from_numpy(w_h).pin_memory(),
           "q": pinned_bf16(q_h), "k": pinned_bf16(k_h), "v": pinned_bf16(v_h)}
    if backward:
        pin["dO"] = pinned_bf16(dO_h)
    del host, q_idx_h, q_h, dO_h

    def host_view(name):
        t = pin[name]
        return t.numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy().view(np.uint16)
    d = {name: t.to(dev) for name, t in pin.items()}
    S, topk = wl.S, wl.topk
    pool_idx = torch.empty((S, topk), dtype=torch.int32, device=dev)
    o = torch.empty_like(d["q"])
    lse = torch.empty((S, wl.Hq), dtype=torch.float32, device=dev)
    ws_idx = torch.empty(dsa.index_topk_workspace_size(S, wl.Hi, wl.Di, wl.chunk, topk), dtype=torch.uint8,
                         device=dev)
    if backward:
        dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
        if args.deterministic:
            bwd = dsa.dsa_sparse_attn_bwd_deterministic
            ws_bwd_bytes = dsa.sparse_attn_bwd_deterministic_workspace_size(S, wl.Hq, wl.D, topk)
        else:
            bwd = dsa.dsa_sparse_attn_bwd
            ws_bwd_bytes = dsa.sparse_attn_bwd_workspace_size(S, wl.Hq, wl.D)
        ws_bwd = torch.empty(ws_bwd_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(t):
        dsa.dsa_index_topk(t["q_idx"], t["k_idx"], t["w"], chunk=wl.chunk, topk=topk, pool_idx=pool_idx,
                           workspace=ws_idx)
        dsa.dsa_sparse_attn_fwd(t["q"], t["k"], t["v"], pool_idx, scale=wl.scale, o=o, lse=lse)
        if backward:
            bwd(t["dO"], t["q"], t["k"], t["v"], o, lse, pool_idx, scale=wl.scale, dq=dq, dk=dk, dv=dv,
                workspace=ws_bwd)

    for _ in range(args.warmup):
        flush.zero_()
        step(d)
    dsa.dsa_sync_status()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region: K steps, device events per step, L2 flush outside the events
    sampler = ClockSampler(gpu_id_for_smi(torch, local_rank))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    dsa.launch_count_reset()
    gc.collect()
    gc.disable()  # no collector pause inside a step's launches
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for s in range(args.steps):
        flush.zero_()
        evs[s][0].record(stream)
        step(d)
        evs[s][1].record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    gc.enable()
    clocks = sampler.stop()
    gpu_launches = dsa.launch_count()
    dsa.dsa_sync_status()
    index_stats = dsa.index_topk_stats(ws_idx)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_s = sum(step_ms) / 1e3
    total_s = max_over_ranks(total_s, dev)
    value = world * S * args.steps / total_s

    # ---- per-kernel device time, live, with events around every launch (one more step)
    flush.zero_()
    torch.cuda.synchronize()
    dsa.profile_enable(True)
    step(d)
    dsa.profile_enable(False)
    prof = dsa.profile_read()
    work = algorithmic_work(wl)
    kernels = {}
    for name, (ms, launches) in prof.items():
        entry = {"ms": ms, "launches": launches}
        if name == "index_topk":
            tf = work["index_topk"]["flops"] / (ms * 1e-3) / 1e12
            entry.update({"algorithmic_tflops": tf, "frac_of_bf16_sustained": tf / peaks["bf16_tflops_sustained"],
                          "executed_tensor_flops_factor": 2.0, "includes": "indexer tiles and top-k rows"})
            traffic, tsrc = profiled_traffic("index_topk", S)
            entry.update({"dram_bytes_per_launch": traffic, "dram_bytes_source": tsrc})
        elif name in ("attn_fwd", "attn_bwd", "det_span"):
            gbs = work[name]["bytes"] / (ms * 1e-3) / 1e9
            entry.update({"algorithmic_gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"]})
            if name == "attn_fwd":
                # the gather and the per-query streams read through L2 (K/V is L2-resident up to S ~ 2^17)
                entry["frac_of_l2_gather"] = gbs / l2["gather_1kb_gbs"]
            if name == "attn_bwd":
                red = work["keys"] * 2 * wl.D * 4 / (ms * 1e-3) / 1e9
                entry.update({"reduction_gbs": red, "frac_of_l2_red": red / l2["red_v4_gbs"]})
        kernels[name] = entry
    if "index_topk" in kernels:
        # the tile loop's handoff measured alone (same warp layout and register cap)
        kernels["index_topk"]["fold_probe_cycles_per_head"] = {
            "loads_and_fold": round(dsa.measure_fold(1), 1), "loads_only": round(dsa.measure_fold(0), 1),
            "tmem_ld32": round(dsa.measure_fold(2), 1), "mma_chain_nominal": 1024}
    dom = max(prof.items(), key=lambda kv: kv[1][0])[0]
    dms, dl = prof[dom]
    if dom == "index_topk":
        ach = work["index_topk"]["flops"] / (dms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops_sustained"], "traffic": None}
    else:
        ach = work.get(dom, {"bytes": 0})["bytes"] / (dms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": None}
    traffic, tsrc = profiled_traffic(dom, S)
    roof["traffic"] = traffic
    roof["traffic_source"] = tsrc
    roof.update({"kernel": dom, "launches_per_step": dl, "avg_launch_ms": dms / max(dl, 1),
                 "peak_source": peaks["source"] + (" (sustained bf16)" if dom == "index_topk" else " (copy bandwidth)")})
    if dom in kernels:
        for key in ("frac_of_l2_red", "reduction_gbs", "frac_of_l2_gather"):
            if key in kernels[dom]:
                roof[key] = kernels[dom][key]
    roof["l2_peaks_measured"] = l2

    # ---- the tcgen05 forward (dsa_sparse_attn_fwd_tc) on the same selection,
    # timed alone after the step (not part of it): the measured tensor-core
    # alternative to attn_fwd, and the cost of one N = 16 tensor-core product
    tc_alt = None
    if not args.no_tc_alt:
        o_tc, lse_tc = torch.empty_like(o), torch.empty_like(lse)
        tms = []
        for _ in range(3):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dsa.dsa_sparse_attn_fwd_tc(d["q"], d["k"], d["v"], pool_idx, scale=wl.scale, o=o_tc, lse=lse_tc)
            b.record(stream)
            torch.cuda.synchronize()
            tms.append(a.elapsed_time(b))
        dsa.dsa_sparse_attn_fwd(d["q"], d["k"], d["v"], pool_idx, scale=wl.scale, o=o, lse=lse)
        dsa.dsa_sync_status()
        tc_alt = {"ms": min(tms), "attn_fwd_ms": kernels.get("attn_fwd", {}).get("ms"),
                  "max_abs_o_diff_vs_attn_fwd": (o_tc.float() - o.float()).abs().max().item(),
                  "max_abs_lse_diff_vs_attn_fwd": (lse_tc - lse).abs().max().item(),
                  "umma_cycles_per_instruction": measure_umma_costs(dsa)}

    # ---- end to end through the public API: pinned host -> device, the calls, device -> host
    e2e = None
    if not args.no_e2e:
        # Three device sets of inputs and outputs, used by steps in turn, the
        # way a training loop with prefetch runs: step s+2's inputs upload into
        # their set while steps s and s+1 compute (once step s-1 is done with
        # that set), pool_idx, o and lse download during the backward, and dq,
        # dk and dv during the next steps (the last step's before the end
        # event).  Every copy is inside the timed region, on its own stream per
        # direction; step 0's indexer inputs upload first, so its indexer
        # starts while the rest of its inputs upload.
        small_names = ("pool_idx", "o", "lse")
        grad_names = ("dq", "dk", "dv") if backward else ()
        outs0 = {"pool_idx": pool_idx, "o": o, "lse": lse}
        if backward:
            outs0.update({"dq": dq, "dk": dk, "dv": dv})
        nsets = 3
        sets = [(d, outs0)] + [({n: torch.empty_like(t) for n, t in d.items()},
                                {n: torch.empty_like(t) for n, t in outs0.items()}) for _ in range(nsets - 1)]
        out_host = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in outs0.items()}
        bi = sum(t.numel() * t.element_size() for t in pin.values())
        bo = sum(t.numel() * t.element_size() for t in out_host.values())
        h2d = torch.cuda.Stream(device=dev)
        d2h = torch.cuda.Stream(device=dev)
        idx_in = ("q_idx", "k_idx", "w")
        attn_in = ("q", "k", "v", "dO") if backward else ("q", "k", "v")

        def upload(dst, names):
            with torch.cuda.stream(h2d):
                for name in names:
                    dst[name].copy_(pin[name], non_blocking=True)
            return h2d.record_event()

        def download(src, names):
            with torch.cuda.stream(d2h):
                for name in names:
                    out_host[name].copy_(src[name], non_blocking=True)
            return d2h.record_event()

        def e2e_run(nsteps, start=None, marks=None):
            if nsteps == 0:
                return
            if start is not None:
                start.record(stream)
            h2d.wait_stream(stream)
            d2h.wait_stream(stream)
            ev_idx_in = [None] * nsteps
            ev_attn_in = [None] * nsteps
            ev_idx_in[0] = upload(sets[0][0], idx_in)
            ev_attn_in[0] = upload(sets[0][0], attn_in)
            for j in range(1, min(nsets - 1, nsteps)):  # the next steps' sets are free from the start
                ev_idx_in[j] = ev_attn_in[j] = upload(sets[j][0], idx_in + attn_in)
            ev_done, ev_out = [None] * nsteps, [None] * nsteps
            for s in range(nsteps):
                t, out = sets[s % nsets]
                nxt = s + nsets - 1
                if nxt < nsteps:
                    if s >= 1:
                        h2d.wait_event(ev_done[s - 1])  # step s-1 is done with the set of step s+2
                    ev_idx_in[nxt] = ev_attn_in[nxt] = upload(sets[nxt % nsets][0], idx_in + attn_in)
                flush.zero_()
                stream.wait_event(ev_idx_in[s])
                if s >= nsets:
                    stream.wait_event(ev_out[s - nsets])  # this set's outputs of step s-3 are on the host
                dsa.dsa_index_topk(t["q_idx"], t["k_idx"], t["w"], chunk=wl.chunk, topk=topk,
                                   pool_idx=out["pool_idx"], workspace=ws_idx)
                stream.wait_event(ev_attn_in[s])
                dsa.dsa_sparse_attn_fwd(t["q"], t["k"], t["v"], out["pool_idx"], scale=wl.scale, o=out["o"],
                                        lse=out["lse"])
                d2h.wait_stream(stream)
                ev_out[s] = download(out, small_names)
                if backward:
                    bwd(t["dO"], t["q"], t["k"], t["v"], out["o"], out["lse"], out["pool_idx"], scale=wl.scale,
                        dq=out["dq"], dk=out["dk"], dv=out["dv"], workspace=ws_bwd)
                ev_done[s] = stream.record_event()
                if backward:
                    d2h.wait_event(ev_done[s])
                    ev_out[s] = download(out, grad_names)
                if marks is not None:
                    marks[s].record(stream)
            stream.wait_stream(d2h)
            stream.wait_stream(h2d)

        e2e_run(args.warmup)  # untimed, like the device loop's warm-up
        barrier()
        # the host enqueues the whole pipelined loop ahead of the device; keep
        # the collector from pausing it mid-way (a training loop does the same)
        gc.collect()
        gc.disable()
        e2e_start, e2e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e2e_run(args.steps, e2e_start, marks)
        e2e_end.record(stream)
        barrier()
        gc.enable()
        e2e_s = e2e_start.elapsed_time(e2e_end) / 1e3
        e2e_s = max_over_ranks(e2e_s, dev)
        bounds = [e2e_start] + marks
        e2e = {"value": world * S * args.steps / e2e_s, "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": 1e3 * e2e_s / args.steps,
               "step_ms": [a.elapsed_time(b) for a, b in zip(bounds[:-1], bounds[1:])],
               "last_step_tail_ms": marks[-1].elapsed_time(e2e_end),
               "pipelining": "three device sets of inputs and outputs used by steps in turn: inputs upload two steps "
                             "ahead, pool_idx/o/lse download during the backward and dq/dk/dv during the next steps; "
                             "all copies inside the timed region"}

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(wl, tuple(host_view(n) if n in pin else None
                                         for n in ("q_idx", "k_idx", "w", "q", "k", "v", "dO")), args.cpu_seconds)
        line = {"metric": metric_for(wl), "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": workload_config(wl, "flushed between timed steps (512 MiB write outside the events)"),
                "parallelism": f"replicas x{world} (one independent sequence per GPU)",
                "clocks": clocks, "gpu_launches": gpu_launches, "e2e": e2e, "roofline": roof,
                "kernels": kernels, "index_topk_stats": index_stats, "cpu_baseline": cpu,
                "wall_s_timed_region": wall, "step_ms": step_ms, "attn_fwd_tcgen05": tc_alt}
        if backward:
            line["backward"] = "deterministic (key-major, fixed order)" if args.deterministic else "atomic dK/dV"
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- packed batches and shards

def varlen_lengths(S, n, seed=7):
    """A seeded mix of n sequence lengths (multiples of 256) summing to S."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, S // 256), size=n - 1, replace=False)) * 256
    return np.diff(np.concatenate([[0], cuts, [S]])).astype(np.int64)


def run_layout(args):
    """--varlen N: the workload's S tokens as N packed sequences (cu_seqlens),
    through the varlen calls.  --zigzag N: the N zig-zag query shards of the
    one sequence, each through the range calls, one after another on this GPU
    (what each of N ranks would run, before the all-gather of pool indices and
    the reduce-scatter of dK/dV that the caller adds).  Both time the device
    with CUDA events, inputs resident, L2 flushed between steps."""
    import torch
    import synth
    import long_context_sparse_index_gb300 as dsa
    from long_context_sparse_index_gb300 import build as libbuild

    libbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS[args.workload]
    S, topk = wl.S, wl.topk
    q_idx_h, k_idx_h, w_h, q_h, k_h, v_h, dO_h = host_inputs(wl)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    q_idx, k_idx, q, k, v, dO = (bf16(a) for a in (q_idx_h, k_idx_h, q_h, k_h, v_h, dO_h))
    w = torch.from_numpy(w_h).to(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    lib = dsa.load()
    extra = {}
    if args.varlen:
        lens = varlen_lengths(S, args.varlen)
        cu = [0] + np.cumsum(lens).tolist()
        cu_c = (ctypes.c_int64 * len(cu))(*cu)
        ws_i = torch.empty(max(256, lib.dsa_index_topk_varlen_workspace(cu_c, args.varlen, wl.Hi, wl.Di, wl.chunk, topk)),
                           dtype=torch.uint8, device=dev)
        ws_b = torch.empty(max(256, lib.dsa_sparse_attn_bwd_varlen_workspace(cu_c, args.varlen, wl.Hq, wl.D)),
                           dtype=torch.uint8, device=dev)
        pool_idx = torch.empty((S, topk), dtype=torch.int32, device=dev)
        o, lse = torch.empty_like(q), torch.empty((S, wl.Hq), dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

        def parts():
            def run():
                dsa.dsa_index_topk_varlen(q_idx, k_idx, w, cu, chunk=wl.chunk, topk=topk, pool_idx=pool_idx,
                                          workspace=ws_i)
                dsa.dsa_sparse_attn_fwd_varlen(q, k, v, pool_idx, cu, scale=wl.scale, o=o, lse=lse)
                dsa.dsa_sparse_attn_bwd_varlen(dO, q, k, v, o, lse, pool_idx, cu, scale=wl.scale, dq=dq, dk=dk, dv=dv,
                                               workspace=ws_b)
            return [run]
        workload = f"dsa_layer_fwd_bwd_varlen{args.varlen}_T{S}"
        extra["seq_lens"] = lens.tolist()
    else:
        n = args.zigzag
        ws_i = torch.empty(dsa.index_topk_workspace_size(S, wl.Hi, wl.Di, wl.chunk, topk), dtype=torch.uint8,
                           device=dev)
        ws_b = torch.empty(dsa.sparse_attn_bwd_workspace_size(S, wl.Hq, wl.D), dtype=torch.uint8, device=dev)
        pool_idx = torch.empty((S, topk), dtype=torch.int32, device=dev)
        o, lse = torch.empty_like(q), torch.empty((S, wl.Hq), dtype=torch.float32, device=dev)
        dq = torch.empty_like(q)
        dks = [(torch.empty_like(k), torch.empty_like(v)) for _ in range(2)]

        def rank_step(r):
            def run():
                for j, (b, e) in enumerate(dsa.zigzag_ranges(S, n, r)):
                    if e <= b:
                        continue
                    sel = pool_idx[b:e]
                    dsa.dsa_index_topk(q_idx, k_idx, w, chunk=wl.chunk, topk=topk, q_begin=b, q_end=e, pool_idx=sel,
                                       workspace=ws_i)
                    dsa.dsa_sparse_attn_fwd(q[b:e], k, v, sel, scale=wl.scale, o=o[b:e], lse=lse[b:e], q_begin=b)
                    dsa.dsa_sparse_attn_bwd(dO[b:e], q[b:e], k, v, o[b:e], lse[b:e], sel, scale=wl.scale, dq=dq[b:e],
                                            dk=dks[j][0], dv=dks[j][1], workspace=ws_b, q_begin=b)
            return run

        def parts():
            return [rank_step(r) for r in range(n)]
        workload = f"dsa_layer_fwd_bwd_zigzag{n}_S{S}"
        extra["ranges"] = [dsa.zigzag_ranges(S, n, r) for r in range(n)]

    fns = parts()
    for _ in range(args.warmup):
        flush.zero_()
        for f in fns:
            f()
    dsa.dsa_sync_status()
    torch.cuda.synchronize()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in fns]
           for _ in range(args.steps)]
    dsa.launch_count_reset()
    for st in range(args.steps):
        flush.zero_()
        for f, (a, b) in zip(fns, evs[st]):
            a.record(stream)
            f()
            b.record(stream)
    torch.cuda.synchronize()
    launches = dsa.launch_count()
    dsa.dsa_sync_status()
    part_ms = np.array([[a.elapsed_time(b) for a, b in row] for row in evs]).mean(0)
    total_ms = float(part_ms.sum())
    line = {"metric": METRIC, "value": S / (total_ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(wl, "flushed between timed steps (512 MiB write outside the events)"),
                           workload=workload),
            "gpu_launches": launches, "e2e": None}
    if args.zigzag:
        line["rank_ms"] = part_ms.tolist()
        line["rank_balance_max_over_mean"] = float(part_ms.max() / part_ms.mean())
        line["note"] = ("value = S / (sum of the N shards' times): the N shards run back to back on one GPU; "
                        "N ranks would each take one rank_ms, plus the caller's collectives")
    line.update(extra)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- indexer item trace

TRACE_KINDS = ("sample", "thresh", "tile", "rows")


def summarize_trace(rec, num_sms):
    """Per-kind and per-CTA time from the item records (see dsa_trace_configure)."""
    kind = rec["kind_sm"] & 0xFF
    sm = rec["kind_sm"] >> 8
    t0, t1, t2, t3 = (rec[f].astype(np.int64) for f in ("t0", "t1", "t2", "t3"))
    start, end = int(t0.min()), int(t3.max())
    out = {"records": int(rec.size), "span_ms": (end - start) / 1e6, "ctas": int(np.unique(sm).size), "kinds": {}}
    ctas = max(out["ctas"], 1)
    for k, name in enumerate(TRACE_KINDS):
        m = kind == k
        if not m.any():
            continue
        out["kinds"][name] = {
            "items": int(m.sum()),
            "fold_ms_per_cta": float((t1[m] - t0[m]).sum()) / 1e6 / ctas,
            "wait_ms_per_cta": float((t2[m] - t1[m]).sum()) / 1e6 / ctas,
            "rest_ms_per_cta": float((t3[m] - t2[m]).sum()) / 1e6 / ctas,
            "mean_us": float((t3[m] - t0[m]).mean()) / 1e3,
        }
    # time between one item's end and the next item's start on the same SM,
    # plus the lead before an SM's first item and the tail after its last
    gaps = 0
    for s_ in np.unique(sm):
        m = sm == s_
        a, b = np.sort(t0[m]), np.sort(t3[m])
        gaps += int(np.clip(a[1:] - b[:-1], 0, None).sum()) + int(a[0] - start) + int(end - b[-1])
    out["between_items_ms_per_cta"] = gaps / 1e6 / ctas
    return out


def run_trace(args, stamps=False):
    import torch
    import synth
    from long_context_sparse_index_gb300 import build as libbuild

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    path = libbuild.build(stamps=True) if stamps else libbuild.build(trace=True)
    lib = ctypes.CDLL(path)
    i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    lib.dsa_index_topk_workspace.argtypes = [i64, i32, i32, i32, i32]
    lib.dsa_index_topk_workspace.restype = sz
    lib.dsa_index_topk.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, i64, i64, vp, vp, sz, vp]
    lib.dsa_trace_configure.argtypes = [vp, sz]
    lib.dsa_sync_status.argtypes = [vp]
    lib.dsa_last_error.restype = ctypes.c_char_p
    wl = synth.WORKLOADS[args.workload]
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, wt = to(q_idx), to(k_idx), torch.from_numpy(w).to(dev)
    del q_idx
    S = wl.S
    out = torch.empty((S, wl.topk), dtype=torch.int32, device=dev)
    ws = torch.empty(lib.dsa_index_topk_workspace(S, wl.Hi, wl.Di, wl.chunk, wl.topk), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        rc = lib.dsa_index_topk(q.data_ptr(), k.data_ptr(), wt.data_ptr(), S, wl.Hi, wl.Di, wl.chunk, wl.topk, 0, S,
                                out.data_ptr(), ws.data_ptr(), ws.numel(), stream)
        if rc != 0:
            raise RuntimeError(lib.dsa_last_error().decode())

    for _ in range(max(1, args.warmup)):
        call()
    rec_dtype = np.dtype([("kind_sm", np.uint32), ("chunk", np.uint32), ("t0", np.uint64), ("t1", np.uint64),
                          ("t2", np.uint64), ("t3", np.uint64)])
    pairs, _ = workload_counts(wl)
    cap = int(pairs // (128 * 256) * 2 + 4 * S // 4 + 100000)
    buf = torch.zeros(64 + cap * rec_dtype.itemsize, dtype=torch.uint8, device=dev)
    if lib.dsa_trace_configure(buf.data_ptr(), buf.numel()) != 0:
        raise RuntimeError("trace build did not accept the buffer")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    call()
    ev1.record()
    torch.cuda.synchronize()
    lib.dsa_trace_configure(None, 0)
    assert lib.dsa_sync_status(None) == 0, lib.dsa_last_error()
    host = buf.cpu().numpy()
    n = int(host[:8].view(np.uint64)[0])
    rec = host[64:64 + min(n, cap) * rec_dtype.itemsize].view(rec_dtype)
    summary = summarize_trace(rec, torch.cuda.get_device_properties(0).multi_processor_count)
    # SM-cycle sums of the trace build (kernel words 37..43): epilogue thread 0 of
    # each CTA and the MMA issuer
    if not stamps:
        words = ws[:64 * 8].cpu().numpy().view(np.uint64)
        fheads, mheads = max(int(words[43]), 1), max(int(words[42]), 1)
        summary["fold_cycles"] = {"per_head_folded": int(words[38]) / fheads,
                                  "acc_wait_per_head": int(words[37]) / fheads,
                                  "mma_q_tile_wait_per_head": int(words[39]) / mheads,
                                  "mma_acc_free_wait_per_head": int(words[40]) / mheads,
                                  "mma_key_tile_wait_per_head": int(words[41]) / mheads,
                                  "heads_issued": int(words[42]), "heads_folded_thread0": int(words[43]),
                                  "fallback_rows": int(words[36])}
        napp = max(int(words[47]), 1)
        summary["append_cycles"] = {"compare_per_tile": int(words[44]) / napp, "atomic_per_tile": int(words[45]) / napp,
                                    "writes_per_tile": int(words[46]) / napp, "tiles_thread0": int(words[47])}
    summary.update({"workload": args.workload, "S": S, "call_ms": ev0.elapsed_time(ev1), "records_dropped": max(0, n - cap),
                    "build": "stamps only (DSA_TRACE_STAMPS_ONLY)" if stamps else "item stamps and SM-cycle counters",
                    "note": "DSA_ITEM_TRACE build (measurement only): epilogue thread 0 stamps each work item; "
                            "fold = taking the item to the end of its fold over heads (waits on the MMAs included), "
                            "wait = its dependency wait, rest = selection / append / store and publish"})
    summary["attn_fwd_tc_profile"] = fwd_tc_profile(lib, wl, out, to, dev)
    print(json.dumps({"trace": summary}), flush=True)


def fwd_tc_profile(lib, wl, pool_idx, to, dev):
    """The tcgen05 forward (dsa_sparse_attn_fwd_tc) in the same measurement
    build: each warp role's clock cycles per 128-key block and pipeline
    segment, summed over the CTAs (DSA_FWD_PROFILE counters)."""
    import torch
    import synth
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.dsa_sparse_attn_fwd_tc.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, ctypes.c_float, vp, vp, vp]
    lib.dsa_fwd_tc_profile.argtypes = [vp, i32]
    qa, ka, va = synth.attention_inputs(wl)
    q, k, v = to(qa), to(ka), to(va)
    del qa, ka, va
    S = wl.S
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((S, wl.Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for rep in range(2):  # the second call is the one read back
        ev0.record()
        rc = lib.dsa_sparse_attn_fwd_tc(q.data_ptr(), k.data_ptr(), v.data_ptr(), pool_idx.data_ptr(), S, wl.Hq, wl.D,
                                        wl.topk, ctypes.c_float(wl.scale), o.data_ptr(), lse.data_ptr(), stream)
        ev1.record()
        if rc != 0:
            raise RuntimeError(lib.dsa_last_error().decode())
        torch.cuda.synchronize()
    ctas = min(S, torch.cuda.get_device_properties(0).multi_processor_count)
    cnt = np.zeros((ctas, 32), dtype=np.uint64)
    if lib.dsa_fwd_tc_profile(cnt.ctypes.data, ctas) != 32 * ctas:
        return {"error": lib.dsa_last_error().decode()}
    c = cnt.astype(np.float64).sum(axis=0)
    roles = {"producers": (0, ["row_buffer_wait", "selection_scan", "free_stage_wait", "block_record", "copy_issue",
                               "drain"], 7),
             "issuer": (8, ["full_stage_wait", "free_s_wait", "s_issue", "o_products_with_p_waits", "drain"], 15),
             "softmax": (16, ["full_stage_wait", "s_wait_and_load", "max_check_and_rescale", "p_buffer_wait",
                              "p_write", "epilogue"], 23)}
    res = {"call_ms": ev0.elapsed_time(ev1), "ctas": ctas}
    for role, (off, names, bw) in roles.items():
        blocks = max(c[bw], 1.0)
        res[role] = {n: round(c[off + j] / blocks, 1) for j, n in enumerate(names)}
        res[role]["blocks"] = int(c[bw])
    res["unit"] = "SM clock cycles per 128-key block, per role (one thread's view)"
    return res


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.trace or args.trace_stamps:
        run_trace(args, stamps=args.trace_stamps)
    elif args.varlen or args.zigzag:
        run_layout(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
