#!/usr/bin/env python
"""Benchmark of the gated DSA attention step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload head8192|val4096|decode64|decode16]

One step = one pass of the whole prefill hot path over one batch:
lightning indexer + top-k -> sparse MLA -> output gate, through the C ABI.
The default workload is the headline prefill: 2 single-document sequences of
8,192 tokens, top-k 2,048, 64x128 indexer, 96 heads, 576-wide latent rows,
hidden 7,168 (seeded synthetic BF16 data shaped like the pages' workloads).

Prints ONE JSON line (rank 0).  ``value`` is whole-job tokens/s with inputs
resident in HBM; ``e2e`` repeats the measurement through the same C ABI with
pinned host buffers copied in and the gated output copied out inside the
timed region; ``roofline`` describes the dominant kernel (sparse MLA);
``cpu_baseline`` times the CPU oracle on a bounded sample of the workload.

With the default workload the same line also carries two more of the pages'
workloads, each timed on its own with its own roofline and clocks:
``decode64`` (64 decode requests over paged caches, HBM-bound) and
``chunk32k`` (a 32,768-token sequence prefilled as 4 chunks of 8,192 queries
over a growing paged cache).  ``--no-extra`` leaves them out.

Multi-GPU: ``torchrun --nproc-per-node N bench.py --gpus N``: every rank runs
an independent replica (no collective on the data path; the path shards by
sequence), timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA indexer+sparse-MLA tokens/s at T=8192,k=2048; % of TC / HBM roofline"
CSRC = os.path.join(ROOT, "sparse_attention_serving_gb300", "csrc")
# Measured DRAM traffic per unit of work for the dominant kernels, one record
# per kernel: the ncu dram read + write bytes of one captured launch divided by
# the units it processed, with the SHA-256 of the kernel's sources at the time
# of the capture.  A record whose sources have changed since is not used
# (traffic is reported as null).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="head8192",
                    choices=["head8192", "val4096", "decode64", "decode16", "tiny", "chunk32k"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the chosen workload (no decode64 / chunk32k sub-objects)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=0, help="oracle sample size (0 = auto)")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="store a kernel's measured DRAM bytes per unit from an ncu --csv log "
                         "(dram__bytes_read.sum / write.sum of one launch) and exit")
    ap.add_argument("--traffic-kernel", default="sparse_mla_kernel",
                    help="kernel-name substring to pick in the ncu log")
    ap.add_argument("--traffic-key", default=None, help="record name (default: the kernel)")
    ap.add_argument("--traffic-units", type=float, default=0.0,
                    help="units the captured launch processed (queries, or requests)")
    ap.add_argument("--traffic-launch", type=int, default=0,
                    help="which matching launch of the log to use (0 = first)")
    ap.add_argument("--traffic-note", default="", help="how the capture was taken")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# algorithmic work
# ----------------------------------------------------------------------------

def sel_pairs(T: int, k: int, q0: int = 0) -> int:
    """sum over queries t in [q0, T) of min(t+1, k)"""
    return sum(min(t + 1, k) for t in range(q0, T))


def indexer_flops(T: int, k: int, H_I: int, D_I: int) -> int:
    """2*H_I*D_I per scored (t, s), counted for queries with more than k causal keys"""
    return sum(t + 1 for t in range(k, T)) * 2 * H_I * D_I


def mla_flops_per_pair(H: int) -> int:
    return 2 * H * (576 + 512)


def gate_flops(N: int, hid: int, H: int, dv: int) -> int:
    return 2 * N * (hid * H * dv + H * 512 * dv)


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ----------------------------------------------------------------------------

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


def tensor_peaks(peaks):
    """(burst, sustained, source) dense BF16 TFLOP/s.  A kernel timed on its own
    for a fraction of a second is held against the burst figure; the sustained
    one (a seconds-long loop under the power cap) is reported beside it."""
    if peaks.get("bf16_tflops"):
        return peaks["bf16_tflops"], peaks.get("bf16_tflops_sustained"), "measured"
    return 1900.0, 1700.0, "fallback"


def hbm_peak(peaks):
    if peaks.get("hbm_gbs"):
        return peaks["hbm_gbs"], "measured"
    return 6800.0, "fallback"


def _sources_sha(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_per_unit(kernel: str):
    """(bytes per unit, capture note) of a kernel's measured DRAM traffic, or
    (None, reason) when there is no record or the kernel has changed since."""
    try:
        rec = json.load(open(TRAFFIC_FILE))[kernel]
    except Exception:
        return None, "no ncu capture recorded for this kernel"
    if _sources_sha(rec["sources"]) != rec["sources_sha256"]:
        return None, "kernel sources changed since the ncu capture"
    return rec["bytes_per_unit"], rec["capture"]


# sources whose change invalidates a kernel's traffic record
TRAFFIC_SOURCES = {
    "sparse_mla_kernel": ["sparse_mla.cu", "sm103.cuh", "internal.h", "dsa_status.cuh"],
    "sparse_mla_kernel_decode": ["sparse_mla.cu", "sm103.cuh", "internal.h", "dsa_status.cuh"],
}


def record_traffic(args):
    """Read one launch's dram__bytes_read.sum + dram__bytes_write.sum for a kernel
    from an ncu --csv log and store bytes per unit with the SHA-256 of the
    kernel's sources (so the record goes stale when they change)."""
    import csv
    rows = list(csv.reader(open(args.record_traffic)))
    hdr = next(i for i, r in enumerate(rows) if "Kernel Name" in r and "Metric Name" in r)
    H = rows[hdr]
    ki, ii, mi = H.index("Kernel Name"), H.index("ID"), H.index("Metric Name")
    vi, ui = H.index("Metric Value"), H.index("Metric Unit")
    launches = {}
    for r in rows[hdr + 1:]:
        if len(r) <= vi or args.traffic_kernel not in r[ki]:
            continue
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(r[ui], 1)
        launches.setdefault(r[ii], {})[r[mi]] = float(r[vi].replace(",", "")) * scale
    ids = sorted(launches, key=int)
    m = launches[ids[args.traffic_launch]]
    total = m["dram__bytes_read.sum"] + m["dram__bytes_write.sum"]
    key = args.traffic_key or args.traffic_kernel
    src = TRAFFIC_SOURCES[key]
    try:
        recs = json.load(open(TRAFFIC_FILE))
    except Exception:
        recs = {}
    recs[key] = {"bytes_per_unit": total / args.traffic_units, "sources": src,
                 "sources_sha256": _sources_sha(src),
                 "capture": f"{args.traffic_note}: dram read {m['dram__bytes_read.sum']:.0f} + "
                            f"write {m['dram__bytes_write.sum']:.0f} bytes over "
                            f"{args.traffic_units:g} units"}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(recs, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({key: recs[key]}))


def shared_config(cfg, world):
    """The workload description both arms print (the same dict, key for key)."""
    c = {"workload": cfg.name, "B": cfg.B, "T": cfg.T, "topk": cfg.topk, "H": cfg.H,
         "H_I": cfg.H_I, "D_I": cfg.D_I, "latent": 576, "hid": cfg.hid,
         "parallelism": f"replicas x{world}"}
    if cfg.decode:
        c.update({"T": 1, "context": [cfg.L_min, cfg.L_max], "page": 64,
                  "step": "dsa_indexer_topk (decode) -> sparse_mla_fwd (split-K)",
                  "l2": "caches 6.6 GB > L2; between timed steps a 256 MB buffer is "
                        "rewritten, then another 256 MB read (no dirty lines left in L2)"})
    elif cfg.chunk:
        c.update({"chunk": cfg.chunk, "page": 64,
                  "step": "per chunk: dsa_indexer_topk -> sparse_mla_fwd -> mla_gate_apply",
                  "l2": "inputs larger than L2 each step (q_lat alone 3.6 GB)"})
    else:
        c.update({"step": "dsa_indexer_topk -> sparse_mla_fwd -> mla_gate_apply",
                  "l2": "inputs larger than L2 each step (q_lat alone 1.81 GB at head8192); "
                        "a sequence's latent rows stay L2-resident as they do in serving"})
    return c


# ----------------------------------------------------------------------------
# CPU oracle sample
# ----------------------------------------------------------------------------

def oracle_sample(cfg, d, g, rows, lib=None):
    """indexer + top-k, sparse MLA and the gate for the given flat query rows."""
    import numpy as np
    import oracle
    sc = oracle.indexer_scores(d["q_idx"], d["w"], d["k_idx"], d["q_start"], d["kv_len"], rows, lib)
    Tq = d["q_idx"].shape[1]
    nv = (d["q_start"][rows // Tq] + rows % Tq + 1).astype(np.int32)
    idx, _ = oracle.topk(sc, nv, cfg.topk, lib)
    full_idx = np.full((d["q_idx"].shape[0] * Tq, cfg.topk), -1, np.int32)
    full_idx[rows] = idx
    o, lse = oracle.sparse_mla(d["q_lat"], d["kv"], full_idx.reshape(d["q_idx"].shape[0], Tq, -1),
                               d["q_start"], d["kv_len"], cfg.scale, rows, lib)
    out = oracle.gate(g["x"][rows], g["W_g"], o, g["W_uv"], None, lib)
    return out


def cpu_baseline(cfg, d, g, n_rows: int):
    import numpy as np
    import oracle
    lib = oracle.load()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores, lib)
    B, T = cfg.B, cfg.T
    rng = np.random.default_rng(12345)
    rows = np.sort(rng.choice(B * T, n_rows, replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    oracle_sample(cfg, d, g, rows, lib)
    dt = time.perf_counter() - t0
    return {"value": n_rows / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "seconds": dt,
            "sample": f"{n_rows} query rows drawn uniformly from the {B*T} of {cfg.name}; each row "
                      f"runs indexer scores over all causal keys, top-{cfg.topk}, sparse MLA over "
                      f"the selected rows and the gate (float64 C oracle, {cores} threads)"}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(args, rank, world, local):
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_serving_gb300 as dsa
    from workloads import CONFIGS, gate_inputs, prefill

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = CONFIGS[args.workload]
    if cfg.decode:
        return run_decode(args, rank, world, local, cfg)
    if cfg.chunk:
        return run_chunked(args, dsa, world, local, cfg)
    B, T = cfg.B, cfg.T
    N = B * T
    d = prefill(cfg)
    g = gate_inputs(cfg, N)

    def up(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    q_idx, w, k_idx, q_lat, kv = (up(d[k]) for k in ("q_idx", "w", "k_idx", "q_lat", "kv"))
    x, W_g, W_uv = up(g["x"]), up(g["W_g"]), up(g["W_uv"])
    qs = torch.from_numpy(d["q_start"]).to(dev)
    kl = torch.from_numpy(d["kv_len"]).to(dev)
    idx = torch.empty((B, T, cfg.topk), dtype=torch.int32, device=dev)
    o_lat = torch.empty((B, T, cfg.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, cfg.H), dtype=torch.float32, device=dev)
    out = torch.empty((N, cfg.H * cfg.dv), dtype=torch.bfloat16, device=dev)
    ws_bytes = max(dsa.workspace_bytes(op, B, T, T, h, cfg.topk)
                   for op, h in ((dsa.OP_INDEXER_TOPK, cfg.H_I), (dsa.OP_SPARSE_MLA, cfg.H),
                                 (dsa.OP_GATE, cfg.H)))
    ws = dsa.new_workspace(ws_bytes, dev)
    krows, kvrows = dsa.Rows(k_idx), dsa.Rows(kv)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dsa.dsa_indexer_topk(q_idx, w, krows, qs, kl, cfg.topk, T, out_idx=idx, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        dsa.sparse_mla_fwd(q_lat, kvrows, idx, qs, kl, T, cfg.scale, o_lat=o_lat, lse=lse,
                           workspace=ws)
        if ev is not None:
            ev[2].record(stream)
        dsa.mla_gate_apply(x, W_g, o_lat.view(N, cfg.H, 512), W_uv, out=out, workspace=ws)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"device status {code} at {where:#x} ({detail})")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(K):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed = max_over_ranks(elapsed, world)
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"device status {code} at {where:#x} ({detail})")
    t_idx = sum(e[0].elapsed_time(e[1]) for e in evs) / K / 1e3
    t_mla = sum(e[1].elapsed_time(e[2]) for e in evs) / K / 1e3
    t_gate = sum(e[2].elapsed_time(e[3]) for e in evs) / K / 1e3

    peaks = measured_peaks()
    peak, pk_sust, peak_src = tensor_peaks(peaks)
    f_idx = B * indexer_flops(T, cfg.topk, cfg.H_I, cfg.D_I)
    pairs = B * sel_pairs(T, cfg.topk)
    f_mla = pairs * mla_flops_per_pair(cfg.H)
    f_gate = gate_flops(N, cfg.hid, cfg.H, cfg.dv)
    tflops = lambda f, t: f / t / 1e12
    ach = tflops(f_mla, t_mla)
    kern = lambda f, t: {"ms": t * 1e3, "tflops": tflops(f, t), "frac": tflops(f, t) / peak,
                         "frac_of_sustained": tflops(f, t) / pk_sust if pk_sust else None,
                         "flop": f}
    kernels = {"dsa_indexer_topk": kern(f_idx, t_idx), "sparse_mla_fwd": kern(f_mla, t_mla),
               "mla_gate_apply": kern(f_gate, t_gate)}
    bpq, tnote = traffic_per_unit("sparse_mla_kernel")
    tokens = N * world * K
    res = {
        "metric": METRIC,
        "value": tokens / elapsed,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(args.warmup, 3),
        "ms_per_step": elapsed / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) BF16 activations, N(0,0.02) weights)",
        "config": shared_config(cfg, world),
        "value_indexer_mla_only": N * world / max(t_idx + t_mla, 1e-12),
        "kernels": kernels,
        "roofline": {"kernel": "sparse_mla_fwd", "bound": "tensor", "achieved": ach,
                     "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                     "peak_source": f"{peak_src} bf16 burst (the kernel timed on its own "
                                    "launches, each well under a second)",
                     "peak_sustained": pk_sust,
                     "frac_of_sustained": ach / pk_sust if pk_sust else None,
                     "traffic": bpq * N if bpq is not None else None,
                     "traffic_unit": "bytes per launch: ncu dram read+write per query of one "
                                     "captured launch, times the launch's queries",
                     "traffic_capture": tnote,
                     "algorithmic": f"{pairs} (query, selected key) pairs x 2*H*(576+512) FLOP"},
        "gpu_launches": K * launches_per_step(dsa, B, T, cfg),
        "clocks": clk,
    }
    res["variants"] = {"fp8_indexer": run_prefill_fp8(args, dsa, cfg, dev, stream, q_idx, w,
                                                      k_idx, qs, kl, idx, ws, T, f_idx, peak,
                                                      t_mla),
                       "sparse_mla_bwd": run_prefill_bwd(dsa, cfg, dev, stream, q_lat, kvrows,
                                                         idx, o_lat, lse, T, peak)}
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, dsa, d, g, cfg, dev, stream, ws, krows, kvrows, world,
                             tensors=dict(q_idx=q_idx, w=w, k_idx=k_idx, q_lat=q_lat, kv=kv, x=x,
                                          W_g=W_g, W_uv=W_uv, qs=qs, kl=kl, idx=idx, o_lat=o_lat,
                                          lse=lse, out=out))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, d, g, args.cpu_rows or 768)
    if cfg.name == "head8192" and not args.no_extra:
        # free the headline's buffers before the other workloads allocate theirs
        del q_idx, w, k_idx, q_lat, kv, x, W_g, W_uv, idx, o_lat, lse, out, ws, krows, kvrows
        d = g = None
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        res["decode64"] = run_decode(args, rank, world, local, CONFIGS["decode64"])
        torch.cuda.empty_cache()
        res["chunk32k"] = run_chunked(args, dsa, world, local, CONFIGS["chunk32k"])
    return res


def run_prefill_fp8(args, dsa, cfg, dev, stream, q_idx, w, k_idx, qs, kl, idx, ws, T, f_idx,
                    peak_bf16, t_mla):
    """The prefill indexer with FP8 (E4M3) operands, timed on its own: the query
    heads are quantised inside each step, the keys once (as the FP8 cache append
    would have stored them).  Reported beside the BF16 step, not as the headline.
    The FP8 tensor peak is taken as twice the measured BF16 one (the nominal
    dense ratio, 4.5 vs 2.25 PFLOP/s)."""
    import torch
    kc, ksc = dsa.dsa_quant_fp8(k_idx)
    krows8 = dsa.Rows(kc)
    qc = torch.empty(q_idx.shape, dtype=torch.uint8, device=dev)
    qsc = torch.empty(q_idx.shape[:-1], dtype=torch.float32, device=dev)
    idx8 = torch.empty_like(idx)  # the BF16 step's index sets stay as they are

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dsa.dsa_quant_fp8(q_idx, codes=qc, scale=qsc)
        if ev is not None:
            ev[1].record(stream)
        dsa.dsa_indexer_topk_fp8(qc, qsc, w, krows8, ksc, qs, kl, cfg.topk, T, out_idx=idx8,
                                 workspace=ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"fp8 device status {code} at {where:#x} ({detail})")
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        step(evs[i])
    torch.cuda.synchronize(dev)
    t_q = sum(e[0].elapsed_time(e[1]) for e in evs) / K / 1e3
    t_i = sum(e[1].elapsed_time(e[2]) for e in evs) / K / 1e3
    tf = f_idx / t_i / 1e12
    return {"quant_ms": t_q * 1e3, "indexer_ms": t_i * 1e3, "tflops": tf,
            "frac_of_fp8_peak": tf / (2 * peak_bf16),
            "value_indexer_mla_only": cfg.B * T / (t_q + t_i + t_mla), "unit": "tokens/s",
            "step": "dsa_quant_fp8 (queries) -> dsa_indexer_topk_fp8; sparse MLA as in the BF16 step",
            "gpu_launches": K * 2}


def run_prefill_bwd(dsa, cfg, dev, stream, q_lat, kvrows, idx, o_lat, lse, T, peak_bf16, nq=512):
    """The sparse MLA backward on a bounded slice of the workload: the last `nq`
    queries of sequence 0 (each with the full k selected keys), using the step's
    own forward outputs; upstream gradient seeded N(0,1) BF16.  Work per
    (query, selected key): 2*H*(3*576 + 2*512) FLOP (the logits and dp again,
    dq, the key and the value gradients)."""
    import numpy as np
    import torch
    from workloads import normal_bf16
    q0 = T - nq
    sl = lambda t: t[0:1, q0:T].contiguous()
    q, ix, o, ls = sl(q_lat), sl(idx), sl(o_lat), sl(lse)
    g = normal_bf16(cfg.seed, "w", (1, nq, cfg.H, 512), sub=7)
    d_o = torch.from_numpy(g.view(np.int16)).to(dev).view(torch.bfloat16)
    qs = torch.tensor([q0], dtype=torch.int32, device=dev)
    kl = torch.tensor([T], dtype=torch.int32, device=dev)
    dkv = torch.zeros((1, T, 576), dtype=torch.float32, device=dev)
    dq = torch.empty((1, nq, cfg.H, 576), dtype=torch.float32, device=dev)
    # a workspace of dsa_workspace_bytes selects the tcgen05 kernels; the bare
    # status header, the warp-level MMA path (timed beside it for comparison)
    ws_tc = dsa.new_workspace(dsa.workspace_bytes(dsa.OP_SPARSE_MLA_BWD, 1, nq, T, cfg.H, cfg.topk), dev)
    ws_w = dsa.new_workspace(256, dev)

    def timed(ws, K=2):
        run = lambda: dsa.sparse_mla_bwd(q, kvrows, ix, qs, kl, T, o, ls, d_o, dkv, cfg.scale,
                                         dq=dq, workspace=ws)
        run()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            run()
        b.record(stream)
        torch.cuda.synchronize(dev)
        code, where, detail = dsa.read_device_status(ws)
        if code != dsa.DSA_OK:
            raise RuntimeError(f"bwd device status {code} at {where:#x} ({detail})")
        return a.elapsed_time(b) / K / 1e3

    K = 2
    t = timed(ws_tc, K)
    t_warp = timed(ws_w, K)
    flop = nq * cfg.topk * 2 * cfg.H * (3 * 576 + 2 * 512)
    tf = flop / t / 1e12
    return {"ms": t * 1e3, "queries": nq, "tflops": tf, "frac_of_bf16_peak": tf / peak_bf16,
            "flop": flop, "unit": "TFLOP/s",
            "note": "tcgen05 kernels (P and dz from S^T and dP^T, dq from rows^T.dz^T, dKV from "
                    "dz^T.q + p^T.dO with vector atomics); slice: last 512 queries of sequence 0",
            "warp_mma_ms": t_warp * 1e3,
            "gpu_launches": K * 2}


def launches_per_step(dsa, B, T, cfg):
    # indexer 1, sparse MLA 1 (+1 split combine when B*T is below the SM count), gate 1
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 3 + (1 if B * T < sms else 0)


def run_e2e(args, dsa, d, g, cfg, dev, stream, ws, krows, kvrows, world, tensors):
    """The step through the C ABI with pinned host inputs copied in and the gated
    output copied out inside the timed region (weights stay resident), run the
    way a serving loop runs it: each sequence's queries in chunks of 2,048 (a
    chunk is the public calls at q_start = its offset, kv_len = its end, over the
    sequence's keys and latent rows, which are copied in first).  A chunk's
    inputs go in on one stream, its indexer + sparse MLA + gate run on a second
    and its output comes back on a third, so that copies and kernels overlap.
    Every byte of the step's inputs and outputs crosses the host link every step;
    the keys and latent rows alternate between two device copies from step to
    step, and each chunk's buffers are reused only once the previous step is
    done with them."""
    import numpy as np
    import torch
    t = tensors
    B, T, N = cfg.B, cfg.T, cfg.B * cfg.T
    C = min(T, 2048)
    nc = (T + C - 1) // C
    host = {k: torch.from_numpy(d[k].view(np.int16)).view(torch.bfloat16).pin_memory()
            for k in ("q_idx", "w", "k_idx", "q_lat", "kv")}
    host["x"] = torch.from_numpy(g["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    out_h = torch.empty(t["out"].shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size()
    # the step's own output, to check the chunked pipeline against: the same
    # computation per query, up to the order of each index list (candidates are
    # appended by racing warps), hence of the attention's FP32 sums
    ref_out = t["out"].clone()
    kb = [t["k_idx"], torch.empty_like(t["k_idx"])]
    kvb = [t["kv"], torch.empty_like(t["kv"])]
    rows = [[(dsa.Rows(kb[p][b:b + 1]), dsa.Rows(kvb[p][b:b + 1])) for b in range(B)]
            for p in range(2)]
    qs_c = [torch.tensor([c * C], dtype=torch.int32, device=dev) for c in range(nc)]
    kl_c = [torch.tensor([min(T, (c + 1) * C)], dtype=torch.int32, device=dev) for c in range(nc)]
    s_in, s_out, s_cmp = torch.cuda.Stream(dev), torch.cuda.Stream(dev), stream
    done, drained, keys_free = {}, {}, [None, None]

    def step(i, first):
        p = i & 1
        ev_keys = torch.cuda.Event()
        if first:  # the copies start after the caller's point (the start event)
            s_in.wait_stream(s_cmp)
        with torch.cuda.stream(s_in):
            if keys_free[p] is not None:
                s_in.wait_event(keys_free[p])
            kb[p].copy_(host["k_idx"], non_blocking=True)
            kvb[p].copy_(host["kv"], non_blocking=True)
            ev_keys.record(s_in)
        s_cmp.wait_event(ev_keys)
        for b in range(B):
            for c in range(nc):
                q0, q1 = c * C, min(T, (c + 1) * C)
                r0, r1 = b * T + q0, b * T + q1
                ev_in = torch.cuda.Event()
                with torch.cuda.stream(s_in):
                    if (b, c) in done:
                        s_in.wait_event(done[(b, c)])
                    for k in ("q_idx", "w", "q_lat"):
                        t[k][b, q0:q1].copy_(host[k][b, q0:q1], non_blocking=True)
                    t["x"][r0:r1].copy_(host["x"][r0:r1], non_blocking=True)
                    ev_in.record(s_in)
                s_cmp.wait_event(ev_in)
                if (b, c) in drained:
                    s_cmp.wait_event(drained[(b, c)])
                kr, kvr = rows[p][b]
                idx_c, o_c = t["idx"][b:b + 1, q0:q1], t["o_lat"][b:b + 1, q0:q1]
                dsa.dsa_indexer_topk(t["q_idx"][b:b + 1, q0:q1], t["w"][b:b + 1, q0:q1], kr,
                                     qs_c[c], kl_c[c], cfg.topk, T, out_idx=idx_c, workspace=ws,
                                     stream=s_cmp)
                dsa.sparse_mla_fwd(t["q_lat"][b:b + 1, q0:q1], kvr, idx_c, qs_c[c], kl_c[c], T,
                                   cfg.scale, o_lat=o_c, lse=t["lse"][b:b + 1, q0:q1],
                                   workspace=ws, stream=s_cmp)
                dsa.mla_gate_apply(t["x"][r0:r1], t["W_g"], o_c.view(q1 - q0, cfg.H, 512),
                                   t["W_uv"], out=t["out"][r0:r1], workspace=ws, stream=s_cmp)
                ev_done = torch.cuda.Event()
                ev_done.record(s_cmp)
                done[(b, c)] = ev_done
                s_out.wait_event(ev_done)
                with torch.cuda.stream(s_out):
                    out_h[r0:r1].copy_(t["out"][r0:r1], non_blocking=True)
                    ev_out = torch.cuda.Event()
                    ev_out.record(s_out)
                    drained[(b, c)] = ev_out
        kf = torch.cuda.Event()
        kf.record(s_cmp)
        keys_free[p] = kf

    for i in range(2):
        step(i, i == 0)
    torch.cuda.synchronize(dev)
    diff = out_h.to(dev).float() - ref_out.float()
    rel_l2 = float(diff.norm() / ref_out.float().norm())
    max_abs = float(diff.abs().max())
    K = max(2, min(args.steps, 10))
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    a.record(s_cmp)
    for i in range(K):
        step(i, i == 0)
    s_cmp.wait_stream(s_out)
    b_.record(s_cmp)
    torch.cuda.synchronize(dev)
    el = max_over_ranks(a.elapsed_time(b_) / 1e3, world)
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"e2e device status {code} at {where:#x} ({detail})")
    return {"value": N * world * K / el, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K, "ms_per_step": el / K * 1e3,
            "pipeline": f"{B * nc} chunks of {C} queries; copy in, kernels and copy out on "
                        "three streams",
            "vs_step_output": {"rel_l2": rel_l2, "max_abs": max_abs}}


def decode_bytes(lens, topk, H, H_I, D_I):
    """Compulsory HBM bytes of one decode step: every cached indexer key once,
    the selected latent rows once, the queries, weights and outputs."""
    import numpy as np
    lens = np.asarray(lens, np.int64)
    keys = int(lens.sum()) * D_I * 2
    rows = int(np.minimum(lens, topk).sum()) * 576 * 2
    q = len(lens) * (H_I * D_I * 2 + H_I * 2 + H * 576 * 2)
    out = len(lens) * (topk * 4 + H * 512 * 2 + H * 4)
    return keys + rows + q + out


def decode_mla_bytes(lens, topk, H):
    """Compulsory HBM bytes of the decode sparse MLA alone: the selected latent
    rows once, the queries and index lists in, the outputs out."""
    import numpy as np
    lens = np.asarray(lens, np.int64)
    rows = int(np.minimum(lens, topk).sum()) * 576 * 2
    per_req = H * 576 * 2 + topk * 4 + H * 512 * 2 + H * 4
    return rows + len(lens) * per_req


class L2Flush:
    """Empties L2 between timed steps: rewrites a 256 MB buffer (twice L2), then
    reads a second one, so the write-back of the rewrite's dirty lines happens
    here, before the next timed region, not inside its first kernel."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self, i):
        import torch
        self.w.fill_(i & 255)
        torch.sum(self.r, dtype=torch.int64)


def run_decode(args, rank, world, local, cfg):
    """Decode step (indexer + top-k and sparse MLA for one new token per request)
    over paged caches; HBM-bound, reported against the measured copy bandwidth."""
    import numpy as np
    import torch
    import sparse_attention_serving_gb300 as dsa
    from workloads import decode
    dev = torch.device("cuda", local)
    d = decode(cfg)

    def up(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    q_idx, w, q_lat = up(d["q_idx"]), up(d["w"]), up(d["q_lat"])
    k_pool, kv_pool = up(d["k_pool"]), up(d["kv_pool"])
    bt = torch.from_numpy(d["block_table"]).to(dev)
    qs = torch.from_numpy(d["q_start"]).to(dev)
    kl = torch.from_numpy(d["kv_len"]).to(dev)
    B, S = cfg.B, int(d["kv_len"].max())
    idx = torch.empty((B, 1, cfg.topk), dtype=torch.int32, device=dev)
    o_lat = torch.empty((B, 1, cfg.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, 1, cfg.H), dtype=torch.float32, device=dev)
    ws_bytes = max(dsa.workspace_bytes(dsa.OP_INDEXER_TOPK, B, 1, S, cfg.H_I, cfg.topk),
                   dsa.workspace_bytes(dsa.OP_SPARSE_MLA, B, 1, S, cfg.H, cfg.topk))
    ws = dsa.new_workspace(ws_bytes, dev)
    krows, kvrows = dsa.Rows(k_pool, bt), dsa.Rows(kv_pool, bt)
    stream = torch.cuda.current_stream(dev)
    # between timed steps a buffer larger than L2 is rewritten and a second one
    # read (the caches are larger than L2 anyway): L2 then holds none of the
    # previous step's data (score vectors, rows) and none of the rewrite's dirty
    # lines, whose write-back would otherwise land in the next timed kernel
    flush = L2Flush(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dsa.dsa_indexer_topk(q_idx, w, krows, qs, kl, cfg.topk, S, out_idx=idx, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        dsa.sparse_mla_fwd(q_lat, kvrows, idx, qs, kl, S, cfg.scale, o_lat=o_lat, lse=lse,
                           workspace=ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"device status {code} at {where:#x} ({detail})")
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    for i in range(K):
        flush(i)
        step(evs[i])
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    t_idx = sum(e[0].elapsed_time(e[1]) for e in evs) / K / 1e3
    t_mla = sum(e[1].elapsed_time(e[2]) for e in evs) / K / 1e3
    t_step = max_over_ranks(t_idx + t_mla, world)
    peaks = measured_peaks()
    hbm, hbm_src = hbm_peak(peaks)
    nbytes = decode_bytes(d["kv_len"], cfg.topk, cfg.H, cfg.H_I, cfg.D_I)
    ach = nbytes / t_step / 1e9
    idx_bytes = int(d["kv_len"].astype(np.int64).sum()) * cfg.D_I * 2
    mla_bytes = decode_mla_bytes(d["kv_len"], cfg.topk, cfg.H)
    # the cache append that precedes a decode step (indexer-key LayerNorm + the
    # two row writes), timed on its own after the steps so that the caches the
    # steps read are not changed under them; not part of the step's number
    from workloads import append_inputs
    ap = append_inputs(cfg.seed, B, 1, cfg.D_I)
    k_pre, kv_new = torch.from_numpy(ap["k_pre"]).to(dev), up(ap["kv_new"])
    ws_app = dsa.new_workspace(dsa.workspace_bytes(dsa.OP_CACHE_APPEND, B, 1, 0, 0, 0), dev)
    for _ in range(3):
        dsa.dsa_cache_append(k_pre, kv_new, krows, kvrows, qs, workspace=ws_app)
    torch.cuda.synchronize(dev)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(K):
        dsa.dsa_cache_append(k_pre, kv_new, krows, kvrows, qs, workspace=ws_app)
    a1.record(stream)
    torch.cuda.synchronize(dev)
    code, where, detail = dsa.read_device_status(ws_app)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"append device status {code} at {where:#x} ({detail})")
    t_app = a0.elapsed_time(a1) / K / 1e3
    app_bytes = B * (cfg.D_I * 4 + 1152 + cfg.D_I * 2 + 1152)
    fp8 = run_decode_fp8(args, dev, cfg, d, k_pool, bt, qs, kl, q_idx, w, q_lat, kvrows, idx,
                         o_lat, lse, ws, flush, stream, S, hbm)
    gbs = lambda nb, t: nb / t / 1e9
    bps_mla, tnote = traffic_per_unit("sparse_mla_kernel_decode")
    res = {
        "metric": METRIC, "value": B * world / t_step, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) BF16, paged caches with permuted pages)",
        "config": shared_config(cfg, world),
        "kernels": {"dsa_indexer_topk": {"ms": t_idx * 1e3, "bytes": idx_bytes,
                                         "gbs": gbs(idx_bytes, t_idx),
                                         "frac": gbs(idx_bytes, t_idx) / hbm},
                    "sparse_mla_fwd": {"ms": t_mla * 1e3, "bytes": mla_bytes,
                                       "gbs": gbs(mla_bytes, t_mla),
                                       "frac": gbs(mla_bytes, t_mla) / hbm,
                                       "traffic": (bps_mla * B if bps_mla is not None
                                                   else None),
                                       "traffic_capture": tnote,
                                       "bytes_what": "selected latent rows (min(L,k) x 1,152 B "
                                                     "per request) + q_lat + idx in, o_lat + "
                                                     "lse out"},
                    "dsa_cache_append": {"us": t_app * 1e6, "gbs": gbs(app_bytes, t_app),
                                         "bytes": app_bytes,
                                         "note": "timed separately, back to back; not in the step"}},
        "variants": {"fp8_indexer": fp8},
        "roofline": {"kernel": "decode step", "bound": "hbm", "achieved": ach, "peak": hbm,
                     "unit": "GB/s", "frac": ach / hbm, "traffic": None,
                     "peak_source": f"{hbm_src} HBM copy bandwidth",
                     "algorithmic": f"{nbytes} compulsory bytes per step"},
        # scores + select, sparse MLA (+ split combine): no gate in the decode step
        "gpu_launches": K * launches_per_step(dsa, B, 1, cfg),
        "clocks": clk,
    }
    return res


def run_decode_fp8(args, dev, cfg, d, k_pool, bt, qs, kl, q_idx, w, q_lat, kvrows, idx, o_lat,
                   lse, ws, flush, stream, S, hbm):
    """The same decode step with the FP8 (E4M3) indexer: the query heads are
    quantised inside the step, the key cache is held as E4M3 codes plus one FP32
    scale per token (quantised once here, as the FP8 cache append would have
    written it).  Reported beside the BF16 step, not as the headline."""
    import numpy as np
    import torch
    import sparse_attention_serving_gb300 as dsa
    kc, ksc = dsa.dsa_quant_fp8(k_pool)
    qc = torch.empty(q_idx.shape, dtype=torch.uint8, device=dev)
    qsc = torch.empty(q_idx.shape[:-1], dtype=torch.float32, device=dev)
    krows8 = dsa.Rows(kc, bt)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dsa.dsa_quant_fp8(q_idx, codes=qc, scale=qsc)
        dsa.dsa_indexer_topk_fp8(qc, qsc, w, krows8, ksc, qs, kl, cfg.topk, S, out_idx=idx,
                                 workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        dsa.sparse_mla_fwd(q_lat, kvrows, idx, qs, kl, S, cfg.scale, o_lat=o_lat, lse=lse,
                           workspace=ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"fp8 device status {code} at {where:#x} ({detail})")
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush(i)
        step(evs[i])
    torch.cuda.synchronize(dev)
    t_idx = sum(e[0].elapsed_time(e[1]) for e in evs) / K / 1e3
    t_mla = sum(e[1].elapsed_time(e[2]) for e in evs) / K / 1e3
    keys = int(d["kv_len"].astype(np.int64).sum())
    idx_bytes = keys * (cfg.D_I + 4)
    return {"ms_per_step": (t_idx + t_mla) * 1e3, "value": cfg.B / (t_idx + t_mla),
            "unit": "tokens/s",
            "indexer_ms": t_idx * 1e3, "indexer_gbs": idx_bytes / t_idx / 1e9,
            "indexer_frac": idx_bytes / t_idx / 1e9 / hbm, "sparse_mla_ms": t_mla * 1e3,
            "indexer_bytes": idx_bytes,
            "step": "dsa_quant_fp8 (queries) -> dsa_indexer_topk_fp8 -> sparse_mla_fwd",
            "gpu_launches": K * 5}


def run_chunked(args, dsa, world, local, cfg):
    """Chunked long-context prefill: one sequence of cfg.T tokens whose queries
    are processed in chunks of cfg.chunk against a paged cache (page 64, pages
    permuted) that holds the keys up to the chunk's end.  One step = every
    chunk's indexer + top-k, sparse MLA and gate, in order, through the C ABI."""
    import numpy as np
    import torch
    from workloads import gate_inputs, page_table, prefill_keys, prefill_queries, to_pages
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    T, C = cfg.T, cfg.chunk
    nc = T // C
    keys = prefill_keys(cfg, T)
    lens = np.full(cfg.B, T, np.int64)
    bt_h, num_pages = page_table(cfg.seed, lens)
    q = prefill_queries(cfg, 0, T)
    g = gate_inputs(cfg, T)

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    k_pool = up(to_pages(keys["k_idx"], lens, bt_h, num_pages))
    kv_pool = up(to_pages(keys["kv"], lens, bt_h, num_pages))
    bt = torch.from_numpy(bt_h).to(dev)
    q_idx, w, q_lat = up(q["q_idx"]), up(q["w"]), up(q["q_lat"])
    x, W_g, W_uv = up(g["x"]), up(g["W_g"]), up(g["W_uv"])
    del q, g, keys
    idx = torch.empty((1, T, cfg.topk), dtype=torch.int32, device=dev)
    o_lat = torch.empty((1, T, cfg.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((1, T, cfg.H), dtype=torch.float32, device=dev)
    out = torch.empty((T, cfg.H * cfg.dv), dtype=torch.bfloat16, device=dev)
    krows, kvrows = dsa.Rows(k_pool, bt), dsa.Rows(kv_pool, bt)
    ws_bytes = max(dsa.workspace_bytes(op, 1, C, T, h, cfg.topk)
                   for op, h in ((dsa.OP_INDEXER_TOPK, cfg.H_I), (dsa.OP_SPARSE_MLA, cfg.H),
                                 (dsa.OP_GATE, cfg.H)))
    ws = dsa.new_workspace(ws_bytes, dev)
    qs = [torch.tensor([c * C], dtype=torch.int32, device=dev) for c in range(nc)]
    kl = [torch.tensor([(c + 1) * C], dtype=torch.int32, device=dev) for c in range(nc)]

    def step(ev=None):
        for c in range(nc):
            q0, q1 = c * C, (c + 1) * C
            e = ev[c] if ev is not None else None
            if e is not None:
                e[0].record(stream)
            dsa.dsa_indexer_topk(q_idx[:, q0:q1], w[:, q0:q1], krows, qs[c], kl[c], cfg.topk, T,
                                 out_idx=idx[:, q0:q1], workspace=ws)
            if e is not None:
                e[1].record(stream)
            dsa.sparse_mla_fwd(q_lat[:, q0:q1], kvrows, idx[:, q0:q1], qs[c], kl[c], T, cfg.scale,
                               o_lat=o_lat[:, q0:q1], lse=lse[:, q0:q1], workspace=ws)
            if e is not None:
                e[2].record(stream)
            dsa.mla_gate_apply(x[q0:q1], W_g, o_lat[0, q0:q1], W_uv, out=out[q0:q1],
                               workspace=ws)
            if e is not None:
                e[3].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"chunked device status {code} at {where:#x} ({detail})")
    K = max(2, min(args.steps, 10))
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nc)]
           for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    for i in range(K):
        step(evs[i])
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    code, where, detail = dsa.read_device_status(ws)
    if code != dsa.DSA_OK:
        raise RuntimeError(f"chunked device status {code} at {where:#x} ({detail})")
    per = lambda a, b: [sum(evs[i][c][a].elapsed_time(evs[i][c][b]) for i in range(K)) / K / 1e3
                        for c in range(nc)]
    t_idx_c, t_mla_c, t_gate_c = per(0, 1), per(1, 2), per(2, 3)
    t_idx, t_mla, t_gate = sum(t_idx_c), sum(t_mla_c), sum(t_gate_c)
    t_step = max_over_ranks(t_idx + t_mla + t_gate, world)
    peak, pk_sust, peak_src = tensor_peaks(measured_peaks())
    f_idx = sum(t + 1 for t in range(cfg.topk, T)) * 2 * cfg.H_I * cfg.D_I
    f_mla = sel_pairs(T, cfg.topk) * mla_flops_per_pair(cfg.H)
    f_gate = gate_flops(T, cfg.hid, cfg.H, cfg.dv)
    tf = lambda f, t: f / t / 1e12
    ach = tf(f_mla, t_mla)
    return {
        "metric": METRIC, "value": T * world / t_step, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) BF16 activations, N(0,0.02) weights; paged caches "
                "with permuted pages)",
        "config": shared_config(cfg, world),
        "value_indexer_mla_only": T * world / (t_idx + t_mla),
        "kernels": {
            "dsa_indexer_topk": {"ms": t_idx * 1e3, "ms_per_chunk": [t * 1e3 for t in t_idx_c],
                                 "tflops": tf(f_idx, t_idx), "frac": tf(f_idx, t_idx) / peak,
                                 "flop": f_idx},
            "sparse_mla_fwd": {"ms": t_mla * 1e3, "ms_per_chunk": [t * 1e3 for t in t_mla_c],
                               "tflops": ach, "frac": ach / peak, "flop": f_mla},
            "mla_gate_apply": {"ms": t_gate * 1e3, "tflops": tf(f_gate, t_gate),
                               "frac": tf(f_gate, t_gate) / peak, "flop": f_gate}},
        "roofline": {"kernel": "indexer + top-k + sparse MLA (all chunks)", "bound": "tensor",
                     "achieved": tf(f_idx + f_mla, t_idx + t_mla), "peak": peak,
                     "unit": "TFLOP/s", "frac": tf(f_idx + f_mla, t_idx + t_mla) / peak,
                     "peak_source": f"{peak_src} bf16 burst", "peak_sustained": pk_sust,
                     "traffic": None,
                     "algorithmic": f"indexer {f_idx} FLOP (2*H_I*D_I per scored pair of a "
                                    f"query with more than k causal keys) + sparse MLA {f_mla} "
                                    "FLOP (2*H*(576+512) per selected pair)"},
        "gpu_launches": K * nc * launches_per_step(dsa, 1, C, cfg),
        "clocks": clk,
    }


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle, as it stands, on the machine's host cores
# ----------------------------------------------------------------------------

def run_reference(args, rank, world):
    import numpy as np
    import oracle
    from workloads import CONFIGS, gate_inputs, prefill
    if rank != 0:
        return None
    cfg = CONFIGS[args.workload]
    if cfg.decode or cfg.chunk:
        return {"impl": "reference", "unavailable": "reference arm wired for unchunked prefill only"}
    d = prefill(cfg)
    g = gate_inputs(cfg, cfg.B * cfg.T)
    lib = oracle.load()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores, lib)
    rows_per_step = args.cpu_rows or 32
    rng = np.random.default_rng(777)
    W = max(args.warmup, 0)
    times = []
    for i in range(W + args.steps):
        rows = np.sort(rng.choice(cfg.B * cfg.T, rows_per_step, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle_sample(cfg, d, g, rows, lib)
        if i >= W:
            times.append(time.perf_counter() - t0)
    el = sum(times)
    val = rows_per_step * args.steps / el
    sample = (f"each step: {rows_per_step} query rows drawn uniformly from the {cfg.B*cfg.T} of "
              f"{cfg.name}, indexer + top-{cfg.topk} + sparse MLA + gate in the float64 C oracle")
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": W, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) BF16 activations, N(0,0.02) weights)",
        "config": shared_config(cfg, world),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    if args.record_traffic:
        record_traffic(args)
        return
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
