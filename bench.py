#!/usr/bin/env python3
"""Benchmark of HeadTail ring (context-parallel) causal attention, fwd + bwd.

One step = the whole hot path over one batch of synthetic inputs resident in
HBM: HeadTail shard of q, k, v, dO -> ring attention forward (O, LSE) ->
backward (D preprocess, dK/dV kernel, dQ kernel) -> unshard of O, dQ, dK, dV.
Every step of it runs in libcpattn's CUDA kernels, called through the C ABI.

value  = algorithmic causal fwd+bwd TFLOP/s (7 * B * H * T^2 * d / 2 ... see
         flops below) summed over ranks / max-over-ranks step time.
e2e    = the same metric with pinned-host -> device copies of q, k, v, dO and
         device -> host copies of O, LSE, dQ, dK, dV inside the timed region.
roofline: the kernel with the most device time per step, timed live with CUDA
         events that the library records at kernel boundaries.
cpu_baseline: the float64 CPU oracle, timed on a bounded sample (rank 0, N=1).

N > 1: every rank runs its own replica on its own batch (the (b, h) problems
are independent), so there is no collective on the data path; only the timing
uses a barrier and a max over ranks. Under a launcher (torchrun) the world size
must equal --gpus; without one, --gpus N > 1 starts N ranks through
torch.distributed.run itself.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal attn fwd+bwd TFLOP/s & tokens/s at T=32k, % of GB300 BF16 TC peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "window_32k"

# DRAM bytes (read + write) per launch of a kernel on a workload, from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum), each tagged with the
# digest of the kernel sources it was taken on (KERNEL_SOURCES, see
# kernel_digest). A capture whose digest no longer matches the sources in the
# tree describes an older kernel: the bench then reports the traffic as null.
NCU_TRAFFIC = {
    ("window_32k", "fwd"): (0.499014e9 + 0.118961e9, "15648c3798d7"),
    ("window_32k", "bwd_dkdv"): (0.543523e9 + 0.238607e9, "6a778e6f4486"),
    ("window_32k", "bwd_dq"): (0.673456e9 + 0.123740e9, "5182bf0ed1d2"),
}
CSRC = os.path.join(ROOT, "context_causal_attention_headtail_gb300", "csrc")
KERNEL_SOURCES = {
    "fwd": ("attn_fwd_tc.cu", "tc_common.cuh", "attn_common.cuh", "device_common.cuh"),
    "bwd_dkdv": ("attn_bwd2_tc.cu", "tc_common.cuh", "attn_common.cuh", "device_common.cuh"),
    "bwd_dq": ("attn_dq_pair.cu", "tc_common.cuh", "attn_common.cuh", "device_common.cuh"),
}


def kernel_digest(kernel: str) -> str:
    """First 12 hex digits of the SHA-256 of the kernel's source files, in order."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def ncu_traffic(workload: str, kernel: str):
    """(bytes per launch, source note) of the kernel's last ncu capture, or (None, why)."""
    entry = NCU_TRAFFIC.get((workload, kernel))
    if entry is None:
        return None, "no ncu capture of this kernel on this workload"
    nbytes, digest = entry
    if digest is None or digest != kernel_digest(kernel):
        return None, "kernel sources changed since the ncu capture"
    return nbytes, f"ncu dram__bytes_read.sum + dram__bytes_write.sum, sources {digest}"


def launch_plan(gpus: int, env) -> tuple[str, str]:
    """How to honour --gpus N: run here, relaunch under torch.distributed.run
    (one process per GPU) or refuse when a launcher already set another world size."""
    if gpus < 1:
        return "refuse", f"--gpus {gpus}: need at least one GPU"
    world = env.get("WORLD_SIZE")
    if world is None:
        return ("run", "") if gpus == 1 else ("relaunch", "")
    if int(world) != gpus:
        return "refuse", f"--gpus {gpus} but the launcher started WORLD_SIZE={world} ranks"
    return "run", ""


def relaunch_cmd(gpus: int, argv: list[str], port: int) -> list[str]:
    """torch.distributed.run line that starts this script once per GPU on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port),
            os.path.abspath(__file__)] + list(argv)


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-merge", action="store_true", help="skip timing the standalone merge kernel")
    ap.add_argument("--rope-in-kernel", action="store_true",
                    help="rotate q, k inside the attention calls (cpattn_fwd_rope_save / cpattn_bwd_rotated) "
                         "instead of in shard/unshard")
    return ap.parse_args()


def host_link_gbs(host_in, dev_in, host_out, dev_out, h2d_s, d2h_s, reps=3):
    """Pinned host <-> device copy rates of this machine, measured with the e2e
    buffers before the timed region: H2D alone, D2H alone and both at once on
    the two copy streams (GB/s, the best of a few rounds after a warm-up round).
    The e2e step cannot be faster than its copies."""
    import torch

    def best(fn):
        times = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            times.append(time.perf_counter() - t0)
        return min(times)

    def h2d():
        with torch.cuda.stream(h2d_s):
            for k in dev_in:
                dev_in[k].copy_(host_in[k], non_blocking=True)

    def d2h():
        with torch.cuda.stream(d2h_s):
            for k in dev_out:
                host_out[k].copy_(dev_out[k], non_blocking=True)

    bi = sum(t.numel() * t.element_size() for t in host_in.values())
    bo = sum(t.numel() * t.element_size() for t in host_out.values())
    h2d(), d2h()
    torch.cuda.synchronize()
    t_in, t_out = best(h2d), best(d2h)
    t_both = best(lambda: (h2d(), d2h()))
    return {"h2d": round(bi / t_in / 1e9, 1), "d2h": round(bo / t_out / 1e9, 1),
            "both": round((bi + bo) / t_both / 1e9, 1)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def input_bytes(w, elt=2):
    """Bytes of q, k, v, dO (and of o, dq, dk, dv) in the storage dtype."""
    return 2 * (w.H + w.kv_heads) * w.B * w.T * w.d * elt


def workload_config(w):
    cfg = {"workload": w.name, "B": w.B, "T": w.T, "T_valid": w.T_valid, "H": w.H, "d": w.d,
           "cp": w.cp, "causal": w.causal, "rope": w.rope,
           "l2": "inputs larger than L2: q,k,v,dO = %d MiB per step vs 129 MB L2"
                 % (input_bytes(w) // 2 ** 20)}
    if w.kv_heads != w.H:
        cfg["H_kv"] = w.kv_heads
    if w.yarn:
        cfg["yarn"] = {"factor": w.yarn_factor, "original_max_position": w.yarn_original}
    if w.ulysses:
        cfg["ulysses_ranks"] = w.ulysses
    if w.packed:
        cu = w.cu_seqlens()
        cfg["documents"] = {"n": len(cu) - 1, "length_range": list(w.doc_len),
                            "lengths": [int(x) for x in np.diff(cu)]}
    return cfg


# ----------------------------------------------------------- rank logic ----
# Every rank runs its own replica on its own batch (the (b, h) problems are
# independent), so the only cross-rank traffic is timing: a barrier around the
# timed region and the max of the per-rank step times.

def rank_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(w, rank: int) -> int:
    """Seed of rank `rank`'s batch: the workload's seed, shifted per rank."""
    from context_causal_attention_headtail_gb300.synth import SEEDS
    return SEEDS.get(w.name, 1234) + rank


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, flops_per_rank: float, ms_max: float) -> float:
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's step time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        sm, smax, reasons, power = [], [], set(), []
        for line in self.out.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ---------------------------------------------------------- CPU oracle ----

_INPUT_CACHE = {}


def _workload_inputs(w):
    from context_causal_attention_headtail_gb300.synth import SEEDS, make_inputs
    if w.name not in _INPUT_CACHE:
        _INPUT_CACHE[w.name] = make_inputs(w, SEEDS.get(w.name, 1234))
    return _INPUT_CACHE[w.name]


def oracle_sample(w, seconds_target=12.0, max_heads=64):
    """Times the float64 oracle on a bounded sample of the workload.

    Sample: full forward + backward of whole heads (b=0, h=0,1,...) over the
    first T_s tokens of the workload's own inputs. For causal attention the
    first T_s output rows of a head are exactly that prefix's attention, so
    this is a slice of the same problem; its algorithmic work is
    7 * T_s^2 * d flops per head (3.5 x the causal forward 2 * T_s^2 * d), or
    the same count over the prefix's documents for packed workloads.
    """
    from oracle import attention as A

    T_s = min(w.T_valid, 4096)
    rope = (A.RopeSpec(factor=w.yarn_factor, original_max_position=w.yarn_original)
            if w.yarn else w.rope)
    docs, pairs = None, T_s * T_s * (0.5 if w.causal else 1.0)
    if w.packed:          # the documents of the prefix, the last one cut at T_s
        cu = w.cu_seqlens()
        docs = np.append(cu[cu < T_s], T_s)
        lens = np.diff(docs).astype(np.float64)
        pairs = float(np.sum(lens * lens)) * (0.5 if w.causal else 1.0)
    inp = _workload_inputs(w)
    q, k, v, do = (inp[n][0:1, :, :T_s].double().numpy() for n in ("q", "k", "v", "do"))
    heads, t0 = 0, time.perf_counter()
    while heads < min(max_heads, w.H):
        sl = slice(heads, heads + 1)
        hk = heads // (w.H // w.kv_heads)     # the K/V head this query head reads
        kl = slice(hk, hk + 1)
        O, L = A.forward(q[:, sl], k[:, kl], v[:, kl], w.causal, T_s, rope, docs=docs)
        A.backward(q[:, sl], k[:, kl], v[:, kl], O, L, do[:, sl], w.causal, T_s, rope, docs=docs)
        heads += 1
        if time.perf_counter() - t0 >= seconds_target:
            break
    dt = time.perf_counter() - t0
    flops = heads * 3.5 * 4.0 * pairs * w.d          # 3.5 x the forward's 4 d flops per live pair
    return {"seconds": dt, "flops": flops, "tokens": heads * T_s, "T_s": T_s, "heads": heads,
            "cores": os.cpu_count(),
            "blas_threads": os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
            or str(os.cpu_count())}


def cpu_baseline_entry(w, s):
    tflops = s["flops"] / s["seconds"] / 1e12
    return {"value": tflops, "unit": UNIT, "cores": int(s["blas_threads"]), "kind": "oracle",
            "tokens_per_s": s["tokens"] / s["seconds"],
            "sample": (f"float64 oracle forward+backward of {s['heads']} head(s), first {s['T_s']} "
                       f"tokens of the {w.name} inputs (b=0), {s['seconds']:.1f} s on the host")}


def run_reference(args):
    """--impl reference: the oracle, timed as it stands on the host cores."""
    world, rank, _ = rank_env()
    if rank != 0:
        return
    from context_causal_attention_headtail_gb300.synth import WORKLOADS
    w = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        oracle_sample(w, seconds_target=0.0, max_heads=1)
    times, samples = [], []
    for _ in range(args.steps):
        s = oracle_sample(w, seconds_target=0.0, max_heads=1)
        times.append(s["seconds"])
        samples.append(s)
    tot_flops = sum(s["flops"] for s in samples)
    tot_t = sum(times)
    value = tot_flops / tot_t / 1e12
    base = cpu_baseline_entry(w, {**samples[0], "seconds": tot_t, "flops": tot_flops,
                                  "tokens": sum(s["tokens"] for s in samples),
                                  "heads": sum(s["heads"] for s in samples)})
    base["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w), "cpu_baseline": base,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU ----

def run_ours(args):
    import torch
    import torch.distributed as dist

    from context_causal_attention_headtail_gb300 import cpattn
    from context_causal_attention_headtail_gb300.synth import SEEDS, WORKLOADS, make_inputs

    world, rank, local = rank_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    if w.dtype != "bf16":
        raise SystemExit("bench runs the bf16 tensor-core path; pick a bf16 workload")

    inp = make_inputs(w, rank_seed(w, rank))
    if rank == 0:
        _INPUT_CACHE[w.name] = inp
    P = w.ulysses
    if P:
        # Ulysses: the caller holds P sequence shards (contiguous token blocks,
        # stacked rank-major as [P*B, H, T/P, d]); the attention runs on the
        # head shards [P*B, H/P, T, d] at cp = 1.
        Tl = w.T // P
        inp = {k: torch.cat([v[:, :, r * Tl:(r + 1) * Tl] for r in range(P)], dim=0).contiguous()
               for k, v in inp.items()}
    host_in = {k: v.pin_memory() for k, v in inp.items()}
    nat = {k: v.to(dev) for k, v in inp.items()}
    if P:
        sh = {k: torch.empty((v.shape[0], max(v.shape[1] // P, 1), w.T, w.d), dtype=v.dtype, device=dev)
              for k, v in nat.items()}
    else:
        sh = {k: torch.empty_like(v) for k, v in nat.items()}
    o, dq = torch.empty_like(sh["q"]), torch.empty_like(sh["q"])
    dk, dv = torch.empty_like(sh["k"]), torch.empty_like(sh["v"])
    Bx, Hx = sh["q"].shape[0], sh["q"].shape[1]       # batch and heads the attention sees
    cp_attn = 1 if P else w.cp
    lse = torch.empty((Bx, Hx, w.T), dtype=torch.float32, device=dev)
    ws = torch.empty(cpattn.cpattn_bwd_workspace_bytes(Bx, w.T, Hx, w.d), dtype=torch.uint8, device=dev)
    outs = {"o": o, "dq": dq, "dk": dk, "dv": dv}
    out_like = {"o": "q", "dq": "q", "dk": "k", "dv": "v"}
    outs_nat = {k: torch.empty_like(nat[out_like[k]]) for k in outs}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs_nat.items()}
    host_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    stream = torch.cuda.current_stream(dev)

    kernels = ["shard", "fwd", "bwd_D", "bwd_dkdv", "bwd_dq", "unshard"]
    # the ring path shards q, k, v, dO in one launch and unshards o, dq, dk, dv in one;
    # the Ulysses all-to-all runs per tensor
    n_passes = 4 if P else 1
    # at d = 128 the paired dQ kernel computes D = rowsum(dO * O) itself: no D launch
    d_fused = w.d == 128
    launches_per_step = 2 * n_passes + 1 + (2 if d_fused else 3) + (1 if w.packed else 0)

    def new_events():
        evs = {"shard": [], "unshard": []}
        for _ in range(n_passes):
            evs["shard"].append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
            evs["unshard"].append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
        evs["fwd"] = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        # backward: start, after the D pass, dK/dV start / end, dQ start / end
        evs["bwd"] = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for e in [x for p in evs["shard"] + evs["unshard"] for x in p] + evs["fwd"] + evs["bwd"]:
            e.record(stream)   # creates the underlying CUDA event so its handle can be passed down
        return evs

    # RoPE at global positions: fused into the shard / unshard passes of q, k
    # and dq, dk (default), or applied inside the attention kernels.
    fused = w.rope and not args.rope_in_kernel
    rope_flag = w.rope and not fused
    if rope_flag and P:
        raise SystemExit("the Ulysses workload takes RoPE from its all-to-all; drop --rope-in-kernel")
    rope_cfg = (cpattn.RopeCfg(factor=w.yarn_factor, original_max_position=w.yarn_original)
                if w.yarn else None)
    # in-kernel RoPE: the forward rotates as it streams and stores the rotated
    # q, k, which the backward reads in place of q, k
    q_rot = torch.empty_like(sh["q"]) if rope_flag else None
    k_rot = torch.empty_like(sh["k"]) if rope_flag else None
    docs = cu_dev = cu_host = None
    if w.packed:          # cu_seqlens -> per-position document bounds, every step
        cu_host = torch.from_numpy(w.cu_seqlens()).pin_memory()
        cu_dev = cu_host.to(dev)
        docs = (torch.empty(w.T, dtype=torch.int32, device=dev), torch.empty(w.T, dtype=torch.int32, device=dev))

    names_in, names_out = ("q", "k", "v", "do"), ("o", "dq", "dk", "dv")

    def step(evs=None, nat=nat, outs_nat=outs_nat, lse=lse):
        if P:
            for i, name in enumerate(names_in):
                if evs:
                    cpattn.cpattn_set_trace_events([e.cuda_event for e in evs["shard"][i]])
                cpattn.ulysses_a2a(nat[name], sh[name], P, rope=fused and name in ("q", "k"), cfg=rope_cfg,
                                   stream=stream)
        else:   # one launch for the four tensors, q and k rotated when RoPE is fused into it
            if evs:
                cpattn.cpattn_set_trace_events([e.cuda_event for e in evs["shard"][0]])
            cpattn.shard_batch([nat[n_] for n_ in names_in], [sh[n_] for n_ in names_in], w.cp,
                               rope=[fused and n_ in ("q", "k") for n_ in names_in], stream=stream, cfg=rope_cfg)
        if docs is not None:
            cpattn.doc_bounds(cu_dev, w.T, docs[0], docs[1], stream)
        if evs:
            cpattn.cpattn_set_trace_events([e.cuda_event for e in evs["fwd"]])
        if rope_flag:
            cpattn.fwd_rope_save(sh["q"], sh["k"], sh["v"], o, lse, q_rot, k_rot, cp_attn, w.T_valid, w.causal,
                                 stream, docs=docs, rope_cfg=rope_cfg)
        else:
            cpattn.fwd(sh["q"], sh["k"], sh["v"], o, lse, cp_attn, w.T_valid, w.causal, False, stream, docs=docs)
        if evs:
            cpattn.cpattn_set_trace_events([e.cuda_event for e in evs["bwd"]])
        if rope_flag:
            cpattn.bwd_rotated(q_rot, k_rot, sh["v"], o, lse, sh["do"], dq, dk, dv, ws, cp_attn, w.T_valid,
                               w.causal, stream, docs=docs, rope_cfg=rope_cfg)
        else:
            cpattn.bwd(sh["q"], sh["k"], sh["v"], o, lse, sh["do"], dq, dk, dv, ws, cp_attn, w.T_valid,
                       w.causal, False, stream, docs=docs)
        if P:
            for i, name in enumerate(names_out):
                if evs:
                    cpattn.cpattn_set_trace_events([e.cuda_event for e in evs["unshard"][i]])
                cpattn.ulysses_a2a(outs[name], outs_nat[name], P, inverse=True,
                                   rope=fused and name in ("dq", "dk"), cfg=rope_cfg, stream=stream)
        else:
            if evs:
                cpattn.cpattn_set_trace_events([e.cuda_event for e in evs["unshard"][0]])
            cpattn.shard_batch([outs[n_] for n_ in names_out], [outs_nat[n_] for n_ in names_out], w.cp,
                               rope=[fused and n_ in ("dq", "dk") for n_ in names_out], stream=stream,
                               cfg=rope_cfg, inverse=True)
        if evs:
            cpattn.cpattn_set_trace_events([])

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    cpattn.cpattn_sync_status(stream.cuda_stream)

    step_events = [new_events() for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    sampler = ClockSampler(gpu_id)
    torch.cuda.synchronize(dev)
    barrier()
    sampler.start()
    time.sleep(0.3)
    start.record(stream)
    for i in range(args.steps):
        step(step_events[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    cpattn.cpattn_sync_status(stream.cuda_stream)
    ms_local = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms_local, world, dev)

    # per-kernel device time per step (averaged over the timed steps)
    ker_ms = {k: 0.0 for k in kernels}
    for evs in step_events:
        ker_ms["shard"] += sum(a.elapsed_time(b) for a, b in evs["shard"])
        ker_ms["unshard"] += sum(a.elapsed_time(b) for a, b in evs["unshard"])
        ker_ms["fwd"] += evs["fwd"][0].elapsed_time(evs["fwd"][1])
        b = evs["bwd"]
        ker_ms["bwd_D"] += b[0].elapsed_time(b[1])
        ker_ms["bwd_dkdv"] += b[2].elapsed_time(b[3])
        ker_ms["bwd_dq"] += b[4].elapsed_time(b[5])
    ker_ms = {k: v / args.steps for k, v in ker_ms.items()}

    # e2e through the same public API, host buffers in and out. Every step
    # copies its inputs in from pinned host memory and its results (o, lse,
    # dq, dk, dv) back out, on two copy streams with double-buffered device
    # buffers: the inputs of step i+1 and the outputs of step i-1 move while
    # step i computes, as an input pipeline of a training loop would do.
    e2e = None
    if not args.no_e2e:
        nat_b = [nat, {k: torch.empty_like(v) for k, v in nat.items()}]
        out_b = [outs_nat, {k: torch.empty_like(v) for k, v in outs_nat.items()}]
        lse_b = [lse, torch.empty_like(lse)]
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        link = host_link_gbs(host_in, nat_b[1], host_out, out_b[1], h2d_s, d2h_s)
        for _ in range(2):
            step()
        torch.cuda.synchronize(dev)
        barrier()
        mk = lambda: torch.cuda.Event()
        h2d_done, done, d2h_done = [mk(), mk()], [mk(), mk()], [mk(), mk()]
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def h2d(j):
            bj = j % 2
            with torch.cuda.stream(h2d_s):
                if j >= 2:
                    h2d_s.wait_event(done[bj])          # step j-2 has read this buffer
                for k_ in nat:
                    nat_b[bj][k_].copy_(host_in[k_], non_blocking=True)
                if cu_dev is not None:
                    cu_dev.copy_(cu_host, non_blocking=True)
                h2d_done[bj].record(h2d_s)

        s2.record(stream)
        h2d_s.wait_event(s2)
        d2h_s.wait_event(s2)
        h2d(0)
        for i in range(args.steps):
            bi = i % 2
            if i + 1 < args.steps:
                h2d(i + 1)
            stream.wait_event(h2d_done[bi])
            if i >= 2:
                stream.wait_event(d2h_done[bi])          # outputs of step i-2 are out
            step(nat=nat_b[bi], outs_nat=out_b[bi], lse=lse_b[bi])
            done[bi].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[bi])
                for k_ in outs_nat:
                    host_out[k_].copy_(out_b[bi][k_], non_blocking=True)
                host_lse.copy_(lse_b[bi], non_blocking=True)
                d2h_done[bi].record(d2h_s)
        stream.wait_event(d2h_done[(args.steps - 1) % 2])
        e2.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2) / args.steps, world, dev)
        h2d_bytes = sum(t.numel() * t.element_size() for t in host_in.values())
        if cu_host is not None:
            h2d_bytes += cu_host.numel() * 4
        d2h_bytes = sum(t.numel() * t.element_size() for t in host_out.values()) + host_lse.numel() * 4
        e2e = {"value": weak_scaling_value(world, w.fwdbwd_flops(), e2e_ms), "unit": UNIT,
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "tokens_per_s": world * w.B * w.T_valid / (e2e_ms * 1e-3),
               "copies": "every step: inputs in, outputs out, on two copy streams overlapping the "
                         "neighbouring steps' compute (double-buffered)",
               "host_link_gbs": link,
               "copy_bound_ms_per_step": round(max(h2d_bytes / (link["h2d"] * 1e9),
                                                   d2h_bytes / (link["d2h"] * 1e9),
                                                   (h2d_bytes + d2h_bytes) / (link["both"] * 1e9)) * 1e3, 3)}

    peaks = measured_peaks()
    unit_flops = w.fwd_flops() / 2.0          # one GEMM over the live causal pairs
    elt = 2
    tensor_bytes = w.B * w.H * w.T * w.d * elt
    ker_work = {
        "fwd": ("tensor", 2 * unit_flops),
        "bwd_dkdv": ("tensor", 4 * unit_flops),
        "bwd_dq": ("tensor", 1 * unit_flops),     # S and dP recomputation is not credited
        "bwd_D": ("hbm", 2 * tensor_bytes + w.B * w.H * w.T * 4),   # dropped below when fused
        "shard": ("hbm", 2 * input_bytes(w, elt)),     # read + write of q, k, v, dO
        "unshard": ("hbm", 2 * input_bytes(w, elt)),   # of o, dq, dk, dv
    }
    if d_fused:
        del ker_work["bwd_D"]
    ker_rep = {}
    for name, (bound, work) in ker_work.items():
        t = ker_ms[name] * 1e-3
        if bound == "tensor":
            ach = work / t / 1e12
            ker_rep[name] = {"ms": ker_ms[name], "bound": "tensor", "achieved": ach, "unit": "TFLOP/s",
                             "frac": ach / peaks["bf16_tflops"],
                             "frac_sustained": ach / peaks["bf16_tflops_sustained"]}
        else:
            ach = work / t / 1e9
            ker_rep[name] = {"ms": ker_ms[name], "bound": "hbm", "achieved": ach, "unit": "GB/s",
                             "frac": ach / peaks["hbm_gbs"]}
    # The standalone SDPAMerger (cpattn_merge) is not on the step's path (the
    # forward merges in its softmax epilogue); it is timed here on its own, on
    # two fp32 partials of the workload's size, and reported beside the step's
    # kernels with its HBM roofline.
    if not args.no_merge:
        n_parts = 2
        o_parts = [torch.randn((Bx, Hx, w.T, w.d), device=dev, dtype=torch.float32) for _ in range(n_parts)]
        l_parts = [torch.randn((Bx, Hx, w.T), device=dev, dtype=torch.float32) for _ in range(n_parts)]
        o_m = torch.empty((Bx, Hx, w.T, w.d), device=dev, dtype=torch.bfloat16)
        l_m = torch.empty((Bx, Hx, w.T), device=dev, dtype=torch.float32)
        for _ in range(3):
            cpattn.merge(o_parts, l_parts, o_m, l_m, stream)
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for _ in range(10):
            cpattn.merge(o_parts, l_parts, o_m, l_m, stream)
        m1.record(stream)
        torch.cuda.synchronize(dev)
        merge_ms = m0.elapsed_time(m1) / 10
        rows = Bx * Hx * w.T
        merge_bytes = n_parts * rows * (w.d + 1) * 4 + rows * (w.d * 2 + 4)
        ach = merge_bytes / (merge_ms * 1e-3) / 1e9
        ker_rep["merge_standalone"] = {"ms": merge_ms, "bound": "hbm", "achieved": ach, "unit": "GB/s",
                                       "frac": ach / peaks["hbm_gbs"],
                                       "note": "cpattn_merge of 2 fp32 partials, timed outside the step"}
        del o_parts, l_parts, o_m, l_m
    dom = max((k_ for k_ in ("fwd", "bwd_dkdv", "bwd_dq", "bwd_D") if k_ in ker_work), key=lambda k: ker_ms[k])
    d = ker_rep[dom]
    traffic, traffic_src = ncu_traffic(w.name, dom) if not rope_flag else (None, "in-kernel RoPE build")
    # The timed region lasts well under a second, so the burst peak applies;
    # the sustained (power-capped, seconds-long) figure is reported beside it.
    roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"],
                "peak": peaks["bf16_tflops"] if d["bound"] == "tensor" else peaks["hbm_gbs"],
                "unit": d["unit"], "frac": d["frac"],
                "traffic": traffic, "traffic_source": traffic_src,
                "peak_source": f"{peaks['source']} "
                               + ("bf16_tflops (burst)" if d["bound"] == "tensor" else "hbm_gbs"),
                "work_per_launch": ker_work[dom][1]}
    if d["bound"] == "tensor":
        roofline["frac_sustained"] = d["frac_sustained"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry(w, oracle_sample(w))

    value = weak_scaling_value(world, w.fwdbwd_flops(), ms)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {**workload_config(w), "parallelism": f"replica per GPU x{world}",
                           "rope_path": ("fused into shard/unshard" if fused else
                                         "inside the attention kernels (forward stores the rotated q, k)"
                                         if rope_flag else "none")},
                "tokens_per_s": world * w.B * w.T_valid / (ms * 1e-3),
                "frac_of_bf16_peak": value / world / peaks["bf16_tflops"],
                "frac_of_bf16_peak_sustained": value / world / peaks["bf16_tflops_sustained"],
                "fwd_tflops": w.fwd_flops() / (ker_ms["fwd"] * 1e-3) / 1e12,
                "e2e": e2e, "roofline": roofline, "kernels": ker_rep, "cpu_baseline": cpu,
                "clocks": clocks, "gpu_launches": launches_per_step * args.steps}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    plan, why = launch_plan(args.gpus, os.environ)
    if plan == "refuse":
        print(f"bench.py: {why}", file=sys.stderr)
        raise SystemExit(2)
    if plan == "relaunch":
        raise SystemExit(subprocess.call(relaunch_cmd(args.gpus, sys.argv[1:], free_port())))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
