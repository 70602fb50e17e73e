"""Benchmark: exact attention forward + backward on one GB300 per process.

One step = the whole hot path on one batch: fa_fwd (O, L) then fa_bwd
(Delta, dK/dV, dQ; at D <= 64 the dQ pass computes Delta and runs first) on
the causal B4 H16 S4096 D64 fp16 workload, inputs resident in HBM.  Prints ONE JSON line (rank 0):

  value     whole-job TFLOP/s over the timed steps, counting 4*B*H*S^2*D / 2
            (causal) for the forward and 2.5x that for the backward;
  e2e       the same metric through the C ABI with host buffers: every step
            copies q, k, v, dO from pinned host memory and O, L, dQ, dK, dV back
            (copy streams and two buffer sets overlap neighbouring steps' copies
            with the kernels);
  roofline  the dominant kernel's algorithmic FLOPs (or bytes) per launch over
            its CUDA-event duration, against the measured peak (kernel times come
            from a second pass of the same steps with events between the
            backward's kernels; the timed steps have none there, since such an
            event keeps the dK/dV pass from overlapping the dQ pass's end);
  cpu_baseline  the fp64 CPU oracle on a bounded sample (rank 0, N = 1).

`--impl reference` times the CPU oracle (the reference arm of this build) on
the same workload, one (b, h) head per step.

`--workload gqa` / `--workload mqa` run the same measurement on the same shape
with 2 K/V heads (8 query heads each) or 1 K/V head (grouped-query and
multi-query attention, fa_fwd_gqa / fa_bwd_gqa); the default is the multi-head
workload above.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU with no
data exchange (weak scaling); value = all ranks' FLOPs / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS and % of GB300 FP16 tensor peak (B4 H16 S4096 D64 causal)"
WORKLOAD = "c2"
WORKLOADS = ("c2", "c4", "c5", "leaderboard", "gqa", "mqa", "varlen", "window", "splitkv")
FLUSH_BYTES = 256 << 20  # > 129 MB L2
_CSRC = "exact_attention_18_gb300/csrc/"
_COMMON = [_CSRC + f for f in ("fa_kernel_common.cuh", "sm103_ptx.cuh", "fa_internal.cuh")]
# The sources each kernel is compiled from: a committed ncu traffic figure is used only while
# these are unchanged since its capture.
KERNEL_SOURCES = {
    "fa_fwd4_kernel": [_CSRC + "fa_fwd4.cu", _CSRC + "fa_softmax.cuh"] + _COMMON,
    "fa_fwd4p_kernel": [_CSRC + "fa_fwd4p.cu", _CSRC + "fa_softmax.cuh"] + _COMMON,
    "fa_fwd_kernel": [_CSRC + "fa_fwd.cu", _CSRC + "fa_softmax.cuh"] + _COMMON,
    "fa_bwd_preprocess_kernel": [_CSRC + "fa_bwd.cu"] + _COMMON,
    "fa_bwd_dkdv_kernel": [_CSRC + "fa_bwd.cu"] + _COMMON,
    "fa_bwd_dq_kernel": [_CSRC + "fa_bwd.cu"] + _COMMON,
}


def is_packed(w):
    return hasattr(w, "lengths")


def head_list(w):
    """Every attention head of the workload as (b, h, rows): B*H heads of S rows, or, for a
    packed batch, H heads per sample of that sample's length."""
    if is_packed(w):
        return [(b, h, n) for b, n in enumerate(w.lengths) for h in range(w.H)]
    return [(b, h, w.S) for b in range(w.B) for h in range(w.H)]


def sq_rows(w):
    """Sum over heads of rows^2 (the S^2 of the FLOP convention, per head)."""
    return float(sum(n * n for _, _, n in head_list(w)))


def band_pairs(n, causal, window):
    """Exact count of visible (query, key) pairs of one head of n rows under a window band."""
    left, right = window
    total = 0
    for i in range(n):
        lo = 0 if left < 0 else max(0, i - left)
        hi = i if causal else (n - 1 if right < 0 else min(n - 1, i + right))
        if causal and right >= 0:
            hi = min(hi, i + right)
        total += max(0, hi - lo + 1)
    return total


def pairs(w):
    """Score pairs the FLOP convention counts: S^2 per head (halved when causal), or, with
    a window band, the exact number of visible pairs."""
    if getattr(w, "window", None) is not None:
        return float(sum(band_pairs(n, w.causal, w.window) for _, _, n in head_list(w)))
    return sq_rows(w) / (2.0 if w.causal else 1.0)


def conv_flops(w):
    """FLOP convention: forward 4*S^2*D per head (halved when causal; with a window band,
    4*D per visible pair), summed over heads (B*H*S^2 fixed length, H * sum of squared
    sample lengths packed); backward 2.5x forward."""
    f = 4.0 * pairs(w) * w.D
    return f, 2.5 * f


PERSISTENT_MAX_S = 6144  # the library's switch between its two D <= 64 forward kernels


def fwd_kernel_name(w, general=False):
    """The forward kernel the library launches for this workload: at D <= 64 the persistent
    two-pipeline kernel for fixed-length sequences of up to 6144 rows, the four-tile kernel for
    longer ones and for packed batches, windows and split-KV (``general``)."""
    if w.D > 64:
        return "fa_fwd_kernel"
    if general or is_packed(w) or getattr(w, "window", None) is not None or w.S > PERSISTENT_MAX_S:
        return "fa_fwd4_kernel"
    return "fa_fwd4p_kernel"


def bwd_fuses_delta(w):
    """Whether the library's dQ pass computes Delta itself (D <= 64, fixed length, no window
    band): the backward then runs the dQ pass first and the dK/dV pass after it, with no
    separate Delta kernel."""
    return w.D <= 64 and not is_packed(w) and getattr(w, "window", None) is None


def bwd_intervals(w):
    """The backward kernels between fa_bwd_marked's marks 0-1, 1-2 and 2-3 (None: no launch)."""
    if bwd_fuses_delta(w):
        return ["fa_bwd_dq_kernel", "fa_bwd_dkdv_kernel", None]
    return ["fa_bwd_preprocess_kernel", "fa_bwd_dkdv_kernel", "fa_bwd_dq_kernel"]


def kernel_work(w, general=False):
    """Algorithmic work per launch of each kernel (FLOPs of its tensor-core GEMMs, or HBM bytes)."""
    units = pairs(w) * w.D
    rows = sum(n for _, _, n in head_list(w))
    work = {
        fwd_kernel_name(w, general): ("tensor", 4.0 * units),        # S = QK^T, O += PV
        "fa_bwd_dkdv_kernel": ("tensor", 8.0 * units),       # S^T, dP^T, dV, dK
        "fa_bwd_dq_kernel": ("tensor", 6.0 * units),         # S, dP, dQ (and Delta's row sums when fused)
    }
    if not bwd_fuses_delta(w):
        work["fa_bwd_preprocess_kernel"] = ("hbm", rows * w.D * 2 * 2 + rows * 4)  # read O, dO; write Delta
    return work


def sources_digest(kernel):
    """Digest of the sources `kernel` is compiled from."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "tensor_tflops": d["bf16_tflops"],
                "tensor_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "tensor_tflops": 1900.0, "tensor_tflops_sustained": 1700.0, "source": "fallback"}


def load_traffic(workload):
    """DRAM bytes per launch from the committed ncu summaries: the kernels captured on this
    workload whose sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        d = json.load(f)
    out = {}
    for kernel, rec in d.get("bytes_per_launch", {}).get(workload, {}).items():
        if kernel in KERNEL_SOURCES and rec.get("sources_digest") == sources_digest(kernel):
            out[kernel] = rec["bytes"]
    return out


class ClockSampler:
    """nvidia-smi clock / throttle sampling every 100 ms while the benchmark runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.marks = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [p for t, p in self.samples if t0 - 0.25 <= t <= t1 + 0.25] or [p for _, p in self.samples]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower().startswith("active")})
        power = [num(p[3]) for p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "power_w_max": max(power) if power else None}


def cpu_oracle_step(inp, w, heads):
    """The fp64 oracle forward + backward on the listed (b, h) heads (test infrastructure).

    With grouped K/V heads, query head h reads K/V head h // (H / H_kv).
    """
    import oracle
    grp = w.H // w.kv_heads
    cu = inp["cu_seqlens"].tolist() if is_packed(w) else None
    for b, h, _ in heads:
        if cu is None:
            q, do = inp["q"][b, h], inp["do"][b, h]
            k, v = inp["k"][b, h // grp], inp["v"][b, h // grp]
        else:
            a, e = cu[b], cu[b + 1]
            q, do = inp["q"][a:e, h], inp["do"][a:e, h]
            k, v = inp["k"][a:e, h // grp], inp["v"][a:e, h // grp]
        win = getattr(w, "window", None)
        oracle.forward(q, k, v, w.causal, w.scale, window=win)
        oracle.backward(q, k, v, do, w.causal, w.scale, window=win)


def head_flops(w, heads):
    """Convention FLOPs (forward + backward) of the listed heads."""
    if getattr(w, "window", None) is not None:
        f = 4.0 * w.D * sum(band_pairs(n, w.causal, w.window) for _, _, n in heads)
    else:
        f = 4.0 * w.D * sum(n * n for _, _, n in heads) * (0.5 if w.causal else 1.0)
    return 3.5 * f


def time_oracle_heads(inp, w, heads):
    """Wall time of the fp64 oracle's forward + backward over `heads`, one head per call,
    after one untimed head (thread pool and allocator warm-up).  The cpu_baseline leg and the
    reference arm both time the oracle this way."""
    cpu_oracle_step(inp, w, heads[:1])
    t0 = time.perf_counter()
    for hd in heads:
        cpu_oracle_step(inp, w, [hd])
    return time.perf_counter() - t0


def cpu_threads():
    import torch
    return {"cores": torch.get_num_threads(), "host_cpus": os.cpu_count()}


def cpu_baseline(inp, w, n_heads: int):
    all_heads = head_list(w)
    heads = [all_heads[i % len(all_heads)] for i in range(n_heads)]
    dt = time_oracle_heads(inp, w, heads)
    return {"value": head_flops(w, heads) / dt / 1e12, "unit": "TFLOP/s", **cpu_threads(), "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd, one head at a time, on {n_heads} of the {len(all_heads)} heads of "
                      f"{w.describe()}, {dt:.2f} s; convention FLOPs of those heads / wall time"}


def cpu_table():
    """The fp64 oracle on the configured workloads' shapes (bounded samples), TFLOP/s by the
    convention FLOPs of what was computed: forward of c1 (all threads and one thread), of one
    c2 head, of 512 sampled rows of one c5 head; forward + backward of one c4 head and of one
    batch entry of c3 at D = 64 and S = 256, 1024, 4096."""
    import torch
    import oracle
    from seeded_inputs import CONFIGS, make_inputs
    rows_out = []

    def timed(case, fn, flops, threads=None):
        old = torch.get_num_threads()
        if threads:
            torch.set_num_threads(threads)
        try:
            fn()  # untimed warm-up
            t0 = time.perf_counter()
            fn()
            dt = time.perf_counter() - t0
        finally:
            torch.set_num_threads(old)
        rows_out.append({"case": case, "TFLOP/s": flops / dt / 1e12, "s": dt, "threads": threads or old})

    def head(w, b=0, h=0):
        inp = make_inputs(w, with_dout=True)
        return [inp[n][b, h] for n in ("q", "k", "v", "do")]

    w = CONFIGS["c1"]
    q, k, v, do = head(w)
    f = 4.0 * w.S * w.S * w.D
    timed("c1 fwd", lambda: oracle.forward(q, k, v, False, w.scale), f)
    timed("c1 fwd, 1 thread", lambda: oracle.forward(q, k, v, False, w.scale), f, threads=1)
    w = CONFIGS["c2"]
    q, k, v, do = head(w)
    timed("c2 fwd, one head", lambda: oracle.forward(q, k, v, True, w.scale), 4.0 * w.S * w.S * w.D / 2)
    w = CONFIGS["c5"]
    q, k, v, do = head(w)
    rows = list(range(w.S - 512, w.S))
    timed("c5 fwd, 512 rows of one head", lambda: oracle.forward_rows(q, k, v, True, w.scale, rows),
          4.0 * w.D * sum(r + 1 for r in rows))
    w = CONFIGS["c4"]
    q, k, v, do = head(w)
    timed("c4 fwd+bwd, one head",
          lambda: (oracle.forward(q, k, v, False, w.scale, row_block=2048),
                   oracle.backward(q, k, v, do, False, w.scale, row_block=2048)), 3.5 * 4.0 * w.S * w.S * w.D)
    for S in (256, 1024, 4096):
        w = CONFIGS[f"c3_d64_s{S}"]
        q, k, v, do = head(w)
        timed(f"c3 D64 S{S} fwd+bwd, one batch entry",
              lambda: (oracle.forward(q, k, v, True, w.scale), oracle.backward(q, k, v, do, True, w.scale)),
              3.5 * 4.0 * S * S * w.D / 2)
    return rows_out


def workload_inputs(w):
    from seeded_inputs import make_inputs, make_packed_inputs
    return make_packed_inputs(w) if is_packed(w) else make_inputs(w, with_dout=True)


def workload_config(w):
    if is_packed(w):
        return {"workload": w.name, "samples": w.batch, "lengths": list(w.lengths), "total_tokens": w.total,
                "max_seqlen": w.max_seqlen, "H": w.H, "H_kv": w.kv_heads, "D": w.D, "causal": w.causal}
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.kv_heads, "S": w.S, "D": w.D, "causal": w.causal}
    if w.window is not None:
        cfg["window"] = list(w.window)
    return cfg


def run_reference(args, w):
    """Reference arm: the CPU oracle as it stands, one head per step, rank 0 only."""
    import torch
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = workload_inputs(w)
    all_heads = head_list(w)
    nh = len(all_heads)
    for i in range(args.warmup):
        cpu_oracle_step(inp, w, [all_heads[i % nh]])
    done = [all_heads[(args.warmup + i) % nh] for i in range(args.steps)]
    t0 = time.perf_counter()
    for hd in done:
        cpu_oracle_step(inp, w, [hd])
    dt = time.perf_counter() - t0
    value = head_flops(w, done) / dt / 1e12
    sample = f"fp64 CPU oracle fwd+bwd of one head of {w.describe()} per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(w), sample_per_step="one (b,h) head"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", **cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-heads", type=int, default=48,
                    help="heads in the CPU oracle baseline sample (48 of c2's 64: about 10-15 s of CPU work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-table", action="store_true",
                    help="add the oracle timed on the configured workloads' shapes to cpu_baseline")
    ap.add_argument("--workload", default=WORKLOAD, choices=WORKLOADS)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import dataclasses
    from seeded_inputs import CONFIGS, PACKED_CONFIGS
    if args.workload in PACKED_CONFIGS:
        w = PACKED_CONFIGS[args.workload]
    else:
        w = dataclasses.replace(CONFIGS[args.workload], backward=True)
    global METRIC
    if args.workload != WORKLOAD:
        METRIC = f"attention fwd/bwd TFLOPS and % of GB300 FP16 tensor peak ({w.describe()})"
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import exact_attention_18_gb300 as fa
    from exact_attention_18_gb300.sharding import job_throughput, max_over_ranks

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    inp = workload_inputs(w)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    packed = is_packed(w)
    H, D, Hkv = w.H, w.D, w.kv_heads
    lse_shape = (H, w.total) if packed else q.shape[:3]
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    if packed:
        cu = inp["cu_seqlens"].to(dev)
        nb, ms, T = w.batch, w.max_seqlen, w.total
        ws_bytes = fa.fa_bwd_varlen_workspace_size(nb, ms, T, H, Hkv, D)
    else:
        B, S = w.B, w.S
        ws_bytes = fa.fa_bwd_gqa_workspace_size(B, H, Hkv, S, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    # Split-KV forward (the splitkv workload): shard count and the partials' workspace.
    n_split = fa.fa_splitkv_num_splits(B, H, S, D) if args.workload == "splitkv" else 0
    split_bytes = fa.fa_fwd_splitkv_workspace_size(B, H, S, D, n_split) if n_split else 0
    split_ws = torch.empty(max(split_bytes, 256), dtype=torch.uint8, device=dev)
    # Kernel launches per step: forward (+ merge when split), Delta (unless the dQ pass computes
    # it), dK/dV (+ partial-sum reduction when the grouped pass splits), dQ.
    delta_bytes = ((H * (w.total if packed else B * S) * 4) + 255) // 256 * 256
    launches_per_step = (3 + (0 if bwd_fuses_delta(w) else 1) + (1 if n_split else 0)
                         + (1 if ws_bytes > delta_bytes else 0))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    dt_code = fa.FA_FP16 if w.dtype == "fp16" else fa.FA_BF16

    win = None if packed else w.window

    def fwd_call(q_, k_, v_, o_, lse_, cu_=None):
        if n_split:
            return fa.fa_fwd_splitkv(q_, k_, v_, o_, lse_, B, H, Hkv, S, D, w.causal, n_split, w.scale, dt_code,
                                     split_ws.data_ptr(), split_bytes, sp)
        if win is not None:
            return fa.fa_fwd_window(q_, k_, v_, o_, lse_, B, H, Hkv, S, D, w.causal, win[0], win[1], w.scale, dt_code,
                                    sp)
        if packed:
            return fa.fa_fwd_varlen(q_, k_, v_, o_, lse_, cu_ or cu.data_ptr(), nb, ms, T, H, Hkv, D, w.causal, w.scale,
                                    dt_code, sp)
        if Hkv == H:
            return fa.fa_fwd(q_, k_, v_, o_, lse_, B, H, S, D, w.causal, w.scale, dt_code, sp)
        return fa.fa_fwd_gqa(q_, k_, v_, o_, lse_, B, H, Hkv, S, D, w.causal, w.scale, dt_code, sp)

    def bwd_call(q_, k_, v_, o_, do_, lse_, dq_, dk_, dv_, marks, cu_=None):
        if win is not None:
            return fa.fa_bwd_window_marked(q_, k_, v_, o_, do_, lse_, dq_, dk_, dv_, B, H, Hkv, S, D, w.causal, win[0],
                                           win[1], w.scale, dt_code, ws.data_ptr(), ws_bytes, sp, marks)
        if packed:
            return fa.fa_bwd_varlen_marked(q_, k_, v_, o_, do_, lse_, dq_, dk_, dv_, cu_ or cu.data_ptr(), nb, ms, T, H, Hkv,
                                           D, w.causal, w.scale, dt_code, ws.data_ptr(), ws_bytes, sp, marks)
        if Hkv == H:
            return fa.fa_bwd_marked(q_, k_, v_, o_, do_, lse_, dq_, dk_, dv_, B, H, S, D, w.causal, w.scale,
                                    dt_code, ws.data_ptr(), ws_bytes, sp, marks)
        return fa.fa_bwd_gqa_marked(q_, k_, v_, o_, do_, lse_, dq_, dk_, dv_, B, H, Hkv, S, D, w.causal, w.scale,
                                    dt_code, ws.data_ptr(), ws_bytes, sp, marks)

    def step(ev=None, inner=False):
        """One step; ev: five events, e0 before the forward, e1 between forward and backward, e4
        after the backward, and with `inner` e2, e3 between the backward's kernels (an event
        between two kernels keeps the second from starting before the first has finished, so
        the timed steps record none there)."""
        if ev is not None:
            ev[0].record(stream)
        st = fwd_call(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
        if st:
            raise RuntimeError(f"forward: {fa.fa_status_string(st)} {fa.fa_last_error_detail()}")
        marks = [e.cuda_event for e in ev[1:5]] if ev is not None and inner else None
        if ev is not None and not inner:
            ev[1].record(stream)
        st = bwd_call(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), marks)
        if st:
            raise RuntimeError(f"backward: {fa.fa_status_string(st)} {fa.fa_last_error_detail()}")
        if ev is not None and not inner:
            ev[4].record(stream)

    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_id = visible.split(",")[local].strip() if visible else str(local)
    sampler = ClockSampler(gpu_id)
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if fa.fa_check_device_errors(sp) != 0:
        raise RuntimeError("device error during warm-up: " + fa.fa_last_error_detail())

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for e in evs + kevs:  # create the CUDA events (torch creates them on first record) before the C side records them
        for x in e:
            x.record(stream)
    barrier()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()  # L2 flush between timed steps, outside the step's events
        step(evs[i])
    barrier()
    t_wall1 = time.time()
    # The same steps again with events between the backward's kernels: each kernel's time.
    for i in range(args.steps):
        flush.zero_()
        step(kevs[i], inner=True)
    torch.cuda.synchronize()
    if fa.fa_check_device_errors(sp) != 0:
        raise RuntimeError("device error during the timed steps: " + fa.fa_last_error_detail())

    slots = [fwd_kernel_name(w, n_split > 0)] + bwd_intervals(w)
    names = [n for n in slots if n is not None]
    per = {n: [] for n in names}
    for e in kevs:
        # fwd = e0->e1 (the forward call); the backward's kernels between the marks e1..e4
        ts = [e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3]), e[3].elapsed_time(e[4])]
        for n, t in zip(slots, ts):
            if n is not None:
                per[n].append(t)
    step_ms = [e[0].elapsed_time(e[4]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    f_fwd, f_bwd = conv_flops(w)
    value = job_throughput(f_fwd + f_bwd, args.steps, world, total_ms) / 1e12
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[4]) for e in evs)
    peaks = load_peaks()
    unsplit = None
    if n_split:
        # The same forward without splitting the keys, for comparison (same protocol).
        ts = []
        for i in range(args.warmup + 20):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, S, D,
                           w.causal, w.scale, dt_code, sp)
            e1.record(stream)
            if st:
                raise RuntimeError(f"fa_fwd: {fa.fa_status_string(st)} {fa.fa_last_error_detail()}")
            if i >= args.warmup:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        unsplit = {"ms": statistics.mean(a.elapsed_time(b) for a, b in ts), "shards": n_split}
    work = kernel_work(w, n_split > 0)
    avg = {n: statistics.mean(per[n]) for n in names}
    dom = max(names, key=lambda n: avg[n])
    kind, amount = work[dom]
    traffic = load_traffic(args.workload).get(dom)
    if kind == "tensor":
        achieved = amount / (avg[dom] * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peaks["tensor_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["tensor_tflops"], "traffic": traffic,
                "peak_note": f"{peaks['source']} bf16 dense burst (fp16 runs at the same nominal rate)"}
    else:
        achieved = amount / (avg[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "peak_note": peaks["source"] + " copy"}

    kernels = {}
    for n in names:
        kd, amt = work[n]
        if kd == "tensor":
            ach = amt / (avg[n] * 1e-3) / 1e12
            kernels[n] = {"ms": avg[n], "TFLOP/s": ach, "frac_of_tensor_peak": ach / peaks["tensor_tflops"]}
        else:
            ach = amt / (avg[n] * 1e-3) / 1e9
            kernels[n] = {"ms": avg[n], "GB/s": ach, "frac_of_hbm_peak": ach / peaks["hbm_gbs"]}
    if "fa_bwd_preprocess_kernel" not in names:
        kernels["fa_bwd_dq_kernel"]["note"] = "computes Delta = rowsum(dO o O) too (no Delta kernel)"

    # ---------------------------------------------------------------- end to end through host buffers
    # Every step copies its inputs q, k, v, dO (and a packed batch's cu_seqlens) from pinned host
    # memory and reads all of its outputs
    # (O, L, dQ, dK, dV) back, inside the timed region.  Two device buffer sets let the copies of
    # neighbouring steps (inputs of step i+1 on one copy stream, outputs of step i-1 on another)
    # overlap step i's kernels, as a training loop would pipeline them.
    e2e = None
    if not args.no_e2e:
        in_names = ("q", "k", "v", "do") + (("cu_seqlens",) if packed else ())
        pin = {n: inp[n].pin_memory() for n in in_names}
        out_shapes = {"o": (o.shape, o.dtype), "lse": (lse.shape, lse.dtype), "dq": (q.shape, q.dtype),
                      "dk": (k.shape, k.dtype), "dv": (k.shape, k.dtype)}
        host_out = [{n: torch.empty(sh, dtype=dt).pin_memory() for n, (sh, dt) in out_shapes.items()}
                    for _ in range(2)]
        dev_in0 = {"q": q, "k": k, "v": v, "do": do}
        if packed:
            dev_in0["cu_seqlens"] = cu
        dev_in = [dev_in0, {n: torch.empty_like(t) for n, t in dev_in0.items()}]
        dev_out = [{"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv},
                   {n: torch.empty(sh, dtype=dt, device=dev) for n, (sh, dt) in out_shapes.items()}]
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
        s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def run_step(bi, bo):
            cu_ = bi["cu_seqlens"].data_ptr() if packed else None
            st = fwd_call(bi["q"].data_ptr(), bi["k"].data_ptr(), bi["v"].data_ptr(), bo["o"].data_ptr(),
                          bo["lse"].data_ptr(), cu_)
            if st:
                raise RuntimeError(f"forward: {fa.fa_status_string(st)} {fa.fa_last_error_detail()}")
            st = bwd_call(bi["q"].data_ptr(), bi["k"].data_ptr(), bi["v"].data_ptr(), bo["o"].data_ptr(),
                          bi["do"].data_ptr(), bo["lse"].data_ptr(), bo["dq"].data_ptr(), bo["dk"].data_ptr(),
                          bo["dv"].data_ptr(), None, cu_)
            if st:
                raise RuntimeError(f"backward: {fa.fa_status_string(st)} {fa.fa_last_error_detail()}")

        def e2e_run(n):
            done_compute, done_d2h = [None, None], [None, None]
            for i in range(n):
                b = i % 2
                with torch.cuda.stream(s_h2d):  # inputs of step i (buffer b was last read by step i-2)
                    if done_compute[b] is not None:
                        s_h2d.wait_event(done_compute[b])
                    for name in pin:
                        dev_in[b][name].copy_(pin[name], non_blocking=True)
                    h_done = torch.cuda.Event()
                    h_done.record(s_h2d)
                stream.wait_event(h_done)
                if done_d2h[b] is not None:  # outputs of step i-2 have left buffer b
                    stream.wait_event(done_d2h[b])
                run_step(dev_in[b], dev_out[b])
                c_done = torch.cuda.Event()
                c_done.record(stream)
                done_compute[b] = c_done
                with torch.cuda.stream(s_d2h):  # outputs of step i
                    s_d2h.wait_event(c_done)
                    for name in host_out[b]:
                        host_out[b][name].copy_(dev_out[b][name], non_blocking=True)
                    d_done = torch.cuda.Event()
                    d_done.record(s_d2h)
                    done_d2h[b] = d_done

        e2e_run(args.warmup)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(s_h2d)
        e2e_run(args.steps)
        e1.record(s_d2h)
        barrier()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
        e2e = {"value": job_throughput(f_fwd + f_bwd, args.steps, world, e2e_ms) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps}
    t_wall2 = time.time()
    sampler.stop()
    # Samples from the device-timed steps and the end-to-end steps (both under load).
    clocks = sampler.summary(t_wall0, t_wall2 if e2e is not None else t_wall1)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, w, args.cpu_heads)
        if args.cpu_table:
            cpu["table"] = cpu_table()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(workload_config(w),
                           global_batch=(w.batch if packed else w.B) * world,
                           seq_len=w.max_seqlen if packed else w.S,
                           parallelism=f"independent x{world}",
                           step=(f"fa_fwd_splitkv ({n_split} shards, merge included in the forward kernel time) + fa_bwd"
                                 if n_split else
                                 "fa_fwd_varlen + fa_bwd_varlen" if packed else
                                 "fa_fwd_window + fa_bwd_window" if win is not None else
                                 "fa_fwd + fa_bwd" if w.kv_heads == w.H else "fa_fwd_gqa + fa_bwd_gqa"),
                           l2="flushed between timed steps (256 MiB write)",
                           flop_convention=("fwd 4*S^2*D per head (/2 causal; S the sample length when packed; "
                                            "4*D per visible pair with a window band), bwd 2.5x fwd")),
            "fwd": {"ms": fwd_ms, "TFLOP/s": f_fwd / (fwd_ms * 1e-3) / 1e12,
                    "frac_of_tensor_peak": f_fwd / (fwd_ms * 1e-3) / 1e12 / peaks["tensor_tflops"]},
            "bwd": {"ms": bwd_ms, "TFLOP/s": f_bwd / (bwd_ms * 1e-3) / 1e12,
                    "frac_of_tensor_peak": f_bwd / (bwd_ms * 1e-3) / 1e12 / peaks["tensor_tflops"]},
            "kernels": kernels,
            **({"fwd_unsplit": unsplit} if unsplit else {}),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
