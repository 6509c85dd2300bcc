"""Benchmark: causal flash attention forward + backward on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole path over one batch: fa_fwd (out, lse) then
fa_bwd (dq, dk, dv) through the C ABI on the long_8k workload (bf16, B=1,
Hq=Hkv=32, S=8192, d=128, causal, synthetic seeded inputs with spike keys).
FLOPs follow the causal convention 2*B*Hq*S^2*d (forward) + 5*B*Hq*S^2*d
(backward), i.e. 4*d (forward) and 10*d (backward) per visible query-key pair
with S^2/2 visible pairs per head; unmasked workloads count Sq*Skv pairs and
a causal query chunk (Sq < Skv, mask aligned to the last key) Sq*Skv - Sq^2/2.
Other workloads (--workload) are timed the same way. Each rank runs its own
replica (no collective on the data path);
`value` is the FLOPs of all ranks divided by the slowest rank's time.

Prints one JSON line (rank 0). `--impl reference` times the fp64 CPU oracle
instead (the reference arm), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import fa_inputs  # noqa: E402

METRIC = "causal attention fwd/bwd TFLOP/s and % of GB300 dense BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
# ex2.approx.ftz.f32 results per clock per SM measured on the GB300 (one
# 1024-thread block per SM, 16 independent chains per thread).
EX2_PER_CLK_SM = 31.9


# ------------------------------------------------------------ arithmetic --
def visible_pairs(Sq, Skv, causal):
    """Query-key pairs per head that the mask leaves visible, by the FLOP
    convention (S^2/2 for causal self-attention)."""
    return Sq * Skv - Sq * Sq / 2 if causal else Sq * Skv


def flops(w, fwd=True, bwd=True):
    """FLOP convention: 4*d per visible pair forward (two GEMMs), 10*d backward
    (five GEMMs); causal self-attention gives 2*B*Hq*S^2*d and 5*B*Hq*S^2*d."""
    base = w.B * w.Hq * visible_pairs(w.S, w.kv_len, w.causal) * w.d
    return (4 * base if fwd else 0) + (10 * base if bwd else 0)


def elem_bytes(w):
    return {"fp32": 4, "fp16": 2, "bf16": 2}[w.dtype]


def tensor_bytes(B, H, S, d, esize):
    return B * H * S * d * esize


def score_matrix_bytes(B, H, S, esize):
    """Bytes of one materialised [B, H, S, S] score (or probability) matrix,
    the tensor flash attention never stores."""
    return B * H * S * S * esize


def fwd_algorithmic_bytes(w):
    """Compulsory HBM traffic of one forward: read Q, K, V, write O and LSE."""
    e = elem_bytes(w)
    return (2 * tensor_bytes(w.B, w.Hq, w.S, w.d, e) + 2 * tensor_bytes(w.B, w.Hkv, w.kv_len, w.d, e)
            + w.B * w.Hq * w.S * 4)


def bwd_algorithmic_bytes(w):
    """Compulsory HBM traffic of one backward: read Q, K, V, O, dO, LSE, write
    dQ, dK, dV."""
    e = elem_bytes(w)
    q = tensor_bytes(w.B, w.Hq, w.S, w.d, e)
    kv = tensor_bytes(w.B, w.Hkv, w.kv_len, w.d, e)
    return 4 * q + 4 * kv + w.B * w.Hq * w.S * 4


def hbm_side(nbytes, nflops, ms, peak_tflops, hbm_gbs):
    """A call against the HBM roof: its algorithmic bytes over its time, its
    arithmetic intensity and the ridge point between the tensor and HBM roofs
    (None without a time or bytes)."""
    if not ms or not nbytes:
        return None
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"achieved_gbs": gbs, "peak_gbs": hbm_gbs, "frac": gbs / hbm_gbs,
            "intensity_flop_per_byte": nflops / nbytes,
            "ridge_flop_per_byte": peak_tflops * 1e12 / (hbm_gbs * 1e9)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {"fa_fwd_kernel": ("fa_fwd.cu", "ptx.cuh", "fa_internal.h"),
                  "fa_bwd_kernel": ("fa_bwd.cu", "ptx.cuh", "fa_internal.h"),
                  "fa_fwd_pair_kernel": ("fa_fwd_pair.cu", "ptx.cuh", "fa_internal.h"),
                  "fa_decode_kernel": ("fa_decode.cu", "ptx.cuh", "fa_internal.h", "fa_decode.h")}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "causal_flash_attention_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch recorded from an ncu capture in
    profiles/dram_traffic.txt (lines: kernel workload source-hash bytes ...),
    valid only while the kernel's sources hash the same as when it was
    captured; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and \
                parts[1] == workload and parts[2] == want:
            return float(parts[3])
    return None


# --------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        under_load = [x for x in sm if x > 0.5 * max(sm)]
        return {"sm_mhz": statistics.median(under_load), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle --
def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = [i["num_threads"] for i in info if i.get("user_api") == "blas"]
        if n:
            return int(max(n)), "BLAS threads (threadpoolctl)"
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0)), "cores available (BLAS default)"
    except AttributeError:
        return os.cpu_count() or 1, "cores available (BLAS default)"


def cpu_model():
    """The host CPU's model name as lscpu or /proc/cpuinfo report it (None if neither does)."""
    try:
        import subprocess
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def oracle_inputs(w, heads):
    """float64 copies of batch 0, query heads [0, heads) and their key/value heads."""
    import torch
    q, k, v, do = fa_inputs.make_inputs(w)
    G = w.Hq // w.Hkv
    f64 = lambda t: t.to(torch.float64).numpy()
    return [(f64(q[:1, h:h + 1]), f64(k[:1, h // G:h // G + 1]), f64(v[:1, h // G:h // G + 1]),
             f64(do[:1, h:h + 1])) for h in range(heads)]


def oracle_block(w, max_rows):
    """The leading block the oracle samples: query rows 0..r-1 and the keys
    they see (causal: keys up to row position r-1 + kv_offset; unmasked: all
    keys). Under the causal mask this is an exact piece of the full problem."""
    r = min(w.S, max_rows)
    kv = min(w.kv_len, r + w.kv_len - w.S) if w.causal else w.kv_len
    return r, kv


def oracle_one_thread(name="tiny_fp32"):
    """Seconds and FLOPs of the fp64 oracle's dense forward + backward of a
    whole small workload with BLAS held to one thread (a child process: the
    thread count is fixed when numpy loads its BLAS)."""
    code = ("import time, fa_inputs, oracle, bench\n"
            f"w = fa_inputs.WORKLOADS[{name!r}]\n"
            "q, k, v, do = (t.double().numpy() for t in fa_inputs.make_inputs(w))\n"
            "oracle.forward(q, k, v, w.causal, w.scale)\n"
            "t0 = time.perf_counter()\n"
            "oracle.forward(q, k, v, w.causal, w.scale)\n"
            "oracle.backward(q, k, v, do, w.causal, w.scale)\n"
            "print(time.perf_counter() - t0, bench.flops(w, True, w.backward))\n")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                             text=True, timeout=300)
        sec, fl = (float(x) for x in out.stdout.split())
        return sec, fl
    except Exception:
        return None, None


def oracle_sample(w, head_inputs, block):
    """Time the fp64 oracle's dense forward + backward on `block` (rows, keys)
    of one head of workload `w`. Returns (seconds, flops of that block by the
    same convention)."""
    import oracle
    r, kv = block
    Q, DO = (x[:, :, :r] for x in (head_inputs[0], head_inputs[3]))
    K, V = (x[:, :, :kv] for x in (head_inputs[1], head_inputs[2]))
    t0 = time.perf_counter()
    oracle.forward(Q, K, V, w.causal, w.scale)
    if w.backward:
        oracle.backward(Q, K, V, DO, w.causal, w.scale)
    dt = time.perf_counter() - t0
    return dt, (14 if w.backward else 4) * visible_pairs(r, kv, w.causal) * w.d


# ------------------------------------------------------------ multi-rank --
def max_over_ranks(times, dist, device):
    """Each timing's maximum over all ranks (the slowest rank sets the job's
    time); `dist` None means a single process."""
    import torch
    t = torch.tensor(times, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tflops(flops_per_rank_step, world, ms_per_step):
    """Whole-job throughput: every rank's FLOPs per step over the slowest
    rank's step time (weak scaling: each rank runs its own replica)."""
    return flops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------- other workloads --
# Timed after the headline workload in the default run, each on its own inputs
# with its own warm-up: the other shapes the metric is quoted on (d = 64 and
# short sequences, grouped-query heads, fp16 at 32K positions) and the
# unmasked, chunked-prefill, decode and paged-decode rows.
PER_CONFIG = ["gpt2_small", "gqa_qwen3", "fp16_32k", "gqa_qwen3_nc", "long_8k_nc", "prefill_8k",
              "decode_8k", "spec_32k", "decode_8k_paged"]


def _calls_for(fa, w, dev):
    """(fwd(), bwd() or None, input bytes) for workload w on fresh device
    buffers; the same entry points run_gpu times."""
    import torch
    q, k, v, do = fa_inputs.make_inputs(w)
    table = None
    if w.page_size:
        k, v, table, _ = fa_inputs.make_paged(k, v, w.page_size, seed=w.page_size)
        table = table.to(dev)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    out = torch.empty_like(qd)
    lse = torch.empty(qd.shape[:3], dtype=torch.float32, device=dev)
    nbytes = sum(x.numel() * x.element_size() for x in (qd, kd, vd, dod))
    if w.decode:
        n = fa.fa_fwd_splitkv_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.kv_len, w.d, 0)
        ws = torch.empty(n, dtype=torch.uint8, device=dev) if n else None
        if w.page_size:
            fwd = lambda: fa.fa_fwd_splitkv_paged(qd, kd, vd, table, out, lse, w.kv_len, w.causal,
                                                  w.scale, 0, ws)
        else:
            fwd = lambda: fa.fa_fwd_splitkv(qd, kd, vd, out, lse, w.causal, w.scale, 0, ws)
        return fwd, None, nbytes
    same = w.S == w.kv_len
    fwd = (lambda: fa.fa_fwd(qd, kd, vd, out, lse, w.causal, w.scale)) if same else \
        (lambda: fa.fa_fwd_kv(qd, kd, vd, out, lse, w.causal, w.scale))
    if not w.backward:
        return fwd, None, nbytes
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = fa.workspace_for(qd, kd)
    bwd = (lambda: fa.fa_bwd(qd, kd, vd, out, dod, lse, dq, dk, dv, ws, w.causal, w.scale)) \
        if same else \
        (lambda: fa.fa_bwd_kv(qd, kd, vd, out, dod, lse, dq, dk, dv, ws, w.causal, w.scale))
    fwd()
    return fwd, bwd, nbytes


# GPU-side wait queued ahead of a timed call's start event, so that the host
# issues the call while the GPU is still busy: the events then bracket the
# call's device time alone (~50 us at 2 GHz, above any call's host time)
HOST_COVER_CYCLES = 100_000


def time_config(fa, w, dev, peaks, warm=20, calls=50, forward_only=False):
    """Per-call CUDA-event times (median over `calls`, after `warm` untimed
    calls) of the workload's
    forward and backward entry points, with its roofline against the measured
    peaks. Inputs smaller than L2 get an L2 flush (a 256 MiB write) before
    every timed call; larger ones need none. A short GPU-side wait before the
    start event covers the call's host issue time, which is reported apart
    (`host_us`, the Python binding plus the C entry point)."""
    import torch
    fwd, bwd, nbytes = _calls_for(fa, w, dev)
    flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev) if nbytes <= L2_BYTES else None
    res = {"workload": w.describe(),
           "l2": "flushed before every timed call" if flush is not None else
                 f"inputs ({nbytes / 2**20:.0f} MiB) larger than L2; no flush"}
    peak, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    if forward_only:
        bwd = None
    for name, fn, fl, nb in (("fwd", fwd, flops(w, True, False), fwd_algorithmic_bytes(w)),
                             ("bwd", bwd, flops(w, False, True), bwd_algorithmic_bytes(w))):
        if fn is None:
            continue
        for _ in range(warm):
            fn()
        torch.cuda.synchronize(dev)
        ts, hs = [], []
        for _ in range(calls):
            if flush is not None:
                flush.fill_(1)
            torch.cuda._sleep(HOST_COVER_CYCLES)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            t0 = time.perf_counter()
            fn()
            hs.append((time.perf_counter() - t0) * 1e6)
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        entry = {"ms": ms, "ms_mean": statistics.mean(ts), "host_us": statistics.median(hs)}
        if w.decode:   # HBM-bound: the split-KV forward streams K and V once
            gbs = nb / (ms * 1e-3) / 1e9
            entry.update({"bound": "hbm", "achieved_gbs": gbs, "frac": gbs / hbm,
                          "peak_gbs": hbm})
        else:
            tf = fl / (ms * 1e-3) / 1e12
            entry.update({"bound": "tensor", "tflops": tf, "frac": tf / peak,
                          "hbm_side": hbm_side(nb, fl, ms, peak, hbm)})
        res[name] = entry
    torch.cuda.synchronize(dev)
    return res


def time_sustained(step, dev, stream, seconds, ms_per_step, local_rank):
    """Back-to-back steps for about `seconds`, timed with CUDA events around
    the whole run, clocks sampled meanwhile."""
    import torch
    n = max(10, int(seconds * 1e3 / max(ms_per_step, 1e-3)))
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
    return n, a.elapsed_time(b), clocks.summary()


# ---------------------------------------------------------------- GPU arm --
def run_gpu(args, w, rank, world, local_rank):
    import torch
    import causal_flash_attention_gb300 as fa

    fa.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    q, k, v, do = fa_inputs.make_inputs(w)
    if w.page_size:   # K and V become the paged caches (block table on the device)
        k, v, table, _ = fa_inputs.make_paged(k, v, w.page_size, seed=w.page_size)
        tables = [table.to(dev), table.to(dev)]
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    out = torch.empty_like(qd)
    lse = torch.empty(qd.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = fa.workspace_for(qd, kd)
    stream = torch.cuda.current_stream(dev)
    # self-attention through fa_fwd / fa_bwd; separate lengths through the *_kv
    # calls; decode workloads (few query rows) through the split-KV forward
    fwd_call = fa.fa_fwd if w.S == w.kv_len else fa.fa_fwd_kv
    bwd_call = fa.fa_bwd if w.S == w.kv_len else fa.fa_bwd_kv
    dec_ws_bytes = 0
    if w.decode:
        dec_ws_bytes = fa.fa_fwd_splitkv_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.kv_len, w.d, 0)
        dec_ws = [torch.empty(max(dec_ws_bytes, 1), dtype=torch.uint8, device=dev) for _ in range(2)]

        def fwd_call(q_, k_, v_, o_, l_, causal, scale, st, _ws=dec_ws):
            ws_ = _ws[1] if (q_.data_ptr() != qd.data_ptr()) else _ws[0]
            if w.page_size:   # k_, v_ are the paged caches; the block table rides along
                fa.fa_fwd_splitkv_paged(q_, k_, v_, tables[0 if q_.data_ptr() == qd.data_ptr() else 1],
                                        o_, l_, w.kv_len, causal, scale, 0,
                                        ws_ if dec_ws_bytes else None, st)
            else:
                fa.fa_fwd_splitkv(q_, k_, v_, o_, l_, causal, scale, 0,
                                  ws_ if dec_ws_bytes else None, st)

    def step():
        fwd_call(qd, kd, vd, out, lse, w.causal, w.scale, stream)
        if w.backward:
            bwd_call(qd, kd, vd, out, dod, lse, dq, dk, dv, ws, w.causal, w.scale, stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    status = fa.fa_last_device_status(stream)
    if status:
        raise RuntimeError(f"device status {status} after warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with ClockSampler(local_rank) as clocks:
        barrier()
        for s in range(K):
            ev[s][0].record(stream)
            fwd_call(qd, kd, vd, out, lse, w.causal, w.scale, stream)
            ev[s][1].record(stream)
            if w.backward:
                bwd_call(qd, kd, vd, out, dod, lse, dq, dk, dv, ws, w.causal, w.scale, stream)
            ev[s][2].record(stream)
        barrier()
        total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
        fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
        fwd_med = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
        bwd_med = statistics.median(e[1].elapsed_time(e[2]) for e in ev)

        # End to end through the public API with host buffers: every step
        # copies its inputs from pinned host memory, runs fa_fwd + fa_bwd and
        # copies every result back to pinned host memory. Steps are pipelined
        # over two device buffer sets: step k's host-to-device copies (one copy
        # stream) and step k-1's device-to-host copies (another) overlap step
        # k's kernels, as a caller streaming batches would run them.
        hq, hk, hv, hdo = (x.pin_memory() for x in (q, k, v, do))
        h_out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        h_lse = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
        h_dq = torch.empty(q.shape, dtype=q.dtype).pin_memory()
        h_dk = torch.empty(k.shape, dtype=k.dtype).pin_memory()
        h_dv = torch.empty(v.shape, dtype=v.dtype).pin_memory()
        ins_h = (hq, hk, hv, hdo) if w.backward else (hq, hk, hv)
        outs_h = (h_out, h_lse, h_dq, h_dk, h_dv) if w.backward else (h_out, h_lse)
        h2d = sum(x.numel() * x.element_size() for x in ins_h)
        d2h = sum(x.numel() * x.element_size() for x in outs_h)
        # at least 32 pipelined steps: with few, the first step's uploads and
        # the last step's downloads (which nothing overlaps) dominate the time
        K2 = 0 if args.no_e2e else max(32, K // 4)
        link = None
        if K2:
            sets = []
            for sidx in range(2):
                if sidx == 0:
                    ins_d = (qd, kd, vd, dod)
                    outs_d = (out, lse, dq, dk, dv)
                    ws_d = ws
                else:
                    ins_d = tuple(torch.empty_like(x) for x in (qd, kd, vd, dod))
                    outs_d = tuple(torch.empty_like(x) for x in (out, lse, dq, dk, dv))
                    ws_d = torch.empty_like(ws)
                sets.append((ins_d, outs_d, ws_d))
            s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
            ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set landed
            ev_comp = [torch.cuda.Event() for _ in range(2)]   # kernels of set done
            ev_out = [torch.cuda.Event() for _ in range(2)]    # results of set copied back
            started = [False, False]

            def e2e_step(kk):
                sidx = kk % 2
                (iq, ik, iv, ido), (oo, ol, oq, okk, ov), wsd = sets[sidx]
                with torch.cuda.stream(s_h2d):
                    if started[sidx]:
                        s_h2d.wait_event(ev_comp[sidx])    # step k-2 has read this set
                    for dst, src in zip((iq, ik, iv, ido), ins_h):
                        dst.copy_(src, non_blocking=True)
                    ev_in[sidx].record(s_h2d)
                stream.wait_event(ev_in[sidx])
                if started[sidx]:
                    stream.wait_event(ev_out[sidx])        # step k-2's results copied out
                fwd_call(iq, ik, iv, oo, ol, w.causal, w.scale, stream)
                if w.backward:
                    bwd_call(iq, ik, iv, oo, ido, ol, oq, okk, ov, wsd, w.causal, w.scale, stream)
                ev_comp[sidx].record(stream)
                with torch.cuda.stream(s_d2h):
                    s_d2h.wait_event(ev_comp[sidx])
                    for dst, src in zip(outs_h, (oo, ol, oq, okk, ov)):
                        dst.copy_(src, non_blocking=True)
                    ev_out[sidx].record(s_d2h)
                started[sidx] = True

            for kk in range(2):
                e2e_step(kk)
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s_h2d)
            for kk in range(K2):
                e2e_step(kk)
            e1.record(s_d2h)
            barrier()
            e2e_ms = e0.elapsed_time(e1) / K2

            # the host link alone: one step's input copies, then its result
            # copies, each timed by itself on its copy stream (best of three)
            def time_copies(cs, pairs):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(cs)
                with torch.cuda.stream(cs):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
                b.record(cs)
                torch.cuda.synchronize(dev)
                return a.elapsed_time(b)
            link = {"h2d_gbs": max(h2d / (time_copies(s_h2d, zip(sets[0][0], ins_h)) * 1e-3) / 1e9
                                   for _ in range(3)),
                    "d2h_gbs": max(d2h / (time_copies(s_d2h, zip(outs_h, sets[0][1])) * 1e-3) / 1e9
                                   for _ in range(3)),
                    "note": "best of 3 isolated copies of one step's inputs / results"}
        else:
            e2e_ms = float("nan")
    status = fa.fa_last_device_status(stream)
    if status:
        raise RuntimeError(f"device status {status} in the timed region")

    sustained = None
    if args.sustain_s > 0:
        n_s, ms_s, clk_s = time_sustained(step, dev, stream, args.sustain_s, total_ms / K, local_rank)
        sustained = {"steps": n_s, "total_ms": ms_s, "clocks": clk_s}
    per_config = {}
    if not args.no_per_config and w.name == "long_8k" and not args.heads:
        peaks, _ = load_peaks()
        for name in PER_CONFIG:
            per_config[name] = time_config(fa, fa_inputs.WORKLOADS[name], dev, peaks)
        # the CTA-pair forward (tcgen05 cta_group::2) on the headline shape, for
        # comparison with the single-CTA forward that fa_fwd runs by default
        prev = os.environ.get("FA_FWD_CTA_PAIR")
        os.environ["FA_FWD_CTA_PAIR"] = "1"
        try:
            per_config["long_8k_cta_pair_forward"] = time_config(
                fa, fa_inputs.WORKLOADS["long_8k"], dev, peaks, forward_only=True)
        finally:
            if prev is None:
                del os.environ["FA_FWD_CTA_PAIR"]
            else:
                os.environ["FA_FWD_CTA_PAIR"] = prev
    status = fa.fa_last_device_status(stream)
    if status:
        raise RuntimeError(f"device status {status} in the sustained or per-workload timing")

    total_ms, fwd_ms, bwd_ms, e2e_ms, fwd_med, bwd_med = max_over_ranks(
        [total_ms, fwd_ms, bwd_ms, e2e_ms, fwd_med, bwd_med], dist, dev)
    return dict(total_ms=total_ms, fwd_ms=fwd_ms, bwd_ms=bwd_ms, e2e_ms=e2e_ms, e2e_steps=K2,
                fwd_med_ms=fwd_med, bwd_med_ms=bwd_med,
                h2d=h2d, d2h=d2h, link=link, clocks=clocks.summary(), dist=dist,
                launches_per_fwd=(2 if dec_ws_bytes else 1), sustained=sustained,
                per_config=per_config)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long_8k", choices=sorted(fa_inputs.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer timing")
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back steps timed after the main region (0: skip)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other workloads after long_8k")
    ap.add_argument("--heads", type=int, default=0,
                    help="override Hq (and Hkv in the same ratio): a smaller case of the same "
                         "workload, e.g. for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    w = fa_inputs.WORKLOADS[args.workload]
    if args.heads:
        import dataclasses
        G = w.Hq // w.Hkv
        if args.heads % G:
            ap.error(f"--heads must be a multiple of {G}")
        w = dataclasses.replace(w, Hq=args.heads, Hkv=args.heads // G)
    peaks, peak_src = load_peaks()
    step_flops = flops(w, True, w.backward)
    e = elem_bytes(w)
    in_bytes = 2 * tensor_bytes(w.B, w.Hq, w.S, w.d, e) + 2 * tensor_bytes(w.B, w.Hkv, w.kv_len, w.d, e)
    l2_note = (f"inputs {'larger' if in_bytes > L2_BYTES else 'NOT larger'} than L2: "
               f"Q,K,V,dO = {in_bytes / 2**20:.0f} MiB read per step vs "
               f"{L2_BYTES / 2**20:.0f} MiB L2; no flush")
    config = {"workload": w.describe(), "global_batch": w.B * world, "seq_len": w.S,
              "heads": [w.Hq, w.Hkv], "head_dim": w.d, "causal": w.causal,
              "parallelism": f"replicas x{world}", "l2": l2_note}
    if w.kv_len != w.S:
        config["kv_len"] = w.kv_len

    if args.impl == "reference":
        if rank != 0:
            return
        cores, how = cpu_threads()
        block = oracle_block(w, 2048 if w.causal else 512)
        inputs = oracle_inputs(w, min(w.Hq, 4))
        times = []
        for i in range(args.warmup + args.steps):
            dt, fl = oracle_sample(w, inputs[i % len(inputs)], block)
            if i >= args.warmup:
                times.append(dt)
        sec = statistics.mean(times)
        value = fl / sec / 1e12
        sample = (f"per step: fp64 dense forward{' + softmax-Jacobian backward' if w.backward else ''} "
                  f"of the leading block (query rows 0..{block[0] - 1}, keys 0..{block[1] - 1}) "
                  f"of one query head of {w.name}, heads 0..{len(inputs) - 1} in turn; "
                  f"{fl / 1e9:.2f} GFLOP by the same convention")
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                                 "cores_source": how, "cpu_model": cpu_model(), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line))
        return

    r = run_gpu(args, w, rank, world, local_rank)
    if rank != 0:
        if r["dist"] is not None:
            r["dist"].destroy_process_group()
        return
    K = args.steps
    ms_per_step = r["total_ms"] / K
    value = job_tflops(step_flops, world, ms_per_step)
    fwd_tf = flops(w, True, False) / (r["fwd_ms"] * 1e-3) / 1e12
    bwd_tf = flops(w, False, True) / (r["bwd_ms"] * 1e-3) / 1e12 if w.backward else None
    e2e_tf = job_tflops(step_flops, world, r["e2e_ms"]) if r["e2e_ms"] == r["e2e_ms"] else None
    peak = peaks["bf16_tflops"]
    hbm = peaks["hbm_gbs"]
    traffic = recorded_traffic("fa_bwd_kernel", w.name)
    if args.heads:
        traffic = None
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else w.dtype,
        "data": "synthetic (seeded N(0,1)-based inputs, no dataset)", "config": config,
        "pct_of_peak": {"step": 100 * value / world / peak, "fwd": 100 * fwd_tf / peak,
                        "bwd": (100 * bwd_tf / peak) if bwd_tf else None,
                        "peak_tflops": peak, "peak_source": f"{peak_src} bf16_tflops (burst)",
                        "step_vs_sustained": 100 * value / world / peaks["bf16_tflops_sustained"]},
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"],
        "per_call_median": {"fwd_ms": r["fwd_med_ms"],
                            "bwd_ms": r["bwd_med_ms"] if w.backward else None,
                            "fwd_tflops": flops(w, True, False) / (r["fwd_med_ms"] * 1e-3) / 1e12,
                            "bwd_tflops": (flops(w, False, True) / (r["bwd_med_ms"] * 1e-3) / 1e12
                                           if w.backward else None)},
        "roofline": {
            "kernel": "fa_bwd_kernel (timed as the fa_bwd call: D pre-pass + main kernel + dQ convert)",
            "bound": "tensor", "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s",
            "frac": (bwd_tf / peak) if bwd_tf else None, "traffic": traffic,
            "traffic_unit": "bytes per launch (dram read + write)",
            "algorithmic_bytes": bwd_algorithmic_bytes(w),
            "peak_source": f"{peak_src} bf16_tflops (burst)",
            "hbm_side": hbm_side(bwd_algorithmic_bytes(w), flops(w, False, True), r["bwd_ms"],
                                 peak, hbm) if w.backward else None,
        },
        "roofline_fwd": {
            "kernel": "fa_fwd_kernel (one launch per fa_fwd call)", "bound": "tensor",
            "achieved": fwd_tf, "peak": peak, "unit": "TFLOP/s", "frac": fwd_tf / peak,
            "traffic": None if args.heads else recorded_traffic("fa_fwd_kernel", w.name),
            "algorithmic_bytes": fwd_algorithmic_bytes(w),
            "hbm_side": hbm_side(fwd_algorithmic_bytes(w), flops(w, True, False), r["fwd_ms"],
                                 peak, hbm),
        },
        "exp_ceiling": {
            "exps_per_step": int(w.B * w.Hq * visible_pairs(w.S, w.kv_len, w.causal)),
            "ex2_per_clk_per_sm": EX2_PER_CLK_SM,
            "fwd_floor_ms": (w.B * w.Hq * visible_pairs(w.S, w.kv_len, w.causal))
                            / (EX2_PER_CLK_SM * 152 * 2.07e9) * 1e3,
            "note": "forward: one ex2 per visible score; floor at 152 SMs x 2.07 GHz",
        },
        "e2e": {"value": e2e_tf, "unit": "TFLOP/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e_ms"],
                "host_link_gbs": r["link"],
                "pipelining": "2 device buffer sets; H2D of step k and D2H of step k-1 on copy "
                              "streams overlap step k's kernels",
                "steps": r["e2e_steps"]},
        "gpu_launches": (r["launches_per_fwd"] + (3 if w.backward else 0)) * K,
        "clocks": r["clocks"],
    }
    if r["sustained"]:
        sus = r["sustained"]
        sus_ms = sus["total_ms"] / sus["steps"]
        sus_tf = job_tflops(step_flops, world, sus_ms)
        mhz = sus["clocks"]["sm_mhz"]
        line["sustained"] = {
            "steps": sus["steps"], "seconds": sus["total_ms"] / 1e3, "ms_per_step": sus_ms,
            "tflops": sus_tf, "frac_of_sustained_peak": sus_tf / world / peaks["bf16_tflops_sustained"],
            "sustained_peak_tflops": peaks["bf16_tflops_sustained"],
            "frac_of_burst_peak": sus_tf / world / peak,
            "clocks": sus["clocks"],
            "ms_x_median_mhz": sus_ms * mhz if mhz else None,
            "burst_ms_x_median_mhz": ms_per_step * r["clocks"]["sm_mhz"] if r["clocks"]["sm_mhz"] else None,
            "note": "back-to-back steps after the burst region; CUDA events around the whole run",
        }
    if r["per_config"]:
        line["per_config"] = r["per_config"]
    if not w.backward:   # forward-only workload: the forward kernel is the whole step
        line["roofline"] = dict(line["roofline_fwd"])
    if w.decode:
        # few query rows: the split-KV forward streams K and V once; HBM-bound
        gbs = fwd_algorithmic_bytes(w) / (r["fwd_ms"] * 1e-3) / 1e9
        line["roofline"] = {
            "kernel": "fa_decode_kernel + decode_merge_kernel (timed as the fa_fwd_splitkv call)",
            "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"],
            "traffic": None if args.heads else recorded_traffic("fa_decode_kernel", w.name),
            "traffic_unit": "bytes per launch (dram read + write)",
            "algorithmic_bytes": fwd_algorithmic_bytes(w),
            "peak_source": f"{peak_src} hbm_gbs (copy)",
        }
        line["roofline_fwd"] = dict(line["roofline"])
    if world == 1 and not args.no_cpu_baseline:
        cores, how = cpu_threads()
        total_t, total_f = 0.0, 0
        # the dense oracle holds rows x keys float64 matrices
        block = oracle_block(w, 8192 if w.causal else 4096)
        for hin in oracle_inputs(w, 2):
            dt, fl = oracle_sample(w, hin, block)
            total_t += dt
            total_f += fl
        line["cpu_baseline"] = {
            "value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": cores,
            "cores_source": how, "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"fp64 dense forward{' + softmax-Jacobian backward' if w.backward else ''} "
                      f"of the leading block (query rows 0..{block[0] - 1}, keys 0..{block[1] - 1}) "
                      f"of query heads 0 and 1 of {w.name} (all of each head when the block "
                      f"covers it): {total_f / 1e9:.1f} GFLOP by the same convention in "
                      f"{total_t:.2f} s"}
        rate = total_f / total_t
        line["cpu_baseline"]["extrapolated_full_step_s"] = step_flops / rate
        line["cpu_baseline"]["extrapolation"] = (
            f"the whole {w.name} step ({step_flops / 1e12:.2f} TFLOP) at the sampled rate: "
            "an extrapolation, not measured")
        sec1, fl1 = oracle_one_thread()
        if sec1:
            line["cpu_baseline"]["tiny_fp32_one_thread"] = {
                "seconds": sec1, "gflop": fl1 / 1e9, "tflops": fl1 / sec1 / 1e12, "threads": 1,
                "sample": "fp64 dense forward + softmax-Jacobian backward of the whole tiny_fp32 "
                          "workload (fp32 B=1 Hq=Hkv=2 S=128 d=64), BLAS held to one thread"}
    if r["dist"] is not None:
        r["dist"].destroy_process_group()
    print(json.dumps(line))


if __name__ == "__main__":
    main()
