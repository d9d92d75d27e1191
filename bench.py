#!/usr/bin/env python3
"""Benchmark of the attention hot path on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
  * attn_fwd on the long-context causal prefill workload (B=1, H=32, N=8192,
    d=128, bf16, Q scaled by 2, causal), and
  * attn_decode_paged on the paged decode workload (B=64, Hq=32, Hkv=8, d=128,
    lengths U[1024, 32768], page_size=16, split-KV with LSE combine).
``value`` is the forward leg's throughput in TFLOP/s (algorithmic FLOPs: 4*d per
visible (query, key) pair and head); the decode leg's HBM GB/s is reported under
``decode``. Both legs are timed with CUDA events on the stream they launch on;
inputs are larger than L2, so no flush is needed between steps.
After the timed steps, attn_decode_paged_fp8 runs the same decode workload with
e4m3 key/value caches for as many timed calls; its GB/s (algorithmic bytes of the
8-bit caches) is reported under ``decode_fp8``, outside ``value``. Likewise
attn_fwd_fp8 on the long causal prefill with e4m3 Q/K/V, under ``prefill_fp8``, and
attn_fwd_hd on the same geometry with head dims (192, 128), under ``prefill_hd``, and
attn_fwd with head width 256 on the same geometry, under ``prefill_d256``.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
With --gpus N > 1 the script runs under torch.distributed.run, one rank per GPU,
each rank processing its own copy of the workload (weak scaling, no data-path
collective). ``--impl reference`` times the float64 CPU oracle on a bounded
sample of the same workload on this machine's host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import workloads as W  # noqa: E402

METRIC = "attn fwd TFLOP/s (bf16 hd128 causal) & paged-decode HBM GB/s vs roofline"
FWD_KERNEL = "attn_fwd_kernel"
DEC_KERNEL = "decode_split_kernel"
DEC8_KERNEL = "decode_split_fp8_kernel"
FWD8_KERNEL = "attn_fwd_kernel<128, 0, 1>"
FWDHD_KERNEL = "attn_fwd_kernel<192, 0, 0, 128, 96>"
FWDW_KERNEL = "attn_fwd_wide_kernel"


# Reduced cases for profiler captures: inputs larger than the L2, a few GB at most on the device.
PROFILE_CASES = {
    "long_causal_h16": lambda: W.PrefillCase("long_causal_h16", 1, 16, 16, 8192, 8192, 128, 1.0 / math.sqrt(128),
                                             True, W.long_causal().seed, 2.0),
    "long_causal_h32": W.long_causal,
    "long_causal_d256": lambda: W.PrefillCase("long_causal_d256", 1, 32, 32, 8192, 8192, 256, 1.0 / 16.0, True,
                                              W.long_causal().seed, 2.0),
    "long_causal_hd": lambda: dataclasses.replace(W.long_causal(), name="long_causal_hd", d=192,
                                                  scale=1.0 / math.sqrt(192), dv=128),
    "long_causal_e4m3": W.long_causal,  # Q/K/V as e4m3 codes
    "prefill_2k": lambda: W.prefill(False),
    "prefill_2k_causal": lambda: W.prefill(True),
    "varlen_gqa": W.varlen_gqa,
    "tiny": W.tiny,
    # the paged decode workload's first 16 sequences (864 MB of bf16 cache, 432 MB of e4m3)
    "decode_b16": lambda: dataclasses.replace(W.decode(), name="decode_b16", B=16, seqlens=W.decode().seqlens[:16]),
    "decode_b16_e4m3": lambda: dataclasses.replace(W.decode_fp8(), name="decode_b16_e4m3", B=16,
                                                   seqlens=W.decode().seqlens[:16]),
}


def run_profile_case(name, options=()):
    """attn_fwd (attn_fwd_hd, attn_fwd_fp8 or the paged decode, as the case needs) four times on
    one case, after the library options given; the fourth launch is the one to capture."""
    import torch
    import exact_softmax_attention_gb300 as A
    for opt in options:
        n, v = opt.split("=", 1)
        A.attn_set_option(n, float(v))
    c = PROFILE_CASES[name]()
    if isinstance(c, W.DecodeCase):
        run_profile_decode(A, c)
        return
    fp8 = name.endswith("_e4m3")
    dev16 = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    if fp8:
        q8, k8, v8, qs, ks, vs = c.generate_fp8("e4m3")
        Q, K, V = (torch.from_numpy(a).cuda() for a in (q8, k8, v8))
    else:
        q, k, v = c.generate()
        Q, K, V = dev16(q), dev16(k), dev16(v)
    dv = c.dv if c.dv else c.d
    O = torch.empty((c.total_q, c.Hq, dv), dtype=torch.bfloat16, device="cuda")
    L = torch.empty((c.total_q, c.Hq), dtype=torch.float32, device="cuda")
    CU = None if c.cu_seqlens is None else torch.from_numpy(c.cu_seqlens).cuda()
    nq, nk = (c.Nq, c.Nk) if CU is None else (c.total_q, c.total_k)
    for _ in range(4):
        if fp8:
            A.attn_fwd_fp8(Q, K, V, O, L, c.B, c.Hq, c.Hkv, nq, nk, c.d, c.scale, c.causal, CU, None, "e4m3", qs, ks, vs)
        elif dv != c.d:
            A.attn_fwd_hd(Q, K, V, O, L, c.B, c.Hq, c.Hkv, nq, nk, c.d, dv, c.scale, c.causal, CU, None)
        else:
            A.attn_fwd(Q, K, V, O, L, c.B, c.Hq, c.Hkv, nq, nk, c.d, c.scale, c.causal, CU)
    torch.cuda.synchronize()
    st = A.attn_get_device_status()
    if st != 0:
        raise RuntimeError(A.status_string(st))
    print(json.dumps({"profile_case": name, "flops_per_call": c.flops()}))


def run_profile_decode(A, c):
    import torch
    dev16 = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    if c.kv_fmt == "bf16":
        q, kc, vc, pt, sl = c.generate()
        KC, VC = dev16(kc), dev16(vc)
    else:
        q, kc, vc, pt, sl, kds, vds = c.generate_fp8()
        KC, VC = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    Q, PT, SL = dev16(q), torch.from_numpy(pt).cuda(), torch.from_numpy(sl).cuda()
    O = torch.empty((c.B, c.Hq, c.d), dtype=torch.bfloat16, device="cuda")
    L = torch.empty((c.B, c.Hq), dtype=torch.float32, device="cuda")
    for _ in range(4):
        if c.kv_fmt == "bf16":
            A.attn_decode_paged(Q, KC, VC, PT, SL, c.page_size, O, L, None, c.B, c.Hq, c.Hkv, c.d, c.max_pages,
                                c.num_pages, c.scale, 0)
        else:
            A.attn_decode_paged_fp8(Q, KC, VC, PT, SL, c.page_size, O, L, None, c.B, c.Hq, c.Hkv, c.d, c.max_pages,
                                    c.num_pages, c.scale, 0, c.kv_fmt, kds, vds)
    torch.cuda.synchronize()
    st = A.attn_get_device_status()
    if st != 0:
        raise RuntimeError(A.status_string(st))
    print(json.dumps({"profile_case": c.name, "bytes_per_call": c.bytes()}))


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU-baseline leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--option", action="append", default=[], metavar="NAME=VALUE",
                    help="library tuning option (attn_set_option) applied before timing; repeatable")
    ap.add_argument("--profile-case", default=None, choices=sorted(PROFILE_CASES),
                    help="run one named workload four times and exit (for ncu captures of one launch)")
    ap.add_argument("--legs", default="all",
                    help="comma-separated legs to run besides the step (decode_fp8, prefill_fp8, prefill_hd, "
                         "prefill_d256, prefill_tiny, prefill_2k, prefill_2k_causal, prefill_varlen_gqa, "
                         "prefill_correction_warp, prefill_unroll_kv, rescale), 'all' or 'none'")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def kernel_sources(kernel: str):
    """The source files a kernel is compiled from."""
    if kernel.startswith("decode"):
        return ["attn_decode.cu", "decode_maps.cuh", "ptx.cuh", "kernels.cuh"]
    return ["attn_fwd.cu", "ptx.cuh", "kernels.cuh"]


def source_sha(kernel: str) -> str:
    """Hash of the sources a kernel is compiled from (to tell whether a profile is stale)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_softmax_attention_gb300", "csrc")
    for name in kernel_sources(kernel):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(leg: str):
    """Per-launch DRAM bytes of the kernel of a bench leg (``step_prefill``, ``step_decode``, or
    the leg's key in the JSON line) from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            e = json.load(f)[leg]
        return float(e["dram_bytes_per_launch"]) if e.get("source_sha") == source_sha(e["kernel"]) else None
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clocks and clock-event (throttle) reasons while the timed region runs.

    Reads NVML through ctypes every ~2 ms (read-only queries); falls back to nvidia-smi
    at 100 ms when NVML cannot be loaded. Changes no GPU setting."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.samples = []  # (sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._handle = None
        self.source = None

    def _open_nvml(self):
        import ctypes
        import torch
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        uuid = getattr(torch.cuda.get_device_properties(self.dev), "uuid", None)
        if uuid is not None:
            ok = nv.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(h)) == 0
        if not ok:
            cnt = ctypes.c_uint()
            if nv.nvmlDeviceGetCount_v2(ctypes.byref(cnt)) == 0 and cnt.value == 1:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) == 0
        if not ok:
            return False
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nvml, self._handle = nv, h
        return True

    def _run_nvml(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        get_r = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(clk)) == 0:
                r = rs.value if get_r(self._handle, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            time.sleep(0.002)

    def _run_smi(self):
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or "0"
        try:
            proc = subprocess.Popen(["nvidia-smi", "-i", vis, f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                     "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        bits = [0x8, 0x40, 0x20, 0x4]
        while not self._stop.is_set():
            line = proc.stdout.readline()
            if not line:
                break
            parts = [x.strip() for x in line.split(",")]
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except (ValueError, IndexError):
                continue
            self.max_mhz = mx
            mask = sum(b for b, v in zip(bits, parts[2:6]) if v.lower().startswith("active"))
            self.samples.append((sm, mask))
        proc.terminate()

    def __enter__(self):
        try:
            use_nvml = self._open_nvml()
        except (OSError, AttributeError):
            use_nvml = False
        self.source = "nvml" if use_nvml else "nvidia-smi"
        self._t = threading.Thread(target=self._run_nvml if use_nvml else self._run_smi, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": self.source}
        mask = 0
        for _, r in self.samples:
            mask |= r
        return {"sm_mhz": statistics.median(x for x, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if mask & b), "samples": len(self.samples),
                "source": self.source}


def max_over_ranks(x: float, world: int, device) -> float:
    """Maximum of a per-rank timing over all ranks (a tiny all-reduce; no data-path collective)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def decode_sample_case(dc, n_seq):
    """The first ``n_seq`` sequences of a decode workload as a workload of their own (same
    lengths, same recipe), so a CPU sample does not have to materialise the whole pool."""
    return W.DecodeCase(dc.name + "_sample", n_seq, dc.Hq, dc.Hkv, dc.d, dc.page_size, dc.seqlens[:n_seq].copy(),
                        dc.max_pages, dc.scale, dc.seed)


# ------------------------------------------------------------------ oracle (CPU) legs

def oracle_fwd_sample(case, q, k, v, n_rows, seed, n_threads):
    import oracle
    T = case.total_q
    rng = np.random.default_rng(seed)
    rows = rng.choice(T * case.Hq, size=n_rows, replace=False).astype(np.int64)
    tok = rows // case.Hq
    pairs = int(np.minimum(tok + 1, case.Nk).sum())  # causal, Nq == Nk
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, case.B, case.Hq, case.Hkv, case.Nq, case.Nk, case.d, case.scale, case.causal,
                    rows=rows, n_threads=n_threads)
    dt = time.perf_counter() - t0
    return 4 * case.d * pairs, dt


def oracle_decode_sample(case, inputs, n_seq, n_threads):
    import oracle
    q, kc, vc, pt, sl = inputs
    sel = np.arange(n_seq)
    t0 = time.perf_counter()
    oracle.attn_decode_paged(q[sel], kc, vc, pt[sel], sl[sel], case.page_size, n_seq, case.Hq, case.Hkv, case.d,
                             case.max_pages, case.scale, n_threads=n_threads)
    dt = time.perf_counter() - t0
    L = sl[sel].astype(np.int64)
    nbytes = int(L.sum()) * case.Hkv * case.d * 4 + 2 * n_seq * case.Hq * case.d * 2 + n_seq * case.Hq * 4
    return nbytes, dt


def cpu_baseline(fwd_case, fwd_inputs, dec_case, dec_inputs, budget_s=15.0):
    """The oracle as it stands, on a bounded sample sized for ~budget_s of CPU time."""
    threads = os.cpu_count() or 1
    # calibrate on a sample large enough to amortise the thread start-up, then size the
    # measured one for ~85 % of the budget (the decode sample takes the rest)
    n0 = 512
    f0, t0 = oracle_fwd_sample(fwd_case, *fwd_inputs, n0, 7, threads)
    rate = f0 / max(t0, 1e-6)
    rows = int(min(fwd_case.total_q * fwd_case.Hq, max(n0, n0 * (budget_s * 0.85) / max(t0, 1e-6))))
    f, t = oracle_fwd_sample(fwd_case, *fwd_inputs, rows, 8, threads)
    d_seq = 2
    b, td = oracle_decode_sample(dec_case, dec_inputs, d_seq, threads)
    return {
        "value": f / t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
        "sample": f"{rows} random (token, head) rows of the long causal prefill ({f / 1e9:.1f} GFLOP, {t:.1f} s); "
                  f"decode: {d_seq} sequences ({b / 1e9:.2f} GB, {td:.1f} s)",
        "decode_gbs": b / td / 1e9,
        "calibration_gflops": rate / 1e9,
    }


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return
    fc = W.long_causal()
    dc = decode_sample_case(W.decode(), 1)
    fin = fc.generate()
    din = dc.generate()
    threads = os.cpu_count() or 1
    # each step: ~4 s of oracle work on a row sample of the prefill and one decode sequence
    f0, t0 = oracle_fwd_sample(fc, *fin, 64, 1, threads)
    rows = int(max(64, 64 * 3.0 / max(t0, 1e-6)))
    for i in range(args.warmup):
        oracle_fwd_sample(fc, *fin, rows, 100 + i, threads)
    tot_f = tot_t = tot_b = tot_td = 0.0
    for i in range(args.steps):
        f, t = oracle_fwd_sample(fc, *fin, rows, 200 + i, threads)
        b, td = oracle_decode_sample(dc, din, 1, threads)
        tot_f += f
        tot_t += t
        tot_b += b
        tot_td += td
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": (tot_t + tot_td) / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "long_causal_prefill+paged_decode", "sample": f"{rows} rows/step, 1 decode seq/step"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} random (token, head) rows of the long causal prefill and one decode "
                                   f"sequence per step"},
        "decode": {"value": tot_b / tot_td / 1e9, "unit": "GB/s"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg

class Timer:
    """CUDA-event timing of repeated library calls on one stream, with the device status
    checked after every timed leg (a watchdog timeout or a bad index fails the run)."""

    def __init__(self, A, stream, barrier):
        import torch
        self.torch, self.A, self.stream, self.barrier = torch, A, stream, barrier

    def check(self, what):
        st = self.A.attn_get_device_status(self.stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"device status after {what}: {self.A.status_string(st)}")

    def per_call_ms(self, fn, calls, warmup, what, flush=None):
        """Average ms of one call. With ``flush`` (a callable that overwrites more than the L2)
        each call is timed alone between its own events, with the flush outside them."""
        torch = self.torch
        for _ in range(warmup):
            fn()
        self.barrier()
        if flush is None:
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(self.stream)
            for _ in range(calls):
                fn()
            e.record(self.stream)
            self.barrier()
            ms = s.elapsed_time(e)
        else:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
            for s, e in evs:
                flush()
                s.record(self.stream)
                fn()
                e.record(self.stream)
            self.barrier()
            ms = sum(s.elapsed_time(e) for s, e in evs)
        self.check(what)
        return ms / calls


def tensor_leg(name, workload, flops, ms, calls, launches, peak, peak_source, kernel, world, extra=None):
    ach = flops / (ms * 1e-3) / 1e12
    leg = {"value": world * ach, "unit": "TFLOP/s", "ms_per_call": ms, "calls": calls, "gpu_launches": launches,
           "workload": workload, "flops_per_call": flops,
           "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                        "traffic": ncu_traffic(name), "kernel": kernel,
                        "peak_source": peak_source}}
    if extra:
        leg.update(extra)
    return name, leg


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import exact_softmax_attention_gb300 as A

    for opt in args.option:
        name, value = opt.split("=", 1)
        A.attn_set_option(name, float(value))
    legs_wanted = set(args.legs.split(",")) if args.legs not in ("all", "none") else (
        set() if args.legs == "none" else None)

    def want(leg):
        return legs_wanted is None or leg in legs_wanted

    hbm, bf16, src = peaks()
    fc, dc = W.long_causal(), W.decode()
    q, k, v = fc.generate()
    dq, kc, vc, pt, sl = dc.generate()

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        Q, K, V = to_dev(q), to_dev(k), to_dev(v)
        O = torch.empty((fc.total_q, fc.Hq, fc.d), dtype=torch.bfloat16, device=dev)
        LSE = torch.empty((fc.total_q, fc.Hq), dtype=torch.float32, device=dev)
        DQ, KC, VC = to_dev(dq), to_dev(kc), to_dev(vc)
        PT, SL = torch.from_numpy(pt).to(dev), torch.from_numpy(sl).to(dev)
        DO = torch.empty((dc.B, dc.Hq, dc.d), dtype=torch.bfloat16, device=dev)
        DLSE = torch.empty((dc.B, dc.Hq), dtype=torch.float32, device=dev)
    stream.synchronize()
    s_handle = stream.cuda_stream

    def fwd_on(q_, k_, v_, o_, lse_):
        A.attn_fwd(q_, k_, v_, o_, lse_, fc.B, fc.Hq, fc.Hkv, fc.Nq, fc.Nk, fc.d, fc.scale, fc.causal, None, s_handle)

    def dec_on(q_, kc_, vc_, pt_, sl_, o_, lse_):
        A.attn_decode_paged(q_, kc_, vc_, pt_, sl_, dc.page_size, o_, lse_, s_handle, dc.B, dc.Hq, dc.Hkv, dc.d,
                            dc.max_pages, dc.num_pages, dc.scale, 0)

    def fwd():
        fwd_on(Q, K, V, O, LSE)

    def dec():
        dec_on(DQ, KC, VC, PT, SL, DO, DLSE)

    _, max_splits = A.attn_decode_plan(dc.B, dc.Hq, dc.Hkv, dc.max_pages, dc.page_size, 0)
    launches_per_step = 1 + (2 if max_splits > 1 else 1)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    timer = Timer(A, stream, barrier)
    for _ in range(args.warmup):
        fwd()
        dec()
    timer.check("warm-up")

    # ---------------------------------------------------------------- the timed step
    K_ = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K_)]
    barrier()
    with ClockSampler(dev) as clk:
        t_wall0 = time.perf_counter()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(K_):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            dec()
            ev[i][2].record(stream)
        end.record(stream)
        barrier()
        t_wall = time.perf_counter() - t_wall0
    timer.check("timed region")
    total_ms = start.elapsed_time(end)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in ev)

    total_ms = max_over_ranks(total_ms, world, dev)
    fwd_ms = max_over_ranks(fwd_ms, world, dev)
    dec_ms = max_over_ranks(dec_ms, world, dev)

    extra = {}
    mx = lambda x: max_over_ranks(x, world, dev)

    # ---------------------------------------------------------------- legs outside `value`
    if want("decode_fp8"):
        dc8 = W.decode_fp8()
        _, kc8, vc8, _, _, kds, vds = dc8.generate_fp8()
        with torch.cuda.stream(stream):
            KC8, VC8 = torch.from_numpy(kc8).to(dev), torch.from_numpy(vc8).to(dev)
        stream.synchronize()
        del kc8, vc8

        def dec8():
            A.attn_decode_paged_fp8(DQ, KC8, VC8, PT, SL, dc8.page_size, DO, DLSE, s_handle, dc8.B, dc8.Hq, dc8.Hkv,
                                    dc8.d, dc8.max_pages, dc8.num_pages, dc8.scale, 0, dc8.kv_fmt, kds, vds)

        ms = mx(timer.per_call_ms(dec8, K_, args.warmup, "the FP8 decode leg"))
        ach = dc8.bytes() / (ms * 1e-3) / 1e9
        extra["decode_fp8"] = {
            "value": world * ach, "unit": "GB/s", "ms_per_call": ms, "calls": K_,
            "gpu_launches": K_ * (launches_per_step - 1),
            "workload": "paged decode as above with e4m3 key/value caches (per-tensor descales)",
            "bytes_per_call": dc8.bytes(), "speedup_vs_bf16_decode": (dec_ms / K_) / ms,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "traffic": ncu_traffic("decode_fp8"), "kernel": DEC8_KERNEL, "peak_source": f"{src} copy"}}
        del KC8, VC8

    if want("prefill_fp8"):
        q8, k8, v8, qds, kds8, vds8 = fc.generate_fp8("e4m3")
        with torch.cuda.stream(stream):
            Q8, K8, V8 = (torch.from_numpy(a).to(dev) for a in (q8, k8, v8))
        stream.synchronize()

        def fwd8():
            A.attn_fwd_fp8(Q8, K8, V8, O, LSE, fc.B, fc.Hq, fc.Hkv, fc.Nq, fc.Nk, fc.d, fc.scale, fc.causal, None,
                           s_handle, "e4m3", qds, kds8, vds8)

        ms = mx(timer.per_call_ms(fwd8, K_, args.warmup, "the FP8 forward leg"))
        name, leg = tensor_leg("prefill_fp8", "long causal prefill as above with e4m3 Q/K/V (per-tensor descales)",
                               fc.flops(), ms, K_, K_, bf16 * 4.0 / 3.0,
                               f"{src} bf16 burst x 4/3 (half the FLOPs in fp8 at 2x, half in f16 at 1x)",
                               FWD8_KERNEL, world, {"speedup_vs_bf16_prefill": (fwd_ms / K_) / ms})
        extra[name] = leg

    if want("prefill_hd"):
        hc = W.PrefillCase("long_causal_hd", fc.B, fc.Hq, fc.Hkv, fc.Nq, fc.Nk, 192, 1.0 / math.sqrt(192), True,
                           fc.seed, fc.q_mult, dv=128)
        hq, hk, hv = hc.generate()
        with torch.cuda.stream(stream):
            HQ, HK, HV = to_dev(hq), to_dev(hk), to_dev(hv)
            HO = torch.empty((hc.total_q, hc.Hq, 128), dtype=torch.bfloat16, device=dev)
        stream.synchronize()

        def fwd_hd():
            A.attn_fwd_hd(HQ, HK, HV, HO, LSE, hc.B, hc.Hq, hc.Hkv, hc.Nq, hc.Nk, 192, 128, hc.scale, True, None,
                          s_handle)

        ms = mx(timer.per_call_ms(fwd_hd, K_, args.warmup, "the (192, 128) forward leg"))
        name, leg = tensor_leg("prefill_hd", "long causal prefill B1 H32 N8192 with head dims (192, 128), bf16",
                               hc.flops(), ms, K_, K_, bf16, f"{src} bf16 burst", FWDHD_KERNEL, world)
        extra[name] = leg
        del HQ, HK, HV, HO

    if want("prefill_d256"):
        wc = W.PrefillCase("long_causal_d256", fc.B, fc.Hq, fc.Hkv, fc.Nq, fc.Nk, 256, 1.0 / math.sqrt(256), True,
                           fc.seed, fc.q_mult)
        wq, wk, wv = wc.generate()
        with torch.cuda.stream(stream):
            WQ, WK, WV = to_dev(wq), to_dev(wk), to_dev(wv)
            WO = torch.empty((wc.total_q, wc.Hq, 256), dtype=torch.bfloat16, device=dev)
        stream.synchronize()
        del wq, wk, wv

        def fwd_w():
            A.attn_fwd(WQ, WK, WV, WO, LSE, wc.B, wc.Hq, wc.Hkv, wc.Nq, wc.Nk, 256, wc.scale, True, None, s_handle)

        ms = mx(timer.per_call_ms(fwd_w, K_, args.warmup, "the d = 256 forward leg"))
        name, leg = tensor_leg("prefill_d256", "long causal prefill B1 H32 N8192 with head width 256, bf16",
                               wc.flops(), ms, K_, K_, bf16, f"{src} bf16 burst", FWDW_KERNEL, world)
        extra[name] = leg
        del WQ, WK, WV, WO

    # the other prefill configurations: tiny (C1), prefill B2 H16 N2048 non-causal and causal
    # (C2), packed GQA (C4, with the heaviest-first order across sequences and without it).
    # C1 and C2 fit in the L2, so each call is timed alone after a write of 512 MB.
    flush_buf = None

    def flush():
        with torch.cuda.stream(stream):  # ordered with the calls it separates
            flush_buf.zero_()

    small = [("prefill_tiny", W.tiny(), True), ("prefill_2k", W.prefill(False), True),
             ("prefill_2k_causal", W.prefill(True), True), ("prefill_varlen_gqa", W.varlen_gqa(), False)]
    for name, c, fits_l2 in small:
        if not want(name):
            continue
        if fits_l2 and flush_buf is None:
            with torch.cuda.stream(stream):
                flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        cq, ck, cv = c.generate()
        with torch.cuda.stream(stream):
            CQ, CK, CV = to_dev(cq), to_dev(ck), to_dev(cv)
            CO = torch.empty((c.total_q, c.Hq, c.d), dtype=torch.bfloat16, device=dev)
            CL = torch.empty((c.total_q, c.Hq), dtype=torch.float32, device=dev)
            CU = None if c.cu_seqlens is None else torch.from_numpy(c.cu_seqlens).to(dev)
        stream.synchronize()
        nq, nk = (c.Nq, c.Nk) if CU is None else (c.total_q, c.total_k)

        def call(c=c, CQ=CQ, CK=CK, CV=CV, CO=CO, CL=CL, CU=CU, nq=nq, nk=nk):
            A.attn_fwd(CQ, CK, CV, CO, CL, c.B, c.Hq, c.Hkv, nq, nk, c.d, c.scale, c.causal, CU, s_handle)

        calls = K_ if not fits_l2 else max(K_, 50)
        ms = mx(timer.per_call_ms(call, calls, args.warmup, f"the {name} leg", flush if fits_l2 else None))
        desc = {"prefill_tiny": "tiny B1 H2 N256 d64 non-causal", "prefill_2k": "prefill B2 H16 N2048 d128 non-causal",
                "prefill_2k_causal": "prefill B2 H16 N2048 d128 causal",
                "prefill_varlen_gqa": "packed GQA: 8 sequences U[512,4096], Hq32 Hkv8 d128 causal"}[name]
        kern = "attn_fwd_kernel<64, 0, 0>" if c.d == 64 else FWD_KERNEL
        lx = {"l2": "each call after a 512 MB write (inputs fit in the L2)" if fits_l2 else "inputs larger than L2"}
        if name == "prefill_varlen_gqa":
            A.attn_set_option("packed_order", 0)
            try:
                ms_plain = mx(timer.per_call_ms(call, calls, args.warmup, "the plain-order packed leg"))
            finally:
                A.attn_set_option("packed_order", 1)
            lx["plain_order"] = {"value": world * c.flops() / (ms_plain * 1e-3) / 1e12, "unit": "TFLOP/s",
                                 "ms_per_call": ms_plain,
                                 "order": "sequences in the given order, each one's blocks heaviest first"}
            lx["sorted_order_gain"] = ms_plain / ms
        extra[name] = tensor_leg(name, desc, c.flops(), ms, calls, calls, bf16, f"{src} bf16 burst", kern, world,
                                 lx)[1]
        del CQ, CK, CV, CO, CL
    del flush_buf

    # the two measured design alternatives of the long causal forward, each as its own leg:
    # the correction warp (option correction = 1) and unroll-KV (option unroll_kv = 1)
    for name, opt, desc in (("prefill_correction_warp", "correction",
                             "long causal prefill as the step, O rescaled by a request-driven correction warp"),
                            ("prefill_unroll_kv", "unroll_kv",
                             "long causal prefill as the step, last P V of a work tile and first S of the next "
                             "in one burst")):
        if not want(name):
            continue
        before = A.attn_get_option(opt)
        A.attn_set_option(opt, 1)
        try:
            ms = mx(timer.per_call_ms(fwd, K_, args.warmup, f"the {name} leg"))
        finally:
            A.attn_set_option(opt, before)
        extra[name] = tensor_leg(name, desc, fc.flops(), ms, K_, K_, bf16, f"{src} bf16 burst", FWD_KERNEL, world,
                                 {"vs_default_step": (fwd_ms / K_) / ms})[1]

    # ---------------------------------------------------------------- rescale rate (untimed)
    if want("rescale"):
        rates = {}
        A.attn_set_option("count", 1)
        try:
            A.attn_read_counters()
            for name, c in (("long_causal", fc), ("prefill_2k_causal", W.prefill(True)),
                            ("prefill_2k", W.prefill(False))):
                if c is fc:
                    fwd()
                else:
                    cq, ck, cv = c.generate()
                    with torch.cuda.stream(stream):
                        CQ, CK, CV = to_dev(cq), to_dev(ck), to_dev(cv)
                        CO = torch.empty((c.total_q, c.Hq, c.d), dtype=torch.bfloat16, device=dev)
                        CL = torch.empty((c.total_q, c.Hq), dtype=torch.float32, device=dev)
                    A.attn_fwd(CQ, CK, CV, CO, CL, c.B, c.Hq, c.Hkv, c.Nq, c.Nk, c.d, c.scale, c.causal, None,
                               s_handle)
                dec_all, raised, _, _, dec1, ores = A.attn_read_counters()
                rates[name] = {"warp_steps": dec_all, "steps_after_first": dec1, "o_rescales": ores,
                               "rescale_rate": ores / max(dec1, 1), "skipped": 1.0 - ores / max(dec1, 1)}
        finally:
            A.attn_set_option("count", 0)
        extra["rescale"] = {"threshold_log2": A.attn_get_option("rescale_threshold"), "per_workload": rates,
                            "note": "softmax warp steps (32 rows x one key tile) after the first key tile of their "
                                    "Q tile, and how many of them rescaled O"}

    # ---------------------------------------------------------------- end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, A, dev, stream, barrier, world, K_, fc, dc, (q, k, v), (dq, kc, vc, pt, sl),
                      (Q, K, V, O, LSE), (DQ, KC, VC, PT, SL, DO, DLSE), fwd_on, dec_on, mx)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    fwd_avg_s = fwd_ms / K_ * 1e-3
    dec_avg_s = dec_ms / K_ * 1e-3
    f_ach = fc.flops() / fwd_avg_s / 1e12
    d_ach = dc.bytes() / dec_avg_s / 1e9
    value = world * K_ * fc.flops() / (fwd_ms * 1e-3) / 1e12
    dvalue = world * K_ * dc.bytes() / (dec_ms * 1e-3) / 1e9
    opts = {n: A.attn_get_option(n) for n in ("correction", "unroll_kv", "rescale_threshold", "exp_poly")}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K_, "warmup": args.warmup,
        "ms_per_step": total_ms / K_, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "long_causal_prefill(B1,H32,N8192,d128,causal,Qx2)+paged_decode(B64,Hq32,Hkv8,d128,"
                               "L~U[1024,32768],page16)",
                   "prefill_flops_per_step": fc.flops(), "decode_bytes_per_step": dc.bytes(),
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}",
                   "decode_splits_max": max_splits, "forward_options": opts},
        "roofline": {"bound": "tensor", "achieved": f_ach, "peak": bf16, "unit": "TFLOP/s", "frac": f_ach / bf16,
                     "traffic": ncu_traffic("step_prefill"), "kernel": FWD_KERNEL, "peak_source": f"{src} bf16 burst"},
        "decode": {"value": dvalue, "unit": "GB/s", "ms_per_step": dec_ms / K_,
                   "roofline": {"bound": "hbm", "achieved": d_ach, "peak": hbm, "unit": "GB/s", "frac": d_ach / hbm,
                                "traffic": ncu_traffic("step_decode"), "kernel": DEC_KERNEL,
                                "peak_source": f"{src} copy"}},
        "prefill_ms_per_step": fwd_ms / K_,
        "gpu_launches": K_ * launches_per_step,
        "clocks": clk.summary(),
        "wall_s_timed": t_wall,
    }
    line.update(extra)
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(fc, (q, k, v), dc, (dq, kc, vc, pt, sl))
    if args.option:
        line["config"]["options"] = dict(o.split("=", 1) for o in args.option)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(torch, A, dev, stream, barrier, world, steps, fc, dc, fin, din, fdev, ddev, fwd_on, dec_on, mx):
    """Both legs end to end from pinned host buffers: every step copies its inputs to the
    device, runs the call and copies the outputs back, inside the timed region. Steps are
    pipelined over two device buffer sets and three streams (host-to-device copies, compute,
    device-to-host copies), so step i+1's inputs travel while step i computes and step i-1's
    outputs return, as a serving loop would overlap them."""
    n = max(3, min(steps, 20))  # enough steps that filling and draining the pipeline weigh little
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def pin(a):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.pin_memory()

    def leg(host_in, dev_sets, host_out_shapes, call):
        h_in = [pin(a) for a in host_in]
        h_out = [[torch.empty(sh, dtype=dt).pin_memory() for sh, dt in host_out_shapes] for _ in range(2)]
        t_in, t_comp, t_out = [], [], []
        barrier()
        start, end = ev(), ev()
        start.record(stream)
        h2d_s.wait_event(start)
        for i in range(n):
            b = dev_sets[i % 2]
            if i >= 2:
                h2d_s.wait_event(t_comp[i - 2][1])  # the set's inputs were last read by step i-2
            e0, e1 = ev(), ev()
            e0.record(h2d_s)
            with torch.cuda.stream(h2d_s):
                for dst, src in zip(b["in"], h_in):
                    (dst.view(torch.int16) if dst.dtype == torch.bfloat16 else dst).copy_(src, non_blocking=True)
            e1.record(h2d_s)
            t_in.append((e0, e1))
            stream.wait_event(e1)
            if i >= 2:
                stream.wait_event(t_out[i - 2][1])  # its outputs of step i-2 have left the device
            c0, c1 = ev(), ev()
            c0.record(stream)
            call(b)
            c1.record(stream)
            t_comp.append((c0, c1))
            d2h_s.wait_event(c1)
            o0, o1 = ev(), ev()
            o0.record(d2h_s)
            with torch.cuda.stream(d2h_s):
                for dst, src in zip(h_out[i % 2], b["out"]):
                    dst.copy_(src, non_blocking=True)
            o1.record(d2h_s)
            t_out.append((o0, o1))
        stream.wait_event(t_out[-1][1])
        end.record(stream)
        barrier()
        st = A.attn_get_device_status(stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"device status after the end-to-end leg: {A.status_string(st)}")
        for o in h_out[(n - 1) % 2]:
            if o.dtype.is_floating_point and not torch.isfinite(o.float()).all():
                raise RuntimeError("non-finite output in the end-to-end leg")
        total = mx(start.elapsed_time(end))
        in_ms = sum(a.elapsed_time(b) for a, b in t_in) / n
        out_ms = sum(a.elapsed_time(b) for a, b in t_out) / n
        bi = sum(t.numel() * t.element_size() for t in h_in)
        bo = sum(t.numel() * t.element_size() for t in h_out[0])
        return total, bi, bo, in_ms, out_ms

    Q, K, V, O, LSE = fdev
    sets_f = [{"in": [Q, K, V], "out": [O, LSE]},
              {"in": [torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)],
               "out": [torch.empty_like(O), torch.empty_like(LSE)]}]
    tf, bif, bof, inf_ms, outf_ms = leg(fin, sets_f, [(O.shape, torch.bfloat16), (LSE.shape, torch.float32)],
                                        lambda b: fwd_on(*b["in"], *b["out"]))
    del sets_f
    DQ, KC, VC, PT, SL, DO, DLSE = ddev
    sets_d = [{"in": [DQ, KC, VC, PT, SL], "out": [DO, DLSE]},
              {"in": [torch.empty_like(x) for x in (DQ, KC, VC, PT, SL)],
               "out": [torch.empty_like(DO), torch.empty_like(DLSE)]}]
    td, bid, bod, ind_ms, outd_ms = leg(din, sets_d, [(DO.shape, torch.bfloat16), (DLSE.shape, torch.float32)],
                                        lambda b: dec_on(*b["in"], *b["out"]))
    del sets_d
    return {"value": world * n * fc.flops() / (tf * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": bif + bid, "d2h_bytes_per_step": bof + bod, "steps": n,
            "pipelined": "2 device buffer sets; H2D, compute and D2H on three streams",
            "prefill": {"ms_per_step": tf / n, "h2d_gbs": bif / (inf_ms * 1e-3) / 1e9,
                        "d2h_gbs": bof / (outf_ms * 1e-3) / 1e9, "h2d_bytes": bif, "d2h_bytes": bof},
            "decode": {"value": world * n * dc.bytes() / (td * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": td / n,
                       "h2d_gbs": bid / (ind_ms * 1e-3) / 1e9, "d2h_gbs": bod / (outd_ms * 1e-3) / 1e9,
                       "h2d_bytes": bid, "d2h_bytes": bod}}


def main():
    args = parse()
    if args.profile_case:
        run_profile_case(args.profile_case, args.option)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
