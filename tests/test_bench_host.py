"""Host logic of bench.py on the CPU: the cross-rank maximum with two gloo ranks, the decode
sample workload, the reference arm's JSON line, and the source hashes of the traffic records."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

from helpers import ROOT

torch = pytest.importorskip("torch")


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    out[rank] = b.max_over_ranks(10.0 + rank * 5.0, world, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_decode_sample_case_matches_the_workload():
    from synth import workloads as W
    b = _bench()
    full = W.decode()
    smp = b.decode_sample_case(full, 2)
    assert smp.B == 2 and list(smp.seqlens) == list(full.seqlens[:2])
    assert smp.num_pages == int(full.pages_per_seq[:2].sum())


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_traffic_records_cover_their_kernel_sources():
    """Every committed DRAM-traffic record names a kernel whose source files exist, and the
    hash that marks a record as current covers each file the kernel is compiled from (a change
    to any of them makes the bench report the traffic as null until it is captured again)."""
    b = _bench()
    csrc = os.path.join(ROOT, "exact_softmax_attention_gb300", "csrc")
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        recs = json.load(f)
    assert {"step_prefill", "step_decode", "decode_fp8"} <= set(recs)
    for leg, e in recs.items():
        files = b.kernel_sources(e["kernel"])
        assert all(os.path.exists(os.path.join(csrc, n)) for n in files), leg
        assert e["dram_bytes_per_launch"] > 0 and len(e["source_sha"]) == 16
    # the decode kernels include their tensor-map header; the forward kernels do not
    assert "decode_maps.cuh" in b.kernel_sources("decode_split_fp8_kernel")
    assert "decode_maps.cuh" not in b.kernel_sources("attn_fwd_kernel")
    # the hash changes with the contents of any listed file
    sha = b.source_sha("decode_split_kernel")
    assert sha == b.source_sha("decode_split_kernel") and sha != b.source_sha("attn_fwd_kernel")
