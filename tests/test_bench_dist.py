"""The multi-process path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The library's work has no exchange step (every stream and head is
independent), so bench.py runs one replica per rank; what needs checking is
the host logic around it: rendezvous, barrier, max-over-ranks timing, and
that only rank 0 prints the reference line.
"""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports a different time; everyone must see the largest
    t = bench.max_over_ranks(1.5 + rank, w)

    class Args:
        steps, warmup = 1, 0
    buf = io.StringIO()
    if rank != 0:
        with redirect_stdout(buf):
            bench.run_reference(Args, w, rank)   # rank > 0 returns without work
    bench.barrier(w)
    out[rank] = (t, buf.getvalue())
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU gloo test")
def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 1.5 + (world - 1)
    assert res[1][1] == ""


def test_algorithmic_bytes_match_the_stated_figures():
    """The roofline's numerator: the per-call algorithmic bytes of the
    batched verify (B=16, T=64, H=16, d=128, bf16 q/k/v). With bf16 o the
    formula B·H·(4·dk·dv + T·(2·dk·2 + dv·2 + 8 + 2·dv + 4·dv + 4)) + 4·B·T
    gives 42,143,744 B; the bench also counts the depth and mask words it
    writes (B·T·4 + B·T·⌈T/32⌉·4 = 12,288 B). The headline's fp32 o adds
    4 MiB; the commit moves S0 once each way."""
    sys.path.insert(0, ROOT)
    import bench
    B, T, H, d = 16, 64, 16, 128
    stated = B * H * (4 * d * d + T * (2 * d * 2 + d * 2 + 8 + 2 * d + 4 * d + 4)) + 4 * B * T
    assert stated == 42_143_744
    assert bench.verify_bytes(B, T, H, d, o_bytes=2) == stated + 12_288
    assert bench.verify_bytes(B, T, H, d) == stated + 12_288 + B * T * H * d * 2 == 46_350_336
    assert bench.commit_bytes(B, T, H, d) == 33_554_432


def test_cpu_baseline_process_pool():
    """The CPU baseline's pool of spawned oracle workers runs, counts whole
    streams and reports its core count and repeats."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    inp = synth.config_inputs(0)
    r = bench.cpu_baseline(inp, seconds=0.3, repeats=2)
    assert r["kind"] == "oracle" and r["value"] > 0 and r["repeats"] == 2
    assert r["cores"] == (os.cpu_count() or 1)
