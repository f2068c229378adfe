"""Failure surfacing on the GPU, without faulting it: a bounded device wait
that runs out reports TQ_ERR_DEVICE_TIMEOUT and leaves the context usable, and
the arch witness declines (TQ_ERR_CAPTURING) instead of being taken inside a
stream capture, then succeeds once the capture is over.

Pages: "fix(qtip): arch-specialise the trellis grouped GEMM ...", sections "The
two changes" and "The arch witness" (a stuck or failed launch must surface as an
error; the witness is never taken during capture and only success is cached)."""
import os
import subprocess
import sys
import textwrap
import time
import zlib

import numpy as np
import pytest

import moe_inputs
import oracle.trellis_moe as O
import trellis_quantized_moe_sort_gb300 as tq
from gpu_util import to_device, grouped_y32, normwise

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TQ_ERR_CAPTURING, TQ_ERR_DEVICE_TIMEOUT, WHERE_PROBE = -5, -6, 10


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_quantized_moe_sort_gb300 import build
    build.build()
    tq.tq_init(0)


def test_bounded_wait_gives_up_and_reports():
    tq.tq_device_error()                       # start from a clear error word
    t0 = time.time()
    done, us = tq.tq_probe_wait_timeout(20_000_000)   # 20 ms on a barrier nothing arrives at
    wall = time.time() - t0
    assert not done
    assert 20_000 <= us < 1_000_000, us
    assert wall < 30, wall
    assert tq.tq_device_error() == (TQ_ERR_DEVICE_TIMEOUT, WHERE_PROBE)
    assert tq.tq_device_error() == (0, 0)      # read and cleared
    # the context is still usable: a small product right after matches the oracle
    name = "after_timeout"
    prob = moe_inputs.make_custom(8, 2, 24, 256, 256, 12, seed=zlib.crc32(name.encode()) % 1000)
    y = grouped_y32(prob, to_device(prob), 16).cpu().numpy()
    ref = O.moe_forward(prob.x_bits, prob.topk_ids, prob.topk_w, prob.packed, prob.lut_bits, prob.shape.L)
    assert normwise(y, ref) <= 1e-2


def test_bounded_wait_rejects_out_of_range_limits():
    for bad in (0, 999, 2_000_000_001):
        with pytest.raises(tq.TQError) as e:
            tq.tq_probe_wait_timeout(bad)
        assert e.value.status == -1


def test_witness_declines_inside_capture_in_a_fresh_process():
    """A fresh process (witness not yet taken) calls a launcher while its
    stream is being captured: the call returns TQ_ERR_CAPTURING before any
    device work; after the capture the same call takes the witness and runs."""
    script = textwrap.dedent("""
        import torch
        import trellis_quantized_moe_sort_gb300 as tq
        torch.cuda.set_device(0)
        tq.lib()                                   # load the library outside the capture
        ids = torch.tensor([[0, 1], [2, 3], [1, 0], [3, 2]], dtype=torch.int32, device="cuda")
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        code = None
        with torch.cuda.stream(side):
            graph.capture_begin()
            try:
                tq.tq_route(ids, 8)
            except tq.TQError as e:
                code = e.status
            ids.add_(0)                            # keep the captured graph non-empty
            graph.capture_end()
        torch.cuda.current_stream().wait_stream(side)
        print("CAPTURE", code)
        counts, offsets, sp = tq.tq_route(ids, 8)
        torch.cuda.synchronize()
        print("AFTER", int(counts.sum()), counts.tolist()[:4], tq.tq_arch_witness(0))
    """)
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=300, cwd=ROOT,
                       env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(line.split(" ", 1) for line in r.stdout.splitlines() if line.startswith(("CAPTURE", "AFTER")))
    assert lines["CAPTURE"] == str(TQ_ERR_CAPTURING), r.stdout
    assert lines["AFTER"] == "8 [2, 2, 2, 2] 1030", r.stdout
