"""The device status word on a GB300: the explicit sync point, and the
bounded-wait path run out on purpose.

A probe kernel allocates tensor memory and waits, through the same bounded
wait every tensor-core pipeline of the library uses, on a barrier that nothing
completes, with a give-up time of about a millisecond.  The wait must end by
itself, raise QRR_DEV_TIMEOUT, free the tensor memory and let the kernel exit;
the context must stay usable, so the next ordinary call on the same stream
still matches the oracle.  No fault, trap or endless loop is involved: the
wait is bounded by construction."""

import time

import numpy as np
import pytest
import torch

import oracle
from quantized_rl_rollout_gb300 import configs, inputs

from .conftest import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def q():
    from quantized_rl_rollout_gb300 import build, qrr

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qrr.lib()
    return qrr


def test_sync_point_reads_the_word(q):
    st = torch.tensor([0x40], dtype=torch.int32, device=DEV)
    assert q.get_last_device_status(st) == 0x40
    st.zero_()
    assert q.get_last_device_status(st) == 0


def test_wait_runs_out_and_reports_timeout(q):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    cyc = torch.zeros(1, dtype=torch.int64, device=DEV)
    limit = 2_000_000  # SM cycles: about 1 ms at 2 GHz
    t0 = time.perf_counter()
    q.wait_probe(limit, 0, st, cyc)
    word = q.get_last_device_status(st)
    wall = time.perf_counter() - t0
    assert word & q.DEV_TIMEOUT, f"status {word:#x}"
    spent = int(cyc.item())
    assert limit <= spent < 50 * limit, spent  # gave up after the limit, not long after
    assert wall < 5.0
    # the barrier completed first: no flag, the wait returns at once
    st.zero_()
    q.wait_probe(limit, 1, st, cyc)
    assert q.get_last_device_status(st) == 0
    assert int(cyc.item()) < limit


def test_context_usable_after_timeout(q):
    """After a timed-out probe, an ordinary quantize + linear on the same
    stream is still bit-exact / within tolerance against the oracle."""
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.wait_probe(1_000_000, 0, st)
    assert q.get_last_device_status(st) & q.DEV_TIMEOUT
    c = configs.TINY
    W = inputs.weight(c["n"], c["k"], inputs.derive_seed(0, "tiny", "W"), device=DEV)
    x = inputs.activations(c["m"], c["k"], inputs.derive_seed(0, "tiny", "x"), device=DEV)
    A, B, _ = inputs.lora(c["r"], c["k"], c["n"], inputs.derive_seed(0, "tiny", "lora"), device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    codes, scales, ts = q.quantize_nvfp4(W, dev_status=st2)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, c["alpha"], dev_status=st2)
    assert q.get_last_device_status(st2) == 0
    rc, rs, rt = oracle.nvfp4.quantize(to_np(W))
    assert np.array_equal(codes.cpu().numpy(), rc) and np.array_equal(scales.cpu().numpy(), rs)
    y_ref = oracle.linear.linear_nvfp4_lora(to_np(x), rc, rs, rt, to_np(A), to_np(B), c["alpha"])
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y), y_ref)
    assert ok, f"normwise {nerr:.3e}, worst {worst:.3f}"


def test_stream_probe_runs_clean(q):
    """The memory-floor probe streams a byte matrix through the decode
    kernels' TMA ring and finishes without flagging anything: a few boxes,
    a ragged share per CTA, and the one-token decode's size."""
    for rows, cols in [(128, 128), (384, 640), (62592, 2048)]:
        data = torch.zeros(rows, cols, dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        q.stream_probe(data, dev_status=st)
        torch.cuda.synchronize()
        assert q.get_last_device_status(st) == 0
