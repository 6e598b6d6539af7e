"""The linear entry point that allocates nothing.

Some callers cannot get device memory of their own (a plugin that only holds
the buffers its host framework handed it, a server that reserved its whole HBM
budget up front), so the library offers a linear call whose scratch is a fixed
block built into the library.  This checks, through the C ABI, that two calls
in a row give the same result as the regular entry point (with its
caller-owned workspace) -- bit for bit, since both run the same plan and the
split-K sums are reduced in a fixed order -- and match the float64 oracle
within the tolerance the other linear tests use, and that a call too large for
the block is refused.

This file is collected last on purpose, and passes both alone in a fresh
process and after the other tests.
"""

import numpy as np
import pytest
import torch

import oracle
from quantized_rl_rollout_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def q():
    from quantized_rl_rollout_gb300 import build, qrr

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qrr.lib()
    return qrr


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("m,n,k,r", [(8, 512, 1024, 32), (64, 1024, 4096, 64), (1, 384, 2048, 0)])
def test_noalloc_matches_workspace_call(q, m, n, k, r):
    lib = q.lib()
    W = inputs.weight(n, k, inputs.derive_seed(0, "noalloc", n, k, "W"), device=DEV)
    codes, scales, ts = q.quantize_nvfp4(W)
    if r:
        A, B, alpha = inputs.lora(r, k, n, inputs.derive_seed(0, "noalloc", n, k, "lora"), device=DEV)
    else:
        A, B, alpha = None, None, 0.0
    x = inputs.activations(m, k, inputs.derive_seed(0, "noalloc", m, k, "x"), device=DEV)
    ref = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    y_oracle = oracle.linear.linear_nvfp4_lora(_np(x), codes.cpu().numpy(), scales.cpu().numpy(),
                                               np.float32(ts.item()), None if A is None else _np(A),
                                               None if B is None else _np(B), alpha)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row share (and reuse) the built-in scratch
        y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        st = lib.qrr_linear_nvfp4_lora_noalloc(x.data_ptr(), m, k, codes.data_ptr(), scales.data_ptr(),
                                               ts.data_ptr(), n, ptr(A), ptr(B), r, float(alpha), y.data_ptr(),
                                               None, stream)
        assert st == 0, q.status_name(st)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"call {call}: differs from the workspace entry point"
        ok, nerr, worst = oracle.linear.within_tolerance(_np(y), y_oracle)
        assert ok, f"call {call}: normwise {nerr:.3e}, worst element ratio {worst:.3f}"


def test_noalloc_refuses_what_does_not_fit(q):
    lib = q.lib()
    limit = lib.qrr_noalloc_scratch_bytes()
    m, n, k, r = 64, 128, 131072, 64  # its f16 copy of x alone fills the built-in block
    assert lib.qrr_linear_nvfp4_lora_workspace_bytes(m, n, k, r) > limit
    fake = 0x10000  # never dereferenced: the call is refused on the host
    st = lib.qrr_linear_nvfp4_lora_noalloc(fake, m, k, fake, fake, fake, n, fake, fake, r, 1.0, fake, None, None)
    assert q.status_name(st) == "QRR_ERR_WORKSPACE"
