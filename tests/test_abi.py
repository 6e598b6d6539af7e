"""Host-only checks of the C ABI: the library loads, exports every function
include/qrr.h declares, and rejects bad arguments before launching anything.
No call here reaches a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_rl_rollout_gb300 import build, qrr

    build.build()
    return qrr.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "qrr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qrr_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    from quantized_rl_rollout_gb300 import qrr

    names = _declared()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name
        assert name in qrr.SIGNATURES, f"{name} has no binding"


def test_status_strings(lib):
    from quantized_rl_rollout_gb300 import qrr

    assert qrr.status_name(0) == "QRR_OK"
    assert qrr.status_name(2) == "QRR_ERR_UNSUPPORTED_SHAPE"
    assert qrr.status_name(99) == "QRR_UNKNOWN_STATUS"
    assert lib.qrr_abi_version() == 1


def test_workspace_queries(lib):
    assert lib.qrr_quantize_nvfp4_workspace_bytes() >= 4
    assert lib.qrr_requantize_workspace_bytes(7) >= 28
    assert lib.qrr_linear_nvfp4_lora_workspace_bytes(64, 4096, 4096, 32) >= 64 * 32 * 4


FAKE = 0x10000  # a 16-byte-aligned non-null address that is never dereferenced


def test_argument_validation(lib):
    q = lib.qrr_quantize_nvfp4
    ws = lib.qrr_quantize_nvfp4_workspace_bytes()
    assert q(FAKE, 4, 30, FAKE, FAKE, FAKE, FAKE, ws, None, None) == 2  # K % 32
    assert q(FAKE, -1, 32, FAKE, FAKE, FAKE, FAKE, ws, None, None) == 1
    assert q(FAKE + 8, 4, 32, FAKE, FAKE, FAKE, FAKE, ws, None, None) == 3  # misaligned W
    assert q(FAKE, 4, 32, FAKE, FAKE, None, FAKE, ws, None, None) == 1  # no tensor scale
    assert q(FAKE, 4, 32, FAKE, FAKE, FAKE, None, ws, None, None) == 4  # no workspace
    lin = lib.qrr_linear_nvfp4_lora
    lws = lib.qrr_linear_nvfp4_lora_workspace_bytes(16, 128, 256, 8)
    assert lin(FAKE, 16, 200, FAKE, FAKE, FAKE, 128, FAKE, FAKE, 8, 16.0, FAKE, FAKE, lws, None, None) == 2
    assert lin(FAKE, 16, 256, FAKE, FAKE, FAKE, 100, FAKE, FAKE, 8, 16.0, FAKE, FAKE, lws, None, None) == 2
    assert lin(FAKE, 16, 256, FAKE, FAKE, FAKE, 128, FAKE, FAKE, 12, 16.0, FAKE, FAKE, lws, None, None) == 2
    assert lin(FAKE, 16, 256, FAKE, FAKE, FAKE, 128, FAKE, FAKE, 8, 16.0, FAKE, FAKE, 4, None, None) == 4
    assert lib.qrr_quantize_fp8_a1x128(FAKE, 4, 100, FAKE, FAKE, 0, None, None) == 2
    assert lib.qrr_quantize_fp8_a1x128(FAKE, 4, 128, FAKE, FAKE, 7, None, None) == 1
    assert lib.qrr_quantize_fp8_w128x128(FAKE, 4, 128, FAKE + 4, FAKE, 0, None, None) == 3
    assert lib.qrr_gemm_fp8_blockwise(FAKE, FAKE, FAKE, FAKE, 4, 100, 128, FAKE, 0, None, None) == 2
    assert lib.qrr_round_probe(FAKE, 4, 5, FAKE, None) == 1
    # adapter rank above 64 is outside the linear's contract
    lws = lib.qrr_linear_nvfp4_lora_workspace_bytes(16, 128, 256, 72)
    assert lin(FAKE, 16, 256, FAKE, FAKE, FAKE, 128, FAKE, FAKE, 72, 16.0, FAKE, FAKE, lws, None, None) == 2


def test_grouped_linear_validation(lib):
    from quantized_rl_rollout_gb300 import qrr

    descs = (qrr.LinearDesc * 9)()
    for i in range(9):
        descs[i] = qrr.LinearDesc(FAKE, 128, 256, FAKE, FAKE, FAKE, None, None, 0, 0.0, FAKE)
    assert lib.qrr_linear_nvfp4_lora_grouped(descs, 9, 16, FAKE, 1 << 20, None, None) == 2  # > 8 layers
    ws = lib.qrr_linear_nvfp4_lora_grouped_workspace_bytes(descs, 3, 16)
    assert ws > 0
    assert lib.qrr_linear_nvfp4_lora_grouped(descs, 3, 16, FAKE, ws - 1, None, None) == 4
    descs[1] = qrr.LinearDesc(FAKE, 100, 256, FAKE, FAKE, FAKE, None, None, 0, 0.0, FAKE)  # N % 128
    assert lib.qrr_linear_nvfp4_lora_grouped(descs, 3, 16, FAKE, ws, None, None) == 2


def test_requant_descriptor_validation(lib):
    from quantized_rl_rollout_gb300 import qrr

    descs = (qrr.WeightDesc * 2)()
    descs[0] = qrr.WeightDesc(FAKE, 4, 64, FAKE, FAKE, FAKE)
    descs[1] = qrr.WeightDesc(FAKE, 4, 48, FAKE, FAKE, FAKE)  # K % 32 != 0
    assert lib.qrr_requantize_weights(descs, 2, 0, 0, FAKE, 4096, None, None) == 2
    assert lib.qrr_requantize_weights(descs, 2, 5, 0, FAKE, 4096, None, None) == 1
    assert lib.qrr_requantize_weights(None, 1, 0, 0, FAKE, 4096, None, None) == 1
    descs[1] = qrr.WeightDesc(FAKE, 4, 64, FAKE, FAKE, FAKE)
    assert lib.qrr_requantize_weights(descs, 2, 0, 0, None, 0, None, None) == 4


def test_injected_cuda_fault_reports_error(lib, monkeypatch):
    """The host-side fault hook makes a valid call fail with QRR_ERR_CUDA
    without launching (no GPU is touched)."""
    monkeypatch.setenv("QRR_INJECT_FAULT", "cuda")
    ws = lib.qrr_quantize_nvfp4_workspace_bytes()
    assert lib.qrr_quantize_nvfp4(FAKE, 4, 32, FAKE, FAKE, FAKE, FAKE, ws, None, None) == 5
    from quantized_rl_rollout_gb300 import qrr

    with pytest.raises(qrr.QrrError) as e:
        qrr._check(5, "probe")
    assert "QRR_ERR_CUDA" in str(e.value)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from quantized_rl_rollout_gb300 import qrr

    monkeypatch.setattr(qrr, "_lib", None)
    monkeypatch.setattr(qrr, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        qrr.lib()


def test_status_sync_and_probe_validation(lib):
    """Argument checks of the sync point and the wait probe (host side only)."""
    assert lib.qrr_get_last_device_status(None, FAKE, None) == 1
    assert lib.qrr_get_last_device_status(FAKE, None, None) == 1
    assert lib.qrr_get_last_device_status(FAKE, FAKE + 2, None) == 3
    assert lib.qrr_wait_probe(0, 0, FAKE, None, None) == 1  # no limit
    assert lib.qrr_wait_probe(1 << 40, 0, FAKE, None, None) == 1  # above the pipelines' own limit
    assert lib.qrr_wait_probe(1000, 2, FAKE, None, None) == 1
    assert lib.qrr_wait_probe(1000, 0, None, None, None) == 1
    assert lib.qrr_wait_probe(1000, 0, FAKE, FAKE + 4, None) == 3
    # the stream probe: shapes in whole 128-row, 128-byte boxes, aligned data
    assert lib.qrr_stream_probe(None, 128, 128, None, None) == 1
    assert lib.qrr_stream_probe(FAKE, -128, 128, None, None) == 1
    assert lib.qrr_stream_probe(FAKE, 130, 128, None, None) == 2
    assert lib.qrr_stream_probe(FAKE, 128, 100, None, None) == 2
    assert lib.qrr_stream_probe(FAKE + 8, 128, 128, None, None) == 3
    assert lib.qrr_stream_probe(FAKE, 128, 128, FAKE + 2, None) == 3
    assert lib.qrr_stream_probe(FAKE, 0, 128, None, None) == 0  # nothing to stream, nothing launched


def test_generic_workspace_query_matches_per_call_queries(lib):
    from quantized_rl_rollout_gb300 import qrr

    assert lib.qrr_workspace_bytes(qrr.OP_QUANTIZE_NVFP4, 0, 0, 0, 0) == lib.qrr_quantize_nvfp4_workspace_bytes()
    for m, n, k, r in [(1, 4096, 4096, 32), (64, 14336, 4096, 32), (4096, 1024, 4096, 0), (3, 128, 256, 8)]:
        assert lib.qrr_workspace_bytes(qrr.OP_LINEAR_NVFP4_LORA, m, n, k, r) == \
            lib.qrr_linear_nvfp4_lora_workspace_bytes(m, n, k, r)
    assert lib.qrr_workspace_bytes(qrr.OP_REQUANTIZE_WEIGHTS, 7, 0, 0, 0) == lib.qrr_requantize_workspace_bytes(7)
    assert lib.qrr_workspace_bytes(qrr.OP_GEMM_FP8, 4096, 4096, 4096, 0) == 0
    assert lib.qrr_workspace_bytes(99, 1, 1, 1, 1) == 0


def test_aqn_and_is_validation(lib):
    from quantized_rl_rollout_gb300 import qrr

    descs = (qrr.WeightDesc * 1)()
    descs[0] = qrr.WeightDesc(FAKE, 4, 64, FAKE, FAKE, FAKE)
    assert lib.qrr_requantize_weights_aqn(descs, 1, 0, 0, -1.0, 1, 0, FAKE, 4096, None, None) == 1  # sigma < 0
    assert lib.qrr_requantize_weights_aqn(descs, 1, 0, 0, float("nan"), 1, 0, FAKE, 4096, None, None) == 1
    assert lib.qrr_requantize_weights_aqn(descs, 1, 0, 0, 1e-3, 1, -2, FAKE, 4096, None, None) == 1  # step < 0
    assert lib.qrr_requantize_weights_aqn(descs, 1, 0, 0, 1e-3, 1, 0, None, 0, None, None) == 4
    assert lib.qrr_aqn_noise_probe(FAKE + 2, 4, 0, 1, 0, 0, None) == 3
    assert lib.qrr_aqn_noise_probe(FAKE, -1, 0, 1, 0, 0, None) == 1
    assert abs(lib.qrr_aqn_sigma(0, 100, 1e-2, 5e-4) - 1e-2) < 1e-9
    assert abs(lib.qrr_aqn_sigma(99, 100, 1e-2, 5e-4) - 5e-4) < 1e-9
    assert lib.qrr_token_logprobs_is(FAKE, 4, 0, FAKE, None, 0.0, FAKE, None, None, None) == 1  # V = 0
    assert lib.qrr_token_logprobs_is(FAKE, 4, 8, FAKE, FAKE, 0.0, FAKE, None, None, None) == 1  # no w
    assert lib.qrr_token_logprobs_is(FAKE + 8, 4, 8, FAKE, None, 0.0, FAKE, None, None, None) == 3
