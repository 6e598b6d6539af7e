"""Thin ctypes binding of the C ABI in ``include/qrr.h``.

Each Python function has the name of the C entry point without its ``qrr_``
prefix and only marshals arguments: it checks dtypes and contiguity, allocates
outputs and workspace with torch when the caller passes none, and hands raw
device pointers and the current CUDA stream to the library.  Every step of the
computation runs in the library's kernels; there is no other code path, and a
missing library is an error.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_qrr.so")

SCALE_FP32 = 0
SCALE_POW2 = 1
FORMAT_NVFP4 = 0
FORMAT_FP8_W128 = 1
DEV_NONFINITE = 0x1
DEV_TIMEOUT = 0x2
DEV_SCALE_RANGE = 0x4
DEV_BAD_INDEX = 0x8
OP_QUANTIZE_NVFP4 = 0
OP_LINEAR_NVFP4_LORA = 1
OP_REQUANTIZE_WEIGHTS = 2
OP_QUANTIZE_FP8 = 3
OP_GEMM_FP8 = 4
OP_LORA_BACKWARD = 5

_c_i64 = ctypes.c_int64
_c_i32 = ctypes.c_int32
_c_p = ctypes.c_void_p
_c_sz = ctypes.c_size_t


class WeightDesc(ctypes.Structure):
    """Mirror of ``qrr_weight_desc``."""

    _fields_ = [("W", _c_p), ("N", _c_i64), ("K", _c_i64), ("codes", _c_p), ("scales", _c_p),
                ("tensor_scale", _c_p)]


class LinearDesc(ctypes.Structure):
    """Mirror of ``qrr_linear_desc``."""

    _fields_ = [("x", _c_p), ("N", _c_i64), ("K", _c_i64), ("codes", _c_p), ("scales", _c_p),
                ("tensor_scale", _c_p), ("lora_A", _c_p), ("lora_B", _c_p), ("r", _c_i32), ("alpha", ctypes.c_float),
                ("y", _c_p)]


# symbol -> (restype, argtypes)
SIGNATURES = {
    "qrr_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qrr_abi_version": (ctypes.c_int, []),
    "qrr_quantize_nvfp4_workspace_bytes": (_c_sz, []),
    "qrr_quantize_nvfp4": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "qrr_linear_nvfp4_lora_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_i64, _c_i32]),
    "qrr_linear_nvfp4_lora": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_p, _c_i32,
                                             ctypes.c_float, _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "qrr_noalloc_scratch_bytes": (_c_sz, []),
    "qrr_linear_nvfp4_lora_noalloc": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_p,
                                                     _c_i32, ctypes.c_float, _c_p, _c_p, _c_p]),
    "qrr_linear_nvfp4_lora_grouped_workspace_bytes": (_c_sz, [ctypes.POINTER(LinearDesc), _c_i32, _c_i64]),
    "qrr_linear_nvfp4_lora_grouped": (ctypes.c_int, [ctypes.POINTER(LinearDesc), _c_i32, _c_i64, _c_p, _c_sz, _c_p,
                                                     _c_p]),
    "qrr_quantize_fp8_w128x128": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i32, _c_p, _c_p]),
    "qrr_quantize_fp8_a1x128": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, _c_i32, _c_p, _c_p]),
    "qrr_gemm_fp8_blockwise": (ctypes.c_int, [_c_p, _c_p, _c_p, _c_p, _c_i64, _c_i64, _c_i64, _c_p, _c_i32, _c_p,
                                              _c_p]),
    "qrr_requantize_workspace_bytes": (_c_sz, [_c_i32]),
    "qrr_requantize_weights": (ctypes.c_int, [ctypes.POINTER(WeightDesc), _c_i32, _c_i32, _c_i32, _c_p, _c_sz, _c_p,
                                              _c_p]),
    "qrr_round_probe": (ctypes.c_int, [_c_p, _c_i64, _c_i32, _c_p, _c_p]),
    "qrr_get_last_device_status": (ctypes.c_int, [_c_p, _c_p, _c_p]),
    "qrr_kv_append_fp8": (ctypes.c_int, [_c_p, _c_p, _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_i32, _c_p,
                                         _c_p]),
    "qrr_attention_decode_fp8_workspace_bytes": (_c_sz, [_c_i32, _c_i32, _c_i32]),
    "qrr_attention_decode_fp8": (ctypes.c_int, [_c_p, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p,
                                                _c_p, _c_sz, _c_p, _c_p]),
    "qrr_lora_backward_workspace_bytes": (_c_sz, [_c_i64, _c_i64, _c_i64, _c_i32]),
    "qrr_lora_backward_nvfp4": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32,
                                               ctypes.c_float, _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "qrr_requantize_weights_aqn": (ctypes.c_int, [ctypes.POINTER(WeightDesc), _c_i32, _c_i32, _c_i32, ctypes.c_float,
                                                  ctypes.c_uint64, _c_i32, _c_p, _c_sz, _c_p, _c_p]),
    "qrr_aqn_sigma": (ctypes.c_float, [_c_i32, _c_i32, ctypes.c_double, ctypes.c_double]),
    "qrr_aqn_noise_probe": (ctypes.c_int, [_c_p, _c_i64, _c_i64, ctypes.c_uint64, _c_i32, _c_i32, _c_p]),
    "qrr_token_logprobs_is": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p, ctypes.c_float, _c_p, _c_p, _c_p,
                                             _c_p]),
    "qrr_workspace_bytes": (_c_sz, [_c_i32, _c_i64, _c_i64, _c_i64, _c_i32]),
    "qrr_wait_probe": (ctypes.c_int, [_c_i64, _c_i32, _c_p, _c_p, _c_p]),
    "qrr_stream_probe": (ctypes.c_int, [_c_p, _c_i64, _c_i64, _c_p, _c_p]),
    "qrr_plan_decode_units": (_c_i64, [_c_i64, _c_i32, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_p, _c_p]),
}

_lib = None


class QrrError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_name(status)}")


def lib() -> ctypes.CDLL:
    """The loaded library (loaded on first use); raises if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"the CUDA library {LIB_PATH} is not built; run __graft_entry__.build() "
                               "(there is no CPU fallback)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_name(status: int) -> str:
    return lib().qrr_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise QrrError(status, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t, dtype, name):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _workspace(nbytes: int, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------

def quantize_nvfp4(W, codes=None, scales=None, tensor_scale=None, workspace=None, dev_status=None, stream=None):
    """NVFP4 quantization of a bf16 [N, K] weight -> (codes, scales, tensor_scale)."""
    _need(W, torch.bfloat16, "W")
    n, k = W.shape
    dev = W.device
    codes = torch.empty(n, k // 2, dtype=torch.uint8, device=dev) if codes is None else codes
    scales = torch.empty(n, k // 16, dtype=torch.uint8, device=dev) if scales is None else scales
    tensor_scale = torch.empty(1, dtype=torch.float32, device=dev) if tensor_scale is None else tensor_scale
    ws_bytes = lib().qrr_quantize_nvfp4_workspace_bytes()
    workspace = _workspace(ws_bytes, dev) if workspace is None else workspace
    _check(lib().qrr_quantize_nvfp4(_ptr(W), n, k, _ptr(codes), _ptr(scales), _ptr(tensor_scale), _ptr(workspace),
                                    workspace.numel(), _ptr(dev_status), _stream(stream)), "qrr_quantize_nvfp4")
    return codes, scales, tensor_scale


def linear_nvfp4_lora_workspace_bytes(M, N, K, r) -> int:
    return int(lib().qrr_linear_nvfp4_lora_workspace_bytes(M, N, K, r))


def linear_nvfp4_lora(x, codes, scales, tensor_scale, lora_A=None, lora_B=None, alpha=0.0, y=None, workspace=None,
                      dev_status=None, stream=None):
    """y = x . dequant(W)^T + (alpha/r) (x . A^T) . B^T in bf16."""
    _need(x, torch.bfloat16, "x")
    m, k = x.shape
    n = codes.shape[0]
    r = 0 if lora_A is None or lora_B is None else int(lora_A.shape[0])
    y = torch.empty(m, n, dtype=torch.bfloat16, device=x.device) if y is None else y
    if workspace is None:
        workspace = _workspace(linear_nvfp4_lora_workspace_bytes(m, n, k, r), x.device)
    _check(lib().qrr_linear_nvfp4_lora(_ptr(x), m, k, _ptr(codes), _ptr(scales), _ptr(tensor_scale), n,
                                       _ptr(lora_A), _ptr(lora_B), r, float(alpha), _ptr(y), _ptr(workspace),
                                       workspace.numel(), _ptr(dev_status), _stream(stream)),
           "qrr_linear_nvfp4_lora")
    return y


def linear_nvfp4_lora_noalloc(x, codes, scales, tensor_scale, lora_A=None, lora_B=None, alpha=0.0, y=None,
                              dev_status=None, stream=None):
    """Same as ``linear_nvfp4_lora`` but on the library's built-in scratch (no workspace)."""
    _need(x, torch.bfloat16, "x")
    m, k = x.shape
    n = codes.shape[0]
    r = 0 if lora_A is None or lora_B is None else int(lora_A.shape[0])
    y = torch.empty(m, n, dtype=torch.bfloat16, device=x.device) if y is None else y
    _check(lib().qrr_linear_nvfp4_lora_noalloc(_ptr(x), m, k, _ptr(codes), _ptr(scales), _ptr(tensor_scale), n,
                                               _ptr(lora_A), _ptr(lora_B), r, float(alpha), _ptr(y),
                                               _ptr(dev_status), _stream(stream)), "qrr_linear_nvfp4_lora_noalloc")
    return y


def _linear_descs(layers):
    descs = (LinearDesc * len(layers))()
    m = None
    for i, d in enumerate(layers):
        x, codes, scales, ts = d["x"], d["codes"], d["scales"], d["tensor_scale"]
        _need(x, torch.bfloat16, f"layers[{i}].x")
        a, b = d.get("lora_A"), d.get("lora_B")
        r = 0 if a is None or b is None else int(a.shape[0])
        if m is None:
            m = x.shape[0]
        elif x.shape[0] != m:
            raise ValueError("every layer of a grouped call has the same token count")
        if d.get("y") is None:
            d["y"] = torch.empty(m, codes.shape[0], dtype=torch.bfloat16, device=x.device)
        descs[i] = LinearDesc(_ptr(x), codes.shape[0], x.shape[1], _ptr(codes), _ptr(scales), _ptr(ts), _ptr(a),
                              _ptr(b), r, float(d.get("alpha", 0.0)), _ptr(d["y"]))
    return descs, (m or 0)


def linear_nvfp4_lora_grouped_workspace_bytes(layers) -> int:
    descs, m = _linear_descs(layers)
    return int(lib().qrr_linear_nvfp4_lora_grouped_workspace_bytes(descs, len(layers), m))


def linear_nvfp4_lora_grouped(layers, workspace=None, dev_status=None, stream=None):
    """Run up to 8 layers sharing the token count in one grouped call.

    ``layers`` is a list of dicts with keys x, codes, scales, tensor_scale and
    optionally lora_A, lora_B, alpha, y (allocated when absent).  Returns the
    list of outputs.
    """
    descs, m = _linear_descs(layers)
    if workspace is None:
        nbytes = lib().qrr_linear_nvfp4_lora_grouped_workspace_bytes(descs, len(layers), m)
        workspace = _workspace(nbytes, layers[0]["x"].device)
    _check(lib().qrr_linear_nvfp4_lora_grouped(descs, len(layers), m, _ptr(workspace), workspace.numel(),
                                               _ptr(dev_status), _stream(stream)), "qrr_linear_nvfp4_lora_grouped")
    return [d["y"] for d in layers]


class GroupedLinear:
    """A grouped linear call prepared once, for the decode loop's case of
    fixed buffers: the layers' tensors (x, weights, adapters, y) and the
    workspace are bound at construction, checked once, and ``run()`` only
    launches.  Refill x in place between runs; y is rewritten by each run.
    The numbers are those of ``linear_nvfp4_lora_grouped`` on the same
    tensors, bit for bit (it is the same C call)."""

    def __init__(self, layers, workspace=None):
        self.layers = layers
        self.descs, self.m = _linear_descs(layers)
        nbytes = int(lib().qrr_linear_nvfp4_lora_grouped_workspace_bytes(self.descs, len(layers), self.m))
        if workspace is None:
            workspace = _workspace(nbytes, layers[0]["x"].device)
        elif workspace.numel() < nbytes:
            raise ValueError(f"workspace of {workspace.numel()} bytes, the call needs {nbytes}")
        self.workspace = workspace
        self.outputs = [d["y"] for d in layers]
        self._args = (self.descs, len(layers), self.m, _ptr(workspace), workspace.numel())
        self._fn = lib().qrr_linear_nvfp4_lora_grouped

    def run(self, dev_status=None, stream=None):
        _check(self._fn(*self._args, _ptr(dev_status), _stream(stream)), "qrr_linear_nvfp4_lora_grouped")
        return self.outputs


def quantize_fp8_w128x128(W, mode=SCALE_FP32, q=None, scales=None, dev_status=None, stream=None):
    _need(W, torch.bfloat16, "W")
    n, k = W.shape
    q = torch.empty(n, k, dtype=torch.uint8, device=W.device) if q is None else q
    scales = torch.empty((n + 127) // 128, k // 128, dtype=torch.float32, device=W.device) if scales is None else scales
    _check(lib().qrr_quantize_fp8_w128x128(_ptr(W), n, k, _ptr(q), _ptr(scales), int(mode), _ptr(dev_status),
                                           _stream(stream)), "qrr_quantize_fp8_w128x128")
    return q, scales


def quantize_fp8_a1x128(x, mode=SCALE_FP32, q=None, scales=None, dev_status=None, stream=None):
    _need(x, torch.bfloat16, "x")
    m, k = x.shape
    q = torch.empty(m, k, dtype=torch.uint8, device=x.device) if q is None else q
    scales = torch.empty(m, k // 128, dtype=torch.float32, device=x.device) if scales is None else scales
    _check(lib().qrr_quantize_fp8_a1x128(_ptr(x), m, k, _ptr(q), _ptr(scales), int(mode), _ptr(dev_status),
                                         _stream(stream)), "qrr_quantize_fp8_a1x128")
    return q, scales


def gemm_fp8_blockwise(qa, sa, qw, sw, mode=SCALE_FP32, y=None, dev_status=None, stream=None):
    m, k = qa.shape
    n = qw.shape[0]
    y = torch.empty(m, n, dtype=torch.bfloat16, device=qa.device) if y is None else y
    _check(lib().qrr_gemm_fp8_blockwise(_ptr(qa), _ptr(sa), _ptr(qw), _ptr(sw), m, n, k, _ptr(y), int(mode),
                                        _ptr(dev_status), _stream(stream)), "qrr_gemm_fp8_blockwise")
    return y


def _weight_descs(weights, outputs, fmt):
    count = len(weights)
    descs = (WeightDesc * max(count, 1))()
    for i, (w, out) in enumerate(zip(weights, outputs)):
        _need(w, torch.bfloat16, f"weights[{i}]")
        ts = out[2] if fmt == FORMAT_NVFP4 else None
        descs[i] = WeightDesc(_ptr(w), w.shape[0], w.shape[1], _ptr(out[0]), _ptr(out[1]), _ptr(ts))
    return descs, count


def requantize_weights(weights, outputs, fmt=FORMAT_NVFP4, mode=SCALE_FP32, workspace=None, dev_status=None,
                       stream=None):
    """Re-quantize every bf16 weight of ``weights`` into ``outputs``.

    ``outputs[i]`` is ``(codes, scales, tensor_scale)`` for NVFP4 or
    ``(q, scales)`` for FP8 128x128.
    """
    descs, count = _weight_descs(weights, outputs, fmt)
    dev = weights[0].device if count else torch.device("cuda")
    if workspace is None:
        workspace = _workspace(lib().qrr_requantize_workspace_bytes(count), dev)
    _check(lib().qrr_requantize_weights(descs, count, int(fmt), int(mode), _ptr(workspace), workspace.numel(),
                                        _ptr(dev_status), _stream(stream)), "qrr_requantize_weights")
    return outputs


def requantize_weights_aqn(weights, outputs, sigma, seed, step, fmt=FORMAT_NVFP4, mode=SCALE_FP32, workspace=None,
                           dev_status=None, stream=None):
    """``requantize_weights`` of the noisy masters bf16(W + sigma z) (see ``qrr_requantize_weights_aqn``)."""
    descs, count = _weight_descs(weights, outputs, fmt)
    dev = weights[0].device if count else torch.device("cuda")
    if workspace is None:
        workspace = _workspace(lib().qrr_requantize_workspace_bytes(count), dev)
    _check(lib().qrr_requantize_weights_aqn(descs, count, int(fmt), int(mode), float(sigma), int(seed), int(step),
                                            _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream)),
           "qrr_requantize_weights_aqn")
    return outputs


def aqn_sigma(step, steps, sigma_start, sigma_end) -> float:
    return float(lib().qrr_aqn_sigma(int(step), int(steps), float(sigma_start), float(sigma_end)))


def aqn_noise_probe(n, seed, tensor, step, start=0, out=None, stream=None):
    out = torch.empty(n, dtype=torch.float32, device="cuda") if out is None else out
    _check(lib().qrr_aqn_noise_probe(_ptr(out), int(n), int(start), int(seed), int(tensor), int(step),
                                     _stream(stream)), "qrr_aqn_noise_probe")
    return out


def round_probe(values, fmt, out=None, stream=None):
    _need(values, torch.float32, "values")
    out = torch.empty(values.numel(), dtype=torch.uint8, device=values.device) if out is None else out
    _check(lib().qrr_round_probe(_ptr(values), values.numel(), int(fmt), _ptr(out), _stream(stream)),
           "qrr_round_probe")
    return out


def get_last_device_status(dev_status, stream=None) -> int:
    """Host copy of the device status word once the stream's earlier work is done."""
    _need(dev_status, torch.int32, "dev_status")
    out = ctypes.c_int32(0)
    _check(lib().qrr_get_last_device_status(ctypes.addressof(out), _ptr(dev_status), _stream(stream)),
           "qrr_get_last_device_status")
    return int(out.value)


def workspace_bytes(op, M=0, N=0, K=0, r=0) -> int:
    return int(lib().qrr_workspace_bytes(int(op), int(M), int(N), int(K), int(r)))


def plan_decode_units(M, shapes, grid, max_units=4096):
    """The decode launch's unit table for layers ``shapes`` = [(N, K, r), ...]
    at M tokens on ``grid`` CTAs (host only; see ``qrr_plan_decode_units``).

    Returns ``(units, offsets)``: a list of decoded units (dicts with layer,
    m_tile, n_tile, pieces, c0, nk, piece, lora) and the per-CTA offsets."""
    n = len(shapes)
    Ns = (ctypes.c_int64 * n)(*[int(s[0]) for s in shapes])
    Ks = (ctypes.c_int64 * n)(*[int(s[1]) for s in shapes])
    rs = (ctypes.c_int32 * n)(*[int(s[2]) for s in shapes])
    units = (ctypes.c_uint32 * (2 * max_units))()
    offsets = (ctypes.c_uint16 * (int(grid) + 1))()
    used = ctypes.c_int32(0)
    got = lib().qrr_plan_decode_units(int(M), n, ctypes.addressof(Ns), ctypes.addressof(Ks), ctypes.addressof(rs),
                                      int(grid), ctypes.addressof(units), int(max_units), ctypes.addressof(offsets),
                                      ctypes.addressof(used))
    if got < 0:
        raise QrrError(int(-got), "qrr_plan_decode_units")
    out = []
    for i in range(got):
        w0, w1 = units[2 * i], units[2 * i + 1]
        out.append(dict(layer=w0 & 0xF, m_tile=(w0 >> 4) & 0xF, n_tile=(w0 >> 8) & 0xFFFF, pieces=w0 >> 24,
                        c0=w1 & 0xFFF, nk=(w1 >> 12) & 0x7FF, piece=(w1 >> 23) & 0xFF, lora=w1 >> 31))
    return out, [int(offsets[b]) for b in range(used.value + 1)]


def wait_probe(limit_cycles, arrive, dev_status, cycles=None, stream=None):
    """Run the bounded-wait probe (see ``qrr_wait_probe``)."""
    _need(dev_status, torch.int32, "dev_status")
    if cycles is not None:
        _need(cycles, torch.int64, "cycles")
    _check(lib().qrr_wait_probe(int(limit_cycles), int(arrive), _ptr(dev_status), _ptr(cycles), _stream(stream)),
           "qrr_wait_probe")


def stream_probe(data, dev_status=None, stream=None):
    """Stream a uint8 [rows, row_bytes] matrix through the TMA ring of the
    decode kernels with no arithmetic (see ``qrr_stream_probe``)."""
    _need(data, torch.uint8, "data")
    if data.dim() != 2:
        raise ValueError("stream_probe: data must be a 2-D uint8 tensor")
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
    _check(lib().qrr_stream_probe(_ptr(data), data.shape[0], data.shape[1], _ptr(dev_status), _stream(stream)),
           "qrr_stream_probe")


def token_logprobs_is(logits, tokens, rollout_logp=None, cap=0.0, logp=None, w=None, dev_status=None, stream=None):
    """Token log-probabilities (and, given the rollout's, importance weights).

    Returns ``logp`` or ``(logp, w)`` when ``rollout_logp`` is given."""
    _need(logits, torch.bfloat16, "logits")
    _need(tokens, torch.int32, "tokens")
    t, v = logits.shape
    logp = torch.empty(t, dtype=torch.float32, device=logits.device) if logp is None else logp
    if rollout_logp is not None:
        _need(rollout_logp, torch.float32, "rollout_logp")
        w = torch.empty(t, dtype=torch.float32, device=logits.device) if w is None else w
    _check(lib().qrr_token_logprobs_is(_ptr(logits), t, v, _ptr(tokens), _ptr(rollout_logp), float(cap), _ptr(logp),
                                       _ptr(w) if rollout_logp is not None else None, _ptr(dev_status),
                                       _stream(stream)), "qrr_token_logprobs_is")
    return logp if rollout_logp is None else (logp, w)


def lora_backward_workspace_bytes(M, N, K, r) -> int:
    return int(lib().qrr_lora_backward_workspace_bytes(M, N, K, r))


def lora_backward_nvfp4(dy, x, codes, scales, tensor_scale, lora_A=None, lora_B=None, alpha=0.0, dx=None, dA=None,
                        dB=None, workspace=None, dev_status=None, stream=None):
    """(dX bf16 [M, K], dA fp32 [r, K], dB fp32 [N, r]) of the linear's backward
    through the frozen NVFP4 weight (dA, dB None without an adapter)."""
    _need(dy, torch.bfloat16, "dy")
    m, n = dy.shape
    k = codes.shape[1] * 2
    r = 0 if lora_A is None or lora_B is None else int(lora_A.shape[0])
    dev = dy.device
    dx = torch.empty(m, k, dtype=torch.bfloat16, device=dev) if dx is None else dx
    if r:
        _need(x, torch.bfloat16, "x")
        dA = torch.empty(r, k, dtype=torch.float32, device=dev) if dA is None else dA
        dB = torch.empty(n, r, dtype=torch.float32, device=dev) if dB is None else dB
    if workspace is None:
        workspace = _workspace(lora_backward_workspace_bytes(m, n, k, r), dev)
    _check(lib().qrr_lora_backward_nvfp4(_ptr(dy), m, n, _ptr(x), k, _ptr(codes), _ptr(scales), _ptr(tensor_scale),
                                         _ptr(lora_A), _ptr(lora_B), r, float(alpha), _ptr(dx),
                                         _ptr(dA) if r else None, _ptr(dB) if r else None, _ptr(workspace),
                                         workspace.numel(), _ptr(dev_status), _stream(stream)),
           "qrr_lora_backward_nvfp4")
    return dx, (dA if r else None), (dB if r else None)


def kv_append_fp8(k_new, v_new, pos, k_cache, k_scales, v_cache, v_scales, mode=SCALE_FP32, dev_status=None,
                  stream=None):
    """Quantize one decode step's key/value rows [B, Hkv, 128] into slot pos[b] of the FP8 caches."""
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(pos, torch.int32, "pos")
    b, hkv, _ = k_new.shape
    lmax = k_cache.shape[2]
    _check(lib().qrr_kv_append_fp8(_ptr(k_new), _ptr(v_new), b, hkv, _ptr(pos), _ptr(k_cache), _ptr(k_scales),
                                   _ptr(v_cache), _ptr(v_scales), lmax, int(mode), _ptr(dev_status), _stream(stream)),
           "qrr_kv_append_fp8")


def attention_decode_fp8(q, k_cache, k_scales, v_cache, v_scales, lens, out=None, workspace=None, dev_status=None,
                         stream=None):
    """o [B, Hq, 128] bf16 of decode attention over the FP8 caches [B, Hkv, Lmax, 128]."""
    _need(q, torch.bfloat16, "q")
    _need(lens, torch.int32, "lens")
    b, hq, _ = q.shape
    hkv, lmax = k_cache.shape[1], k_cache.shape[2]
    out = torch.empty_like(q) if out is None else out
    if workspace is None:
        workspace = _workspace(lib().qrr_attention_decode_fp8_workspace_bytes(b, hq, lmax), q.device)
    _check(lib().qrr_attention_decode_fp8(_ptr(q), b, hq, hkv, _ptr(k_cache), _ptr(k_scales), _ptr(v_cache),
                                          _ptr(v_scales), _ptr(lens), lmax, _ptr(out), _ptr(workspace),
                                          workspace.numel(), _ptr(dev_status), _stream(stream)),
           "qrr_attention_decode_fp8")
    return out
