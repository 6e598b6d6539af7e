"""Benchmark of the low-precision linear-layer hot path on one GB300.

Workload (the decode configuration the headline metric is quoted on): an
8B-class decoder layer set -- q/o 4096x4096, k/v 1024x4096, gate/up
14336x4096, down 4096x14336, bf16 weights ~N(0, 0.02) with 0.1% x20
outliers -- in NVFP4 with LoRA r = 32 (alpha = 64), decoding 1, 8 and 64
tokens.  One step is one pass of the whole hot path over that layer set:

  requant  re-quantize all 7 bf16 weights to NVFP4 (absmax sweep + encode);
           requant_aqn the same with adaptive quantization noise added to the
           masters (Philox noise drawn in the encode sweep, and in the absmax
           sweep only for values that can hold the largest |W'|)
  decode   W4A16 + LoRA linear of all 7 layers at M = 1, 8 and 64 (one
           grouped call per token count)
  prefill  the same linears at M = 4096 (activations with 1% x10 channels)
  lora_bwd the backward of those linears through the frozen NVFP4 weights at
           M = 4096: dX (bf16) and the adapter gradients dA, dB (fp32)
  fp8      FP8 path at M = 4096: 128x128 weight re-quantize (fp8_requant),
           activation 1x128 quantize (fp8_act_quant), blockwise-scaled GEMM
           with fp32 scales (fp8_gemm, promotion) and with power-of-two scales
           (fp8_gemm_pow2, native block-scaled MMA)
  attn     one decode step of attention over an E4M3 key/value cache: append
           the step's rows, then attention for 64 sequences of 2048..4096
           cached tokens, 32 query / 8 KV heads of 128 (attn_fp8)
  is       token log-probabilities and importance-sampling weights of 4096
           tokens over a 128256-entry vocabulary (rollout_is)
  floor    the memory floor of one decode pass: the one-token decode's bytes
           streamed through the decode kernels' TMA ring of [128 x 128 B]
           boxes with no arithmetic (stream_floor; a reference for the decode
           phases, not part of the hot path)

Re-quantization follows a training step: the bf16 masters alternate between W
and W' = bf16(W + N(0, 1e-4)) from step to step, so every step recalibrates
new weights.

After the step, in a timed region of its own, the 32B-class stack (64 layers
of hidden 5120, LoRA r = 64) is measured too (unless --no-32b): the full bf16
-> NVFP4 re-quantization of its 31.2 G weight elements and decode at M = 64
(one grouped call per layer).  It is another configuration, not part of the
step, and is reported in ``breakdown`` beside the step's phases.

Roofline fractions are given against the measured peaks (``MEASURED_PEAKS.json``;
the FP8 dense peak is measured in the same run with torch._scaled_mm) and, as a
second figure, against GB300's published dense numbers (8 TB/s HBM, 2.25
PFLOP/s bf16, 4.5 PFLOP/s FP8).

Each phase is timed with CUDA events on the launching stream after an L2
flush (a 512 MB write, then a read of the same 512 MB), so no phase reads
its weights from L2 left by the previous one, and none starts by writing
back a cache full of the flush's dirty lines (a cost of the flush, not of
the phase: about 4 us of every decode phase).  ``value`` is the decode phase's HBM throughput: its
algorithmic bytes (packed codes, block and tensor scales, LoRA factors,
activations in, outputs out) over its device time; the other phases are
reported in ``breakdown`` with their own roofline fractions.

``--impl reference`` times the CPU oracle instead (a bounded sample of the
same workload per step, on the host's cores) and prints the same line with
``"impl": "reference"``.
"""

import argparse
import csv
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from quantized_rl_rollout_gb300 import configs, inputs  # noqa: E402

METRIC = "NVFP4+LoRA linear: decode HBM GB/s, prefill TFLOPS; % of roofline"
WORKLOAD = "decode, 8B-class layer set (q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096, down 4096x14336), NVFP4 + LoRA r=32, M=1,8,64"
DECODE_TOKENS = (1, 8, 64)
PREFILL_TOKENS = 4096
R = 32
ALPHA = 2.0 * R
IS_TOKENS, IS_VOCAB, IS_CAP = 4096, 128256, 5.0  # importance-sampling phase: tokens x 8B-class vocabulary
ATT_B, ATT_HQ, ATT_HKV, ATT_L = 64, 32, 8, 4096  # decode attention: sequences, query / KV heads, cache length
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
# GB300's published dense figures (per GPU), reported beside the measured peaks
SPEC_PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2250.0, "fp8_tflops": 4500.0}


# DRAM traffic per launch of each phase's main kernel, from an ncu launch list
# (dram__bytes_read.sum + dram__bytes_write.sum).  It is recorded together with
# a hash of the CUDA sources and reported only while the sources are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
PHASE_KERNELS = {  # phase -> (kernel name prefix, template arguments as ncu prints them)
    "prefill": ("w4a16_tc_kernel", "<256, 64, 0, 3, 1>"),
    "decode_m1": ("w4_decode_nvf4_kernel", ""),
    "decode_m8": ("w4_decode_nvf4_kernel", ""),
    "decode_m64": ("w4a16_tc_kernel", "<64, 256, 1, 3, 0>"),
    "requant": ("nvfp4_encode_kernel", ""),
    "requant_aqn": ("nvfp4_encode_kernel", ""),
    "fp8_requant": ("fp8_w128_kernel", ""),
    "fp8_act_quant": ("fp8_a1x128_kernel", ""),
    "fp8_gemm": ("fp8_gemm_tc_kernel", ""),
    "fp8_gemm_pow2": ("fp8_gemm_mx_kernel", ""),
    "rollout_is": ("token_logprob_is_kernel", ""),
    "stream_floor": ("stream_probe_kernel", ""),
    "lora_bwd": ("gemm_bf16_tc_kernel", ""),
    "attn_fp8": ("attn_decode_fp8_kernel", ""),
}


def source_hash():
    h = hashlib.sha256()
    src = os.path.join(ROOT, "quantized_rl_rollout_gb300", "csrc")
    for name in sorted(os.listdir(src)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            h.update(open(os.path.join(src, name), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "qrr.h"), "rb").read())
    return h.hexdigest()


def record_traffic(csv_path):
    """Median DRAM bytes per launch of each phase kernel in an ncu CSV launch
    list, written to profiles/traffic.json with the current source hash."""
    per = {}
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    rows = list(csv.DictReader(lines))
    launches = {}
    for r in rows:
        launches.setdefault(r["ID"], {"name": r["Kernel Name"]})[r["Metric Name"]] = float(
            r["Metric Value"].replace(",", ""))
    for phase, (prefix, targs) in PHASE_KERNELS.items():
        vals = [v["dram__bytes_read.sum"] + v["dram__bytes_write.sum"] for v in launches.values()
                if prefix in v["name"] and targs.replace(" ", "") in v["name"].replace(" ", "")
                and "dram__bytes_read.sum" in v and "dram__bytes_write.sum" in v]
        if vals:
            per[phase] = {"kernel": prefix + targs, "dram_bytes_per_launch": statistics.median(vals),
                          "launches": len(vals)}
    out = {"source_sha256": source_hash(), "from": os.path.basename(csv_path), "phases": per}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out, indent=1))


def load_traffic(phase):
    try:
        d = json.load(open(TRAFFIC_FILE))
    except (OSError, ValueError):
        return None
    if d.get("source_sha256") != source_hash():
        return None
    e = d.get("phases", {}).get(phase)
    return e["dram_bytes_per_launch"] if e else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = dict(FALLBACK_PEAKS)
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                if key in d and isinstance(d[key], (int, float)):
                    out[key] = float(d[key])
            out["source"] = "measured"
            return out
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS)


# ---------------------------------------------------------------------------
# algorithmic bytes / flops


def decode_bytes(layers, m, r):
    total = 0
    for l in layers:
        total += l.n * l.k // 2 + l.n * l.k // 16 + 4  # codes, block scales, tensor scale
        total += 2 * r * (l.k + l.n)  # LoRA A and B
        total += 2 * m * l.k + 2 * m * l.n  # x in, y out
    return total


def linear_flops(layers, m, r):
    return sum(2 * m * l.n * l.k + 2 * m * r * (l.k + l.n) for l in layers)


def requant_nvfp4_bytes(layers):
    # two sweeps over the bf16 weight (the codes depend on the tensor-wide absmax)
    return sum(2 * 2 * l.n * l.k + l.n * l.k // 2 + l.n * l.k // 16 + 4 for l in layers)


def fp8_quant_bytes(layers, m):
    w = sum(2 * l.n * l.k + l.n * l.k + 4 * ((l.n + 127) // 128) * (l.k // 128) for l in layers)
    a = sum(2 * m * l.k + m * l.k + 4 * m * (l.k // 128) for l in layers)
    return w, a


def lora_bwd_flops(layers, m, r):
    """dX = dY . W_hat (2 M N K) + the adapter's five rank-r products:
    dY . B (2 M N r), (.) . A (2 M r K), dA (2 r K M), x . A^T (2 M K r), dB (2 N r M)."""
    return sum(2 * m * l.n * l.k + 2 * m * r * (2 * l.n + 3 * l.k) for l in layers)


def fp8_gemm_flops(layers, m):
    return sum(2 * m * l.n * l.k for l in layers)


def measure_fp8_peak(device, n=8192, reps=10):
    """Dense E4M3 GEMM throughput of torch._scaled_mm (cuBLASLt) at n^3 on this
    GPU: best of `reps` back-to-back launches, TFLOP/s; None if unsupported."""
    try:
        a = torch.randn(n, n, device=device).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=device).to(torch.float8_e4m3fn).t()  # column-major operand
        one = torch.ones((), device=device, dtype=torch.float32)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b
        return 2.0 * n ** 3 / best / 1e9
    except Exception:  # noqa: BLE001 - an unsupported op leaves the nominal ratio in place
        return None


# ---------------------------------------------------------------------------


class Clocks:
    """SM clock, power and throttle reasons sampled DURING a region, read-only.

    Polls NVML directly (libnvidia-ml through ctypes) every 10 ms, so even a
    timed region of a few tens of milliseconds gets several samples; falls back
    to ``nvidia-smi -lms 200`` when NVML cannot be loaded.  Nothing here changes
    a setting of the GPU."""

    # clocks-event-reason bits of NVML
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index, period_s=0.01):
        self.index = index
        self.period = period_s
        self.samples = []  # (sm_mhz, max_mhz, reasons bitmask or names)
        self.proc = None
        self.thread = None
        self.stop_evt = threading.Event()
        self.source = None

    def _nvml_handle(self):
        import ctypes

        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        bus = None
        try:
            props = torch.cuda.get_device_properties(self.index)
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        except (AttributeError, RuntimeError):
            bus = None
        if bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        return nv, h

    def _poll_nvml(self, nv, h):
        import ctypes

        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_evt.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), float(mx.value), int(rs.value)))
            time.sleep(self.period)

    def start(self):
        try:
            nv, h = self._nvml_handle()
            self.source = "nvml 10 ms"
            self.thread = threading.Thread(target=self._poll_nvml, args=(nv, h), daemon=True)
            self.thread.start()
            return
        except OSError:
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi 200 ms"
            self.thread = threading.Thread(target=self._read_smi, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            self.samples.append((sm, mx, [n for n, v in zip(names, parts[4:8]) if v.lower() == "active"]))

    def stop(self):
        self.stop_evt.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        if not self.samples:
            return None
        reasons = set()
        for _, _, r in self.samples:
            if isinstance(r, int):
                reasons.update(name for bit, name in self.REASONS.items() if r & bit)
            else:
                reasons.update(r)
        sm = [a for a, _, _ in self.samples]
        return {"sm_mhz": statistics.median(sm), "sm_mhz_min": min(sm), "sm_max_mhz": max(b for _, b, _ in self.samples),
                "samples": len(sm), "source": self.source, "reasons": sorted(reasons)}


class Workload:
    """Device tensors of one step (weights resident in HBM before timing)."""

    def __init__(self, qrr, device, seed=0):
        self.q = qrr
        self.dev = device
        self.layers = configs.LAYERS_8B
        L = self.layers
        self.W = [inputs.weight(l.n, l.k, inputs.derive_seed(seed, "8b", l.name, "W"), device=device) for l in L]
        # the trainer's N(0, 1e-4) update of every master: successive steps
        # re-quantize W and W' in turn, so each re-quantization sees new weights
        self.Wu = [inputs.updated(w, inputs.derive_seed(seed, "8b", l.name, "update")) for w, l in zip(self.W, L)]
        self.masters = self.W
        self.lora = [inputs.lora(R, l.k, l.n, inputs.derive_seed(seed, "8b", l.name, "lora"), device=device)[:2]
                     for l in L]
        self.nv = [(torch.empty(l.n, l.k // 2, dtype=torch.uint8, device=device),
                    torch.empty(l.n, l.k // 16, dtype=torch.uint8, device=device),
                    torch.empty(1, dtype=torch.float32, device=device)) for l in L]
        self.xd = {m: [inputs.activations(m, l.k, inputs.derive_seed(seed, "8b", l.name, "x", m), device=device)
                       for l in L] for m in DECODE_TOKENS}
        self.yd = {m: [torch.empty(m, l.n, dtype=torch.bfloat16, device=device) for l in L] for m in DECODE_TOKENS}
        self.xp = [inputs.activations(PREFILL_TOKENS, l.k, inputs.derive_seed(seed, "8b", l.name, "xp"), device=device,
                                      channel_outlier_frac=0.01) for l in L]
        self.yp = [torch.empty(PREFILL_TOKENS, l.n, dtype=torch.bfloat16, device=device) for l in L]
        self.f8w = [(torch.empty(l.n, l.k, dtype=torch.uint8, device=device),
                     torch.empty((l.n + 127) // 128, l.k // 128, dtype=torch.float32, device=device)) for l in L]
        self.f8a = [(torch.empty(PREFILL_TOKENS, l.k, dtype=torch.uint8, device=device),
                     torch.empty(PREFILL_TOKENS, l.k // 128, dtype=torch.float32, device=device)) for l in L]
        self.yf = [torch.empty(PREFILL_TOKENS, l.n, dtype=torch.bfloat16, device=device) for l in L]
        # power-of-two-scale operands for the native block-scaled GEMM
        self.f8w2 = [qrr.quantize_fp8_w128x128(w, qrr.SCALE_POW2) for w in self.W]
        self.f8a2 = [qrr.quantize_fp8_a1x128(x, qrr.SCALE_POW2) for x in self.xp]
        self.gd = {m: self._group(self.xd[m], self.yd[m]) for m in DECODE_TOKENS}
        self.gp = self._group(self.xp, self.yp)
        ws = max([qrr.linear_nvfp4_lora_grouped_workspace_bytes(self.gd[m]) for m in DECODE_TOKENS] +
                 [qrr.linear_nvfp4_lora_grouped_workspace_bytes(self.gp)])
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        self.rq_ws = torch.empty(4096, dtype=torch.uint8, device=device)
        self.flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
        self.flush_sum = torch.zeros((), dtype=torch.float32, device=device)
        self.launches = 0

    def next_step(self):
        self.masters = self.Wu if self.masters is self.W else self.W

    # each phase returns the number of library kernels it launched
    def requant(self):
        self.q.requantize_weights(self.masters, self.nv, self.q.FORMAT_NVFP4, workspace=self.rq_ws)
        return 2

    def _group(self, xs, ys):
        out = []
        for i, _ in enumerate(self.layers):
            c, s, t = self.nv[i]
            A, B = self.lora[i]
            out.append(dict(x=xs[i], codes=c, scales=s, tensor_scale=t, lora_A=A, lora_B=B, alpha=ALPHA, y=ys[i]))
        return out

    def decode(self, m):
        # the whole layer set in one grouped call: LoRA/f16 prologue + one GEMM launch
        self.q.linear_nvfp4_lora_grouped(self.gd[m], workspace=self.ws)
        return 2

    def prefill(self):
        self.q.linear_nvfp4_lora_grouped(self.gp, workspace=self.ws)
        return 2

    def fp8_requant(self):
        self.q.requantize_weights(self.masters, self.f8w, self.q.FORMAT_FP8_W128)
        return 1

    def fp8_act_quant(self):
        for i, _ in enumerate(self.layers):
            self.q.quantize_fp8_a1x128(self.xp[i], q=self.f8a[i][0], scales=self.f8a[i][1])
        return len(self.layers)

    def fp8_gemm(self):
        for i, _ in enumerate(self.layers):
            qa, sa = self.f8a[i]
            qw, sw = self.f8w[i]
            self.q.gemm_fp8_blockwise(qa, sa, qw, sw, y=self.yf[i])
        return len(self.layers)

    def fp8_gemm_pow2(self):
        for i, _ in enumerate(self.layers):
            qa, sa = self.f8a2[i]
            qw, sw = self.f8w2[i]
            self.q.gemm_fp8_blockwise(qa, sa, qw, sw, self.q.SCALE_POW2, y=self.yf[i])
        return len(self.layers)

    def requant_aqn(self):
        # step-dependent noise strength of a geometric schedule over 100 steps
        self.aqn_step = getattr(self, "aqn_step", 0) + 1
        sigma = self.q.aqn_sigma(self.aqn_step % 100, 100, 1e-2, 5e-4)
        self.q.requantize_weights_aqn(self.masters, self.nv, sigma, 0x5EED, self.aqn_step, workspace=self.rq_ws)
        return 2

    def _bwd(self):
        if getattr(self, "bw", None) is None:
            L = self.layers
            dy = [inputs.activations(PREFILL_TOKENS, l.n, inputs.derive_seed(0, "8b", l.name, "dy"), device=self.dev)
                  for l in L]
            dx = [torch.empty(PREFILL_TOKENS, l.k, dtype=torch.bfloat16, device=self.dev) for l in L]
            dA = [torch.empty(R, l.k, dtype=torch.float32, device=self.dev) for l in L]
            dB = [torch.empty(l.n, R, dtype=torch.float32, device=self.dev) for l in L]
            ws = torch.empty(max(self.q.lora_backward_workspace_bytes(PREFILL_TOKENS, l.n, l.k, R) for l in L),
                             dtype=torch.uint8, device=self.dev)
            self.bw = (dy, dx, dA, dB, ws)
        return self.bw

    def lora_bwd(self):
        dy, dx, dA, dB, ws = self._bwd()
        for i, _ in enumerate(self.layers):
            c, s, t = self.nv[i]
            A, B = self.lora[i]
            self.q.lora_backward_nvfp4(dy[i], self.xp[i], c, s, t, A, B, ALPHA, dx=dx[i], dA=dA[i], dB=dB[i],
                                       workspace=ws)
        return 7 * 7  # per layer: transpose, factor transpose, rank projections, GEMM, 2 x (partials, reduce)

    def _attn(self):
        if getattr(self, "at", None) is None:
            b, hq, hkv, lmax = ATT_B, ATT_HQ, ATT_HKV, ATT_L
            g = torch.Generator(device="cpu")
            g.manual_seed(inputs.derive_seed(0, "attn", "lens"))
            lens = torch.randint(lmax // 2, lmax, (b,), generator=g, dtype=torch.int32)  # room for the new token
            kq, ks = self.q.quantize_fp8_a1x128(inputs.activations(b * hkv * lmax, 128,
                                                                   inputs.derive_seed(0, "attn", "k"), device=self.dev))
            vq, vs = self.q.quantize_fp8_a1x128(inputs.activations(b * hkv * lmax, 128,
                                                                   inputs.derive_seed(0, "attn", "v"), device=self.dev))
            qq = inputs.activations(b * hq, 128, inputs.derive_seed(0, "attn", "q"), device=self.dev).view(b, hq, 128)
            kn = inputs.activations(b * hkv, 128, inputs.derive_seed(0, "attn", "kn"), device=self.dev).view(b, hkv, 128)
            vn = inputs.activations(b * hkv, 128, inputs.derive_seed(0, "attn", "vn"), device=self.dev).view(b, hkv, 128)
            ws = torch.empty(self.q.lib().qrr_attention_decode_fp8_workspace_bytes(b, hq, lmax), dtype=torch.uint8,
                             device=self.dev)
            self.at = dict(kc=kq.view(b, hkv, lmax, 128), ks=ks.view(b, hkv, lmax), vc=vq.view(b, hkv, lmax, 128),
                           vs=vs.view(b, hkv, lmax), q=qq, kn=kn, vn=vn, pos=lens.to(self.dev),
                           lens=(lens + 1).to(self.dev), out=torch.empty_like(qq), ws=ws,
                           bytes=int((lens + 1).sum()) * hkv * 2 * (128 + 4) + 2 * b * hq * 128 * 2
                           + b * hkv * 2 * (128 * 2 + 128 + 4))
        return self.at

    def attn_fp8(self):
        a = self._attn()
        self.q.kv_append_fp8(a["kn"], a["vn"], a["pos"], a["kc"], a["ks"], a["vc"], a["vs"])
        self.q.attention_decode_fp8(a["q"], a["kc"], a["ks"], a["vc"], a["vs"], a["lens"], out=a["out"],
                                    workspace=a["ws"])
        return 3

    def stream_floor(self):
        # the memory-system floor of one decode pass: the one-token decode's
        # bytes as a [rows x 2048] byte matrix (the shape of a 4096-wide
        # layer's packed codes) through the decode kernels' TMA ring, no arithmetic
        if getattr(self, "sbuf", None) is None:
            rows = -(-decode_bytes(self.layers, 1, R) // (2048 * 128)) * 128
            self.sbuf = torch.zeros(rows, 2048, dtype=torch.uint8, device=self.dev)
        self.q.stream_probe(self.sbuf)
        return 1

    def rollout_is(self):
        if getattr(self, "lg", None) is None:
            # token log-probabilities / importance weights over an 8B-class vocabulary
            self.lg = inputs.logits(IS_TOKENS, IS_VOCAB, inputs.derive_seed(0, "is", "logits"), device=self.dev)
            self.tok = inputs.sampled_tokens(self.lg, inputs.derive_seed(0, "is", "tokens"))
            self.rlp = inputs.jitter(torch.full((IS_TOKENS,), -2.0, device=self.dev), inputs.derive_seed(0, "is", "r"),
                                     1.0)
            self.lp = torch.empty(IS_TOKENS, dtype=torch.float32, device=self.dev)
            self.iw = torch.empty(IS_TOKENS, dtype=torch.float32, device=self.dev)
        self.q.token_logprobs_is(self.lg, self.tok, self.rlp, IS_CAP, logp=self.lp, w=self.iw)
        return 1

    def do_flush(self):
        self.flush.fill_(self.launches & 0xFF)
        torch.sum(self.flush.view(torch.float32), dim=0, out=self.flush_sum)

    # -- 32B-class stack (built on first use: ~62 GB of bf16 masters) --
    def _stack32(self):
        if getattr(self, "s32", None) is None:
            L, c = configs.LAYERS_32B, configs.DECODE_32B
            masters, outs, groups = [], [], []
            for li in range(c["depth"]):
                grp = []
                for l in L:
                    masters.append(inputs.weight(l.n, l.k, inputs.derive_seed(0, "32b", li, l.name, "W"),
                                                 device=self.dev))
                    codes = torch.empty(l.n, l.k // 2, dtype=torch.uint8, device=self.dev)
                    scales = torch.empty(l.n, l.k // 16, dtype=torch.uint8, device=self.dev)
                    ts = torch.empty(1, dtype=torch.float32, device=self.dev)
                    outs.append((codes, scales, ts))
                    A, B, alpha = inputs.lora(c["r"], l.k, l.n, inputs.derive_seed(0, "32b", li, l.name, "lora"),
                                              device=self.dev)
                    x = inputs.activations(c["tokens"], l.k, inputs.derive_seed(0, "32b", li, l.name, "x"),
                                           device=self.dev)
                    grp.append(dict(x=x, codes=codes, scales=scales, tensor_scale=ts, lora_A=A, lora_B=B, alpha=alpha,
                                    y=torch.empty(c["tokens"], l.n, dtype=torch.bfloat16, device=self.dev)))
                groups.append(grp)
            ws = torch.empty(self.q.linear_nvfp4_lora_grouped_workspace_bytes(groups[0]), dtype=torch.uint8,
                             device=self.dev)
            rq_ws = torch.empty(self.q.lib().qrr_requantize_workspace_bytes(len(masters)), dtype=torch.uint8,
                                device=self.dev)
            self.s32 = (masters, outs, groups, ws, rq_ws)
            self.requant32()
        return self.s32

    def requant32(self):
        masters, outs, _, _, rq_ws = self._stack32()
        self.q.requantize_weights(masters, outs, self.q.FORMAT_NVFP4, workspace=rq_ws)
        return 2 * ((len(masters) + 47) // 48)

    def decode32(self):
        _, _, groups, ws, _ = self._stack32()
        for grp in groups:
            self.q.linear_nvfp4_lora_grouped(grp, workspace=ws)
        return 2 * len(groups)


# one step over the 8B-class workload (the hot path's method steps); the
# 32B-class stack (another configuration, ~85 GB resident) and the next rows
# built beside the path (AQN re-quantization, LoRA backward, FP8-KV attention,
# importance weights) are timed after it, each in a region of its own
PHASES = ["requant", "decode_m1", "decode_m8", "decode_m64", "prefill", "fp8_requant", "fp8_act_quant", "fp8_gemm",
          "fp8_gemm_pow2"]
NEXT_PHASES = ["requant_aqn", "lora_bwd", "attn_fp8", "rollout_is", "stream_floor"]
EXTRA_PHASES = ["requant32b", "decode32b"]


def run_phase(w, name):
    if name == "requant":
        return w.requant()
    if name.startswith("decode_m"):
        return w.decode(int(name[len("decode_m"):]))
    if name == "prefill":
        return w.prefill()
    if name == "fp8_requant":
        return w.fp8_requant()
    if name == "fp8_act_quant":
        return w.fp8_act_quant()
    if name == "decode32b":
        return w.decode32()
    if name == "requant32b":
        return w.requant32()
    if name == "fp8_gemm_pow2":
        return w.fp8_gemm_pow2()
    if name == "rollout_is":
        return w.rollout_is()
    if name == "requant_aqn":
        return w.requant_aqn()
    if name == "lora_bwd":
        return w.lora_bwd()
    if name == "attn_fp8":
        return w.attn_fp8()
    if name == "stream_floor":
        return w.stream_floor()
    return w.fp8_gemm()


def timed_steps(w, steps, phases):
    """Per-phase device ms (lists over steps) and kernel launches in the timed region.
    The region is an NVTX range "timed" (free without a tool attached), so a
    profiler can be limited to the timed launches (ncu --nvtx --nvtx-include
    "timed/")."""
    stream = torch.cuda.current_stream()
    times = {p: [] for p in phases}
    launches = 0
    torch.cuda.nvtx.range_push("timed")
    for _ in range(steps):
        w.next_step()
        for p in phases:
            w.do_flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launches += run_phase(w, p)
            e1.record(stream)
            times[p].append((e0, e1))
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    out = {p: [a.elapsed_time(b) for a, b in times[p]] for p in phases}
    return out, launches


def e2e_decode(w, steps):
    """Decode through the public API with host buffers.  Per step, for each
    token count: one copy of every layer's tokens from pinned host memory
    (the layers' x are one contiguous block), the grouped call over the 7
    linears (a ``GroupedLinear`` prepared once on the fixed device buffers, as
    a decode loop holds them), and one copy of every y back.  The copies run on a second stream
    (the copy engines), ordered against the grouped calls by events, so the
    copies of one token count overlap the kernels of another.
    Returns (median ms, h2d bytes, d2h bytes)."""
    L = w.layers
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    hx, hy, dxb, dyb, groups = {}, {}, {}, {}, {}
    for m in DECODE_TOKENS:
        nx = sum(m * l.k for l in L)
        ny = sum(m * l.n for l in L)
        hx[m] = torch.cat([x.reshape(-1) for x in w.xd[m]]).cpu().pin_memory()
        hy[m] = torch.empty(ny, dtype=torch.bfloat16).pin_memory()
        dxb[m] = torch.empty(nx, dtype=torch.bfloat16, device=w.dev)
        dyb[m] = torch.empty(ny, dtype=torch.bfloat16, device=w.dev)
        xs, ys, ox, oy = [], [], 0, 0
        for l in L:
            xs.append(dxb[m][ox:ox + m * l.k].view(m, l.k))
            ys.append(dyb[m][oy:oy + m * l.n].view(m, l.n))
            ox += m * l.k
            oy += m * l.n
        groups[m] = w.q.GroupedLinear(w._group(xs, ys), workspace=w.ws)
    h2d = sum(t.numel() * 2 for t in hx.values())
    landed = {m: torch.cuda.Event() for m in DECODE_TOKENS}
    done = {m: torch.cuda.Event() for m in DECODE_TOKENS}
    d2h = sum(t.numel() * 2 for t in hy.values())

    def one(start):
        copy.wait_event(start)
        with torch.cuda.stream(copy):
            for m in DECODE_TOKENS:
                dxb[m].copy_(hx[m], non_blocking=True)
                landed[m].record(copy)
        for m in DECODE_TOKENS:
            compute.wait_event(landed[m])
            groups[m].run()
            done[m].record(compute)
            copy.wait_event(done[m])
            with torch.cuda.stream(copy):
                hy[m].copy_(dyb[m], non_blocking=True)
        compute.wait_stream(copy)

    for _ in range(3):
        e = torch.cuda.Event()
        e.record(compute)
        one(e)
    torch.cuda.synchronize()
    ms = []
    for _ in range(steps):
        w.do_flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(compute)
        one(e0)
        e1.record(compute)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.median(ms), h2d, d2h


# ---------------------------------------------------------------------------
# CPU oracle timing


def oracle_decode_sample(seconds_target):
    """Time the oracle on a bounded sample of the decode workload: NVFP4
    quantize of the q layer (4096 x 4096) once, then the float64 W4A16 +
    LoRA linear for 1, 8 and 64 tokens, repeated until ~seconds_target.
    Returns (GB/s of decode bytes handled, seconds, sample description)."""
    import oracle

    layer = configs.LAYERS_8B[0]
    g = np.random.default_rng(0)
    w = g.standard_normal((layer.n, layer.k)).astype(np.float32) * np.float32(0.02)
    w = oracle.formats.bf16_rne(w)
    a = oracle.formats.bf16_rne(g.standard_normal((R, layer.k)) * 0.01)
    b = oracle.formats.bf16_rne(g.standard_normal((layer.n, R)) * 0.01)
    t0 = time.perf_counter()
    codes, scales, s_t = oracle.nvfp4.quantize(w)
    bytes_done = 0
    reps = 0
    while True:
        for m in DECODE_TOKENS:
            x = oracle.formats.bf16_rne(g.standard_normal((m, layer.k)))
            oracle.linear.linear_nvfp4_lora(x, codes, scales, s_t, a, b, ALPHA)
            bytes_done += decode_bytes([layer], m, R)
        reps += 1
        if time.perf_counter() - t0 >= seconds_target:
            break
    secs = time.perf_counter() - t0
    desc = (f"oracle NVFP4 quantize of one 4096x4096 layer + float64 W4A16+LoRA linear at M=1,8,64, "
            f"{reps} repetitions, decode bytes of that layer per repetition")
    return bytes_done / secs / 1e9, secs, desc


def oracle_phase_rates(seconds_each=3.0):
    """The oracle's rate on each other phase of the step, on bounded samples
    (each repeated until about `seconds_each`): NVFP4 quantization and FP8
    128x128 quantization of one 4096x4096 weight (GB/s of bf16 read), FP8
    1x128 quantization of 256 tokens x 4096, and the float64 blockwise FP8 GEMM
    for 16 tokens of a 4096x4096 layer (GFLOP/s).  Single process."""
    import oracle

    g = np.random.default_rng(1)
    n = k = 4096
    w = oracle.formats.bf16_rne(g.standard_normal((n, k)).astype(np.float32) * np.float32(0.02))
    x = oracle.formats.bf16_rne(g.standard_normal((256, k)).astype(np.float32))

    def rate(fn, units):
        t0 = time.perf_counter()
        reps = 0
        while True:
            out = fn()
            reps += 1
            if time.perf_counter() - t0 >= seconds_each:
                break
        return units * reps / (time.perf_counter() - t0), reps, out

    out = {}
    r, reps, _ = rate(lambda: oracle.nvfp4.quantize(w), 2.0 * n * k / 1e9)
    out["nvfp4_quantize"] = {"value": r, "unit": "GB/s", "sample": f"one {n}x{k} weight, {reps} reps"}
    r, reps, (qw, sw) = rate(lambda: oracle.fp8.quantize_w128x128(w), 2.0 * n * k / 1e9)
    out["fp8_w128_quantize"] = {"value": r, "unit": "GB/s", "sample": f"one {n}x{k} weight, {reps} reps"}
    r, reps, (qa, sa) = rate(lambda: oracle.fp8.quantize_a1x128(x), 2.0 * x.size / 1e9)
    out["fp8_a1x128_quantize"] = {"value": r, "unit": "GB/s", "sample": f"256x{k} activations, {reps} reps"}
    r, reps, _ = rate(lambda: oracle.fp8.gemm_blockwise(qa[:16], sa[:16], qw, sw), 2.0 * 16 * n * k / 1e9)
    out["fp8_gemm"] = {"value": r, "unit": "GFLOP/s", "sample": f"16 tokens x {n}x{k} layer, {reps} reps"}
    return out


def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001 - threadpoolctl is optional
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ---------------------------------------------------------------------------


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        return rank, world, local, dist
    return 0, 1, 0, None


def max_over_ranks(dist, value):
    """The largest of every rank's value (NCCL on GPU ranks, gloo on CPU)."""
    if dist is None:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job(dist, world, bytes_per_rank, ms_per_rank):
    """Replicas: every rank moves the same bytes; the job's throughput is
    all ranks' bytes over the slowest rank's time (GB/s), or None."""
    ms = max_over_ranks(dist, ms_per_rank)
    return world * bytes_per_rank / ms / 1e6 if ms else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--phases", default=",".join(PHASES))
    ap.add_argument("--skip-extras", action="store_true", help="no e2e or CPU-oracle legs (for profiler runs)")
    ap.add_argument("--no-32b", action="store_true", help="do not build or time the 32B-class stack")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="write profiles/traffic.json from an ncu launch list (dram bytes) and exit")
    args = ap.parse_args()
    if args.record_traffic:
        record_traffic(args.record_traffic)
        return
    warmup = max(3, args.warmup)
    rank, world, local, dist = dist_setup(args.gpus)

    if args.impl == "reference":
        if rank != 0:
            return
        vals = []
        total_s = 0.0
        desc = ""
        for i in range(warmup + args.steps):
            v, s, desc = oracle_decode_sample(seconds_target=2.0)
            if i >= warmup:
                vals.append(v)
                total_s += s
        value = statistics.median(vals)
        cores = cpu_cores()
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
                "steps": args.steps, "warmup": warmup, "ms_per_step": 1000.0 * total_s / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": WORKLOAD, "sample": desc},
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    from quantized_rl_rollout_gb300 import qrr

    qrr.lib()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    asked = [p for p in args.phases.split(",") if p]
    phases = [p for p in asked if p in PHASES]
    nxt = [p for p in asked if p in NEXT_PHASES]
    extra = [p for p in asked if p in EXTRA_PHASES]
    if args.phases == ",".join(PHASES):  # the default: every region
        nxt = list(NEXT_PHASES)
        extra = [] if args.no_32b else list(EXTRA_PHASES)
    peaks = load_peaks()
    fp8_meas = measure_fp8_peak(device)
    w = Workload(qrr, device)
    w.requant()  # valid NVFP4 weights for every phase, whichever phases run
    # warm-up (untimed)
    for _ in range(warmup):
        w.next_step()
        for p in phases:
            run_phase(w, p)
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    per_phase, launches = timed_steps(w, args.steps, phases)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()

    # the next rows beside the path: a region of their own after the step
    # (same protocol: warm-up, L2 flush before every phase)
    per_next, clk_next = {}, None
    if nxt:
        for _ in range(warmup):
            for p in nxt:
                run_phase(w, p)
        torch.cuda.synchronize()
        clocks_n = Clocks(local)
        clocks_n.start()
        per_next, l_next = timed_steps(w, args.steps, nxt)
        torch.cuda.synchronize()
        clk_next = clocks_n.stop()

    # the 32B-class stack: another configuration, timed in a region of its own
    per_extra, clk32, wall32 = {}, None, None
    if extra:
        for p in extra:  # builds the stack on first use
            run_phase(w, p)
        for _ in range(max(1, warmup - 2)):
            for p in extra:
                run_phase(w, p)
        torch.cuda.synchronize()
        clocks32 = Clocks(local)
        clocks32.start()
        t0 = time.perf_counter()
        per_extra, l32 = timed_steps(w, args.steps, extra)
        torch.cuda.synchronize()
        wall32 = time.perf_counter() - t0
        clk32 = clocks32.stop()

    med = {p: statistics.median(v) for p, v in per_phase.items()}
    med_extra = {p: statistics.median(v) for p, v in per_extra.items()}
    med_extra.update({p: statistics.median(v) for p, v in per_next.items()})
    L = configs.LAYERS_8B
    fp8_peak = fp8_meas if fp8_meas else 2.0 * peaks["bf16_tflops"]
    fp8_peak_source = "measured in this run (torch._scaled_mm E4M3 8192^3, best of 10)" if fp8_meas else \
        "2 x measured bf16 (nominal FP8:BF16 ratio)"

    def hbm(ms, b):
        return {"ms": ms, "GB/s": b / ms / 1e6, "frac_hbm": b / ms / 1e6 / peaks["hbm_gbs"],
                "frac_hbm_spec": b / ms / 1e6 / SPEC_PEAKS["hbm_gbs"], "bytes": b}

    breakdown = {}
    dec_bytes = 0
    dec_ms = 0.0
    for p, ms in list(med.items()) + list(med_extra.items()):
        if p.startswith("decode_m"):
            m = int(p[len("decode_m"):])
            b = decode_bytes(L, m, R)
            dec_bytes += b
            dec_ms += ms
            breakdown[p] = hbm(ms, b)
        elif p in ("requant", "requant_aqn"):
            breakdown[p] = hbm(ms, requant_nvfp4_bytes(L))
        elif p == "prefill":
            f = linear_flops(L, PREFILL_TOKENS, R)
            breakdown[p] = {"ms": ms, "TFLOP/s": f / ms / 1e9, "frac_bf16": f / ms / 1e9 / peaks["bf16_tflops"],
                            "frac_bf16_sustained": f / ms / 1e9 / peaks["bf16_tflops_sustained"],
                            "frac_bf16_spec": f / ms / 1e9 / SPEC_PEAKS["bf16_tflops"], "flops": f}
        elif p == "attn_fp8":
            breakdown[p] = hbm(ms, w._attn()["bytes"])
            breakdown[p]["workload"] = (f"{ATT_B} sequences, {ATT_HQ} query / {ATT_HKV} KV heads of 128, "
                                        f"E4M3 cache of {ATT_L // 2}..{ATT_L} tokens: append one step + attention")
        elif p == "lora_bwd":
            f = lora_bwd_flops(L, PREFILL_TOKENS, R)
            breakdown[p] = {"ms": ms, "TFLOP/s": f / ms / 1e9, "frac_bf16": f / ms / 1e9 / peaks["bf16_tflops"],
                            "frac_bf16_spec": f / ms / 1e9 / SPEC_PEAKS["bf16_tflops"], "flops": f}
        elif p == "fp8_requant":
            breakdown[p] = hbm(ms, fp8_quant_bytes(L, PREFILL_TOKENS)[0])
        elif p == "fp8_act_quant":
            breakdown[p] = hbm(ms, fp8_quant_bytes(L, PREFILL_TOKENS)[1])
        elif p in ("fp8_gemm", "fp8_gemm_pow2"):
            f = fp8_gemm_flops(L, PREFILL_TOKENS)
            breakdown[p] = {"ms": ms, "TFLOP/s": f / ms / 1e9, "frac_fp8": f / ms / 1e9 / fp8_peak,
                            "frac_fp8_spec": f / ms / 1e9 / SPEC_PEAKS["fp8_tflops"], "flops": f,
                            "scale_mode": "fp32 (promotion)" if p == "fp8_gemm" else
                            "pow2 (native block-scaled MMA, UE8M0)"}
        elif p == "stream_floor":
            breakdown[p] = hbm(ms, w.sbuf.numel())
            breakdown[p]["workload"] = ("TMA stream of the one-token decode's bytes in [128 x 128 B] boxes, "
                                        "no arithmetic (the memory floor of one such pass)")
            if "decode_m1" in med:
                breakdown[p]["decode_m1_over_floor_time"] = ms / med["decode_m1"]
        elif p == "rollout_is":
            breakdown[p] = hbm(ms, IS_TOKENS * IS_VOCAB * 2 + IS_TOKENS * 16)
            breakdown[p]["workload"] = f"{IS_TOKENS} tokens x {IS_VOCAB} vocabulary, bf16 logits"
        elif p == "decode32b":
            c32 = configs.DECODE_32B
            breakdown[p] = hbm(ms, c32["depth"] * decode_bytes(configs.LAYERS_32B, c32["tokens"], c32["r"]))
            breakdown[p]["region"] = "separate (after the step)"
        elif p == "requant32b":
            breakdown[p] = hbm(ms, configs.DECODE_32B["depth"] * requant_nvfp4_bytes(configs.LAYERS_32B))
            breakdown[p]["region"] = "separate (after the step)"

    for p in per_next:
        breakdown[p]["region"] = "separate (after the step)"
    step_ms = sum(med.values()) if med else sum(med_extra.values())
    step_ms = max_over_ranks(dist, step_ms)
    value = whole_job(dist, world, dec_bytes, dec_ms) if dec_ms else None

    # dominant phase of the step -> roofline object
    all_med = dict(med_extra, **med)
    dom = max(phases, key=lambda p: med[p]) if phases else max(all_med, key=lambda p: all_med[p])
    d = breakdown[dom]
    if "GB/s" in d:
        roof = {"bound": "hbm", "achieved": d["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": d["GB/s"] / peaks["hbm_gbs"], "peak_spec": SPEC_PEAKS["hbm_gbs"],
                "frac_spec": d["GB/s"] / SPEC_PEAKS["hbm_gbs"]}
    elif dom in ("fp8_gemm", "fp8_gemm_pow2"):
        roof = {"bound": "tensor", "achieved": d["TFLOP/s"], "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": d["TFLOP/s"] / fp8_peak, "peak_spec": SPEC_PEAKS["fp8_tflops"],
                "frac_spec": d["TFLOP/s"] / SPEC_PEAKS["fp8_tflops"]}
    else:
        roof = {"bound": "tensor", "achieved": d["TFLOP/s"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": d["TFLOP/s"] / peaks["bf16_tflops"], "peak_spec": SPEC_PEAKS["bf16_tflops"],
                "frac_spec": d["TFLOP/s"] / SPEC_PEAKS["bf16_tflops"]}
    roof["kernel_phase"] = dom
    roof["peak_source"] = peaks["source"]
    roof["traffic"] = load_traffic(dom)

    e2e = None
    cpu = None
    if rank == 0 and not args.skip_extras and any(p.startswith("decode_m") for p in phases):
        e_ms, h2d, d2h = e2e_decode(w, max(3, min(args.steps, 50)))
        e_bytes = sum(decode_bytes(L, m, R) for m in DECODE_TOKENS)
        e2e = {"value": e_bytes / e_ms / 1e6, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms,
               "mode": "grouped C-ABI calls prepared once (GroupedLinear); pinned-host copies on a copy stream, overlapped with the other token counts"}
        v, s, desc = oracle_decode_sample(seconds_target=10.0)
        bt = blas_threads()
        cpu = {"value": v, "unit": "GB/s", "cores": bt or cpu_cores(), "kind": "oracle", "sample": desc, "seconds": s,
               "blas_threads": bt, "host_cores": cpu_cores(),
               "process": "single process; elementwise numpy on one core, float64 matmul on the BLAS threads",
               "phases": oracle_phase_rates(seconds_each=2.5)}

    if clk and clk.get("sm_mhz"):
        clk["step_ms_x_sm_mhz"] = step_ms * clk["sm_mhz"]
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "nvfp4xbf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "phases": phases, "l2": "flushed before every phase: a 512 MB write, then a read of it",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                           "separately_timed": nxt + extra},
                "roofline": roof, "breakdown": breakdown, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "clocks": clk, "clocks_next_region": clk_next, "clocks_32b_region": clk32,
                "wall_s_timed": wall,
                "wall_s_timed_32b": wall32,
                "peaks": dict(peaks, fp8_tflops=fp8_peak, fp8_source=fp8_peak_source, spec=SPEC_PEAKS)}
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
