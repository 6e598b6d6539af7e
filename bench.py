"""Benchmark of the low-precision linear-layer hot path on one GB300.

Workload (the decode configuration the headline metric is quoted on): an
8B-class decoder layer set -- q/o 4096x4096, k/v 1024x4096, gate/up
14336x4096, down 4096x14336, bf16 weights ~N(0, 0.02) with 0.1% x20
outliers -- in NVFP4 with LoRA r = 32 (alpha = 64), decoding 1, 8 and 64
tokens.  One step is one pass of the whole hot path over that layer set:

  requant  re-quantize all 7 bf16 weights to NVFP4 (absmax sweep + encode)
  decode   W4A16 + LoRA linear of all 7 layers at M = 1, 8 and 64 (one
           grouped call per token count)
  prefill  the same linears at M = 4096 (activations with 1% x10 channels)
  fp8      FP8 path at M = 4096: activation 1x128 quantize, 128x128 weight
           re-quantize, blockwise-scaled GEMM

On request (--phases ...,decode32b,requant32b) the 32B-class stack (64 layers
of hidden 5120, LoRA r = 64) is measured too: decode at M = 64 (one grouped
call per layer) and the full bf16 -> NVFP4 re-quantization of its 31.2 G
weight elements.  It is another configuration, not part of the step.

Each phase is timed with CUDA events on the launching stream after an L2
flush (a 512 MB write), so no phase reads its weights from L2 left by the
previous one.  ``value`` is the decode phase's HBM throughput: its
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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# DRAM traffic per launch of each phase's main kernel, from an ncu launch list
# (dram__bytes_read.sum + dram__bytes_write.sum).  It is recorded together with
# a hash of the CUDA sources and reported only while the sources are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
PHASE_KERNELS = {  # phase -> (kernel name prefix, template arguments as ncu prints them)
    "prefill": ("w4a16_tc_kernel", "<256, 64, 0, 3, 1>"),
    "decode_m1": ("w4a16_tc_kernel", "<16, 256, 1, 3, 0>"),
    "decode_m8": ("w4a16_tc_kernel", "<16, 256, 1, 3, 0>"),
    "decode_m64": ("w4a16_tc_kernel", "<64, 256, 1, 3, 0>"),
    "requant": ("nvfp4_encode_kernel", ""),
    "fp8_quant": ("fp8_w128_kernel", ""),
    "fp8_gemm": ("fp8_gemm_tc_kernel", ""),
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


# ---------------------------------------------------------------------------


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


class Workload:
    """Device tensors of one step (weights resident in HBM before timing)."""

    def __init__(self, qrr, device, seed=0):
        self.q = qrr
        self.dev = device
        self.layers = configs.LAYERS_8B
        L = self.layers
        self.W = [inputs.weight(l.n, l.k, inputs.derive_seed(seed, "8b", l.name, "W"), device=device) for l in L]
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
        self.gd = {m: self._group(self.xd[m], self.yd[m]) for m in DECODE_TOKENS}
        self.gp = self._group(self.xp, self.yp)
        ws = max([qrr.linear_nvfp4_lora_grouped_workspace_bytes(self.gd[m]) for m in DECODE_TOKENS] +
                 [qrr.linear_nvfp4_lora_grouped_workspace_bytes(self.gp)])
        self.ws = torch.empty(ws, dtype=torch.uint8, device=device)
        self.rq_ws = torch.empty(4096, dtype=torch.uint8, device=device)
        self.flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
        self.launches = 0

    # each phase returns the number of library kernels it launched
    def requant(self):
        self.q.requantize_weights(self.W, self.nv, self.q.FORMAT_NVFP4, workspace=self.rq_ws)
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

    def fp8_quant(self):
        self.q.requantize_weights(self.W, self.f8w, self.q.FORMAT_FP8_W128)
        for i, _ in enumerate(self.layers):
            self.q.quantize_fp8_a1x128(self.xp[i], q=self.f8a[i][0], scales=self.f8a[i][1])
        return 1 + len(self.layers)

    def fp8_gemm(self):
        for i, _ in enumerate(self.layers):
            qa, sa = self.f8a[i]
            qw, sw = self.f8w[i]
            self.q.gemm_fp8_blockwise(qa, sa, qw, sw, y=self.yf[i])
        return len(self.layers)

    def do_flush(self):
        self.flush.fill_(self.launches & 0xFF)

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


# one step over the 8B-class workload; the 32B-class stack (another
# configuration, ~85 GB resident) is measured only when asked for by --phases
PHASES = ["requant", "decode_m1", "decode_m8", "decode_m64", "prefill", "fp8_quant", "fp8_gemm"]
EXTRA_PHASES = ["decode32b", "requant32b"]


def run_phase(w, name):
    if name == "requant":
        return w.requant()
    if name.startswith("decode_m"):
        return w.decode(int(name[len("decode_m"):]))
    if name == "prefill":
        return w.prefill()
    if name == "fp8_quant":
        return w.fp8_quant()
    if name == "decode32b":
        return w.decode32()
    if name == "requant32b":
        return w.requant32()
    return w.fp8_gemm()


def timed_steps(w, steps, phases):
    """Per-phase device ms (lists over steps) and kernel launches in the timed region."""
    stream = torch.cuda.current_stream()
    times = {p: [] for p in phases}
    launches = 0
    for _ in range(steps):
        for p in phases:
            w.do_flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launches += run_phase(w, p)
            e1.record(stream)
            times[p].append((e0, e1))
    torch.cuda.synchronize()
    out = {p: [a.elapsed_time(b) for a, b in times[p]] for p in phases}
    return out, launches


def e2e_decode(w, steps):
    """Decode through the public API with host buffers.  Per step, for each
    token count: one copy of every layer's tokens from pinned host memory
    (the layers' x are one contiguous block), the grouped call over the 7
    linears, and one copy of every y back.  The copies run on a second stream
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
        groups[m] = w._group(xs, ys)
    h2d = sum(t.numel() * 2 for t in hx.values())
    d2h = sum(t.numel() * 2 for t in hy.values())

    def one(start):
        copy.wait_event(start)
        landed = {}
        with torch.cuda.stream(copy):
            for m in DECODE_TOKENS:
                dxb[m].copy_(hx[m], non_blocking=True)
                landed[m] = torch.cuda.Event()
                landed[m].record(copy)
        for m in DECODE_TOKENS:
            compute.wait_event(landed[m])
            w.q.linear_nvfp4_lora_grouped(groups[m], workspace=w.ws)
            done = torch.cuda.Event()
            done.record(compute)
            copy.wait_event(done)
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
    phases = [p for p in args.phases.split(",") if p]
    w = Workload(qrr, device)
    w.requant()  # valid NVFP4 weights for every phase, whichever phases run
    # warm-up (untimed)
    for _ in range(warmup):
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

    med = {p: statistics.median(v) for p, v in per_phase.items()}
    L = configs.LAYERS_8B
    peaks = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # nominal FP8:BF16 dense ratio of 2
    breakdown = {}
    dec_bytes = 0
    dec_ms = 0.0
    for p in phases:
        ms = med[p]
        if p.startswith("decode_m"):
            m = int(p[len("decode_m"):])
            b = decode_bytes(L, m, R)
            dec_bytes += b
            dec_ms += ms
            breakdown[p] = {"ms": ms, "GB/s": b / ms / 1e6, "frac_hbm": b / ms / 1e6 / peaks["hbm_gbs"],
                            "bytes": b}
        elif p == "requant":
            b = requant_nvfp4_bytes(L)
            breakdown[p] = {"ms": ms, "GB/s": b / ms / 1e6, "frac_hbm": b / ms / 1e6 / peaks["hbm_gbs"], "bytes": b}
        elif p == "prefill":
            f = linear_flops(L, PREFILL_TOKENS, R)
            breakdown[p] = {"ms": ms, "TFLOP/s": f / ms / 1e9, "frac_bf16": f / ms / 1e9 / peaks["bf16_tflops"],
                            "flops": f}
        elif p == "fp8_quant":
            bw, ba = fp8_quant_bytes(L, PREFILL_TOKENS)
            breakdown[p] = {"ms": ms, "GB/s": (bw + ba) / ms / 1e6, "frac_hbm": (bw + ba) / ms / 1e6 / peaks["hbm_gbs"],
                            "bytes": bw + ba}
        elif p == "decode32b":
            c32 = configs.DECODE_32B
            b = c32["depth"] * decode_bytes(configs.LAYERS_32B, c32["tokens"], c32["r"])
            breakdown[p] = {"ms": ms, "GB/s": b / ms / 1e6, "frac_hbm": b / ms / 1e6 / peaks["hbm_gbs"], "bytes": b}
        elif p == "requant32b":
            b = configs.DECODE_32B["depth"] * requant_nvfp4_bytes(configs.LAYERS_32B)
            breakdown[p] = {"ms": ms, "GB/s": b / ms / 1e6, "frac_hbm": b / ms / 1e6 / peaks["hbm_gbs"], "bytes": b}
        elif p == "fp8_gemm":
            f = sum(2 * PREFILL_TOKENS * l.n * l.k for l in L)
            breakdown[p] = {"ms": ms, "TFLOP/s": f / ms / 1e9, "frac_fp8_nominal": f / ms / 1e9 / fp8_peak, "flops": f}

    step_ms = sum(med.values())
    step_ms = max_over_ranks(dist, step_ms)
    value = whole_job(dist, world, dec_bytes, dec_ms) if dec_ms else None

    # dominant phase -> roofline object
    dom = max(phases, key=lambda p: med[p])
    d = breakdown[dom]
    if "GB/s" in d:
        roof = {"bound": "hbm", "achieved": d["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": d["GB/s"] / peaks["hbm_gbs"], "traffic": None, "kernel_phase": dom}
    elif dom == "fp8_gemm":
        roof = {"bound": "tensor", "achieved": d["TFLOP/s"], "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": d["TFLOP/s"] / fp8_peak, "traffic": None, "kernel_phase": dom}
    else:
        roof = {"bound": "tensor", "achieved": d["TFLOP/s"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": d["TFLOP/s"] / peaks["bf16_tflops"], "traffic": None, "kernel_phase": dom}
    roof["peak_source"] = peaks["source"]
    roof["traffic"] = load_traffic(dom)

    e2e = None
    cpu = None
    if rank == 0 and not args.skip_extras and any(p.startswith("decode_m") for p in phases):
        e_ms, h2d, d2h = e2e_decode(w, max(3, min(args.steps, 50)))
        e_bytes = sum(decode_bytes(L, m, R) for m in DECODE_TOKENS)
        e2e = {"value": e_bytes / e_ms / 1e6, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms,
               "mode": "grouped C-ABI calls; pinned-host copies on a copy stream, overlapped with the other token counts"}
        v, s, desc = oracle_decode_sample(seconds_target=12.0)
        cpu = {"value": v, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc, "seconds": s}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "nvfp4xbf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "phases": phases, "l2": "flushed (512 MB write) before every phase",
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "roofline": roof, "breakdown": breakdown, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "clocks": clk, "wall_s_timed": wall,
                "peaks": peaks}
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
