"""Benchmark of the dropless MoE layer forward pass on GB300.

Default workload (one GPU): T=8192 tokens, d=7168, d_e=2048, E=8 routed
SwiGLU experts, top-4, per-expert logit bias N(0, 0.5), one shared expert of
width 2048 (the pages' fused-MoE default shape).  A step is one whole layer
forward: router -> offsets -> permute -> grouped GEMMs -> shared expert ->
combine, on synthetic seeded inputs already resident in HBM.

Prints one JSON line:
  value    useful TFLOP/s of the layer (routed rows without padding + shared
           expert), aggregated over ranks; replicas only for N > 1
  e2e      the same metric through MoeLayer.forward with the token rows copied
           from pinned host memory and the output copied back every step
  roofline the grouped-GEMM stage (GEMM1 + SwiGLU, GEMM2 + gate) against the
           measured bf16 tensor peak
  stages   per-stage milliseconds and the permute / combine HBM GB/s
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the workload

``--impl reference`` times the CPU oracle as the reference arm.
``--weights fp8`` runs the layer with e4m3 expert weights (per-output-channel
fp32 scales; moe_layer_fwd_fp8) instead of bf16 ones.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from routing_permute_grouped_gb300 import ledger, synth  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    except OSError:
        p = dict(FALLBACK)
        p["source"] = "fallback"
        return p


# ------------------------------------------------------------ clocks ------
# NVML clock-event reason bits (nvml.h): the ones a measurement must report
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock, clock-event reasons and board power of one GPU, read every
    ``period_s`` seconds on a background thread while a region runs.

    NVML is read through ctypes (libnvidia-ml ships with the driver); where
    it cannot be loaded, ``nvidia-smi -lms`` is the fallback.  Readings only:
    nothing here changes a setting of the GPU.  ``mark(name)`` / ``window``
    record wall-clock spans (the host enqueues far ahead and synchronises at
    the end of each span, so the device is busy during it) and ``summary``
    reports the samples taken inside a span."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.idx = device_index
        self.period = period_s
        self.samples = []  # (wall time, sm MHz, reason bits, power W or None)
        self.sm_max = None
        self.power_limit = None
        self.spans = {}
        self._stop = threading.Event()
        self.thread = None
        self.proc = None
        self.source = None

    # -- NVML through ctypes
    def _nvml_open(self):
        import ctypes

        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None or lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        try:  # the CUDA device's own GPU, matched by UUID
            uuid = str(torch.cuda.get_device_properties(self.idx).uuid)
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) == 0
        except Exception:  # noqa: BLE001
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.idx, ctypes.byref(h)) != 0:
            return None
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
            self.sm_max = float(mx.value)
        if lib.nvmlDeviceGetEnforcedPowerLimit(h, ctypes.byref(mx)) == 0:  # milliwatts
            self.power_limit = mx.value / 1e3
        return lib, h

    def _nvml_loop(self, lib, h):
        import ctypes

        class FieldValue(ctypes.Structure):  # nvmlFieldValue_t
            _fields_ = [("fieldId", ctypes.c_uint), ("scopeId", ctypes.c_uint),
                        ("timestamp", ctypes.c_longlong), ("latencyUsec", ctypes.c_longlong),
                        ("valueType", ctypes.c_int), ("nvmlReturn", ctypes.c_int),
                        ("value", ctypes.c_ulonglong)]

        def power_w():
            # instantaneous board power (NVML_FI_DEV_POWER_INSTANT, milliwatts);
            # nvmlDeviceGetPowerUsage, a one-second average on recent GPUs,
            # where the field is not served
            fv = FieldValue(fieldId=186)
            if lib.nvmlDeviceGetFieldValues(h, 1, ctypes.byref(fv)) == 0 and fv.nvmlReturn == 0:
                if fv.valueType == 0:
                    return ctypes.cast(ctypes.pointer(ctypes.c_ulonglong(fv.value)),
                                       ctypes.POINTER(ctypes.c_double))[0] / 1e3
                if fv.valueType in (1, 5):
                    return (fv.value & 0xFFFFFFFF) / 1e3
                return fv.value / 1e3
            return mw.value / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0 else None

        mhz = ctypes.c_uint()
        mw = ctypes.c_uint()
        bits = ctypes.c_ulonglong()
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            t = time.time()
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                r = bits.value if reasons(h, ctypes.byref(bits)) == 0 else 0
                self.samples.append((t, float(mhz.value), int(r), power_w()))
            time.sleep(self.period)

    # -- nvidia-smi fallback
    def _smi_read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) < 8:
                continue
            try:
                sm = float(parts[0])
                self.sm_max = float(parts[1])
            except ValueError:
                continue
            bits = 0
            for b, v in zip((0x8, 0x40, 0x20, 0x4), parts[4:8]):
                if v.lower().startswith("active"):
                    bits |= b
            try:
                w = float(parts[2])
            except ValueError:
                w = None
            self.samples.append((time.time(), sm, bits, w))

    def start(self):
        nv = None
        try:
            nv = self._nvml_open()
        except Exception:  # noqa: BLE001
            nv = None
        if nv is not None:
            self.source = "nvml"
            self.thread = threading.Thread(target=self._nvml_loop, args=nv, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._smi_read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def window(self, name: str, t0: float, t1: float):
        self.spans[name] = (t0, t1)

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, span: str = None):
        """Median SM MHz, the reasons seen and the median and largest board
        power (W) among the samples inside the span (all samples when span is
        None), with the enforced power limit."""
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock readings unavailable"]}
        sel = self.samples
        if span is not None and span in self.spans:
            t0, t1 = self.spans[span]
            sel = [x for x in self.samples if t0 <= x[0] <= t1]
        reasons = sorted({n for x in sel for bit, n in _NVML_REASONS.items() if x[2] & bit})
        sm = [x[1] for x in sel]
        pw = [x[3] for x in sel if len(x) > 3 and x[3] is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.sm_max,
                "reasons": reasons, "samples": len(sm), "source": self.source,
                "period_ms": self.period * 1e3 if self.source == "nvml" else 100.0,
                "power_w_median": round(statistics.median(pw), 1) if pw else None,
                "power_w_max": round(max(pw), 1) if pw else None,
                "power_limit_w": self.power_limit}


def clock_normalised(stage_ms: float, roof: dict, clk):
    """Stage time against the SM clock seen while it ran: ms x median MHz
    (thousands of SM cycles) and the rate the same cycles would give at the
    maximum SM clock.  A stage held back by the power cap shows a median
    below the maximum; one held back by its code does not."""
    if not clk or not clk.get("sm_mhz") or not clk.get("sm_max_mhz"):
        return None
    scale = clk["sm_max_mhz"] / clk["sm_mhz"]
    return {"sm_mhz_median": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
            "samples": clk.get("samples"), "stage_ms_x_mhz": stage_ms * clk["sm_mhz"],
            "achieved_at_max_clock": roof["achieved"] * scale,
            "frac_at_max_clock": roof["achieved"] * scale / roof["peak"]}


# --------------------------------------------------------- distributed ----
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(v: float, world: int) -> float:
    """Maximum of a host value over all ranks (the slowest rank sets the
    job time)."""
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------ oracle ------
def oracle_sample_tflops(shape, inp_host: dict, n_tokens: int):
    """fp64 CPU oracle on n_tokens tokens of the workload: router for those
    tokens, their routed experts (direct per-token evaluation) and the shared
    expert.  Returns (useful TFLOP/s, seconds, threads)."""
    import numpy as np

    import oracle

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    tok = np.arange(n_tokens, dtype=np.int32)
    x = bits(inp_host["x"][:n_tokens])
    t0 = time.perf_counter()
    if inp_host.get("Wg") is not None:
        bias = None if inp_host.get("bias") is None else inp_host["bias"].numpy()
        lg = oracle.router_logits(x, bits(inp_host["Wg"]), bias)
        idx, w, _ = oracle.route(lg, shape.k, shape.n_groups, shape.topk_groups)
    else:
        idx = inp_host["topk_idx"][:n_tokens].numpy()
        w = inp_host["topk_w"][:n_tokens].double().numpy()
    ys = None
    if shape.d_shared:
        _, ys = oracle.shared_expert(x, bits(inp_host["Ws1"]), bits(inp_host["Ws3"]),
                                     bits(inp_host["Ws2"]))
    oracle.direct_layer(np.arange(n_tokens, dtype=np.int32), x, bits(inp_host["W1"]),
                        bits(inp_host["W3"]), bits(inp_host["W2"]), idx, w, ys)
    dt = time.perf_counter() - t0
    flops = ledger.layer_useful_flops(n_tokens, shape.k, shape.d, shape.d_e, shape.d_shared)
    if inp_host.get("Wg") is not None:
        flops += ledger.router_flops(n_tokens, shape.d, shape.E)
    return flops / dt / 1e12, dt, oracle.num_threads()


def oracle_train_sample_tflops(shape, inp_host: dict, n_tokens: int):
    """fp64 CPU oracle forward + backward of the layer on the first n_tokens
    tokens of the workload (the same weights; upstream gradient seeded).
    Returns (useful TFLOP/s, seconds, threads)."""
    import dataclasses

    import numpy as np

    import oracle

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    sub = dataclasses.replace(shape, T=n_tokens)
    oi = {}
    for key, v in inp_host.items():
        if v is None:
            oi[key] = None
        elif key in ("topk_idx", "topk_w", "x"):
            v = v[:n_tokens]
            oi[key] = bits(v) if v.dtype == torch.bfloat16 else (
                v.double().numpy() if key == "topk_w" else v.numpy())
        elif v.dtype == torch.bfloat16:
            oi[key] = bits(v)
        else:
            oi[key] = v.numpy()
    gen = torch.Generator().manual_seed(shape.seed + 1000)
    dout = torch.randn((n_tokens, shape.d), generator=gen).to(torch.bfloat16).double().numpy()
    t0 = time.perf_counter()
    fwd = oracle.layer_forward(oi, sub)
    oracle.layer_backward(oi, sub, fwd, dout)
    dt = time.perf_counter() - t0
    flops = train_useful_flops(sub)
    return flops / dt / 1e12, dt, oracle.num_threads()


def train_useful_flops(shape) -> int:
    """Forward + backward useful FLOP of one layer step (router included when
    the layer routes)."""
    E = 0 if shape.prerouted else shape.E
    fwd = ledger.layer_useful_flops(shape.T, shape.k, shape.d, shape.d_e, shape.d_shared)
    fwd += ledger.router_flops(shape.T, shape.d, E) if E else 0
    return fwd + ledger.layer_backward_useful_flops(shape.T, shape.k, shape.d, shape.d_e,
                                                    shape.d_shared, E)


def host_inputs(shape):
    """CPU copies of the workload (seeded; same generator as the GPU run)."""
    return synth.make_inputs(shape, device="cpu")


# -------------------------------------------------------- reference arm ---
def run_reference(args, shape, rank, world):
    if rank != 0:
        return
    import oracle

    inp = host_inputs(shape)
    if args.pass_ == "train":
        return run_reference_train(args, shape, inp)
    n_tok = max(1, oracle.num_threads())  # one token per oracle thread per step
    for _ in range(args.warmup):
        oracle_sample_tflops(shape, inp, n_tok)
    t0 = time.perf_counter()
    flops = 0
    threads = 1
    for _ in range(args.steps):
        _, _, threads = oracle_sample_tflops(shape, inp, n_tok)
        flops += ledger.layer_useful_flops(n_tok, shape.k, shape.d, shape.d_e, shape.d_shared)
        flops += ledger.router_flops(n_tok, shape.d, shape.E) if not shape.prerouted else 0
    dt = time.perf_counter() - t0
    val = flops / dt / 1e12
    sample = (f"{n_tok} token(s) of the workload per step (router, routed experts, shared "
              f"expert), {n_tok} oracle threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(shape, weights=args.weights),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_train(args, shape, inp):
    import oracle

    n_tok = max(1, oracle.num_threads())
    for _ in range(args.warmup):
        oracle_train_sample_tflops(shape, inp, n_tok)
    t0 = time.perf_counter()
    threads = 1
    for _ in range(args.steps):
        _, _, threads = oracle_train_sample_tflops(shape, inp, n_tok)
    dt = time.perf_counter() - t0
    flops = train_useful_flops(__import__("dataclasses").replace(shape, T=n_tok)) * args.steps
    val = flops / dt / 1e12
    sample = (f"{n_tok} token(s) of the workload per step: the oracle's layer forward and "
              f"backward on them")
    line = {
        "impl": "reference", "metric": METRIC_TRAIN, "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(config_dict(shape, weights=args.weights), **{"pass": "train"}),
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "MoE layer fwd useful TFLOP/s (bf16, fp32 accumulate)"
METRIC_TRAIN = "MoE layer fwd+bwd useful TFLOP/s (bf16, fp32 accumulate)"
METRIC_FP8 = "MoE layer fwd useful TFLOP/s (e4m3 expert weights, fp32 accumulate)"


def config_dict(shape, permute="layer", weights="bf16", schedule="padded", combine="kernel"):
    return {"workload": f"{shape.name}: T={shape.T} d={shape.d} d_e={shape.d_e} E={shape.E} "
                        f"k={shape.k} groups={shape.n_groups}/{shape.topk_groups} "
                        f"pad={shape.pad} shared={shape.d_shared}",
            "permute": permute, "combine": combine, "expert_weights": weights,
            "schedule": schedule,
            "l2": "inputs larger than L2 (expert weights and permuted rows exceed 129 MB)",
            "parallelism": "replicas"}


# -------------------------------------------------------------- ours ------
def run_ours(args, shape, rank, world, local):
    import routing_permute_grouped_gb300 as moe
    from routing_permute_grouped_gb300 import build as moe_build

    moe_build.build()
    moe.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    # token rows, router weight and routing on the host (the same draws as the
    # tests and the Zipf calibration), expert weights drawn on the GPU
    inp = synth.make_inputs(shape, device="cpu", weights_device=dev)
    for key in ("x", "Wg", "bias", "topk_idx", "topk_w"):
        if inp.get(key) is not None:
            inp[key] = inp[key].to(dev)
    cfg = moe.config_of(shape)
    fp8 = args.weights == "fp8"
    if fp8 and (args.permute == "gather" or args.combine != "kernel"):
        raise SystemExit("--weights fp8 runs with the layer's permute and combine")
    unpadded = args.schedule == "unpadded"
    if unpadded and (fp8 or args.permute == "gather" or args.combine != "kernel" or
                     shape.T * shape.k <= 32 * shape.E):
        raise SystemExit("--schedule unpadded runs the CTA-pair GEMMs with bf16 weights and the "
                         "permute and combine kernels")
    layer = moe.MoeLayer(cfg, inp["W1"], inp["W3"], inp["W2"], Wg=inp.get("Wg"),
                         bias=inp.get("bias"), Ws1=inp.get("Ws1"), Ws3=inp.get("Ws3"),
                         Ws2=inp.get("Ws2"), fp8=fp8)
    x = inp["x"]
    out = torch.empty_like(x)
    L = layer.layout
    ws = layer.ws
    i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
    T, k, E, d, de, ds = shape.T, shape.k, shape.E, shape.d, shape.d_e, shape.d_shared
    A, R, NB = shape.A, shape.rows_capacity, shape.blocks_capacity
    buf = layer.buffer
    topk_idx = buf("topk_idx", i32, (T, k)) if not shape.prerouted else inp["topk_idx"]
    topk_w = buf("topk_w", f32, (T, k)) if not shape.prerouted else inp["topk_w"]
    counts, po = buf("counts", i32, (E,)), buf("padded_offsets", i32, (E + 1,))
    meta, nb = buf("block_metadata", i32, (NB, 3)), buf("num_blocks", i32, (1,))
    perm_row, row_src = buf("perm_row", i32, (A,)), buf("row_src", i32, (R,))
    row_gate = buf("row_gate", f32, (R,))
    h, y = buf("h", bf, (R, de)), buf("y", bf, (R, d))
    hs = buf("hs", bf, (T, ds)) if ds else None
    ys = buf("ys", bf, (T, d)) if ds else None
    # the layer's kernel choice: the small-M kernel (shared expert merged
    # into its launches) when the mean rows per expert is at most 32; above
    # that, e4m3 weights are widened to bf16 for the CTA-pair kernel
    skinny = T * k <= 32 * E
    wide = fp8 and not skinny
    if wide:  # the widened codes: routed W13, W2, then shared Ws13, Ws2
        n13, n2, ns13 = E * 2 * de * d, E * d * de, 2 * ds * d
        W13w = buf("w16", bf, (n13,))
        W2w = buf("w16", bf, (n2,), offset=2 * n13)
        Ws13w = buf("w16", bf, (ns13,), offset=2 * (n13 + n2)) if ds else None
        Ws2w = buf("w16", bf, (ns13 // 2,), offset=2 * (n13 + n2 + ns13)) if ds else None
    if fp8 and not wide:  # e4m3 pairs of the activations and their row scales
        u8 = torch.uint8
        x_perm = buf("x_perm", u8, (2 * R, d))
        h8 = buf("h8", u8, (2 * R, de))
        x_scale = buf("row_scale", f32, (R,))
        h_scale = buf("row_scale", f32, (R,), offset=4 * R)
        xs8 = buf("xs8", u8, (2 * T, d)) if ds else None
        hs8 = buf("h8", u8, (2 * T, ds), offset=2 * R * de) if ds else None
        xs_scale = buf("row_scale", f32, (T,), offset=8 * R) if ds else None
        hs_scale = buf("row_scale", f32, (T,), offset=8 * R + 4 * T) if ds else None
    else:
        x_perm = buf("x_perm", bf, (R, d))
    status_word = buf("status", i32, (1,))
    nsplit = moe.moe_route_splitk_scratch_size(cfg) // 4 if not shape.prerouted else 0
    router_partial = buf("router_partial", f32, (nsplit,)) if nsplit else None
    offs_ws = ws[L["status"]:L["topk_idx"]]

    # The stages in enqueue order, (name, call).  By default they mirror
    # moe_layer_fwd: on the bf16 CTA-pair path with a shared expert, the
    # shared GEMM1 runs before the routed GEMMs with the permute in its
    # epilogue, the shared GEMM2 after them, then the combine.  (With e4m3
    # weights widened for the CTA-pair kernel the layer does the same with the
    # scaled GEMMs; the stage pass there runs the permute kernel and the whole
    # scaled shared expert after the routed GEMMs.)
    pair_shared = bool(ds) and not skinny and not fp8 and not unpadded
    perm_in_shared = pair_shared and args.permute == "layer"
    # --permute gemm: the permute in GEMM1's copy warps (stage calls)
    perm_in_gemm = not skinny and not fp8 and not unpadded and args.permute == "gemm"
    visit_ready = buf("visit_ready", i32, (NB,))
    stages = []
    if not shape.prerouted:
        # the router the layer runs: split-K for small batches
        stages.append(("route", lambda: moe.moe_route_splitk(
            cfg, x, layer.Wg_t, layer.bias, topk_idx, topk_w, router_partial)))
    if unpadded:  # group offsets in po, no block table
        stages.append(("offsets", lambda: moe.moe_build_offsets_unpadded(
            cfg, topk_idx, topk_w, counts, po, perm_row, row_src, row_gate, offs_ws)))
    else:
        stages.append(("offsets", lambda: moe.moe_build_offsets(
            cfg, topk_idx, topk_w, counts, po, meta, nb, perm_row, row_src, row_gate, offs_ws)))
    if perm_in_shared:
        stages.append(("shared_up_permute", lambda: moe.moe_shared_expert_up(
            cfg, x, layer.Ws13, hs, perm_row, x_perm, status_word)))
    elif fp8 and not wide:
        stages.append(("permute", lambda: moe.moe_permute_fp8(
            cfg, x, perm_row, x_perm, x_scale, xs8, xs_scale)))
    elif args.permute != "gather" and not perm_in_gemm:
        stages.append(("permute", lambda: moe.moe_permute(cfg, x, perm_row, x_perm)))

    def grouped():
        if wide:  # widen the routed codes, then the scaled bf16 GEMMs
            moe.moe_widen_e4m3(layer.W13q, W13w)
            moe.moe_widen_e4m3(layer.W2q, W2w)
            moe.moe_grouped_gemm_swiglu_scaled(cfg, x_perm, W13w, layer.s13, W2w, layer.s2, meta,
                                               nb, po, row_gate, h, y, status_word)
        elif fp8:
            moe.moe_grouped_gemm_swiglu_fp8(cfg, x_perm, x_scale, layer.W13q, layer.s13, layer.W2q,
                                            layer.s2, meta, nb, row_gate, h, h8, h_scale, y,
                                            status_word)
        elif unpadded:
            moe.moe_grouped_gemm_swiglu_unpadded(cfg, x_perm, layer.W13, layer.W2_t, po, row_gate,
                                                 h, y, status_word)
        elif skinny:
            moe.moe_grouped_gemm_swiglu_skinny(cfg, x_perm, layer.W13, layer.W2_t, meta, nb,
                                               row_gate, h, y, status_word)
        elif perm_in_gemm:
            moe.moe_grouped_gemm_swiglu_permute(cfg, x, row_src, x_perm, visit_ready, layer.W13,
                                                layer.W2_t, meta, nb, po, row_gate, h, y,
                                                status_word)
        elif args.permute != "gather":
            moe.moe_grouped_gemm_swiglu(cfg, x_perm, layer.W13, layer.W2_t, meta, nb, po, row_gate,
                                        h, y, status_word)
        else:
            moe.moe_grouped_gemm_swiglu_gather(cfg, x, row_src, layer.W13, layer.W2_t, meta, nb, po,
                                               row_gate, h, y, status_word)

    stages.append(("grouped_gemm", grouped))
    fused_combine = pair_shared and args.combine == "fused"
    if pair_shared:
        if not perm_in_shared:
            stages.append(("shared_up", lambda: moe.moe_shared_expert_up(
                cfg, x, layer.Ws13, hs, None, None, status_word)))
        if fused_combine:
            stages.append(("shared_down_combine", lambda: moe.moe_shared_expert_down_combine(
                cfg, hs, layer.Ws2_t, y, perm_row, out, status_word)))
        else:
            stages.append(("shared_down", lambda: moe.moe_shared_expert_down(
                cfg, hs, layer.Ws2_t, ys, status_word)))
    elif ds:
        def shared():
            if wide:
                moe.moe_widen_e4m3(layer.Ws13q, Ws13w)
                moe.moe_widen_e4m3(layer.Ws2q, Ws2w)
                moe.moe_shared_expert_scaled(cfg, x, Ws13w, layer.ss13, Ws2w, layer.ss2, hs, ys,
                                             status_word)
            elif fp8:
                moe.moe_shared_expert_fp8(cfg, xs8, xs_scale, layer.Ws13q, layer.ss13, layer.Ws2q,
                                          layer.ss2, hs, hs8, hs_scale, ys, status_word)
            else:
                moe.moe_shared_expert(cfg, x, layer.Ws13, layer.Ws2_t, hs, ys, status_word)

        stages.append(("shared", shared))
    if not fused_combine:
        stages.append(("combine", lambda: moe.moe_combine(cfg, y, perm_row, ys, out)))
    stage_names = [n for n, _ in stages]

    def step(ev=None):
        for i, (_, call) in enumerate(stages):
            if ev is not None:
                ev[i].record()
            call()
        if ev is not None:
            ev[len(stages)].record()

    launches_per_step = forward_launches(shape, skinny, fp8,
                                         "kernel" if unpadded else args.permute, args.combine)
    topk_kw_dev = dict(topk_idx=inp["topk_idx"], topk_w=inp["topk_w"]) if shape.prerouted else {}

    def layer_step():
        if args.permute == "layer" and args.combine == "kernel" and not unpadded:
            layer(x, out, **topk_kw_dev)  # moe_layer_fwd: the whole layer, one call
        else:
            step()

    for _ in range(max(args.warmup, 3)):
        layer_step()
        step()
    torch.cuda.synchronize()
    timed_step = layer_step
    if args.graph:
        # the whole-layer call recorded once into a CUDA graph (the layer only
        # enqueues kernels: no host sync, no allocation); each timed step
        # replays it, so the host issues one launch per step instead of one
        # per kernel
        if not (args.permute == "layer" and args.combine == "kernel" and not unpadded):
            raise SystemExit("--graph records the whole-layer call: default --permute, "
                             "--combine and --schedule only")
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            layer_step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer_step()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        timed_step = graph.replay
    # timed region: K whole-layer forwards (moe_layer_fwd: every stage on the
    # calling stream, or the replay of its graph), bracketed by CUDA events on
    # that stream
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    t_start.record()
    for i in range(args.steps):
        timed_step()
    t_end.record()
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    ms_total = t_start.elapsed_time(t_end)
    ms_max = reduce_max(ms_total, world)
    # stage pass, also timed: the same kernels called stage by stage on one
    # stream, each stage bracketed by CUDA events on that stream, for the
    # per-stage breakdown and the grouped-GEMM roofline
    n_stage = min(args.steps, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stage_names) + 1)]
           for _ in range(n_stage)]
    torch.cuda.synchronize()
    w2 = time.time()
    for i in range(n_stage):
        step(evs[i])
    torch.cuda.synchronize()
    w3 = time.time()
    # per-stage median over the stage-pass steps
    stage_ms = {n: statistics.median(ev[j].elapsed_time(ev[j + 1]) for ev in evs)
                for j, n in enumerate(stage_names)}

    counts_h = counts.cpu().tolist()
    useful = ledger.layer_useful_flops(T, k, d, de, ds)
    flops_job = reduce_sum(useful * args.steps, world)
    value = flops_job / (ms_max / 1e3) / 1e12
    st = layer.device_status()
    if st:
        raise RuntimeError(f"device status bits {st:#x}")

    # e2e through the public API with host buffers: every step copies its
    # token rows from pinned host memory and its output back; HostPipeline
    # overlaps the copies of neighbouring steps with the layer's compute
    x_host = x.cpu().pin_memory()
    out_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    topk_kw = {}
    h2d = x_host.numel() * 2
    if shape.prerouted:
        idx_host = inp["topk_idx"].cpu().pin_memory()
        w_host = inp["topk_w"].cpu().pin_memory()
        topk_kw = dict(topk_idx=idx_host, topk_w=w_host)
        h2d += idx_host.numel() * 4 + w_host.numel() * 4
    d2h = x_host.numel() * 2
    e2e_steps = max(1, min(args.steps, 100))
    pipe = moe.HostPipeline(layer)
    for i in range(3):
        pipe.submit(x_host, out_host[i % 2], **topk_kw)
    pipe.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w4 = time.time()
    e0.record(pipe.s_in)
    for i in range(e2e_steps):
        pipe.submit(x_host, out_host[i % 2], **topk_kw)
    e1.record(pipe.s_out)
    pipe.synchronize()
    w5 = time.time()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world)
    e2e_val = reduce_sum(useful * e2e_steps, world) / (e2e_ms / 1e3) / 1e12
    clocks = stage_clocks = e2e_clocks = None
    if sampler:  # one sampler over the three regions, summarised per region
        sampler.stop()
        sampler.window("timed", w0, w1)
        sampler.window("stages", w2, w3)
        sampler.window("e2e", w4, w5)
        clocks = sampler.summary("timed")
        stage_clocks = sampler.summary("stages")
        e2e_clocks = sampler.summary("e2e")

    pk = peaks()
    gemm_flops = ledger.routed_flops(A, d, de)
    active = sum(1 for c in counts_h if c > 0)
    gemm_bytes = ledger.grouped_gemm_bytes_alg(A, active, d, de, fp8_weights=fp8)
    gemm_s = stage_ms["grouped_gemm"] / 1e3
    # the stage is timed by CUDA events launch by launch (about 2 ms each,
    # well under a second), so its peak is the burst bf16 figure; the
    # sustained one (a seconds-long loop under the power cap) is context
    peak_t = pk["bf16_tflops"]
    # the stage is tensor-bound when its FLOP per byte exceeds the machine
    # balance (measured bf16 FLOP/s over measured HBM bytes/s), else HBM-bound
    hbm_bound = gemm_flops / gemm_bytes < peak_t * 1e12 / (pk["hbm_gbs"] * 1e9)
    if hbm_bound:
        roof = {"bound": "hbm", "achieved": gemm_bytes / gemm_s / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "peak_source": pk["source"] + " copy bandwidth"}
    else:
        roof = {"bound": "tensor", "achieved": gemm_flops / gemm_s / 1e12, "peak": peak_t,
                "unit": "TFLOP/s", "peak_source": pk["source"] + " burst bf16"}
        if "bf16_tflops_sustained" in pk:
            roof["frac_of_sustained"] = roof["achieved"] / pk["bf16_tflops_sustained"]
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["clock"] = clock_normalised(stage_ms["grouped_gemm"], roof, stage_clocks)
    roof["algorithmic"] = {"flop": gemm_flops, "bytes": gemm_bytes, "active_experts": active}
    perm_bytes = ledger.permute_bytes_alg(T, k, d)
    comb_bytes = ledger.combine_bytes_alg(T, k, d, bool(ds))
    perm_gbs = perm_bytes / (stage_ms["permute"] / 1e3) / 1e9 if "permute" in stage_ms else None
    comb_gbs = comb_bytes / (stage_ms["combine"] / 1e3) / 1e9 if "combine" in stage_ms else None
    traffic = recorded_traffic("skinny_gemm" if skinny else "grouped_gemm",
                               shape.name + ("_fp8" if fp8 else ""))
    line = {
        "metric": METRIC_FP8 if fp8 else METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 (weights, widened to bf16 for the MMAs; per-channel scales on the fp32 "
                  "accumulators)" if wide else
                  "e4m3 (weights; activations as e4m3 pairs), fp32 accumulate" if fp8 else "bf16"),
        "data": "synthetic", "config": dict(config_dict(shape, args.permute, args.weights,
                                                          args.schedule, args.combine),
                                              **({"timed_call": "CUDA graph replay of the layer"}
                                                 if args.graph else {})),
        "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "clocks": e2e_clocks},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": dict(roof, kernel="grouped GEMM stage (GEMM1+SwiGLU, GEMM2+gate)",
                         timing="stage pass: CUDA events around " + (
                             "moe_widen_e4m3 (routed codes) + moe_grouped_gemm_swiglu_scaled"
                             if wide else
                             "moe_grouped_gemm_swiglu_fp8" if fp8 else
                             "moe_grouped_gemm_swiglu_skinny" if skinny else
                             "moe_grouped_gemm_swiglu"),
                         traffic=traffic),
        "stages": {"ms": {n: round(v, 4) for n, v in stage_ms.items()},
                   "clocks": stage_clocks,
                   "serial_sum_ms": round(sum(stage_ms.values()), 4),
                   "permute_gbs": perm_gbs,
                   "permute_frac_hbm": perm_gbs / pk["hbm_gbs"] if perm_gbs else None,
                   "combine_gbs": comb_gbs,
                   "combine_frac_hbm": comb_gbs / pk["hbm_gbs"] if comb_gbs else None,
                   "expert_counts": counts_h,
                   "padded_rows": ledger.padded_rows(counts_h, shape.pad),
                   # 256-row windows the CTA pairs execute under each schedule
                   "visits": {"padded": ledger.padded_tiles(counts_h, shape.pad, 256),
                              "unpadded": ledger.unpadded_tiles(counts_h, 256)}},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {kk: (v.cpu() if isinstance(v, torch.Tensor) else v) for kk, v in inp.items()}
        # calibrate to ~20 s of oracle work: one token per thread first
        import oracle

        n0 = max(1, oracle.num_threads())
        _, dt1, _ = oracle_sample_tflops(shape, host, n0)
        n = max(n0, min(shape.T, n0 * int(round(20.0 / max(dt1, 1e-3)))))
        tf, dt, threads = oracle_sample_tflops(shape, host, n)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {n} tokens of the workload: router, routed "
                                          f"experts and shared expert ({dt:.1f} s)"
                                          + (", bf16 weights (the e4m3 evaluation does the same "
                                             "fp64 work)" if fp8 else "")}
    if rank == 0:
        print(json.dumps(line), flush=True)


def forward_launches(shape, skinny: bool, fp8: bool = False, permute: str = "layer",
                     combine: str = "kernel") -> int:
    """Kernels of one layer forward: router (2 when split-K with a scratch:
    partial logits + reduce; 1 fused or clustered), offsets (1 to 3), permute
    (none where the layer runs it in the shared expert's GEMM1 epilogue,
    on the CTA-pair path with a shared expert, nor in GEMM1's A load or its
    copy warps), 2 routed GEMMs, 2 shared-expert GEMMs (none on the small-M
    kernel,
    whose launches carry the shared tiles), combine (none when it runs in the
    shared expert's GEMM2 epilogue), and with e4m3 weights the split of h
    between the GEMMs."""
    import routing_permute_grouped_gb300 as moe

    cfg = moe.config_of(shape)
    nsplit = moe.moe_route_splitk_scratch_size(cfg) // 4 if not shape.prerouted else 0
    # one-CTA offsets kernel for small batches; else the chunk histograms and
    # the scatter (with the scan inside it while chunks x experts <= 8192),
    # or histograms, scan and scatter
    n_chunks = (shape.A + 2047) // 2048
    offsets_launches = 1 if shape.A <= 4096 else (2 if n_chunks * shape.E <= 8192 else 3)
    widen = (2 + (2 if shape.d_shared else 0)) if fp8 and not skinny else 0
    pair_shared = bool(shape.d_shared) and not skinny
    # on the CTA-pair path with a shared expert the layer's permute rides in
    # the shared GEMM1's epilogue
    permute_kernel = skinny or permute == "kernel" or (permute == "layer" and not pair_shared)
    fused_combine = pair_shared and not fp8 and combine == "fused"
    return ((0 if shape.prerouted else (2 if nsplit else 1)) + offsets_launches
            + (1 if permute_kernel else 0) + 2
            + (2 if pair_shared else 0) + (0 if fused_combine else 1)
            + (1 if fp8 and skinny else 0)  # e4m3 pairs of h between the small-M GEMMs
            + widen)


def backward_launches(shape, router_grads: bool = True, recompute: bool = True) -> int:
    """Kernels of one moe_layer_bwd call."""
    # permutes of dout and x; dh, SwiGLU backward, dx_perm; dW2, dW1 + dW3
    n = 2 + 3 + 2
    if recompute:
        n += 1  # the gate/up values recomputed (else read from the forward's save)
    if not shape.prerouted:
        n += 2  # router backward; dx from the router
        if router_grads:
            n += 2  # dbias column sums; dWg
    if shape.d_shared:
        # [gate/up,] dh, SwiGLU backward, dx; 2 weight gradients
        n += (6 if recompute else 5)
    return n + 1  # dx combine


def run_train(args, shape, rank, world, local):
    """Forward + backward of the layer per step (moe_layer_fwd, moe_layer_bwd)."""
    import routing_permute_grouped_gb300 as moe
    from routing_permute_grouped_gb300 import build as moe_build

    if args.weights != "bf16":
        raise SystemExit("--pass train runs with bf16 expert weights")
    moe_build.build()
    moe.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = synth.make_inputs(shape, device="cpu", weights_device=dev)
    for key in ("x", "Wg", "bias", "topk_idx", "topk_w"):
        if inp.get(key) is not None:
            inp[key] = inp[key].to(dev)
    cfg = moe.config_of(shape)
    layer = moe.MoeLayer(cfg, inp["W1"], inp["W3"], inp["W2"], Wg=inp.get("Wg"),
                         bias=inp.get("bias"), Ws1=inp.get("Ws1"), Ws3=inp.get("Ws3"),
                         Ws2=inp.get("Ws2"), keep_gate_up=args.keep_gate_up)
    T, k, d, de, ds = shape.T, shape.k, shape.d, shape.d_e, shape.d_shared
    x = inp["x"]
    out = torch.empty_like(x)
    gen = torch.Generator().manual_seed(shape.seed + 1000)
    dout = torch.randn((T, d), generator=gen).to(torch.bfloat16).to(dev)
    pre = bool(shape.prerouted)
    kw = dict(topk_idx=inp["topk_idx"], topk_w=inp["topk_w"]) if pre else {}
    layer(x, out, **kw)
    grads = layer.backward(x, dout, prerouted=pre)

    def train_step():
        layer(x, out, **kw)
        layer.backward(x, dout, grads=grads, prerouted=pre)

    for _ in range(max(args.warmup, 3)):
        train_step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    t0.record()
    for _ in range(args.steps):
        train_step()
    t1.record()
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    ms_max = reduce_max(t0.elapsed_time(t1), world)
    # split pass: forward and backward bracketed separately
    n_split = min(args.steps, 20)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_split)]
    w2 = time.time()
    for i in range(n_split):
        evs[i][0].record()
        layer(x, out, **kw)
        evs[i][1].record()
        layer.backward(x, dout, grads=grads, prerouted=pre)
        evs[i][2].record()
    torch.cuda.synchronize()
    w3 = time.time()
    clocks = split_clocks = None
    if sampler:
        sampler.stop()
        sampler.window("timed", w0, w1)
        sampler.window("split", w2, w3)
        clocks = sampler.summary("timed")
        split_clocks = sampler.summary("split")
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    st = layer.device_status()
    if st:
        raise RuntimeError(f"device status bits {st:#x}")
    useful = train_useful_flops(shape)
    value = reduce_sum(useful * args.steps, world) / (ms_max / 1e3) / 1e12

    # e2e through the public API with host buffers: every step copies its
    # token rows and output gradient from pinned host memory and dx back
    # (weight gradients stay on the device); HostPipeline.submit_train
    # overlaps the copies of neighbouring steps with the compute
    x_host = x.cpu().pin_memory()
    dout_host = dout.cpu().pin_memory()
    dx_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    h2d = x_host.numel() * 2 + dout_host.numel() * 2
    kw_host = {}
    if pre:
        kw_host = dict(topk_idx=inp["topk_idx"].cpu().pin_memory(),
                       topk_w=inp["topk_w"].cpu().pin_memory())
        h2d += kw_host["topk_idx"].numel() * 4 + kw_host["topk_w"].numel() * 4
    d2h = x_host.numel() * 2
    e2e_steps = max(1, min(args.steps, 50))
    pipe = moe.HostPipeline(layer)
    for i in range(3):
        pipe.submit_train(x_host, dout_host, dx_host[i % 2], grads, **kw_host)
    pipe.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(pipe.s_in)
    for i in range(e2e_steps):
        pipe.submit_train(x_host, dout_host, dx_host[i % 2], grads, **kw_host)
    e1.record(pipe.s_out)
    pipe.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world)
    e2e_val = reduce_sum(useful * e2e_steps, world) / (e2e_ms / 1e3) / 1e12

    pk = peaks()
    E_r = 0 if pre else shape.E
    counts_h = layer.buffer("counts", torch.int32, (shape.E,)).cpu().tolist()
    active = sum(1 for c in counts_h if c > 0)
    bwd_flops = ledger.layer_backward_gemm_flops(T, k, d, de, ds, E_r,
                                                 recompute=not args.keep_gate_up)
    bwd_bytes = ledger.layer_backward_bytes_alg(T, k, d, de, ds, shape.E, active, not pre,
                                                recompute=not args.keep_gate_up)
    # the backward is timed call by call (a few ms each, well under a
    # second): the burst bf16 peak applies; the sustained one is context
    peak_t = pk["bf16_tflops"]
    bwd_s = bwd_ms / 1e3
    # tensor-bound when the backward's FLOP per byte exceeds the machine
    # balance (measured bf16 FLOP/s over measured HBM bytes/s), else HBM-bound
    if bwd_flops / bwd_bytes < peak_t * 1e12 / (pk["hbm_gbs"] * 1e9):
        roof = {"bound": "hbm", "achieved": bwd_bytes / bwd_s / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "peak_source": pk["source"] + " copy bandwidth"}
    else:
        roof = {"bound": "tensor", "achieved": bwd_flops / bwd_s / 1e12, "peak": peak_t,
                "unit": "TFLOP/s", "peak_source": pk["source"] + " burst bf16"}
        if "bf16_tflops_sustained" in pk:
            roof["frac_of_sustained"] = roof["achieved"] / pk["bf16_tflops_sustained"]
    roof["clock"] = clock_normalised(bwd_ms, dict(roof, frac=None), split_clocks)
    roof.update({"frac": roof["achieved"] / roof["peak"],
                 "kernel": "layer backward (moe_layer_bwd: all its kernels; GEMM FLOP incl. the "
                           "gate/up recomputation; bytes: weights read, weight gradients "
                           "written, token rows)",
                 "timing": "split pass: CUDA events around moe_layer_bwd",
                 "algorithmic": {"flop": bwd_flops, "bytes": bwd_bytes, "active_experts": active},
                 "traffic": None})
    skinny = T * k <= 32 * shape.E
    line = {
        "metric": METRIC_TRAIN, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(config_dict(shape, weights="bf16"), **{
            "pass": "train",
            "gate_up": "saved by the forward" if args.keep_gate_up else "recomputed"}),
        "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": (forward_launches(shape, skinny)
                         + backward_launches(shape, recompute=not args.keep_gate_up)) * args.steps,
        "roofline": roof,
        "stages": {"ms": {"forward": round(fwd_ms, 4), "backward": round(bwd_ms, 4)},
                   "clocks": split_clocks},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = {kk: (v.cpu() if isinstance(v, torch.Tensor) else v) for kk, v in inp.items()}
        import oracle

        n0 = max(1, oracle.num_threads())
        _, dt1, _ = oracle_train_sample_tflops(shape, host, n0)
        n = max(n0, min(T, n0 * int(round(20.0 / max(dt1, 1e-3)))))
        tf, dt, threads = oracle_train_sample_tflops(shape, host, n)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {n} tokens of the workload: the oracle's "
                                          f"layer forward and backward ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ep(args, shape, rank, world, local):
    """Expert parallelism (ep.GpuEp): rank r holds experts [r E/W, (r+1) E/W)
    and routes its own T tokens (the workload's token rows on every rank);
    dispatch and combine move one piece per (rank, expert): batched NCCL
    point-to-point operations between ranks, one gather kernel for the
    pieces a rank keeps.  At N = 1 the group has one rank and the exchange
    is that gather in each direction."""
    import socket

    import torch.distributed as dist

    import routing_permute_grouped_gb300 as moe
    from routing_permute_grouped_gb300 import build as moe_build
    from routing_permute_grouped_gb300 import ep

    moe_build.build()
    moe.load()
    if not dist.is_initialized():
        s = socket.socket()
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
        s.close()
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0,
                                world_size=1)
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = synth.make_inputs(shape, device="cpu", weights_device=dev)
    for key in ("x", "Wg", "bias", "topk_idx", "topk_w"):
        if inp.get(key) is not None:
            inp[key] = inp[key].to(dev)
    cfg = moe.config_of(shape)
    W = dist.get_world_size()
    if shape.E % W:
        raise SystemExit(f"--parallel ep needs E ({shape.E}) divisible by the ranks ({W})")
    El = shape.E // W
    sl = slice(dist.get_rank() * El, (dist.get_rank() + 1) * El)
    layer = ep.GpuEp(cfg, inp["W1"][sl].contiguous(), inp["W3"][sl].contiguous(),
                     inp["W2"][sl].contiguous(), Wg=inp.get("Wg"), bias=inp.get("bias"),
                     Ws1=inp.get("Ws1"), Ws3=inp.get("Ws3"), Ws2=inp.get("Ws2"))
    x = inp["x"]
    kw = dict(topk_idx=inp["topk_idx"], topk_w=inp["topk_w"]) if shape.prerouted else {}
    for _ in range(max(args.warmup, 3)):
        layer.forward(x, **kw)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    t0.record()
    for _ in range(args.steps):
        layer.forward(x, **kw)
    t1.record()
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    clocks = None
    if sampler:
        sampler.stop()
        sampler.window("timed", w0, w1)
        clocks = sampler.summary("timed")
    ms_max = reduce_max(t0.elapsed_time(t1), world)
    assert layer.device_status() == 0
    T, k, d, de, ds = shape.T, shape.k, shape.d, shape.d_e, shape.d_shared
    useful = ledger.layer_useful_flops(T, k, d, de, ds)
    value = reduce_sum(useful * args.steps, world) / (ms_max / 1e3) / 1e12
    # e2e: token rows in from pinned host memory, the output back, every
    # step; the copies run on their own streams with two device buffers, so
    # that they overlap the neighbouring steps' layers (as HostPipeline does
    # for the single-GPU layer)
    x_host = x.cpu().pin_memory()
    out_host = [torch.empty_like(x_host).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(1, min(args.steps, 50))

    def e2e_step(i):
        j = i % 2
        s_in.wait_event(ev_run[j])  # the buffer's previous layer has read it
        with torch.cuda.stream(s_in):
            xd[j].copy_(x_host, non_blocking=True)
            ev_in[j].record(s_in)
        cur.wait_event(ev_in[j])
        o = layer.forward(xd[j], **kw)
        ev_run[j].record(cur)
        s_out.wait_event(ev_run[j])
        with torch.cuda.stream(s_out):
            out_host[j].copy_(o, non_blocking=True)
        o.record_stream(s_out)

    for j in range(2):
        ev_run[j].record(cur)
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world)
    e2e_val = reduce_sum(useful * e2e_steps, world) / (e2e_ms / 1e3) / 1e12
    pk = peaks()
    peak_t = pk["bf16_tflops"]  # K calls of a few ms: the burst figure
    achieved = useful / (ms_max / args.steps / 1e3) / 1e12
    skinny = T * k <= 32 * shape.E
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(config_dict(shape), parallelism=f"expert parallel over {world} rank(s)"),
        "clocks": clocks,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": x_host.numel() * 2,
                "d2h_bytes_per_step": x_host.numel() * 2},
        # the layer's kernels (the routed GEMMs are two launches on either
        # kernel; the shared expert always runs its own two) plus the two
        # gathers of the exchange's reorder
        "gpu_launches": (forward_launches(shape, False) + 2) * args.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": achieved / peak_t, "peak_source": pk["source"] + " burst bf16",
                     "kernel": "the whole expert-parallel layer per rank (its kernels, the two "
                               "all-to-alls, the host sync for the split sizes)",
                     "timing": "CUDA events around the K layer calls", "traffic": None},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except OSError:
        return None
    from routing_permute_grouped_gb300 import build as moe_build

    ent = rec.get(kernel, {}).get(workload)
    if not ent or ent.get("source_digest") != moe_build.kernel_digest(moe_build.KERNEL_SOURCES[kernel]):
        return None
    return ent.get("dram_bytes_per_launch")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="default", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--permute", choices=["layer", "kernel", "gather", "gemm"], default="layer",
                    help="layer: as moe_layer_fwd (in the shared expert's GEMM1 epilogue when "
                         "there is one on the CTA-pair kernel, else its own kernel); kernel: "
                         "always its own kernel; gather: fused into GEMM1's A load; gemm: in "
                         "GEMM1's copy warps (stage calls)")
    ap.add_argument("--combine", choices=["kernel", "fused"], default="kernel",
                    help="kernel: the combine as its own kernel (the layer); fused: in the "
                         "shared expert's GEMM2 epilogue (stage calls)")
    ap.add_argument("--weights", choices=["bf16", "fp8"], default="bf16",
                    help="expert weights in bf16, or e4m3 with per-output-channel scales")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "train"], default="fwd",
                    help="fwd: the layer forward; train: forward + backward per step")
    ap.add_argument("--parallel", choices=["replicas", "ep"], default="replicas",
                    help="replicas: every rank runs the whole layer on its tokens; ep: the "
                         "routed experts are split over the ranks (NCCL all-to-alls)")
    ap.add_argument("--schedule", choices=["padded", "unpadded"], default="padded",
                    help="padded: segments padded to the block multiple (the layer); unpadded: "
                         "no padding, windows cut by an expert boundary visited once per "
                         "expert (stage calls)")
    ap.add_argument("--graph", action="store_true",
                    help="fwd: time replays of one CUDA graph of the whole-layer call")
    ap.add_argument("--keep-gate-up", action="store_true",
                    help="train: the forward saves the gate/up values, the backward skips "
                         "recomputing them")
    args = ap.parse_args()
    if args.graph and (args.impl != "ours" or args.parallel != "replicas" or args.pass_ != "fwd"):
        ap.error("--graph applies to the forward of our layer on replicas")
    rank, world, local = dist_setup(args.gpus)
    shape = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, shape, rank, world)
    elif args.parallel == "ep":
        run_ep(args, shape, rank, world, local)
    elif args.pass_ == "train":
        run_train(args, shape, rank, world, local)
    else:
        run_ours(args, shape, rank, world, local)
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
