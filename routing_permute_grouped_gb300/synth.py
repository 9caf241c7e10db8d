"""Seeded synthetic inputs for the dropless MoE layer forward pass.

This module only draws random numbers: it holds none of the layer's
arithmetic and is shared by the tests (which feed the same tensors to the CPU
oracle and to the CUDA library) and by ``bench.py``.

Workloads (the shapes of the pages' running examples):
  tiny       T=256,  d=512,  de=256,  E=8,   k=2, no shared expert
  default    T=8192, d=7168, de=2048, E=8,   k=4, logit bias N(0, 0.5),
             shared expert of width 2048 ("MoE & MLA operators", sec. 1.2
             default shape; "Dropless and grouped GEMM", sec. 1)
  prerouted  65,536 assignments of 8192 tokens x top-8 onto 4 experts with
             sizes 21733/15004/17982/10817 ("Dropless and grouped GEMM",
             sec. 1 table), gates U(0.05, 1), no router
  decode     T=64, d=7168, de=2048, E=256, k=8, 8 expert groups of which 4
             are kept, shared expert 2048 ("Dropless and grouped GEMM",
             sec. 10 decode regime; group limit from "MoE & MLA operators",
             sec. 2.2)
  imbalance  T=16384, d=4096, de=1024, E=64, k=6, Zipf(s) logit bias with
             s set for a hottest-expert load of 1x / 2x / 4x the mean,
             padding multiple 64 or 128
  decode_e32 the decode layer's expert width with E=32, k=2, no shared
             expert: 2.8 GB of bf16 weights, every expert active; small
             enough for hardware-counter captures of the small-M kernel
  decode_e8  the same expert shapes with E=8, k=2, T=16: a small backward
             in the decode regime for captures of the weight-gradient kernel
  mid_e8     T=4096, d=4096, de=1024, E=8, k=4, shared 1024: a mid-size
             layer for captures of the backward kernels

Distributions: x ~ N(0, 1); every weight ~ N(0, std = 1/sqrt(fan_in)); all
bf16 (torch's round-to-nearest-even conversion from fp32 draws).  Each tensor
has its own generator stream, seeded from the workload's base seed
(1234 + workload index) and the tensor's name.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoeShape:
    name: str
    T: int
    d: int
    d_e: int
    E: int
    k: int
    n_groups: int = 0
    topk_groups: int = 0
    pad: int = 128
    d_shared: int = 0
    bias_std: float = 0.0          # N(0, bias_std) per-expert logit bias
    zipf_target: float = 0.0       # hottest/mean load target for a Zipf bias
    prerouted: tuple = ()          # fixed per-expert sizes (pre-routed input)
    seed: int = 1234

    @property
    def A(self) -> int:
        return self.T * self.k

    @property
    def rows_capacity(self) -> int:
        return self.A + self.E * (self.pad - 1)

    @property
    def blocks_capacity(self) -> int:
        return self.A // self.pad + self.E


def _imb(target: float, pad: int) -> MoeShape:
    return MoeShape(f"imbalance_x{int(target)}_p{pad}", T=16384, d=4096, d_e=1024, E=64, k=6,
                    pad=pad, zipf_target=target, seed=1234 + 4)


WORKLOADS = {
    "tiny": MoeShape("tiny", T=256, d=512, d_e=256, E=8, k=2, seed=1234 + 0),
    "default": MoeShape("default", T=8192, d=7168, d_e=2048, E=8, k=4, d_shared=2048,
                        bias_std=0.5, seed=1234 + 1),
    "prerouted": MoeShape("prerouted", T=8192, d=7168, d_e=2048, E=4, k=8,
                          prerouted=(21733, 15004, 17982, 10817), seed=1234 + 2),
    "decode": MoeShape("decode", T=64, d=7168, d_e=2048, E=256, k=8, n_groups=8, topk_groups=4,
                       d_shared=2048, seed=1234 + 3),
    "decode_e32": MoeShape("decode_e32", T=64, d=7168, d_e=2048, E=32, k=2, seed=5),
    # the decode expert shapes with 8 experts and 4 rows each: a small
    # backward (about 2.5 GB) for counter captures of the weight-gradient
    # kernel in the decode regime
    "decode_e8": MoeShape("decode_e8", T=16, d=7168, d_e=2048, E=8, k=2, seed=7),
    # a mid-size layer (a few GB with its backward) for counter captures
    "mid_e8": MoeShape("mid_e8", T=4096, d=4096, d_e=1024, E=8, k=4, d_shared=1024,
                       bias_std=0.5, seed=6),
}
for _t in (1.0, 2.0, 4.0):
    for _p in (64, 128):
        _w = _imb(_t, _p)
        WORKLOADS[_w.name] = _w


def stream_seed(base: int, name: str) -> int:
    """Per-tensor seed: the base seed mixed with a CRC of the tensor name."""
    return (base * 1000003 + zlib.crc32(name.encode())) & 0x7FFFFFFFFFFF


def _gen(base: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(stream_seed(base, name))
    return g


def normal_bf16(shape, std: float, base: int, name: str, device="cpu", chunk_dim0: bool = False):
    """N(0, std) drawn in fp32 and rounded to bf16.  With chunk_dim0 the
    leading dimension is drawn slice by slice from the same stream (bounded
    fp32 temporaries for very large weights)."""
    g = _gen(base, name, device)
    if not chunk_dim0:
        return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(
            torch.bfloat16)
    out = torch.empty(shape, device=device, dtype=torch.bfloat16)
    for i in range(shape[0]):
        out[i] = (torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32) *
                  std).to(torch.bfloat16)
    return out


# Zipf exponents s of the imbalance workloads, for a hottest-expert load of
# 1x, 2x and 4x the mean.  Written by tests/golden/make_zipf_s.py, which
# bisects s on the CPU oracle's routing counts of the workload's seeded token
# rows until max/mean is within 2 % of the target (s = 0 for 1x; the routing
# of the unbiased draws already puts 1.117x the mean on the hottest expert).
# tests/test_oracle_pins.py re-derives the loads these values give.  The
# padding multiple does not enter the routing, so both paddings share s.
ZIPF_S = {
    "imbalance_x1_p128": 0.0,
    "imbalance_x1_p64": 0.0,
    "imbalance_x2_p128": 0.1328125,
    "imbalance_x2_p64": 0.1328125,
    "imbalance_x4_p128": 0.328125,
    "imbalance_x4_p64": 0.328125,
}
# hottest / mean expert load that the oracle's routing gives at these s
ZIPF_HOT_OVER_MEAN = {
    "imbalance_x1_p128": 1.1172,
    "imbalance_x1_p64": 1.1172,
    "imbalance_x2_p128": 1.9753,
    "imbalance_x2_p64": 1.9753,
    "imbalance_x4_p128": 4.0026,
    "imbalance_x4_p64": 4.0026,
}


def zipf_bias(E: int, s: float, base: int) -> torch.Tensor:
    """bias_e = -s * ln(rank_e), rank a seeded permutation of 1..E."""
    g = _gen(base, "zipf_rank", "cpu")
    rank = torch.randperm(E, generator=g) + 1
    return (-s * torch.log(rank.to(torch.float64))).to(torch.float32)


def make_inputs(shape: MoeShape, device="cpu", weights_device=None, zipf_s: Optional[float] = None
                ) -> dict:
    """All tensors of one workload.  Small tensors are drawn on ``device``;
    expert weights on ``weights_device`` (defaults to ``device``)."""
    wdev = weights_device or device
    b = shape.seed
    T, d, de, E, k = shape.T, shape.d, shape.d_e, shape.E, shape.k
    inp = {"x": normal_bf16((T, d), 1.0, b, "x", device)}
    big = E * d * de > (1 << 28)
    inp["W1"] = normal_bf16((E, d, de), 1.0 / math.sqrt(d), b, "W1", wdev, chunk_dim0=big)
    inp["W3"] = normal_bf16((E, d, de), 1.0 / math.sqrt(d), b, "W3", wdev, chunk_dim0=big)
    inp["W2"] = normal_bf16((E, de, d), 1.0 / math.sqrt(de), b, "W2", wdev, chunk_dim0=big)
    if shape.prerouted:
        sizes = shape.prerouted
        assert sum(sizes) == T * k and len(sizes) == E
        labels = torch.cat([torch.full((n,), e, dtype=torch.int32) for e, n in enumerate(sizes)])
        perm = torch.randperm(T * k, generator=_gen(b, "assign", "cpu"))
        inp["topk_idx"] = labels[perm].reshape(T, k).contiguous().to(device)
        u = torch.rand((T, k), generator=_gen(b, "gates", "cpu"), dtype=torch.float64)
        inp["topk_w"] = (0.05 + 0.95 * u).to(torch.float32).to(device)
        inp["Wg"] = None
        inp["bias"] = None
    else:
        inp["Wg"] = normal_bf16((d, E), 1.0 / math.sqrt(d), b, "Wg", device)
        if shape.bias_std > 0:
            g = _gen(b, "bias", "cpu")
            inp["bias"] = (torch.randn(E, generator=g, dtype=torch.float64) *
                           shape.bias_std).to(torch.float32).to(device)
        elif shape.zipf_target > 0:
            s = zipf_s if zipf_s is not None else ZIPF_S.get(shape.name, 0.0)
            inp["bias"] = zipf_bias(E, s, b).to(device)
        else:
            inp["bias"] = None
    if shape.d_shared:
        ds = shape.d_shared
        inp["Ws1"] = normal_bf16((d, ds), 1.0 / math.sqrt(d), b, "Ws1", wdev)
        inp["Ws3"] = normal_bf16((d, ds), 1.0 / math.sqrt(d), b, "Ws3", wdev)
        inp["Ws2"] = normal_bf16((ds, d), 1.0 / math.sqrt(ds), b, "Ws2", wdev)
    return inp


def redraw_rows(x: torch.Tensor, rows, base: int, attempt: int) -> None:
    """Replace the listed token rows of x by fresh N(0, 1) bf16 draws from a
    stream keyed by (base seed, attempt).  Used to move token rows away from
    near-ties of the routing decision."""
    rows = torch.as_tensor(rows, dtype=torch.long)
    if rows.numel() == 0:
        return
    g = _gen(base, f"redraw{attempt}", "cpu")
    fresh = torch.randn((rows.numel(), x.shape[1]), generator=g, dtype=torch.float32)
    x[rows.to(x.device)] = fresh.to(torch.bfloat16).to(x.device)
