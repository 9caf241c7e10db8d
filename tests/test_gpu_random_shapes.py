"""Seeded random layer shapes, forward and backward, against the oracle.

Twelve small layers drawn from a fixed seed: widths d, d_e, d_shared
(multiples of 128, the shared expert present or not), E from 1 to 96, k up
to min(E, 8), padding 64 or 128, group-limited routing where E allows it, a
logit bias or not, and T from 1 to 1500 (so that both the small-M and the
CTA-pair paths run).  Each layer's forward output and backward gradients are
compared with the oracle under the tolerances of the dedicated parity files
(forward 5e-3 / 3e-2, backward 1e-2 / 5e-2, relative Frobenius / max over
max|ref|); routing indices are compared bit-exactly after the margin filter.
The same layers also run with e4m3 expert weights (forward) and with the
gate/up values kept from the forward (backward).
"""
import numpy as np
import pytest
import torch

import oracle
import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build
from routing_permute_grouped_gb300 import synth
from routing_permute_grouped_gb300.synth import MoeShape
from tests.helpers import enforce_margin, oracle_inputs

pytestmark = pytest.mark.gpu


def _shapes(n=12, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([1, 2, 3, 5, 8, 13, 32, 64, 96]))
        k = int(rng.integers(1, min(E, 8) + 1))
        groups = 0
        topk_groups = 0
        if E % 4 == 0 and E >= 8 and rng.random() < 0.5:
            groups = 4
            topk_groups = int(rng.integers(1, 5))
            while topk_groups * (E // groups) < k:
                topk_groups += 1
        out.append(MoeShape(
            f"r{i}", T=int(rng.choice([1, 60, 400, 900, 1500], p=[0.15, 0.15, 0.25, 0.25, 0.2])),
            d=128 * int(rng.integers(1, 5)),
            d_e=128 * int(rng.integers(1, 4)), E=E, k=k, n_groups=groups,
            topk_groups=topk_groups, pad=int(rng.choice([64, 128])),
            d_shared=128 * int(rng.integers(0, 3)), bias_std=float(rng.choice([0.0, 0.4])),
            seed=3000 + i))
    return out


SHAPES = {s.name: s for s in _shapes()}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    moe_build.build()
    moe.load()


def _close(got, ref, what, rel_fro, max_rel):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    nref = np.linalg.norm(ref)
    if nref == 0:
        assert np.abs(got).max() == 0, what
        return
    rel = np.linalg.norm(got - ref) / nref
    mx = np.abs(got - ref).max()
    assert rel <= rel_fro, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= max_rel * np.abs(ref).max(), f"{what}: max error {mx:.3e}"


@pytest.mark.parametrize("name", list(SHAPES))
def test_random_layer_forward_and_backward(name):
    shape = SHAPES[name]
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    oi = oracle_inputs(inp)
    ref = oracle.layer_forward(oi, shape)
    g = torch.Generator().manual_seed(shape.seed + 1000)
    dout = torch.randn((shape.T, shape.d), generator=g).to(torch.bfloat16)
    bref = oracle.layer_backward(oi, shape, ref, dout.double().numpy())
    cuda = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    layer = moe.MoeLayer(moe.config_of(shape), cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]),
                         Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")),
                         Ws1=cuda(inp.get("Ws1")), Ws3=cuda(inp.get("Ws3")),
                         Ws2=cuda(inp.get("Ws2")))
    x = cuda(inp["x"])
    out = layer(x)
    grads = layer.backward(x, cuda(dout))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    T, k = shape.T, shape.k
    idx = layer.buffer("topk_idx", torch.int32, (T, k)).cpu().numpy()
    assert np.array_equal(idx, ref["topk_idx"])
    _close(out.double().cpu().numpy(), ref["out"], "out", 5e-3, 3e-2)
    for key in ("dx", "dW1", "dW3", "dW2", "dWs1", "dWs3", "dWs2"):
        if key in bref:
            _close(grads[key].double().cpu().numpy(), bref[key], key, 1e-2, 5e-2)


@pytest.mark.parametrize("name", list(SHAPES))
def test_random_layer_e4m3_forward(name):
    """The same layers with e4m3 expert weights (the small-M kernel's 8-bit
    MMAs below T*k = 32*E, the widened codes on the CTA-pair kernel above),
    against the oracle's evaluation of the quantized weights."""
    shape = SHAPES[name]
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    oi = oracle_inputs(inp)
    oi.update(oracle.quantize_experts(oi))
    if shape.d_shared:
        oi.update(oracle.quantize_shared(oi))
    ref = oracle.layer_forward(oi, shape)
    cuda = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    layer = moe.MoeLayer(moe.config_of(shape), cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]),
                         Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")),
                         Ws1=cuda(inp.get("Ws1")), Ws3=cuda(inp.get("Ws3")),
                         Ws2=cuda(inp.get("Ws2")), fp8=True)
    out = layer(cuda(inp["x"]))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    idx = layer.buffer("topk_idx", torch.int32, (shape.T, shape.k)).cpu().numpy()
    assert np.array_equal(idx, ref["topk_idx"])
    _close(out.double().cpu().numpy(), ref["out"], "out (e4m3)", 5e-3, 3e-2)


@pytest.mark.parametrize("name", list(SHAPES))
def test_random_layer_backward_with_saved_gate_up(name):
    """The same layers with the gate/up values kept from the forward
    (keep_gate_up): the gradients equal the recomputing layer's bit for bit
    where the forward ran the CTA-pair kernel, and stay within the backward
    tolerances of the oracle where it ran the small-M kernel."""
    shape = SHAPES[name]
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    cuda = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    g = torch.Generator().manual_seed(shape.seed + 1000)
    dout = torch.randn((shape.T, shape.d), generator=g).to(torch.bfloat16)
    kw = dict(Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")), Ws1=cuda(inp.get("Ws1")),
              Ws3=cuda(inp.get("Ws3")), Ws2=cuda(inp.get("Ws2")))
    cfg = moe.config_of(shape)
    W = [cuda(inp[n]) for n in ("W1", "W3", "W2")]
    plain = moe.MoeLayer(cfg, *W, **kw)
    keep = moe.MoeLayer(cfg, *W, keep_gate_up=True, **kw)
    x, dz = cuda(inp["x"]), cuda(dout)
    out_p, out_k = plain(x), keep(x)
    g_p, g_k = plain.backward(x, dz), keep.backward(x, dz)
    torch.cuda.synchronize()
    assert keep.device_status() == 0
    assert torch.equal(out_p, out_k)
    if shape.T * shape.k > 32 * shape.E:
        for key in g_p:
            assert torch.equal(g_p[key], g_k[key]), key
        return
    oi = oracle_inputs(inp)
    ref = oracle.layer_forward(oi, shape)
    bref = oracle.layer_backward(oi, shape, ref, dout.double().numpy())
    for key in ("dx", "dW1", "dW3", "dW2", "dWs1", "dWs3", "dWs2"):
        if key in bref:
            _close(g_k[key].double().cpu().numpy(), bref[key], key, 1e-2, 5e-2)
