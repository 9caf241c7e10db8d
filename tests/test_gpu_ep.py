"""The expert-parallel layer forward (ep.GpuEp) on the CUDA library, through
NCCL, with world size 1: the one GPU of a box holds every expert, so the
all-to-alls move rows within the rank, and the dispatch plan, the receiver's
block table and the stage calls run exactly as they do across ranks.  The
output must be bit-identical to MoeLayer's where both run the CTA-pair
kernel, and within the parity bound of the oracle everywhere.  (The exchange
between ranks is tested on CPU process groups in tests/test_ep_gloo.py.)
"""
import socket

import numpy as np
import pytest
import torch

import oracle
import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build
from routing_permute_grouped_gb300 import ep, synth
from routing_permute_grouped_gb300.synth import MoeShape
from tests.helpers import enforce_margin, oracle_inputs

pytestmark = pytest.mark.gpu

SHAPES = {
    "pair_shared": MoeShape("ep_pair", T=777, d=1024, d_e=384, E=8, k=4, bias_std=0.5,
                            d_shared=256, seed=501),
    "small_m_groups": MoeShape("ep_small", T=37, d=512, d_e=256, E=64, k=8, n_groups=8,
                               topk_groups=4, d_shared=128, seed=502),
    "prerouted": MoeShape("ep_pre", T=300, d=512, d_e=256, E=4, k=8,
                          prerouted=(900, 321, 1000, 179), seed=503),
}


@pytest.fixture(scope="module", autouse=True)
def _group():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    moe_build.build()
    moe.load()
    import torch.distributed as dist

    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    yield
    dist.destroy_process_group()


def _close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    assert rel <= 5e-3, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= 3e-2 * np.abs(ref).max(), f"{what}: max error {mx:.3e}"


@pytest.mark.parametrize("name", list(SHAPES))
def test_ep_world1_matches_the_layer(name):
    shape = SHAPES[name]
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    ref = oracle.layer_forward(oracle_inputs(inp), shape)
    cuda = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    cfg = moe.config_of(shape)
    kw = dict(Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")), Ws1=cuda(inp.get("Ws1")),
              Ws3=cuda(inp.get("Ws3")), Ws2=cuda(inp.get("Ws2")))
    W1, W3, W2 = cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"])
    layer = moe.MoeLayer(cfg, W1, W3, W2, **kw)
    eplayer = ep.GpuEp(cfg, W1, W3, W2, **kw)
    x = cuda(inp["x"])
    pre = dict(topk_idx=cuda(inp["topk_idx"]), topk_w=cuda(inp["topk_w"])) if shape.prerouted else {}
    out_l = layer(x, **pre)
    out_e = eplayer.forward(x, **pre)
    out_e2 = eplayer.forward(x, **pre)
    torch.cuda.synchronize()
    assert eplayer.device_status() == 0 and layer.device_status() == 0
    assert torch.equal(out_e, out_e2)
    _close(out_e.double().cpu().numpy(), ref["out"], "out (expert parallel)")
    if shape.T * shape.k > 32 * shape.E:  # both on the CTA-pair kernel
        assert torch.equal(out_e, out_l)


def test_gather_rows():
    """moe_gather_rows: dst[i] = src[idx[i]] bit for bit, gates alongside;
    a negative index leaves the row and its gate as they were."""
    g = torch.Generator().manual_seed(9)
    src = torch.randn((300, 264), generator=g).to(torch.bfloat16).cuda()
    sg = torch.rand(300, generator=g).cuda()
    idx = torch.randint(-1, 300, (517,), generator=g, dtype=torch.int32)
    dst = torch.full((517, 264), 7.0, dtype=torch.bfloat16, device="cuda")
    dg = torch.full((517,), 7.0, device="cuda")
    moe.moe_gather_rows(src, idx.cuda(), dst, sg, dg)
    torch.cuda.synchronize()
    ii = idx.long()
    ok = ii >= 0
    expect = torch.full((517, 264), 7.0, dtype=torch.bfloat16)
    expect[ok] = src.cpu()[ii[ok]]
    assert torch.equal(dst.cpu(), expect)
    eg = torch.full((517,), 7.0)
    eg[ok] = sg.cpu()[ii[ok]]
    assert torch.equal(dg.cpu(), eg)


def _random_shapes():
    from tests.test_gpu_random_shapes import SHAPES as RANDOM

    return {k: v for k, v in RANDOM.items() if k in ("r0", "r2", "r3", "r6", "r7", "r11")}


@pytest.mark.parametrize("name", list(_random_shapes()))
def test_ep_world1_random_layers(name):
    """Seeded random layers (E from 2 to 64, shared expert or not, both GEMM
    paths) through the piece-by-piece exchange at world size 1: bit-identical
    to MoeLayer where both run the CTA-pair kernel, within the parity bound
    of the oracle everywhere."""
    shape = _random_shapes()[name]
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    ref = oracle.layer_forward(oracle_inputs(inp), shape)
    cuda = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    cfg = moe.config_of(shape)
    kw = dict(Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")), Ws1=cuda(inp.get("Ws1")),
              Ws3=cuda(inp.get("Ws3")), Ws2=cuda(inp.get("Ws2")))
    W1, W3, W2 = cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"])
    x = cuda(inp["x"])
    out_l = moe.MoeLayer(cfg, W1, W3, W2, **kw)(x)
    eplayer = ep.GpuEp(cfg, W1, W3, W2, **kw)
    out_e = eplayer.forward(x)
    torch.cuda.synchronize()
    assert eplayer.device_status() == 0
    _close(out_e.double().cpu().numpy(), ref["out"], "out (expert parallel)")
    if shape.T * shape.k > 32 * shape.E:
        assert torch.equal(out_e, out_l)
