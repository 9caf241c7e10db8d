"""The expert-parallel layer forward (ep.GpuEp) on the CUDA library, through
NCCL, with world size 1: the one GPU of a box holds every expert, so the
counts all-to-all stays within the rank, the receiver's layout is built on
the device from the exchanged counts, and the rank's own layout serves as the
expert-major one.  The output must be bit-identical to MoeLayer's where both
run the CTA-pair kernel, and within the parity bound of the oracle
everywhere.  The device entry points of the exchange with several senders
(the receiver's layout from counts, the piece copies) are compared with the
oracle's layout and with plain indexing here; the exchange between ranks is
tested on CPU process groups in tests/test_ep_gloo.py.
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


@pytest.mark.parametrize("W, El, P", [(1, 8, 128), (2, 4, 64), (4, 32, 128), (8, 256, 64),
                                      (3, 1, 128)])
def test_blocks_from_counts_match_the_oracle(W, El, P):
    """moe_build_blocks_from_counts: padded offsets, block table and landing
    rows bit-exact against the oracle's layout of the same counts (empty
    experts and senders included), twice on stale outputs."""
    rng = np.random.default_rng(W * 1000 + El)
    counts = rng.integers(0, 3 * P, (W, El)).astype(np.int32)
    counts[rng.random((W, El)) < 0.2] = 0
    ref = oracle.blocks_from_counts(counts, P)
    cap = int(counts.sum()) // P + El
    dev = "cuda"
    po = torch.full((El + 1,), -9, dtype=torch.int32, device=dev)
    meta = torch.full((cap, 3), -9, dtype=torch.int32, device=dev)
    nb = torch.full((1,), -9, dtype=torch.int32, device=dev)
    pr = torch.full((W, El), -9, dtype=torch.int32, device=dev)
    st = torch.zeros((1,), dtype=torch.int32, device=dev)
    for _ in range(2):
        moe.moe_build_blocks_from_counts(torch.from_numpy(counts).to(dev), P, po, meta, nb, pr, st)
        torch.cuda.synchronize()
        n = int(nb.item())
        assert n == ref["num_blocks"] and int(st.item()) == 0
        assert np.array_equal(po.cpu().numpy(), ref["padded_offsets"])
        assert np.array_equal(meta.cpu().numpy()[:n], ref["block_metadata"])
        assert np.array_equal(pr.cpu().numpy(), ref["piece_row"])


def test_blocks_from_counts_flags_overflow():
    """A table that does not fit its capacity is cut at nb_cap and flagged."""
    counts = torch.tensor([[300, 5]], dtype=torch.int32, device="cuda")
    meta = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
    po = torch.zeros((3,), dtype=torch.int32, device="cuda")
    nb = torch.zeros((1,), dtype=torch.int32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    moe.moe_build_blocks_from_counts(counts, 128, po, meta, nb, None, st)
    torch.cuda.synchronize()
    assert int(nb.item()) == 2 and int(st.item()) & 0x4
    assert po.cpu().tolist() == [0, 384, 512]


def test_copy_pieces():
    """moe_copy_pieces: each piece's rows (and gates) land at its destination
    bit for bit; rows outside the pieces keep their contents."""
    g = torch.Generator().manual_seed(11)
    src = torch.randn((500, 264), generator=g).to(torch.bfloat16).cuda()
    sg = torch.rand(500, generator=g).cuda()
    pieces = [(0, 40, 17), (100, 0, 33), (300, 90, 0), (37, 200, 64), (450, 300, 50)]
    s_row, d_row, rows = (torch.tensor(v, dtype=torch.int32, device="cuda") for v in zip(*pieces))
    dst = torch.full((400, 264), 3.0, dtype=torch.bfloat16, device="cuda")
    dg = torch.full((400,), 3.0, device="cuda")
    moe.moe_copy_pieces(src, dst, s_row, d_row, rows, 64, sg, dg)
    torch.cuda.synchronize()
    expect = torch.full((400, 264), 3.0, dtype=torch.bfloat16)
    eg = torch.full((400,), 3.0)
    for a, b, n in pieces:
        expect[b:b + n] = src.cpu()[a:a + n]
        eg[b:b + n] = sg.cpu()[a:a + n]
    assert torch.equal(dst.cpu(), expect)
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
