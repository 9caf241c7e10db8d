"""The unpadded schedule ("Dropless and grouped GEMM", sec. 11) on the GPU:
moe_build_offsets_unpadded against the oracle's offsets with no padding
(P = 1: group offsets = the prefix sum of the counts), bit-exact; then
moe_permute, moe_grouped_gemm_swiglu_unpadded and moe_combine on that layout
against the oracle, every row of h and y and every token of the output
within the parity tolerances.  The shapes put expert boundaries inside
256-row windows (visited twice), on window edges, and leave experts empty.
"""
import numpy as np
import pytest
import torch

import oracle
import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build
from routing_permute_grouped_gb300 import synth
from routing_permute_grouped_gb300.synth import MoeShape
from tests.helpers import bits, enforce_margin, oracle_inputs

pytestmark = pytest.mark.gpu

REL_FRO = 5e-3
MAX_REL = 3e-2

SHAPES = {
    "routed_e8": MoeShape("unp_e8", T=777, d=1024, d_e=384, E=8, k=4, bias_std=0.5,
                          d_shared=256, seed=601),
    "routed_e64": MoeShape("unp_e64", T=1500, d=512, d_e=256, E=64, k=6, bias_std=1.0,
                           seed=602),
    "prerouted_ragged": MoeShape("unp_pre", T=300, d=512, d_e=256, E=5, k=8,
                                 prerouted=(900, 0, 321, 1000, 179), seed=603),
    # segment starts on window edges: 512, 768 are multiples of 256
    "prerouted_aligned": MoeShape("unp_aligned", T=256, d=384, d_e=128, E=3, k=4,
                                  prerouted=(512, 256, 256), seed=604),
    "one_expert": MoeShape("unp_e1", T=333, d=256, d_e=128, E=1, k=1, seed=605),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    moe_build.build()
    moe.load()


def _close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= MAX_REL * np.abs(ref).max(), f"{what}: max error {mx:.3e}"


@pytest.mark.parametrize("name", list(SHAPES))
def test_unpadded_schedule_matches_the_oracle(name):
    shape = SHAPES[name]
    inp = synth.make_inputs(shape)
    enforce_margin(inp, shape)
    oi = oracle_inputs(inp)
    T, k, E, d, de = shape.T, shape.k, shape.E, shape.d, shape.d_e
    A = T * k
    if shape.prerouted:
        idx, w = oi["topk_idx"], oi["topk_w"]
    else:
        lg = oracle.router_logits(oi["x"], oi["Wg"], oi.get("bias"))
        idx, w, _ = oracle.route(lg, k)
    ref = oracle.build_offsets(idx, w, E, 1)  # no padding: group offsets
    cfg = moe.config_of(shape)
    dev = "cuda"
    i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
    counts = torch.full((E,), -3, dtype=i32, device=dev)
    go = torch.full((E + 1,), -3, dtype=i32, device=dev)
    perm_row = torch.full((A,), -3, dtype=i32, device=dev)
    row_src = torch.full((A,), -3, dtype=i32, device=dev)
    row_gate = torch.full((A,), -3.0, dtype=f32, device=dev)
    ws = torch.zeros(moe.moe_offsets_workspace_size(cfg), dtype=torch.uint8, device=dev)
    idx_d = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev)
    w_d = torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev)
    moe.moe_build_offsets_unpadded(cfg, idx_d, w_d, counts, go, perm_row, row_src, row_gate, ws)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(go.cpu().numpy(), ref["padded_offsets"])
    assert np.array_equal(perm_row.cpu().numpy(), ref["perm_row"])
    assert np.array_equal(row_src.cpu().numpy(), ref["row_src"][:A])
    assert np.array_equal(row_gate.cpu().numpy(), ref["row_gate"][:A].astype(np.float32))

    W13 = torch.empty((E, 2 * de, d), dtype=bf, device=dev)
    W2t = torch.empty((E, d, de), dtype=bf, device=dev)
    moe.moe_pack_experts(inp["W1"].to(dev), inp["W3"].to(dev), inp["W2"].to(dev), W13, W2t)
    x = inp["x"].to(dev)
    x_perm = torch.empty((A, d), dtype=bf, device=dev)
    h = torch.full((A, de), float("nan"), dtype=bf, device=dev)
    y = torch.full((A, d), float("nan"), dtype=bf, device=dev)
    status = torch.zeros((1,), dtype=i32, device=dev)
    moe.moe_permute(cfg, x, perm_row, x_perm)
    for _ in range(2):  # twice: the second call runs on the first call's outputs
        moe.moe_grouped_gemm_swiglu_unpadded(cfg, x_perm, W13, W2t, go, row_gate, h, y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # every row of the layout belongs to exactly one expert
    seg = np.searchsorted(ref["padded_offsets"], np.arange(A), side="right") - 1
    xp = oracle.permute(oi["x"], ref["row_src"][:A], k)
    eh, ey = oracle.expert_rows(xp, seg.astype(np.int32), ref["row_gate"][:A], oi["W1"], oi["W3"],
                                oi["W2"])
    _close(h.double().cpu().numpy(), eh, "h")
    _close(y.double().cpu().numpy(), ey, "y")

    ys = None
    ys_ref = None
    if shape.d_shared:
        Ws13 = torch.empty((1, 2 * shape.d_shared, d), dtype=bf, device=dev)
        Ws2t = torch.empty((1, d, shape.d_shared), dtype=bf, device=dev)
        moe.moe_pack_experts(inp["Ws1"][None].to(dev), inp["Ws3"][None].to(dev),
                             inp["Ws2"][None].to(dev), Ws13, Ws2t)
        hs = torch.empty((T, shape.d_shared), dtype=bf, device=dev)
        ys = torch.empty((T, d), dtype=bf, device=dev)
        moe.moe_shared_expert(cfg, x, Ws13, Ws2t, hs, ys, status)
        _, ys_ref = oracle.shared_expert(oi["x"], oi["Ws1"], oi["Ws3"], oi["Ws2"])
    out = torch.empty((T, d), dtype=bf, device=dev)
    moe.moe_combine(cfg, y, perm_row, ys, out)
    torch.cuda.synchronize()
    ref_out = oracle.direct_layer(np.arange(T, dtype=np.int32), oi["x"], oi["W1"], oi["W3"],
                                  oi["W2"], np.ascontiguousarray(idx, np.int32),
                                  np.ascontiguousarray(w, np.float64), ys_ref)
    _close(out.double().cpu().numpy(), ref_out, "out")
