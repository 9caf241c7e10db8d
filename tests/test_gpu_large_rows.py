"""GPU parity for a layer whose padded buffers pass 2^31 elements.

With T = 40960 tokens, k = 8 and d = 7168 the padded row buffers x_perm and y
(forward) and dz, x_perm and dx_perm (backward) are [R, d] with R * d above
2^31 elements and 4 GiB, so every row and element offset in the permute, the
GEMMs' tile coordinates and epilogues, the combine, the SwiGLU backward and
the weight-gradient GEMMs must be taken in 64 bits.  The rows and tokens
checked against the oracle are chosen above that line on purpose (the last
expert's segment lies there), next to a few random ones.  Routing and offsets
are compared in full and bit-exactly, as at the pages' sizes.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build
from routing_permute_grouped_gb300 import synth
from routing_permute_grouped_gb300.synth import MoeShape
from tests.helpers import bits, enforce_margin

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SHAPE = MoeShape("rows_beyond_2e31", T=40960, d=7168, d_e=256, E=16, k=8, bias_std=0.5,
                 d_shared=256, seed=601)
# first padded row whose element offset row * d no longer fits in 31 bits
FIRST_HIGH_ROW = -(-(1 << 31) // SHAPE.d)


def _close(got, ref, what, rel_fro, max_rel):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    assert rel <= rel_fro, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= max_rel * np.abs(ref).max(), f"{what}: max error {mx:.3e}"


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.fail("GPU parity tests need a CUDA device")
    moe_build.build()
    moe.load()
    s = SHAPE
    assert s.rows_capacity * s.d > (1 << 31)
    dev = torch.device("cuda")
    inp = synth.make_inputs(s, device="cpu")
    enforce_margin(inp, s)
    g = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    layer = moe.MoeLayer(moe.config_of(s), g(inp["W1"]), g(inp["W3"]), g(inp["W2"]),
                         Wg=g(inp["Wg"]), bias=g(inp["bias"]), Ws1=g(inp["Ws1"]),
                         Ws3=g(inp["Ws3"]), Ws2=g(inp["Ws2"]))
    x = g(inp["x"])
    out = layer(x)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    x_bits = bits(inp["x"])
    lg = oracle.router_logits(x_bits, bits(inp["Wg"]), inp["bias"].numpy())
    idx, w, margin = oracle.route(lg, s.k)
    assert margin.min() >= 1e-3
    off = oracle.build_offsets(idx, w, s.E, s.pad)
    host = {key: bits(inp[key]) for key in ("W1", "W3", "W2", "Ws1", "Ws3", "Ws2", "Wg")}
    return dict(inp=inp, layer=layer, x=x, out=out, x_bits=x_bits, idx=idx, w=w, off=off,
                host=host)


def _high_tokens(row_src, k, n, rng):
    """n tokens that have an assignment at or above FIRST_HIGH_ROW (the last
    rows of the buffer first) and n random tokens."""
    valid = np.flatnonzero(row_src >= 0)
    high = valid[valid >= FIRST_HIGH_ROW]
    assert high.size > 0, "the shape must place rows above the 31-bit element line"
    tok_high = np.unique(row_src[high[-4 * n:]] // k)[-n:]
    tok_rand = rng.choice(SHAPE.T, size=n, replace=False)
    return np.unique(np.concatenate([tok_high, tok_rand])).astype(np.int32)


def test_forward_beyond_31_bit_offsets(run):
    s, layer, off = SHAPE, run["layer"], run["off"]
    T, k, E, d, de = s.T, s.k, s.E, s.d, s.d_e
    A, R, NB = s.A, s.rows_capacity, s.blocks_capacity
    dev = torch.device("cuda")
    i32 = torch.int32

    # routing and offsets: full, bit-exact
    assert np.array_equal(layer.buffer("topk_idx", i32, (T, k)).cpu().numpy(), run["idx"])
    assert np.array_equal(layer.buffer("counts", i32, (E,)).cpu().numpy(), off["counts"])
    assert np.array_equal(layer.buffer("padded_offsets", i32, (E + 1,)).cpu().numpy(),
                          off["padded_offsets"])
    nb = int(layer.buffer("num_blocks", i32, (1,)).item())
    assert nb == off["num_blocks"]
    assert np.array_equal(layer.buffer("block_metadata", i32, (NB, 3)).cpu().numpy()[:nb],
                          off["block_metadata"])
    assert np.array_equal(layer.buffer("perm_row", i32, (A,)).cpu().numpy(), off["perm_row"])
    row_src = layer.buffer("row_src", i32, (R,)).cpu().numpy()
    assert np.array_equal(row_src, off["row_src"])
    assert off["padded_offsets"][-1] > FIRST_HIGH_ROW

    # permute: every valid row is its token's row
    xp = layer.buffer("x_perm", torch.bfloat16, (R, d))
    valid = torch.from_numpy(row_src >= 0).to(dev)
    src_tok = torch.from_numpy(np.where(row_src >= 0, row_src // k, 0)).to(dev)
    assert torch.equal(xp[valid], run["x"][src_tok[valid]])

    # h and y of the last valid rows and of random ones
    rng = np.random.default_rng(17)
    vrows = np.flatnonzero(row_src >= 0)
    samp = np.unique(np.concatenate([vrows[-12:], rng.choice(vrows, size=12, replace=False)]))
    assert (samp >= FIRST_HIGH_ROW).sum() >= 12
    ref_xp = oracle.permute(run["x_bits"], np.where(np.isin(np.arange(R), samp), row_src, -1), k)
    seg = (np.searchsorted(off["padded_offsets"], samp, side="right") - 1).astype(np.int32)
    hw = run["host"]
    eh, ey = oracle.expert_rows(ref_xp[samp], seg, off["row_gate"][samp], hw["W1"], hw["W3"],
                                hw["W2"])
    st = torch.as_tensor(samp, device=dev)
    h = layer.buffer("h", torch.bfloat16, (R, de))
    y = layer.buffer("y", torch.bfloat16, (R, d))
    _close(h[st].double().cpu().numpy(), eh, "h (sampled rows)", 5e-3, 3e-2)
    _close(y[st].double().cpu().numpy(), ey, "y (sampled rows)", 5e-3, 3e-2)

    # the output of tokens routed above the line, by direct evaluation
    toks = _high_tokens(row_src, k, 6, rng)
    _, ys = oracle.shared_expert(run["x_bits"][toks], hw["Ws1"], hw["Ws3"], hw["Ws2"])
    ref_out = oracle.direct_layer(np.arange(toks.size, dtype=np.int32), run["x_bits"][toks],
                                  hw["W1"], hw["W3"], hw["W2"], run["idx"][toks],
                                  run["w"][toks], ys)
    got = run["out"][torch.as_tensor(toks, device=dev, dtype=torch.long)]
    _close(got.double().cpu().numpy(), ref_out, "out (sampled tokens)", 5e-3, 3e-2)
    assert torch.isfinite(run["out"].float()).all()


def test_backward_beyond_31_bit_offsets(run):
    s, layer, off = SHAPE, run["layer"], run["off"]
    T, k, E, d, de = s.T, s.k, s.E, s.d, s.d_e
    dev = torch.device("cuda")
    gen = torch.Generator().manual_seed(s.seed + 1000)
    dout = torch.randn((T, d), generator=gen).to(torch.bfloat16)
    grads = layer.backward(run["x"], dout.to(dev))
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    for key, t in grads.items():
        assert torch.isfinite(t.float()).all(), key
    hw, idx, w = run["host"], run["idx"], run["w"]
    dout64 = dout.double().numpy()

    # dx and dgates of tokens routed above the line: the oracle's backward on
    # those tokens alone
    rng = np.random.default_rng(19)
    toks = _high_tokens(off["row_src"], k, 4, rng)
    sub = dict(x=run["x_bits"][toks], W1=hw["W1"], W3=hw["W3"], W2=hw["W2"], Wg=hw["Wg"],
               bias=run["inp"]["bias"].numpy(), Ws1=hw["Ws1"], Ws3=hw["Ws3"], Ws2=hw["Ws2"])
    sub_shape = dataclasses.replace(s, T=toks.size)
    fwd = oracle.layer_forward(sub, sub_shape)
    assert np.array_equal(fwd["topk_idx"], idx[toks])
    ref = oracle.layer_backward(sub, sub_shape, fwd, dout64[toks])
    tt = torch.as_tensor(toks, device=dev, dtype=torch.long)
    _close(grads["dx"][tt].double().cpu().numpy(), ref["dx"], "dx (sampled tokens)", 1e-2, 5e-2)
    _close(grads["dgates"][tt].double().cpu().numpy(), ref["dgates"], "dgates (sampled)",
           1e-2, 5e-2)

    # columns of the last expert's weight gradients (its segment lies above
    # the line) and of the shared expert's, over all their rows
    e = E - 1
    assert off["padded_offsets"][e + 1] > FIRST_HIGH_ROW
    J = np.array([0, de // 2 + 1, de - 1], np.int32)
    t, j = np.nonzero(idx == e)
    dW1c, dW3c, dW2r = oracle.weight_grad_columns(run["x_bits"][t], dout64[t], w[t, j],
                                                  hw["W1"][e], hw["W3"][e], hw["W2"][e], J)
    Jt = torch.as_tensor(J, device=dev, dtype=torch.long)
    _close(grads["dW1"][e][:, Jt].double().cpu().numpy(), dW1c, "dW1 columns", 1e-2, 5e-2)
    _close(grads["dW3"][e][:, Jt].double().cpu().numpy(), dW3c, "dW3 columns", 1e-2, 5e-2)
    _close(grads["dW2"][e][Jt, :].double().cpu().numpy(), dW2r, "dW2 rows", 1e-2, 5e-2)
    Js = np.array([1, s.d_shared - 1], np.int32)
    dW1c, dW3c, dW2r = oracle.weight_grad_columns(run["x_bits"], dout64, np.ones(T), hw["Ws1"],
                                                  hw["Ws3"], hw["Ws2"], Js)
    Jt = torch.as_tensor(Js, device=dev, dtype=torch.long)
    _close(grads["dWs1"][:, Jt].double().cpu().numpy(), dW1c, "dWs1 columns", 1e-2, 5e-2)
    _close(grads["dWs3"][:, Jt].double().cpu().numpy(), dW3c, "dWs3 columns", 1e-2, 5e-2)
    _close(grads["dWs2"][Jt, :].double().cpu().numpy(), dW2r, "dWs2 rows", 1e-2, 5e-2)
