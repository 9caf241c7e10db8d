"""GPU parity at the full workload sizes, in the launch configuration that
bench.py times (the same entry points, persistent grids and workspace).

At these sizes the oracle runs the full routing and the full offsets (cheap)
and compares them bit-exactly.  It then computes sampled rows one by one:
  - permuted rows, compared bit-exactly;
  - h and y of sampled padded rows;
  - the output of sampled tokens, by direct per-token evaluation.
On top of that come properties that hold at any size: every valid permuted
row is a copy of its token row, and nothing non-finite appears.  The expert
weights are drawn on the GPU (the decode workload holds 22.5 GB of them), and
only the experts that the sampled rows use are copied to the host for the
oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build
from routing_permute_grouped_gb300 import synth
from tests.helpers import bits, enforce_margin

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

REL_FRO = 5e-3
MAX_REL = 3e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU parity tests need a CUDA device")
    moe_build.build()
    moe.load()


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= MAX_REL * np.abs(ref).max(), f"{what}: max error {mx:.3e}"


def _expert_subset(W, experts):
    """Host copy of the listed experts' weights (uint16 bits)."""
    return bits(W[torch.as_tensor(experts, device=W.device, dtype=torch.long)].cpu())


@pytest.mark.parametrize("name", ["default", "prerouted", "decode", "imbalance_x1_p64",
                                  "imbalance_x1_p128", "imbalance_x2_p64", "imbalance_x2_p128",
                                  "imbalance_x4_p64", "imbalance_x4_p128"])
def test_full_size_layer(name):
    shape = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    inp = synth.make_inputs(shape, device="cpu", weights_device=dev)
    enforce_margin(inp, shape)
    cfg = moe.config_of(shape)
    g = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    layer = moe.MoeLayer(cfg, inp["W1"], inp["W3"], inp["W2"], Wg=g(inp.get("Wg")),
                         bias=g(inp.get("bias")), Ws1=inp.get("Ws1"), Ws3=inp.get("Ws3"),
                         Ws2=inp.get("Ws2"))
    x = g(inp["x"])
    if shape.prerouted:
        out = layer(x, topk_idx=g(inp["topk_idx"]), topk_w=g(inp["topk_w"]))
    else:
        out = layer(x)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    T, k, E, d, de = shape.T, shape.k, shape.E, shape.d, shape.d_e
    A, R, NB = shape.A, shape.rows_capacity, shape.blocks_capacity
    x_bits = bits(inp["x"])

    # routing: full, bit-exact indices
    if shape.prerouted:
        idx = inp["topk_idx"].numpy()
        w = inp["topk_w"].double().numpy()
    else:
        bias = None if inp.get("bias") is None else inp["bias"].numpy()
        lg = oracle.router_logits(x_bits, bits(inp["Wg"]), bias)
        idx, w, margin = oracle.route(lg, k, shape.n_groups, shape.topk_groups)
        assert margin.min() >= 1e-3
        gidx = layer.buffer("topk_idx", torch.int32, (T, k)).cpu().numpy()
        assert np.array_equal(gidx, idx)
        gw = layer.buffer("topk_w", torch.float32, (T, k)).cpu().double().numpy()
        np.testing.assert_allclose(gw, w, rtol=0, atol=2e-5)

    # offsets: full, bit-exact
    off = oracle.build_offsets(idx, w, E, shape.pad)
    i32 = torch.int32
    assert np.array_equal(layer.buffer("counts", i32, (E,)).cpu().numpy(), off["counts"])
    assert np.array_equal(layer.buffer("padded_offsets", i32, (E + 1,)).cpu().numpy(),
                          off["padded_offsets"])
    nb = int(layer.buffer("num_blocks", i32, (1,)).item())
    assert nb == off["num_blocks"]
    assert np.array_equal(layer.buffer("block_metadata", i32, (NB, 3)).cpu().numpy()[:nb],
                          off["block_metadata"])
    perm_row = layer.buffer("perm_row", i32, (A,)).cpu().numpy()
    assert np.array_equal(perm_row, off["perm_row"])
    row_src = layer.buffer("row_src", i32, (R,)).cpu().numpy()
    assert np.array_equal(row_src, off["row_src"])
    if name == "prerouted":
        assert off["padded_offsets"].tolist() == [0, 21760, 36864, 54912, 65792]

    # permute: property over all valid rows, plus sampled rows from the oracle
    xp = layer.buffer("x_perm", torch.bfloat16, (R, d))
    valid = torch.from_numpy(row_src >= 0).to(dev)
    src_tok = torch.from_numpy(np.where(row_src >= 0, row_src // k, 0)).to(dev)
    assert torch.equal(xp[valid], x[src_tok[valid]])
    rng = np.random.default_rng(7)
    vrows = np.flatnonzero(row_src >= 0)
    n_rows, n_tok = (16, 4) if E > 64 else (24, 8)  # bounds the expert weights copied to the host
    samp = np.sort(rng.choice(vrows, size=min(n_rows, vrows.size), replace=False))
    ref_xp = oracle.permute(x_bits, np.where(np.isin(np.arange(R), samp), row_src, -1), k)
    assert np.array_equal(bits(xp[torch.as_tensor(samp, device=dev)].cpu()), ref_xp[samp])

    # h, y of sampled padded rows
    seg = np.searchsorted(off["padded_offsets"], samp, side="right") - 1
    used = np.unique(seg)
    remap = {e: i for i, e in enumerate(used)}
    W1s = _expert_subset(inp["W1"], used)
    W3s = _expert_subset(inp["W3"], used)
    W2s = _expert_subset(inp["W2"], used)
    eh, ey = oracle.expert_rows(ref_xp[samp], np.array([remap[e] for e in seg], np.int32),
                                off["row_gate"][samp], W1s, W3s, W2s)
    h = layer.buffer("h", torch.bfloat16, (R, de))
    y = layer.buffer("y", torch.bfloat16, (R, d))
    st = torch.as_tensor(samp, device=dev)
    assert_close(h[st].double().cpu().numpy(), eh, "h (sampled rows)")
    assert_close(y[st].double().cpu().numpy(), ey, "y (sampled rows)")

    # output of sampled tokens by direct per-token evaluation
    toks = np.sort(rng.choice(T, size=min(n_tok, T), replace=False)).astype(np.int32)
    used = np.unique(idx[toks])
    remap = {e: i for i, e in enumerate(used)}
    idx_s = np.vectorize(remap.get)(idx[toks]).astype(np.int32)
    ys = None
    if shape.d_shared:
        _, ys = oracle.shared_expert(x_bits[toks], bits(inp["Ws1"].cpu()),
                                     bits(inp["Ws3"].cpu()), bits(inp["Ws2"].cpu()))
    ref_out = oracle.direct_layer(np.arange(toks.size, dtype=np.int32), x_bits[toks],
                                  _expert_subset(inp["W1"], used), _expert_subset(inp["W3"], used),
                                  _expert_subset(inp["W2"], used), idx_s, w[toks], ys)
    got = out[torch.as_tensor(toks, device=dev, dtype=torch.long)].double().cpu().numpy()
    assert_close(got, ref_out, "out (sampled tokens)")
    assert torch.isfinite(out.float()).all()


def _packed_rows(de):
    """Packed W13 row r -> (0 gate / 1 up, output column)."""
    r = np.arange(2 * de)
    return (r % 256 >= 128).astype(np.int64), (r // 256) * 128 + r % 128


@pytest.mark.parametrize("name", ["decode", "default"])
def test_full_size_layer_fp8(name):
    """The e4m3-weight layer at the full decode size (8-bit MMAs on the small-M
    kernel) and the full default size (the codes widened to bf16 for the
    CTA-pair kernel), in the bench's launch configuration: routing and tables bit-exact, the packed codes and scales of
    the sampled experts bit-exact against the oracle's quantizer, sampled h, y
    and token outputs within the tolerances against the oracle evaluating the
    dequantized weights."""
    shape = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    inp = synth.make_inputs(shape, device="cpu", weights_device=dev)
    enforce_margin(inp, shape)
    cfg = moe.config_of(shape)
    g = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    layer = moe.MoeLayer(cfg, inp["W1"], inp["W3"], inp["W2"], Wg=g(inp.get("Wg")),
                         bias=g(inp.get("bias")), Ws1=inp.get("Ws1"), Ws3=inp.get("Ws3"),
                         Ws2=inp.get("Ws2"), fp8=True)
    x = g(inp["x"])
    out = layer(x)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    T, k, E, d, de = shape.T, shape.k, shape.E, shape.d, shape.d_e
    A, R = shape.A, shape.rows_capacity
    x_bits = bits(inp["x"])
    bias = None if inp.get("bias") is None else inp["bias"].numpy()
    lg = oracle.router_logits(x_bits, bits(inp["Wg"]), bias)
    idx, w, margin = oracle.route(lg, k, shape.n_groups, shape.topk_groups)
    assert margin.min() >= 1e-3
    i32 = torch.int32
    assert np.array_equal(layer.buffer("topk_idx", i32, (T, k)).cpu().numpy(), idx)
    off = oracle.build_offsets(idx, w, E, shape.pad)
    perm_row = layer.buffer("perm_row", i32, (A,)).cpu().numpy()
    assert np.array_equal(perm_row, off["perm_row"])

    rng = np.random.default_rng(11)
    row_src = off["row_src"]
    samp = np.sort(rng.choice(np.flatnonzero(row_src >= 0), size=6, replace=False))
    seg = np.searchsorted(off["padded_offsets"], samp, side="right") - 1
    toks = np.sort(rng.choice(T, size=2, replace=False)).astype(np.int32)
    used = np.unique(np.concatenate([seg, idx[toks].reshape(-1)]))
    remap = {e: i for i, e in enumerate(used)}
    q = oracle.quantize_experts(dict(W1=_expert_subset(inp["W1"], used),
                                     W3=_expert_subset(inp["W3"], used),
                                     W2=_expert_subset(inp["W2"], used)))
    # the GPU's packed codes and scales of these experts
    ut = torch.as_tensor(used, device=dev, dtype=torch.long)
    which, col = _packed_rows(de)
    q13 = layer.W13q[ut].cpu().numpy()
    exp13 = np.where(which[None, :, None] == 0, q["Q1"].transpose(0, 2, 1)[:, col, :],
                     q["Q3"].transpose(0, 2, 1)[:, col, :])
    assert np.array_equal(q13, exp13)
    assert np.array_equal(layer.s13[ut].cpu().numpy(),
                          np.where(which[None, :] == 0, q["S1"][:, col], q["S3"][:, col]))
    assert np.array_equal(layer.W2q[ut].cpu().numpy(), q["Q2"].transpose(0, 2, 1))
    assert np.array_equal(layer.s2[ut].cpu().numpy(), q["S2"])

    # h, y of sampled padded rows
    ref_xp = oracle.permute(x_bits, np.where(np.isin(np.arange(R), samp), row_src, -1), k)
    eh, ey = oracle.expert_rows_w8(ref_xp[samp], np.array([remap[e] for e in seg], np.int32),
                                   off["row_gate"][samp], q)
    st = torch.as_tensor(samp, device=dev)
    h = layer.buffer("h", torch.bfloat16, (R, de))
    y = layer.buffer("y", torch.bfloat16, (R, d))
    assert_close(h[st].double().cpu().numpy(), eh, "h (sampled rows, e4m3)")
    assert_close(y[st].double().cpu().numpy(), ey, "y (sampled rows, e4m3)")

    # sampled tokens: routed experts through the oracle's rows, plus the shared expert
    qs = oracle.quantize_shared(dict(Ws1=bits(inp["Ws1"].cpu()), Ws3=bits(inp["Ws3"].cpu()),
                                     Ws2=bits(inp["Ws2"].cpu())))
    _, ys = oracle.shared_expert_w8(x_bits[toks], qs)
    rows = np.repeat(toks, k)
    _, yr = oracle.expert_rows_w8(x_bits[rows], np.array([remap[e] for e in idx[toks].reshape(-1)],
                                                          np.int32), w[toks].reshape(-1), q)
    ref_out = yr.reshape(toks.size, k, d).sum(axis=1) + ys
    got = out[torch.as_tensor(toks, device=dev, dtype=torch.long)].double().cpu().numpy()
    assert_close(got, ref_out, "out (sampled tokens, e4m3)")
    assert torch.isfinite(out.float()).all()


def _close_bwd(got, ref, what, rel_fro=1e-2, max_rel=5e-2):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), what
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    assert rel <= rel_fro, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= max_rel * np.abs(ref).max(), f"{what}: max error {mx:.3e}"


@pytest.mark.parametrize("name", ["default", "prerouted"])
def test_full_size_backward(name):
    """moe_layer_bwd at the full workload sizes, as bench.py --pass train runs
    it.  Sampled from the oracle: dx and dgates of sampled tokens (the
    oracle's layer backward on those tokens alone: dx of a token depends on
    that token only), and three columns of the weight gradients of two
    experts and of the shared expert (the oracle over every row routed to the
    expert).  Tolerances as the small-size backward parity."""
    import dataclasses

    shape = synth.WORKLOADS[name]
    dev = torch.device("cuda")
    inp = synth.make_inputs(shape, device="cpu", weights_device=dev)
    enforce_margin(inp, shape)
    cfg = moe.config_of(shape)
    g = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
    layer = moe.MoeLayer(cfg, inp["W1"], inp["W3"], inp["W2"], Wg=g(inp.get("Wg")),
                         bias=g(inp.get("bias")), Ws1=inp.get("Ws1"), Ws3=inp.get("Ws3"),
                         Ws2=inp.get("Ws2"))
    x = g(inp["x"])
    pre = bool(shape.prerouted)
    if pre:
        layer(x, topk_idx=g(inp["topk_idx"]), topk_w=g(inp["topk_w"]))
    else:
        layer(x)
    T, k, E, d, de = shape.T, shape.k, shape.E, shape.d, shape.d_e
    gen = torch.Generator().manual_seed(shape.seed + 1000)
    dout = torch.randn((T, d), generator=gen).to(torch.bfloat16)
    grads = layer.backward(x, dout.to(dev), prerouted=pre)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    for key, t in grads.items():
        assert torch.isfinite(t.float()).all(), key
    x_bits = bits(inp["x"])
    dout64 = dout.double().numpy()
    idx = layer.buffer("topk_idx", torch.int32, (T, k)).cpu().numpy() if not pre \
        else inp["topk_idx"].numpy()
    gates = layer.buffer("topk_w", torch.float32, (T, k)).cpu().double().numpy() if not pre \
        else inp["topk_w"].double().numpy()
    host = lambda key: None if inp.get(key) is None else bits(inp[key].cpu())  # noqa: E731
    W1, W3, W2 = host("W1"), host("W3"), host("W2")

    # sampled tokens: the oracle's layer backward on those tokens alone
    rng = np.random.default_rng(11)
    toks = np.sort(rng.choice(T, size=8, replace=False))
    sub = dict(x=x_bits[toks], W1=W1, W3=W3, W2=W2, Wg=host("Wg"),
               bias=None if inp.get("bias") is None else inp["bias"].numpy(),
               Ws1=host("Ws1"), Ws3=host("Ws3"), Ws2=host("Ws2"))
    if pre:
        sub.update(Wg=None, topk_idx=idx[toks], topk_w=gates[toks])
    sub_shape = dataclasses.replace(shape, T=toks.size)
    fwd = oracle.layer_forward(sub, sub_shape)
    if not pre:
        assert np.array_equal(fwd["topk_idx"], idx[toks])
    ref = oracle.layer_backward(sub, sub_shape, fwd, dout64[toks])
    tt = torch.as_tensor(toks, device=dev, dtype=torch.long)
    _close_bwd(grads["dx"][tt].double().cpu().numpy(), ref["dx"], "dx (sampled tokens)")
    _close_bwd(grads["dgates"][tt].double().cpu().numpy(), ref["dgates"], "dgates (sampled)")

    # three columns of the weight gradients of two experts, over all their rows
    J = np.array([3, de // 2, de - 1], np.int32)
    for e in (0, E - 1):
        t, j = np.nonzero(idx == e)
        dW1c, dW3c, dW2r = oracle.weight_grad_columns(x_bits[t], dout64[t], gates[t, j],
                                                      W1[e], W3[e], W2[e], J)
        Jt = torch.as_tensor(J, device=dev, dtype=torch.long)
        _close_bwd(grads["dW1"][e][:, Jt].double().cpu().numpy(), dW1c, f"dW1[{e}] columns")
        _close_bwd(grads["dW3"][e][:, Jt].double().cpu().numpy(), dW3c, f"dW3[{e}] columns")
        _close_bwd(grads["dW2"][e][Jt, :].double().cpu().numpy(), dW2r, f"dW2[{e}] rows")
    if shape.d_shared:
        Js = np.array([5, shape.d_shared - 3], np.int32)
        dW1c, dW3c, dW2r = oracle.weight_grad_columns(x_bits, dout64, np.ones(T), host("Ws1"),
                                                      host("Ws3"), host("Ws2"), Js)
        Jt = torch.as_tensor(Js, device=dev, dtype=torch.long)
        _close_bwd(grads["dWs1"][:, Jt].double().cpu().numpy(), dW1c, "dWs1 columns")
        _close_bwd(grads["dWs3"][:, Jt].double().cpu().numpy(), dW3c, "dWs3 columns")
        _close_bwd(grads["dWs2"][Jt, :].double().cpu().numpy(), dW2r, "dWs2 rows")
