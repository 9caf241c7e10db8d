"""GPU parity of the layer backward (moe_layer_bwd) against the oracle's fp64
layer backward, on the same seeded inputs and the same routing.

The backward runs bf16 GEMMs with fp32 accumulation and rounds each GEMM
output to bf16 once, so a gradient passes through at most five bf16
roundings (dz scaled by the routing weight, dh, the recomputed gate/up
values, dgu, the output itself), each a relative error of at most 2^-9 per
element.  Random rounding errors add in quadrature: the bound below,
a relative Frobenius error of 1e-2 and a max error of 5e-2 * max|ref|, is
about three times that sum.  dgates is held to the same bound.  The router
gradients come from dgates through the softmax over the chosen logits,
dlogit_j = p_j (dp_j - sum_i p_i dp_i), a difference that cancels when the
dp_j are close: their error is bounded by dgates' error times the terms
before cancellation, p_j (|dp_j| + sum_i p_i |dp_i|), so dWg and dbias are
measured against that scale (propagated through x^T and the column sums)
instead of against their own size.

Shapes: routed with a logit bias and a shared expert (several row tiles per
expert, ragged tails), group-limited routing with padding 64 and a model
width that is not a multiple of 256, a pre-routed batch with an empty expert
and repeated experts within a token, many experts (E = 100, most of them
empty), a decode-sized batch whose forward runs on the small-M kernel, a
single token, a single expert (k = 1: every gate is 1 and the router gets no
gradient) and k = E (every expert chosen by every token).
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

REL_FRO = 1e-2
MAX_REL = 5e-2

SHAPES = {
    "routed_shared": MoeShape("routed_shared", T=777, d=1024, d_e=384, E=8, k=4, bias_std=0.5,
                              d_shared=256, seed=201),
    "groups_p64_d384": MoeShape("groups_p64_d384", T=400, d=384, d_e=256, E=16, k=4, n_groups=4,
                                topk_groups=2, pad=64, seed=202),
    "prerouted_empty": MoeShape("prerouted_empty", T=150, d=256, d_e=256, E=4, k=8,
                                prerouted=(500, 0, 600, 100), seed=203),
    "e100": MoeShape("e100", T=300, d=384, d_e=128, E=100, k=3, bias_std=0.3, seed=204),
    "decode_small_m": MoeShape("decode_small_m", T=37, d=512, d_e=256, E=64, k=8, n_groups=8,
                               topk_groups=4, d_shared=128, seed=205),
    "one_token": MoeShape("one_token", T=1, d=256, d_e=128, E=8, k=2, d_shared=128, seed=206),
    "single_expert": MoeShape("single_expert", T=300, d=384, d_e=256, E=1, k=1, d_shared=128,
                              seed=207),
    "k_equals_E": MoeShape("k_equals_E", T=130, d=256, d_e=128, E=4, k=4, bias_std=0.5, seed=208),
}

_cache = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU backward tests need a CUDA device")
    moe_build.build()
    moe.load()


def _dout(shape):
    g = torch.Generator().manual_seed(shape.seed + 1000)
    return torch.randn((shape.T, shape.d), generator=g).to(torch.bfloat16)


def prepared(name):
    """(shape, CPU inputs, dout bf16, oracle forward, oracle backward)."""
    if name not in _cache:
        shape = SHAPES[name]
        inp = synth.make_inputs(shape)
        enforce_margin(inp, shape)
        oi = oracle_inputs(inp)
        fwd = oracle.layer_forward(oi, shape)
        dout = _dout(shape)
        bwd = oracle.layer_backward(oi, shape, fwd, dout.double().numpy())
        _cache[name] = (shape, inp, dout, fwd, bwd)
    return _cache[name]


def cuda(t):
    return None if t is None else t.cuda().contiguous()


def f64(t):
    return t.detach().cpu().double().numpy()


def assert_close(got, ref, what, scale=None):
    """Relative Frobenius and max error of got against ref, both measured
    against |ref| (or against ``scale``, an array of ref's shape)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref) if scale is None else np.asarray(scale, np.float64)
    assert got.shape == ref.shape == scale.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    nref = np.linalg.norm(scale)
    rel = np.linalg.norm(got - ref) / (nref if nref > 0 else 1.0)
    mx = np.abs(got - ref).max() if got.size else 0.0
    bound = MAX_REL * (scale.max() if scale.size else 0.0)
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e}"
    assert mx <= bound + 1e-30, f"{what}: max error {mx:.3e} > {bound:.3e}"


def router_scales(inp, fwd, ref):
    """Error scales of dWg and dbias: the terms of each token's dlogits
    before cancellation, summed over tokens in quadrature (the rounding errors
    of different tokens are independent), never below |ref| itself."""
    p, dp = fwd["topk_w"], np.abs(ref["dgates"])
    terms = p * (dp + (p * dp).sum(axis=1, keepdims=True))
    T, _ = p.shape
    E = ref["dbias"].shape[0]
    dl2 = np.zeros((T, E))
    for j in range(p.shape[1]):
        np.add.at(dl2, (np.arange(T), fwd["topk_idx"][:, j]), terms[:, j] ** 2)
    x = oracle.bf16_to_f64(oracle_inputs({"x": inp["x"]})["x"])
    s_wg = np.sqrt((x ** 2).T @ dl2)
    s_bias = np.sqrt(dl2.sum(axis=0))
    return np.maximum(s_wg, np.abs(ref["dWg"])), np.maximum(s_bias, np.abs(ref["dbias"]))


def run(shape, inp, dout):
    cfg = moe.config_of(shape)
    layer = moe.MoeLayer(cfg, cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]),
                         Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")),
                         Ws1=cuda(inp.get("Ws1")), Ws3=cuda(inp.get("Ws3")),
                         Ws2=cuda(inp.get("Ws2")))
    x = cuda(inp["x"])
    if shape.prerouted:
        layer(x, topk_idx=cuda(inp["topk_idx"]), topk_w=cuda(inp["topk_w"]))
    else:
        layer(x)
    g = layer.backward(x, cuda(dout), prerouted=bool(shape.prerouted))
    torch.cuda.synchronize()
    return layer, x, g


@pytest.mark.parametrize("name", list(SHAPES))
def test_backward_matches_oracle(name):
    shape, inp, dout, fwd, ref = prepared(name)
    layer, x, g = run(shape, inp, dout)
    assert layer.device_status() == 0
    for key in ("dx", "dgates", "dW1", "dW3", "dW2"):
        assert_close(f64(g[key]), ref[key], key)
    if not shape.prerouted:
        s_wg, s_bias = router_scales(inp, fwd, ref)
        assert_close(f64(g["dWg"]), ref["dWg"], "dWg", s_wg)
        assert_close(f64(g["dbias"]), ref["dbias"], "dbias", s_bias)
    else:
        assert "dWg" not in g
    if shape.d_shared:
        for key in ("dWs1", "dWs3", "dWs2"):
            assert_close(f64(g[key]), ref[key], key)
    # experts that received no rows have exactly zero weight gradients
    empty = np.flatnonzero(fwd["counts"] == 0)
    for key in ("dW1", "dW3", "dW2"):
        assert not g[key][torch.as_tensor(empty)].any() if empty.size else True


def test_backward_needs_only_the_routing_state():
    """The backward reads the forward workspace's routing state (everything
    before x_perm) and nothing else: overwriting the rest changes nothing, the
    state itself is left as it was, and a second run is bit-identical."""
    shape, inp, dout, _, _ = prepared("routed_shared")
    layer, x, g1 = run(shape, inp, dout)
    front = layer.layout["x_perm"]
    before = layer.ws[256:front].clone()
    layer.ws[front:].fill_(0xFF)
    g2 = layer.backward(x, cuda(dout))
    torch.cuda.synchronize()
    assert torch.equal(before, layer.ws[256:front])
    for key in g1:
        assert torch.equal(g1[key], g2[key]), key
    assert layer.device_status() == 0


@pytest.mark.parametrize("name", ["routed_shared", "groups_p64_d384", "decode_small_m", "e100"])
def test_backward_workspace_contents_do_not_matter(name):
    """The backward workspace filled with NaN bit patterns before a run gives
    the same gradients bit for bit: every row a kernel reads is written
    first in the same call (pad rows of 64-row blocks that hold data are
    zeroed; all-pad blocks are never read)."""
    shape, inp, dout, _, _ = prepared(name)
    layer, x, g1 = run(shape, inp, dout)
    layer.bws.fill_(0xFF)
    g2 = layer.backward(x, cuda(dout))
    torch.cuda.synchronize()
    for key in g1:
        assert torch.equal(g1[key], g2[key]), key
    assert layer.device_status() == 0


def test_frozen_router_still_differentiates_through_it():
    """dWg/dbias left NULL: dx keeps the router's term."""
    shape, inp, dout, _, ref = prepared("e100")
    layer, x, g = run(shape, inp, dout)
    grads = {k: torch.empty_like(v) for k, v in g.items() if k not in ("dWg", "dbias")}
    layer.backward(x, cuda(dout), grads=grads)
    torch.cuda.synchronize()
    assert_close(f64(grads["dx"]), ref["dx"], "dx, frozen router")
    assert torch.equal(grads["dx"], g["dx"])


def test_backward_captures_into_a_cuda_graph():
    shape, inp, dout, _, ref = prepared("groups_p64_d384")
    layer, x, g = run(shape, inp, dout)
    dz = cuda(dout)
    grads = {k: torch.zeros_like(v) for k, v in g.items()}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.backward(x, dz, grads=grads, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.backward(x, dz, grads=grads)
    for v in grads.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for key in g:
        assert torch.equal(grads[key], g[key]), key
    assert layer.device_status() == 0


def test_backward_weight_packs():
    """moe_pack_experts_bwd interleaves W1 and W3 per 128 columns along d_e;
    moe_pack_router_bwd pads Wg to a multiple of 128 columns with zeros."""
    g = torch.Generator().manual_seed(11)
    E, d, de = 3, 256, 384
    W1 = torch.randn((E, d, de), generator=g).to(torch.bfloat16).cuda()
    W3 = torch.randn((E, d, de), generator=g).to(torch.bfloat16).cuda()
    W13t = torch.empty((E, d, 2 * de), dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_experts_bwd(W1, W3, W13t)
    expect = torch.stack([W1.view(E, d, de // 128, 128), W3.view(E, d, de // 128, 128)], dim=3)
    assert torch.equal(W13t, expect.reshape(E, d, 2 * de))
    Wg = torch.randn((d, 5), generator=g).to(torch.bfloat16).cuda()
    WgP = torch.full((d, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_pack_router_bwd(Wg, WgP)
    torch.cuda.synchronize()
    assert torch.equal(WgP[:, :5], Wg) and not WgP[:, 5:].any()


def test_empty_batch_backward_is_a_noop():
    shape = MoeShape("t0", T=0, d=256, d_e=128, E=4, k=2, d_shared=128, seed=209)
    cfg = moe.config_of(shape)
    inp = synth.make_inputs(MoeShape("t1", T=1, d=256, d_e=128, E=4, k=2, d_shared=128, seed=209))
    layer = moe.MoeLayer(cfg, cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]), Wg=cuda(inp["Wg"]),
                         Ws1=cuda(inp["Ws1"]), Ws3=cuda(inp["Ws3"]), Ws2=cuda(inp["Ws2"]))
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    layer(x)
    grads = layer.backward(x, torch.empty_like(x))
    torch.cuda.synchronize()
    assert grads["dx"].shape == (0, 256)
    assert layer.device_status() == 0


def test_host_pipeline_train_matches_the_direct_calls():
    """HostPipeline.submit_train: x and dout from pinned host memory, dx back;
    the same bits as forward + backward called directly."""
    shape, inp, dout, _, _ = prepared("groups_p64_d384")
    layer, x, g = run(shape, inp, dout)
    x_host = inp["x"].pin_memory()
    dout_host = dout.pin_memory()
    dx_host = [torch.empty_like(x_host).pin_memory() for _ in range(3)]
    grads = {k: torch.empty_like(v) for k, v in g.items()}
    pipe = moe.HostPipeline(layer)
    for i in range(3):
        pipe.submit_train(x_host, dout_host, dx_host[i], grads)
    pipe.synchronize()
    for i in range(3):
        assert torch.equal(dx_host[i], g["dx"].cpu()), i
    for key in g:
        if key != "dx":
            assert torch.equal(grads[key], g[key]), key
    assert layer.device_status() == 0


def _layer(shape, inp, **kw):
    cfg = moe.config_of(shape)
    return moe.MoeLayer(cfg, cuda(inp["W1"]), cuda(inp["W3"]), cuda(inp["W2"]),
                        Wg=cuda(inp.get("Wg")), bias=cuda(inp.get("bias")),
                        Ws1=cuda(inp.get("Ws1")), Ws3=cuda(inp.get("Ws3")),
                        Ws2=cuda(inp.get("Ws2")), **kw)


@pytest.mark.parametrize("name", ["routed_shared", "prerouted_empty", "decode_small_m"])
def test_saved_gate_up_matches_the_recomputation(name):
    """moe_layer_fwd_save keeps [g|u]; the backward that reads it gives the
    forward output and gradients of the recomputing one, bit for bit where the
    forward and the recomputation run the same GEMM kernel (the CTA-pair
    kernel), and within the parity bound where the forward ran the small-M
    kernel (decode sizes)."""
    shape, inp, dout, _, ref = prepared(name)
    pre = bool(shape.prerouted)
    kw = dict(topk_idx=cuda(inp["topk_idx"]), topk_w=cuda(inp["topk_w"])) if pre else {}
    x, dz = cuda(inp["x"]), cuda(dout)
    plain, keep = _layer(shape, inp), _layer(shape, inp, keep_gate_up=True)
    out_p, out_k = plain(x, **kw), keep(x, **kw)
    g_p = plain.backward(x, dz, prerouted=pre)
    g_k = keep.backward(x, dz, prerouted=pre)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_k)
    assert keep.device_status() == 0
    if shape.T * shape.k > 32 * shape.E:  # the forward ran the CTA-pair kernel
        for key in g_p:
            assert torch.equal(g_p[key], g_k[key]), key
        return
    for key in ("dx", "dgates", "dW1", "dW3", "dW2", "dWs1", "dWs3", "dWs2"):
        if key in ref:
            assert_close(f64(g_k[key]), ref[key], key)
    if not pre:
        s_wg, s_bias = router_scales(inp, _cache[name][3], ref)
        assert_close(f64(g_k["dWg"]), ref["dWg"], "dWg", s_wg)
        assert_close(f64(g_k["dbias"]), ref["dbias"], "dbias", s_bias)
