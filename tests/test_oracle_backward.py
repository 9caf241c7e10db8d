"""Pins of the oracle's layer backward, CPU only.

The hand-derived gradients of ``oracle.layer_backward`` are checked against
torch's automatic differentiation in fp64 (a library routine that derives them
independently) on tiny layers: routed with a logit bias and a shared expert,
group-limited routing, pre-routed input that repeats an expert within a token,
and k = 1.  The routing choice is held constant and the bf16 rounding of h
passes its gradient through, as the oracle's reading states; the rounded
values themselves come from the oracle.  Invariants of the softmax over the
chosen logits are checked as well.
"""
import numpy as np
import pytest
import torch

import oracle
from routing_permute_grouped_gb300.synth import MoeShape
from tests.helpers import rand_bf16

SHAPES = {
    "routed_shared": MoeShape("routed_shared", T=7, d=32, d_e=16, E=4, k=2, bias_std=0.5,
                              d_shared=16, seed=3),
    "groups": MoeShape("groups", T=6, d=32, d_e=16, E=8, k=3, n_groups=4, topk_groups=2, seed=4),
    "prerouted_repeat": MoeShape("prerouted_repeat", T=5, d=16, d_e=16, E=2, k=3,
                                 prerouted=(9, 6), seed=5),
    "top1": MoeShape("top1", T=6, d=16, d_e=16, E=3, k=1, d_shared=16, seed=6),
}


def _inputs(shape):
    rng = np.random.default_rng(shape.seed)
    T, d, de, E, k = shape.T, shape.d, shape.d_e, shape.E, shape.k
    inp = dict(x=rand_bf16((T, d), 1.0, shape.seed),
               W1=rand_bf16((E, d, de), d ** -0.5, shape.seed + 1),
               W3=rand_bf16((E, d, de), d ** -0.5, shape.seed + 2),
               W2=rand_bf16((E, de, d), de ** -0.5, shape.seed + 3))
    if shape.prerouted:
        labels = np.concatenate([np.full(n, e) for e, n in enumerate(shape.prerouted)])
        inp["topk_idx"] = rng.permutation(labels).reshape(T, k).astype(np.int32)
        inp["topk_w"] = rng.uniform(0.05, 1.0, (T, k))
        inp["Wg"] = None
    else:
        inp["Wg"] = rand_bf16((d, E), d ** -0.5, shape.seed + 4)
        inp["bias"] = (rng.standard_normal(E) * shape.bias_std).astype(np.float32) \
            if shape.bias_std else None
    if shape.d_shared:
        ds = shape.d_shared
        inp["Ws1"] = rand_bf16((d, ds), d ** -0.5, shape.seed + 5)
        inp["Ws3"] = rand_bf16((d, ds), d ** -0.5, shape.seed + 6)
        inp["Ws2"] = rand_bf16((ds, d), ds ** -0.5, shape.seed + 7)
    return inp


def _torch_grads(inp, shape, fwd, dout):
    """The same layer in torch fp64 with autograd; routing indices fixed."""
    f = lambda b: torch.tensor(oracle.bf16_to_f64(b), dtype=torch.float64,  # noqa: E731
                               requires_grad=True)
    x, W1, W3, W2 = f(inp["x"]), f(inp["W1"]), f(inp["W3"]), f(inp["W2"])
    idx = torch.as_tensor(fwd["topk_idx"]).long()
    T, k = idx.shape
    leaves = dict(x=x, W1=W1, W3=W3, W2=W2)
    if inp.get("Wg") is not None:
        Wg = f(inp["Wg"])
        leaves["Wg"] = Wg
        bias = torch.zeros(shape.E, dtype=torch.float64, requires_grad=True)
        if inp.get("bias") is not None:
            bias = torch.tensor(inp["bias"].astype(np.float64), requires_grad=True)
        leaves["bias"] = bias
        logits = x @ Wg + bias
        leaves["logits_probe"] = logits
        logits.retain_grad()
        gates = torch.softmax(logits.gather(1, idx), dim=1)
    else:
        gates = torch.tensor(np.asarray(fwd["topk_w"], np.float64), requires_grad=True)
        leaves["gates"] = gates

    def round_st(h):  # the oracle's bf16 rounding, gradient passed straight through
        r = torch.from_numpy(oracle.round_bf16(h.detach().numpy()))
        return h + (r - h).detach()

    rows = []
    for t in range(T):
        acc = torch.zeros(shape.d, dtype=torch.float64)
        for j in range(k):
            e = int(idx[t, j])
            g = x[t] @ W1[e]
            u = x[t] @ W3[e]
            acc = acc + gates[t, j] * (round_st(torch.nn.functional.silu(g) * u) @ W2[e])
        rows.append(acc)
    out = torch.stack(rows)
    if shape.d_shared:
        Ws1, Ws3, Ws2 = f(inp["Ws1"]), f(inp["Ws3"]), f(inp["Ws2"])
        leaves.update(Ws1=Ws1, Ws3=Ws3, Ws2=Ws2)
        out = out + round_st(torch.nn.functional.silu(x @ Ws1) * (x @ Ws3)) @ Ws2
    (out * torch.from_numpy(dout)).sum().backward()
    return out.detach().numpy(), leaves


def _close(a, b, what, rtol=1e-9):
    a, b = np.asarray(a), np.asarray(b)
    scale = max(np.abs(b).max(), 1e-300)
    assert np.abs(a - b).max() <= rtol * scale, f"{what}: {np.abs(a - b).max():.3e} vs {scale:.3e}"


@pytest.mark.parametrize("name", list(SHAPES))
def test_backward_matches_autograd(name):
    shape = SHAPES[name]
    inp = _inputs(shape)
    fwd = oracle.layer_forward(inp, shape)
    dout = np.random.default_rng(shape.seed + 99).standard_normal((shape.T, shape.d))
    g = oracle.layer_backward(inp, shape, fwd, dout)
    out_t, L = _torch_grads(inp, shape, fwd, dout)
    _close(out_t, fwd["out"], "forward of the torch reference", rtol=1e-12)
    _close(g["dx"], L["x"].grad, "dx")
    _close(g["dW1"], L["W1"].grad, "dW1")
    _close(g["dW3"], L["W3"].grad, "dW3")
    _close(g["dW2"], L["W2"].grad, "dW2")
    if "Wg" in L:
        _close(g["dWg"], L["Wg"].grad, "dWg")
        _close(g["dbias"], L["bias"].grad, "dbias")
        _close(g["dlogits"], L["logits_probe"].grad, "dlogits")
    else:
        _close(g["dgates"], L["gates"].grad, "dgates")
    if shape.d_shared:
        _close(g["dWs1"], L["Ws1"].grad, "dWs1")
        _close(g["dWs3"], L["Ws3"].grad, "dWs3")
        _close(g["dWs2"], L["Ws2"].grad, "dWs2")


def test_router_gradient_invariants():
    shape = SHAPES["routed_shared"]
    inp = _inputs(shape)
    fwd = oracle.layer_forward(inp, shape)
    dout = np.random.default_rng(1).standard_normal((shape.T, shape.d))
    g = oracle.layer_backward(inp, shape, fwd, dout)
    dl = g["dlogits"]
    idx = fwd["topk_idx"]
    chosen = np.zeros_like(dl, bool)
    np.put_along_axis(chosen, idx.astype(np.int64), True, axis=1)
    assert np.all(dl[~chosen] == 0.0)
    # softmax over the chosen logits: its Jacobian rows sum to zero
    assert np.abs(dl.sum(axis=1)).max() < 1e-12 * np.abs(dl).max()
    assert np.allclose(g["dbias"], dl.sum(axis=0), rtol=0, atol=1e-14)
    # dlogits from dgates by the closed form p * (dp - <p, dp>)
    p, dp = fwd["topk_w"], g["dgates"]
    expect = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    assert np.allclose(np.take_along_axis(dl, idx.astype(np.int64), axis=1), expect, rtol=1e-12,
                       atol=1e-15)


def test_top1_router_has_no_gradient():
    shape = SHAPES["top1"]
    inp = _inputs(shape)
    fwd = oracle.layer_forward(inp, shape)
    g = oracle.layer_backward(inp, shape, fwd, np.ones((shape.T, shape.d)))
    assert np.all(fwd["topk_w"] == 1.0)
    assert not g["dlogits"].any() and not g["dWg"].any() and not g["dbias"].any()


@pytest.mark.parametrize("name", ["routed_shared", "prerouted_repeat"])
def test_weight_grad_columns_match_autograd(name):
    """oracle.weight_grad_columns (columns of one expert's weight gradients
    over the rows routed to it) against torch fp64 autograd, for every expert
    and the shared expert."""
    shape = SHAPES[name]
    inp = _inputs(shape)
    fwd = oracle.layer_forward(inp, shape)
    dout = np.random.default_rng(shape.seed + 77).standard_normal((shape.T, shape.d))
    _, L = _torch_grads(inp, shape, fwd, dout)
    idx, gates = fwd["topk_idx"], fwd["topk_w"]
    J = np.array([0, shape.d_e - 1, shape.d_e // 2 + 1], np.int32)
    for e in range(shape.E):
        t, j = np.nonzero(idx == e)
        if t.size == 0:
            continue
        dW1c, dW3c, dW2r = oracle.weight_grad_columns(inp["x"][t], dout[t], gates[t, j],
                                                      inp["W1"][e], inp["W3"][e], inp["W2"][e], J)
        _close(dW1c, L["W1"].grad[e][:, J].numpy(), f"dW1[{e}] columns")
        _close(dW3c, L["W3"].grad[e][:, J].numpy(), f"dW3[{e}] columns")
        _close(dW2r, L["W2"].grad[e][J, :].numpy(), f"dW2[{e}] rows")
    if shape.d_shared:
        Js = np.array([1, shape.d_shared - 2], np.int32)
        dW1c, dW3c, dW2r = oracle.weight_grad_columns(inp["x"], dout, np.ones(shape.T),
                                                      inp["Ws1"], inp["Ws3"], inp["Ws2"], Js)
        _close(dW1c, L["Ws1"].grad[:, Js].numpy(), "dWs1 columns")
        _close(dW3c, L["Ws3"].grad[:, Js].numpy(), "dWs3 columns")
        _close(dW2r, L["Ws2"].grad[Js, :].numpy(), "dWs2 rows")
