"""Test-side helpers: tensor <-> oracle array conversion and the routing
margin filter.  Tests only; never imported by the library."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from routing_permute_grouped_gb300 import synth


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def rand_bf16(shape, std=1.0, seed=0) -> np.ndarray:
    g = torch.Generator().manual_seed(seed)
    return bits((torch.randn(shape, generator=g) * std).to(torch.bfloat16))


def oracle_inputs(inp: dict) -> dict:
    """The synth tensors as numpy arrays in the oracle's conventions."""
    out = {}
    for key, v in inp.items():
        if v is None:
            out[key] = None
        elif v.dtype == torch.bfloat16:
            out[key] = bits(v)
        elif v.dtype == torch.int32:
            out[key] = v.cpu().numpy()
        else:
            out[key] = v.cpu().to(torch.float64).numpy() if key == "topk_w" else v.cpu().numpy()
    return out


def enforce_margin(inp: dict, shape, min_margin: float = 1e-3, max_attempts: int = 50) -> int:
    """Redraw token rows of inp['x'] (in place, CPU tensor) whose routing
    decision is closer than min_margin to a tie, as judged by the oracle's
    fp64 logits.  Returns the number of redraws."""
    if inp.get("Wg") is None:
        return 0
    x = inp["x"]
    Wg = bits(inp["Wg"])
    bias = None if inp.get("bias") is None else inp["bias"].cpu().numpy()
    rows = np.arange(shape.T)
    redrawn = 0
    for attempt in range(max_attempts):
        lg = oracle.router_logits(bits(x[torch.as_tensor(rows)]), Wg, bias)
        _, _, m = oracle.route(lg, shape.k, shape.n_groups, shape.topk_groups)
        bad = rows[m < min_margin]
        if bad.size == 0:
            return redrawn
        synth.redraw_rows(x, bad, shape.seed, attempt)
        redrawn += bad.size
        rows = bad
    raise RuntimeError("could not reach the routing margin")
