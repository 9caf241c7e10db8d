"""The allocation-free offsets entry point (moe_build_offsets_noalloc).

It serves callers that cannot allocate device memory where they build the
routing tables (runtimes that only use a pool reserved at start-up, for one):
its scratch is a fixed array inside the library.  The
GPU test checks, through the C ABI, that two calls in a row give the same
tables as moe_build_offsets with a caller-allocated scratch; tables are
integer (and copied gates), so the comparison is exact.  The file is named to
be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build


def _tables(E, T, k, P, dev):
    A, R, NB = T * k, T * k + E * (P - 1), (T * k) // P + E
    z = lambda n, dt=torch.int32: torch.full(n, -3, dtype=dt, device=dev)  # noqa: E731
    return dict(counts=z((E,)), padded_offsets=z((E + 1,)), block_metadata=z((NB, 3)),
                num_blocks=z((1,)), perm_row=z((A,)), row_src=z((R,)),
                row_gate=z((R,), torch.float32))


def _order(t):
    return (t["counts"], t["padded_offsets"], t["block_metadata"], t["num_blocks"], t["perm_row"],
            t["row_src"], t["row_gate"])


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    moe_build.build()
    moe.load()
    dev = "cuda"
    # the larger scratch user first, so stale counts from it would show in
    # the later, smaller calls; the third case (T*k <= 4096) takes the
    # one-CTA offsets kernel, the fourth carries expert ids outside [0, E),
    # which both entry points skip and flag in their status words
    cases = [(256, 1111, 8, 64, 11, False), (8, 4097, 4, 128, 12, False),
             (16, 300, 6, 64, 13, False), (32, 2500, 4, 128, 14, True)]
    for E, T, k, P, seed, bad in cases:
        rng = np.random.default_rng(seed)
        p = rng.dirichlet(np.full(E, 0.2))
        idx_h = rng.choice(E, size=(T, k), p=p).astype(np.int32)
        if bad:
            idx_h[3, 1] = E
            idx_h[T - 1, 0] = E + 7
        idx = torch.from_numpy(idx_h).to(dev)
        w = torch.from_numpy(rng.random((T, k)).astype(np.float32)).to(dev)
        cfg = moe.config_of(T=T, d=128, d_e=128, E=E, k=k, pad_multiple=P)
        ref = _tables(E, T, k, P, dev)
        ws = torch.zeros(moe.moe_offsets_workspace_size(cfg), dtype=torch.uint8, device=dev)
        moe.moe_build_offsets(cfg, idx, w, *_order(ref), ws)
        got = _tables(E, T, k, P, dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        moe.moe_build_offsets_noalloc(cfg, idx, w, *_order(got), status=status)
        torch.cuda.synchronize()
        want = moe.DEVERR_EXPERT_RANGE if bad else 0
        assert int(status.item()) == want
        assert int(ws[:4].view(torch.int32).item()) == want
        nb = int(ref["num_blocks"].item())
        assert nb == int(got["num_blocks"].item()) and nb > 0
        for key in ("counts", "padded_offsets", "perm_row", "row_src", "row_gate"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["block_metadata"][:nb], ref["block_metadata"][:nb])


def test_noalloc_rejects_configs_beyond_its_static_scratch():
    moe_build.build()
    lib = moe.load()
    cfg = moe.config_of(T=20000, d=128, d_e=128, E=256, k=8)  # 79 chunks x 256 experts
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the size check comes first
    st = lib.moe_build_offsets_noalloc(ctypes.byref(cfg), fake, None, fake, fake, fake, fake,
                                       fake, fake, fake, None, None)
    assert st == 3
    assert "static" in lib.moe_last_error().decode()
