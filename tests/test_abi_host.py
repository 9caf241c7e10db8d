"""CPU tests of the C ABI: the library builds, loads and exports every entry
point that include/moe.h declares, and the host-side argument checks return
their errors before anything is enqueued (no GPU is touched here)."""
import ctypes
import os
import re

import pytest

import routing_permute_grouped_gb300 as moe
from routing_permute_grouped_gb300 import build as moe_build
from routing_permute_grouped_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "moe_layer_fwd" in names and "moe_build_offsets" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"


def test_status_strings(lib):
    assert moe.moe_status_string(0) == "ok"
    assert "workspace" in moe.moe_status_string(3)


def _cfg(**kw):
    base = dict(T=256, d=512, d_e=256, E=8, k=2)
    base.update(kw)
    return moe.config_of(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(d=500), 2), (dict(d_e=200), 2), (dict(E=300), 2), (dict(k=9, E=16), 2),
    (dict(pad_multiple=32), 2), (dict(d_shared=100), 2), (dict(T=-1), 1), (dict(E=0), 1),
])
def test_check_config_rejects(lib, kw, status):
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_check_config(_cfg(**kw))
    assert ei.value.status == status


@pytest.mark.parametrize("kw", [dict(k=5, E=4), dict(n_groups=3, E=8), dict(n_groups=4, topk_groups=1, k=3),
                                dict(n_groups=4, topk_groups=5)])
def test_route_rejects_before_launch(lib, kw):
    cfg = _cfg(**kw)
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the checks fail first
    st = lib.moe_route(ctypes.byref(cfg), fake, fake, None, fake, fake, None)
    assert st == 1


def test_workspace_sizes_follow_the_capacities(lib):
    for name in ("tiny", "default", "prerouted", "decode", "imbalance_x2_p64"):
        s = synth.WORKLOADS[name]
        cfg = moe.config_of(s)
        L = moe.moe_workspace_layout(cfg)
        assert L["total"] == moe.moe_workspace_size(cfg)
        R = s.A + s.E * (s.pad - 1)
        assert L["h"] - L["x_perm"] >= R * s.d * 2
        assert L["y"] - L["h"] >= R * s.d_e * 2
        offs = [L[n] for n in ("status", "topk_idx", "topk_w", "counts", "padded_offsets",
                               "block_metadata", "num_blocks", "perm_row", "row_src", "row_gate",
                               "x_perm", "h", "y", "hs", "ys")]
        assert offs == sorted(offs) and all(o % 1024 == 0 for o in offs)


def test_layer_rejects_small_workspace_and_nulls(lib):
    cfg = _cfg()
    fake = ctypes.c_void_p(0x1000)
    w = moe.MoeWeights(Wg_t=0x1000, bias=None, W13=0x1000, W2=0x1000, Ws13=None, Ws2=None)
    need = moe.moe_workspace_size(cfg)
    assert lib.moe_layer_fwd(ctypes.byref(cfg), ctypes.byref(w), fake, fake, fake, need - 1, None) == 3
    assert lib.moe_layer_fwd(ctypes.byref(cfg), ctypes.byref(w), None, fake, fake, need, None) == 1
    w2 = moe.MoeWeights(Wg_t=None, bias=None, W13=0x1000, W2=0x1000, Ws13=None, Ws2=None)
    assert lib.moe_layer_fwd(ctypes.byref(cfg), ctypes.byref(w2), fake, fake, fake, need, None) == 1
    cfg_s = _cfg(d_shared=256)
    need_s = moe.moe_workspace_size(cfg_s)
    assert lib.moe_layer_fwd(ctypes.byref(cfg_s), ctypes.byref(w), fake, fake, fake, need_s, None) == 1
    assert "shared" in lib.moe_last_error().decode()


def test_offsets_scratch_checked(lib):
    cfg = _cfg()
    fake = ctypes.c_void_p(0x1000)
    need = moe.moe_offsets_workspace_size(cfg)
    assert need >= 256 + cfg.E * 4
    st = lib.moe_build_offsets(ctypes.byref(cfg), fake, None, fake, fake, fake, fake, fake, fake,
                               fake, fake, need - 4, None)
    assert st == 3


def test_empty_batch_is_a_noop(lib):
    cfg = _cfg(T=0)
    fake = ctypes.c_void_p(0x1000)
    assert lib.moe_permute(ctypes.byref(cfg), fake, fake, fake, None) == 0
    assert lib.moe_combine(ctypes.byref(cfg), fake, fake, None, fake, None) == 0
    assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, fake, fake, None) == 0


def test_fp8_entry_points_check_arguments_before_launch(lib):
    cfg = _cfg()
    fake = ctypes.c_void_p(0x1000)
    need = moe.moe_workspace_size_fp8(cfg)
    assert need > moe.moe_workspace_size(cfg)  # the e4m3 layer needs its extra regions
    L8 = moe.moe_workspace_layout_fp8(cfg)
    assert L8["total"] == need and L8["row_scale"] > L8["h8"] >= L8["xs8"] >= L8["router_partial"]
    w = moe.MoeWeightsFp8(Wg_t=0x1000, bias=None, W13q=0x1000, s13=0x1000, W2q=0x1000, s2=0x1000)
    assert lib.moe_layer_fwd_fp8(ctypes.byref(cfg), ctypes.byref(w), fake, fake, fake, need - 1,
                                 None) == 3
    w_noscale = moe.MoeWeightsFp8(Wg_t=0x1000, W13q=0x1000, s13=None, W2q=0x1000, s2=0x1000)
    assert lib.moe_layer_fwd_fp8(ctypes.byref(cfg), ctypes.byref(w_noscale), fake, fake, fake,
                                 need, None) == 1
    assert "scales" in lib.moe_last_error().decode()
    cfg_s = _cfg(d_shared=256)
    need_s = moe.moe_workspace_size_fp8(cfg_s)
    assert lib.moe_layer_fwd_fp8(ctypes.byref(cfg_s), ctypes.byref(w), fake, fake, fake, need_s,
                                 None) == 1
    assert lib.moe_layer_fwd_fp8_prerouted(ctypes.byref(cfg), ctypes.byref(w), fake, None, fake,
                                           fake, fake, need, None) == 1
    # null operands of the stage calls
    args15 = [fake] * 15
    args15[11] = None  # h8
    assert lib.moe_grouped_gemm_swiglu_fp8(ctypes.byref(cfg), *args15) == 1
    assert lib.moe_grouped_gemm_swiglu_skinny(ctypes.byref(cfg), fake, fake, fake, None, fake,
                                              None, fake, fake, None, None) == 1
    assert lib.moe_permute_fp8(ctypes.byref(cfg), fake, fake, fake, None, None, None, None) == 1
    assert lib.moe_permute_fp8(ctypes.byref(cfg), fake, fake, fake, fake, fake, None, None) == 1
    assert lib.moe_shared_expert_fp8(ctypes.byref(cfg_s), *([fake] * 9), None, None, None) == 1
    # packing: shape rules
    assert lib.moe_pack_experts_fp8(2, 200, 128, fake, fake, fake, fake, fake, fake, fake,
                                    None) == 2
    assert lib.moe_pack_experts_fp8(2, 256, 128, fake, fake, fake, fake, None, fake, fake,
                                    None) == 1
    # T = 0 is a no-op
    cfg0 = _cfg(T=0)
    assert lib.moe_layer_fwd_fp8(ctypes.byref(cfg0), ctypes.byref(w), fake, fake, fake,
                                 moe.moe_workspace_size_fp8(cfg0), None) == 0
    args15 = [fake] * 15
    args15[13] = None  # status
    args15[14] = None  # stream
    assert lib.moe_grouped_gemm_swiglu_fp8(ctypes.byref(cfg0), *args15) == 0


def test_backward_entry_points_check_arguments_before_launch(lib):
    cfg = _cfg(d_shared=256)
    fake = 0x1000
    fp = ctypes.c_void_p(fake)
    need_f = moe.moe_workspace_size(cfg)
    need_b = moe.moe_backward_workspace_size(cfg)
    assert need_b > 0 and moe.moe_backward_workspace_size(_cfg(d=500)) == 0
    w = moe.MoeWeights(Wg_t=fake, bias=None, W13=fake, W2=fake, Ws13=fake, Ws2=fake)
    wb = moe.MoeWeightsBwd(W13t=fake, W2=fake, WgP=fake, Ws13t=fake, Ws2=fake)
    full = {n: fake for n in moe._GRAD_FIELDS}
    g = moe.MoeGrads(**full)

    def call(c=cfg, w=w, wb=wb, g=g, fwd_bytes=need_f, bws_bytes=need_b, x=fp, gu=None, gu_bytes=0):
        return lib.moe_layer_bwd(ctypes.byref(c), ctypes.byref(w), ctypes.byref(wb), x, fp, fp,
                                 fwd_bytes, gu, gu_bytes, ctypes.byref(g), fp, bws_bytes, None)

    assert call(bws_bytes=need_b - 1) == 3
    # the backward needs only the routing state at the front of the forward workspace
    assert call(fwd_bytes=moe.moe_workspace_layout(cfg)["x_perm"] - 1) == 3
    assert call(x=None) == 1
    assert call(g=moe.MoeGrads(**dict(full, dW2=None))) == 1
    assert call(g=moe.MoeGrads(**dict(full, dWs3=None))) == 1
    assert "shared" in lib.moe_last_error().decode()
    assert call(wb=moe.MoeWeightsBwd(W13t=fake, W2=fake, WgP=None, Ws13t=fake, Ws2=fake)) == 1
    assert "WgP" in lib.moe_last_error().decode()
    assert call(c=_cfg(d_shared=256, d_e=200)) == 2
    # a gate/up save shorter than its size
    need_gu = moe.moe_gate_up_save_size(cfg)
    R = 256 * 2 + 8 * 127
    assert need_gu >= R * 2 * 256 * 2 + 256 * 2 * 256 * 2
    assert call(gu=fp, gu_bytes=need_gu - 1) == 3
    assert lib.moe_layer_fwd_save(ctypes.byref(cfg), ctypes.byref(w), fp, None, None, fp, fp,
                                  moe.moe_workspace_size(cfg), fp, need_gu - 1, None) == 3
    # T = 0: nothing to do, nothing enqueued
    c0 = _cfg(T=0, d_shared=256)
    assert call(c=c0, fwd_bytes=moe.moe_workspace_size(c0),
                bws_bytes=moe.moe_backward_workspace_size(c0)) == 0
    # packs: shape rules
    assert lib.moe_pack_experts_bwd(2, 200, 128, fp, fp, fp, None) == 2
    assert lib.moe_pack_experts_bwd(2, 256, 128, fp, None, fp, None) == 1
    assert lib.moe_pack_router_bwd(256, 0, fp, fp, None) == 1


def test_exchange_and_widened_entry_points_check_arguments_before_launch(lib):
    """moe_gather_rows, moe_widen_e4m3 and the scaled (widened e4m3) stage
    calls reject bad sizes and null operands before any launch, and are
    no-ops for empty inputs."""
    fake = ctypes.c_void_p(0x1000)
    # gather: sizes, d % 8, gates both or neither; n = 0 touches nothing
    assert lib.moe_gather_rows(fake, fake, fake, ctypes.c_int64(-1), 64, None, None, None) == 1
    assert lib.moe_gather_rows(fake, fake, fake, ctypes.c_int64(4), 60, None, None, None) == 2
    assert lib.moe_gather_rows(fake, fake, fake, ctypes.c_int64(4), 64, fake, None, None) == 1
    assert lib.moe_gather_rows(None, None, None, ctypes.c_int64(0), 64, None, None, None) == 0
    assert lib.moe_gather_rows(None, fake, fake, ctypes.c_int64(4), 64, None, None, None) == 1
    # widen: n % 16, null buffers; n = 0 is a no-op
    assert lib.moe_widen_e4m3(fake, fake, ctypes.c_int64(24), None) == 2
    assert lib.moe_widen_e4m3(None, fake, ctypes.c_int64(32), None) == 1
    assert lib.moe_widen_e4m3(None, None, ctypes.c_int64(0), None) == 0
    # scaled stages: null operands; the shared one needs d_shared > 0
    cfg = _cfg()
    args = [fake] * 13
    args[2] = None  # s13
    assert lib.moe_grouped_gemm_swiglu_scaled(ctypes.byref(cfg), *args) == 1
    assert lib.moe_shared_expert_scaled(ctypes.byref(cfg), *([fake] * 7), None, None) == 1
    cfg_s = _cfg(d_shared=256)
    sargs = [fake] * 7
    sargs[2] = None  # ss13
    assert lib.moe_shared_expert_scaled(ctypes.byref(cfg_s), *sargs, None, None) == 1


def test_pack_weights_checks_arguments_before_launch(lib):
    """moe_pack_weights takes the layer's config: the config rules and null
    operands are rejected before anything is enqueued."""
    fake = ctypes.c_void_p(0x1000)
    assert lib.moe_pack_weights(ctypes.byref(_cfg(d=500)), fake, fake, fake, None) == 2
    assert lib.moe_pack_weights(ctypes.byref(_cfg(d_e=200)), fake, fake, fake, None) == 2
    assert lib.moe_pack_weights(ctypes.byref(_cfg()), fake, None, fake, None) == 1
    assert lib.moe_pack_weights(ctypes.byref(_cfg()), fake, fake, None, None) == 1
    assert lib.moe_pack_weights(None, fake, fake, fake, None) == 1


def test_exchange_table_entry_points_check_arguments_before_launch(lib):
    """moe_build_blocks_from_counts and moe_copy_pieces reject bad sizes and
    null operands before any launch."""
    fake = ctypes.c_void_p(0x1000)
    f = lib.moe_build_blocks_from_counts
    assert f(fake, 0, 8, 128, fake, fake, fake, 10, None, None, None) == 1   # no sender
    assert f(fake, 2, 300, 128, fake, fake, fake, 10, None, None, None) == 2  # E > 256
    assert f(fake, 2, 8, 96, fake, fake, fake, 10, None, None, None) == 2    # P
    assert f(None, 2, 8, 128, fake, fake, fake, 10, None, None, None) == 1
    assert f(fake, 2, 8, 128, fake, None, fake, 10, None, None, None) == 1
    c = lib.moe_copy_pieces
    assert c(fake, fake, 60, fake, fake, fake, 3, 8, None, None, None) == 2  # d % 8
    assert c(fake, fake, 64, fake, fake, fake, 3, 8, fake, None, None) == 1  # gates both or neither
    assert c(fake, fake, 64, None, fake, fake, 3, 8, None, None, None) == 1
    assert c(None, None, 64, None, None, None, 0, 0, None, None, None) == 0  # nothing to move


def test_unpadded_entry_points_check_arguments_before_launch(lib):
    fake = ctypes.c_void_p(0x1000)
    cfg = _cfg()
    small = moe.moe_offsets_workspace_size(cfg) - 1
    assert lib.moe_build_offsets_unpadded(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake,
                                          fake, fake, small, None) == 3
    assert lib.moe_build_offsets_unpadded(ctypes.byref(cfg), fake, fake, None, fake, fake, fake,
                                          fake, fake, small + 1, None) == 1
    assert lib.moe_grouped_gemm_swiglu_unpadded(ctypes.byref(cfg), fake, fake, fake, None, fake,
                                                fake, fake, None, None) == 1
    assert lib.moe_grouped_gemm_swiglu_unpadded(ctypes.byref(_cfg(d_e=200)), fake, fake, fake,
                                                fake, fake, fake, fake, None, None) == 2


def test_shared_expert_halves_check_arguments_before_launch(lib):
    """moe_shared_expert_up / _down / _down_combine need a shared expert and
    their operands; the permute of _up takes perm_row and x_perm both or
    neither; an empty batch is a no-op."""
    fake = ctypes.c_void_p(0x1000)
    cfg, cfg_s = _cfg(), _cfg(d_shared=256)
    up, down, dc = lib.moe_shared_expert_up, lib.moe_shared_expert_down, \
        lib.moe_shared_expert_down_combine
    assert up(ctypes.byref(cfg), fake, fake, fake, None, None, None, None) == 1       # no shared
    assert up(ctypes.byref(cfg_s), fake, fake, fake, fake, None, None, None) == 1     # perm alone
    assert up(ctypes.byref(cfg_s), fake, fake, fake, None, fake, None, None) == 1     # x_perm alone
    assert up(ctypes.byref(cfg_s), None, fake, fake, None, None, None, None) == 1
    assert down(ctypes.byref(cfg_s), fake, fake, None, None, None) == 1
    assert down(ctypes.byref(cfg), fake, fake, fake, None, None) == 1
    assert dc(ctypes.byref(cfg_s), fake, fake, fake, None, fake, None, None) == 1     # no perm_row
    assert dc(ctypes.byref(cfg_s), fake, fake, fake, fake, None, None, None) == 1     # no out
    empty = _cfg(d_shared=256, T=0)
    assert up(ctypes.byref(empty), None, None, None, None, None, None, None) == 0
    assert down(ctypes.byref(empty), None, None, None, None, None) == 0
    assert dc(ctypes.byref(empty), None, None, None, None, None, None, None) == 0


def test_binding_signatures_match_the_header(lib):
    """Every entry point the binding declares to ctypes takes as many
    arguments as include/moe.h gives it (a mismatch would only show at the
    first call on a GPU)."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    decls = dict(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", src))
    checked = 0
    for name, params in decls.items():
        argtypes = getattr(getattr(lib, name), "argtypes", None)
        if argtypes is None:
            continue
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        assert len(argtypes) == n, f"{name}: {len(argtypes)} argtypes, {n} parameters in the header"
        checked += 1
    assert checked >= 40
