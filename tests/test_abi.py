"""The C-ABI library: it loads, exports every symbol the header declares, and
rejects bad arguments on the host before anything reaches a GPU.  CPU only:
every call here fails validation before its first CUDA call."""
import ctypes as C
import re

import pytest

import moe_expert_layer_router_gb300 as m
from moe_expert_layer_router_gb300 import _native as N


@pytest.fixture(scope="module")
def L():
    from moe_expert_layer_router_gb300 import build
    build.build()
    return m.load()


def header_functions():
    txt = open(N.HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(L):
    names = header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(N._SIG), "binding and header disagree"


def test_abi_version_and_strings(L):
    assert L.moe_abi_version() == 2
    for s in range(7):
        assert L.moe_status_string(s)


def test_config_struct_layout():
    assert C.sizeof(N.MoeConfig) == 48
    assert N.MoeConfig.route_scale.offset == 36


def cfg(**kw):
    base = dict(T=256, H=512, E=8, k=2, I=1024, I_shared=0, score="softmax")
    base.update(kw)
    return m.make_config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(E=0), N.MOE_ERR_UNSUPPORTED), (dict(E=300), N.MOE_ERR_UNSUPPORTED),
    (dict(k=0), N.MOE_ERR_INVALID_ARG), (dict(k=9), N.MOE_ERR_INVALID_ARG),
    (dict(E=32, k=17), N.MOE_ERR_INVALID_ARG), (dict(H=500), N.MOE_ERR_UNSUPPORTED),
    (dict(H=64), N.MOE_ERR_UNSUPPORTED), (dict(I=100), N.MOE_ERR_UNSUPPORTED),
    (dict(I_shared=64), N.MOE_ERR_UNSUPPORTED), (dict(T=-1), N.MOE_ERR_INVALID_ARG),
    (dict(T=1 << 29, k=8, E=8), N.MOE_ERR_UNSUPPORTED),
])
def test_bad_config_rejected(L, kw, status):
    c = cfg(**kw)
    n = C.c_size_t(0)
    assert L.moe_workspace_size(C.byref(c), N.MOE_OP_FORWARD, C.byref(n)) == status
    assert L.moe_last_error_message()


def test_bad_enums_rejected(L):
    for field, val in (("score", 7), ("renormalize", 2), ("wtype", 5)):
        c = cfg()
        setattr(c, field, val)
        n = C.c_size_t(0)
        assert L.moe_workspace_size(C.byref(c), 0, C.byref(n)) == N.MOE_ERR_INVALID_ARG
    c = cfg()
    c.route_scale = float("nan")
    assert L.moe_workspace_size(C.byref(c), 0, C.byref(C.c_size_t())) == N.MOE_ERR_INVALID_ARG


def test_workspace_sizes_grow_with_op(L):
    c = cfg(T=1000, E=32, k=4, H=1024, I=512, I_shared=256)
    sizes = {op: m.moe_workspace_size(c, op) for op in ("route", "permute", "grouped_ffn",
                                                         "combine", "forward")}
    assert all(v % 256 == 0 for v in sizes.values())
    assert sizes["route"] == sizes["combine"] == 256
    R = 1000 * 4
    # forward holds x_perm and y_perm (bf16 [R, H]) at least
    assert sizes["forward"] >= 2 * R * 1024 * 2 + sizes["grouped_ffn"]
    assert sizes["grouped_ffn"] >= R * 512 * 2 + 1000 * 256 * 2


def test_workspace_checks_before_launch(L):
    c = cfg()
    # NULL and misaligned workspaces fail before any device work
    assert L.moe_route(C.byref(c), 16, 16, None, 16, 16, None, None, 0, None) == N.MOE_ERR_WORKSPACE
    assert L.moe_route(C.byref(c), 16, 16, None, 16, 16, None, 0x1008, 4096, None) == N.MOE_ERR_WORKSPACE
    assert L.moe_combine(C.byref(c), 16, 16, None, 32, 0x1000, 16, None) == N.MOE_ERR_WORKSPACE


def test_pointer_checks_before_launch(L):
    c = cfg()
    ws = 0x10000
    # NULL x, misaligned x, NULL outputs
    assert L.moe_route(C.byref(c), None, 16, None, 16, 16, None, ws, 256, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_route(C.byref(c), 0x1002, 16, None, 16, 16, None, ws, 256, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_route(C.byref(c), 16, 16, None, None, 16, None, ws, 256, None) == N.MOE_ERR_INVALID_ARG
    assert b"topk_ids" in L.moe_last_error_message()
    assert L.moe_combine(C.byref(c), 16, 16, None, 16, ws, 256, None) == N.MOE_ERR_INVALID_ARG  # alias
    assert L.moe_combine(C.byref(c), None, 16, None, 32, ws, 256, None) == N.MOE_ERR_INVALID_ARG


def test_zero_tokens_is_a_noop(L):
    c = cfg(T=0)
    # T = 0 returns OK without touching any pointer or launching anything
    assert L.moe_route(C.byref(c), None, None, None, None, None, None, 0x10000, 256, None) == N.MOE_OK
    assert L.moe_combine(C.byref(c), None, None, None, None, 0x10000, 256, None) == N.MOE_OK


def test_weights_create_validates(L):
    c = cfg()
    wl = N.MoeWeightList()
    h = C.c_void_p()
    assert L.moe_weights_create(C.byref(c), C.byref(wl), C.byref(h)) == N.MOE_ERR_INVALID_ARG
    arr = (C.c_void_p * 8)(*([0x1000] * 7 + [0x1001]))
    wl.gate = wl.up = wl.down = C.cast(arr, C.POINTER(C.c_void_p))
    assert L.moe_weights_create(C.byref(c), C.byref(wl), C.byref(h)) == N.MOE_ERR_INVALID_ARG
    assert b"gate[7]" in L.moe_last_error_message()
    assert h.value is None
    assert L.moe_weights_create(None, C.byref(wl), C.byref(h)) == N.MOE_ERR_INVALID_ARG


def test_quantize_validation(L):
    assert L.moe_quantize_weight_fp8(16, 100, 128, 16, 16, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_act_fp8(16, 4, 100, 16, 16, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_act_fp8(None, 0, 128, None, None, None) == N.MOE_OK


def test_forward_ex_rejects_unknown_flags(L):
    c = cfg()
    ws = 0x10000
    nb = C.c_size_t()
    assert L.moe_workspace_size(C.byref(c), N.MOE_OP_FORWARD, C.byref(nb)) == 0
    rc = L.moe_forward_ex(C.byref(c), None, 16, 16, None, 16, None, None, 0x8, ws, nb.value, None)
    assert rc == N.MOE_ERR_INVALID_ARG and b"flags" in L.moe_last_error_message()


def test_stack_create_validates(L):
    """moe_stack_create checks every layer's list before touching the device."""
    c = cfg()
    h = C.c_void_p()
    good = (C.c_void_p * 8)(*([0x1000] * 8))
    bad = (C.c_void_p * 8)(*([0x1000] * 5 + [0x1001] + [0x1000] * 2))
    wls = (N.MoeWeightList * 2)()
    for wl, arr in zip(wls, (good, bad)):
        wl.gate = wl.up = wl.down = C.cast(arr, C.POINTER(C.c_void_p))
    routers = (C.c_void_p * 2)(0x2000, 0x2000)
    assert L.moe_stack_create(C.byref(c), 0, wls, routers, None, C.byref(h)) == N.MOE_ERR_INVALID_ARG
    assert L.moe_stack_create(C.byref(c), 2, None, routers, None, C.byref(h)) == N.MOE_ERR_INVALID_ARG
    assert L.moe_stack_create(C.byref(c), 2, wls, routers, None, C.byref(h)) == N.MOE_ERR_INVALID_ARG
    assert b"gate[5]" in L.moe_last_error_message()      # layer 1's bad pointer
    assert h.value is None


def test_forward_stack_validates(L):
    c = cfg()
    nb = C.c_size_t()
    assert L.moe_workspace_size(C.byref(c), N.MOE_OP_FORWARD, C.byref(nb)) == 0
    ws = 0x10000
    assert L.moe_forward_stack(C.byref(c), None, 16, 16, 16, None, None, ws, nb.value,
                               None) == N.MOE_ERR_INVALID_ARG
    assert b"stack" in L.moe_last_error_message()


def test_nvfp4_config_and_entry_points(L):
    """NVFP4 layers need H, I, I_shared multiples of 256, and run only through
    moe_forward / moe_forward_stack."""
    n = C.c_size_t(0)
    for kw in (dict(H=384), dict(I=384), dict(I_shared=128)):
        c = cfg(wtype="nvfp4", **kw)
        assert L.moe_workspace_size(C.byref(c), N.MOE_OP_FORWARD, C.byref(n)) == N.MOE_ERR_UNSUPPORTED
    c = cfg(wtype="nvfp4", I_shared=256)
    assert L.moe_workspace_size(C.byref(c), N.MOE_OP_FORWARD, C.byref(n)) == N.MOE_OK
    # the padded NVFP4 rows: at most T*k + 127 E, in 128-row blocks, times H/2 + H/16 bytes
    Rp = (256 * 2 + 127 * 8 + 127) // 128 * 128
    assert n.value >= Rp * (512 // 2 + 512 // 16)
    ws = 0x100000
    assert L.moe_permute(C.byref(c), 16, None, None, 16, 16, 16, 16, None, None, None, ws,
                         n.value, None) == N.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_ffn(C.byref(c), 16, 16, None, 16, None, None, None, 16, None, ws,
                             n.value, None) == N.MOE_ERR_UNSUPPORTED


def test_nvfp4_weight_list_layout():
    assert N.MoeWeightList.gate_sf.offset == 12 * 8
    assert N.MoeWeightList.input_scale.offset == 20 * 8
    assert C.sizeof(N.MoeWeightList) == 20 * 8 + 8


def test_nvfp4_weights_create_validates(L):
    c = cfg(wtype="nvfp4", I=512)
    h = C.c_void_p()
    wl = N.MoeWeightList()
    good = (C.c_void_p * 8)(*([0x1000] * 8))
    P = C.POINTER(C.c_void_p)
    wl.gate = wl.down = C.cast(good, P)
    # scale and tensor-scale arrays missing
    assert L.moe_weights_create(C.byref(c), C.byref(wl), C.byref(h)) == N.MOE_ERR_INVALID_ARG
    assert b"gate_sf" in L.moe_last_error_message()
    bad_sf = (C.c_void_p * 8)(*([0x1000] * 3 + [0x1008] + [0x1000] * 4))
    wl.gate_sf = C.cast(bad_sf, P)
    wl.down_sf = wl.gate_tscale = wl.down_tscale = C.cast(good, P)
    wl.input_scale, wl.hidden_scale = 1.0, 0.0
    assert L.moe_weights_create(C.byref(c), C.byref(wl), C.byref(h)) == N.MOE_ERR_INVALID_ARG
    assert b"hidden_scale" in L.moe_last_error_message()
    wl.hidden_scale = 0.0625
    assert L.moe_weights_create(C.byref(c), C.byref(wl), C.byref(h)) == N.MOE_ERR_INVALID_ARG
    assert b"gate_sf[3]" in L.moe_last_error_message()
    assert h.value is None


def test_nvfp4_quantize_validation(L):
    assert L.moe_quantize_weight_nvfp4(16, None, 100, 128, 16, 16, 16, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_weight_nvfp4(16, 16, 64, 128, 16, 16, 16, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_weight_nvfp4(16, None, 128, 96, 16, 16, 16, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_act_nvfp4(16, 4, 100, 1.0, 16, 16, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_act_nvfp4(16, 4, 128, 0.0, 16, 16, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_act_nvfp4(None, 0, 128, 1.0, None, None, None) == N.MOE_OK


def test_nvfp4_step_calls_validate(L):
    """The NVFP4 step calls: buffer sizes, and host checks before any launch."""
    c = cfg(wtype="nvfp4", I_shared=256)
    rows, toks = C.c_int64(0), C.c_int64(0)
    assert L.moe_nvfp4_rows(C.byref(c), C.byref(rows), C.byref(toks)) == N.MOE_OK
    assert rows.value == (256 * 2 + 127 * 8 + 127) // 128 * 128 and toks.value == 256
    b = cfg()
    assert L.moe_nvfp4_rows(C.byref(b), C.byref(rows), None) == N.MOE_ERR_INVALID_ARG
    n = C.c_size_t(0)
    assert L.moe_workspace_size(C.byref(c), N.MOE_OP_PERMUTE, C.byref(n)) == N.MOE_OK
    ws = 0x100000
    args = (16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16)
    assert L.moe_permute_nvfp4(C.byref(b), 16, *args, ws, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    assert b"NVFP4 layers only" in L.moe_last_error_message()
    assert L.moe_permute_nvfp4(C.byref(c), None, *args, ws, n.value, None) == N.MOE_ERR_INVALID_ARG
    assert b"weights" in L.moe_last_error_message()
    assert L.moe_permute_nvfp4(C.byref(c), 16, *args, ws, 64, None) == N.MOE_ERR_WORKSPACE
    assert L.moe_workspace_size(C.byref(c), N.MOE_OP_GROUPED_FFN, C.byref(n)) == N.MOE_OK
    fargs = (16, 16, 16, 16, 16, 16, 16, 16, 16)
    assert L.moe_grouped_ffn_nvfp4(C.byref(b), 16, *fargs, ws, 1 << 30, None) == N.MOE_ERR_INVALID_ARG
    assert L.moe_grouped_ffn_nvfp4(C.byref(c), None, *fargs, ws, n.value, None) == N.MOE_ERR_INVALID_ARG


def test_failure_test_hook_and_noalloc_checks(L):
    """moe_test_stall_gemm1 rejects a negative count; moe_permute_noalloc validates
    exactly as moe_permute (E > 256 is unsupported, not an invalid argument)."""
    assert L.moe_test_stall_gemm1(-1) == N.MOE_ERR_INVALID_ARG
    assert L.moe_test_stall_gemm1(0) == N.MOE_OK
    c = cfg(E=300)
    assert L.moe_permute_noalloc(C.byref(c), 16, None, None, 16, 16, 16, 16, None, None, None,
                                 None, None) == N.MOE_ERR_UNSUPPORTED
    c = cfg(wtype="nvfp4", I_shared=256)
    assert L.moe_permute_noalloc(C.byref(c), 16, None, None, 16, 16, 16, 16, None, None, None,
                                 None, None) == N.MOE_ERR_UNSUPPORTED
