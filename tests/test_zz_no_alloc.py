"""moe_permute_noalloc: the permutation step for callers that cannot allocate
device memory (graph-recording code, runtimes with a memory plan fixed at
start-up, plugins handed only their tensors).  It keeps its scratch in a
fixed array inside the library instead of a caller workspace.

Called through the C ABI twice in a row -- a larger layer, then a smaller one,
so the second call meets the first call's leftovers in the shared array --
and compared with moe_permute (workspace version) output by output.  The
permutation is integer work plus row copies, so the comparison is exact.
Also: an fp8 layer with no status word, a layer at the scratch's size limit,
a call recorded into a CUDA graph and replayed, and a repeated expert id.
This file is collected last so that a failure here leaves every other test
already run."""
import ctypes as C

import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from moe_expert_layer_router_gb300 import _native as N

pytestmark = pytest.mark.gpu


def _random_routing(T, E, k, seed, dev):
    g = np.random.default_rng(seed)
    ids = np.argsort(g.random((T, E)), axis=1)[:, :k].astype(np.int32)
    w = g.random((T, k)).astype(np.float32)
    return torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)


def _outputs(cfg, dev):
    """Output buffers of one call, made by the test (the entry point allocates
    nothing), filled with a marker so that an unwritten entry shows."""
    T, k, E, H = cfg.T, cfg.k, cfg.E, cfg.H
    fp8 = cfg.wtype == N.MOE_DTYPE_FP8_E4M3
    return {"expert_counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
            "expert_offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            "perm_token": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
            "inv_row": torch.full((T, k), -7, dtype=torch.int32, device=dev),
            "row_weight": torch.full((T * k,), -7.0, dtype=torch.float32, device=dev),
            "x_perm": torch.zeros(T * k, H, dtype=torch.uint8 if fp8 else torch.bfloat16,
                                  device=dev),
            "x_perm_scales": (torch.full((T * k, H // 128), -7.0, dtype=torch.float32, device=dev)
                              if fp8 else None)}


def _call(cfg, ids, w, x, out, status):
    """The C entry point, called directly with the test's buffers."""
    sc = out["x_perm_scales"]
    return N.lib().moe_permute_noalloc(
        C.byref(cfg), ids.data_ptr(), w.data_ptr(), x.data_ptr(),
        out["expert_counts"].data_ptr(), out["expert_offsets"].data_ptr(),
        out["perm_token"].data_ptr(), out["inv_row"].data_ptr(), out["row_weight"].data_ptr(),
        out["x_perm"].data_ptr(), None if sc is None else sc.data_ptr(),
        None if status is None else status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _noalloc_via_c_abi(cfg, ids, w, x, status):
    out = _outputs(cfg, ids.device)
    N.check(_call(cfg, ids, w, x, out, status), "moe_permute_noalloc")
    return out


def _reference(cfg, ids, w, x):
    ws = m.Workspace(cfg, "permute")
    ref = m.moe_permute(cfg, ids, w, x, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    return ref


def _assert_same(got, ref, what):
    for name in ("expert_counts", "expert_offsets", "perm_token", "inv_row", "row_weight",
                 "x_perm", "x_perm_scales"):
        if got[name] is None:
            assert ref[name] is None
            continue
        assert torch.equal(got[name], ref[name]), f"{what}: {name} differs"


def test_noalloc_permute_matches_workspace_permute_on_two_calls():
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    layers = [wl.DSV3.with_(name="first", T=3000, E=256, k=8, H=1024),
              wl.TINY.with_(name="second", T=333, E=16, k=4, H=256)]
    for i, lc in enumerate(layers):
        cfg = m.config_from(lc)
        ids, w = _random_routing(lc.T, lc.E, lc.k, seed=11 + i, dev=dev)
        x = wl.gen_x(lc, dev)
        got = _noalloc_via_c_abi(cfg, ids, w, x, status)
        ref = _reference(cfg, ids, w, x)
        _assert_same(got, ref, f"call {i + 1}")
        assert int(status.item()) == 0, f"call {i + 1}: device status {int(status.item())}"


def test_noalloc_fp8_and_without_status_word():
    """fp8 layers (each token quantised once, codes and 1x128 scales gathered) and a
    NULL device_status, which discards the status bits."""
    dev = torch.device("cuda")
    lc = wl.DSV3_FP8.with_(name="fp8_noalloc", T=700, E=64, k=6, H=512)
    cfg = m.config_from(lc)
    ids, w = _random_routing(lc.T, lc.E, lc.k, seed=21, dev=dev)
    x = wl.gen_x(lc, dev)
    got = _noalloc_via_c_abi(cfg, ids, w, x, None)
    _assert_same(got, _reference(cfg, ids, w, x), "fp8")


def test_noalloc_at_its_size_limit():
    """E * ceil(T/64) = 262144 exactly: T = 65536 tokens over E = 256 experts."""
    dev = torch.device("cuda")
    lc = wl.DSV3.with_(name="limit", T=65536, E=256, k=8, H=128)
    cfg = m.config_from(lc)
    ids, w = _random_routing(lc.T, lc.E, lc.k, seed=31, dev=dev)
    x = wl.gen_x(lc, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = _noalloc_via_c_abi(cfg, ids, w, x, status)
    _assert_same(got, _reference(cfg, ids, w, x), "T=65536, E=256")
    assert int(status.item()) == 0


def test_noalloc_recorded_in_a_cuda_graph():
    """A caller that records its step into a CUDA graph: one call before the
    capture, then the call recorded and the graph replayed on new routing."""
    dev = torch.device("cuda")
    lc = wl.DSV3.with_(name="graph", T=1000, E=64, k=4, H=256)
    cfg = m.config_from(lc)
    ids, w = _random_routing(lc.T, lc.E, lc.k, seed=41, dev=dev)
    x = wl.gen_x(lc, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = _outputs(cfg, dev)
    N.check(_call(cfg, ids, w, x, out, status), "warm-up call")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rc = _call(cfg, ids, w, x, out, status)
    N.check(rc, "moe_permute_noalloc during capture")
    for seed in (42, 43):
        ids2, w2 = _random_routing(lc.T, lc.E, lc.k, seed=seed, dev=dev)
        ids.copy_(ids2)
        w.copy_(w2)
        for t in out.values():
            if t is not None:
                t.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        _assert_same(out, _reference(cfg, ids, w, x), f"graph replay {seed}")
        assert int(status.item()) == 0


def test_noalloc_flags_a_repeated_expert_id():
    """Routing whose token lists one expert twice is reported (status bit 3)."""
    dev = torch.device("cuda")
    lc = wl.TINY.with_(name="dup", T=100, E=8, k=2, H=256)
    cfg = m.config_from(lc)
    ids, w = _random_routing(lc.T, lc.E, lc.k, seed=51, dev=dev)
    ids[17, 1] = ids[17, 0]
    x = wl.gen_x(lc, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _noalloc_via_c_abi(cfg, ids, w, x, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 8


def test_noalloc_rejects_layers_beyond_its_scratch():
    cfg = m.config_from(wl.DSV3.with_(T=65537))        # ceil(T/64) * 256 > 262144
    rc = N.lib().moe_permute_noalloc(C.byref(cfg), 16, None, None, 16, 16, 16, 16, None, None,
                                     None, None, None)
    assert rc == N.MOE_ERR_UNSUPPORTED
    assert b"exceeds the fixed scratch" in N.lib().moe_last_error_message()
