"""moe_permute_noalloc: the permutation step for callers that cannot allocate
device memory (graph-recording code, runtimes with a memory plan fixed at
start-up, plugins handed only their tensors).  It keeps its scratch in a
fixed array inside the library instead of a caller workspace.

Called through the C ABI twice in a row -- a larger layer, then a smaller one,
so the second call meets the first call's leftovers in the shared array --
and compared with moe_permute (workspace version) output by output.  The
permutation is integer work plus row copies, so the comparison is exact.
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


def _noalloc_via_c_abi(cfg, ids, w, x, status):
    """Call the C entry point directly; every output buffer is made here, by the
    test, since the entry point itself allocates nothing."""
    dev = ids.device
    T, k, E, H = cfg.T, cfg.k, cfg.E, cfg.H
    out = {"expert_counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
           "expert_offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
           "perm_token": torch.full((T * k,), -7, dtype=torch.int32, device=dev),
           "inv_row": torch.full((T, k), -7, dtype=torch.int32, device=dev),
           "row_weight": torch.full((T * k,), -7.0, dtype=torch.float32, device=dev),
           "x_perm": torch.zeros(T * k, H, dtype=torch.bfloat16, device=dev)}
    rc = N.lib().moe_permute_noalloc(
        C.byref(cfg), ids.data_ptr(), w.data_ptr(), x.data_ptr(),
        out["expert_counts"].data_ptr(), out["expert_offsets"].data_ptr(),
        out["perm_token"].data_ptr(), out["inv_row"].data_ptr(), out["row_weight"].data_ptr(),
        out["x_perm"].data_ptr(), None, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    N.check(rc, "moe_permute_noalloc")
    return out


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
        ws = m.Workspace(cfg, "permute")
        ref = m.moe_permute(cfg, ids, w, x, ws=ws)
        torch.cuda.synchronize()
        m.moe_get_device_error(ws)
        for name in ("expert_counts", "expert_offsets", "perm_token", "inv_row", "row_weight",
                     "x_perm"):
            assert torch.equal(got[name], ref[name]), f"call {i + 1}: {name} differs"
        assert int(status.item()) == 0, f"call {i + 1}: device status {int(status.item())}"


def test_noalloc_rejects_layers_beyond_its_scratch():
    cfg = m.config_from(wl.DSV3.with_(T=65537))        # ceil(T/64) * 256 > 262144
    rc = N.lib().moe_permute_noalloc(C.byref(cfg), 16, None, None, 16, 16, 16, 16, None, None,
                                     None, None, None)
    assert rc == N.MOE_ERR_UNSUPPORTED
    assert b"exceeds the fixed scratch" in N.lib().moe_last_error_message()
