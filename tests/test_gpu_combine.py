"""moe_combine on the GPU: exact-input sums within the fp32-sum + bf16-rounding bound."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import moe as om
from parity import f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,k,H,shared", [(256, 2, 512, False), (97, 8, 7168, True),
                                          (1, 1, 128, True), (300, 16, 256, False)])
def test_combine_matches_oracle(T, k, H, shared):
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=T, k=k, H=H, E=max(k, 8))
    cfg = m.config_from(lc)
    g = np.random.default_rng(T * 31 + k)
    inv = g.permutation(T * k).reshape(T, k)
    y = wl.rng.normal_f32(3, 11, (T * k, H), 1.0, dev)
    s = wl.rng.normal_f32(3, 12, (T, H), 1.0, dev) if shared else None
    ws = m.Workspace(cfg, "combine")
    out = m.moe_combine(cfg, y, torch.from_numpy(inv.astype(np.int32)).to(dev), s, ws=ws)
    torch.cuda.synchronize()
    m.moe_get_device_error(ws)
    ref = om.combine(f64(y), inv, None if s is None else f64(s))
    # fp32 sum of <= k+1 fp32 terms (gamma_{k+1} with u = 2^-24), then one rounding to
    # bf16 (unit roundoff 2^-8, relative to the value rounded)
    absum = np.abs(f64(y))[inv].sum(axis=1) + (np.abs(f64(s)) if shared else 0)
    g = (k + 1) * 2.0 ** -24 * absum
    bound = g + 2.0 ** -8 * (np.abs(ref) + g) + 1e-30
    assert (np.abs(f64(out) - ref) <= bound).all()


def test_combine_flags_bad_rows():
    dev = torch.device("cuda")
    lc = wl.TINY.with_(T=4, k=2, H=128)
    cfg = m.config_from(lc)
    inv = torch.tensor([[0, 1], [2, 3], [4, 5], [6, 1000]], dtype=torch.int32, device=dev)
    y = torch.ones(8, 128, dtype=torch.float32, device=dev)
    ws = m.Workspace(cfg, "combine")
    out = m.moe_combine(cfg, y, inv, ws=ws)
    torch.cuda.synchronize()
    with pytest.raises(m.MoeError):
        m.moe_get_device_error(ws)
    assert (out[:3].float().cpu() == 2).all() and (out[3].float().cpu() == 1).all()
