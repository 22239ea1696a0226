"""NVFP4 path on the GPU: the quantisers bit-exact against the oracle's codec
(E2M1 codes, e4m3 block scales, tensor scales), and the whole layer against
the oracle's NVFP4 layer (max |err| <= 6e-2 x RMS, mean relative <= 5e-3),
small layers on every token and full size on sampled tokens; layer stacks
give each layer's bits."""
import numpy as np
import pytest
import torch

import moe_expert_layer_router_gb300 as m
import workload as wl
from oracle import moe as om
from oracle import nvfp4 as onv
from parity import (NVFP4_MAX_OVER_RMS, NVFP4_MEAN_REL, Case, Routing, assert_close_layer,
                    check_sampled, f64, family_parity, with_flips)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- layouts (test side)
def unpack(codes) -> np.ndarray:
    """uint8 [rows, K/2] (element 2i in the low nibble of byte i) -> codes [rows, K]."""
    c = codes.cpu().numpy() if hasattr(codes, "cpu") else np.asarray(codes)
    out = np.empty((c.shape[0], 2 * c.shape[1]), np.uint8)
    out[:, 0::2] = c & 15
    out[:, 1::2] = c >> 4
    return out


def sf_rowmajor(sf, rows, K) -> np.ndarray:
    """MMA scale layout (512-byte atoms of 128 rows x 4 blocks) -> [rows, K/16]."""
    s = sf.cpu().numpy() if hasattr(sf, "cpu") else np.asarray(sf)
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4
    return s[off]


def stacked_order(I) -> np.ndarray:
    """Row v of the interleaved gate/up matrix -> row of [W_g; W_u]."""
    v = np.arange(2 * I)
    b, i = v // 256, v % 256
    return np.where(i < 128, 128 * b + i, I + 128 * b + (i - 128))


# ---------------------------------------------------------------- quantisers
def test_weight_quantiser_bit_exact_stacked_and_plain():
    dev = torch.device("cuda")
    I, H = 384, 320
    wg = wl.rng.normal_bf16(0, 91, (I, H), 0.02, dev)
    wu = wl.rng.normal_bf16(0, 92, (I, H), 0.03, dev)
    wg[:64, :64] = 0                                    # all-zero blocks
    wu[7, 5] = 0.9                                      # the tensor's amax, in the up half
    wg[200:, 64:80] = 0                                 # zero blocks in the second 128-row block
    codes, sf, ts = m.moe_quantize_weight_nvfp4(wg, wu)
    torch.cuda.synchronize()
    ref_q, ref_s, ref_g = onv.quantize_weight(np.concatenate([f64(wg), f64(wu)]))
    order = stacked_order(I)
    assert ts.item() == float(ref_g)
    assert (unpack(codes) == ref_q[order]).all()
    assert (sf_rowmajor(sf, 2 * I, H) == ref_s[order]).all()

    wd = wl.rng.normal_bf16(0, 93, (256, 192), 0.02, dev)
    codes, sf, ts = m.moe_quantize_weight_nvfp4(wd)
    torch.cuda.synchronize()
    ref_q, ref_s, ref_g = onv.quantize_weight(f64(wd))
    assert ts.item() == float(ref_g)
    assert (unpack(codes) == ref_q).all()
    assert (sf_rowmajor(sf, 256, 192) == ref_s).all()


def test_weight_quantiser_all_zero_matrix():
    dev = torch.device("cuda")
    w = torch.zeros(128, 64, dtype=torch.bfloat16, device=dev)
    codes, sf, ts = m.moe_quantize_weight_nvfp4(w)
    torch.cuda.synchronize()
    assert ts.item() == 1.0 and int(codes.sum()) == 0 and int(sf.sum()) == 0


def test_activation_quantiser_bit_exact():
    dev = torch.device("cuda")
    g = 2.0 ** -8
    x = wl.rng.normal_bf16(0, 94, (300, 512), 1.0, dev)
    x[3] = 0                                            # zero blocks
    x[5, :16] = 5000.0                                  # saturates the block scale (448)
    x[6, 16:32] = 1e-4                                  # scale in the e4m3 subnormal range
    # a block whose scale is exactly 1 (amax = 6 g): every other quotient is an
    # exact rounding threshold (ties to the even code), and the negative ones
    # that round to zero must give +0 (code 0, not 8)
    ties = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -0.1]
    x[7, :16] = torch.tensor(ties, dtype=torch.float32).to(x.dtype).to(dev) * g
    codes, sf = m.moe_quantize_act_nvfp4(x, g)
    torch.cuda.synchronize()
    ref_q, ref_s = onv.quantize_blocks(f64(x).astype(np.float32), np.float32(g))
    assert (unpack(codes) == ref_q).all()
    assert (sf.cpu().numpy() == ref_s).all()
    assert ref_s[5, 0] == 0x7E and ref_s[3].max() == 0
    # codes of 6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 and their negatives, -0.1
    assert ref_s[7, 0] == 0x38 and list(ref_q[7, :16]) == [7, 0, 2, 2, 4, 4, 6, 6,
                                                           0, 10, 10, 12, 12, 14, 14, 0]


# ---------------------------------------------------------------- the layer
class Nvfp4Layer:
    """Seeded NVFP4 layer: bf16 weights on the device, quantised by the library
    for the GPU path; the oracle quantises its own copy of the same bf16 values."""

    def __init__(self, lc, dev):
        self.lc, self.dev = lc, dev
        self.x = wl.gen_x(lc, dev)
        self.wr = wl.gen_router(lc, dev)
        b = wl.gen_bias(lc)
        self.bias = b.to(dev) if b is not None else None
        self.gx, self.gh = wl.nvfp4_act_scales(lc)
        self.Wb = [tuple(wl.gen_expert(lc, e, w, dev) for w in ("gate", "up", "down"))
                   for e in range(lc.E)]
        self.Sb = (tuple(wl.gen_shared(lc, w, dev) for w in ("gate", "up", "down"))
                   if lc.I_shared else None)
        self.cfg = m.config_from(lc)
        self.weights = m.quantize_experts_nvfp4(
            self.cfg, [w[0] for w in self.Wb], [w[1] for w in self.Wb], [w[2] for w in self.Wb],
            shared=self.Sb, input_scale=self.gx, hidden_scale=self.gh)
        self._cache = {}

    def oracle_expert(self, e):
        if e not in self._cache:
            self._cache[e] = onv.dequantize_expert(*onv.quantize_expert(*(f64(t) for t in self.Wb[e])))
        return self._cache[e]

    def oracle_shared(self):
        if self.Sb is None:
            return None
        if "shared" not in self._cache:
            self._cache["shared"] = onv.dequantize_expert(
                *onv.quantize_expert(*(f64(t) for t in self.Sb)))
        return self._cache["shared"]

    def forward(self, ws=None):
        ws = ws or m.Workspace(self.cfg, "forward")
        out, ids, w = m.moe_forward(self.cfg, self.weights, self.x, self.wr, self.bias,
                                    return_routing=True, ws=ws)
        torch.cuda.synchronize()
        assert m.moe_get_device_error(ws) == 0
        return out, ids.cpu().numpy(), w


def check_layer(L, full_size=False):
    """Routing over every token (bit-exact off measured near ties); then every
    output row against the oracle's NVFP4 layer (small layers), or the
    stratified sample of at least 512 rows reaching every expert (full size)."""
    lc = L.lc
    out, ids, _ = L.forward()
    r = Routing(lc.name, lc, L.cfg, L.x, L.wr, L.bias, ids, m)
    assert torch.isfinite(out.float()).all()
    if full_size:
        rec = check_sampled(lc.name, lc, r, L.x, out, NVFP4_MAX_OVER_RMS, NVFP4_MEAN_REL)
        assert rec["experts_covered"] == rec["experts_with_rows"]
        return out
    b = None if L.bias is None else f64(L.bias)
    ref = onv.moe_layer_nvfp4(f64(L.x), f64(L.wr), b, L.oracle_expert, L.oracle_shared(), lc.k,
                              lc.score, lc.renormalize, lc.route_scale, L.gx, L.gh)
    ref_out = with_flips(r, ref["out"], lambda t, i, w_: onv.moe_tokens_nvfp4(
        f64(L.x)[t], i, w_, L.oracle_expert, L.oracle_shared(), L.gx, L.gh))
    assert_close_layer(out, ref_out, max_over_rms=NVFP4_MAX_OVER_RMS, mean_rel=NVFP4_MEAN_REL,
                       what=lc.name)
    return out


SMALL = [
    wl.DSV3_NVFP4.with_(name="nvfp4_small", T=200, H=512, E=8, k=2, I=256, I_shared=256),
    # ragged expert rows (some experts with a few rows, maybe none), no shared expert
    wl.DSV3_NVFP4.with_(name="nvfp4_ragged", T=150, H=1024, E=16, k=4, I=512, I_shared=0,
                        score="softmax", route_scale=1.0),
    # one token, one expert: every row block is 1 real row + 127 padding rows
    wl.DSV3_NVFP4.with_(name="nvfp4_one_token", T=1, H=512, E=4, k=1, I=256, I_shared=256),
    # several 128-row blocks per expert and a ragged last block
    wl.DSV3_NVFP4.with_(name="nvfp4_multi_block", T=700, H=768, E=4, k=2, I=768, I_shared=512),
    # Zipf-biased routing: a few hot experts with many row blocks, the coldest with none
    wl.DSV3_NVFP4.with_(name="nvfp4_skewed", T=600, H=512, E=16, k=4, I=256, I_shared=256,
                        zipf_bias=True),
]


@pytest.mark.parametrize("lc", SMALL, ids=lambda c: c.name)
def test_nvfp4_forward_matches_oracle(lc):
    check_layer(Nvfp4Layer(lc, torch.device("cuda")))


# Full-size NVFP4 layers sharing the DeepSeek-V3 weights (the bench workload, its
# 512-token batch and the skewed batch), plus the Qwen3 shape on its own.
NVFP4_FAMILY = [wl.DSV3_NVFP4,                                         # the bench workload
                wl.DSV3_NVFP4.with_(name="dsv3_nvfp4_t512", T=512),    # 16 rows per expert
                wl.DSV3_SKEW.with_(name="dsv3_skewed_nvfp4", wtype="nvfp4")]  # ~10x hottest


@pytest.fixture(scope="module")
def nvfp4_family():
    """Each DeepSeek-V3-shaped NVFP4 layer in the launch configuration the bench
    times: routing over every token, and the stratified samples of all of them
    through one oracle pass."""
    dev = torch.device("cuda")
    L = Nvfp4Layer(wl.DSV3_NVFP4.with_(T=max(lc.T for lc in NVFP4_FAMILY)), dev)
    cases, failed = [], {}
    for lc in NVFP4_FAMILY:
        x = L.x[:lc.T]
        b = wl.gen_bias(lc)
        bias = b.to(dev) if b is not None else None
        cfg = m.config_from(lc)
        ws = m.Workspace(cfg, "forward")
        out, ids, _ = m.moe_forward(cfg, L.weights, x, L.wr, bias, return_routing=True, ws=ws)
        torch.cuda.synchronize()
        try:
            m.moe_get_device_error(ws)
            r = Routing(lc.name, lc, cfg, x, L.wr, bias, ids.cpu().numpy(), m)
            cases.append(Case(lc.name, lc, r, x, out, NVFP4_MAX_OVER_RMS, NVFP4_MEAN_REL))
        except (AssertionError, m.MoeError) as e:
            failed[lc.name] = str(e)
    res = family_parity(cases)
    res.update(failed)
    return res


@pytest.mark.parametrize("lc", NVFP4_FAMILY, ids=lambda c: c.name)
def test_nvfp4_forward_full_size(nvfp4_family, lc):
    rec = nvfp4_family[lc.name]
    assert isinstance(rec, dict), rec
    assert rec["experts_covered"] == rec["experts_with_rows"]


def test_nvfp4_forward_full_size_qwen3():
    """The Qwen3 shape with NVFP4 weights (softmax routing, no shared expert)."""
    L = Nvfp4Layer(wl.QWEN3.with_(name="qwen3_nvfp4", wtype="nvfp4"), torch.device("cuda"))
    check_layer(L, full_size=True)


def test_nvfp4_deterministic_and_empty_batch():
    lc = SMALL[0]
    L = Nvfp4Layer(lc, torch.device("cuda"))
    a = L.forward()[0]
    b = L.forward()[0]
    assert torch.equal(a, b)
    cfg0 = m.config_from(lc, T=0)
    W0 = m.quantize_experts_nvfp4(cfg0, [w[0] for w in L.Wb], [w[1] for w in L.Wb],
                                  [w[2] for w in L.Wb], shared=L.Sb, input_scale=L.gx,
                                  hidden_scale=L.gh)
    out = m.moe_forward(cfg0, W0, L.x[:0], L.wr)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, lc.H)


def test_nvfp4_stack_layers_match_single_layer_calls():
    """A layer stack of NVFP4 layers: every layer gives the bits of that layer
    run alone, directly and through one CUDA graph replayed for every layer."""
    dev = torch.device("cuda")
    lc = SMALL[0]
    layers = [Nvfp4Layer(lc.with_(seed=s), dev) for s in range(2)]
    x = layers[0].x
    cfg = layers[0].cfg
    refs, oracle = [], []
    for l, L in enumerate(layers):
        out, ids, _ = m.moe_forward(cfg, L.weights, x, L.wr, return_routing=True)
        torch.cuda.synchronize()
        refs.append(out)
        r = Routing(f"nvfp4_stack_layer{l}", lc, cfg, x, L.wr, None, ids.cpu().numpy(), m)
        ref = onv.moe_layer_nvfp4(f64(x), f64(L.wr), None, L.oracle_expert, L.oracle_shared(),
                                  lc.k, lc.score, lc.renormalize, lc.route_scale, L.gx, L.gh)
        oracle.append(with_flips(r, ref["out"], lambda t, i, w_, L=L: onv.moe_tokens_nvfp4(
            f64(x)[t], i, w_, L.oracle_expert, L.oracle_shared(), L.gx, L.gh)))
    stack = m.LayerStack(cfg, [L.weights for L in layers], [L.wr for L in layers])
    layer = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = m.Workspace(cfg, "forward")
    out = torch.empty(lc.T, lc.H, dtype=torch.bfloat16, device=dev)
    for l in (1, 0, 1):
        layer.fill_(l)
        m.moe_forward_stack(cfg, stack, layer, x, out=out, ws=ws)
        torch.cuda.synchronize()
        assert_close_layer(out, oracle[l], max_over_rms=NVFP4_MAX_OVER_RMS,
                           mean_rel=NVFP4_MEAN_REL, what=f"NVFP4 stack layer {l}")
        assert torch.equal(out, refs[l]), f"layer {l}"
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        m.moe_forward_stack(cfg, stack, layer, x, out=out, ws=ws, stream=torch.cuda.current_stream())
    for l in (0, 1):
        layer.fill_(l)
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert_close_layer(out, oracle[l], max_over_rms=NVFP4_MAX_OVER_RMS,
                           mean_rel=NVFP4_MEAN_REL, what=f"graph, NVFP4 stack layer {l}")
        assert torch.equal(out, refs[l]), f"graph, layer {l}"
    assert m.moe_get_device_error(ws) == 0


# ---------------------------------------------------------------- the step calls
@pytest.mark.parametrize("lc", [SMALL[0], SMALL[1], SMALL[3], SMALL[4]], ids=lambda c: c.name)
def test_nvfp4_four_calls_match_forward_and_oracle(lc):
    """moe_route -> moe_permute_nvfp4 -> moe_grouped_ffn_nvfp4 -> moe_combine: the
    maps and the padded segments against the oracle's permutation, every
    quantised row against the oracle's codec, and the output bit-exact against
    moe_forward (the same fp16 expert rows, widened exactly) and within the
    NVFP4 bound of the oracle's layer."""
    dev = torch.device("cuda")
    L = Nvfp4Layer(lc, dev)
    cfg = L.cfg
    out_f, ids_f, w_f = m.moe_forward(cfg, L.weights, L.x, L.wr, L.bias, return_routing=True)
    ids, w, _ = m.moe_route(cfg, L.x, L.wr, L.bias)
    p = m.moe_permute_nvfp4(cfg, L.weights, ids, w, L.x)
    y, s = m.moe_grouped_ffn_nvfp4(cfg, L.weights, p, p["row_weight"])
    out4 = m.moe_combine(cfg, y, p["inv_row"], s)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids_f) and torch.equal(w, w_f)
    assert torch.equal(out4, out_f), "the four calls differ from moe_forward"

    ids_np = ids.cpu().numpy()
    counts, offsets = om.expert_histogram(ids_np, lc.E)
    perm, slot, inv = om.permutation(ids_np, lc.E)
    pad = np.zeros(lc.E + 1, np.int64)
    pad[1:] = np.cumsum((counts + 127) // 128 * 128)
    assert (p["expert_counts"].cpu().numpy() == counts).all()
    assert (p["expert_offsets"].cpu().numpy() == offsets).all()
    assert (p["pad_offsets"].cpu().numpy() == pad).all()
    assert (p["perm_token"].cpu().numpy() == perm).all()
    assert (p["inv_row"].cpu().numpy() == inv).all()
    assert (p["row_weight"].cpu().numpy() == w.cpu().numpy()[perm, slot]).all()
    # quantised rows: routed row r of expert e sits at pad[e] + (r - offsets[e])
    xq, xs = onv.quantize_blocks(f64(L.x).astype(np.float32), np.float32(L.gx))
    Rp, Tp = m.moe_nvfp4_rows(cfg)
    codes, sf = unpack(p["x_perm"]), sf_rowmajor(p["x_perm_sf"], Rp, lc.H)
    e_of = np.repeat(np.arange(lc.E), counts)
    dst = pad[e_of] + (np.arange(lc.R) - offsets[e_of])
    assert (codes[dst] == xq[perm]).all() and (sf[dst] == xs[perm]).all()
    padding = np.setdiff1d(np.arange(pad[-1]), dst)
    assert (sf[padding] == 0).all()
    if lc.I_shared:
        assert (unpack(p["x_tok"])[:lc.T] == xq).all()
        assert (sf_rowmajor(p["x_tok_sf"], Tp, lc.H)[:lc.T] == xs).all()

    r = Routing(lc.name, lc, cfg, L.x, L.wr, L.bias, ids_np, m)
    b = None if L.bias is None else f64(L.bias)
    ref = onv.moe_layer_nvfp4(f64(L.x), f64(L.wr), b, L.oracle_expert, L.oracle_shared(), lc.k,
                              lc.score, lc.renormalize, lc.route_scale, L.gx, L.gh)
    ref_out = with_flips(r, ref["out"], lambda t, i, w_: onv.moe_tokens_nvfp4(
        f64(L.x)[t], i, w_, L.oracle_expert, L.oracle_shared(), L.gx, L.gh))
    assert_close_layer(out4, ref_out, max_over_rms=NVFP4_MAX_OVER_RMS, mean_rel=NVFP4_MEAN_REL,
                       what=f"{lc.name} four calls")


def test_nvfp4_step_calls_validate_their_layer():
    """The bf16 step calls refuse NVFP4 layers (pointing at the NVFP4 calls), and
    the NVFP4 calls refuse other layers."""
    dev = torch.device("cuda")
    lc = SMALL[0]
    L = Nvfp4Layer(lc, dev)
    ids, w, _ = m.moe_route(L.cfg, L.x, L.wr)
    with pytest.raises(m.MoeError, match="moe_permute_nvfp4"):
        m.moe_permute(L.cfg, ids, w, L.x)
    bcfg = m.config_from(lc.with_(wtype="bf16"))
    with pytest.raises(m.MoeError, match="NVFP4"):
        m.moe_permute_nvfp4(bcfg, L.weights, ids, w, L.x)
