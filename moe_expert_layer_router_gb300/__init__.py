"""GB300 (sm_103a) forward pass of one Mixture-of-Experts FFN layer.

Thin Python binding over the C ABI of ``include/moe_layer.h``: every function
here only checks tensor metadata, allocates outputs with torch (device memory
plumbing) and calls the library.  Every step of the layer runs in the
library's CUDA kernels; there is no Python or CPU implementation behind these
calls.

    cfg = make_config(T=..., H=..., E=..., k=..., I=..., score="sigmoid", route_scale=2.5)
    W = ExpertWeights(cfg, gate, up, down, shared=(sg, su, sd))
    ws = Workspace(cfg, "forward")
    out = moe_forward(cfg, W, x, w_router, ws=ws)
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _native as N
from ._native import MoeConfig, MoeError

__all__ = ["MoeConfig", "MoeError", "make_config", "config_from", "Workspace", "ExpertWeights",
           "moe_route", "moe_permute", "moe_permute_noalloc", "moe_grouped_ffn", "moe_combine",
           "moe_nvfp4_rows", "moe_permute_nvfp4", "moe_grouped_ffn_nvfp4",
           "moe_forward", "LayerStack", "moe_forward_stack",
           "moe_quantize_weight_fp8", "moe_quantize_act_fp8", "moe_get_device_error",
           "moe_workspace_size", "load", "Nvfp4ExpertWeights", "moe_quantize_weight_nvfp4",
           "moe_quantize_act_nvfp4", "quantize_experts_nvfp4"]

_OPS = {"route": N.MOE_OP_ROUTE, "permute": N.MOE_OP_PERMUTE, "grouped_ffn": N.MOE_OP_GROUPED_FFN,
        "combine": N.MOE_OP_COMBINE, "forward": N.MOE_OP_FORWARD}


def load():
    """Load the shared library (raises ImportError if it was not built)."""
    return N.lib()


def make_config(T, H, E, k, I, I_shared=0, score="softmax", renormalize=True, route_scale=1.0,
                wtype="bf16") -> MoeConfig:
    return MoeConfig(int(T), int(H), int(E), int(k), int(I), int(I_shared),
                     {"softmax": N.MOE_SCORE_SOFTMAX, "sigmoid": N.MOE_SCORE_SIGMOID}[score],
                     1 if renormalize else 0, float(route_scale),
                     {"bf16": N.MOE_DTYPE_BF16, "fp8_e4m3": N.MOE_DTYPE_FP8_E4M3,
                      "nvfp4": N.MOE_DTYPE_NVFP4}[wtype])


def config_from(layer, T: int | None = None) -> MoeConfig:
    """MoeConfig of an object with the fields of workload.LayerConfig."""
    return make_config(layer.T if T is None else T, layer.H, layer.E, layer.k, layer.I,
                       layer.I_shared, layer.score, layer.renormalize, layer.route_scale,
                       layer.wtype)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t, name, dtype, shape, device):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def moe_workspace_size(cfg: MoeConfig, op: str = "forward") -> int:
    n = C.c_size_t(0)
    N.check(N.lib().moe_workspace_size(C.byref(cfg), _OPS[op], C.byref(n)), "moe_workspace_size")
    return int(n.value)


class Workspace:
    """Caller-owned workspace for one op (device memory from torch), initialised once."""

    def __init__(self, cfg: MoeConfig, op: str = "forward", device=None, stream=None):
        self.nbytes = max(moe_workspace_size(cfg, op), 256)
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=dev)
        off = (-self.buf.data_ptr()) % 256
        self.view = self.buf[off:off + self.nbytes]
        self.ptr = self.view.data_ptr()
        self.device = dev
        N.check(N.lib().moe_workspace_init(self.ptr, self.nbytes, _stream(stream)),
                "moe_workspace_init")


def moe_get_device_error(ws: Workspace, stream=None) -> int:
    """Raise MoeError if a kernel flagged a bounds/timeout error; returns the raw bits."""
    bits = C.c_int32(0)
    N.check(N.lib().moe_get_device_error(ws.ptr, _stream(stream), C.byref(bits)),
            "device status")
    return int(bits.value)


def _ptr_array(ts):
    arr = (C.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return arr


class ExpertWeights:
    """Per-expert weight pointer list -> device table of TMA descriptors.

    The tensors are referenced, not copied; keep them alive (this object holds
    references).  gate[e], up[e]: [I, H]; down[e]: [H, I]; shared: (gate, up,
    down) of the shared expert or None.  bf16 tensors, or uint8 e4m3 codes
    plus fp32 block scales (``scales=(gate_s, up_s, down_s)`` lists and
    ``shared_scales``) for fp8 layers."""

    def __init__(self, cfg: MoeConfig, gate, up, down, shared=None, scales=None,
                 shared_scales=None):
        E = cfg.E
        if not (len(gate) == len(up) == len(down) == E):
            raise ValueError("gate/up/down must each list E tensors")
        fp8 = cfg.wtype == N.MOE_DTYPE_FP8_E4M3
        wdt = torch.uint8 if fp8 else torch.bfloat16
        for e in range(E):
            _need(gate[e], f"gate[{e}]", wdt, (cfg.I, cfg.H), None)
            _need(up[e], f"up[{e}]", wdt, (cfg.I, cfg.H), None)
            _need(down[e], f"down[{e}]", wdt, (cfg.H, cfg.I), None)
        self._keep = [list(gate), list(up), list(down), shared, scales, shared_scales]
        self._arrays = [_ptr_array(gate), _ptr_array(up), _ptr_array(down)]
        wl = N.MoeWeightList()
        wl.gate = C.cast(self._arrays[0], C.POINTER(C.c_void_p))
        wl.up = C.cast(self._arrays[1], C.POINTER(C.c_void_p))
        wl.down = C.cast(self._arrays[2], C.POINTER(C.c_void_p))
        if scales is not None:
            sa = [_ptr_array(s) for s in scales]
            self._arrays += sa
            wl.gate_scales, wl.up_scales, wl.down_scales = (
                C.cast(a, C.POINTER(C.c_void_p)) for a in sa)
        if shared is not None:
            sg, su, sd = shared
            _need(sg, "shared_gate", wdt, (cfg.I_shared, cfg.H), None)
            _need(su, "shared_up", wdt, (cfg.I_shared, cfg.H), None)
            _need(sd, "shared_down", wdt, (cfg.H, cfg.I_shared), None)
            wl.shared_gate, wl.shared_up, wl.shared_down = sg.data_ptr(), su.data_ptr(), sd.data_ptr()
        if shared_scales is not None:
            wl.shared_gate_scales, wl.shared_up_scales, wl.shared_down_scales = (
                s.data_ptr() for s in shared_scales)
        self.cfg = cfg
        self._wl = wl
        h = C.c_void_p()
        N.check(N.lib().moe_weights_create(C.byref(cfg), C.byref(wl), C.byref(h)),
                "moe_weights_create")
        self.handle = h.value

    def close(self):
        if getattr(self, "handle", None):
            N.lib().moe_weights_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Nvfp4ExpertWeights:
    """NVFP4 expert weights (MOE_DTYPE_NVFP4) -> device descriptor table.

    Per expert e: ``gate_up[e]`` uint8 [2I, H/2] (stacked gate/up E2M1 codes,
    rows interleaved in 128-row blocks), ``down[e]`` uint8 [H, I/2], their
    MMA-layout block scales ``gate_up_sf[e]`` / ``down_sf[e]`` (uint8, rows*K/16
    bytes) and fp32 tensor scales ``gate_up_ts`` / ``down_ts`` (device float32
    tensors [E]: entry e is expert e's).  ``shared`` = (gate_up, down,
    gate_up_sf, down_sf, tensor scales [2]) or None.  ``input_scale`` and
    ``hidden_scale`` are the static activation tensor scales g_x, g_h.  The
    tensors are referenced, not copied; this object keeps them alive."""

    def __init__(self, cfg: MoeConfig, gate_up, down, gate_up_sf, down_sf, gate_up_ts, down_ts,
                 input_scale, hidden_scale, shared=None):
        E, H, I = cfg.E, cfg.H, cfg.I
        if not (len(gate_up) == len(down) == len(gate_up_sf) == len(down_sf) == E):
            raise ValueError("gate_up/down and their scales must each list E tensors")
        for e in range(E):
            _need(gate_up[e], f"gate_up[{e}]", torch.uint8, (2 * I, H // 2), None)
            _need(down[e], f"down[{e}]", torch.uint8, (H, I // 2), None)
            _need(gate_up_sf[e], f"gate_up_sf[{e}]", torch.uint8, (2 * I * H // 16,), None)
            _need(down_sf[e], f"down_sf[{e}]", torch.uint8, (H * I // 16,), None)
        _need(gate_up_ts, "gate_up_ts", torch.float32, (E,), None)
        _need(down_ts, "down_ts", torch.float32, (E,), None)
        self._keep = [list(gate_up), list(down), list(gate_up_sf), list(down_sf), gate_up_ts,
                      down_ts, shared]
        ts = lambda t: (C.c_void_p * E)(*[t.data_ptr() + 4 * e for e in range(E)])
        self._arrays = [_ptr_array(gate_up), _ptr_array(down), _ptr_array(gate_up_sf),
                        _ptr_array(down_sf), ts(gate_up_ts), ts(down_ts)]
        wl = N.MoeWeightList()
        P = C.POINTER(C.c_void_p)
        wl.gate = C.cast(self._arrays[0], P)
        wl.down = C.cast(self._arrays[1], P)
        wl.gate_sf = C.cast(self._arrays[2], P)
        wl.down_sf = C.cast(self._arrays[3], P)
        wl.gate_tscale = C.cast(self._arrays[4], P)
        wl.down_tscale = C.cast(self._arrays[5], P)
        wl.input_scale = float(input_scale)
        wl.hidden_scale = float(hidden_scale)
        if shared is not None:
            sgu, sd, sgu_sf, sd_sf, sts = shared
            Is = cfg.I_shared
            _need(sgu, "shared gate_up", torch.uint8, (2 * Is, H // 2), None)
            _need(sd, "shared down", torch.uint8, (H, Is // 2), None)
            _need(sts, "shared tensor scales", torch.float32, (2,), None)
            wl.shared_gate, wl.shared_down = sgu.data_ptr(), sd.data_ptr()
            wl.shared_gate_sf, wl.shared_down_sf = sgu_sf.data_ptr(), sd_sf.data_ptr()
            wl.shared_gate_tscale, wl.shared_down_tscale = sts.data_ptr(), sts.data_ptr() + 4
        self.cfg = cfg
        self.input_scale = float(input_scale)
        self.hidden_scale = float(hidden_scale)
        self._wl = wl
        h = C.c_void_p()
        N.check(N.lib().moe_weights_create(C.byref(cfg), C.byref(wl), C.byref(h)),
                "moe_weights_create")
        self.handle = h.value

    def close(self):
        if getattr(self, "handle", None):
            N.lib().moe_weights_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LayerStack:
    """L layers of one shape behind one device descriptor table (moe_stack_create):
    ``layers`` is a list of ExpertWeights (kept alive here), ``w_router`` a list of
    bf16 [E, H] router matrices, ``bias`` None or a list of fp32 [E] tensors (or
    None entries).  moe_forward_stack picks the layer from a device int32 tensor
    when its kernels run, so one recorded CUDA graph serves every layer."""

    def __init__(self, cfg: MoeConfig, layers, w_router, bias=None):
        L = len(layers)
        if L < 1 or len(w_router) != L or (bias is not None and len(bias) != L):
            raise ValueError("layers, w_router (and bias) must list the same L >= 1 layers")
        for l, w in enumerate(w_router):
            _need(w, f"w_router[{l}]", torch.bfloat16, (cfg.E, cfg.H), None)
        self._keep = [list(layers), list(w_router), bias]
        wls = (N.MoeWeightList * L)(*[lw._wl for lw in layers])
        routers = (C.c_void_p * L)(*[w.data_ptr() for w in w_router])
        biases = None
        if bias is not None:
            biases = (C.c_void_p * L)(*[0 if b is None else b.data_ptr() for b in bias])
        self._arrays = [wls, routers, biases]
        self.cfg = cfg
        self.num_layers = L
        h = C.c_void_p()
        N.check(N.lib().moe_stack_create(C.byref(cfg), L, wls, routers, biases, C.byref(h)),
                "moe_stack_create")
        self.handle = h.value

    def close(self):
        if getattr(self, "handle", None):
            N.lib().moe_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _ws(ws, cfg, op, device):
    return ws if ws is not None else Workspace(cfg, op, device)


def moe_route(cfg: MoeConfig, x, w_router, bias=None, *, return_logits=False, ws=None,
              stream=None):
    """Router logits + top-k + gate weights.  Returns (topk_ids int32 [T,k],
    topk_w fp32 [T,k], logits fp32 [T,E] or None)."""
    dev = x.device
    _need(x, "x", torch.bfloat16, (cfg.T, cfg.H), dev)
    _need(w_router, "w_router", torch.bfloat16, (cfg.E, cfg.H), dev)
    if bias is not None:
        _need(bias, "bias", torch.float32, (cfg.E,), dev)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
    w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev) if return_logits else None
    ws = _ws(ws, cfg, "route", dev)
    N.check(N.lib().moe_route(C.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(ids),
                              _ptr(w), _ptr(logits), ws.ptr, ws.nbytes, _stream(stream)),
            "moe_route")
    return ids, w, logits


def moe_permute(cfg: MoeConfig, topk_ids, topk_w=None, x=None, *, ws=None, stream=None):
    """Histogram + permutation.  Returns a dict with expert_counts, expert_offsets,
    perm_token, inv_row, row_weight (if topk_w), x_perm (if x) and
    x_perm_scales (fp8)."""
    dev = topk_ids.device
    T, k, E, H = cfg.T, cfg.k, cfg.E, cfg.H
    R = T * k
    _need(topk_ids, "topk_ids", torch.int32, (T, k), dev)
    if topk_w is not None:
        _need(topk_w, "topk_w", torch.float32, (T, k), dev)
    fp8 = cfg.wtype == N.MOE_DTYPE_FP8_E4M3
    o = {"expert_counts": torch.empty(E, dtype=torch.int32, device=dev),
         "expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "perm_token": torch.empty(R, dtype=torch.int32, device=dev),
         "inv_row": torch.empty(T, k, dtype=torch.int32, device=dev),
         "row_weight": torch.empty(R, dtype=torch.float32, device=dev) if topk_w is not None else None,
         "x_perm": None, "x_perm_scales": None}
    if x is not None:
        _need(x, "x", torch.bfloat16, (T, H), dev)
        o["x_perm"] = torch.empty(R, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
        if fp8:
            o["x_perm_scales"] = torch.empty(R, H // 128, dtype=torch.float32, device=dev)
    ws = _ws(ws, cfg, "permute", dev)
    N.check(N.lib().moe_permute(C.byref(cfg), _ptr(topk_ids), _ptr(topk_w), _ptr(x),
                                _ptr(o["expert_counts"]), _ptr(o["expert_offsets"]),
                                _ptr(o["perm_token"]), _ptr(o["inv_row"]), _ptr(o["row_weight"]),
                                _ptr(o["x_perm"]), _ptr(o["x_perm_scales"]), ws.ptr, ws.nbytes,
                                _stream(stream)), "moe_permute")
    return o


def moe_permute_noalloc(cfg: MoeConfig, topk_ids, topk_w=None, x=None, *, device_status=None,
                        stream=None):
    """moe_permute for callers that cannot allocate device scratch: the library's
    fixed scratch array replaces the workspace (E * ceil(T/64) <= 262144).  The
    outputs here are still allocated by torch for convenience; a caller that
    cannot allocate passes its own buffers to the C entry point directly.
    device_status: optional int32 [1] device tensor that receives the status bits."""
    dev = topk_ids.device
    T, k, E, H = cfg.T, cfg.k, cfg.E, cfg.H
    R = T * k
    _need(topk_ids, "topk_ids", torch.int32, (T, k), dev)
    if topk_w is not None:
        _need(topk_w, "topk_w", torch.float32, (T, k), dev)
    fp8 = cfg.wtype == N.MOE_DTYPE_FP8_E4M3
    o = {"expert_counts": torch.empty(E, dtype=torch.int32, device=dev),
         "expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "perm_token": torch.empty(R, dtype=torch.int32, device=dev),
         "inv_row": torch.empty(T, k, dtype=torch.int32, device=dev),
         "row_weight": torch.empty(R, dtype=torch.float32, device=dev) if topk_w is not None else None,
         "x_perm": None, "x_perm_scales": None}
    if x is not None:
        _need(x, "x", torch.bfloat16, (T, H), dev)
        o["x_perm"] = torch.empty(R, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
        if fp8:
            o["x_perm_scales"] = torch.empty(R, H // 128, dtype=torch.float32, device=dev)
    N.check(N.lib().moe_permute_noalloc(C.byref(cfg), _ptr(topk_ids), _ptr(topk_w), _ptr(x),
                                        _ptr(o["expert_counts"]), _ptr(o["expert_offsets"]),
                                        _ptr(o["perm_token"]), _ptr(o["inv_row"]),
                                        _ptr(o["row_weight"]), _ptr(o["x_perm"]),
                                        _ptr(o["x_perm_scales"]), _ptr(device_status),
                                        _stream(stream)), "moe_permute_noalloc")
    return o


def moe_grouped_ffn(cfg: MoeConfig, weights: ExpertWeights, x_perm, expert_offsets,
                    row_weight=None, x_shared=None, *, x_perm_scales=None,
                    x_shared_scales=None, ws=None, stream=None):
    """Grouped SwiGLU experts over the permuted rows (+ the shared expert on
    x_shared).  Returns (y_perm fp32 [T*k,H], shared_out fp32 [T,H] or None)."""
    dev = x_perm.device
    T, k, H = cfg.T, cfg.k, cfg.H
    R = T * k
    fp8 = cfg.wtype == N.MOE_DTYPE_FP8_E4M3
    _need(x_perm, "x_perm", torch.uint8 if fp8 else torch.bfloat16, (R, H), dev)
    _need(expert_offsets, "expert_offsets", torch.int32, (cfg.E + 1,), dev)
    if row_weight is not None:
        _need(row_weight, "row_weight", torch.float32, (R,), dev)
    y = torch.empty(R, H, dtype=torch.float32, device=dev)
    s = None
    if x_shared is not None and cfg.I_shared > 0:
        _need(x_shared, "x_shared", torch.uint8 if fp8 else torch.bfloat16, (T, H), dev)
        s = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = _ws(ws, cfg, "grouped_ffn", dev)
    N.check(N.lib().moe_grouped_ffn(C.byref(cfg), weights.handle, _ptr(x_perm),
                                    _ptr(x_perm_scales), _ptr(expert_offsets), _ptr(row_weight),
                                    _ptr(x_shared), _ptr(x_shared_scales), _ptr(y), _ptr(s),
                                    ws.ptr, ws.nbytes, _stream(stream)), "moe_grouped_ffn")
    return y, s


def moe_nvfp4_rows(cfg: MoeConfig) -> tuple[int, int]:
    """(padded_rows, padded_tokens) of the NVFP4 step buffers of a layer."""
    r, t = C.c_int64(0), C.c_int64(0)
    N.check(N.lib().moe_nvfp4_rows(C.byref(cfg), C.byref(r), C.byref(t)), "moe_nvfp4_rows")
    return int(r.value), int(t.value)


def moe_permute_nvfp4(cfg: MoeConfig, weights, topk_ids, topk_w, x, *, shared=True, ws=None,
                      stream=None):
    """Histogram + permutation of an NVFP4 layer: the moe_permute outputs plus
    pad_offsets, x_perm (E2M1 codes over the 128-row-padded expert segments),
    x_perm_sf (their MMA-layout scales) and, with ``shared``, the token-order
    copy x_tok / x_tok_sf for the shared expert."""
    dev = topk_ids.device
    T, k, E, H = cfg.T, cfg.k, cfg.E, cfg.H
    R = T * k
    Rp, Tp = moe_nvfp4_rows(cfg)
    _need(topk_ids, "topk_ids", torch.int32, (T, k), dev)
    _need(topk_w, "topk_w", torch.float32, (T, k), dev)
    _need(x, "x", torch.bfloat16, (T, H), dev)
    sh = shared and cfg.I_shared > 0
    o = {"expert_counts": torch.empty(E, dtype=torch.int32, device=dev),
         "expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "pad_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "perm_token": torch.empty(R, dtype=torch.int32, device=dev),
         "inv_row": torch.empty(T, k, dtype=torch.int32, device=dev),
         "row_weight": torch.empty(R, dtype=torch.float32, device=dev),
         "x_perm": torch.empty(Rp, H // 2, dtype=torch.uint8, device=dev),
         "x_perm_sf": torch.empty(Rp * H // 16, dtype=torch.uint8, device=dev),
         "x_tok": torch.empty(Tp, H // 2, dtype=torch.uint8, device=dev) if sh else None,
         "x_tok_sf": torch.empty(Tp * H // 16, dtype=torch.uint8, device=dev) if sh else None}
    ws = _ws(ws, cfg, "permute", dev)
    N.check(N.lib().moe_permute_nvfp4(
        C.byref(cfg), weights.handle, _ptr(topk_ids), _ptr(topk_w), _ptr(x),
        _ptr(o["expert_counts"]), _ptr(o["expert_offsets"]), _ptr(o["pad_offsets"]),
        _ptr(o["perm_token"]), _ptr(o["inv_row"]), _ptr(o["row_weight"]), _ptr(o["x_perm"]),
        _ptr(o["x_perm_sf"]), _ptr(o["x_tok"]), _ptr(o["x_tok_sf"]), ws.ptr, ws.nbytes,
        _stream(stream)), "moe_permute_nvfp4")
    return o


def moe_grouped_ffn_nvfp4(cfg: MoeConfig, weights, p, row_weight=None, *, shared=True, ws=None,
                          stream=None):
    """Grouped SwiGLU experts of an NVFP4 layer on the outputs ``p`` of
    moe_permute_nvfp4.  Returns (y_perm fp32 [T*k,H], shared_out fp32 [T,H] or None)."""
    dev = p["x_perm"].device
    T, k, H = cfg.T, cfg.k, cfg.H
    if row_weight is not None:
        _need(row_weight, "row_weight", torch.float32, (T * k,), dev)
    y = torch.empty(T * k, H, dtype=torch.float32, device=dev)
    s = None
    if shared and cfg.I_shared > 0 and p.get("x_tok") is not None:
        s = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = _ws(ws, cfg, "grouped_ffn", dev)
    N.check(N.lib().moe_grouped_ffn_nvfp4(
        C.byref(cfg), weights.handle, _ptr(p["x_perm"]), _ptr(p["x_perm_sf"]),
        _ptr(p["expert_offsets"]), _ptr(p["pad_offsets"]), _ptr(row_weight),
        _ptr(p["x_tok"]) if s is not None else None,
        _ptr(p["x_tok_sf"]) if s is not None else None, _ptr(y), _ptr(s), ws.ptr, ws.nbytes,
        _stream(stream)), "moe_grouped_ffn_nvfp4")
    return y, s


def moe_combine(cfg: MoeConfig, y_perm, inv_row, shared_out=None, *, ws=None, stream=None):
    """out[t] = sum_j y_perm[inv_row[t,j]] (+ shared_out[t]) -> bf16 [T,H]; y_perm and
    shared_out are fp32."""
    dev = y_perm.device
    T, k, H = cfg.T, cfg.k, cfg.H
    _need(y_perm, "y_perm", torch.float32, (T * k, H), dev)
    _need(inv_row, "inv_row", torch.int32, (T, k), dev)
    if shared_out is not None:
        _need(shared_out, "shared_out", torch.float32, (T, H), dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = _ws(ws, cfg, "combine", dev)
    N.check(N.lib().moe_combine(C.byref(cfg), _ptr(y_perm), _ptr(inv_row), _ptr(shared_out),
                                _ptr(out), ws.ptr, ws.nbytes, _stream(stream)), "moe_combine")
    return out


def moe_forward(cfg: MoeConfig, weights: ExpertWeights, x, w_router, bias=None, *, out=None,
                return_routing=False, fused_dispatch=False, ws=None, stream=None):
    """The whole layer.  Returns out bf16 [T,H] (and (topk_ids, topk_w) when
    return_routing).  fused_dispatch: GEMM1 gathers its rows from x instead of
    a permuted copy (moe_forward_ex with MOE_FORWARD_FUSED_DISPATCH)."""
    dev = x.device
    _need(x, "x", torch.bfloat16, (cfg.T, cfg.H), dev)
    _need(w_router, "w_router", torch.bfloat16, (cfg.E, cfg.H), dev)
    if bias is not None:
        _need(bias, "bias", torch.float32, (cfg.E,), dev)
    if out is None:
        out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    else:
        _need(out, "out", torch.bfloat16, (cfg.T, cfg.H), dev)
    ids = w = None
    if return_routing:
        ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
        w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    ws = _ws(ws, cfg, "forward", dev)
    flags = N.MOE_FORWARD_FUSED_DISPATCH if fused_dispatch else 0
    N.check(N.lib().moe_forward_ex(C.byref(cfg), weights.handle, _ptr(x), _ptr(w_router),
                                   _ptr(bias), _ptr(out), _ptr(ids), _ptr(w), flags, ws.ptr,
                                   ws.nbytes, _stream(stream)), "moe_forward_ex")
    return (out, ids, w) if return_routing else out


def moe_forward_stack(cfg: MoeConfig, stack: LayerStack, layer, x, *, out=None,
                      return_routing=False, ws=None, stream=None):
    """moe_forward on layer ``layer`` (a device int32 tensor of one element, read
    when the kernels run) of a LayerStack.  Returns out bf16 [T,H] (and (topk_ids,
    topk_w) when return_routing)."""
    dev = x.device
    _need(x, "x", torch.bfloat16, (cfg.T, cfg.H), dev)
    if layer.dtype != torch.int32 or layer.numel() != 1 or layer.device != dev:
        raise ValueError("layer must be a one-element int32 tensor on the device of x")
    if out is None:
        out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    else:
        _need(out, "out", torch.bfloat16, (cfg.T, cfg.H), dev)
    ids = w = None
    if return_routing:
        ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
        w = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    ws = _ws(ws, cfg, "forward", dev)
    N.check(N.lib().moe_forward_stack(C.byref(cfg), stack.handle, _ptr(layer), _ptr(x),
                                      _ptr(out), _ptr(ids), _ptr(w), ws.ptr, ws.nbytes,
                                      _stream(stream)), "moe_forward_stack")
    return (out, ids, w) if return_routing else out


def moe_quantize_weight_fp8(w, stream=None):
    """fp32 [N,K] -> (e4m3 codes uint8 [N,K], fp32 scales [N/128, K/128])."""
    Nr, K = w.shape
    _need(w, "w", torch.float32, (Nr, K), w.device)
    q = torch.empty(Nr, K, dtype=torch.uint8, device=w.device)
    s = torch.empty(Nr // 128, K // 128, dtype=torch.float32, device=w.device)
    N.check(N.lib().moe_quantize_weight_fp8(_ptr(w), Nr, K, _ptr(q), _ptr(s), _stream(stream)),
            "moe_quantize_weight_fp8")
    return q, s


def moe_quantize_act_fp8(x, stream=None):
    """bf16 [M,K] -> (e4m3 codes uint8 [M,K], fp32 scales [M, K/128])."""
    M, K = x.shape
    _need(x, "x", torch.bfloat16, (M, K), x.device)
    q = torch.empty(M, K, dtype=torch.uint8, device=x.device)
    s = torch.empty(M, K // 128, dtype=torch.float32, device=x.device)
    N.check(N.lib().moe_quantize_act_fp8(_ptr(x), M, K, _ptr(q), _ptr(s), _stream(stream)),
            "moe_quantize_act_fp8")
    return q, s


def moe_quantize_weight_nvfp4(w, w2=None, tensor_scale=None, stream=None):
    """NVFP4 weights (moe_quantize_weight_nvfp4): bf16 [N, K] (w2: a second
    [N, K] matrix stacked with w, rows interleaved in 128-row blocks) ->
    (codes uint8 [rows, K/2], MMA-layout scales uint8 [rows*K/16], tensor scale
    float32 [1], or written into ``tensor_scale`` (a float32 view of one element))."""
    Nr, K = w.shape
    _need(w, "w", torch.bfloat16, (Nr, K), None)
    if w2 is not None:
        _need(w2, "w2", torch.bfloat16, (Nr, K), w.device)
    rows = 2 * Nr if w2 is not None else Nr
    codes = torch.empty(rows, K // 2, dtype=torch.uint8, device=w.device)
    sf = torch.empty(rows * K // 16, dtype=torch.uint8, device=w.device)
    ts = tensor_scale if tensor_scale is not None else torch.empty(1, dtype=torch.float32,
                                                                    device=w.device)
    N.check(N.lib().moe_quantize_weight_nvfp4(w.data_ptr(), _ptr(w2), Nr, K, codes.data_ptr(),
                                              sf.data_ptr(), ts.data_ptr(), _stream(stream)),
            "moe_quantize_weight_nvfp4")
    return codes, sf, ts


def moe_quantize_act_nvfp4(x, g, stream=None):
    """bf16 [M, K] -> (codes uint8 [M, K/2], e4m3 scale codes uint8 [M, K/16]) with
    the static tensor scale g."""
    M, K = x.shape
    _need(x, "x", torch.bfloat16, (M, K), None)
    codes = torch.empty(M, K // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(M, K // 16, dtype=torch.uint8, device=x.device)
    N.check(N.lib().moe_quantize_act_nvfp4(x.data_ptr(), M, K, float(g), codes.data_ptr(),
                                           sf.data_ptr(), _stream(stream)),
            "moe_quantize_act_nvfp4")
    return codes, sf


def quantize_experts_nvfp4(cfg: MoeConfig, gate, up, down, shared=None, *, input_scale,
                           hidden_scale, stream=None) -> Nvfp4ExpertWeights:
    """Quantise bf16 expert weights (lists of [I, H] gate/up and [H, I] down
    tensors, and the shared expert's triple) to NVFP4 on the GPU and build the
    layer's weight table.  The quantised tensors are owned by the result."""
    E = cfg.E
    dev = gate[0].device
    gu_ts = torch.empty(E, dtype=torch.float32, device=dev)
    d_ts = torch.empty(E, dtype=torch.float32, device=dev)
    gu, dn, gu_sf, dn_sf = [], [], [], []
    for e in range(E):
        c, s, _ = moe_quantize_weight_nvfp4(gate[e], up[e], gu_ts[e:e + 1], stream)
        gu.append(c)
        gu_sf.append(s)
        c, s, _ = moe_quantize_weight_nvfp4(down[e], None, d_ts[e:e + 1], stream)
        dn.append(c)
        dn_sf.append(s)
    sh = None
    if shared is not None:
        sg, su, sd = shared
        sts = torch.empty(2, dtype=torch.float32, device=dev)
        c1, s1, _ = moe_quantize_weight_nvfp4(sg, su, sts[0:1], stream)
        c2, s2, _ = moe_quantize_weight_nvfp4(sd, None, sts[1:2], stream)
        sh = (c1, c2, s1, s2, sts)
    return Nvfp4ExpertWeights(cfg, gu, dn, gu_sf, dn_sf, gu_ts, d_ts, input_scale, hidden_scale,
                              shared=sh)
