"""Thin ctypes binding of libmoe (include/moe.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmoe.so.  PyTorch supplies device memory, streams and events.  There is no
fallback: if libmoe.so is missing or a call fails, an exception is raised.
Function names follow the C ABI.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(5)
MOE_F32, MOE_BF16 = 0, 1
MOE_DEVERR_BAD_EXPERT_ID, MOE_DEVERR_BAD_ROW_INDEX, MOE_DEVERR_BAD_OFFSETS, MOE_DEVERR_TIMEOUT = 1, 2, 4, 8
MOE_WS_HEADER_BYTES = 256
MOE_NUM_STAGES = 8
WS_FIELDS = ["logits", "topk_ids", "topk_w", "tokens_per_expert", "expert_offsets", "expanded_row_idx",
             "expanded_x", "h_routed", "h_shared", "y_routed", "y_shared", "x_in", "out", "xq", "xq_scales",
             "expanded_xq", "expanded_xq_scales", "hq", "hq_scales", "hq_shared", "hq_shared_scales"]
WS_FIELDS_EP = ["x_sorted", "gathered_ids_unsort", "recv_start", "expert_offsets"]
MOE_WEIGHTS_NATIVE, MOE_WEIGHTS_FP8, MOE_WEIGHTS_FP8_POW2 = 0, 1, 2
WEIGHT_FORMATS = {"native": MOE_WEIGHTS_NATIVE, "fp8": MOE_WEIGHTS_FP8, "fp8_pow2": MOE_WEIGHTS_FP8_POW2}
MOE_LAYOUT_ROWS, MOE_LAYOUT_TILED = 0, 1
WEIGHT_LAYOUTS = {"rows": MOE_LAYOUT_ROWS, "tiled": MOE_LAYOUT_TILED}

# The exported entry points (name -> (restype, argtypes)).
P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t


class LayerDesc(ctypes.Structure):
    _fields_ = [("T", I32), ("H", I32), ("E", I32), ("k", I32), ("I", I32), ("S", I32), ("dtype", I32),
                ("renormalize", I32), ("w_router", P), ("expert_bias", P), ("w13", P), ("w2", P),
                ("w13_shared", P), ("w2_shared", P), ("n_group", I32), ("topk_group", I32), ("group_rule", I32),
                ("weight_format", I32), ("w13_scales", P), ("w2_scales", P), ("w13_shared_scales", P),
                ("w2_shared_scales", P), ("weight_layout", I32)]


_DP = ctypes.POINTER(LayerDesc)
SIGNATURES = {
    "moe_abi_version": (I32, []),
    "moe_status_string": (ctypes.c_char_p, [I32]),
    "moe_kernel_launch_count": (ctypes.c_uint64, []),
    "moe_check_device_status": (I32, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_diag_bounded_wait": (I32, [ctypes.c_uint64, P, P, P]),
    "moe_gate_logits": (I32, [P, P, I32, I32, I32, I32, P, P]),
    "moe_route_topk": (I32, [P, P, I32, I32, I32, I32, P, P, P]),
    "moe_route_topk_grouped": (I32, [P, P, I32, I32, I32, I32, I32, I32, I32, P, P, P]),
    "moe_init_routing_workspace_bytes": (SZ, [I32, I32, I32]),
    "moe_init_routing": (I32, [P, I32, P, I32, I32, I32, I32, P, P, P, P, P, SZ, P]),
    "moe_init_routing_noalloc": (I32, [P, I32, P, I32, I32, I32, I32, P, P, P, P, P]),
    "moe_w13_packed_bytes": (SZ, [I32, I32, I32, I32]),
    "moe_pack_w13": (I32, [P, P, I32, I32, I32, I32, P, P]),
    "moe_grouped_ffn_workspace_bytes": (SZ, [I32, I32, I32]),
    "moe_grouped_ffn": (I32, [P, I32, P, I32, I32, I32, I32, P, P, P, P, SZ, P]),
    "moe_grouped_ffn_tiled": (I32, [P, I32, P, I32, I32, I32, I32, P, P, P, P, SZ, P]),
    "moe_tiled_weight_bytes": (SZ, [I32, I32, I32]),
    "moe_tile_weights": (I32, [P, I32, I32, I32, P, P]),
    "moe_finalize_routing": (I32, [P, I64, P, P, P, I32, I32, I32, I32, P, P, P]),
    "moe_re_routing_workspace_bytes": (SZ, [I32, I32]),
    "moe_re_routing": (I32, [P, I32, P, I32, I32, I32, I32, P, P, P, P, P, SZ, P]),
    "moe_unsort_rows": (I32, [P, I32, P, I32, I32, P, P, P]),
    "moe_layer_workspace_bytes_ep": (SZ, [_DP, I32]),
    "moe_layer_forward_ep": (I32, [_DP, I32, P, P, P, SZ, P]),
    "moe_layer_workspace_field_ep": (I32, [_DP, I32, I32, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]),
    "moe_quantize_rows_fp8": (I32, [P, I32, I64, I32, P, P, I32, P]),
    "moe_quantize_weights_fp8": (I32, [P, I32, I32, I32, I32, P, P, P]),
    "moe_quantize_rows_fp8_pow2": (I32, [P, I32, I64, I32, P, P, I32, P]),
    "moe_quantize_weights_fp8_pow2": (I32, [P, I32, I32, I32, I32, P, P, P]),
    "moe_grouped_ffn_fp8_workspace_bytes": (SZ, [I32, I32]),
    "moe_grouped_ffn_fp8": (I32, [P, P, I32, P, I32, I32, I32, I32, P, P, P, P, P, P, SZ, P]),
    "moe_grouped_ffn_fp8_pow2": (I32, [P, P, I32, P, I32, I32, I32, I32, P, P, P, P, P, P, SZ, P]),
    "moe_stage_name": (ctypes.c_char_p, [I32]),
    "moe_layer_workspace_bytes": (SZ, [_DP]),
    "moe_layer_workspace_field": (I32, [_DP, I32, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]),
    "moe_layer_forward": (I32, [_DP, P, P, P, SZ, P]),
    "moe_layer_forward_timed": (I32, [_DP, P, P, P, SZ, P, ctypes.POINTER(P)]),
    "moe_layer_shared_expert_sms": (I32, [_DP]),
    "moe_layer_forward_host": (I32, [_DP, P, P, P, SZ, P]),
}

_lock = threading.Lock()
_lib = None


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = lib().moe_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what} failed: {name}")


def lib():
    """Load libmoe.so (built by __graft_entry__.build() or python -m ...build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libmoe.so not found at {LIB_PATH}: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _check(st: int, what: str):
    if st != MOE_OK:
        raise MoEError(st, what)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensors expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensors expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise TypeError(f"float32 or bfloat16 expected, got {t.dtype}")


def launch_count() -> int:
    return int(lib().moe_kernel_launch_count())


def moe_check_device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and return the status word of a workspace (0 = no device error)."""
    word = ctypes.c_uint32(0)
    st = lib().moe_check_device_status(_ptr(ws), _stream(stream), ctypes.byref(word))
    if st not in (MOE_OK, MOE_ERR_DEVICE):
        _check(st, "moe_check_device_status")
    return int(word.value)


def moe_gate_logits(x: torch.Tensor, w_router: torch.Tensor, stream=None) -> torch.Tensor:
    T, H = x.shape
    E = w_router.shape[0]
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _check(lib().moe_gate_logits(_ptr(x), _ptr(w_router), _dt(x), T, H, E, _ptr(logits), _stream(stream)),
           "moe_gate_logits")
    return logits


def moe_route_topk(logits: torch.Tensor, k: int, renormalize: bool = True, expert_bias=None, stream=None):
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topk(_ptr(logits), _ptr(expert_bias), T, E, k, int(bool(renormalize)), _ptr(ids),
                                _ptr(w), _stream(stream)), "moe_route_topk")
    return ids, w


GROUP_RULES = {"max": 0, "top2_sum": 1}


def moe_route_topk_grouped(logits: torch.Tensor, k: int, n_group: int, topk_group: int, rule: str = "max",
                           renormalize: bool = True, expert_bias=None, stream=None):
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route_topk_grouped(_ptr(logits), _ptr(expert_bias), T, E, k, n_group, topk_group,
                                        GROUP_RULES[rule], int(bool(renormalize)), _ptr(ids), _ptr(w),
                                        _stream(stream)), "moe_route_topk_grouped")
    return ids, w


def moe_init_routing(x: torch.Tensor, topk_ids: torch.Tensor, E: int, stream=None, ws=None) -> dict:
    T, H = x.shape
    k = topk_ids.shape[1]
    dev = x.device
    need = lib().moe_init_routing_workspace_bytes(T, E, k)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out = dict(expanded_x=torch.empty((T * k, H), dtype=x.dtype, device=dev),
               expanded_row_idx=torch.empty(T * k, dtype=torch.int32, device=dev),
               tokens_per_expert=torch.empty(E, dtype=torch.int32, device=dev),
               expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev), ws=ws)
    _check(lib().moe_init_routing(_ptr(x), _dt(x), _ptr(topk_ids), T, H, E, k, _ptr(out["expanded_x"]),
                                  _ptr(out["expanded_row_idx"]), _ptr(out["tokens_per_expert"]),
                                  _ptr(out["expert_offsets"]), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_init_routing")
    return out


def moe_init_routing_noalloc(x: torch.Tensor, topk_ids: torch.Tensor, E: int, stream=None) -> dict:
    """moe_init_routing without a workspace: the library's fixed device array is the
    scratch (for callers that cannot allocate; calls must not overlap on the GPU)."""
    T, H = x.shape
    k = topk_ids.shape[1]
    dev = x.device
    out = dict(expanded_x=torch.empty((T * k, H), dtype=x.dtype, device=dev),
               expanded_row_idx=torch.empty(T * k, dtype=torch.int32, device=dev),
               tokens_per_expert=torch.empty(E, dtype=torch.int32, device=dev),
               expert_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev))
    _check(lib().moe_init_routing_noalloc(_ptr(x), _dt(x), _ptr(topk_ids), T, H, E, k, _ptr(out["expanded_x"]),
                                          _ptr(out["expanded_row_idx"]), _ptr(out["tokens_per_expert"]),
                                          _ptr(out["expert_offsets"]), _stream(stream)),
           "moe_init_routing_noalloc")
    return out


def moe_pack_w13(w_gate: torch.Tensor, w_up: torch.Tensor, stream=None) -> torch.Tensor:
    """w_gate, w_up [E,I,H] (or [I,H] for one expert) -> packed [E, 2*Ip, H]."""
    if w_gate.dim() == 2:
        w_gate, w_up = w_gate.unsqueeze(0), w_up.unsqueeze(0)
    E, I, H = w_gate.shape
    dt = _dt(w_gate)
    nbytes = lib().moe_w13_packed_bytes(dt, E, H, I)
    packed = torch.empty(nbytes // w_gate.element_size(), dtype=w_gate.dtype, device=w_gate.device)
    _check(lib().moe_pack_w13(_ptr(w_gate), _ptr(w_up), dt, E, H, I, _ptr(packed), _stream(stream)),
           "moe_pack_w13")
    return packed.view(E, -1, H)


def moe_grouped_ffn(a: torch.Tensor, expert_offsets, E: int, I: int, w13_packed: torch.Tensor,
                    w2: torch.Tensor, y: torch.Tensor | None = None, ws=None, stream=None, tiled: bool = False):
    """tiled: w13_packed and w2 are moe_tile_weights outputs (moe_grouped_ffn_tiled)."""
    rows, H = a.shape
    dt = _dt(a)
    need = lib().moe_grouped_ffn_workspace_bytes(dt, rows, I)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=a.device)
    if y is None:
        y = torch.zeros((rows, H), dtype=a.dtype, device=a.device)
    name = "moe_grouped_ffn_tiled" if tiled else "moe_grouped_ffn"
    _check(getattr(lib(), name)(_ptr(a), dt, _ptr(expert_offsets), E, rows, H, I, _ptr(w13_packed), _ptr(w2),
                                _ptr(y), _ptr(ws), ws.numel(), _stream(stream)), name)
    return y, ws


def moe_tile_weights(w: torch.Tensor, stream=None) -> torch.Tensor:
    """w [G, n_rows, K] (or [n_rows, K]) -> the tiled layout as a flat uint8 tensor."""
    if w.dim() == 2:
        w = w.unsqueeze(0)
    w = w.contiguous()
    G, n, k = w.shape
    row_bytes = k * w.element_size()
    nbytes = lib().moe_tiled_weight_bytes(G, n, row_bytes)
    if nbytes == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_tiled_weight_bytes")
    out = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    _check(lib().moe_tile_weights(_ptr(w), G, n, row_bytes, _ptr(out), _stream(stream)), "moe_tile_weights")
    return out


def moe_finalize_routing(y: torch.Tensor, topk_w: torch.Tensor, expanded_row_idx: torch.Tensor,
                         skip: torch.Tensor | None = None, ws=None, stream=None) -> torch.Tensor:
    T, k = topk_w.shape
    H = y.shape[1]
    out = torch.empty((T, H), dtype=y.dtype, device=y.device)
    _check(lib().moe_finalize_routing(_ptr(y), y.shape[0], _ptr(skip), _ptr(topk_w), _ptr(expanded_row_idx),
                                      _dt(y), T, H, k, _ptr(out), _ptr(ws), _stream(stream)),
           "moe_finalize_routing")
    return out


def moe_re_routing(x_recv: torch.Tensor, counts: torch.Tensor, stream=None) -> dict:
    """Second routing of Double-Routing; counts [W, E_local] int32 on the device."""
    N, H = x_recv.shape
    W, El = counts.shape
    dev = x_recv.device
    ws = torch.empty(lib().moe_re_routing_workspace_bytes(W, El), dtype=torch.uint8, device=dev)
    out = dict(x_sorted=torch.empty_like(x_recv), gathered_ids_unsort=torch.empty(N, dtype=torch.int32, device=dev),
               tokens_per_local_expert=torch.empty(El, dtype=torch.int32, device=dev),
               local_offsets=torch.empty(El + 1, dtype=torch.int32, device=dev), ws=ws)
    _check(lib().moe_re_routing(_ptr(x_recv), _dt(x_recv), _ptr(counts.contiguous()), W, El, N, H,
                                _ptr(out["x_sorted"]), _ptr(out["gathered_ids_unsort"]),
                                _ptr(out["tokens_per_local_expert"]), _ptr(out["local_offsets"]), _ptr(ws),
                                ws.numel(), _stream(stream)), "moe_re_routing")
    return out


def moe_unsort_rows(y_sorted: torch.Tensor, gathered_ids_unsort: torch.Tensor, ws=None, stream=None):
    N, H = y_sorted.shape
    out = torch.empty_like(y_sorted)
    _check(lib().moe_unsort_rows(_ptr(y_sorted), _dt(y_sorted), _ptr(gathered_ids_unsort), N, H, _ptr(out),
                                 _ptr(ws), _stream(stream)), "moe_unsort_rows")
    return out


def scale_ld(cols: int) -> int:
    """Row stride (floats) of the 1x128 activation scales the layer uses."""
    return -(-(-(-cols // 128)) // 4) * 4


def moe_quantize_rows_fp8(a: torch.Tensor, ld_scales: int | None = None, stream=None, pow2: bool = False):
    """1x128 blocks; pow2 selects the power-of-two scale format (moe_quantize_rows_fp8_pow2)."""
    rows, cols = a.shape
    ld = ld_scales or -(-cols // 128)
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=a.device)
    scales = torch.empty((rows, ld), dtype=torch.float32, device=a.device)
    name = "moe_quantize_rows_fp8_pow2" if pow2 else "moe_quantize_rows_fp8"
    _check(getattr(lib(), name)(_ptr(a), _dt(a), rows, cols, _ptr(codes), _ptr(scales), ld, _stream(stream)), name)
    return codes, scales


def moe_quantize_weights_fp8(w: torch.Tensor, stream=None, pow2: bool = False):
    """w [G, n_out, k_in] (or [n_out, k_in]) -> (codes, scales [G, n/128, k/128]); pow2 as above."""
    if w.dim() == 2:
        w = w.unsqueeze(0)
    G, n, k = w.shape
    codes = torch.empty((G, n, k), dtype=torch.uint8, device=w.device)
    scales = torch.empty((G, -(-n // 128), -(-k // 128)), dtype=torch.float32, device=w.device)
    name = "moe_quantize_weights_fp8_pow2" if pow2 else "moe_quantize_weights_fp8"
    _check(getattr(lib(), name)(_ptr(w.contiguous()), _dt(w), G, n, k, _ptr(codes), _ptr(scales), _stream(stream)),
           name)
    return codes, scales


def moe_grouped_ffn_fp8(aq, a_scales, expert_offsets, E: int, I: int, w13q, w13s, w2q, w2s, stream=None,
                        pow2: bool = False):
    """pow2: every scale a power of two, products on block-scaled MMAs (moe_grouped_ffn_fp8_pow2)."""
    rows, H = aq.shape
    ws = torch.empty(lib().moe_grouped_ffn_fp8_workspace_bytes(rows, I), dtype=torch.uint8, device=aq.device)
    y = torch.zeros((rows, H), dtype=torch.bfloat16, device=aq.device)
    name = "moe_grouped_ffn_fp8_pow2" if pow2 else "moe_grouped_ffn_fp8"
    _check(getattr(lib(), name)(_ptr(aq), _ptr(a_scales), a_scales.shape[1], _ptr(expert_offsets), E, rows, H, I,
                                _ptr(w13q), _ptr(w13s), _ptr(w2q), _ptr(w2s), _ptr(y), _ptr(ws), ws.numel(),
                                _stream(stream)), name)
    return y, ws


def stage_names() -> list[str]:
    return [lib().moe_stage_name(i).decode() for i in range(MOE_NUM_STAGES)]


class MoELayer:
    """A MoE layer whose weights live on the device, with its workspace.

    Weights: w_router [E,H]; w_gate, w_up [E,I,H]; w2 [E,H,I]; shared experts
    s_gate, s_up [S,I,H], s2 [S,H,I] (S may be 0); expert_bias [E] fp32 or None.
    The gate/up weights are packed once (moe_pack_w13)."""

    def __init__(self, *, T: int, k: int, w_router, w_gate, w_up, w2, s_gate=None, s_up=None, s2=None,
                 expert_bias=None, renormalize: bool = True, n_group: int = 1, topk_group: int = 1,
                 group_rule: str = "max", weight_format: str = "native", weight_layout: str | None = None,
                 stream=None):
        E, I, H = w_gate.shape
        S = 0 if s_gate is None else s_gate.shape[0]
        self.T, self.H, self.E, self.k, self.I, self.S = T, H, E, k, I, S
        self.dtype = w_gate.dtype
        self.w_router = w_router.contiguous()
        self.w13 = moe_pack_w13(w_gate.contiguous(), w_up.contiguous(), stream)
        self.w2 = w2.contiguous()
        if S:
            self.w13_shared = moe_pack_w13(s_gate.reshape(S * I, H).contiguous(),
                                           s_up.reshape(S * I, H).contiguous(), stream)
            # [S,H,I] -> [H, S*I]: the shared down projections side by side
            self.w2_shared = s2.permute(1, 0, 2).reshape(H, S * I).contiguous()
        else:
            self.w13_shared = self.w2_shared = None
        self.expert_bias = None if expert_bias is None else expert_bias.to(torch.float32).contiguous()
        self.weight_format = weight_format
        scales = [None] * 4
        if weight_format not in WEIGHT_FORMATS:
            raise ValueError(f"weight_format must be one of {sorted(WEIGHT_FORMATS)}, got {weight_format!r}")
        if weight_format != "native":
            # static 128x128-tile quantisation of the packed gate/up and the down weights
            p2 = weight_format == "fp8_pow2"
            self.w13, s13 = moe_quantize_weights_fp8(self.w13, stream, pow2=p2)
            self.w2, s2_ = moe_quantize_weights_fp8(self.w2, stream, pow2=p2)
            scales[0], scales[1] = s13, s2_
            if S:
                self.w13_shared, ss13 = moe_quantize_weights_fp8(self.w13_shared, stream, pow2=p2)
                self.w2_shared, ss2 = moe_quantize_weights_fp8(self.w2_shared, stream, pow2=p2)
                scales[2], scales[3] = ss13, ss2
        # bf16 expert weights go to the tiled layout (each 256-row x 128-byte weight box one contiguous
        # block of HBM) unless asked otherwise.  FP8 codes stay row-major by default: tiled, the FP8 up
        # projection gains (power-of-two scales: 1271 -> 1238 us at the DeepSeek-V3 prefill shape) but
        # both FP8 down projections lose more (700 -> 741 and 764 -> 806 us).  fp32 layers keep rows.
        if weight_layout is None:
            weight_layout = "tiled" if (self.dtype == torch.bfloat16 and weight_format == "native") else "rows"
        if weight_layout not in WEIGHT_LAYOUTS:
            raise ValueError(f"weight_layout must be one of {sorted(WEIGHT_LAYOUTS)}, got {weight_layout!r}")
        self.weight_layout = weight_layout
        if weight_layout == "tiled":
            self.w13 = moe_tile_weights(self.w13, stream)
            self.w2 = moe_tile_weights(self.w2, stream)
            if S:
                self.w13_shared = moe_tile_weights(self.w13_shared, stream)
                self.w2_shared = moe_tile_weights(self.w2_shared, stream)
        self.scales = scales
        sp = [0 if t is None else t.data_ptr() for t in scales]
        self.desc = LayerDesc(T, H, E, k, I, S, _dt(w_gate), int(bool(renormalize)), self.w_router.data_ptr(),
                              0 if self.expert_bias is None else self.expert_bias.data_ptr(), self.w13.data_ptr(),
                              self.w2.data_ptr(), 0 if S == 0 else self.w13_shared.data_ptr(),
                              0 if S == 0 else self.w2_shared.data_ptr(), n_group, topk_group,
                              GROUP_RULES[group_rule], WEIGHT_FORMATS[weight_format], *sp,
                              WEIGHT_LAYOUTS[weight_layout])
        nbytes = lib().moe_layer_workspace_bytes(ctypes.byref(self.desc))
        if nbytes == 0:
            raise MoEError(MOE_ERR_INVALID_ARG, "moe_layer_workspace_bytes")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=w_gate.device)

    def field(self, name: str, ws: torch.Tensor | None = None) -> torch.Tensor:
        """A view of one intermediate in the workspace (see moe_ws_field); ws: another
        workspace laid out from the same descriptor (forward_ep's), else the layer's."""
        off, nb = SZ(0), SZ(0)
        _check(lib().moe_layer_workspace_field(ctypes.byref(self.desc), WS_FIELDS.index(name), ctypes.byref(off),
                                               ctypes.byref(nb)), "moe_layer_workspace_field")
        raw = (self.ws if ws is None else ws)[off.value:off.value + nb.value]
        T, H, E, k, I, S = self.T, self.H, self.E, self.k, self.I, self.S
        shapes = dict(logits=((T, E), torch.float32), topk_ids=((T, k), torch.int32),
                      topk_w=((T, k), torch.float32), tokens_per_expert=((E,), torch.int32),
                      expert_offsets=((E + 1,), torch.int32), expanded_row_idx=((T * k,), torch.int32),
                      expanded_x=((T * k, H), self.dtype), h_routed=((T * k, I), self.dtype),
                      h_shared=((T, S * I), self.dtype), y_routed=((T * k, H), self.dtype),
                      y_shared=((T, H), self.dtype), x_in=((T, H), self.dtype), out=((T, H), self.dtype),
                      xq=((T, H), torch.uint8), xq_scales=((T, scale_ld(H)), torch.float32),
                      expanded_xq=((T * k, H), torch.uint8), expanded_xq_scales=((T * k, scale_ld(H)), torch.float32),
                      hq=((T * k, I), torch.uint8), hq_scales=((T * k, scale_ld(I)), torch.float32),
                      hq_shared=((T, S * I), torch.uint8), hq_shared_scales=((T, scale_ld(S * I) if S else 0),
                                                                             torch.float32))
        shape, dtype = shapes[name]
        n = 1
        for dim in shape:
            n *= dim
        return raw.view(dtype)[:n].view(shape)  # the logits region also holds the gate's K slices

    def forward(self, x: torch.Tensor, out: torch.Tensor | None = None, stream=None, events=None):
        if out is None:
            out = torch.empty_like(x)
        if events is None:
            st = lib().moe_layer_forward(ctypes.byref(self.desc), _ptr(x), _ptr(out), _ptr(self.ws),
                                         self.ws.numel(), _stream(stream))
        else:
            if len(events) != 2 * MOE_NUM_STAGES:
                raise ValueError(f"{2 * MOE_NUM_STAGES} events expected (start, end per stage; None skips one)")
            for e in events:  # torch creates the CUDA event on its first record
                if e is not None and e.cuda_event == 0:
                    e.record()
            arr = (P * (2 * MOE_NUM_STAGES))(*[ctypes.c_void_p(0 if e is None else e.cuda_event) for e in events])
            st = lib().moe_layer_forward_timed(ctypes.byref(self.desc), _ptr(x), _ptr(out), _ptr(self.ws),
                                               self.ws.numel(), _stream(stream), arr)
        _check(st, "moe_layer_forward")
        return out

    def forward_host(self, x_host: torch.Tensor, out_host: torch.Tensor, stream=None):
        """End to end from host memory (blocks until out_host is written)."""
        if x_host.is_cuda or out_host.is_cuda:
            raise ValueError("host tensors expected")
        st = lib().moe_layer_forward_host(ctypes.byref(self.desc), ctypes.c_void_p(x_host.data_ptr()),
                                          ctypes.c_void_p(out_host.data_ptr()), _ptr(self.ws), self.ws.numel(),
                                          _stream(stream))
        _check(st, "moe_layer_forward_host")
        return out_host

    def forward_ep(self, x: torch.Tensor, W: int, out: torch.Tensor | None = None, stream=None):
        """The layer through Double-Routing with W virtual expert-parallel ranks."""
        if out is None:
            out = torch.empty_like(x)
        need = lib().moe_layer_workspace_bytes_ep(ctypes.byref(self.desc), W)
        if need == 0:
            raise MoEError(MOE_ERR_INVALID_ARG, "moe_layer_workspace_bytes_ep")
        if getattr(self, "ws_ep", None) is None or self.ws_ep.numel() < need:
            self.ws_ep = torch.empty(need, dtype=torch.uint8, device=x.device)
        _check(lib().moe_layer_forward_ep(ctypes.byref(self.desc), W, _ptr(x), _ptr(out), _ptr(self.ws_ep),
                                          self.ws_ep.numel(), _stream(stream)), "moe_layer_forward_ep")
        return out

    def field_ep(self, name: str, W: int) -> torch.Tensor:
        """A view of one intermediate left in the workspace by forward_ep(x, W)
        (see moe_ws_field_ep)."""
        off, nb = SZ(0), SZ(0)
        _check(lib().moe_layer_workspace_field_ep(ctypes.byref(self.desc), W, WS_FIELDS_EP.index(name),
                                                  ctypes.byref(off), ctypes.byref(nb)), "moe_layer_workspace_field_ep")
        raw = self.ws_ep[off.value:off.value + nb.value]
        R = self.T * self.k
        shapes = dict(x_sorted=((R, self.H), self.dtype), gathered_ids_unsort=((R,), torch.int32),
                      recv_start=((W + 1,), torch.int32), expert_offsets=((self.E + 1,), torch.int32))
        shape, dtype = shapes[name]
        return raw.view(dtype).view(shape)

    def shared_expert_sms(self) -> int:
        """SMs the shared experts' GEMMs take beside the routed up projection (0: no split)."""
        return int(lib().moe_layer_shared_expert_sms(ctypes.byref(self.desc)))

    def device_status(self, stream=None) -> int:
        return moe_check_device_status(self.ws, stream)
