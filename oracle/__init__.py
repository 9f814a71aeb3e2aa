"""CPU oracle for the MoE layer hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls it; the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 sums, OpenMP over
tokens/rows).  This module only compiles it with gcc and marshals numpy arrays.
bf16 arrays are passed as their uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_int64
        lib.oracle_num_threads.restype = I
        lib.oracle_set_num_threads.argtypes = [I]
        lib.oracle_round_array.argtypes = [P, I, L, P]
        lib.oracle_gate_logits.argtypes = [P, P, I, I, I, I, P]
        lib.oracle_route_topk.argtypes = [P, P, I, I, I, I, P, P]
        lib.oracle_route_topk_grouped.argtypes = [P, P, I, I, I, I, I, I, I, P, P]
        lib.oracle_init_routing.argtypes = [P, I, I, I, P, I, I, P, P, P, P]
        lib.oracle_init_routing.restype = I
        lib.oracle_expert_ffn_rows.argtypes = [P, I, L, P, P, P, P, I, I, P]
        lib.oracle_re_routing.argtypes = [P, I, P, I, I, I, P, P, P, P]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_rows_fp8.argtypes = [P, I, L, I, P, P, I]
        lib.oracle_quantize_tiles_fp8.argtypes = [P, I, I, I, P, P, I]
        lib.oracle_gemm_fp8.argtypes = [P, P, P, P, I, I, I, P]
        lib.oracle_expert_ffn_rows_fp8.argtypes = [P, P, L, P, P, P, P, P, P, P, I, I, P, I]
        lib.oracle_layer_fp8.argtypes = [P, I, I, I, I, I, I, I, P, P] + [P] * 12 + [P, I, P, P, P, P, I, I, I, I]
        lib.oracle_unsort_rows.argtypes = [P, I, P, L, I, P]
        lib.oracle_finalize_routing.argtypes = [P, I, L, P, P, P, I, I, I, P]
        lib.oracle_layer.argtypes = [P, I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, I,
                                     P, P, P, P, I, I, I]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle arrays are float32 or bf16 bit patterns (uint16), got {a.dtype}")


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def round_to(values: np.ndarray, dt: int) -> np.ndarray:
    """Round fp64 values to the storage dtype (fp32 or bf16, RNE); fp64 out."""
    v = _c(values, np.float64)
    out = np.empty_like(v)
    _load().oracle_round_array(_ptr(v), dt, v.size, _ptr(out))
    return out


def gate_logits(x: np.ndarray, wg: np.ndarray) -> np.ndarray:
    """logits[t,e] = sum_h x[t,h] wg[e,h] in fp64.  x [T,H], wg [E,H]."""
    x, wg = _c(x), _c(wg)
    dt = _dt(x)
    assert _dt(wg) == dt
    T, H = x.shape
    E = wg.shape[0]
    out = np.empty((T, E), np.float64)
    _load().oracle_gate_logits(_ptr(x), _ptr(wg), dt, T, H, E, _ptr(out))
    return out


def route_topk(logits: np.ndarray, k: int, renorm: bool = True, bias: np.ndarray | None = None):
    """Top-k routing on fp32 scores.  Returns (ids int32 [T,k], w fp64 [T,k])."""
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().oracle_route_topk(_ptr(logits), _ptr(bias), T, E, k, int(bool(renorm)), _ptr(ids), _ptr(w))
    return ids, w


def route_topk_grouped(logits: np.ndarray, k: int, n_group: int, topk_group: int, rule: str = "max",
                       renorm: bool = True, bias: np.ndarray | None = None):
    """Group-limited top-k (rule "max" or "top2_sum").  Returns (ids [T,k], w [T,k])."""
    logits = _c(logits, np.float32)
    bias = _c(bias, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().oracle_route_topk_grouped(_ptr(logits), _ptr(bias), T, E, k, n_group, topk_group,
                                      {"max": 0, "top2_sum": 1}[rule], int(bool(renorm)), _ptr(ids), _ptr(w))
    return ids, w


def init_routing(ids: np.ndarray, x: np.ndarray | None, E: int, H: int | None = None):
    """Init-routing.  ids [T,k] int32, x [T,H] (float32 or bf16 bits) or None.

    Returns dict(expanded_x, expanded_row_idx, tokens_per_expert, expert_offsets, bad)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    if x is not None:
        x = _c(x)
        dt, H = _dt(x), x.shape[1]
        ex = np.zeros((T * k, H), x.dtype)
    else:
        dt, H, ex = F32, 0 if H is None else H, None
    idx = np.empty(T * k, np.int32)
    cnt = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    bad = _load().oracle_init_routing(_ptr(ids), T, k, E, _ptr(x), dt, H, _ptr(ex), _ptr(idx),
                                      _ptr(cnt), _ptr(off))
    return dict(expanded_x=ex, expanded_row_idx=idx, tokens_per_expert=cnt, expert_offsets=off,
                bad=bad)


def re_routing(x_recv: np.ndarray, counts: np.ndarray):
    """Second routing of Double-Routing.  counts [W, E_local] (rows from source p for
    local expert e, arrival order p-major).  Returns dict(x_sorted, gathered_ids_unsort,
    tokens_per_local_expert, local_offsets)."""
    x_recv = _c(x_recv)
    counts = _c(counts, np.int32)
    W, El = counts.shape
    N, H = x_recv.shape
    assert counts.sum() == N
    xs = np.zeros_like(x_recv)
    gidx = np.empty(N, np.int32)
    tpl = np.empty(El, np.int32)
    off = np.empty(El + 1, np.int32)
    _load().oracle_re_routing(_ptr(x_recv), _dt(x_recv), _ptr(counts), W, El, H, _ptr(xs), _ptr(gidx), _ptr(tpl),
                              _ptr(off))
    return dict(x_sorted=xs, gathered_ids_unsort=gidx, tokens_per_local_expert=tpl, local_offsets=off)


def unsort_rows(y_sorted: np.ndarray, gathered_ids_unsort: np.ndarray) -> np.ndarray:
    y_sorted = _c(y_sorted)
    gidx = _c(gathered_ids_unsort, np.int32)
    out = np.zeros_like(y_sorted)
    _load().oracle_unsort_rows(_ptr(y_sorted), _dt(y_sorted), _ptr(gidx), gidx.size, y_sorted.shape[1], _ptr(out))
    return out


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


E4M3_VALUES = None


def e4m3_table() -> np.ndarray:
    """Values of all 256 e4m3 codes (fp64; NaN for the two NaN codes)."""
    global E4M3_VALUES
    if E4M3_VALUES is None:
        E4M3_VALUES = np.array([e4m3_decode(c) for c in range(256)])
    return E4M3_VALUES


def quantize_rows_fp8(a: np.ndarray, pow2: bool = False):
    """1x128 blocks along the columns.  Returns (codes uint8 [rows, cols], scales f32 [rows, ceil(cols/128)]).
    pow2: each scale the smallest power of two that brings the block's largest magnitude to <= 448."""
    a = _c(a)
    rows, cols = a.shape
    codes = np.empty((rows, cols), np.uint8)
    scales = np.empty((rows, (cols + 127) // 128), np.float32)
    _load().oracle_quantize_rows_fp8(_ptr(a), _dt(a), rows, cols, _ptr(codes), _ptr(scales), int(bool(pow2)))
    return codes, scales


def quantize_tiles_fp8(w: np.ndarray, pow2: bool = False):
    """128x128 tiles of a [n_out, k_in] weight.  Returns (codes, scales [ceil(n/128), ceil(k/128)]).
    pow2: power-of-two tile scales, as quantize_rows_fp8."""
    w = _c(w)
    n, k = w.shape
    codes = np.empty((n, k), np.uint8)
    scales = np.empty(((n + 127) // 128, (k + 127) // 128), np.float32)
    _load().oracle_quantize_tiles_fp8(_ptr(w), _dt(w), n, k, _ptr(codes), _ptr(scales), int(bool(pow2)))
    return codes, scales


def gemm_fp8(qa, sa, qb, sb) -> np.ndarray:
    """C[m,n] = sum_b sa[m,b] sb[n/128,b] sum_(k in b) e4m3(qa[m,k]) e4m3(qb[n,k])  (fp64)."""
    qa, qb = _c(qa, np.uint8), _c(qb, np.uint8)
    sa, sb = _c(sa, np.float32), _c(sb, np.float32)
    M, K = qa.shape
    N = qb.shape[0]
    c = np.empty((M, N), np.float64)
    _load().oracle_gemm_fp8(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K, _ptr(c))
    return c


def quantize_experts_fp8(w: np.ndarray, pow2: bool = False):
    """[E, n_out, k_in] weights -> (codes [E, n_out, k_in], scales [E, n_out/128, k_in/128])."""
    E = w.shape[0]
    pairs = [quantize_tiles_fp8(w[e], pow2) for e in range(E)]
    return np.stack([p[0] for p in pairs]), np.stack([p[1] for p in pairs])


def expert_ffn_rows_fp8(xq, xs, expert, q: dict, pow2: bool = False) -> np.ndarray:
    """y[r] = FP8 SwiGLU expert expert[r] on quantised row r, stored in bf16 (fp64 out).
    pow2: h is quantised with power-of-two block scales."""
    xq, xs = _c(xq, np.uint8), _c(xs, np.float32)
    expert = _c(expert, np.int32)
    n, H = xq.shape
    I = q["gq"].shape[1]
    assert xs.shape[1] == (H + 127) // 128
    arrs = [_c(q[k_], np.uint8 if k_.endswith("q") else np.float32) for k_ in ("gq", "gs", "uq", "us", "dq", "ds")]
    y = np.zeros((n, H), np.float64)
    _load().oracle_expert_ffn_rows_fp8(_ptr(xq), _ptr(xs), n, _ptr(expert), *[_ptr(a) for a in arrs], H, I, _ptr(y),
                                       int(bool(pow2)))
    return y


def layer_fp8(x, wg, q: dict, *, k: int, renorm: bool = True, bias=None, tokens=None, n_group: int = 1,
              topk_group: int = 1, group_rule: str = "max", pow2: bool = False):
    """Brute-force layer with FP8 expert weights (x, wg bf16 bit patterns).  q holds the codes
    and scales from quantize_experts_fp8: gq, gs, uq, us, dq, ds and the shared sgq ... sds.
    pow2: the activations (x and h) get power-of-two block scales."""
    x, wg = _c(x, np.uint16), _c(wg, np.uint16)
    T, H = x.shape
    E, I = q["gq"].shape[0], q["gq"].shape[1]
    S = 0 if q.get("sgq") is None else q["sgq"].shape[0]
    arrs = [_c(q[n], np.uint8 if n.endswith("q") else np.float32) if q.get(n) is not None else None
            for n in ("gq", "gs", "uq", "us", "dq", "ds", "sgq", "sgs", "suq", "sus", "sdq", "sds")]
    bias = _c(bias, np.float32)
    toks = None if tokens is None else _c(np.asarray(tokens, np.int32), np.int32)
    n = T if toks is None else toks.size
    logits = np.empty((n, E), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    out = np.empty((n, H), np.float64)
    _load().oracle_layer_fp8(_ptr(x), T, H, E, k, I, S, int(bool(renorm)), _ptr(wg), _ptr(bias),
                             *[_ptr(a) for a in arrs], _ptr(toks), n, _ptr(logits), _ptr(ids), _ptr(w), _ptr(out),
                             n_group, topk_group, {"max": 0, "top2_sum": 1}[group_rule], int(bool(pow2)))
    return dict(logits64=logits, ids=ids, w=w, out=out)


def expert_ffn_rows(a: np.ndarray, expert: np.ndarray, wgate, wup, w2) -> np.ndarray:
    """y[r] = FFN_{expert[r]}(a[r]) stored in a's dtype (returned as fp64).

    a [n,H]; wgate/wup [E,I,H]; w2 [E,H,I]; rows with expert < 0 stay zero."""
    a, expert = _c(a), _c(expert, np.int32)
    wgate, wup, w2 = _c(wgate), _c(wup), _c(w2)
    dt = _dt(a)
    n, H = a.shape
    I = wgate.shape[1]
    y = np.zeros((n, H), np.float64)
    _load().oracle_expert_ffn_rows(_ptr(a), dt, n, _ptr(expert), _ptr(wgate), _ptr(wup), _ptr(w2),
                                   H, I, _ptr(y))
    return y


def finalize_routing(y: np.ndarray, scales: np.ndarray, expanded_row_idx: np.ndarray,
                     skip: np.ndarray | None = None) -> np.ndarray:
    """out[t] = skip[t] + sum_j scales[t,j] y[expanded_row_idx[t*k+j]]  (fp64, unrounded)."""
    y = _c(y)
    dt = _dt(y)
    scales = _c(np.asarray(scales, np.float64), np.float64)
    idx = _c(expanded_row_idx, np.int32).reshape(-1)
    T, k = scales.shape
    H = y.shape[1]
    skip = _c(skip)
    if skip is not None:
        assert _dt(skip) == dt
    out = np.empty((T, H), np.float64)
    _load().oracle_finalize_routing(_ptr(y), dt, y.shape[0], _ptr(skip), _ptr(scales), _ptr(idx),
                                    T, H, k, _ptr(out))
    return out


def layer(x, wg, wgate, wup, w2, sgate=None, sup=None, s2=None, *, k: int, renorm: bool = True,
          bias=None, tokens=None, n_group: int = 1, topk_group: int = 1, group_rule: str = "max"):
    """Brute-force per-token MoE layer.

    x [T,H]; wg [E,H]; wgate/wup [E,I,H]; w2 [E,H,I]; sgate/sup [S,I,H]; s2 [S,H,I].
    tokens: optional int array of token indices to evaluate.
    Returns dict(logits64 [n,E], ids [n,k], w [n,k], out [n,H] (rounded to x's dtype))."""
    x, wg = _c(x), _c(wg)
    wgate, wup, w2 = _c(wgate), _c(wup), _c(w2)
    dt = _dt(x)
    T, H = x.shape
    E, I = wgate.shape[0], wgate.shape[1]
    S = 0 if sgate is None else sgate.shape[0]
    sgate, sup, s2 = _c(sgate), _c(sup), _c(s2)
    bias = _c(bias, np.float32)
    toks = None if tokens is None else _c(np.asarray(tokens, np.int32), np.int32)
    n = T if toks is None else toks.size
    logits = np.empty((n, E), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    out = np.empty((n, H), np.float64)
    _load().oracle_layer(_ptr(x), dt, T, H, E, k, I, S, int(bool(renorm)), _ptr(wg), _ptr(bias),
                         _ptr(wgate), _ptr(wup), _ptr(w2), _ptr(sgate), _ptr(sup), _ptr(s2),
                         _ptr(toks), n, _ptr(logits), _ptr(ids), _ptr(w), _ptr(out), n_group, topk_group,
                         {"max": 0, "top2_sum": 1}[group_rule])
    return dict(logits64=logits, ids=ids, w=w, out=out)
