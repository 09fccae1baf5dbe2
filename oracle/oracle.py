"""ctypes wrapper around the C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py, never by the product package. All arrays are
numpy; bf16 tensors travel as uint16 bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class OrcMat(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("g", ctypes.c_float),
                ("n", ctypes.c_int64), ("k", ctypes.c_int64)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        L.orc_e2m1_value.restype = ctypes.c_double
        L.orc_e2m1_value.argtypes = [ctypes.c_int]
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_e4m3_value.argtypes = [ctypes.c_int]
        L.orc_e2m1_encode.restype = ctypes.c_int
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_int
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_bf16_round.restype = ctypes.c_uint16
        L.orc_bf16_round.argtypes = [ctypes.c_double]
        L.orc_bf16_value.restype = ctypes.c_double
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_quantize.restype = ctypes.c_int
        L.orc_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P, P, P]
        L.orc_dequantize.restype = None
        L.orc_dequantize.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, P]
        L.orc_route.restype = None
        L.orc_route.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P, ctypes.c_int32,
                                ctypes.c_int32, P, P, P, P, P]
        L.orc_moe_layer.restype = None
        L.orc_moe_layer.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P, P, P, P, P,
                                    ctypes.c_int32, P, P, P]
        L.orc_rms_norm.restype = None
        L.orc_rms_norm.argtypes = [P, ctypes.c_int32, ctypes.c_int64, ctypes.c_double, P]
        L.orc_lm_head.restype = None
        L.orc_lm_head.argtypes = [P, P, ctypes.c_int32, P]
        L.orc_lm_head_rows.restype = None
        L.orc_lm_head_rows.argtypes = [P, P, ctypes.c_int32, P, ctypes.c_int64, P]
        L.orc_fp8_quantize.restype = ctypes.c_int
        L.orc_fp8_quantize.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P, P]
        L.orc_shared_fp8.restype = None
        L.orc_shared_fp8.argtypes = [P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_float, P,
                                     ctypes.c_float, P, P]
        L.orc_set_threads.restype = None
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_get_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int):
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return lib().orc_get_threads()


# ---- codecs ---------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return lib().orc_e4m3_value(int(byte))


def e2m1_encode(v: float) -> int:
    return lib().orc_e2m1_encode(float(v))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def bf16_round(x: float) -> int:
    return lib().orc_bf16_round(float(x))


def bf16_value(b: int) -> float:
    return lib().orc_bf16_value(int(b))


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


# ---- quantiser ------------------------------------------------------------
PER_TENSOR, PER_ROW, GIVEN = 0, 1, 2


def quantize(x: np.ndarray, mode: int = PER_TENSOR, g: float = None):
    """x: float32 [rows][cols] (or uint16 bf16). Returns (codes, scales, g)."""
    if x.dtype == np.uint16:
        x = bf16_to_f32(x)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    gio = np.zeros(rows if mode == PER_ROW else 1, np.float32)
    if mode == GIVEN:
        gio[0] = g
    rc = lib().orc_quantize(_p(x), rows, cols, mode, _p(gio), _p(codes), _p(scales))
    if rc != 0:
        raise ValueError("orc_quantize rejected its arguments")
    return codes, scales, gio


def dequantize(codes, scales, g, cols: int = None) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    g = np.ascontiguousarray(np.atleast_1d(g), np.float32)
    rows = codes.shape[0]
    cols = codes.shape[1] * 2 if cols is None else cols
    out = np.zeros((rows, cols), np.float64)
    lib().orc_dequantize(_p(codes), _p(scales), _p(g), int(g.size > 1), rows, cols, _p(out))
    return out


class Mat:
    """An NVFP4 matrix held by the oracle: codes [n][k/2], scales [n][k/16], global g."""

    def __init__(self, codes, scales, g):
        self.codes = np.ascontiguousarray(codes, np.uint8)
        self.scales = np.ascontiguousarray(scales, np.uint8)
        self.g = float(np.asarray(g).reshape(-1)[0])
        self.n = self.codes.shape[0]
        self.k = self.codes.shape[1] * 2

    def c(self):
        return OrcMat(self.codes.ctypes.data, self.scales.ctypes.data, self.g, self.n, self.k)

    @staticmethod
    def from_master(w):
        c, s, g = quantize(w, PER_TENSOR)
        return Mat(c, s, g[0])


# ---- router ---------------------------------------------------------------
def route(h_bf16: np.ndarray, Wg: np.ndarray, bias: np.ndarray, k: int):
    """Returns dict(idx int32 [T][k], w f64 [T][k], z, c, tau f64 [T][E])."""
    h = np.ascontiguousarray(h_bf16, np.uint16)
    if h.ndim == 1:
        h = h[None, :]
    T, H = h.shape
    Wg = np.ascontiguousarray(Wg, np.float32)
    bias = np.ascontiguousarray(bias, np.float32)
    E = Wg.shape[0]
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    z = np.zeros((T, E), np.float64)
    c = np.zeros((T, E), np.float64)
    tau = np.zeros((T, E), np.float64)
    lib().orc_route(_p(h), T, H, _p(Wg), _p(bias), E, k, _p(idx), _p(w), _p(z), _p(c), _p(tau))
    return dict(idx=idx, w=w, z=z, c=c, tau=tau)


def rms_norm_slack(h_bf16, eps, Wg, window=2.0 ** -18):
    """Logit slack [T][E] of routing on an RMS norm evaluated in binary32
    instead of this oracle's binary64 (the pages fix the norm's bf16 output,
    card-int4 "Left at bfloat16", not the precision it is computed in). An
    element whose exact normalised value lies within `window` (relative) of a
    bf16 rounding midpoint may round to the other neighbour in binary32 (the
    binary32 sum of squares and reciprocal square root are good to a few
    2^-24), moving logit e by up to |Wg[e][i]| times the gap between the two
    neighbours; the slack adds this up over such elements. Zero for eps <= 0
    (no norm, the input is used as it is)."""
    h = np.ascontiguousarray(h_bf16, np.uint16)
    if h.ndim == 1:
        h = h[None, :]
    Wg = np.asarray(Wg, np.float64)
    if eps <= 0:
        return np.zeros((h.shape[0], Wg.shape[0]))
    hv = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    inv = 1.0 / np.sqrt((hv * hv).sum(axis=1) / hv.shape[1] + eps)
    x = hv * inv[:, None]
    lo_bits = x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    lo = lo_bits.view(np.float32).astype(np.float64)
    hi = (lo_bits + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    gap = np.abs(hi - lo)
    near = (np.abs(x - 0.5 * (lo + hi)) <= window * np.abs(x)) & (x != 0)
    return (near * gap) @ np.abs(Wg).T


# ---- MoE layer / lm_head --------------------------------------------------
def rms_norm(h_bf16, eps):
    """Unit-weight RMS norm of each bf16 row -> bf16 (uint16 bits)."""
    h = np.ascontiguousarray(h_bf16, np.uint16)
    if h.ndim == 1:
        h = h[None, :]
    out = np.zeros_like(h)
    lib().orc_rms_norm(_p(h), h.shape[0], h.shape[1], float(eps), _p(out))
    return out


def moe_layer(h_bf16, idx, w, up: dict, down: dict, sh_up: Mat, sh_down: Mat, w4a4: bool,
              residual, num_experts: int):
    """up/down: {expert_id: Mat}; only the experts named in idx are needed.
    residual: None, or a bf16 [T][H] array added before the final rounding.
    Returns (out_bf16 uint16 [T][H], out_f64 [T][H])."""
    h = np.ascontiguousarray(h_bf16, np.uint16)
    if h.ndim == 1:
        h = h[None, :]
    T, H = h.shape
    idx = np.ascontiguousarray(idx, np.int32).reshape(T, -1)
    k = idx.shape[1]
    w = np.ascontiguousarray(w, np.float64).reshape(T, k)
    ups = (OrcMat * num_experts)()
    downs = (OrcMat * num_experts)()
    for e in range(num_experts):
        if e in up:
            ups[e] = up[e].c()
            downs[e] = down[e].c()
    for e in np.unique(idx):
        if int(e) not in up:
            raise KeyError(f"expert {int(e)} weights not supplied")
    shu, shd = sh_up.c(), sh_down.c()
    out = np.zeros((T, H), np.uint16)
    outf = np.zeros((T, H), np.float64)
    res = None
    if residual is not None:
        res = np.ascontiguousarray(residual, np.uint16).reshape(T, H)
    lib().orc_moe_layer(_p(h), T, k, _p(idx), _p(w), ctypes.cast(ups, ctypes.c_void_p),
                        ctypes.cast(downs, ctypes.c_void_p), ctypes.byref(shu), ctypes.byref(shd),
                        int(w4a4), _p(res) if res is not None else None, _p(out), _p(outf))
    return out, outf


def lm_head(W: Mat, h_bf16) -> np.ndarray:
    h = np.ascontiguousarray(h_bf16, np.uint16)
    if h.ndim == 1:
        h = h[None, :]
    T = h.shape[0]
    out = np.zeros((T, W.n), np.float64)
    m = W.c()
    lib().orc_lm_head(ctypes.byref(m), _p(h), T, _p(out))
    return out


def lm_head_rows(W: Mat, h_bf16, rows) -> np.ndarray:
    h = np.ascontiguousarray(h_bf16, np.uint16)
    if h.ndim == 1:
        h = h[None, :]
    T = h.shape[0]
    rows = np.ascontiguousarray(rows, np.int64)
    out = np.zeros((T, rows.size), np.float64)
    m = W.c()
    lib().orc_lm_head_rows(ctypes.byref(m), _p(h), T, _p(rows), rows.size, _p(out))
    return out


# ---- FP8 shared expert ------------------------------------------------------
def fp8_quantize(x: np.ndarray, mode: int = PER_TENSOR, g: float = None):
    """x: float32 [rows][cols] (or uint16 bf16). Returns (codes uint8 [rows][cols], g)."""
    if x.dtype == np.uint16:
        x = bf16_to_f32(x)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    rows, cols = x.shape
    q = np.zeros((rows, cols), np.uint8)
    gio = np.zeros(rows if mode == PER_ROW else 1, np.float32)
    if mode == GIVEN:
        gio[0] = g
    if lib().orc_fp8_quantize(_p(x), rows, cols, mode, _p(gio), _p(q)) != 0:
        raise ValueError("orc_fp8_quantize rejected its arguments")
    return q, gio


def shared_fp8(x_bf16, w_up, g_up, w_dn, g_dn):
    """The FP8 W8A8 shared expert on bf16 rows x [T][H]: returns (y f64 [T][H],
    act bf16 bits [T][S])."""
    x = np.ascontiguousarray(x_bf16, np.uint16)
    T, H = x.shape
    w_up = np.ascontiguousarray(w_up, np.uint8)
    w_dn = np.ascontiguousarray(w_dn, np.uint8)
    S = w_up.shape[0]
    y = np.zeros((T, H), np.float64)
    act = np.zeros((T, S), np.uint16)
    lib().orc_shared_fp8(_p(x), T, H, S, _p(w_up), float(g_up), _p(w_dn), float(g_dn), _p(y), _p(act))
    return y, act
