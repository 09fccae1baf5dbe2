"""Seeded synthetic inputs (see gen.h): host (numpy) and device (torch CUDA) fills
that produce identical values. Holds no part of the method's arithmetic.

Recipe (the workloads of the pages, stated as distributions):
  * expert / shared-expert / lm_head masters: bf16 sigma * N(0, 1), sigma = 0.02;
  * router gate: bf16 N(0, 0.02) values held as float32 (the gate is a bf16
    tensor computed in fp32);
  * e_score_correction_bias: float32 U(lo, hi);
  * hidden states: bf16 N(0, 1); with correlation rho between tokens,
    h_t = sqrt(rho) z_0 + sqrt(1 - rho) z_{t+1}.
"""
import ctypes
import math

import numpy as np

from . import build as _build

KIND_ROUTER_W, KIND_ROUTER_B, KIND_UP, KIND_DOWN = 1, 2, 3, 4
KIND_SH_UP, KIND_SH_DOWN, KIND_LM_HEAD, KIND_HIDDEN = 5, 6, 7, 8
WEIGHT_SIGMA = 0.02

_host = None
_dev = None


def tensor_id(kind: int, layer: int, index: int) -> int:
    return ((kind << 28) | ((layer & 0xFF) << 20) | (index & 0xFFFFF)) & 0xFFFFFFFF


def host():
    global _host
    if _host is None:
        L = ctypes.CDLL(_build.build_host())
        P, I64, U32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
        L.gen_fill_normal_bf16.argtypes = [P, I64, U32, U32, F]
        L.gen_fill_normal_bf16_range.argtypes = [P, I64, I64, U32, U32, F]
        L.gen_fill_normal_bf16_range.restype = None
        L.gen_fill_normal_f32.argtypes = [P, I64, U32, U32]
        L.gen_fill_uniform_f32.argtypes = [P, I64, U32, U32, F, F]
        L.gen_fill_hidden_bf16.argtypes = [P, ctypes.c_int32, ctypes.c_int32, I64, U32, U32, F, F]
        L.gen_philox.argtypes = [P, P, P]
        L.gen_log_test.argtypes = [F]
        L.gen_log_test.restype = F
        for f in (L.gen_fill_normal_bf16, L.gen_fill_normal_f32, L.gen_fill_uniform_f32,
                  L.gen_fill_hidden_bf16, L.gen_philox):
            f.restype = None
        _host = L
    return _host


def dev():
    global _dev
    if _dev is None:
        L = ctypes.CDLL(_build.build_cuda())
        P, I64, U32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
        L.gen_dev_normal_bf16.argtypes = [P, I64, U32, U32, F, P]
        L.gen_dev_normal_bf16_as_f32.argtypes = [P, P, I64, U32, U32, F, P]
        L.gen_dev_uniform_f32.argtypes = [P, I64, U32, U32, F, F, P]
        L.gen_dev_hidden_bf16.argtypes = [P, ctypes.c_int32, ctypes.c_int32, I64, U32, U32, F, F, P]
        for f in (L.gen_dev_normal_bf16, L.gen_dev_normal_bf16_as_f32, L.gen_dev_uniform_f32,
                  L.gen_dev_hidden_bf16):
            f.restype = ctypes.c_int
        _dev = L
    return _dev


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rho(rho):
    return float(np.float32(math.sqrt(rho))), float(np.float32(math.sqrt(1.0 - rho)))


# ---------------------------------------------------------------- host fills
def philox(ctr, key):
    c = np.asarray(ctr, np.uint32)
    k = np.asarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    host().gen_philox(_p(c), _p(k), _p(out))
    return out


def normal_bf16(n, seed, tid, sigma):
    out = np.zeros(n, np.uint16)
    host().gen_fill_normal_bf16(_p(out), n, seed, tid, sigma)
    return out


def normal_f32(n, seed, tid):
    out = np.zeros(n, np.float32)
    host().gen_fill_normal_f32(_p(out), n, seed, tid)
    return out


def uniform_f32(n, seed, tid, lo, hi):
    out = np.zeros(n, np.float32)
    host().gen_fill_uniform_f32(_p(out), n, seed, tid, lo, hi)
    return out


def hidden_bf16(T, H, seed, layer=0, rho=0.0, t0=0):
    out = np.zeros((T, H), np.uint16)
    sr, s1 = _rho(rho)
    host().gen_fill_hidden_bf16(_p(out), t0, T, H, seed, layer, sr, s1)
    return out


def bf16_bits_to_f32(a):
    return (a.astype(np.uint32) << 16).view(np.float32)


def router_w(seed, layer, E, H):
    w = normal_bf16(E * H, seed, tensor_id(KIND_ROUTER_W, layer, 0), WEIGHT_SIGMA)
    return bf16_bits_to_f32(w).reshape(E, H)


def router_bias(seed, layer, E, lo, hi):
    return uniform_f32(E, seed, tensor_id(KIND_ROUTER_B, layer, 0), lo, hi)


def up_master(seed, layer, e, I, H):
    return normal_bf16(I * H, seed, tensor_id(KIND_UP, layer, e), WEIGHT_SIGMA).reshape(I, H)


def down_master(seed, layer, e, H, I):
    return normal_bf16(H * I, seed, tensor_id(KIND_DOWN, layer, e), WEIGHT_SIGMA).reshape(H, I)


def sh_up_master(seed, layer, S, H):
    return normal_bf16(S * H, seed, tensor_id(KIND_SH_UP, layer, 0), WEIGHT_SIGMA).reshape(S, H)


def sh_down_master(seed, layer, H, S):
    return normal_bf16(H * S, seed, tensor_id(KIND_SH_DOWN, layer, 0), WEIGHT_SIGMA).reshape(H, S)


def lm_head_master(seed, V, H, row0=0, nrows=None):
    """Rows [row0, row0+nrows) of the lm_head master; elements are addressed by
    their flat index, so any slice regenerates exactly."""
    nrows = V - row0 if nrows is None else nrows
    return normal_bf16_range(row0 * H, nrows * H, seed, tensor_id(KIND_LM_HEAD, 0, 0),
                             WEIGHT_SIGMA).reshape(nrows, H)


def normal_bf16_range(i0, n, seed, tid, sigma):
    out = np.zeros(n, np.uint16)
    host().gen_fill_normal_bf16_range(_p(out), i0, n, seed, tid, sigma)
    return out


# --------------------------------------------------------------- device fills
def _stream_ptr(stream):
    return ctypes.c_void_p(stream.cuda_stream if stream is not None else 0)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what}: CUDA error {rc}")


def dev_normal_bf16(t, seed, tid, sigma, stream=None):
    """Fill a contiguous torch.bfloat16/int16 CUDA tensor in place."""
    _check(dev().gen_dev_normal_bf16(ctypes.c_void_p(t.data_ptr()), t.numel(), seed, tid, sigma,
                                     _stream_ptr(stream)), "gen_dev_normal_bf16")


def dev_normal_bf16_as_f32(t, tmp, seed, tid, sigma, stream=None):
    _check(dev().gen_dev_normal_bf16_as_f32(ctypes.c_void_p(t.data_ptr()),
                                            ctypes.c_void_p(tmp.data_ptr()), t.numel(), seed, tid,
                                            sigma, _stream_ptr(stream)), "gen_dev_normal_bf16_as_f32")


def dev_uniform_f32(t, seed, tid, lo, hi, stream=None):
    _check(dev().gen_dev_uniform_f32(ctypes.c_void_p(t.data_ptr()), t.numel(), seed, tid, lo, hi,
                                     _stream_ptr(stream)), "gen_dev_uniform_f32")


def dev_hidden_bf16(t, seed, layer=0, rho=0.0, t0=0, stream=None):
    T, H = t.shape
    sr, s1 = _rho(rho)
    _check(dev().gen_dev_hidden_bf16(ctypes.c_void_p(t.data_ptr()), t0, T, H, seed, layer, sr, s1,
                                     _stream_ptr(stream)), "gen_dev_hidden_bf16")
