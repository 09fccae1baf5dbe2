"""Shared helpers for the parity tests (test infrastructure)."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")

# floating-point parity bar: |gpu - ref| <= ATOL + RTOL * |ref|, elementwise
ATOL, RTOL = 1e-2, 2e-2


def header_functions():
    """Names of the functions include/nvfp4moe.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-zA-Z_][\w\s\*]*?\b([a-z][a-z0-9_]+)\s*\(", src, re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def bf16_bits(t):
    """torch bf16 tensor -> numpy uint16 bit patterns."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().astype(np.uint16)


def to_dev_bf16(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_to_f64(a):
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside {ATOL} + {RTOL}|ref|; "
                           f"worst |err| {err.max():.4g} at {np.unravel_index(err.argmax(), err.shape)}")
    return err.max()


def check_routing(gpu_idx, gpu_w, orc, k):
    """Routing parity: indices must equal the oracle's; a difference is allowed
    only where the oracle's biased scores of the swapped experts are within
    their binary32 error bounds (tau). Weights agree to 1e-5 relative, plus,
    when the oracle routed a normalised input, what the input's bf16 rounding
    decisions may move them by (zslack). Returns the number of exempted tokens."""
    gpu_idx = np.asarray(gpu_idx)
    T, E = orc["c"].shape
    exempt = 0
    for t in range(T):
        gi = list(gpu_idx[t])
        if gi == list(orc["idx"][t]):
            bound = 0.0
            if orc.get("zslack") is not None:
                # the input's own bf16 rounding may differ (rms_norm_slack):
                # sigma moves by at most slack / 4, w_j = sigma_j / S by at
                # most (dsigma_j + w_j sum_l dsigma_l) / S
                sel = orc["idx"][t]
                sig = 1.0 / (1.0 + np.exp(-orc["z"][t][sel]))
                ds = 0.25 * orc["zslack"][t][sel]
                bound = (ds + orc["w"][t] * ds.sum()) / sig.sum()
            err = np.abs(np.asarray(gpu_w[t], np.float64) - orc["w"][t])
            assert (err <= 1e-7 + 1e-5 * np.abs(orc["w"][t]) + bound).all(), \
                f"token {t}: weights {gpu_w[t]} vs {orc['w'][t]} (slack {bound})"
            continue
        c, tau = orc["c"][t], orc["tau"][t]
        assert len(set(gi)) == k and all(0 <= e < E for e in gi), f"token {t}: invalid {gi}"
        inside = np.zeros(E, bool)
        inside[gi] = True
        lo = np.min(c[inside] + tau[inside])
        hi = np.max(c[~inside] - tau[~inside]) if (~inside).any() else -np.inf
        assert lo >= hi, f"token {t}: gpu set {gi} vs oracle {list(orc['idx'][t])} not a near-tie"
        for a, b in zip(gi[:-1], gi[1:]):
            assert c[a] + tau[a] >= c[b] - tau[b], f"token {t}: order {gi}"
        exempt += 1
    return exempt


def colblock_loops(codes, scales):
    """The column-block order of nvfp4_colblock_layout as include/nvfp4moe.h
    states it, byte by byte."""
    B, R, C2 = codes.shape
    out = np.zeros((B, 2 * C2 // 16, 9 * R), np.uint8)
    for b in range(B):
        for c in range(2 * C2 // 16):
            for p in range(R // 32):
                for L in range(32):
                    g, q = L // 4, L % 4
                    for mt in range(2):
                        for i in range(4):
                            row = 32 * p + 16 * mt + g + 8 * (i >> 1)
                            col = 16 * c + 4 * q + 2 * (i & 1)
                            out[b, c, 256 * p + 8 * L + 4 * mt + i] = codes[b, row, col // 2]
                for g in range(8):
                    for mt in range(2):
                        for j in range(2):
                            out[b, c, 8 * R + 32 * p + 4 * g + 2 * mt + j] = scales[b, 32 * p + 16 * mt + g + 8 * j, c]
    return out


def colblock_vectorised(codes, scales):
    """colblock_loops with numpy indexing, for the large cases."""
    B, R, C2 = codes.shape
    P, NB = R // 32, 2 * C2 // 16
    L = np.arange(32)
    g, q = L // 4, L % 4
    mt, i = np.arange(2), np.arange(4)
    rows = (32 * np.arange(P)[:, None, None, None] + 16 * mt[None, None, :, None] + g[None, :, None, None]
            + 8 * (i[None, None, None, :] >> 1))                                       # [P, 32, 2, 4]
    cbyte = 8 * np.arange(NB)[:, None, None] + 2 * q[None, :, None] + (i[None, None, :] & 1)  # [NB, 32, 4]
    cod = codes[:, rows[None], cbyte[:, None, :, None, :]].reshape(B, NB, 256 * P)
    gg = np.arange(8)
    srow = (32 * np.arange(P)[:, None, None, None] + 16 * mt[None, None, :, None] + gg[None, :, None, None]
            + 8 * np.arange(2)[None, None, None, :])                                     # [P, 8, 2, 2]
    sc = scales[:, srow[None], np.arange(NB)[:, None, None, None, None]].reshape(B, NB, 32 * P)
    return np.concatenate([cod, sc], axis=2)
