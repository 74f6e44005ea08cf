"""The C++ oracle (oracle/csa_oracle_ref.cpp) with the numpy oracle's call
signatures -- TEST INFRASTRUCTURE ONLY, like the rest of oracle/.

compress, n_visible, indexer_scores, topk and attend_one run in the C++
library in double precision; the conversions between bf16 bit patterns and
float64 and the window rows are the numpy oracle's (plain definitions, no
arithmetic of the method).  The library is built by the repository's build
step (g++); importing this module without it raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

from .csa_oracle import bf16_to_f64, round_bf16, window_rows  # noqa: F401  (shared bf16 helpers)

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csa_oracle_ref.cpp")
LIB = os.path.join(HERE, "liboracle_ref.so")


def build(force: bool = False) -> str:
    """Compile the C++ oracle with g++ (-O2, no fast-math: IEEE double)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        r = subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-o", LIB, SRC],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"g++ failed for the C++ oracle:\n{r.stderr}")
    return LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} is missing: build it with oracle.ref_cpp.build()")
        L = ctypes.CDLL(LIB)
        dp, ip, i, d = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_double
        L.oref_compress.argtypes = [dp, dp, i, i, i, dp]
        L.oref_compress.restype = i
        L.oref_n_visible.argtypes = [i, i, i]
        L.oref_n_visible.restype = i
        L.oref_indexer_scores.argtypes = [dp, dp, dp, i, i, i, i, i, dp]
        L.oref_indexer_scores.restype = i
        L.oref_topk.argtypes = [dp, i, i, ip]
        L.oref_topk.restype = None
        L.oref_attend_one.argtypes = [dp, i, i, dp, dp, ip, i, dp, dp, ip, i, d, dp, dp]
        L.oref_attend_one.restype = None
        _lib = L
    return _lib


def _d(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a, t=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(t))


def compress(x: np.ndarray, g: np.ndarray, m: int) -> np.ndarray:
    x, g = _d(x), _d(g)
    T, D = x.shape
    out = np.zeros((T // m, D))
    _L().oref_compress(_p(x), _p(g), T, D, m, _p(out))
    return out


def n_visible(t: int, m: int, N: int) -> int:
    return int(_L().oref_n_visible(int(t), int(m), int(N)))


def indexer_scores(q_idx: np.ndarray, k_idx: np.ndarray, w: np.ndarray, t: int, m: int) -> np.ndarray:
    q, k, w = _d(q_idx), _d(k_idx), _d(w)
    H, dI = q.shape
    N = k.shape[0]
    S = np.zeros(max(N, 1))
    n = _L().oref_indexer_scores(_p(q), _p(k), _p(w), H, dI, N, int(t), int(m), _p(S))
    return S[:n].copy()


def topk(S: np.ndarray, k: int) -> np.ndarray:
    S = _d(S)
    out = np.zeros(k, dtype=np.int32)
    _L().oref_topk(_p(S), S.shape[0], k, _p(out, ctypes.c_int32))
    return out


def attend_one(q: np.ndarray, k_cmp: np.ndarray, v_cmp: np.ndarray, sel: Sequence[int], k_raw: np.ndarray,
               v_raw: np.ndarray, win: np.ndarray, scale: float):
    q = _d(q)
    H, d = q.shape
    kc = _d(k_cmp).reshape(-1, d) if np.size(k_cmp) else np.zeros((1, d))
    vc = _d(v_cmp).reshape(-1, d) if np.size(v_cmp) else np.zeros((1, d))
    kr = _d(k_raw).reshape(-1, d) if np.size(k_raw) else np.zeros((1, d))
    vr = _d(v_raw).reshape(-1, d) if np.size(v_raw) else np.zeros((1, d))
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1))
    win = np.ascontiguousarray(np.asarray(win, dtype=np.int32).reshape(-1))
    O = np.zeros((H, d))
    lse = np.zeros(H)
    _L().oref_attend_one(_p(q), H, d, _p(kc), _p(vc), _p(sel, ctypes.c_int32), sel.shape[0], _p(kr), _p(vr),
                         _p(win, ctypes.c_int32), win.shape[0], float(scale), _p(O), _p(lse))
    return O, lse


# batched entry points (the library's calls), looping over sequences and queries

def csa_compress(x_bits, g_bits, m: int) -> np.ndarray:
    x, g = bf16_to_f64(x_bits), bf16_to_f64(g_bits)
    return np.stack([compress(x[b], g[b], m) for b in range(x.shape[0])])


def csa_index_scores(q_idx_bits, k_idx_bits, w, q_pos, m: int):
    qi, ki = bf16_to_f64(q_idx_bits), bf16_to_f64(k_idx_bits)
    w = np.asarray(w, dtype=np.float64)
    return [[indexer_scores(qi[b, j], ki[b], w if w.ndim == 1 else w[b, j], int(q_pos[b][j]), m)
             for j in range(qi.shape[1])] for b in range(qi.shape[0])]


def csa_index_topk(q_idx_bits, k_idx_bits, w, q_pos, m: int, k: int):
    S = csa_index_scores(q_idx_bits, k_idx_bits, w, q_pos, m)
    return np.stack([np.stack([topk(s, k) for s in row]) for row in S]), S


def _attend_all(q_bits, kc_bits, vc_bits, sel_of, kr_bits, vr_bits, raw_base, q_pos, W, scale):
    q = bf16_to_f64(q_bits)
    kc, vc = bf16_to_f64(kc_bits), bf16_to_f64(vc_bits)
    kr, vr = bf16_to_f64(kr_bits), bf16_to_f64(vr_bits)
    B, Tq, H, d = q.shape
    O = np.zeros((B, Tq, H, d))
    L = np.zeros((B, Tq, H))
    for b in range(B):
        for j in range(Tq):
            t = int(q_pos[b][j])
            win = window_rows(t, W, int(raw_base[b]), kr.shape[1])
            O[b, j], L[b, j] = attend_one(q[b, j], kc[b], vc[b], sel_of(b, j, t, kc.shape[1]), kr[b], vr[b], win,
                                          scale)
    return O, L


def csa_attend(q_bits, k_cmp_bits, v_cmp_bits, idx, k_raw_bits, v_raw_bits, raw_base, q_pos, W: int, scale: float):
    return _attend_all(q_bits, k_cmp_bits, v_cmp_bits, lambda b, j, t, N: idx[b][j], k_raw_bits, v_raw_bits,
                       raw_base, q_pos, W, scale)


def hca_attend(q_bits, k_cmp_bits, v_cmp_bits, k_raw_bits, v_raw_bits, raw_base, q_pos, m: int, W: int,
               scale: float):
    return _attend_all(q_bits, k_cmp_bits, v_cmp_bits, lambda b, j, t, N: np.arange(n_visible(t, m, N)),
                       k_raw_bits, v_raw_bits, raw_base, q_pos, W, scale)
