"""CPU oracle for the Compressed Sparse Attention (CSA) / Heavily Compressed
Attention (HCA) path -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  The product path (the CUDA library and its Python
binding) never calls it and shares no code with it.

Everything is computed in float64 from the bf16 bit patterns of the inputs,
plainly and in the order the method states it, with numpy library primitives
(matmul, exp, sort) as the only building blocks.

Sources (page title, then section):
* "DeepSeek V4: Compressed Sparse Attention and the Million-Token Context"
  (octagono.org), section "Hybrid Attention: CSA and HCA": a learned
  compressor folds each run of m tokens of the KV cache into one entry; the
  Lightning Indexer rates every query against the compressed blocks and keeps
  the best 1024; a window over the last 128 raw tokens supplies local context;
  HCA folds every m' >> m tokens and then attends to all of them.
* "DeepSeek V4 technical review" (takeshell.com), section 2.1 CSA: each entry
  is a weighted sum over m tokens (the sequence shrinks to 1/m of its length);
  per query token the indexer forms its own queries, rates the compressed
  entries and keeps the k best blocks, and attention is then computed over
  those k blocks only; the constants are m = 4, 64 indexer heads of width 128,
  k = 1024.  Section 2.2 HCA: m' = 128.
* The workload specification that accompanies those pages fixes what the pages
  leave open: the compressor is a per-channel softmax over the block of given
  gate logits multiplied with the raw vectors; the indexer score is
  sum_h w_h * ReLU(q_h . k); top-k ties go to the lowest index; block b is
  visible to query position t iff (b+1)*m - 1 <= t; the softmax scale is
  1/sqrt(d); one K/V stream is shared by all query heads (MQA).

Readings taken where the pages are silent (each is listed with its reason in
the design notes of the repository):
* window = raw tokens u with max(0, t-W+1) <= u <= t (t included);
* selected compressed entries and the window tokens share ONE softmax; they are
  not de-duplicated;
* a trailing partial block (T mod m tokens) is not compressed;
* selected indices are returned in ascending block order, padded with -1;
* compressed entries are rounded to bf16 (round-to-nearest-even) before they
  are used downstream, as a bf16 cache holds them;
* an empty key set gives output 0 and log-sum-exp -inf.

Pins (tests/test_oracle_pins.py): hand-worked m=2 compression values and a
hand-worked two-key attention value (tests/golden/), closed forms, shift /
permutation / homogeneity invariants, brute force over all k-subsets for
top-k, and reductions to torch's scaled_dot_product_attention and scipy's
logsumexp.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np


# --------------------------------------------------------------------------
# bf16 <-> float64
# --------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x) -> np.ndarray:
    """float64 -> bf16 bit patterns, round-to-nearest-even, one rounding.

    bf16 keeps 8 significant bits.  Finite, normal-range values only (the
    path's values are O(1)); raises on inf / nan.
    """
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("round_bf16: non-finite input")
    mant, ex = np.frexp(x)                    # x = mant * 2**ex, 0.5 <= |mant| < 1
    q = np.round(mant * 256.0) / 256.0        # np.round: half to even
    y = np.ldexp(q, ex).astype(np.float32)    # exactly representable in fp32
    return (y.view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# (1) block compression
# --------------------------------------------------------------------------

def compress(x: np.ndarray, g: np.ndarray, m: int) -> np.ndarray:
    """Compress one sequence's stream x [T, D] with gate logits g [T, D].

    Entry b, channel c: sum_{j<m} softmax_j(g[b*m + j, c]) * x[b*m + j, c]
    (a weighted sum over the block's m tokens whose weights are the
    per-channel softmax of the block's gate logits).  T mod m trailing
    tokens are dropped.  Returns float64 [T // m, D].
    """
    T, D = x.shape
    nb = T // m
    X = x[: nb * m].reshape(nb, m, D)
    G = g[: nb * m].reshape(nb, m, D)
    G = G - G.max(axis=1, keepdims=True)      # softmax is shift-invariant
    P = np.exp(G)
    P = P / P.sum(axis=1, keepdims=True)
    return (P * X).sum(axis=1)


def append_blocks(x_win: np.ndarray, g_win: np.ndarray, raw_base: int, positions: Sequence[int],
                  m: int) -> Dict[int, np.ndarray]:
    """Decode-time compression of one sequence: every m tokens become one
    entry, so a query at position t with (t+1) mod m == 0 completes block
    b = (t+1)/m - 1 (tokens t-m+1 .. t), which is compressed from the raw rows
    the window buffer holds (row r = token raw_base + r) exactly as ``compress``
    folds a block.  x_win, g_win [T_raw, D].  Returns {b: float64 [D]} for the
    positions that complete a block (none for the others)."""
    out = {}
    for t in positions:
        t = int(t)
        if t < 0 or (t + 1) % m != 0:
            continue
        r0 = t - m + 1 - raw_base
        if r0 < 0 or r0 + m > x_win.shape[0]:
            raise IndexError("block rows outside the window buffer")
        out[(t + 1) // m - 1] = compress(x_win[r0:r0 + m], g_win[r0:r0 + m], m)[0]
    return out


# --------------------------------------------------------------------------
# (2) Lightning Indexer scores, (3) top-k
# --------------------------------------------------------------------------

def n_visible(t: int, m: int, N: int) -> int:
    """Number of compressed blocks visible at query position t.

    Block b (tokens b*m .. b*m+m-1) is visible iff (b+1)*m - 1 <= t, i.e.
    b < floor((t+1)/m); at most N blocks exist.
    """
    return max(0, min(N, (t + 1) // m))


def indexer_scores(q_idx: np.ndarray, k_idx: np.ndarray, w: np.ndarray,
                   t: int, m: int) -> np.ndarray:
    """Scores of one query against its visible compressed indexer keys.

    q_idx [H_I, d_I], k_idx [N, d_I], w [H_I].
    S[b] = sum_h w[h] * ReLU(q_idx[h] . k_idx[b]) for b < n_visible(t).
    Returns float64 [n_vis].
    """
    n = n_visible(t, m, k_idx.shape[0])
    dots = k_idx[:n] @ q_idx.T                # [n, H_I]
    return np.maximum(dots, 0.0) @ w


# --------------------------------------------------------------------------
# (2') FP8 indexer: e4m3 codes, one power-of-two scale per row
# --------------------------------------------------------------------------
# "DeepSeek V4 technical review", section 5 (and "Muon Optimizer and FP4 QAT"
# on dataforcee): the indexer's QK product runs in low precision.  Reading
# taken here: keys and indexer queries are stored as OCP FP8 E4M3 codes (max
# 448, round to nearest even) with one power-of-two scale per row (one
# compressed entry, or one (query, head)); the scale 2^e is the smallest with
# max|row| <= 448 * 2^e, so the division by it is exact and rounding to the
# code is the only inexact step.  Scores are the float64 definition applied to
# the dequantised rows.

E4M3_MAX = 448.0


def e4m3_round(y) -> np.ndarray:
    """float64 -> the nearest E4M3 value (ties to even), |y| <= 448.  Normal
    values have 3 fraction bits (exponents -6 .. 8), below 2^-6 the step is
    2^-9 (subnormals)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    if np.any(a > E4M3_MAX):
        raise ValueError("e4m3_round: value beyond 448")
    _, ex = np.frexp(np.where(a > 0, a, 1.0))      # a = f * 2^ex, 0.5 <= f < 1: leading bit 2^(ex-1)
    q = np.maximum(ex - 4, -9)                      # quantum: 2^(ex-1-3), at least 2^-9
    v = np.ldexp(np.round(np.ldexp(a, -q)), q)      # np.round: half to even
    return np.copysign(v, y)


def e4m3_code(v: np.ndarray, sign_of: np.ndarray) -> np.ndarray:
    """Byte codes (sign, 4 exponent bits bias 7, 3 mantissa bits) of E4M3
    values ``v``; the sign bit is taken from ``sign_of`` (so -0 is 0x80)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    lead = ex - 1                                   # a = 1.mmm * 2^lead for normal values
    normal = a >= 2.0 ** -6
    e_field = np.where(normal, lead + 7, 0)
    mant = np.where(normal, np.ldexp(a, -lead) * 8 - 8, np.ldexp(a, 9))
    code = (e_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    return (code | np.where(np.signbit(sign_of), 0x80, 0)).astype(np.uint8)


def quantize_e4m3_rows(x) -> tuple:
    """Rows of x (float64 [R, D]) -> (values on the e4m3 grid [R, D], scales
    [R], byte codes [R, D]); row r is scale[r] * values[r].  scale = 2^e with
    e the smallest integer such that max|x_r| <= 448 * 2^e (e in [-126, 127];
    an all-zero row gets scale 1)."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=1)
    _, ex = np.frexp(np.where(amax > 0, amax, 1.0))
    e = (ex - 1) - 8
    e = np.where(amax > np.ldexp(E4M3_MAX, e), e + 1, e)
    e = np.clip(np.where(amax > 0, e, 0), -126, 127)
    scale = np.ldexp(1.0, e)
    v = e4m3_round(x / scale[:, None])
    return v, scale, e4m3_code(v, x)


def indexer_scores_fp8(qv: np.ndarray, q_scale: np.ndarray, kv: np.ndarray, k_scale: np.ndarray,
                       w: np.ndarray, t: int, m: int) -> np.ndarray:
    """indexer_scores on the dequantised rows: query head h is q_scale[h] *
    qv[h], entry b is k_scale[b] * kv[b] (qv [H_I, d_I], kv [N, d_I] e4m3
    values)."""
    return indexer_scores(qv * q_scale[:, None], kv * k_scale[:, None], w, t, m)


def topk(S: np.ndarray, k: int) -> np.ndarray:
    """Top-k over the visible scores S [n_vis].

    Keeps the min(k, n_vis) entries with the largest score; among equal scores
    the lower index wins.  Returns int32 [k]: the kept indices ascending, then
    -1 padding.
    """
    n = S.shape[0]
    order = np.lexsort((np.arange(n), -S))    # primary: -S, secondary: index
    kept = np.sort(order[: min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[: kept.shape[0]] = kept
    return out


# --------------------------------------------------------------------------
# (4) attention over selected entries + sliding window, and the HCA mode
# --------------------------------------------------------------------------

def window_rows(t: int, W: int, raw_base: int, T_raw: int) -> np.ndarray:
    """Rows of the raw buffer holding tokens u, max(0, t-W+1) <= u <= t."""
    lo = max(0, t - W + 1)
    u = np.arange(lo, t + 1) if W > 0 else np.arange(0)
    r = u - raw_base
    if r.size and (r[0] < 0 or r[-1] >= T_raw):
        raise IndexError("window token outside the raw buffer")
    return r


def attend_one(q: np.ndarray, k_cmp: np.ndarray, v_cmp: np.ndarray,
               sel: Sequence[int], k_raw: np.ndarray, v_raw: np.ndarray,
               win: np.ndarray, scale: float):
    """One query, all heads: one softmax over the union of keys.

    q [H, d]; keys = k_cmp[sel] followed by k_raw[win] (no de-duplication);
    O[h] = sum_j softmax_j(scale * q[h] . K_j) V_j;  lse[h] = log sum_j exp(...).
    An empty key set gives O = 0, lse = -inf.
    """
    sel = np.asarray([s for s in sel if s >= 0], dtype=np.int64)
    K = np.concatenate([k_cmp[sel], k_raw[win]], axis=0)
    V = np.concatenate([v_cmp[sel], v_raw[win]], axis=0)
    H, d = q.shape
    if K.shape[0] == 0:
        return np.zeros((H, d)), np.full(H, -np.inf)
    s = scale * (q @ K.T)                     # [H, L]
    mx = s.max(axis=1, keepdims=True)
    p = np.exp(s - mx)
    l = p.sum(axis=1, keepdims=True)
    O = (p @ V) / l
    lse = (mx + np.log(l))[:, 0]
    return O, lse


# --------------------------------------------------------------------------
# batched entry points (mirror the library's calls)
# --------------------------------------------------------------------------

def csa_compress(x_bits, g_bits, m: int) -> np.ndarray:
    """[B, T, D] bf16 bits -> float64 [B, T//m, D]."""
    x = bf16_to_f64(x_bits)
    g = bf16_to_f64(g_bits)
    return np.stack([compress(x[b], g[b], m) for b in range(x.shape[0])])


def csa_append(x_win_bits, g_win_bits, raw_base, q_pos, m: int) -> List[Dict[int, np.ndarray]]:
    """[B, T_raw, D] bf16 bits -> per sequence {block: float64 [D]}."""
    x = bf16_to_f64(x_win_bits)
    g = bf16_to_f64(g_win_bits)
    return [append_blocks(x[b], g[b], int(raw_base[b]), q_pos[b], m) for b in range(x.shape[0])]


def csa_index_scores(q_idx_bits, k_idx_bits, w, q_pos, m: int) -> List[List[np.ndarray]]:
    """Per (b, query) float64 score vectors over the visible prefix.  ``w`` is
    one [H_I] vector shared by every query, or [B, Tq, H_I]: each query's own
    head weights (the DSA-style indexer produces them per token)."""
    qi = bf16_to_f64(q_idx_bits)
    ki = bf16_to_f64(k_idx_bits)
    w = np.asarray(w, dtype=np.float64)
    out = []
    for b in range(qi.shape[0]):
        out.append([indexer_scores(qi[b, j], ki[b], w if w.ndim == 1 else w[b, j], int(q_pos[b][j]), m)
                    for j in range(qi.shape[1])])
    return out


def csa_index_topk(q_idx_bits, k_idx_bits, w, q_pos, m: int, k: int):
    """Returns (idx int32 [B, Tq, k], scores list) -- steps (2) and (3)."""
    S = csa_index_scores(q_idx_bits, k_idx_bits, w, q_pos, m)
    idx = np.stack([np.stack([topk(s, k) for s in row]) for row in S])
    return idx, S


def csa_attend(q_bits, k_cmp_bits, v_cmp_bits, idx, k_raw_bits, v_raw_bits,
               raw_base, q_pos, W: int, scale: float):
    """Step (4): returns (O float64 [B, Tq, H, d], lse float64 [B, Tq, H])."""
    q = bf16_to_f64(q_bits)
    kc, vc = bf16_to_f64(k_cmp_bits), bf16_to_f64(v_cmp_bits)
    kr, vr = bf16_to_f64(k_raw_bits), bf16_to_f64(v_raw_bits)
    B, Tq, H, d = q.shape
    O = np.zeros((B, Tq, H, d))
    L = np.zeros((B, Tq, H))
    for b in range(B):
        for j in range(Tq):
            t = int(q_pos[b][j])
            win = window_rows(t, W, int(raw_base[b]), kr.shape[1])
            O[b, j], L[b, j] = attend_one(q[b, j], kc[b], vc[b], idx[b][j], kr[b], vr[b], win, scale)
    return O, L


def hca_attend(q_bits, k_cmp_bits, v_cmp_bits, k_raw_bits, v_raw_bits,
               raw_base, q_pos, m: int, W: int, scale: float):
    """HCA mode: every visible compressed entry (no selection) + the window."""
    q = bf16_to_f64(q_bits)
    kc, vc = bf16_to_f64(k_cmp_bits), bf16_to_f64(v_cmp_bits)
    kr, vr = bf16_to_f64(k_raw_bits), bf16_to_f64(v_raw_bits)
    B, Tq, H, d = q.shape
    N = kc.shape[1]
    O = np.zeros((B, Tq, H, d))
    L = np.zeros((B, Tq, H))
    for b in range(B):
        for j in range(Tq):
            t = int(q_pos[b][j])
            sel = np.arange(n_visible(t, m, N))
            win = window_rows(t, W, int(raw_base[b]), kr.shape[1])
            O[b, j], L[b, j] = attend_one(q[b, j], kc[b], vc[b], sel, kr[b], vr[b], win, scale)
    return O, L


def csa_layer_prefill(inp: Dict[str, np.ndarray], m: int, k: int, W: int,
                      scale: Optional[float] = None) -> Dict[str, np.ndarray]:
    """Steps (1)-(4) for prefill: compress K, V and the indexer keys, score,
    select, attend.  ``inp`` holds bf16 bit arrays q, q_idx, k_raw, v_raw,
    i_raw, g_k, g_v, g_i, and w, q_pos, raw_base.  Compressed entries are
    rounded to bf16 before use."""
    d = inp["q"].shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    kc = round_bf16(csa_compress(inp["k_raw"], inp["g_k"], m))
    vc = round_bf16(csa_compress(inp["v_raw"], inp["g_v"], m))
    ic = round_bf16(csa_compress(inp["i_raw"], inp["g_i"], m))
    idx, S = csa_index_topk(inp["q_idx"], ic, inp["w"], inp["q_pos"], m, k)
    O, L = csa_attend(inp["q"], kc, vc, idx, inp["k_raw"], inp["v_raw"],
                      inp["raw_base"], inp["q_pos"], W, scale)
    return {"k_cmp": kc, "v_cmp": vc, "i_cmp": ic, "idx": idx, "scores": S,
            "out": O, "lse": L}
