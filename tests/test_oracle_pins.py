"""Pins for the CPU oracle: checks against hand-worked values, closed forms,
invariants, brute force and library routines -- never against the oracle's own
formulas retyped.  CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle as O
from oracle import ref_cpp


@pytest.fixture(scope="module", params=["numpy", "cpp"])
def OC(request):
    """The oracle under test: the numpy oracle, or the C++ oracle (same call
    signatures).  Both are held to the same pins."""
    if request.param == "cpp":
        ref_cpp.build()
        return ref_cpp
    return O


def _rows(s):
    return np.array([[float(v) for v in r.split()] for r in s.split("|")])


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_ties_and_single_rounding():
    one = np.float64(1.0)
    cases = {
        one + 2 ** -8: 1.0,                        # tie -> even (1.0)
        one + 3 * 2 ** -8: 1.0 + 2 ** -6,          # tie -> even (1 + 2^-6)
        one + 2 ** -8 + 2 ** -40: 1.0 + 2 ** -7,   # just above the tie: up (a second
                                                   # rounding through fp32 would give 1.0)
        -(one + 2 ** -8 + 2 ** -40): -(1.0 + 2 ** -7),
    }
    for x, want in cases.items():
        got = O.bf16_to_f64(O.round_bf16(np.array([x])))[0]
        assert got == want, (x, got, want)


# ---------------------------------------------------------------- (1) compression

def test_compress_golden_m2(OC, golden_dir):
    for ln in _load(golden_dir, "compress_m2.txt"):
        p = [s for s in ln.split("|")]
        x = np.array([[float(v) for v in p[0].split()], [float(v) for v in p[1].split()]])
        g = np.array([[float(v) for v in p[2].split()], [float(v) for v in p[3].split()]])
        want = np.array([float(v) for v in p[4].split()])
        got = OC.compress(x, g, 2)
        assert got.shape == (1, 2)
        np.testing.assert_allclose(got[0], want, rtol=0, atol=1e-14)


def test_compress_invariants(OC):
    rng = np.random.default_rng(1)
    T, D, m = 64, 8, 4
    x = rng.standard_normal((T, D))
    g = rng.standard_normal((T, D)) * 3
    base = OC.compress(x, g, m)
    # adding one constant per (block, channel) to the gates changes nothing
    shift = np.repeat(rng.standard_normal((T // m, D)) * 50, m, axis=0)
    np.testing.assert_allclose(OC.compress(x, g + shift, m), base, rtol=1e-12, atol=1e-12)
    # a stream constant within each block is reproduced exactly
    c = np.repeat(rng.standard_normal((T // m, D)), m, axis=0)
    np.testing.assert_allclose(OC.compress(c, g, m), c[::m], rtol=1e-13, atol=1e-13)
    # permuting tokens inside a block (with their gates) changes nothing
    perm = np.concatenate([b * m + rng.permutation(m) for b in range(T // m)])
    np.testing.assert_allclose(OC.compress(x[perm], g[perm], m), base, rtol=1e-12, atol=1e-12)
    # a convex combination: inside [min, max] of the block
    X = x.reshape(T // m, m, D)
    assert np.all(base <= X.max(axis=1) + 1e-12) and np.all(base >= X.min(axis=1) - 1e-12)
    # m = 1 is the identity
    np.testing.assert_array_equal(OC.compress(x, g, 1), x)
    # a trailing partial block is dropped
    assert OC.compress(x[:T - 3], g[:T - 3], m).shape == (T // m - 1, D)
    # one dominant gate selects its token
    g2 = np.zeros((T, D))
    g2[2::m] = 800.0
    np.testing.assert_allclose(OC.compress(x, g2, m), x[2::m], rtol=0, atol=1e-300)


# ---------------------------------------------------------------- visibility

@pytest.mark.parametrize("m", [1, 2, 4, 128])
def test_n_visible_boundaries(OC, m):
    N = 10
    if m >= 2:
        assert OC.n_visible(m - 2, m, N) == 0      # first block not yet complete
    assert OC.n_visible(m - 1, m, N) == 1          # first block complete at t = m-1
    assert OC.n_visible(2 * m - 2, m, N) == 1      # second block one token short
    assert OC.n_visible(2 * m - 1, m, N) == 2
    assert OC.n_visible(100 * m, m, N) == N        # capped by the blocks that exist
    assert OC.n_visible(-1, m, N) == 0


# ---------------------------------------------------------------- (2)+(3) indexer, top-k

def test_indexer_golden_and_tie(OC, golden_dir):
    lines = _load(golden_dir, "indexer_tie.txt")
    kv = dict(ln.split("=", 1) for ln in lines if "=" in ln)
    w = np.array([float(v) for v in kv["w "].split()])
    q = _rows(kv["q "])
    keys = _rows(kv["keys "])
    want_scores = np.array([float(v) for v in kv["scores "].split()])
    np.testing.assert_array_equal(OC.indexer_scores(q, keys, w, t=100, m=1), want_scores)
    cases = [ln for ln in lines if "=" not in ln]
    assert len(cases) == 5
    for ln in cases:
        a, b = ln.split("|")
        m, t, k = (int(v) for v in a.split())
        want = np.array([int(v) for v in b.split()])
        S = OC.indexer_scores(q, keys, w, t=t, m=m)
        np.testing.assert_array_equal(OC.topk(S, k), want)


def test_indexer_homogeneity_and_positive_closed_form(OC):
    rng = np.random.default_rng(2)
    H, d, N = 6, 16, 40
    q = rng.standard_normal((H, d))
    k = rng.standard_normal((N, d))
    w = rng.uniform(0, 1, H)
    S = OC.indexer_scores(q, k, w, t=10 ** 6, m=1)
    # ReLU is positively homogeneous: scaling q by a > 0 scales S by a
    np.testing.assert_allclose(OC.indexer_scores(2.5 * q, k, w, 10 ** 6, 1), 2.5 * S, rtol=1e-13)
    # with non-negative q and k every ReLU is the identity, so
    # S[b] = (sum_h w_h q_h) . k_b  -- one dot product with the weighted query
    qp, kp = np.abs(q), np.abs(k)
    closed = np.array([np.dot(w @ qp, kp[b]) for b in range(N)])
    np.testing.assert_allclose(OC.indexer_scores(qp, kp, w, 10 ** 6, 1), closed, rtol=1e-13)
    # with non-positive dots every term vanishes
    np.testing.assert_array_equal(OC.indexer_scores(qp, -kp, w, 10 ** 6, 1), np.zeros(N))


def _brute_topk(S, k):
    """argmax over all k-subsets of (sum of scores, -sum of indices)."""
    n = len(S)
    kk = min(k, n)
    best = max(itertools.combinations(range(n), kk),
               key=lambda c: (sum(S[i] for i in c), -sum(c)))
    out = np.full(k, -1)
    out[:kk] = sorted(best)
    return out


def test_topk_brute_force_with_ties(OC):
    rng = np.random.default_rng(3)
    for trial in range(300):
        n = int(rng.integers(0, 9))
        k = int(rng.integers(1, 6))
        # small integer scores force many ties; halves keep sums exact
        S = rng.integers(0, 4, n).astype(np.float64) * 0.5
        np.testing.assert_array_equal(OC.topk(S, k), _brute_topk(S, k), err_msg=str((S, k)))


def test_topk_never_selects_future_blocks(OC):
    rng = np.random.default_rng(4)
    H, d, N, m = 4, 8, 32, 4
    q = np.abs(rng.standard_normal((H, d)))
    k = np.abs(rng.standard_normal((N, d)))
    k[N // 2:] *= 1000.0                     # future blocks score far higher
    w = np.ones(H)
    for t in range(0, N * m):
        idx = OC.topk(OC.indexer_scores(q, k, w, t, m), 5)
        sel = idx[idx >= 0]
        assert len(sel) == min(5, (t + 1) // m)
        assert np.all((sel + 1) * m - 1 <= t)


# ---------------------------------------------------------------- (4) attention

def test_attend_golden_two_keys(OC, golden_dir):
    kv = dict(ln.split("=", 1) for ln in _load(golden_dir, "attend_2key.txt"))
    q = np.array([[float(v) for v in kv["q "].split()]])
    K, V = _rows(kv["K "]), _rows(kv["V "])
    out, lse = OC.attend_one(q, K, V, [0, 1], K[:0], V[:0], np.arange(0), 1 / math.sqrt(2))
    np.testing.assert_allclose(out[0], [float(v) for v in kv["O "].split()], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0], float(kv["lse "]), rtol=0, atol=1e-15)
    # the same two keys reached through the window branch give the same result
    out2, _ = OC.attend_one(q, K[:0], V[:0], [], K, V, np.arange(2), 1 / math.sqrt(2))
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-15)


def test_attend_special_cases(OC):
    rng = np.random.default_rng(5)
    H, d = 3, 8
    q = rng.standard_normal((H, d))
    K = rng.standard_normal((5, d))
    V = rng.standard_normal((5, d))
    empty = np.arange(0)
    # one key -> its value
    o1, l1 = OC.attend_one(q, K, V, [3], K[:0], V[:0], empty, 0.3)
    np.testing.assert_allclose(o1, np.repeat(V[3:4], H, 0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(l1, 0.3 * q @ K[3], rtol=1e-14)
    # equal logits (q = 0) -> mean of the values
    o2, l2 = OC.attend_one(np.zeros((H, d)), K, V, [0, 1, 2, 3, 4], K[:0], V[:0], empty, 0.3)
    np.testing.assert_allclose(o2, np.repeat(V.mean(0, keepdims=True), H, 0), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(l2, np.full(H, math.log(5)), rtol=1e-14)
    # -1 entries are skipped; no keys at all -> zeros and -inf
    o3, l3 = OC.attend_one(q, K, V, [-1, -1], K[:0], V[:0], empty, 0.3)
    assert np.all(o3 == 0) and np.all(np.isneginf(l3))
    # lse agrees with scipy's logsumexp
    _, l4 = OC.attend_one(q, K, V, [4, 0, 2], K, V, np.array([1, 2]), 0.3)
    keys = np.concatenate([K[[4, 0, 2]], K[[1, 2]]])
    np.testing.assert_allclose(l4, logsumexp(0.3 * q @ keys.T, axis=1), rtol=1e-14)


def _sdpa(q, K, V, mask, scale):
    """torch's scaled_dot_product_attention in float64; q [T,H,d], K/V [L,d]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]           # [1,H,T,d]
    kt = torch.from_numpy(K)[None, None].expand(1, q.shape[1], -1, -1)
    vt = torch.from_numpy(V)[None, None].expand(1, q.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask)[None, None], scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def _bits(x):
    return O.round_bf16(x)


def test_csa_reduces_to_causal_attention_at_m1(OC):
    """m = 1, k >= n_vis, W = 0: CSA is textbook causal softmax attention."""
    rng = np.random.default_rng(6)
    T, H, d, HI, dI = 24, 2, 8, 2, 4
    q = _bits(rng.standard_normal((1, T, H, d)))
    kr = _bits(rng.standard_normal((1, T, d)))
    vr = _bits(rng.standard_normal((1, T, d)))
    g = _bits(rng.standard_normal((1, T, d)))
    inp = dict(q=q, q_idx=_bits(rng.standard_normal((1, T, HI, dI))), k_raw=kr, v_raw=vr,
               i_raw=_bits(rng.standard_normal((1, T, dI))), g_k=g, g_v=g, g_i=_bits(rng.standard_normal((1, T, dI))),
               w=rng.uniform(0, 1, HI), q_pos=np.arange(T)[None], raw_base=np.zeros(1, np.int64))
    res = O.csa_layer_prefill(inp, m=1, k=T, W=0, scale=0.25)
    mask = np.tril(np.ones((T, T), dtype=bool))
    ref = _sdpa(O.bf16_to_f64(q[0]), O.bf16_to_f64(kr[0]), O.bf16_to_f64(vr[0]), mask, 0.25)
    np.testing.assert_allclose(res["out"][0], ref, rtol=1e-12, atol=1e-12)


def test_hca_is_block_causal_dense_attention_and_csa_agrees(OC):
    rng = np.random.default_rng(7)
    N, m, H, d, T = 12, 4, 2, 8, 48
    q = _bits(rng.standard_normal((1, T, H, d)))
    kc = _bits(rng.standard_normal((1, N, d)))
    vc = _bits(rng.standard_normal((1, N, d)))
    kr = _bits(rng.standard_normal((1, T, d)))
    pos = np.arange(T)[None]
    base = np.zeros(1, np.int64)
    o_h, _ = OC.hca_attend(q, kc, vc, kr, kr, base, pos, m, 0, 0.3)
    # (b+1)*m - 1 <= t, written as a boolean table
    mask = np.array([[(b + 1) * m - 1 <= t for b in range(N)] for t in range(T)])
    rows = mask.any(1)
    ref = _sdpa(O.bf16_to_f64(q[0]), O.bf16_to_f64(kc[0]), O.bf16_to_f64(vc[0]), mask, 0.3)
    np.testing.assert_allclose(o_h[0][rows], ref[rows], rtol=1e-12, atol=1e-12)
    assert np.all(o_h[0][~rows] == 0)
    # CSA with every visible block selected equals HCA
    idx = np.full((1, T, N), -1)
    for t in range(T):
        nv = OC.n_visible(t, m, N)
        idx[0, t, :nv] = np.arange(nv)
    o_c, _ = OC.csa_attend(q, kc, vc, idx, kr, kr, base, pos, 0, 0.3)
    np.testing.assert_allclose(o_c, o_h, rtol=0, atol=1e-15)


def test_window_only_is_banded_attention(OC):
    """n_vis = 0 (t < m-1 of a huge m) leaves the sliding window alone."""
    rng = np.random.default_rng(8)
    T, H, d, W = 20, 2, 8, 5
    q = _bits(rng.standard_normal((1, T, H, d)))
    kr = _bits(rng.standard_normal((1, T, d)))
    vr = _bits(rng.standard_normal((1, T, d)))
    kc = _bits(np.zeros((1, 0, d)))
    o, _ = OC.hca_attend(q, kc, kc, kr, vr, np.zeros(1, np.int64), np.arange(T)[None], 128, W, 0.4)
    mask = np.array([[t - W < u <= t for u in range(T)] for t in range(T)])
    ref = _sdpa(O.bf16_to_f64(q[0]), O.bf16_to_f64(kr[0]), O.bf16_to_f64(vr[0]), mask, 0.4)
    np.testing.assert_allclose(o[0], ref, rtol=1e-12, atol=1e-12)
    # window rows honour the raw buffer's base position
    assert list(O.window_rows(10, 4, 5, 100)) == [2, 3, 4, 5]
    assert list(O.window_rows(1, 4, 0, 100)) == [0, 1]
    with pytest.raises(IndexError):
        O.window_rows(10, 4, 8, 100)


# ---------------------------------------------------------------- batched wrappers

def _rand_bf16(rng, shape):
    return O.round_bf16(rng.standard_normal(shape))


def test_batched_wrappers_equal_each_sequence_alone(OC):
    """B = 3 sequences with different inputs, positions and window offsets:
    every batched wrapper returns, for sequence b, exactly what it returns for
    that sequence alone (B = 1, itself pinned by the reductions above), and
    the three sequences' results differ, so a wrapper that paired one
    sequence's tensor with another's (or read sequence 0 for all) fails."""
    rng = np.random.default_rng(11)
    B, T, m, H, d, HI, dI, k, W = 3, 64, 4, 2, 8, 3, 4, 5, 6
    N = T // m
    x, g = _rand_bf16(rng, (B, T, d)), _rand_bf16(rng, (B, T, d))
    xi, gi = _rand_bf16(rng, (B, T, dI)), _rand_bf16(rng, (B, T, dI))
    q, qi = _rand_bf16(rng, (B, 2, H, d)), _rand_bf16(rng, (B, 2, HI, dI))
    w = rng.uniform(0, 1, HI)
    q_pos = np.array([[63, 50], [61, 45], [59, 47]])
    T_raw = 24
    raw_base = np.array([T - T_raw, T - T_raw - 2, T - T_raw - 4])
    kr, vr = _rand_bf16(rng, (B, T_raw, d)), _rand_bf16(rng, (B, T_raw, d))
    # window rows must exist for every query: t - W + 1 >= raw_base, t < raw_base + T_raw
    for b in range(B):
        for t in q_pos[b]:
            assert t - W + 1 >= raw_base[b] and t < raw_base[b] + T_raw
    scale = 0.3

    kc = OC.csa_compress(x, g, m)
    ic = OC.csa_compress(xi, gi, m)
    kcb, icb = O.round_bf16(kc), O.round_bf16(ic)
    idx, S = OC.csa_index_topk(qi, icb, w, q_pos, m, k)
    Oc, Lc = OC.csa_attend(q, kcb, kcb, idx, kr, vr, raw_base, q_pos, W, scale)
    Oh, Lh = OC.hca_attend(q, kcb, kcb, kr, vr, raw_base, q_pos, m, W, scale)
    for b in range(B):
        one = slice(b, b + 1)
        np.testing.assert_array_equal(kc[b], OC.csa_compress(x[one], g[one], m)[0])
        idx1, S1 = OC.csa_index_topk(qi[one], icb[one], w, q_pos[one], m, k)
        np.testing.assert_array_equal(idx[b], idx1[0])
        for j in range(2):
            np.testing.assert_array_equal(S[b][j], S1[0][j])
        o1, l1 = OC.csa_attend(q[one], kcb[one], kcb[one], idx[one], kr[one], vr[one], raw_base[one],
                              q_pos[one], W, scale)
        np.testing.assert_array_equal(Oc[b], o1[0])
        np.testing.assert_array_equal(Lc[b], l1[0])
        o1, l1 = OC.hca_attend(q[one], kcb[one], kcb[one], kr[one], vr[one], raw_base[one], q_pos[one], m, W,
                              scale)
        np.testing.assert_array_equal(Oh[b], o1[0])
        np.testing.assert_array_equal(Lh[b], l1[0])
    for res in (kc, idx, Oc, Oh):
        assert not np.array_equal(res[0], res[1]) and not np.array_equal(res[1], res[2])
    # the window really reaches into each sequence's own raw buffer: the HCA
    # output of query (1, 1) changes when only sequence 1's window rows change
    vr2 = vr.copy()
    vr2[1] = _rand_bf16(rng, (T_raw, d))
    Oh2, _ = OC.hca_attend(q, kcb, kcb, kr, vr2, raw_base, q_pos, m, W, scale)
    assert not np.array_equal(Oh2[1], Oh[1])
    np.testing.assert_array_equal(Oh2[0], Oh[0])
    np.testing.assert_array_equal(Oh2[2], Oh[2])


# ---------------------------------------------------------------- decode-time append

def test_append_golden_m2(golden_dir):
    """A window whose last two tokens complete a block reproduces the
    hand-worked m = 2 values; a position that completes no block appends
    nothing."""
    for ln in _load(golden_dir, "compress_m2.txt"):
        p = ln.split("|")
        x = np.array([[float(v) for v in p[0].split()], [float(v) for v in p[1].split()]])
        g = np.array([[float(v) for v in p[2].split()], [float(v) for v in p[3].split()]])
        want = np.array([float(v) for v in p[4].split()])
        # window rows hold tokens 10, 11 (raw_base 10); t = 11 completes block 5
        got = O.append_blocks(x, g, 10, [11], 2)
        assert list(got) == [5]
        np.testing.assert_allclose(got[5], want, rtol=0, atol=1e-14)
        assert O.append_blocks(x, g, 10, [10], 2) == {}


def test_append_equals_prefill_compression_of_the_same_block():
    """Every block a decode step completes equals the entry that compressing
    the whole stream gives for it (the prefill path), for windows at several
    offsets and a step with several queries."""
    rng = np.random.default_rng(5)
    T, D, m, T_raw = 96, 8, 4, 20
    x, g = rng.standard_normal((T, D)), rng.standard_normal((T, D)) * 2
    full = O.compress(x, g, m)
    for t_last in (19, 43, 44, 63, 95):
        raw_base = t_last + 1 - T_raw
        pos = [t_last - 5, t_last - 2, t_last]      # a step of three queries
        got = O.append_blocks(x[raw_base:t_last + 1], g[raw_base:t_last + 1], raw_base, pos, m)
        assert sorted(got) == sorted((t + 1) // m - 1 for t in pos if (t + 1) % m == 0)
        for b, v in got.items():
            np.testing.assert_array_equal(v, full[b])


# ---------------------------------------------------------------- per-query indexer weights

def test_per_query_weights():
    """[B, Tq, H_I] weights: a query whose weights equal the shared vector
    scores as with the shared vector; a one-hot weight vector scores
    ReLU(q_h . k) of that head alone (closed form); weights of mixed sign give
    sum_h w_h ReLU(.) with negative scores allowed, and top-k still keeps the
    largest (ties to the lower index, checked by brute force)."""
    rng = np.random.default_rng(21)
    B, Tq, HI, dI, N, m = 2, 3, 4, 8, 40, 4
    qi = O.round_bf16(rng.standard_normal((B, Tq, HI, dI)))
    ki = O.round_bf16(rng.standard_normal((B, N, dI)))
    q_pos = np.array([[159, 100, 57], [159, 120, 3]])
    w_shared = rng.uniform(0, 1, HI)
    w_q = np.broadcast_to(w_shared, (B, Tq, HI)).copy()
    S_shared = O.csa_index_scores(qi, ki, w_shared, q_pos, m)
    S_q = O.csa_index_scores(qi, ki, w_q, q_pos, m)
    for b in range(B):
        for j in range(Tq):
            np.testing.assert_array_equal(S_q[b][j], S_shared[b][j])
    # one-hot per query: head j % HI of query j
    w_oh = np.zeros((B, Tq, HI))
    for j in range(Tq):
        w_oh[:, j, j % HI] = 1.0
    S_oh = O.csa_index_scores(qi, ki, w_oh, q_pos, m)
    q64, k64 = O.bf16_to_f64(qi), O.bf16_to_f64(ki)
    for b in range(B):
        for j in range(Tq):
            n = O.n_visible(int(q_pos[b, j]), m, N)
            want = [max(0.0, sum(q64[b, j, j % HI, c] * k64[b, i, c] for c in range(dI))) for i in range(n)]
            np.testing.assert_allclose(S_oh[b][j], want, rtol=1e-12, atol=1e-12)
    # mixed signs: some scores negative; top-k by brute force over the key order
    w_mix = rng.uniform(-1, 1, (B, Tq, HI))
    S_mix = O.csa_index_scores(qi, ki, w_mix, q_pos, m)
    assert min(v.min() for row in S_mix for v in row if v.size) < 0
    for row in S_mix:
        for v in row:
            k = 5
            order = sorted(range(len(v)), key=lambda i: (-v[i], i))[:k]
            got = O.topk(v, k)
            assert list(got[got >= 0]) == sorted(order)


# ---------------------------------------------------------------- FP8 (e4m3) indexer

def test_e4m3_rounding_matches_torch():
    """Round-to-nearest-even onto the E4M3 grid (normals, subnormals, exact
    ties) and the byte codes, against torch's float8_e4m3fn conversion."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal(200000) * np.exp2(rng.uniform(-12, 8.7, 200000))
    x = np.clip(x, -448, 448).astype(np.float32).astype(np.float64)
    grid = O.e4m3_round(np.arange(-448, 449, dtype=np.float64))             # all are integers or on the grid
    ties = (grid[1:] + grid[:-1]) / 2                                       # midpoints: exact ties
    sub = np.arange(0, 8) * 2.0 ** -9 + 2.0 ** -10                          # subnormal ties
    x = np.concatenate([x, ties, -ties, sub, -sub, [0.0, -0.0, 448.0, -448.0, 2.0 ** -6, 2.0 ** -9]])
    t = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)       # every input is exact in fp32
    np.testing.assert_array_equal(O.e4m3_round(x), t.float().numpy().astype(np.float64))
    np.testing.assert_array_equal(O.e4m3_code(O.e4m3_round(x), x), t.view(torch.uint8).numpy())


def test_e4m3_row_quantisation():
    """Scale 2^e, the smallest with max|row| <= 448 * 2^e: the largest code
    magnitude lies in [224, 448] (max|row| / 2^e in (224, 448] before the
    rounding); dequantised values within half a step
    (2^-4 relative for normal codes) of the input; an all-zero row keeps
    scale 1 and zero codes; scales are exact powers of two."""
    rng = np.random.default_rng(4)
    x = O.bf16_to_f64(O.round_bf16(rng.standard_normal((300, 128)) * np.exp2(rng.uniform(-20, 20, (300, 1)))))
    x[7] = 0.0
    v, s, c = O.quantize_e4m3_rows(x)
    nz = np.abs(x).max(axis=1) > 0
    top = np.abs(v).max(axis=1)
    assert np.all((top[nz] >= 224) & (top[nz] <= 448))
    pre = np.abs(x).max(axis=1)[nz] / s[nz]
    assert np.all((pre > 224) & (pre <= 448))
    assert s[7] == 1.0 and not c[7].any() and not v[7].any()
    assert np.all(np.frexp(s)[0] == 0.5)                                     # powers of two
    normal = np.abs(v) >= 2.0 ** -6
    rel = np.abs(v * s[:, None] - x)[normal] / np.abs(x)[normal]
    assert rel.max() <= 2.0 ** -4 + 1e-15
    # the codes decode to the values (torch's e4m3 decoding of the bytes)
    dec = torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(dec, v)


def test_fp8_scores_reduce_to_the_definition():
    """With rows already on the E4M3 grid the quantisation is exact (up to the
    power-of-two scale), so the FP8 scores equal indexer_scores of the
    original rows; in general they equal indexer_scores of the dequantised
    rows (checked against a brute-force double loop)."""
    rng = np.random.default_rng(6)
    H, d, N, m, t = 3, 16, 24, 4, 95
    qg = O.e4m3_round(np.clip(rng.standard_normal((H, d)) * 8, -448, 448))
    kg = O.e4m3_round(np.clip(rng.standard_normal((N, d)) * 8, -448, 448))
    w = rng.uniform(0, 1, H)
    qv, qs, _ = O.quantize_e4m3_rows(qg)
    kv, ks, _ = O.quantize_e4m3_rows(kg)
    np.testing.assert_allclose(O.indexer_scores_fp8(qv, qs, kv, ks, w, t, m), O.indexer_scores(qg, kg, w, t, m),
                               rtol=1e-14, atol=0)
    q, k = rng.standard_normal((H, d)), rng.standard_normal((N, d))
    qv, qs, _ = O.quantize_e4m3_rows(q)
    kv, ks, _ = O.quantize_e4m3_rows(k)
    got = O.indexer_scores_fp8(qv, qs, kv, ks, w, t, m)
    n = O.n_visible(t, m, N)
    for b in range(n):
        want = 0.0
        for h in range(H):
            dot = sum((qs[h] * qv[h, c]) * (ks[b] * kv[b, c]) for c in range(d))
            want += w[h] * max(dot, 0.0)
        assert abs(got[b] - want) <= 1e-12 * (1 + abs(want))
