"""(3) Top-k on the GPU vs the oracle, both fed the same fp32 scores: the
decision is taken in the same precision on both sides, so the indices must be
bit-exact (ties included)."""
import numpy as np
import pytest
import torch

import oracle as O
from long_context_sparse_23_b300 import scores_ld

pytestmark = pytest.mark.gpu


def _run(scores_np, q_pos, N, m, k):
    import long_context_sparse_23_b300 as csa
    B, Tq = q_pos.shape
    ld = scores_ld(N)
    full = np.zeros((B, Tq, ld), np.float32)
    full[:, :, :N] = scores_np
    S = torch.from_numpy(full).cuda()
    qp = torch.from_numpy(q_pos.astype(np.int32)).cuda()
    idx, sel = csa.csa_topk(S, qp, N, m, k, with_scores=True)
    return idx.cpu().numpy(), sel.cpu().numpy()


def _check(scores_np, q_pos, N, m, k):
    idx, sel = _run(scores_np, q_pos, N, m, k)
    B, Tq = q_pos.shape
    for b in range(B):
        for j in range(Tq):
            n = O.n_visible(int(q_pos[b, j]), m, N)
            s = scores_np[b, j, :n].astype(np.float64)
            want = O.topk(s, k)
            np.testing.assert_array_equal(idx[b, j], want, err_msg=f"b={b} j={j} n={n}")
            kept = want[want >= 0]
            np.testing.assert_array_equal(sel[b, j, :len(kept)], scores_np[b, j, kept])


def _normal_scores(rng, B, Tq, N, loc=150.0, sd=30.0):
    return (rng.standard_normal((B, Tq, N)) * sd + loc).astype(np.float32)


def test_topk_tiny_prefill():
    rng = np.random.default_rng(0)
    N, m, k = 64, 4, 16
    q_pos = np.arange(256)[None]
    _check(_normal_scores(rng, 1, 256, N), q_pos, N, m, k)


def test_topk_prefill_8k_sampled_rows():
    rng = np.random.default_rng(1)
    N, m, k = 2048, 4, 1024
    pos = np.concatenate([np.arange(0, 16), rng.integers(0, 8192, 100), np.arange(8180, 8192)])
    _check(_normal_scores(rng, 1, len(pos), N), pos[None], N, m, k)


@pytest.mark.parametrize("N", [32768, 262144, 262144 - 37, 40000])
def test_topk_decode_sizes(N):
    rng = np.random.default_rng(N)
    m, k = 4, 1024
    q_pos = np.array([[4 * N - 1], [4 * N - 2], [4 * N - 5], [2 * N + 3]])
    _check(_normal_scores(rng, 4, 1, N), q_pos, N, m, k)


def test_topk_heavy_ties():
    rng = np.random.default_rng(2)
    N, m, k = 50000, 4, 1024
    q_pos = np.array([[4 * N - 1, 4 * N - 1, 1000, 4 * N - 1]])
    s = rng.integers(0, 4, (1, 4, N)).astype(np.float32)      # four distinct values
    s[0, 1] = 5.0                                              # every score equal
    s[0, 3, ::2] = -0.0                                        # -0 and +0 are the same score
    s[0, 3, 1::2] = 0.0
    _check(s, q_pos, N, m, k)


def test_topk_signs_small_k_and_short_rows():
    rng = np.random.default_rng(3)
    N, m = 3000, 4
    s = (rng.standard_normal((1, 6, N)) * 10).astype(np.float32)   # negative scores too
    q_pos = np.array([[0, 2, 3, 7, 4 * N - 1, 4 * N + 100]])        # n_vis 0, 0, 1, 2, N, N
    for k in (1, 2, 7, 1024, 4096):
        _check(s, q_pos, N, m, k)


def test_topk_bucket_path_with_quantised_ties():
    """Long rows take the 12-bit bucket path; scores on a 1/4 grid put many
    exact ties inside the bucket that holds the k-th score."""
    rng = np.random.default_rng(4)
    N, m, k = 262144, 4, 1024
    s = np.round((rng.standard_normal((3, 1, N)) * 30 + 150) * 4) / 4
    q_pos = np.array([[4 * N - 1], [4 * N - 1], [4 * N - 9]])
    _check(s.astype(np.float32), q_pos, N, m, k)


def test_topk_bucket_overflow_falls_back():
    """A bucket too full to gather (a narrow score range) takes the digit path."""
    rng = np.random.default_rng(5)
    N, m, k = 100000, 4, 1024
    s = (1000.0 + rng.integers(0, 512, (2, 1, N)) / 4096.0).astype(np.float32)
    _check(s, np.array([[4 * N - 1], [4 * N - 1]]), N, m, k)


@pytest.mark.parametrize("N", [16385, 24001, 32768])
def test_topk_mid_rows(N):
    """Rows of 16385..32768 entries: one CTA per query finishes the selection
    from the bucket histogram.  Visible lengths of the whole row, odd lengths
    (scalar loads at the end of the row), just above k and equal to k."""
    rng = np.random.default_rng(100 + N)
    m = 4
    q_pos = np.array([[4 * N - 1], [4 * N - 2], [4 * N - 7], [4 * 1025 - 1], [4 * 1024 - 1], [2 * N + 5]])
    for k in (1, 1024, 4096):
        _check(_normal_scores(rng, 6, 1, N), q_pos, N, m, k)


def test_topk_mid_rows_ties_and_full_buckets():
    """Mid rows with ties inside the k-th score's bucket (kept by lowest
    index), every score equal and a narrow score range (the bucket holds more
    keys than the CTA stages: digit passes over the whole row), and -0 / +0."""
    rng = np.random.default_rng(7)
    N, m, k = 30000, 4, 1024
    s = np.empty((5, 1, N), np.float32)
    s[0, 0] = rng.integers(0, 4, N)                                  # four values, ~7500 each
    s[1, 0] = 5.0                                                    # every score equal
    s[2, 0, ::2] = -0.0
    s[2, 0, 1::2] = 0.0
    s[3, 0] = 1000.0 + rng.integers(0, 512, N) / 4096.0              # one bucket holds the row
    s[4, 0] = np.round((rng.standard_normal(N) * 30 + 150) * 4) / 4  # quarter grid
    _check(s, np.full((5, 1), 4 * N - 1), N, m, k)


def test_topk_mid_rows_one_half_overflows():
    """The two halves of a mid row are selected by the two CTAs of a cluster:
    a first half of equal top scores overflows its candidate list alone (the
    whole row is then selected by digit passes: the lowest indices win), and
    ties at the threshold that straddle the two halves keep the lowest
    indices of the whole row."""
    rng = np.random.default_rng(8)
    N, m, k = 32768, 4, 1024
    s = (rng.standard_normal((3, 1, N)) * 30 + 150).astype(np.float32)
    s[0, 0, :16384] = 1000.0                       # 16384 equal keys in the first half
    s[1, 0, 16000:16800] = 400.0                   # 800 tied top keys across the halves,
    s[1, 0, 100:400] = 400.0                       # 300 more in the first half: 1100 ties > k
    s[2, 0, 16384:16384 + 2000] = 900.0            # the top 2000, all in the second half
    _check(s, np.full((3, 1), 4 * N - 1), N, m, k)
