"""(4)/(5) Decode attention on the tcgen05 kernel (H = 64, d = 128, fewer than 16
queries per sequence) against the oracle, |err| <= 1e-2 + 1e-2 |ref| and lse to
1e-4.

Dense HCA (TMA key tiles, ranges of up to four tiles): one key range (output
written directly), up to eight ranges merged inside their thread-block
cluster and more ranges merged by the combine kernel (some ranges empty for the shorter query), entries that are not a whole number of 128-key tiles, the
window clipped at token 0, the window alone, no window, an empty key set, and
window rows outside the raw buffer.

CSA (gathered rows, ranges of up to five tiles): ragged index lists with
holes, lists spanning several ranges (cluster merge, and the combine kernel
beyond eight), the window alone (k = 0), an empty key set, and indices outside the
entries (flagged and skipped)."""
import math

import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import assert_attention_close, bits
from tests.test_gpu_attend import _attn_case

pytestmark = pytest.mark.gpu


def test_hca_tc_one_range_ragged_entries_and_window_edges():
    """N = 300 entries (2 full tiles + 44), W = 128: 4 tiles, one range.  Positions
    from 0 (one window key) through partial visibility to all entries visible."""
    pos = np.array([[0, 5, 126, 127, 300, 16383, 38399], [1, 128, 255, 4095, 20000, 38398, 39999]])
    _attn_case(31, 2, 7, 300, 64, 128, 0, 128, 128, pos, 40000, 0, hca=True)
    _attn_case(32, 2, 7, 300, 64, 128, 0, 128, 128, pos, 40000, 0, hca=True, out_dtype=torch.float32)


def test_hca_tc_many_ranges_with_empty_ones():
    """140000 entries at m = 1: 1094 + 1 tiles, 274 ranges merged by the combine
    kernel; the second query sees half of them (its later ranges are empty)."""
    pos = np.array([[139999, 70000]])
    _attn_case(33, 1, 2, 140000, 64, 128, 0, 128, 1, pos, 140000, 0, hca=True)


def test_hca_tc_cluster_merged_ranges_with_empty_ones():
    """2000 entries at m = 1 with W = 128: 16 + 1 tiles, 5 ranges merged inside
    their cluster; the second query sees 301 entries (its later ranges are
    empty), the third only its window; bf16 and fp32 outputs."""
    pos = np.array([[1999, 300, 0]])
    _attn_case(37, 1, 3, 2000, 64, 128, 0, 128, 1, pos, 4000, 0, hca=True)
    _attn_case(38, 1, 3, 2000, 64, 128, 0, 128, 1, pos, 4000, 0, hca=True, out_dtype=torch.float32)


def test_hca_tc_two_ranges_of_three_tiles():
    """600 entries at m = 1 with W = 128: 5 + 1 tiles -> 2 ranges of 3 tiles
    merged inside their cluster; queries that see all, some and none of the
    entries."""
    pos = np.array([[599, 200, 0, 383]])
    _attn_case(39, 1, 4, 600, 64, 128, 0, 128, 1, pos, 1200, 0, hca=True)


def test_hca_tc_no_window_and_empty_key_set():
    """W = 0: the compressed entries alone; t < m' - 1 leaves no key at all
    (output 0, lse -inf)."""
    pos = np.array([[0, 126, 127, 5000, 8191]])
    out, lse = _attn_case(34, 1, 5, 64, 64, 128, 0, 0, 128, pos, 64, 0, hca=True)
    assert torch.all(out[0, :2] == 0)
    assert torch.all(torch.isneginf(lse[0, :2]))


def test_hca_tc_window_only_exact_tile():
    """t < m' - 1 with W = 128: only window keys, the first query's window is
    cut at token 0; the raw buffer starts at a non-zero position."""
    pos = np.array([[60, 126], [100, 120]])
    _attn_case(35, 2, 2, 16, 64, 128, 0, 128, 128, pos, 256, -20, hca=True)


def test_hca_tc_window_outside_raw_buffer_is_flagged_and_skipped():
    import long_context_sparse_23_b300 as csa
    B, Tq, N, H, d, m, W, T_raw = 1, 1, 512, 64, 128, 128, 128, 256
    t = 65535
    raw_base = t - 100          # tokens t-127 .. t-101 are not in the buffer
    q = S.normal_bf16(36, 1, (B, Tq, H, d), "cuda")
    kc, vc = S.normal_bf16(36, 10, (B, N, d), "cuda"), S.normal_bf16(36, 11, (B, N, d), "cuda")
    kr, vr = S.normal_bf16(36, 3, (B, T_raw, d), "cuda"), S.normal_bf16(36, 4, (B, T_raw, d), "cuda")
    qp = torch.tensor([[t]], dtype=torch.int32, device="cuda")
    rb = torch.tensor([raw_base], dtype=torch.int32, device="cuda")
    ws = csa.Workspace()
    out, lse = csa.hca_attend(q, kc, vc, kr, vr, rb, qp, m, W, out_dtype=torch.float32, with_lse=True, ws=ws)
    assert ws.check_error() == 2                 # CSA_FLAG_INDEX
    # the result is the attention over the keys that do exist
    f64 = lambda x: O.bf16_to_f64(bits(x.cpu()))
    win = np.arange(t - W + 1, t + 1) - raw_base
    win = win[(win >= 0) & (win < T_raw)]
    ref, ref_lse = O.attend_one(f64(q)[0, 0], f64(kc)[0], f64(vc)[0], np.arange(O.n_visible(t, m, N)),
                                f64(kr)[0], f64(vr)[0], win, 1.0 / math.sqrt(d))
    assert_attention_close(out[0, 0].cpu().numpy(), ref, "hca with a partly missing window")
    np.testing.assert_allclose(lse[0, 0].cpu().numpy(), ref_lse, rtol=1e-4, atol=1e-4)


def test_csa_tc_ragged_lists_with_holes_one_range():
    """k = 100 with -1 holes, W = 37: 137 slots in two tiles; positions with fewer
    visible entries than k; bf16 and fp32 outputs."""
    pos = np.array([[401, 1000, 40000], [999, 5000, 65535]])
    _attn_case(41, 2, 3, 16384, 64, 128, 100, 37, 4, pos, 70000, 0, holes=True)
    _attn_case(42, 2, 3, 16384, 64, 128, 100, 37, 4, pos, 70000, 0, holes=True, out_dtype=torch.float32)


def test_csa_tc_many_ranges():
    """k = 2000, W = 128: 17 tiles -> 4 ranges of at most 5 tiles (two P
    buffers in turn), merged inside their cluster, for 3 queries of one
    sequence; k = 5200: 42 tiles -> 9 ranges, merged by the combine kernel."""
    pos = np.array([[131071, 100000, 9000]])
    _attn_case(43, 1, 3, 32768, 64, 128, 2000, 128, 4, pos, 140000, 0, holes=True)
    _attn_case(47, 1, 3, 32768, 64, 128, 5200, 128, 4, pos, 140000, 0, holes=True, out_dtype=torch.float32)


def test_csa_tc_decode_128k_shape_two_ranges():
    """k = 1000, W = 128 (the shape of decode at 128K context): 9 tiles -> ranges
    of 5 and 4 tiles merged inside their cluster; 2 sequences, ragged lists
    with holes, a query that sees fewer entries than k."""
    pos = np.array([[131071, 3000], [100000, 131071]])
    _attn_case(48, 2, 2, 32768, 64, 128, 1000, 128, 4, pos, 140000, 0, holes=True)
    _attn_case(49, 2, 2, 32768, 64, 128, 1000, 128, 4, pos, 140000, 0, holes=True, out_dtype=torch.float32)


def test_csa_tc_window_only_and_empty():
    """k = 0 (only the window); W = 0 with every slot a hole (no key at all)."""
    import long_context_sparse_23_b300 as csa
    pos = np.array([[0, 50, 127, 128, 3000]])
    _attn_case(44, 1, 5, 64, 64, 128, 0, 128, 4, pos, 4096, 0)
    B, Tq, N, H, d, k = 1, 2, 64, 64, 128, 8
    q = S.normal_bf16(45, 1, (B, Tq, H, d), "cuda")
    kc, vc = S.normal_bf16(45, 10, (B, N, d), "cuda"), S.normal_bf16(45, 11, (B, N, d), "cuda")
    idx = torch.full((B, Tq, k), -1, dtype=torch.int32, device="cuda")
    qp = torch.tensor([[200, 300]], dtype=torch.int32, device="cuda")
    rb = torch.zeros((B,), dtype=torch.int32, device="cuda")
    out, lse = csa.csa_attend(q, kc, vc, idx, kc, vc, rb, qp, 0, out_dtype=torch.float32, with_lse=True)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_csa_tc_bad_indices_are_flagged_and_skipped():
    import long_context_sparse_23_b300 as csa
    B, Tq, N, H, d, k, W = 1, 2, 512, 64, 128, 8, 4
    q = S.normal_bf16(46, 1, (B, Tq, H, d), "cuda")
    kc, vc = S.normal_bf16(46, 10, (B, N, d), "cuda"), S.normal_bf16(46, 11, (B, N, d), "cuda")
    kr, vr = S.normal_bf16(46, 3, (B, 32, d), "cuda"), S.normal_bf16(46, 4, (B, 32, d), "cuda")
    idx = torch.tensor([[[0, 5, N + 3, 9, -1, 2, 7, 1], [1, 2, 3, 4, 5, 6, 7, 8]]], dtype=torch.int32, device="cuda")
    qp = torch.tensor([[2000, 2000]], dtype=torch.int32, device="cuda")
    rb = torch.tensor([1980], dtype=torch.int32, device="cuda")  # window rows 17..20 exist
    ws = csa.Workspace()
    out = csa.csa_attend(q, kc, vc, idx, kr, vr, rb, qp, W, ws=ws)
    assert ws.check_error() == 2                # CSA_FLAG_INDEX
    clean = idx.clone()
    clean[0, 0, 2] = -1
    out2 = csa.csa_attend(q, kc, vc, clean, kr, vr, rb, qp, W, ws=ws)
    assert ws.check_error() == 0
    assert torch.equal(out, out2)
    # a window that falls outside the raw buffer is flagged too
    csa.csa_attend(q, kc, vc, clean, kr, vr, torch.tensor([1990], dtype=torch.int32, device="cuda"), qp, W + 10,
                   ws=ws)
    assert ws.check_error() == 2
