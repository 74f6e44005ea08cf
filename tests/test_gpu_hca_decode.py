"""(5) Dense HCA attention, decode-shaped calls with H = 64 and d = 128: the
tcgen05 kernel (TMA key tiles, scores and output accumulated in tensor memory)
against the oracle, |err| <= 1e-2 + 1e-2 |ref| and lse to 1e-4.  Covers one
key range (output written directly), many ranges with partials merged by the
combine kernel (some ranges empty for the shorter query), entries that are not
a whole number of 128-key tiles, the window clipped at token 0, the window
alone, no window, an empty key set, and window rows outside the raw buffer."""
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
