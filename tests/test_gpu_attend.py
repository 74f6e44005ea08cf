"""(4) Attention over selected entries + window (CSA) and the dense HCA mode on
the GPU vs the oracle, both given the same index sets: |err| <= 1e-2 + 1e-2|ref|."""
import math

import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import assert_attention_close, bits, random_selection

pytestmark = pytest.mark.gpu


def _mk(seed, shape, tid, device):
    return S.normal_bf16(seed, tid, shape, device)


def _attn_case(seed, B, Tq, N, H, d, k, W, m, pos, T_raw, raw_base, hca=False, holes=False,
               rows=None, out_dtype=torch.bfloat16):
    import long_context_sparse_23_b300 as csa
    rng = np.random.default_rng(seed)
    pos = np.asarray(pos, np.int64)
    idx = None
    if not hca:
        idx = np.stack([np.stack([random_selection(rng, O.n_visible(int(pos[b, j]), m, N), k, holes)
                                  for j in range(Tq)]) for b in range(B)])
    tens = {}
    for dev in ("cuda", "cpu"):
        tens[dev] = dict(q=_mk(seed, (B, Tq, H, d), 1, dev), kc=_mk(seed, (B, N, d), 10, dev),
                         vc=_mk(seed, (B, N, d), 11, dev), kr=_mk(seed, (B, T_raw, d), 3, dev),
                         vr=_mk(seed, (B, T_raw, d), 4, dev))
    g = tens["cuda"]
    qp = torch.from_numpy(pos.astype(np.int32)).cuda()
    rb = torch.full((B,), raw_base, dtype=torch.int32, device="cuda")
    if hca:
        out, lse = csa.hca_attend(g["q"], g["kc"], g["vc"], g["kr"], g["vr"], rb, qp, m, W,
                                  out_dtype=out_dtype, with_lse=True)
    else:
        it = torch.from_numpy(idx).cuda()
        out, lse = csa.csa_attend(g["q"], g["kc"], g["vc"], it, g["kr"], g["vr"], rb, qp, W,
                                  out_dtype=out_dtype, with_lse=True)
    torch.cuda.synchronize()
    c = tens["cpu"]
    out_np = out.float().cpu().numpy()
    lse_np = lse.cpu().numpy()
    scale = 1.0 / math.sqrt(d)
    rows = rows if rows is not None else [(b, j) for b in range(B) for j in range(Tq)]
    q64, kc64, vc64 = O.bf16_to_f64(bits(c["q"])), O.bf16_to_f64(bits(c["kc"])), O.bf16_to_f64(bits(c["vc"]))
    kr64, vr64 = O.bf16_to_f64(bits(c["kr"])), O.bf16_to_f64(bits(c["vr"]))
    for b, j in rows:
        t = int(pos[b, j])
        win = O.window_rows(t, W, raw_base, T_raw)
        sel = np.arange(O.n_visible(t, m, N)) if hca else idx[b, j]
        ref, ref_lse = O.attend_one(q64[b, j], kc64[b], vc64[b], sel, kr64[b], vr64[b], win, scale)
        assert_attention_close(out_np[b, j], ref, f"out b={b} j={j}")
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse_np[b, j])), f"lse finiteness b={b} j={j}"
        np.testing.assert_allclose(lse_np[b, j][fin], ref_lse[fin], rtol=1e-4, atol=1e-4)
    return out, lse


def test_attend_tiny_prefill():
    """H=4 (padded head group), d=64, 64 entries, top-16, W=32, every position."""
    _attn_case(0, 1, 256, 64, 4, 64, 16, 32, 4, np.arange(256)[None], 256, 0)


def test_attend_prefill_8k_sampled():
    """H=16 (one head group, four key sub-ranges per tile), top-1024, W=128."""
    rng = np.random.default_rng(1)
    rows = [(0, int(j)) for j in np.concatenate([np.arange(8), rng.integers(0, 8192, 120), np.arange(8184, 8192)])]
    _attn_case(1, 1, 8192, 2048, 16, 128, 1024, 128, 4, np.arange(8192)[None], 8192, 0, rows=rows)


def test_attend_decode_128k_full():
    """B=64, H=64, 1024 selected + 128 window keys, split over key ranges."""
    _attn_case(2, 64, 1, 32768, 64, 128, 1024, 128, 4, np.full((64, 1), 131071), 256, 131072 - 256)


def test_attend_decode_1m_tail_holes_f32():
    """B=4 x 4 tail queries, -1 holes inside the index lists, fp32 output."""
    pos = np.array([list(range((1 << 20) - 4, 1 << 20))] * 4)
    _attn_case(4, 4, 4, 262144, 64, 128, 1024, 128, 4, pos, 256, (1 << 20) - 256, holes=True,
               out_dtype=torch.float32)


def test_hca_decode_1m_given_entries():
    """B=8, 8192 entries (m'=128) all visible + 128 window keys."""
    _attn_case(3, 8, 1, 8192, 64, 128, 0, 128, 128, np.full((8, 1), (1 << 20) - 1), 256, (1 << 20) - 256, hca=True)


def test_hca_short_positions_and_window_edges():
    """t < m'-1 (window only), window clipped at token 0, partial visibility."""
    pos = np.array([[0, 5, 126, 127, 300, 1000, 4095]])
    _attn_case(6, 1, 7, 32, 32, 64, 0, 128, 128, pos, 4096, 0, hca=True)


def test_csa_empty_and_window_only():
    """W = 0 with nothing visible -> 0 / -inf; k > n_vis; window only."""
    pos = np.array([[0, 1, 2, 3, 9, 40]])
    out, lse = _attn_case(8, 1, 6, 16, 16, 64, 8, 0, 4, pos, 64, 0)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.all(o[0, :3] == 0) and np.all(np.isneginf(l[0, :3]))
    _attn_case(9, 1, 6, 16, 16, 64, 8, 5, 4, pos, 64, 0)


def test_attend_bad_indices_are_flagged_and_skipped():
    import long_context_sparse_23_b300 as csa
    B, Tq, N, H, d, k, W = 1, 2, 64, 16, 64, 8, 4
    q = _mk(11, (B, Tq, H, d), 1, "cuda")
    kc, vc = _mk(11, (B, N, d), 10, "cuda"), _mk(11, (B, N, d), 11, "cuda")
    kr, vr = _mk(11, (B, 32, d), 3, "cuda"), _mk(11, (B, 32, d), 4, "cuda")
    idx = torch.tensor([[[0, 5, N + 3, 9, -1, 2, 7, 1], [1, 2, 3, 4, 5, 6, 7, 8]]], dtype=torch.int32, device="cuda")
    qp = torch.tensor([[200, 200]], dtype=torch.int32, device="cuda")
    rb = torch.tensor([180], dtype=torch.int32, device="cuda")  # window rows 17..20 exist
    ws = csa.Workspace()
    out = csa.csa_attend(q, kc, vc, idx, kr, vr, rb, qp, W, ws=ws)
    assert ws.check_error() == 2                # CSA_FLAG_INDEX
    clean = idx.clone()
    clean[0, 0, 2] = -1
    out2 = csa.csa_attend(q, kc, vc, clean, kr, vr, rb, qp, W, ws=ws)
    assert ws.check_error() == 0
    assert torch.equal(out, out2)
    # a window that falls outside the raw buffer is flagged too
    csa.csa_attend(q, kc, vc, clean, kr, vr, torch.tensor([190], dtype=torch.int32, device="cuda"), qp, W + 10, ws=ws)
    assert ws.check_error() == 2


def test_hca_long_list_partials_in_workspace():
    """140000 entries at m = 1 (over 131072 keys): the splits keep their
    partials in the workspace and merge in the combine kernel."""
    pos = np.array([[139999, 70000]])
    _attn_case(12, 1, 2, 140000, 16, 128, 0, 128, 1, pos, 140000, 0, hca=True)
