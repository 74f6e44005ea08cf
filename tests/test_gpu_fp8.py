"""FP8 (E4M3) indexer on the GPU vs the oracle: the row quantisation bit for
bit (codes and power-of-two scales), the FP8 tensor-core scores element by
element against the oracle's float64 scores of the same dequantised rows, the
top-k by the near-tie rule on those scores, and csa_layer with FP8 indexer
keys end to end."""
import math

import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import assert_attention_close, assert_scores_close, bits, check_topk_near_tie

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [32, 64, 128, 256])
def test_quantize_matches_oracle_bit_for_bit(D):
    import long_context_sparse_23_b300 as csa
    R = 1000
    x = S.normal_bf16(11, S.TID["i_cmp"], (R, D), "cpu")
    # rows over a wide range of magnitudes, an all-zero row, a row of tiny
    # (bf16-subnormal) values, a row with a single non-zero element
    mag = torch.exp2(torch.linspace(-30, 30, R)).view(R, 1)
    x = (x.float() * mag).to(torch.bfloat16)
    x[3] = 0
    x[5] = (x[5].float() * 2.0 ** -110).to(torch.bfloat16)
    x[7] = 0
    x[7, 1] = -3.0
    codes, scales = csa.csa_quantize_fp8(x.cuda())
    torch.cuda.synchronize()
    v, s, c = O.quantize_e4m3_rows(O.bf16_to_f64(bits(x)))
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.float64), s)
    np.testing.assert_array_equal(codes.cpu().numpy(), c)


def _fp8_case(seed, B, Tq, N, H_I, m, k, pos, per_query_w=False, rows=None):
    import long_context_sparse_23_b300 as csa
    d_I = 128
    q = S.normal_bf16(seed, S.TID["q_idx"], (B, Tq, H_I, d_I), "cuda")
    kk = S.normal_bf16(seed, S.TID["i_cmp"], (B, N, d_I), "cuda")
    if per_query_w:
        w = S.uniform_f32(seed, S.TID["w"], (B, Tq, H_I), "cuda") * 2 - 1
    else:
        w = S.uniform_f32(seed, S.TID["w"], (H_I,), "cuda")
    qp = torch.from_numpy(np.asarray(pos, np.int32)).cuda()
    q8, qs = csa.csa_quantize_fp8(q)
    k8, ks = csa.csa_quantize_fp8(kk)
    sc = csa.csa_index_scores_fp8(q8, qs, k8, ks, w, qp, m)
    idx = csa.csa_topk(sc, qp, N, m, k)
    torch.cuda.synchronize()
    # the oracle quantises the same bf16 rows itself
    qv, qsc, _ = O.quantize_e4m3_rows(O.bf16_to_f64(bits(q)).reshape(-1, d_I))
    kv, ksc, _ = O.quantize_e4m3_rows(O.bf16_to_f64(bits(kk)).reshape(-1, d_I))
    qv, qsc = qv.reshape(B, Tq, H_I, d_I), qsc.reshape(B, Tq, H_I)
    kv, ksc = kv.reshape(B, N, d_I), ksc.reshape(B, N)
    w64 = w.cpu().double().numpy()
    scg, ixg = sc.cpu().numpy(), idx.cpu().numpy()
    rows = rows if rows is not None else [(b, j) for b in range(B) for j in range(Tq)]
    for b, j in rows:
        t = int(pos[b][j])
        wq = w64 if w64.ndim == 1 else w64[b, j]
        ref = O.indexer_scores_fp8(qv[b, j], qsc[b, j], kv[b], ksc[b], wq, t, m)
        n = ref.shape[0]
        scale = (np.abs(kv[b, :n]) * ksc[b, :n, None]) @ (np.abs(qv[b, j]) * qsc[b, j][:, None]).T @ np.abs(wq)
        assert_scores_close(scg[b, j, :n], ref, scale, f"b={b} j={j}")
        check_topk_near_tie(ixg[b, j], O.topk(ref, k), ref, k, f"b={b} j={j}")


@pytest.mark.parametrize("H_I", [16, 32, 64, 128])
def test_fp8_scores_head_shapes(H_I):
    """Every head count, ragged N (not a multiple of the 128-key tile), a
    partial query group."""
    pos = np.array([[3, 100, 1999, 2000, 4003, 4010, 5000]] * 2)
    _fp8_case(5, 2, 7, 1004, H_I, 4, 64, pos)


def test_fp8_scores_decode_128k_and_per_query_weights():
    _fp8_case(2, 8, 1, 32768, 64, 4, 1024, np.full((8, 1), 131071))
    _fp8_case(3, 2, 1, 32768, 64, 4, 1024, np.full((2, 1), 131071), per_query_w=True)


def test_fp8_scores_1m_causal_tail():
    pos = np.array([list(range((1 << 20) - 4, 1 << 20))] * 2)
    _fp8_case(4, 2, 4, 262144, 64, 4, 1024, pos)


def test_fp8_scores_prefill_sampled():
    """1024 queries of one sequence (256 query groups of four, several per
    CTA), 256 entries: 40 rows checked."""
    rng = np.random.default_rng(0)
    rows = [(0, int(j)) for j in np.concatenate([np.arange(8), rng.integers(0, 1024, 24), np.arange(1016, 1024)])]
    _fp8_case(6, 1, 1024, 256, 64, 4, 16, np.arange(1024)[None], rows=rows)


def test_layer_decode_1m_fp8_indexer():
    """csa_layer at 1M context with E4M3 indexer keys: indices by the near-tie
    rule against the oracle's top-k of its FP8 scores (queries quantised by
    the oracle from the same bf16 rows), output against the oracle's
    attention on the GPU's indices."""
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["decode_1m"].replace(B=2)
    inp = S.make_inputs(wl, "cuda")
    k8, ks = csa.csa_quantize_fp8(inp["i_cmp"])
    out = torch.empty(wl.B, 1, wl.H, wl.d, dtype=torch.float32, device="cuda")
    idx = torch.empty(wl.B, 1, wl.k, dtype=torch.int32, device="cuda")
    a = csa.layer_args(B=wl.B, Tq=1, N=wl.N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k, W=wl.W,
                       T_raw=wl.raw_len, k_cmp=inp["k_cmp"], v_cmp=inp["v_cmp"], i_cmp=k8, k_win=inp["k_raw"],
                       v_win=inp["v_raw"], raw_base=inp["raw_base"], q=inp["q"], q_idx=inp["q_idx"], w=inp["w"],
                       q_pos=inp["q_pos"], idx_out=idx, out=out, out_dtype=torch.float32, i_scale=ks)
    ws = csa.Workspace()
    csa.csa_layer(a, ws)
    assert ws.check_error() == 0
    c = {n: (bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()) for n, v in inp.items()}
    t = wl.q_positions[0]
    kv, ksc, _ = O.quantize_e4m3_rows(O.bf16_to_f64(c["i_cmp"]).reshape(-1, wl.d_I))
    kv, ksc = kv.reshape(wl.B, wl.N, wl.d_I), ksc.reshape(wl.B, wl.N)
    gidx = idx.cpu().numpy()
    for b in range(wl.B):
        qv, qsc, _ = O.quantize_e4m3_rows(O.bf16_to_f64(c["q_idx"][b, 0]))
        ref = O.indexer_scores_fp8(qv, qsc, kv[b], ksc[b], c["w"].astype(np.float64), t, wl.m)
        check_topk_near_tie(gidx[b, 0], O.topk(ref, wl.k), ref, wl.k, f"b={b}")
        win = O.window_rows(t, wl.W, wl.raw_base, wl.raw_len)
        o, _ = O.attend_one(O.bf16_to_f64(c["q"][b, 0]), O.bf16_to_f64(c["k_cmp"][b]), O.bf16_to_f64(c["v_cmp"][b]),
                            gidx[b, 0], O.bf16_to_f64(c["k_raw"][b]), O.bf16_to_f64(c["v_raw"][b]), win,
                            1 / math.sqrt(wl.d))
        assert_attention_close(out[b, 0].cpu().numpy(), o, f"b={b}")
