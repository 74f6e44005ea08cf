"""csa_layer end to end (1)->(4) on the GPU vs the oracle; determinism, batch
invariance and the 1M decode / causal-tail consistency."""
import math

import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import (assert_attention_close, assert_compressed_bf16, bits,
                           check_topk_near_tie)

pytestmark = pytest.mark.gpu


def _decode_layer(inp, wl, out_dtype=torch.bfloat16):
    import long_context_sparse_23_b300 as csa
    B, Tq = inp["q_pos"].shape
    out = torch.empty(B, Tq, wl.H, wl.d, dtype=out_dtype, device="cuda")
    idx = torch.empty(B, Tq, wl.k, dtype=torch.int32, device="cuda")
    a = csa.layer_args(B=B, Tq=Tq, N=wl.N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k, W=wl.W,
                       T_raw=wl.raw_len, k_cmp=inp["k_cmp"], v_cmp=inp["v_cmp"], i_cmp=inp["i_cmp"],
                       k_win=inp["k_raw"], v_win=inp["v_raw"], raw_base=inp["raw_base"], q=inp["q"],
                       q_idx=inp["q_idx"], w=inp["w"], q_pos=inp["q_pos"], idx_out=idx, out=out,
                       out_dtype=out_dtype)
    csa.csa_layer(a)
    torch.cuda.synchronize()
    return idx, out


def _prefill_case(name, rows=None):
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS[name]
    g = S.make_inputs(wl, "cuda")
    res = csa.csa_layer_prefill(g, wl.m, wl.k, wl.W)
    torch.cuda.synchronize()
    c = {k: (bits(v) if v.dtype == torch.bfloat16 else v.numpy()) for k, v in S.make_inputs(wl, "cpu").items()}
    kc = O.csa_compress(c["k_raw"], c["g_k"], wl.m)
    vc = O.csa_compress(c["v_raw"], c["g_v"], wl.m)
    ic = O.csa_compress(c["i_raw"], c["g_i"], wl.m)
    for ref, key, xk, gk in ((kc, "k_cmp", "k_raw", "g_k"), (vc, "v_cmp", "v_raw", "g_v"),
                             (ic, "i_cmp", "i_raw", "g_i")):
        absx = O.round_bf16(np.abs(O.bf16_to_f64(c[xk])))  # |x| is exact in bf16
        assert_compressed_bf16(bits(res[key]), ref, O.csa_compress(absx, c[gk], wl.m), key)
    # downstream steps on the oracle's own bf16 caches
    kcb, vcb, icb = O.round_bf16(kc), O.round_bf16(vc), O.round_bf16(ic)
    q64 = O.bf16_to_f64(c["q"])
    qi64, ic64 = O.bf16_to_f64(c["q_idx"]), O.bf16_to_f64(icb)
    kc64, vc64 = O.bf16_to_f64(kcb), O.bf16_to_f64(vcb)
    kr64, vr64 = O.bf16_to_f64(c["k_raw"]), O.bf16_to_f64(c["v_raw"])
    w64 = c["w"].astype(np.float64)
    gidx = res["idx"].cpu().numpy()
    gout = res["out"].float().cpu().numpy()
    scale = 1 / math.sqrt(wl.d)
    rows = rows if rows is not None else range(wl.T)
    for t in rows:
        # the GPU scored its own bf16 caches; a one-ulp cache difference moves a
        # score by far less than the near-tie band
        S_ref = O.indexer_scores(qi64[0, t], ic64[0], w64, t, wl.m)
        check_topk_near_tie(gidx[0, t], O.topk(S_ref, wl.k), S_ref, wl.k, f"t={t}")
        # attention on the GPU's own index set
        win = O.window_rows(t, wl.W, 0, wl.T)
        ref, _ = O.attend_one(q64[0, t], kc64[0], vc64[0], gidx[0, t], kr64[0], vr64[0], win, scale)
        assert_attention_close(gout[0, t], ref, f"t={t}")


def test_layer_tiny_prefill_end_to_end():
    _prefill_case("tiny_prefill")


def test_layer_prefill_8k_end_to_end_sampled():
    rng = np.random.default_rng(0)
    rows = sorted(set(np.concatenate([np.arange(6), rng.integers(0, 8192, 60), np.arange(8186, 8192)]).tolist()))
    _prefill_case("prefill_8k", rows)


def _decode_check(wl, inp_cpu, idx, out, rows):
    c = {k: (bits(v) if v.dtype == torch.bfloat16 else v.numpy()) for k, v in inp_cpu.items()}
    gidx, gout = idx.cpu().numpy(), out.float().cpu().numpy()
    w64 = c["w"].astype(np.float64)
    scale = 1 / math.sqrt(wl.d)
    for b, j in rows:
        t = int(c["q_pos"][b, j])
        ic64 = O.bf16_to_f64(c["i_cmp"][b])
        S_ref = O.indexer_scores(O.bf16_to_f64(c["q_idx"][b, j]), ic64, w64, t, wl.m)
        check_topk_near_tie(gidx[b, j], O.topk(S_ref, wl.k), S_ref, wl.k, f"b={b} j={j}")
        sel = gidx[b, j][gidx[b, j] >= 0]
        kc = O.bf16_to_f64(bits(S.rows_bf16(wl.seed, S.TID["k_cmp"], wl.N, wl.d, b, torch.from_numpy(sel.astype(np.int64)))))
        vc = O.bf16_to_f64(bits(S.rows_bf16(wl.seed, S.TID["v_cmp"], wl.N, wl.d, b, torch.from_numpy(sel.astype(np.int64)))))
        win = O.window_rows(t, wl.W, int(c["raw_base"][b]), wl.raw_len)
        ref, _ = O.attend_one(O.bf16_to_f64(c["q"][b, j]), kc, vc, np.arange(len(sel)),
                              O.bf16_to_f64(c["k_raw"][b]), O.bf16_to_f64(c["v_raw"][b]), win, scale)
        assert_attention_close(gout[b, j], ref, f"b={b} j={j}")


def test_layer_decode_128k_batch_invariant_and_deterministic():
    wl = S.WORKLOADS["decode_128k"]
    g = S.make_inputs(wl, "cuda")
    idx1, out1 = _decode_layer(g, wl)
    idx2, out2 = _decode_layer(g, wl)
    assert torch.equal(idx1, idx2) and torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    # sequence 5 alone gives the bits it gets inside the batch of 64
    one = {k: (v[5:6].contiguous() if v.dim() > 1 or k == "raw_base" else v) for k, v in g.items()}
    idx3, out3 = _decode_layer(one, wl)
    assert torch.equal(idx3[0], idx1[5]) and torch.equal(out3[0].view(torch.int16), out1[5].view(torch.int16))
    rows = [(b, 0) for b in (0, 5, 31, 63)]
    cpu = S.make_inputs(wl, "cpu", only={"q", "q_idx", "w", "q_pos", "k_raw", "v_raw", "i_cmp"})
    _decode_check(wl, cpu, idx1, out1, rows)


def test_layer_decode_1m_and_causal_tail_agree():
    wl = S.WORKLOADS["decode_1m"]
    wt = S.WORKLOADS["decode_1m_tail"]
    g = S.make_inputs(wl, "cuda")
    gt = S.make_inputs(wt, "cuda", only={"q", "q_idx", "q_pos"})
    gt.update({k: g[k] for k in ("k_cmp", "v_cmp", "i_cmp", "k_raw", "v_raw", "w", "raw_base")})
    idx, out = _decode_layer(g, wl)
    idx_t, out_t = _decode_layer(gt, wt)
    # the tail's last query (t = 1048575) is the decode query: identical bits
    assert torch.equal(idx_t[:, 3], idx[:, 0])
    assert torch.equal(out_t[:, 3].view(torch.int16), out[:, 0].view(torch.int16))
    # only the last tail query sees the last block
    it = idx_t.cpu().numpy()
    assert np.all(it[:, :3] < 262143) and np.all(it[:, :3] >= -1)
    cpu = S.make_inputs(wt, "cpu", only={"q", "q_idx", "w", "q_pos", "k_raw", "v_raw", "i_cmp"})
    _decode_check(wt, cpu, idx_t, out_t, [(b, j) for b in range(4) for j in range(4)])


def test_layer_decode_fused_tail_matches_separate_calls():
    """Decode csa_layer at 1M context runs the fused top-k + attention kernel;
    csa_index_topk followed by csa_attend runs the separate kernels.  Same
    indices, bit for bit; outputs within the attention tolerance of each other."""
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["decode_1m"]
    g = S.make_inputs(wl, "cuda", batches=[0, 1])
    idx_l, out_l = _decode_layer(g, wl, out_dtype=torch.float32)
    idx_s = csa.csa_index_topk(g["q_idx"], g["i_cmp"], g["w"], g["q_pos"], wl.m, wl.k)
    out_s = csa.csa_attend(g["q"], g["k_cmp"], g["v_cmp"], idx_s, g["k_raw"], g["v_raw"], g["raw_base"],
                           g["q_pos"], wl.W, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(idx_l, idx_s)
    assert_attention_close(out_l.cpu().numpy(), out_s.double().cpu().numpy(), "fused vs separate")


@pytest.mark.parametrize("N", [70000, 30000], ids=["fused_tail", "mid_rows"])
def test_layer_decode_tail_ties_and_short_visibility(N):
    """The decode top-k on degenerate inputs, in the fused decode tail (rows
    over 65536 entries) and in the one-CTA-per-query selection (rows up to
    32768): every score equal (the lowest indices win; the tie bucket is too
    large to stage), scores tied in groups of eight (ties at the threshold),
    and a query that sees fewer blocks than k (everything visible kept, -1
    padding)."""
    B, m, H, d, H_I, d_I, k, W = 3, 4, 64, 128, 64, 128, 1024, 128
    wl = S.WORKLOADS["decode_128k"].replace(B=B, T=N * m, positions=(N * m - 1,), raw_len=256)
    g = S.make_inputs(wl, "cuda")
    g["q_idx"][0].zero_()                                      # sequence 0: all scores 0
    g["i_cmp"][1] = g["i_cmp"][1][::8].repeat_interleave(8, 0)[:N]   # sequence 1: ties in groups of 8
    g["q_pos"][2, 0] = 2001                                    # sequence 2: n_vis = 500 < k
    g["raw_base"][2] = 2002 - 256
    for name in ("k_raw", "v_raw"):                            # its window rows: tokens 1746..2001
        g[name][2] = S.rows_bf16(wl.seed, S.TID[name], wl.T, d, 2,
                                 torch.arange(2002 - 256, 2002, device="cuda"))
    idx, out = _decode_layer(g, wl)
    gi = idx.cpu().numpy()
    np.testing.assert_array_equal(gi[0, 0], np.arange(k))
    np.testing.assert_array_equal(gi[2, 0], np.concatenate([np.arange(500), -np.ones(k - 500, np.int32)]))
    cpu = {key: v.cpu() for key, v in g.items()}
    _decode_check(wl, cpu, idx, out, [(0, 0), (1, 0), (2, 0)])


def test_layer_decode_per_query_weights():
    """csa_layer with per-query indexer weights at 1M context (the fused
    top-k + attention kernel): the indices equal csa_index_topk's with the
    same weights, and the output matches the oracle on those indices."""
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["decode_1m"].replace(B=2)
    inp = S.make_inputs(wl, "cuda")
    w = S.uniform_f32(9, S.TID["w"], (wl.B, 1, wl.H_I), "cuda") * 2 - 1
    inp["w"] = w
    idx, out = _decode_layer(inp, wl, out_dtype=torch.float32)
    idx_s = csa.csa_index_topk(inp["q_idx"], inp["i_cmp"], w, inp["q_pos"], wl.m, wl.k)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_s)
    c = {k: (bits(v) if v.dtype == torch.bfloat16 else v.cpu().numpy()) for k, v in inp.items()}
    t = wl.q_positions[0]
    for b in range(wl.B):
        win = O.window_rows(t, wl.W, wl.raw_base, wl.raw_len)
        o, _ = O.attend_one(O.bf16_to_f64(c["q"][b, 0]), O.bf16_to_f64(c["k_cmp"][b]), O.bf16_to_f64(c["v_cmp"][b]),
                            idx[b, 0].cpu().numpy(), O.bf16_to_f64(c["k_raw"][b]), O.bf16_to_f64(c["v_raw"][b]), win,
                            1 / math.sqrt(wl.d))
        assert_attention_close(out[b, 0].cpu().numpy(), o, f"b={b}")
