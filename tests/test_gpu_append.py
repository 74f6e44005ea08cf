"""Decode-time compression and cache append (every m tokens one entry) on
the GPU: csa_append against the prefill compression of the same blocks
(bit-exact) and against the oracle, and csa_layer decode steps that append
their completed blocks before the indexer, over consecutive positions that
cross block boundaries, against the oracle run on the whole prefix."""
import math

import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import assert_attention_close, assert_compressed_bf16, bits, check_topk_near_tie

pytestmark = pytest.mark.gpu

STREAMS = (("k_raw", "g_k", "k_cmp"), ("v_raw", "g_v", "v_cmp"), ("i_raw", "g_i", "i_cmp"))


def _raw(seed, B, T, d, d_I):
    dev = "cuda"
    x = {}
    for name, width in (("k_raw", d), ("v_raw", d), ("g_k", d), ("g_v", d), ("i_raw", d_I), ("g_i", d_I)):
        x[name] = S.normal_bf16(seed, S.TID[name], (B, T, width), dev)
    return x


def test_append_equals_prefill_compression_and_oracle():
    import long_context_sparse_23_b300 as csa
    B, T, m, d, d_I, T_raw, N = 2, 1024, 4, 128, 64, 40, 300
    x = _raw(41, B, T, d, d_I)
    full = csa.csa_compress([x["k_raw"], x["v_raw"], x["i_raw"]], [x["g_k"], x["g_v"], x["g_i"]], m)
    caches = [torch.zeros(B, N, w, dtype=torch.bfloat16, device="cuda") for w in (d, d, d_I)]
    # sequence 0 at positions ending a block, sequence 1 one token later; three
    # queries per step, two of which complete a block in sequence 0
    t_last = torch.tensor([[1023 - 4 * 20 - 1], [1023 - 4 * 20]], dtype=torch.int64)
    for step in range(6):
        tl = t_last[:, 0] + 4 * step
        q_pos = torch.stack([tl - 4, tl - 2, tl], dim=1).to(torch.int32).cuda()
        rb = (tl + 1 - T_raw).to(torch.int32)
        wins = {n: torch.stack([x[n][b, int(rb[b]):int(rb[b]) + T_raw] for b in range(B)]) for n in x}
        ws = csa.Workspace()
        csa.csa_append([wins["k_raw"], wins["v_raw"], wins["i_raw"]], [wins["g_k"], wins["g_v"], wins["g_i"]],
                       caches, rb.cuda(), q_pos, m, ws=ws)
        assert ws.check_error() == 0
        for b in range(B):
            for t in q_pos[b].tolist():
                if (t + 1) % m:
                    continue
                blk = (t + 1) // m - 1
                for c, f in zip(caches, full):
                    assert torch.equal(c[b, blk], f[b, blk]), (b, t)
        # against the oracle's fold of the same window rows
        for (xn, gn, _), c in zip(STREAMS, caches):
            ref = O.csa_append(bits(wins[xn]), bits(wins[gn]), rb.numpy(), q_pos.cpu().numpy(), m)
            absx = O.round_bf16(np.abs(O.bf16_to_f64(bits(wins[xn]))))
            scale = O.csa_append(absx, bits(wins[gn]), rb.numpy(), q_pos.cpu().numpy(), m)
            got = bits(c)
            for b in range(B):
                for blk, v in ref[b].items():
                    assert_compressed_bf16(got[b, blk][None], v[None], scale[b][blk][None], f"{xn} b={b} blk={blk}")
    # positions that complete no block leave the caches untouched
    before = [c.clone() for c in caches]
    q_pos = torch.tensor([[1000], [1001]], dtype=torch.int32, device="cuda")
    rb = torch.tensor([1000 + 1 - T_raw, 1001 + 1 - T_raw], dtype=torch.int32)
    wins = {n: torch.stack([x[n][b, int(rb[b]):int(rb[b]) + T_raw] for b in range(B)]) for n in x}
    csa.csa_append([wins["k_raw"]], [wins["g_k"]], caches[:1], rb.cuda(), q_pos, m)
    assert torch.equal(before[0], caches[0])


@pytest.mark.parametrize("T0,N", [(4094, 1100), (4 * 65540 + 2, 65600)])
def test_decode_steps_append_then_attend(T0, N):
    """Consecutive decode steps t = T0, T0 + 1, ... (sequence 1 one token
    ahead of sequence 0): each csa_layer call appends the block its position
    completes, then scores, selects and attends.  The caches start as the
    compression of the complete blocks before T0 (the partial block stays
    raw); after every step they must equal the compression of every block
    completed so far, and the indices and output the oracle's on that prefix.
    The second case (65600 entries) takes the fused top-k + attention
    kernel."""
    import long_context_sparse_23_b300 as csa
    B, m, H, d, H_I, d_I, k, W, T_raw = 2, 4, 64, 128, 64, 128, 1024, 128, 256
    steps = 6
    T_tot = T0 + steps + 1
    x = _raw(43, B, T_tot, d, d_I)
    full = csa.csa_compress([x["k_raw"], x["v_raw"], x["i_raw"]], [x["g_k"], x["g_v"], x["g_i"]], m)
    caches = [torch.zeros(B, N, c.shape[2], dtype=torch.bfloat16, device="cuda") for c in full]
    for b in range(B):
        nb = (T0 + b) // m
        for c, f in zip(caches, full):
            c[b, :nb] = f[b, :nb]
    w = S.uniform_f32(43, S.TID["w"], (H_I,), "cuda")
    xc = {n: bits(v) for n, v in x.items()}
    # the oracle's caches: compression of every complete block, rounded to bf16
    ref_c = {cn: O.round_bf16(O.csa_compress(xc[xn], xc[gn], m)) for xn, gn, cn in STREAMS}
    scale = 1 / math.sqrt(d)
    ws = csa.Workspace()
    for s in range(steps):
        t = torch.tensor([T0 + s, T0 + s + 1], dtype=torch.int64)
        q_pos = t.to(torch.int32).view(B, 1).cuda()
        rb = (t + 1 - T_raw).to(torch.int32)
        wins = {n: torch.stack([x[n][b, int(rb[b]):int(rb[b]) + T_raw] for b in range(B)]).contiguous() for n in x}
        q = S.normal_bf16(44 + s, S.TID["q"], (B, 1, H, d), "cuda")
        qi = S.normal_bf16(44 + s, S.TID["q_idx"], (B, 1, H_I, d_I), "cuda")
        out = torch.empty(B, 1, H, d, dtype=torch.float32, device="cuda")
        idx = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
        a = csa.layer_args(B=B, Tq=1, N=N, m=m, H=H, d=d, H_I=H_I, d_I=d_I, k=k, W=W, T_raw=T_raw,
                           k_cmp=caches[0], v_cmp=caches[1], i_cmp=caches[2], k_win=wins["k_raw"],
                           v_win=wins["v_raw"], raw_base=rb.cuda(), q=q, q_idx=qi, w=w, q_pos=q_pos,
                           idx_out=idx, out=out, out_dtype=torch.float32, i_win=wins["i_raw"],
                           gk_win=wins["g_k"], gv_win=wins["g_v"], gi_win=wins["g_i"])
        csa.csa_layer(a, ws)
        assert ws.check_error() == 0
        gidx = idx.cpu().numpy()
        gout = out.cpu().numpy()
        qb, qib = bits(q), bits(qi)
        for b in range(B):
            tb = int(t[b])
            nb = (tb + 1) // m
            for c, f in zip(caches, full):
                assert torch.equal(c[b, :nb], f[b, :nb]), f"cache prefix after step {s}, b={b}"
                assert not c[b, nb:].any(), f"no entry beyond block {nb - 1} after step {s}"
            S_ref = O.indexer_scores(O.bf16_to_f64(qib[b, 0]), O.bf16_to_f64(ref_c["i_cmp"][b, :nb]),
                                     w.cpu().numpy().astype(np.float64), tb, m)
            ref_idx = O.topk(S_ref, k)
            check_topk_near_tie(gidx[b, 0], ref_idx, S_ref, k, f"step {s} b={b}")
            win = O.window_rows(tb, W, int(rb[b]), T_raw)
            o, _ = O.attend_one(O.bf16_to_f64(qb[b, 0]), O.bf16_to_f64(ref_c["k_cmp"][b]),
                                O.bf16_to_f64(ref_c["v_cmp"][b]), gidx[b, 0], O.bf16_to_f64(bits(wins["k_raw"])[b]),
                                O.bf16_to_f64(bits(wins["v_raw"])[b]), win, scale)
            assert_attention_close(gout[b, 0], o, f"step {s} b={b}")
