"""Device-side failure reporting without faulting the GPU: a bounded wait that
runs out sets CSA_FLAG_TIMEOUT in the workspace error word and the kernel
returns; the context stays usable and the next call is correct."""
import numpy as np
import pytest
import torch

import csa_synth as S
from long_context_sparse_23_b300 import _lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", ["decode", "prefill"])
def test_wait_budget_runs_out_and_context_survives(kernel):
    """Indexer waits with a one-cycle budget.  Each CTA streams tens of key
    tiles while every SM reads HBM, so its waits for tiles (and for the
    accumulators of its other epilogue group) last about a tile's streaming
    time: some wait outlasts the budget.  decode: one query per sequence (the
    one-item kernel, whose first tiles are requested before any wait);
    prefill: query groups of four (the persistent kernel)."""
    import long_context_sparse_23_b300 as csa
    if kernel == "decode":
        B, Tq, N = 4, 1, 262144
    else:
        B, Tq, N = 1, 16, 65536
    q = S.normal_bf16(1, 2, (B, Tq, 64, 128), "cuda")
    k = S.normal_bf16(1, 12, (B, N, 128), "cuda")
    w = S.uniform_f32(1, 9, (64,), "cuda")
    qp = torch.full((B, Tq), 4 * N - 1, dtype=torch.int32, device="cuda") - torch.arange(Tq, device="cuda").int()
    ws = csa.Workspace()
    ref = csa.csa_index_scores(q, k, w, qp, 4, ws=ws)
    assert ws.check_error() == 0
    try:
        _lib.lib().csa_set_wait_budget(1)       # one clock cycle: a wait that does not pass at once gives up
        csa.csa_index_scores(q, k, w, qp, 4, ws=ws)
        flags = ws.check_error()
    finally:
        _lib.lib().csa_set_wait_budget(0)       # back to the default budget
    assert flags & _lib.CSA_FLAG_TIMEOUT
    again = csa.csa_index_scores(q, k, w, qp, 4, ws=ws)
    assert ws.check_error() == 0
    # query j sees its first (t_j + 1) // 4 entries; the rest of its row is not written
    for j in range(Tq):
        n = (4 * N - j) // 4
        assert torch.equal(again[:, j, :n], ref[:, j, :n]), j


def _decode_attend_inputs(seed, B, N, k, W, H=64, d=128):
    """Decode-shaped attention inputs at t = 4N - 1 (every entry visible), a
    raw window buffer of 2W rows ending at t, and k distinct sorted indices."""
    t = 4 * N - 1
    g = torch.Generator().manual_seed(seed)
    q = S.normal_bf16(seed, S.TID["q"], (B, 1, H, d), "cuda")
    kc = S.normal_bf16(seed, S.TID["k_cmp"], (B, N, d), "cuda")
    vc = S.normal_bf16(seed, S.TID["v_cmp"], (B, N, d), "cuda")
    kr = S.normal_bf16(seed, S.TID["k_raw"], (B, 2 * W, d), "cuda")
    vr = S.normal_bf16(seed, S.TID["v_raw"], (B, 2 * W, d), "cuda")
    idx = torch.stack([torch.sort(torch.randperm(N, generator=g)[:k])[0] for _ in range(B)])
    idx = idx.to(torch.int32).view(B, 1, k).cuda()
    qp = torch.full((B, 1), t, dtype=torch.int32, device="cuda")
    rb = torch.full((B,), t + 1 - 2 * W, dtype=torch.int32, device="cuda")
    return q, kc, vc, idx, kr, vr, rb, qp


@pytest.mark.parametrize("mode", ["csa_gather", "hca_tiles"])
def test_tensor_core_attention_wait_budget_runs_out(mode):
    """The tcgen05 decode attention (H = 64, d = 128, more than four 128-key
    tiles per query: the CSA case's 2 ranges of 5 and 4 tiles merge inside
    their cluster, the HCA case's 9 in a second kernel) with a one-cycle wait
    budget: CSA_FLAG_TIMEOUT is set, the kernel drains its copies and
    frees its tensor memory, and the next call with the default budget gives
    the reference result bit for bit."""
    import long_context_sparse_23_b300 as csa
    B, N, k, W = 2, 4096, 1024, 128
    q, kc, vc, idx, kr, vr, rb, qp = _decode_attend_inputs(31, B, N, k, W)
    ws = csa.Workspace()

    def call():
        if mode == "csa_gather":
            return csa.csa_attend(q, kc, vc, idx, kr, vr, rb, qp, W, ws=ws)
        return csa.hca_attend(q, kc, vc, kr, vr, rb, qp, 4, W, ws=ws)

    ref = call()
    assert ws.check_error() == 0
    try:
        _lib.lib().csa_set_wait_budget(1)
        call()
        flags = ws.check_error()
    finally:
        _lib.lib().csa_set_wait_budget(0)
    assert flags & _lib.CSA_FLAG_TIMEOUT
    again = call()
    assert ws.check_error() == 0
    assert torch.equal(again, ref)


def test_decode_tail_wait_budget_runs_out():
    """The whole decode layer at a length that takes the fused top-k +
    attention kernel (131072 entries) with a one-cycle wait budget: the
    indexer and the fused kernel report CSA_FLAG_TIMEOUT and drain their
    copies; the next call with the default budget gives the reference
    indices and output bit for bit."""
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["decode_1m"].replace(B=1, T=1 << 19, positions=((1 << 19) - 1,))
    inp = S.make_inputs(wl, "cuda")
    out = torch.empty(1, 1, wl.H, wl.d, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(1, 1, wl.k, dtype=torch.int32, device="cuda")
    a = csa.layer_args(B=1, Tq=1, N=wl.N, m=wl.m, H=wl.H, d=wl.d, H_I=wl.H_I, d_I=wl.d_I, k=wl.k, W=wl.W,
                       T_raw=wl.raw_len, k_cmp=inp["k_cmp"], v_cmp=inp["v_cmp"], i_cmp=inp["i_cmp"],
                       k_win=inp["k_raw"], v_win=inp["v_raw"], raw_base=inp["raw_base"], q=inp["q"],
                       q_idx=inp["q_idx"], w=inp["w"], q_pos=inp["q_pos"], idx_out=idx, out=out)
    ws = csa.Workspace()
    csa.csa_layer(a, ws)
    assert ws.check_error() == 0
    ref_idx, ref_out = idx.clone(), out.clone()
    try:
        _lib.lib().csa_set_wait_budget(1)
        csa.csa_layer(a, ws)
        flags = ws.check_error()
    finally:
        _lib.lib().csa_set_wait_budget(0)
    assert flags & _lib.CSA_FLAG_TIMEOUT
    csa.csa_layer(a, ws)
    assert ws.check_error() == 0
    assert torch.equal(idx, ref_idx) and torch.equal(out, ref_out)
