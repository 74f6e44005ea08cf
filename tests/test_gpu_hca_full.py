"""HCA decode at 1M tokens end to end: the raw K/V streams (8 x 2^20 x 128)
compressed at m' = 128 on the GPU, then dense attention over all 8192 entries
plus the 128-token window; sequence 0 recomputed by the oracle from the raw
streams."""
import math

import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import assert_attention_close, assert_compressed_bf16, bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_hca_decode_1m_from_raw_streams():
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["hca_decode_1m"]
    g = S.make_inputs(wl, "cuda")
    kc, vc = csa.csa_compress([g["k_raw"], g["v_raw"]], [g["g_k"], g["g_v"]], wl.m)
    out = csa.hca_attend(g["q"], kc, vc, g["k_raw"], g["v_raw"], g["raw_base"], g["q_pos"], wl.m, wl.W)
    torch.cuda.synchronize()
    b = 0
    c = S.make_inputs(wl, "cpu", batches=[b])
    for name, gname, got in (("k_raw", "g_k", kc), ("v_raw", "g_v", vc)):
        x = O.bf16_to_f64(bits(c[name][0]))
        gl = O.bf16_to_f64(bits(c[gname][0]))
        ref = O.compress(x, gl, wl.m)
        assert_compressed_bf16(bits(got[b]), ref, O.compress(np.abs(x), gl, wl.m), f"{name} entries")
        if name == "k_raw":
            kref = ref
        else:
            vref = ref
    t = wl.positions[0]
    win = O.window_rows(t, wl.W, 0, wl.T)
    kr = O.bf16_to_f64(bits(c["k_raw"][0, -wl.W:]))
    vr = O.bf16_to_f64(bits(c["v_raw"][0, -wl.W:]))
    ref, _ = O.attend_one(O.bf16_to_f64(bits(c["q"][0, 0])), O.bf16_to_f64(O.round_bf16(kref)),
                          O.bf16_to_f64(O.round_bf16(vref)), np.arange(wl.N), kr, vr,
                          win - (wl.T - wl.W), 1 / math.sqrt(wl.d))
    assert_attention_close(out[b, 0].float().cpu().numpy(), ref, "hca out")
