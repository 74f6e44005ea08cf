"""(1) Block compression on the GPU vs the oracle."""
import numpy as np
import pytest
import torch

import csa_synth as S
import oracle as O
from tests._parity import assert_compressed_bf16, assert_compressed_f32, bits

pytestmark = pytest.mark.gpu


def _streams(seed, B, T, Ds, device):
    xs = [S.normal_bf16(seed, 100 + i, (B, T, D), device) for i, D in enumerate(Ds)]
    gs = [S.normal_bf16(seed, 200 + i, (B, T, D), device) for i, D in enumerate(Ds)]
    return xs, gs


@pytest.mark.parametrize("B,T,m,Ds", [
    (1, 256, 4, (64, 64, 32)),            # tiny prefill: K, V, indexer keys in one launch
    (1, 8192, 4, (128, 128, 128)),        # 8K prefill
    (2, 128 * 37 + 5, 128, (128, 128)),   # HCA block size, ragged tail dropped
    (3, 50, 3, (8, 16)),                  # odd m, narrow rows
    (2, 96, 6, (32,)),
    (1, 64, 1, (64,)),                    # m = 1: identity
    (1, 3, 4, (64,)),                     # T < m: nothing to compress
])
def test_compress_parity(B, T, m, Ds):
    import long_context_sparse_23_b300 as csa
    xs, gs = _streams(7, B, T, Ds, "cuda")
    out32 = csa.csa_compress(xs, gs, m, out_dtype=torch.float32)
    out16 = csa.csa_compress(xs, gs, m, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    xc, gc = _streams(7, B, T, Ds, "cpu")
    for i in range(len(Ds)):
        assert torch.equal(xs[i].cpu().view(torch.int16), xc[i].view(torch.int16))  # same inputs
        x = O.bf16_to_f64(bits(xc[i]))
        g = O.bf16_to_f64(bits(gc[i]))
        ref = np.stack([O.compress(x[b], g[b], m) for b in range(B)])
        scale = np.stack([O.compress(np.abs(x[b]), g[b], m) for b in range(B)])
        assert out32[i].shape == (B, T // m, Ds[i])
        if T // m == 0:
            continue
        assert_compressed_f32(out32[i].cpu().numpy(), ref, scale, f"stream {i}")
        assert_compressed_bf16(bits(out16[i]), ref, scale, f"stream {i}")
        if m == 1:
            assert torch.equal(out16[i].cpu(), xc[i])


def test_compress_full_1m_hca_sampled():
    """The 1M-token HCA streams (8 x 2^20 x 128, K and V) at m' = 128, the launch
    the benchmark times; 256 sampled entries checked against the oracle."""
    import long_context_sparse_23_b300 as csa
    wl = S.WORKLOADS["hca_decode_1m"]
    inp = S.make_inputs(wl, "cuda", only={"k_raw", "v_raw", "g_k", "g_v"})
    kc, vc = csa.csa_compress([inp["k_raw"], inp["v_raw"]], [inp["g_k"], inp["g_v"]], wl.m)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    got_all, ref_all, scale_all = [], [], []
    for b, blk in zip(rng.integers(0, wl.B, 256), rng.integers(0, wl.N, 256)):
        rows = torch.arange(blk * wl.m, (blk + 1) * wl.m, dtype=torch.int64)
        for name, gname, got in (("k_raw", "g_k", kc), ("v_raw", "g_v", vc)):
            x = O.bf16_to_f64(bits(S.rows_bf16(wl.seed, S.TID[name], wl.T, wl.d, int(b), rows)))
            g = O.bf16_to_f64(bits(S.rows_bf16(wl.seed, S.TID[gname], wl.T, wl.d, int(b), rows)))
            ref_all.append(O.compress(x, g, wl.m)[0])
            scale_all.append(O.compress(np.abs(x), g, wl.m)[0])
            got_all.append(bits(got[b, blk]))
    assert_compressed_bf16(np.stack(got_all), np.stack(ref_all), np.stack(scale_all), "1M HCA sampled entries")
    del inp
