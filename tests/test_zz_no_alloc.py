"""csa_attend_noalloc: attention for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: operators hosted by a
framework whose memory planner owns the device (they receive only their inputs
and outputs), and latency-bound code that must never reach cudaMalloc or
cudaFree.  csa_attend_noalloc serves them: short key lists merge their split
partials inside a thread-block cluster, and long ones (over 131072 keys per
query) keep them in one fixed device array inside the library.  These tests call it through the C
ABI and check it against csa_attend, which takes a workspace, and against the
oracle on sampled queries, with the attention tolerance |err| <= 1e-2 +
1e-2 |ref| used by every attention test.

The file is named so that pytest collects it last: the shared device array
keeps whatever the previous call left in it, so the GPU test also runs after
every other test of the suite (and passes alone in a fresh process).
"""
import ctypes

import numpy as np
import pytest

from long_context_sparse_23_b300 import _lib

A16 = 1 << 20  # a fake, 16-byte aligned device address; never dereferenced below


@pytest.fixture(scope="module")
def L():
    from long_context_sparse_23_b300 import build
    build.build()
    return _lib.lib()


def _scratch_limit() -> int:
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "csa.h")
    m = re.search(r"#define\s+CSA_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", open(hdr).read())
    return int(m.group(1)) << int(m.group(2))


def test_noalloc_rejects_calls_beyond_its_scratch(L):
    """Partials larger than the fixed array are refused before any device work."""
    limit = _scratch_limit()
    H, d, k, W = 64, 128, 139264, 128
    splits = -(-(k + W) // 8192)                      # over 131072 keys: 8192-key splits, partials in scratch
    per_query = splits * H * (d + 1) * 4
    B_ok, B_bad = limit // per_query, limit // per_query + 1
    args = lambda B: (A16, A16, A16, A16, A16, A16, A16, A16, B, 1, 262144, 256, H, d, k, W, 0.0,
                      A16, 0, None, None)
    assert L.csa_attend_noalloc(*args(B_bad)) == _lib.CSA_ERR_WORKSPACE
    # bad arguments are still refused first, as csa_attend refuses them
    bad = list(args(B_ok))
    bad[0] = None
    assert L.csa_attend_noalloc(*bad) == _lib.CSA_ERR_INVALID
    bad = list(args(B_ok))
    bad[13] = 96                                      # d outside {64, 128}
    assert L.csa_attend_noalloc(*bad) == _lib.CSA_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_matches_workspace_attention_twice(L):
    """Two calls in a row (different inputs and shapes) through the shared
    array, each against csa_attend on the same inputs."""
    import torch

    import csa_synth as S
    from tests._parity import assert_attention_close

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream().cuda_stream

    def case(seed, B, N, k, W, H, d, t):
        g = torch.Generator().manual_seed(seed)
        q = S.normal_bf16(seed, S.TID["q"], (B, 1, H, d), dev)
        kc = S.normal_bf16(seed, S.TID["k_cmp"], (B, N, d), dev)
        vc = S.normal_bf16(seed, S.TID["v_cmp"], (B, N, d), dev)
        T_raw = 2 * W
        kr = S.normal_bf16(seed, S.TID["k_raw"], (B, T_raw, d), dev)
        vr = S.normal_bf16(seed, S.TID["v_raw"], (B, T_raw, d), dev)
        n_vis = (t + 1) // 4
        idx = torch.stack([torch.sort(torch.randperm(n_vis, generator=g)[:k])[0] for _ in range(B)])
        idx = idx.to(torch.int32).view(B, 1, k).to(dev)
        idx[:, :, -3:] = -1                               # a few skipped slots
        qp = torch.full((B, 1), t, dtype=torch.int32, device=dev)
        rb = torch.full((B,), t + 1 - T_raw, dtype=torch.int32, device=dev)
        return dict(q=q, kc=kc, vc=vc, kr=kr, vr=vr, idx=idx, qp=qp, rb=rb, B=B, N=N, k=k, W=W, H=H,
                    d=d, T_raw=T_raw)

    def run(c, noalloc):
        out = torch.empty(c["B"], 1, c["H"], c["d"], dtype=torch.float32, device=dev)
        lse = torch.empty(c["B"], 1, c["H"], dtype=torch.float32, device=dev)
        common = (c["q"].data_ptr(), c["kc"].data_ptr(), c["vc"].data_ptr(), c["idx"].data_ptr(),
                  c["kr"].data_ptr(), c["vr"].data_ptr(), c["rb"].data_ptr(), c["qp"].data_ptr(),
                  c["B"], 1, c["N"], c["T_raw"], c["H"], c["d"], c["k"], c["W"], 0.0,
                  out.data_ptr(), _lib.CSA_F32, lse.data_ptr())
        if noalloc:
            r = L.csa_attend_noalloc(*common, st)
        else:
            need = ctypes.c_size_t(0)
            assert L.csa_attend_workspace(c["B"], 1, c["H"], c["d"], c["k"], c["W"], ctypes.byref(need)) == 0
            ws = torch.empty(need.value + 256, dtype=torch.uint8, device=dev)
            base = (ws.data_ptr() + 255) // 256 * 256
            assert L.csa_workspace_init(base, need.value, st) == 0
            r = L.csa_attend(*common, base, need.value, st)
        assert r == _lib.CSA_OK, _lib.lib().csa_status_string(r)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy()

    # two calls in a row whose split partials go through the shared array (over
    # 131072 keys per query), then a 1M-decode-shaped call that merges inside
    # a thread-block cluster and does not touch it
    cases = [case(21, 2, 150000, 139264, 128, 64, 128, 4 * 150000 - 1),
             case(22, 3, 140000, 135000, 64, 32, 64, 4 * 140000 - 1),
             case(23, 4, 65536, 1024, 128, 64, 128, 262143)]
    import oracle as O
    from tests._parity import bits

    for c in cases:
        ref_o, ref_l = run(c, noalloc=False)
        got_o, got_l = run(c, noalloc=True)
        assert_attention_close(got_o, ref_o.astype(np.float64), "noalloc vs workspace output")
        np.testing.assert_allclose(got_l, ref_l, rtol=1e-4, atol=1e-4)
        # and against the oracle itself on the first and last query of the call
        t = int(c["qp"][0, 0])
        for b in (0, c["B"] - 1):
            win = O.window_rows(t, c["W"], int(c["rb"][b]), c["T_raw"])
            o, lse = O.attend_one(O.bf16_to_f64(bits(c["q"][b, 0])), O.bf16_to_f64(bits(c["kc"][b])),
                                  O.bf16_to_f64(bits(c["vc"][b])), c["idx"][b, 0].cpu().numpy(),
                                  O.bf16_to_f64(bits(c["kr"][b])), O.bf16_to_f64(bits(c["vr"][b])), win,
                                  1 / np.sqrt(c["d"]))
            assert_attention_close(got_o[b, 0], o, f"noalloc vs oracle, H={c['H']} d={c['d']} b={b}")
            np.testing.assert_allclose(got_l[b, 0], lse, rtol=1e-4, atol=1e-4)
