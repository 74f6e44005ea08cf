"""The checking half of __graft_entry__.smoke() on the CPU: the oracle's own
results stand in for the GPU's, so every shape and index the check uses is
exercised without a GPU, and planted mistakes in the stand-in results must be
caught."""
import numpy as np
import pytest

import csa_synth as S

import __graft_entry__ as E


@pytest.fixture(scope="module")
def case():
    wl = S.WORKLOADS["tiny_prefill"]
    c, ref = E.smoke_reference(wl)
    gpu = {key: ref[key].copy() for key in ("k_cmp", "v_cmp", "i_cmp")}
    gpu["idx"] = ref["idx"].copy()
    gpu["out"] = ref["out"].astype(np.float32)
    gpu["out_on_ref"] = ref["out"].astype(np.float32)
    return wl, c, ref, gpu


def test_smoke_check_accepts_the_oracles_own_results(case):
    wl, c, ref, gpu = case
    assert E.smoke_check(wl, c, ref, gpu) == wl.T


def _planted(gpu, key, fn):
    g = {k: v.copy() for k, v in gpu.items()}
    fn(g[key])
    return g


@pytest.mark.parametrize("key,fn", [
    ("out", lambda a: a.__setitem__((0, 100, 2, 5), a[0, 100, 2, 5] + 0.05)),
    ("out_on_ref", lambda a: a.__setitem__((0, 7, 0, 0), -a[0, 7, 0, 0] - 0.1)),
    ("k_cmp", lambda a: a.__setitem__((0, 3, 3), a[0, 3, 3] + 2)),
    ("i_cmp", lambda a: a.__setitem__((0, 60, 31), a[0, 60, 31] ^ 0x8000)),
])
def test_smoke_check_catches_planted_mistakes(case, key, fn):
    wl, c, ref, gpu = case
    with pytest.raises(AssertionError):
        E.smoke_check(wl, c, ref, _planted(gpu, key, fn))


def test_smoke_check_catches_a_wrong_selection(case):
    wl, c, ref, gpu = case
    g = {k: v.copy() for k, v in gpu.items()}
    # keep the lowest visible blocks instead of the best ones on many queries
    for t in range(200, 256):
        n = (t + 1) // wl.m
        g["idx"][0, t, :] = np.arange(wl.k, dtype=np.int32) if n >= wl.k else -1
    with pytest.raises(AssertionError):
        E.smoke_check(wl, c, ref, g)


# ---- the decode-shaped half of smoke(): two sequences over 3000 cached
# entries (the smoke itself runs 20000 and 70000 on the GPU)

@pytest.fixture(scope="module")
def decode_case():
    import math

    import torch

    import oracle as O
    wl = E.smoke_decode_workload(3000)
    inp = S.make_inputs(wl, "cpu")
    c = {k: (S.bf16_bits(v) if v.dtype == torch.bfloat16 else v.numpy()) for k, v in inp.items()}
    B, Tq = c["q_pos"].shape
    idx = np.empty((B, Tq, wl.k), np.int32)
    out = np.empty((B, Tq, wl.H, wl.d), np.float32)
    for b in range(B):
        kc, vc, ic = (O.bf16_to_f64(c[key][b]) for key in ("k_cmp", "v_cmp", "i_cmp"))
        kr, vr = O.bf16_to_f64(c["k_raw"][b]), O.bf16_to_f64(c["v_raw"][b])
        for j in range(Tq):
            t = int(c["q_pos"][b, j])
            s_ref = O.indexer_scores(O.bf16_to_f64(c["q_idx"][b, j]), ic, c["w"].astype(np.float64), t, wl.m)
            idx[b, j] = O.topk(s_ref, wl.k)
            win = O.window_rows(t, wl.W, int(c["raw_base"][b]), kr.shape[0])
            out[b, j], _ = O.attend_one(O.bf16_to_f64(c["q"][b, j]), kc, vc, idx[b, j], kr, vr, win,
                                        1 / math.sqrt(wl.d))
    return wl, c, idx, out


def test_smoke_decode_check_accepts_the_oracles_own_results(decode_case):
    wl, c, idx, out = decode_case
    assert E.smoke_decode_check(wl, c, idx, out) == 2


def test_smoke_decode_check_catches_planted_mistakes(decode_case):
    wl, c, idx, out = decode_case
    bad_out = out.copy()
    bad_out[1, 0, 63, 127] += 0.05
    with pytest.raises(AssertionError):
        E.smoke_decode_check(wl, c, idx, bad_out)
    bad_idx = idx.copy()
    bad_idx[0, 0] = np.arange(wl.k, dtype=np.int32)   # the lowest blocks instead of the best
    with pytest.raises(AssertionError):
        E.smoke_decode_check(wl, c, bad_idx, out)
