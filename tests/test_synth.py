"""The shared seeded input generator: its definition (SplitMix64 output function,
Irwin-Hall of twelve 16-bit lanes), its moments, and its virtual indexing.  CPU only."""
import numpy as np
import torch

import csa_synth as S

GAMMA = np.uint64(0x9E3779B97F4A7C15)


def _np_mix(z):
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def _np_normal(seed, tid, idx):
    key = np.uint64(S.stream_key(seed, tid))
    acc = np.zeros(idx.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        for r in range(3):
            h = _np_mix(key + (np.uint64(3) * idx.astype(np.uint64) + np.uint64(r + 1)) * GAMMA)
            for q in range(4):
                acc += ((h >> np.uint64(16 * q)) & np.uint64(0xFFFF)).astype(np.int64)
    z = ((acc - 6 * 65535).astype(np.float32) * np.float32(2.0 ** -16))
    return torch.from_numpy(z).to(torch.bfloat16)


def test_splitmix_reference_vector():
    # SplitMix64 seeded with 0 yields 0xE220A8397B1DCDAF as its first output
    # (Vigna's reference implementation; state advanced by GAMMA before mixing).
    assert S._mix_int(0 + 0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_generator_matches_numpy_uint64_definition():
    idx = np.arange(0, 200000, dtype=np.int64) * 7919 + 12345
    got = S.normal_bf16_at(3, S.TID["k_raw"], torch.from_numpy(idx))
    want = _np_normal(3, S.TID["k_raw"], idx)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_moments_and_bounds():
    x = S.normal_bf16(1, S.TID["q"], (1 << 20,)).float()
    assert abs(x.mean().item()) < 5e-3
    assert abs(x.var().item() - 1.0) < 1e-2
    assert x.abs().max().item() <= 6.0
    u = S.uniform_f32(1, S.TID["w"], (1 << 16,))
    assert u.min().item() >= 0.0 and u.max().item() < 1.0
    assert abs(u.mean().item() - 0.5) < 1e-2


def test_virtual_indexing_is_consistent():
    wl = S.WORKLOADS["tiny_prefill"]
    full = S.make_inputs(wl)
    sub = S.make_inputs(wl, batches=[0])
    for key in full:
        assert torch.equal(full[key], sub[key]), key
    rows = torch.tensor([3, 17, 200])
    r = S.rows_bf16(wl.seed, S.TID["k_raw"], wl.T, wl.d, 0, rows)
    assert torch.equal(r, full["k_raw"][0, rows])
    qh = S.rows_bf16_heads(wl.seed, S.TID["q"], wl.T, wl.H, wl.d, 0, rows)
    assert torch.equal(qh, full["q"][0, rows])


def test_decode_tail_shares_inputs_with_decode_query():
    """The 1M tail's last query is the 1M decode query: same caches, same q."""
    a = S.WORKLOADS["decode_1m"].replace(T=4096, raw_len=256)
    b = S.WORKLOADS["decode_1m_tail"].replace(T=4096, raw_len=256, positions=(4092, 4093, 4094, 4095))
    a = a.replace(positions=(4095,))
    ia, ib = S.make_inputs(a), S.make_inputs(b)
    assert torch.equal(ia["q"][:, 0], ib["q"][:, 3])
    assert torch.equal(ia["q_idx"][:, 0], ib["q_idx"][:, 3])
    for key in ("k_cmp", "v_cmp", "i_cmp", "k_raw", "v_raw", "w"):
        assert torch.equal(ia[key], ib[key]), key
