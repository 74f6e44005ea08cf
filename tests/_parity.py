"""Acceptance rules shared by the GPU parity tests.

* compressed entries, fp32 output: |gpu - ref| <= 1e-3 * sum_j p_j |x_j| (the
  softmax-weighted magnitude, which bounds |ref| and avoids blow-ups where the
  pooled value cancels);  bf16 output: the same budget plus the final
  rounding, |gpu - ref| <= 1e-3 * sum_j p_j |x_j| + ulp_bf16(ref) / 2, and
  bit-equal to the oracle's bf16 rounding on >= 99.9% of entries (one bf16 ulp
  everywhere cannot hold where the pooled value cancels towards zero);
* top-k indices: bit-exact, except at near-ties -- the valid counts match and
  every index in the symmetric difference has an oracle score within 1e-3 of
  the oracle's k-th largest score (relative);
* attention: |err| <= 1e-2 + 1e-2 * |ref| (fp32 accumulation, bf16 inputs).
"""
import numpy as np
import torch

import csa_synth as S
import oracle as O

ATT_ATOL = 1e-2
ATT_RTOL = 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return S.bf16_bits(t)


def assert_attention_close(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    err = np.abs(gpu.astype(np.float64) - ref)
    lim = ATT_ATOL + ATT_RTOL * np.abs(ref)
    bad = err > lim
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside 1e-2+1e-2|ref|, max err {err.max():.3g}"


def assert_compressed_f32(gpu: np.ndarray, ref: np.ndarray, scale: np.ndarray, what: str = "") -> None:
    err = np.abs(gpu.astype(np.float64) - ref)
    bad = err > 1e-3 * scale + 1e-30
    assert not bad.any(), f"{what}: {bad.sum()} entries beyond 1e-3 * sum p|x| (max rel {np.max(err / (scale + 1e-30)):.3g})"


def assert_compressed_bf16(gpu_bits: np.ndarray, ref_f64: np.ndarray, scale: np.ndarray, what: str = "") -> None:
    g = O.bf16_to_f64(gpu_bits)
    half_ulp = np.ldexp(1.0, np.frexp(np.abs(ref_f64))[1] - 9)
    err = np.abs(g - ref_f64)
    lim = 1e-3 * scale + half_ulp
    bad = err > lim
    if bad.any():
        i = np.argmax(err / lim)
        raise AssertionError(f"{what}: {bad.sum()} entries beyond 1e-3*sum p|x| + ulp/2 (worst: gpu "
                             f"{g.flat[i]:.6g}, ref {ref_f64.flat[i]:.6g}, sum p|x| {scale.flat[i]:.4g})")
    frac = np.mean(gpu_bits == O.round_bf16(ref_f64))
    assert frac >= 0.999, f"{what}: only {frac:.5f} bit-equal to the oracle's bf16 rounding"


def check_topk_near_tie(gpu_idx: np.ndarray, ref_idx: np.ndarray, ref_scores: np.ndarray, k: int,
                        what: str = "") -> int:
    """One query.  Returns the number of near-tie swaps accepted."""
    n = ref_scores.shape[0]
    valid = gpu_idx[gpu_idx >= 0]
    # structure: ascending, unique, visible, padded at the end
    assert np.all(np.diff(valid) > 0), f"{what}: not strictly ascending"
    assert np.all(gpu_idx[len(valid):] == -1), f"{what}: padding not at the end"
    assert valid.size == 0 or (valid[0] >= 0 and valid[-1] < n), f"{what}: invisible block selected"
    assert valid.size == min(k, n), f"{what}: {valid.size} kept, want {min(k, n)}"
    if np.array_equal(gpu_idx, ref_idx):
        return 0
    g = set(valid.tolist())
    r = set(ref_idx[ref_idx >= 0].tolist())
    diff = sorted(g ^ r)
    sk = np.sort(ref_scores)[::-1][min(k, n) - 1]
    far = [b for b in diff if abs(ref_scores[b] - sk) > 1e-3 * abs(sk)]
    assert not far, f"{what}: {len(far)} index differences are not near-ties (e.g. {far[:5]})"
    return len(diff)


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, scale: np.ndarray, what: str = "") -> None:
    """fp32 tensor-core scores vs float64: error relative to sum_h w_h |q_h|.|k|."""
    err = np.abs(gpu.astype(np.float64) - ref)
    bad = err > 1e-4 * scale + 1e-6
    assert not bad.any(), f"{what}: {bad.sum()} scores off (max rel {np.max(err / (scale + 1e-12)):.3g})"


def index_scale(q_idx: np.ndarray, k_idx: np.ndarray, w: np.ndarray) -> np.ndarray:
    """sum_h w_h * (|q_h| . |k_b|) for one query: [H_I, d_I] x [n, d_I] -> [n]."""
    return (np.abs(k_idx) @ np.abs(q_idx).T) @ np.abs(w)


def random_selection(rng, n_vis: int, k: int, extra_minus=False) -> np.ndarray:
    """A valid index list: min(k, n_vis) distinct visible blocks, ascending, -1 padded."""
    c = min(k, n_vis)
    sel = np.sort(rng.choice(n_vis, size=c, replace=False)) if c else np.zeros(0, np.int64)
    out = np.full(k, -1, dtype=np.int32)
    out[:c] = sel
    if extra_minus and c > 4:
        out[c // 2] = -1  # a hole in the middle must be skipped
    return out
