"""Seeded synthetic inputs for the CSA / HCA attention path.

This module is shared by both sides of every parity check: the CUDA library's
tests and benchmark, and the CPU oracle's tests.  It holds no arithmetic of the
method itself -- only counter-based random draws and the shapes of the
workloads -- so that neither side depends on the other.

Generator (one definition, evaluated with the same integer operations on the
CPU and on a CUDA device, hence bit-identical on both):

* stream key      K = mix(((seed << 20) ^ tensor_id) mod 2^64)
* element draw    h_r(i) = mix(K + (3*i + r + 1) * GAMMA mod 2^64),  r = 0, 1, 2
  where ``mix`` is the SplitMix64 output function of Steele, Lea & Flood,
  "Fast splittable pseudorandom number generators" (OOPSLA 2014), with Vigna's
  constants, and GAMMA = 0x9E3779B97F4A7C15.
* ~N(0, 1): Irwin-Hall sum of the twelve 16-bit lanes of h_0, h_1, h_2:
  z = (S - 6 * 65535) * 2^-16, exact in fp32 (|S - 6*65535| < 2^19), then
  rounded to bf16 with round-to-nearest-even.  Mean 0, variance 1 - 2^-32,
  tails bounded at +-6.
* ~U(0, 1): (h_0 >> 40) * 2^-24, exact in fp32.

Each tensor is a *virtual* full-size array addressed by its flat row-major
index, so any sub-block (a few sampled rows, the queries at chosen positions)
can be regenerated on demand without materialising the rest.

Workload shapes follow the five configurations the CSA/HCA method is measured
on (DeepSeek-V4 pages: CSA every m=4 tokens, top-1024, a 128-token window,
indexer 64 heads x 128; HCA every m'=128 tokens).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# tensor ids (part of the stream key): fixed forever, so stored expected values
# stay valid.
TID = {
    "q": 1, "q_idx": 2, "k_raw": 3, "v_raw": 4, "i_raw": 5,
    "g_k": 6, "g_v": 7, "g_i": 8, "w": 9,
    "k_cmp": 10, "v_cmp": 11, "i_cmp": 12,
}


def _s64(u: int) -> int:
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def _mix_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tid: int) -> int:
    return _mix_int(((seed << 20) ^ tid) & MASK64)


def _srl(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes viewed as uint64."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(_M1)
    z = (z ^ _srl(z, 27)) * _s64(_M2)
    return z ^ _srl(z, 31)


def hash_u64(seed: int, tid: int, counter: torch.Tensor) -> torch.Tensor:
    """h = mix(K + counter * GAMMA) for an int64 counter tensor (uint64 bits)."""
    return _mix(counter * _s64(GAMMA) + _s64(stream_key(seed, tid)))


_CHUNK = 1 << 24


def normal_bf16_at(seed: int, tid: int, flat: torch.Tensor) -> torch.Tensor:
    """~N(0,1) bf16 draws of tensor ``tid`` at the given flat indices."""
    out = torch.empty(flat.shape, dtype=torch.bfloat16, device=flat.device)
    f = flat.reshape(-1)
    o = out.view(-1)
    for s in range(0, f.numel(), _CHUNK):
        c3 = f[s:s + _CHUNK].to(torch.int64) * 3
        acc = None
        for r in range(3):
            h = hash_u64(seed, tid, c3 + (r + 1))
            for q in range(4):
                lane = _srl(h, 16 * q) & 0xFFFF if q else h & 0xFFFF
                acc = lane if acc is None else acc + lane
        z = (acc - 6 * 65535).to(torch.float32) * (2.0 ** -16)
        o[s:s + _CHUNK] = z.to(torch.bfloat16)
    return out


def normal_bf16(seed: int, tid: int, shape, device="cpu", offset: int = 0) -> torch.Tensor:
    """Contiguous block [offset, offset + prod(shape)) of tensor ``tid``."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        idx = torch.arange(offset + s, offset + e, dtype=torch.int64, device=device)
        out[s:e] = normal_bf16_at(seed, tid, idx)
    return out.view(*shape)


def uniform_f32(seed: int, tid: int, shape, device="cpu") -> torch.Tensor:
    n = 1
    for s in shape:
        n *= int(s)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    h = hash_u64(seed, tid, idx * 3 + 1)
    return (_srl(h, 40).to(torch.float32) * (2.0 ** -24)).view(*shape)


def rows_bf16(seed: int, tid: int, n_rows_total: int, width: int, b: int,
              rows: torch.Tensor) -> torch.Tensor:
    """Rows ``rows`` (int64 tensor) of sequence ``b`` of a virtual [B, n_rows_total, width] tensor."""
    flat = ((b * n_rows_total + rows.to(torch.int64))[:, None] * width
            + torch.arange(width, dtype=torch.int64, device=rows.device)[None, :])
    return normal_bf16_at(seed, tid, flat)


def rows_bf16_heads(seed: int, tid: int, T: int, H: int, width: int, b: int,
                    pos: torch.Tensor) -> torch.Tensor:
    """Rows [len(pos), H, width] of sequence b of a virtual [B, T, H, width] tensor."""
    dev = pos.device
    base = (b * T + pos.to(torch.int64))[:, None, None] * H
    flat = ((base + torch.arange(H, dtype=torch.int64, device=dev)[None, :, None]) * width
            + torch.arange(width, dtype=torch.int64, device=dev)[None, None, :])
    return normal_bf16_at(seed, tid, flat)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one CSA / HCA workload.

    mode: "prefill" -- raw streams of T tokens are compressed and every token
          is a query (q_pos = 0..T-1);
          "decode"  -- the compressed caches (N = T/m entries) are given and
          each sequence asks the queries at ``positions``; the most recent raw
          tokens are given as a window buffer starting at ``raw_base``;
          "hca"     -- the raw streams of T tokens are compressed at m (=128)
          and each sequence asks the queries at ``positions``.
    """
    name: str
    mode: str
    B: int
    T: int
    m: int
    H: int
    d: int
    k: int
    W: int
    seed: int
    H_I: int = 0
    d_I: int = 0
    positions: Optional[tuple] = None   # decode / hca query positions
    raw_len: int = 0                    # decode: raw window buffer length

    @property
    def N(self) -> int:
        return self.T // self.m

    @property
    def Tq(self) -> int:
        return self.T if self.mode == "prefill" else len(self.positions)

    @property
    def q_positions(self) -> List[int]:
        return list(range(self.T)) if self.mode == "prefill" else list(self.positions)

    @property
    def raw_base(self) -> int:
        if self.mode == "decode":
            return self.T - self.raw_len
        return 0

    @property
    def T_raw(self) -> int:
        return self.raw_len if self.mode == "decode" else self.T

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    # B=1, T=256, m=4 (64 entries), H=4, d=64, indexer 4 x 32, top-16, W=32, seed 0
    "tiny_prefill": Workload("tiny_prefill", "prefill", B=1, T=256, m=4, H=4, d=64,
                             k=16, W=32, seed=0, H_I=4, d_I=32),
    # B=1, T=8192, m=4 (2048 entries), H=16, d=128, indexer 64 x 128, top-1024, W=128, seed 1
    "prefill_8k": Workload("prefill_8k", "prefill", B=1, T=8192, m=4, H=16, d=128,
                           k=1024, W=128, seed=1, H_I=64, d_I=128),
    # B=64, one query at 131071, 32768 entries given, H=64, top-1024, W=128, seed 2
    "decode_128k": Workload("decode_128k", "decode", B=64, T=131072, m=4, H=64, d=128,
                            k=1024, W=128, seed=2, H_I=64, d_I=128,
                            positions=(131071,), raw_len=256),
    # B=8, one query at 1048575, m'=128 (8192 entries from 2^20 raw tokens), H=64, W=128, seed 3
    "hca_decode_1m": Workload("hca_decode_1m", "hca", B=8, T=1 << 20, m=128, H=64, d=128,
                              k=0, W=128, seed=3, positions=((1 << 20) - 1,)),
    # B=4, one query at 1048575, 262144 entries given, H=64, top-1024, W=128, seed 4
    "decode_1m": Workload("decode_1m", "decode", B=4, T=1 << 20, m=4, H=64, d=128,
                          k=1024, W=128, seed=4, H_I=64, d_I=128,
                          positions=((1 << 20) - 1,), raw_len=256),
    # the 4-query causal tail of the same 1M-token sequences (same seed, same caches)
    "decode_1m_tail": Workload("decode_1m_tail", "decode", B=4, T=1 << 20, m=4, H=64, d=128,
                               k=1024, W=128, seed=4, H_I=64, d_I=128,
                               positions=tuple(range((1 << 20) - 4, 1 << 20)), raw_len=256),
}


def make_inputs(wl: Workload, device="cpu", batches: Optional[List[int]] = None,
                only: Optional[set] = None) -> Dict[str, torch.Tensor]:
    """Materialise the inputs of ``wl`` (optionally only sequences ``batches``).

    Returned keys depend on the mode:
      prefill: q, q_idx, k_raw, v_raw, i_raw, g_k, g_v, g_i, w, q_pos, raw_base
      decode : q, q_idx, k_cmp, v_cmp, i_cmp, k_raw, v_raw, w, q_pos, raw_base
      hca    : q, k_raw, v_raw, g_k, g_v, q_pos, raw_base
    bf16 tensors are [B, ...] row-major; q_pos [B, Tq] int32; raw_base [B] int32;
    w [H_I] fp32.  ``only`` restricts the result to the named tensors.
    """
    bl = list(range(wl.B)) if batches is None else list(batches)
    s = wl.seed
    pos = torch.tensor(wl.q_positions, dtype=torch.int64, device=device)
    out: Dict[str, torch.Tensor] = {}

    def want(name):
        return only is None or name in only

    def heads(name, H, width):
        return torch.stack([rows_bf16_heads(s, TID[name], wl.T, H, width, b, pos) for b in bl])

    def raw(name, width, base, length):
        rows = torch.arange(base, base + length, dtype=torch.int64, device=device)
        if base == 0 and length == wl.T:
            return torch.stack([normal_bf16(s, TID[name], (wl.T, width), device,
                                            offset=b * wl.T * width) for b in bl])
        return torch.stack([rows_bf16(s, TID[name], wl.T, width, b, rows) for b in bl])

    def cache(name, width):
        return torch.stack([normal_bf16(s, TID[name], (wl.N, width), device,
                                        offset=b * wl.N * width) for b in bl])

    if want("q"):
        out["q"] = heads("q", wl.H, wl.d)
    if wl.mode != "hca":
        if want("q_idx"):
            out["q_idx"] = heads("q_idx", wl.H_I, wl.d_I)
        if want("w"):
            out["w"] = uniform_f32(s, TID["w"], (wl.H_I,), device)
    if wl.mode in ("prefill", "hca"):
        names = ["k_raw", "v_raw", "g_k", "g_v"] + (["i_raw", "g_i"] if wl.mode == "prefill" else [])
        for name in names:
            if want(name):
                out[name] = raw(name, wl.d_I if name in ("i_raw", "g_i") else wl.d, 0, wl.T)
    else:
        for name, width in (("k_cmp", wl.d), ("v_cmp", wl.d), ("i_cmp", wl.d_I)):
            if want(name):
                out[name] = cache(name, width)
        for name in ("k_raw", "v_raw"):
            if want(name):
                out[name] = raw(name, wl.d, wl.raw_base, wl.raw_len)
    out["q_pos"] = pos.to(torch.int32)[None, :].repeat(len(bl), 1).contiguous()
    out["raw_base"] = torch.full((len(bl),), wl.raw_base, dtype=torch.int32, device=device)
    return out


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
