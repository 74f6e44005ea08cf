// Attention building blocks shared by the attention kernels and the fused
// decode tail: virtual key slots (selected compressed rows, then the raw
// window), the XOR-swizzled K/V tile layout, and one warp's share of one
// staged tile on mma.sync (S = Q K^T, online softmax, O += P V).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace csa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Row code of virtual key slot vk of query (qi, b, t): >= 0 a compressed row,
// <= -2 the raw-window row (-code - 2), -1 no key.  *bad is set for an index
// or window row outside its buffer (the slot is then skipped).
__device__ __forceinline__ int slot_code(const AttendArgs& a, long long qi, int b, int t, int n_c,
                                         int raw_base, int vk, bool* bad) {
  if (vk < n_c) {
    const int row = a.idx ? a.idx[qi * a.k + vk] : vk;
    if (row < 0) return -1;
    if (row >= a.N) {
      *bad = true;
      return -1;
    }
    return row;
  }
  const int w = vk - n_c;
  const int u = t - a.W + 1 + w;
  if (w >= a.W || u < 0) return -1;
  const int r = u - raw_base;
  if (r < 0 || r >= a.T_raw) {
    *bad = true;
    return -1;
  }
  return -r - 2;
}

// byte offset of 16-byte chunk ch of row r in a swizzled [rows][D] bf16 tile
template <int D>
__device__ __forceinline__ int swz(int r, int ch) {
  return r * (D * 2) + ((ch ^ (r & 7)) << 4);
}

// byte offset of chunk ch of row r in a K/V tile: swizzled rows (PITCH = 0),
// or plain rows PITCH bytes apart (PITCH = D * 2 + 16: each row contiguous,
// and the 16-byte pad spreads the eight rows of an ldmatrix phase over all
// banks)
template <int D, int PITCH>
__device__ __forceinline__ int kv_off(int r, int ch) {
  if constexpr (PITCH == 0)
    return swz<D>(r, ch);
  else
    return r * PITCH + (ch << 4);
}

// One warp's share of one staged tile: keys [key0, key0 + KW) of the K/V
// tile (rows addressed through kv_off), slot codes cs[0 .. KW) (-1 = no key),
// for the warp's 16 query heads (fragments qf).  S = Q K^T on mma.sync, the
// online softmax in the log2 domain (sl2 = scale * log2 e), then O += P V.
// Updates the running (o, m, l) of the warp's rows g and g + 8.
template <int D, int KW, int PITCH = 0>
__device__ __forceinline__ void tile_step(const uint32_t (&qf)[D / 16][4], const char* Kt, const char* Vt,
                                          int key0, const int* cs, float sl2, float (&o)[D / 8][4], float& m0,
                                          float& m1, float& l0, float& l1) {
  constexpr int NT = KW / 8;  // S n-tiles
  constexpr int DT = D / 8;   // O n-tiles
  const int lane = threadIdx.x & 31, c = lane & 3;
  bool any = false;
#pragma unroll
  for (int i = 0; i < KW; i += 32) any |= __any_sync(0xffffffffu, cs[min(i + lane, KW - 1)] != -1);
  if (!any) return;
  // ---- S = Q K^T over this warp's KW keys
  float s[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int jp = 0; jp < NT / 2; ++jp) {
      uint32_t r[4];
      const int key = key0 + jp * 16 + ((lane >> 4) << 3) + (lane & 7);
      const int ch = 2 * kk + ((lane >> 3) & 1);
      ldsm_x4(r, Kt + kv_off<D, PITCH>(key, ch));
      mma_16816(s[2 * jp], qf[kk], r[0], r[1]);
      mma_16816(s[2 * jp + 1], qf[kk], r[2], r[3]);
    }
  }
  // ---- online softmax (log2 domain)
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float b0 = cs[8 * j + 2 * c] != -1 ? 0.f : -INFINITY;
    const float b1 = cs[8 * j + 2 * c + 1] != -1 ? 0.f : -INFINITY;
    s[j][0] = fmaf(s[j][0], sl2, b0);
    s[j][1] = fmaf(s[j][1], sl2, b1);
    s[j][2] = fmaf(s[j][2], sl2, b0);
    s[j][3] = fmaf(s[j][3], sl2, b1);
    mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
    mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
  const float r0 = n0 == -INFINITY ? 0.f : n0;
  const float r1 = n1 == -INFINITY ? 0.f : n1;
  const float al0 = ex2(m0 - r0), al1 = ex2(m1 - r1);
  m0 = n0;
  m1 = n1;
  l0 *= al0;
  l1 *= al1;
#pragma unroll
  for (int i = 0; i < DT; ++i) {
    o[i][0] *= al0;
    o[i][1] *= al0;
    o[i][2] *= al1;
    o[i][3] *= al1;
  }
  uint32_t pf[KW / 16][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float p0 = ex2(s[j][0] - r0), p1 = ex2(s[j][1] - r0);
    const float p2 = ex2(s[j][2] - r1), p3 = ex2(s[j][3] - r1);
    l0 += p0 + p1;
    l1 += p2 + p3;
    pf[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
    pf[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
  }
  // ---- O += P V
#pragma unroll
  for (int kk = 0; kk < KW / 16; ++kk) {
    // A fragment order: (g, k-lo), (g+8, k-lo), (g, k-hi), (g+8, k-hi)
    const uint32_t af[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
    for (int dp = 0; dp < DT / 2; ++dp) {
      uint32_t r[4];
      const int key = key0 + kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
      const int ch = 2 * dp + (lane >> 4);
      ldsm_x4_t(r, Vt + kv_off<D, PITCH>(key, ch));
      mma_16816(o[2 * dp], af, r[0], r[1]);
      mma_16816(o[2 * dp + 1], af, r[2], r[3]);
    }
  }
}

}  // namespace
}  // namespace csa
