// (4) Attention over the selected compressed entries merged with the sliding
// window of raw tokens (CSA), and the dense HCA mode.
// "DeepSeek V4 technical review", section 2.1: attention runs only over the
// selected compressed blocks; octagono "Hybrid Attention: CSA and HCA": a
// window over the most recent 128 raw tokens gives local context, and HCA
// attends to every (heavily) compressed entry.  For query (n, j) at position
// t and head h, with K/V shared by all heads:
//   keys J = {k_cmp[idx[i]] : idx[i] >= 0}  ++  {k_raw[u - raw_base] : t-W < u <= t, u >= 0}
//   out[h] = sum_{x in J} softmax_x(scale * q[h] . K_x) V_x    (one softmax over J)
//
// Design: a query's key list J is a virtual sequence of n_c compressed slots
// followed by W window slots.  It is cut into 64-key tiles; a CTA (4 warps)
// handles one query and a contiguous range of tiles (split-KV), gathering the
// tile's K and V rows into XOR-swizzled shared memory with 16-byte cp.async
// (double-buffered; invalid slots are zero-filled and masked with -inf).
// Warps are (head group of 16) x (key sub-range of the tile): S = Q K^T and
// O += P V run on mma.sync m16n8k16 (bf16 in, fp32 out) with an online
// softmax in the log2 domain.  Sub-range partials merge in shared memory.
// The key-range splits of one query (up to 16) form a thread-block cluster:
// each CTA publishes its (O, max, sum) in shared memory and then folds every
// split's partial into its slice of the output through distributed shared
// memory, in split order, so results never depend on scheduling.  Longer key
// lists keep split partials in the workspace and merge in a second kernel.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kThreads = 128;
constexpr int kTile = 64;  // keys per tile
constexpr int kMaxTilesPerCta = 128;
constexpr int kMaxCluster = 16;  // CTAs of one query merged through distributed shared memory
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

// mode: 0 = one split (write the output), 1 = split partials to global
// memory (merged by attend_combine_kernel), 2 = the splits of a query form a
// thread-block cluster and merge through distributed shared memory.
template <int D, int HG>
__global__ void __launch_bounds__(kThreads) attend_kernel(AttendArgs a, int nsplit, int tps, int mode) {
  pdl_wait_then_release();
  constexpr int KS = 4 / HG;      // key sub-ranges per tile
  constexpr int KW = kTile / KS;  // keys per warp per tile: 64, 32, 16
  constexpr int CH = D / 8;       // 16-byte chunks per row
  constexpr int NT = KW / 8;      // S n-tiles per warp
  constexpr int DT = D / 8;       // O n-tiles
  constexpr int TILE_BYTES = kTile * D * 2;

  extern __shared__ __align__(128) char smem[];
  char* Ks = smem;                    // [2][kTile][D]
  char* Vs = smem + 2 * TILE_BYTES;   // [2][kTile][D]
  int* codes = reinterpret_cast<int*>(smem + 4 * TILE_BYTES);  // [tps * kTile] slot row codes

  const int split = blockIdx.x;
  const long long qi = blockIdx.y;
  const int b = static_cast<int>(qi / a.Tq);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hg = warp % HG, ks = warp / HG;
  const int g = lane >> 2, c = lane & 3;

  const int t = a.q_pos[qi];
  int n_c;
  if (a.idx) {
    n_c = a.k;
  } else {
    n_c = t >= 0 ? (t + 1) / a.m : 0;
    n_c = n_c < a.N ? n_c : a.N;
  }
  const int L = n_c + a.W;
  const int n_tiles = (L + kTile - 1) / kTile;
  const int tile0 = split * tps;
  const int tile1 = min(n_tiles, tile0 + tps);

  // Q fragments (rows h = hg*16 + g and + 8), zero for heads >= H
  uint32_t qf[D / 16][4];
  {
    const int h0 = hg * 16 + g, h1 = h0 + 8;
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(
        static_cast<const char*>(a.q) + (static_cast<size_t>(qi) * a.H + h0) * D * 2);
    const uint32_t* q1 = reinterpret_cast<const uint32_t*>(
        static_cast<const char*>(a.q) + (static_cast<size_t>(qi) * a.H + h1) * D * 2);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[kk][0] = h0 < a.H ? q0[kk * 8 + c] : 0u;
      qf[kk][1] = h1 < a.H ? q1[kk * 8 + c] : 0u;
      qf[kk][2] = h0 < a.H ? q0[kk * 8 + 4 + c] : 0u;
      qf[kk][3] = h1 < a.H ? q1[kk * 8 + 4 + c] : 0u;
    }
  }

  float o[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = a.scale * kLog2e;

  // resolve every key slot of this CTA's tile range once (one coalesced pass
  // over the index list), so the gathers below need no dependent loads
  {
    const int raw_base = a.W > 0 ? a.raw_base[b] : 0;
    bool bad = false;
    const int nslots = (tile1 - tile0) * kTile;
    for (int i = tid; i < nslots; i += kThreads)
      codes[i] = slot_code(a, qi, b, t, n_c, raw_base, tile0 * kTile + i, &bad);
    if (bad) raise_flag(a.errw, kFlagIndex);
  }
  __syncthreads();
  const char* kc_base = static_cast<const char*>(a.k_cmp) + static_cast<size_t>(b) * a.N * D * 2;
  const char* vc_base = static_cast<const char*>(a.v_cmp) + static_cast<size_t>(b) * a.N * D * 2;
  const char* kr_base = static_cast<const char*>(a.k_raw) + static_cast<size_t>(b) * a.T_raw * D * 2;
  const char* vr_base = static_cast<const char*>(a.v_raw) + static_cast<size_t>(b) * a.T_raw * D * 2;

  auto load_tile = [&](int stage, int tile) {
    const int* cs = codes + (tile - tile0) * kTile;
#pragma unroll
    for (int rr = 0; rr < kTile * CH / kThreads; ++rr) {
      const int i = tid + rr * kThreads;
      const int r = i / CH, ch = i % CH;
      const int code = cs[r];
      const char* ks = code >= 0 ? kc_base + static_cast<size_t>(code) * D * 2
                                 : kr_base + static_cast<size_t>(code <= -2 ? -code - 2 : 0) * D * 2;
      const char* vs = code >= 0 ? vc_base + static_cast<size_t>(code) * D * 2
                                 : vr_base + static_cast<size_t>(code <= -2 ? -code - 2 : 0) * D * 2;
      const bool valid = code != -1;
      cp_async16(Ks + stage * TILE_BYTES + swz<D>(r, ch), valid ? ks + ch * 16 : kc_base, valid);
      cp_async16(Vs + stage * TILE_BYTES + swz<D>(r, ch), valid ? vs + ch * 16 : vc_base, valid);
    }
    cp_async_commit();
  };

  if (tile0 < tile1) load_tile(0, tile0);
  for (int tile = tile0; tile < tile1; ++tile) {
    const int stage = (tile - tile0) & 1;
    if (tile + 1 < tile1) {
      load_tile(stage ^ 1, tile + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const int* cs = codes + (tile - tile0) * kTile + ks * KW;
    bool any = false;
#pragma unroll
    for (int i = 0; i < KW; i += 32) any |= __any_sync(0xffffffffu, cs[min(i + lane, KW - 1)] != -1);
    if (any) {
      const char* Kt = Ks + stage * TILE_BYTES;
      const char* Vt = Vs + stage * TILE_BYTES;
      // ---- S = Q K^T over this warp's KW keys
      float s[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int jp = 0; jp < NT / 2; ++jp) {
          uint32_t r[4];
          const int key = ks * KW + jp * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int ch = 2 * kk + ((lane >> 3) & 1);
          ldsm_x4(r, Kt + swz<D>(key, ch));
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
          const int key = ks * KW + kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
          const int ch = 2 * dp + (lane >> 4);
          ldsm_x4_t(r, Vt + swz<D>(key, ch));
          mma_16816(o[2 * dp], af, r[0], r[1]);
          mma_16816(o[2 * dp + 1], af, r[2], r[3]);
        }
      }
    }
    __syncthreads();
  }

  // ---- per-row totals over the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- merge the KS key sub-ranges of each head group (shared memory)
  if constexpr (KS > 1) {
    float* xo = reinterpret_cast<float*>(smem);                 // [4 warps][16][D]
    float* xm = reinterpret_cast<float*>(smem + 4 * 16 * D * 4);  // [4 warps][16]
    float* xl = xm + 4 * 16;
    float* mo = xo + warp * 16 * D;
#pragma unroll
    for (int i = 0; i < DT; ++i) {
      mo[g * D + 8 * i + 2 * c] = o[i][0];
      mo[g * D + 8 * i + 2 * c + 1] = o[i][1];
      mo[(g + 8) * D + 8 * i + 2 * c] = o[i][2];
      mo[(g + 8) * D + 8 * i + 2 * c + 1] = o[i][3];
    }
    if (c == 0) {
      xm[warp * 16 + g] = m0;
      xm[warp * 16 + g + 8] = m1;
      xl[warp * 16 + g] = l0;
      xl[warp * 16 + g + 8] = l1;
    }
    __syncthreads();
    if (ks == 0) {
      float M0 = -INFINITY, M1 = -INFINITY;
      for (int k2 = 0; k2 < KS; ++k2) {
        const int w2 = hg + k2 * HG;
        M0 = fmaxf(M0, xm[w2 * 16 + g]);
        M1 = fmaxf(M1, xm[w2 * 16 + g + 8]);
      }
      const float R0 = M0 == -INFINITY ? 0.f : M0, R1 = M1 == -INFINITY ? 0.f : M1;
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      for (int k2 = 0; k2 < KS; ++k2) {
        const int w2 = hg + k2 * HG;
        const float f0 = ex2(xm[w2 * 16 + g] - R0), f1 = ex2(xm[w2 * 16 + g + 8] - R1);
        L0 += f0 * xl[w2 * 16 + g];
        L1 += f1 * xl[w2 * 16 + g + 8];
        const float* so = xo + w2 * 16 * D;
#pragma unroll
        for (int i = 0; i < DT; ++i) {
          o[i][0] += f0 * so[g * D + 8 * i + 2 * c];
          o[i][1] += f0 * so[g * D + 8 * i + 2 * c + 1];
          o[i][2] += f1 * so[(g + 8) * D + 8 * i + 2 * c];
          o[i][3] += f1 * so[(g + 8) * D + 8 * i + 2 * c + 1];
        }
      }
      m0 = M0;
      m1 = M1;
      l0 = L0;
      l1 = L1;
    }
  }
  const int h0 = hg * 16 + g, h1 = h0 + 8;
  if (mode == 2) {
    // ---- cluster merge: every CTA publishes (o, m, l) in its shared memory,
    // then owns a slice of the (head, column) outputs and folds the cluster's
    // partials into it in split order
    float* po = reinterpret_cast<float*>(smem);   // [H][D] unnormalised
    float* pm = po + a.H * D;                      // [H] running max (log2 domain)
    float* pl = pm + a.H;                          // [H] sum of exponentials
    __syncthreads();                               // the merge above is done with smem
    if (ks == 0) {
#pragma unroll
      for (int i = 0; i < DT; ++i) {
        const int col = 8 * i + 2 * c;
        if (h0 < a.H) *reinterpret_cast<float2*>(po + h0 * D + col) = make_float2(o[i][0], o[i][1]);
        if (h1 < a.H) *reinterpret_cast<float2*>(po + h1 * D + col) = make_float2(o[i][2], o[i][3]);
      }
      if (c == 0) {
        if (h0 < a.H) {
          pm[h0] = m0;
          pl[h0] = l0;
        }
        if (h1 < a.H) {
          pm[h1] = m1;
          pl[h1] = l1;
        }
      }
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    // every split's (max, sum) of every head, fetched once into local shared
    // memory (after the partial o, which nothing overwrites)
    float* wgt = pl + a.H;  // [kMaxCluster][H] weights 2^(m_r - M) / L
    for (int i = tid; i < C * a.H; i += kThreads) {
      const int r = i / a.H, h = i % a.H;
      wgt[i] = *cluster.map_shared_rank(pm + h, r);
      wgt[kMaxCluster * a.H + i] = *cluster.map_shared_rank(pl + h, r);
    }
    __syncthreads();
    if (tid < a.H) {
      const int h = tid;
      float M = -INFINITY;
      for (int r = 0; r < C; ++r) M = fmaxf(M, wgt[r * a.H + h]);
      float den = 0.f;
      for (int r = 0; r < C; ++r) {
        const float f = M == -INFINITY ? 0.f : ex2(wgt[r * a.H + h] - M);
        wgt[r * a.H + h] = f;
        den = fmaf(f, wgt[kMaxCluster * a.H + r * a.H + h], den);
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      for (int r = 0; r < C; ++r) wgt[r * a.H + h] *= inv;
      if (a.lse && rank == 0) a.lse[qi * a.H + h] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    // this CTA's slice of the output, four columns per thread, all splits'
    // partials requested before any is used
    const int n4 = a.H * D / 4;
    for (int e4 = rank * kThreads + tid; e4 < n4; e4 += C * kThreads) {
      const int h = (4 * e4) / D;
      float4 v[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < C) v[r] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(po + 4 * e4, r));
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r < C) {
          const float f = wgt[r * a.H + h];
          acc.x = fmaf(f, v[r].x, acc.x);
          acc.y = fmaf(f, v[r].y, acc.y);
          acc.z = fmaf(f, v[r].z, acc.z);
          acc.w = fmaf(f, v[r].w, acc.w);
        }
      }
      const long long o0 = qi * static_cast<long long>(a.H) * D + 4 * e4;
      if (a.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o0) = acc;
      } else {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + o0) = pk;
      }
    }
    cluster.sync();  // peers may still read this CTA's partials until here
    return;
  }
  if (ks != 0) return;

  // ---- write: final output (single split) or the split partial
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const float lse0 = l0 > 0.f ? m0 + __log2f(l0) : -INFINITY;
  const float lse1 = l1 > 0.f ? m1 + __log2f(l1) : -INFINITY;
  if (mode == 0) {
#pragma unroll
    for (int i = 0; i < DT; ++i) {
      const int col = 8 * i + 2 * c;
      if (a.out_f32) {
        float* op = static_cast<float*>(a.out);
        if (h0 < a.H)
          *reinterpret_cast<float2*>(op + (static_cast<size_t>(qi) * a.H + h0) * D + col) =
              make_float2(o[i][0] * inv0, o[i][1] * inv0);
        if (h1 < a.H)
          *reinterpret_cast<float2*>(op + (static_cast<size_t>(qi) * a.H + h1) * D + col) =
              make_float2(o[i][2] * inv1, o[i][3] * inv1);
      } else {
        uint32_t* op = static_cast<uint32_t*>(a.out);
        if (h0 < a.H)
          op[((static_cast<size_t>(qi) * a.H + h0) * D + col) / 2] = pack_bf16x2(o[i][0] * inv0, o[i][1] * inv0);
        if (h1 < a.H)
          op[((static_cast<size_t>(qi) * a.H + h1) * D + col) / 2] = pack_bf16x2(o[i][2] * inv1, o[i][3] * inv1);
      }
    }
    if (a.lse && c == 0) {
      if (h0 < a.H) a.lse[qi * a.H + h0] = lse0 * kLn2;
      if (h1 < a.H) a.lse[qi * a.H + h1] = lse1 * kLn2;
    }
  } else {
    // partial layout: [nq][nsplit][H][D + 1]  (normalised O, then log2-sum-exp)
    const size_t stride = D + 1;
    float* pb = a.part + (static_cast<size_t>(qi) * nsplit + split) * a.H * stride;
#pragma unroll
    for (int i = 0; i < DT; ++i) {
      const int col = 8 * i + 2 * c;
      if (h0 < a.H) {
        pb[h0 * stride + col] = o[i][0] * inv0;
        pb[h0 * stride + col + 1] = o[i][1] * inv0;
      }
      if (h1 < a.H) {
        pb[h1 * stride + col] = o[i][2] * inv1;
        pb[h1 * stride + col + 1] = o[i][3] * inv1;
      }
    }
    if (c == 0) {
      if (h0 < a.H) pb[h0 * stride + D] = lse0;
      if (h1 < a.H) pb[h1 * stride + D] = lse1;
    }
  }
}

// Merge split partials of one (query, head) in split order.
template <int D>
__global__ void __launch_bounds__(D) attend_combine_kernel(AttendArgs a, int nsplit) {
  pdl_wait_then_release();
  const long long qh = blockIdx.x;  // qi * H + h
  const long long qi = qh / a.H;
  const int h = static_cast<int>(qh % a.H);
  const size_t stride = D + 1;
  const float* pb = a.part + static_cast<size_t>(qi) * nsplit * a.H * stride + h * stride;
  const size_t sstride = static_cast<size_t>(a.H) * stride;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pb[s * sstride + D]);
  float acc = 0.f, den = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float f = ex2(pb[s * sstride + D] - M);
      den += f;
      acc = fmaf(f, pb[s * sstride + threadIdx.x], acc);
    }
  }
  const float val = den > 0.f ? acc / den : 0.f;
  if (a.out_f32)
    static_cast<float*>(a.out)[qh * D + threadIdx.x] = val;
  else
    static_cast<__nv_bfloat16*>(a.out)[qh * D + threadIdx.x] = __float2bfloat16_rn(val);
  if (a.lse && threadIdx.x == 0) a.lse[qh] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
}

template <int D, int HG>
cudaError_t launch_impl(const AttendArgs& a, const AttendPlan& p, cudaStream_t s) {
  constexpr int TILE_BYTES = kTile * D * 2;
  constexpr int KS = 4 / HG;
  size_t smem = 4 * TILE_BYTES + static_cast<size_t>(p.tiles_per_split) * kTile * sizeof(int);
  if (KS > 1) {
    const size_t need = 4 * 16 * D * 4 + 2 * 4 * 16 * 4;
    smem = smem > need ? smem : need;
  }
  if (p.mode == 2) {
    // the CTA's partial (o, m, l), then every split's (m, l) of every head
    const size_t need = static_cast<size_t>(a.H) * (D + 2 + 2 * kMaxCluster) * 4;
    smem = smem > need ? smem : need;
  }
  cudaError_t e = ensure_dyn_smem<attend_kernel<D, HG>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  const dim3 grid(p.nsplit, static_cast<unsigned>(nq));
  if (p.mode == 2 && p.nsplit > 8) {
    static bool nonportable_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!nonportable_set[dev]) {
      e = cudaFuncSetAttribute(attend_kernel<D, HG>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      nonportable_set[dev] = true;
    }
  }
  e = launch_k(attend_kernel<D, HG>, grid, dim3(kThreads), smem, s, p.mode == 2 ? p.nsplit : 1, a, p.nsplit,
               p.tiles_per_split, p.mode);
  if (e != cudaSuccess || p.mode != 1) return e;
  return launch_k(attend_combine_kernel<D>, dim3(static_cast<unsigned>(nq * a.H)), dim3(D), 0, s, 1, a,
                  p.nsplit);
}

template <int D>
cudaError_t launch_d(const AttendArgs& a, const AttendPlan& p, cudaStream_t s) {
  const int hg = (a.H + 15) / 16;
  if (hg <= 1) return launch_impl<D, 1>(a, p, s);
  if (hg <= 2) return launch_impl<D, 2>(a, p, s);
  return launch_impl<D, 4>(a, p, s);
}

}  // namespace

AttendPlan plan_attend(int Tq, long long nq, int n_keys_max, int H, int d) {
  // The split depends only on the queries per sequence and the key count, never
  // on the batch size or the GPU, so a sequence gives bit-identical results
  // alone or inside any batch.  Prefill-like calls (many queries per sequence)
  // fill the GPU without splitting (up to 128 tiles per CTA); decode-like calls
  // split every query's keys over up to kMaxCluster CTAs.  Up to kMaxCluster
  // splits of a query run as one thread-block cluster and merge through
  // distributed shared memory; more splits (over kMaxCluster * 128 tiles) keep
  // their partials in the workspace and merge in a second kernel.
  AttendPlan p;
  const int n_tiles = (n_keys_max + kTile - 1) / kTile;
  int tps;
  if (Tq >= 16) {
    tps = n_tiles < kMaxTilesPerCta ? n_tiles : kMaxTilesPerCta;
  } else {
    tps = (n_tiles + kMaxCluster - 1) / kMaxCluster;
    tps = tps > kMaxTilesPerCta ? kMaxTilesPerCta : tps;
  }
  if (tps > n_tiles) tps = n_tiles;
  if (tps < 1) tps = 1;
  p.tiles_per_split = tps;
  p.nsplit = n_tiles > 0 ? (n_tiles + tps - 1) / tps : 1;
  p.mode = p.nsplit == 1 ? 0 : (p.nsplit <= kMaxCluster ? 2 : 1);
  p.part_bytes = p.mode == 1 ? static_cast<size_t>(nq) * p.nsplit * H * (d + 1) * sizeof(float) : 0;
  return p;
}

cudaError_t launch_attend(const AttendArgs& a, const AttendPlan& p, cudaStream_t s) {
  if (static_cast<long long>(a.B) * a.Tq == 0) return cudaSuccess;
  if (a.d == 128) return launch_d<128>(a, p, s);
  if (a.d == 64) return launch_d<64>(a, p, s);
  return cudaErrorNotSupported;
}

}  // namespace csa
