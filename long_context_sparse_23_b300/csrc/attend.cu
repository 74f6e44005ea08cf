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

#include "attend_tile.cuh"
#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kMaxKeysPerCta = 8192;  // slot codes staged in shared memory
constexpr int kMaxCluster = 16;  // CTAs of one query merged through distributed shared memory
// mode: 0 = one split (write the output), 1 = split partials to global
// memory (merged by attend_combine_kernel), 2 = the splits of a query form a
// thread-block cluster and merge through distributed shared memory.
// NW warps per CTA (4: 64-key tiles, 8: 128-key tiles); warp = (head group
// of 16, key sub-range), each warp owns 16 * HG keys of every tile.
template <int D, int HG, int NW>
__global__ void __launch_bounds__(32 * NW) attend_kernel(AttendArgs a, int nsplit, int tps, int mode) {
  pdl_wait_then_release();
  constexpr int kThreads = 32 * NW;
  constexpr int kTile = 16 * NW;  // keys per tile
  constexpr int KS = NW / HG;     // key sub-ranges per tile
  constexpr int KW = kTile / KS;  // keys per warp per tile: 16 * HG
  constexpr int CH = D / 8;       // 16-byte chunks per row
  constexpr int DT = D / 8;       // O n-tiles
  constexpr int TILE_BYTES = kTile * D * 2;

  extern __shared__ __align__(128) char smem[];
  const int nstage = tps > 1 ? 2 : 1;         // one tile per CTA needs no second buffer
  char* Ks = smem;                            // [nstage][kTile][D]
  char* Vs = smem + nstage * TILE_BYTES;      // [nstage][kTile][D]
  int* codes = reinterpret_cast<int*>(smem + 2 * nstage * TILE_BYTES);  // [tps * kTile] slot row codes

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

    tile_step<D, KW>(qf, Ks + stage * TILE_BYTES, Vs + stage * TILE_BYTES, ks * KW,
                     codes + (tile - tile0) * kTile + ks * KW, sl2, o, m0, m1, l0, l1);
    __syncthreads();
  }

  // ---- per-row totals over the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  const int h0 = hg * 16 + g, h1 = h0 + 8;
  if (mode == 2) {
    // ---- cluster merge.  Every warp's (o, m, l) over its key sub-range is
    // one partial: partial p = rank * KS + ks of the query.  Each CTA owns a
    // slice of the heads and folds all C * KS partials of them, in partial
    // order, through distributed shared memory.
    constexpr int LDO = D + 4;  // padded row: the warps' row stores do not collide on banks
    float* po = reinterpret_cast<float*>(smem);  // [KS][H][LDO] unnormalised o
    float* pm = po + KS * a.H * LDO;              // [KS][H] running max (log2 domain)
    float* pl = pm + KS * a.H;                    // [KS][H] sum of exponentials
    __syncthreads();                              // the last tile's buffers are free
    {
      float* mo = po + (ks * a.H) * LDO;
#pragma unroll
      for (int i = 0; i < DT; ++i) {
        const int col = 8 * i + 2 * c;
        if (h0 < a.H) *reinterpret_cast<float2*>(mo + h0 * LDO + col) = make_float2(o[i][0], o[i][1]);
        if (h1 < a.H) *reinterpret_cast<float2*>(mo + h1 * LDO + col) = make_float2(o[i][2], o[i][3]);
      }
      if (c == 0) {
        if (h0 < a.H) {
          pm[ks * a.H + h0] = m0;
          pl[ks * a.H + h0] = l0;
        }
        if (h1 < a.H) {
          pm[ks * a.H + h1] = m1;
          pl[ks * a.H + h1] = l1;
        }
      }
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int NP = C * KS;                     // partials of the query
    const int hpc = (a.H + C - 1) / C;         // heads per CTA
    const int h_lo = rank * hpc;
    const int nh = max(0, min(a.H, h_lo + hpc) - h_lo);
    float* wm = pl + KS * a.H;                 // [nh][NP] max, then weight
    float* wl = wm + hpc * NP;                 // [nh][NP] sum
    for (int i = tid; i < nh * NP; i += kThreads) {
      const int hl = i / NP, pp = i % NP;
      const int r = pp / KS, s2 = pp % KS;
      wm[i] = *cluster.map_shared_rank(pm + s2 * a.H + h_lo + hl, r);
      wl[i] = *cluster.map_shared_rank(pl + s2 * a.H + h_lo + hl, r);
    }
    __syncthreads();
    if (tid < nh) {
      float* m_ = wm + tid * NP;
      const float* l_ = wl + tid * NP;
      float M = -INFINITY;
      for (int pp = 0; pp < NP; ++pp) M = fmaxf(M, m_[pp]);
      float den = 0.f;
      for (int pp = 0; pp < NP; ++pp) {
        const float f = M == -INFINITY ? 0.f : ex2(m_[pp] - M);
        m_[pp] = f;
        den = fmaf(f, l_[pp], den);
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      for (int pp = 0; pp < NP; ++pp) m_[pp] *= inv;
      if (a.lse) a.lse[qi * a.H + h_lo + tid] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    // the slice's outputs, four columns per item; eight partials in flight
    for (int it = tid; it < nh * (D / 4); it += kThreads) {
      const int hl = it / (D / 4), col = 4 * (it % (D / 4));
      const int h = h_lo + hl;
      const float* w_ = wm + hl * NP;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p0 = 0; p0 < NP; p0 += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int pp = p0 + u;
          if (pp < NP)
            v[u] = *reinterpret_cast<const float4*>(
                cluster.map_shared_rank(po + ((pp % KS) * a.H + h) * LDO + col, pp / KS));
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int pp = p0 + u;
          if (pp < NP) {
            const float f = w_[pp];
            acc.x = fmaf(f, v[u].x, acc.x);
            acc.y = fmaf(f, v[u].y, acc.y);
            acc.z = fmaf(f, v[u].z, acc.z);
            acc.w = fmaf(f, v[u].w, acc.w);
          }
        }
      }
      const long long o0 = (qi * a.H + h) * static_cast<long long>(D) + col;
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

  // ---- merge the KS key sub-ranges of each head group (shared memory)
  if constexpr (KS > 1) {
    float* xo = reinterpret_cast<float*>(smem);                   // [NW warps][16][D]
    float* xm = reinterpret_cast<float*>(smem + NW * 16 * D * 4);  // [NW warps][16]
    float* xl = xm + NW * 16;
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

// Decode-shaped calls (few queries per sequence) with head shapes other than
// the tensor-core kernel's (attend_tc.cu: H = 64, d = 128), and every call of
// csa_attend_noalloc: CTA = (key range, group of 16 heads, query).  The 8 warps own 16 keys each of every 128-key tile, so
// a CTA's tiles (at most a few) are gathered up front through a cp.async
// ring of up to three stages.  The warps' partials merge in shared memory
// (padded rows, no bank conflicts) into one (O, max, sum) per head, and the
// key ranges of one (query, head group) -- a thread-block cluster along x --
// fold their partials into the output through distributed shared memory:
// range r owns heads [r * hpc, (r + 1) * hpc) of the group and reads every
// range's partial of them, in range order.
template <int D>
__global__ void __launch_bounds__(256) attend_decode_kernel(AttendArgs a, int tpr) {
  pdl_wait_then_release();
  constexpr int kThreads = 256, kTile = 128, KW = 16, NWD = 8;
  constexpr int CH = D / 8, DT = D / 8;
  constexpr int TILE_BYTES = kTile * D * 2;
  constexpr int LDO = D + 4;  // padded partial rows
  extern __shared__ __align__(128) char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int gh = blockIdx.y;
  const long long qi = blockIdx.z;
  const int b = static_cast<int>(qi / a.Tq);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int nstage = tpr < 3 ? tpr : 3;
  char* Ks = smem;                                                     // [nstage][kTile][D]
  char* Vs = smem + nstage * TILE_BYTES;                               // [nstage][kTile][D]
  int* codes = reinterpret_cast<int*>(smem + 2 * nstage * TILE_BYTES);  // [tpr * kTile]

  const int t = a.q_pos[qi];
  int n_c;
  if (a.idx) {
    n_c = a.k;
  } else {
    n_c = t >= 0 ? (t + 1) / a.m : 0;
    n_c = n_c < a.N ? n_c : a.N;
  }
  const int n_tiles = (n_c + a.W + kTile - 1) / kTile;
  const int tile0 = rank * tpr;
  const int tile1 = min(n_tiles, tile0 + tpr);
  const int ntile = max(0, tile1 - tile0);

  // Q fragments of the group's heads (rows gh*16 + g and + 8; zero past H)
  uint32_t qf[D / 16][4];
  const int h0 = gh * 16 + g, h1 = h0 + 8;
  {
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
  // slot codes of the range
  {
    const int raw_base = a.W > 0 ? a.raw_base[b] : 0;
    bool bad = false;
    for (int i = tid; i < ntile * kTile; i += kThreads)
      codes[i] = slot_code(a, qi, b, t, n_c, raw_base, tile0 * kTile + i, &bad);
    if (bad) raise_flag(a.errw, kFlagIndex);
  }
  __syncthreads();
  const char* kc_base = static_cast<const char*>(a.k_cmp) + static_cast<size_t>(b) * a.N * D * 2;
  const char* vc_base = static_cast<const char*>(a.v_cmp) + static_cast<size_t>(b) * a.N * D * 2;
  const char* kr_base = static_cast<const char*>(a.k_raw) + static_cast<size_t>(b) * a.T_raw * D * 2;
  const char* vr_base = static_cast<const char*>(a.v_raw) + static_cast<size_t>(b) * a.T_raw * D * 2;
  auto load_tile = [&](int stage, int j) {
    const int* cs = codes + j * kTile;
#pragma unroll
    for (int rr = 0; rr < kTile * CH / kThreads; ++rr) {
      const int i = tid + rr * kThreads;
      const int r = i / CH, ch = i % CH;
      const int code = cs[r];
      const char* kp = code >= 0 ? kc_base + static_cast<size_t>(code) * D * 2
                                 : kr_base + static_cast<size_t>(code <= -2 ? -code - 2 : 0) * D * 2;
      const char* vp = code >= 0 ? vc_base + static_cast<size_t>(code) * D * 2
                                 : vr_base + static_cast<size_t>(code <= -2 ? -code - 2 : 0) * D * 2;
      const bool valid = code != -1;
      cp_async16(Ks + stage * TILE_BYTES + swz<D>(r, ch), valid ? kp + ch * 16 : kc_base, valid);
      cp_async16(Vs + stage * TILE_BYTES + swz<D>(r, ch), valid ? vp + ch * 16 : vc_base, valid);
    }
    cp_async_commit();
  };
  const int S = ntile < nstage ? ntile : nstage;
  for (int j = 0; j < S; ++j) load_tile(j, j);

  float o[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = a.scale * kLog2e;
  for (int j = 0; j < ntile; ++j) {
    // tiles committed so far: min(ntile, S + j); tile j may leave the later ones pending
    const int pending = min(ntile, S + j) - 1 - j;
    if (pending >= 2)
      cp_async_wait<2>();
    else if (pending == 1)
      cp_async_wait<1>();
    else
      cp_async_wait<0>();
    __syncthreads();
    const int stage = j % nstage;
    tile_step<D, KW>(qf, Ks + stage * TILE_BYTES, Vs + stage * TILE_BYTES, warp * KW, codes + j * kTile + warp * KW,
                     sl2, o, m0, m1, l0, l1);
    if (j + S < ntile) {
      __syncthreads();  // every warp is done with this stage
      load_tile(stage, j + S);
    }
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  // ---- the warps' partials -> one (O, max, sum) per head of the CTA
  float* xo = reinterpret_cast<float*>(smem);  // [NWD][16][LDO]
  float* xm = xo + NWD * 16 * LDO;              // [NWD][16]
  float* xl = xm + NWD * 16;                    // [NWD][16]
  float* po = xl + NWD * 16;                    // [16][LDO]  the CTA's partial, read by the cluster
  float* pm = po + 16 * LDO;                    // [16]
  float* pl = pm + 16;                          // [16]
  __syncthreads();                              // the tile buffers are free
  {
    float* mo = xo + warp * 16 * LDO;
#pragma unroll
    for (int i = 0; i < DT; ++i) {
      const int col = 8 * i + 2 * c;
      *reinterpret_cast<float2*>(mo + g * LDO + col) = make_float2(o[i][0], o[i][1]);
      *reinterpret_cast<float2*>(mo + (g + 8) * LDO + col) = make_float2(o[i][2], o[i][3]);
    }
    if (c == 0) {
      xm[warp * 16 + g] = m0;
      xm[warp * 16 + g + 8] = m1;
      xl[warp * 16 + g] = l0;
      xl[warp * 16 + g + 8] = l1;
    }
  }
  __syncthreads();
  {
    // thread -> (row hr, 8 columns)
    const int hr = tid >> 4, c0 = (tid & 15) * (D / 16);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWD; ++w) M = fmaxf(M, xm[w * 16 + hr]);
    const float R = M == -INFINITY ? 0.f : M;
    float f[NWD];
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
      f[w] = ex2(xm[w * 16 + hr] - R);
      L = fmaf(f[w], xl[w * 16 + hr], L);
    }
#pragma unroll
    for (int cc = 0; cc < D / 16; cc += 4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < NWD; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(xo + (w * 16 + hr) * LDO + c0 + cc);
        acc.x = fmaf(f[w], v.x, acc.x);
        acc.y = fmaf(f[w], v.y, acc.y);
        acc.z = fmaf(f[w], v.z, acc.z);
        acc.w = fmaf(f[w], v.w, acc.w);
      }
      *reinterpret_cast<float4*>(po + hr * LDO + c0 + cc) = acc;
    }
    if ((tid & 15) == 0) {
      pm[hr] = M;
      pl[hr] = L;
    }
  }
  cluster.sync();
  // ---- this range's heads of the group, from every range's partial
  const int hpc = (16 + C - 1) / C;
  const int r_lo = rank * hpc;
  const int nr = max(0, min(16, r_lo + hpc) - r_lo);
  for (int it = tid; it < nr * (D / 4); it += kThreads) {
    const int hr = r_lo + it / (D / 4), col = 4 * (it % (D / 4));
    const int h = gh * 16 + hr;
    float mr[kMaxCluster], lr[kMaxCluster];
    float4 v[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      if (r < C) {
        mr[r] = *cluster.map_shared_rank(pm + hr, r);
        lr[r] = *cluster.map_shared_rank(pl + hr, r);
        v[r] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(po + hr * LDO + col, r));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < C) M = fmaxf(M, mr[r]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        if (r < C) {
          const float f = ex2(mr[r] - M);
          den = fmaf(f, lr[r], den);
          acc.x = fmaf(f, v[r].x, acc.x);
          acc.y = fmaf(f, v[r].y, acc.y);
          acc.z = fmaf(f, v[r].z, acc.z);
          acc.w = fmaf(f, v[r].w, acc.w);
        }
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    if (h < a.H) {
      const long long o0 = (qi * a.H + h) * static_cast<long long>(D) + col;
      if (a.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o0) = acc;
      } else {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + o0) = pk;
      }
      if (a.lse && col == 0) a.lse[qi * a.H + h] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
    }
  }
  cluster.sync();  // peers may still read this CTA's partial until here
}

// Merge split partials of one (query, head) in split order.  The splits'
// log2-sum-exps are read in parallel (one split per thread), their weights
// are staged in shared memory a chunk of D splits at a time, and every thread
// folds its column over the chunk with independent loads.
template <int D>
__global__ void __launch_bounds__(D) attend_combine_kernel(AttendArgs a, int nsplit) {
  pdl_wait_then_release();
  __shared__ float wf[D];
  __shared__ float red[D / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long qh = blockIdx.x;  // qi * H + h
  const long long qi = qh / a.H;
  const int h = static_cast<int>(qh % a.H);
  const size_t stride = D + 1;
  const float* pb = a.part + static_cast<size_t>(qi) * nsplit * a.H * stride + h * stride;
  const size_t sstride = static_cast<size_t>(a.H) * stride;
  if (nsplit <= 32) {
    // every split's log2-sum-exp and value in flight at once, then the merge
    // in split order
    float ls[32], vs[32];
#pragma unroll
    for (int s = 0; s < 32; ++s) {
      ls[s] = s < nsplit ? pb[s * sstride + D] : -INFINITY;
      vs[s] = s < nsplit ? pb[s * sstride + tid] : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < 32; ++s) M = fmaxf(M, ls[s]);
    float acc = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int s = 0; s < 32; ++s) {
        if (s < nsplit) {
          const float f = ex2(ls[s] - M);
          den += f;
          acc = fmaf(f, vs[s], acc);
        }
      }
    }
    const float val = den > 0.f ? acc / den : 0.f;
    if (a.out_f32)
      static_cast<float*>(a.out)[qh * D + tid] = val;
    else
      static_cast<__nv_bfloat16*>(a.out)[qh * D + tid] = __float2bfloat16_rn(val);
    if (a.lse && tid == 0) a.lse[qh] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
    return;
  }
  float M = -INFINITY;
  for (int s = tid; s < nsplit; s += D) M = fmaxf(M, pb[s * sstride + D]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) M = fmaxf(M, red[w]);
  float acc = 0.f, den = 0.f;
  if (M != -INFINITY) {  // uniform over the block
    for (int c0 = 0; c0 < nsplit; c0 += D) {
      const int s = c0 + tid;
      wf[tid] = s < nsplit ? ex2(pb[s * sstride + D] - M) : 0.f;
      __syncthreads();
      const int n = nsplit - c0 < D ? nsplit - c0 : D;
      const float* col = pb + c0 * sstride + tid;
#pragma unroll 8
      for (int i = 0; i < n; ++i) {
        const float f = wf[i];
        den += f;
        acc = fmaf(f, col[i * sstride], acc);
      }
      __syncthreads();  // wf is rewritten by the next chunk
    }
  }
  const float val = den > 0.f ? acc / den : 0.f;
  if (a.out_f32)
    static_cast<float*>(a.out)[qh * D + tid] = val;
  else
    static_cast<__nv_bfloat16*>(a.out)[qh * D + tid] = __float2bfloat16_rn(val);
  if (a.lse && tid == 0) a.lse[qh] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
}

template <int D, int HG, int NW>
cudaError_t launch_impl(const AttendArgs& a, const AttendPlan& p, cudaStream_t s) {
  constexpr int kTile = 16 * NW;
  constexpr int TILE_BYTES = kTile * D * 2;
  constexpr int KS = NW / HG;
  const int nstage = p.tiles_per_split > 1 ? 2 : 1;
  size_t smem = 2 * nstage * TILE_BYTES + static_cast<size_t>(p.tiles_per_split) * kTile * sizeof(int);
  if (KS > 1) {
    const size_t need = NW * 16 * D * 4 + 2 * NW * 16 * 4;
    smem = smem > need ? smem : need;
  }
  if (p.mode == 2) {
    // every warp's partial (o on padded rows, m, l), then the (max, sum) of
    // this CTA's heads over all the query's partials
    const int np = p.nsplit * KS, hpc = (a.H + p.nsplit - 1) / p.nsplit;
    const size_t need = static_cast<size_t>(KS) * a.H * (D + 4 + 2) * 4 + 2 * static_cast<size_t>(hpc) * np * 4;
    smem = smem > need ? smem : need;
  }
  auto kern = attend_kernel<D, HG, NW>;
  cudaError_t e = ensure_dyn_smem<attend_kernel<D, HG, NW>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  const dim3 grid(p.nsplit, static_cast<unsigned>(nq));
  if (p.mode == 2 && p.nsplit > 8) {
    static std::atomic<bool> nonportable_set[64] = {};
    e = ensure_nonportable_cluster(kern, nonportable_set);
    if (e != cudaSuccess) return e;
  }
  e = launch_k(kern, grid, dim3(32 * NW), smem, s, p.mode == 2 ? p.nsplit : 1, a, p.nsplit, p.tiles_per_split,
               p.mode);
  if (e != cudaSuccess || p.mode != 1) return e;
  return launch_k(attend_combine_kernel<D>, dim3(static_cast<unsigned>(nq * a.H)), dim3(D), 0, s, 1, a,
                  p.nsplit);
}

template <int D>
cudaError_t launch_decode(const AttendArgs& a, const AttendPlan& p, cudaStream_t s) {
  constexpr int TILE_BYTES = 128 * D * 2;
  const int nstage = p.tiles_per_split < 3 ? p.tiles_per_split : 3;
  size_t smem = 2 * nstage * TILE_BYTES + static_cast<size_t>(p.tiles_per_split) * 128 * sizeof(int);
  const size_t merge = (8 * 16 * (D + 4) + 2 * 8 * 16 + 16 * (D + 4) + 2 * 16) * 4;
  smem = smem > merge ? smem : merge;
  auto kern = attend_decode_kernel<D>;
  cudaError_t e = ensure_dyn_smem<attend_decode_kernel<D>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (p.nsplit > 8) {
    static std::atomic<bool> nonportable_set[64] = {};
    e = ensure_nonportable_cluster(kern, nonportable_set);
    if (e != cudaSuccess) return e;
  }
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  const dim3 grid(p.nsplit, (a.H + 15) / 16, static_cast<unsigned>(nq));
  return launch_k(kern, grid, dim3(256), smem, s, p.nsplit, a, p.tiles_per_split);
}

template <int D, int NW>
cudaError_t launch_d(const AttendArgs& a, const AttendPlan& p, cudaStream_t s) {
  if (p.mode == 3) return launch_decode<D>(a, p, s);
  const int hg = (a.H + 15) / 16;
  if (hg <= 1) return launch_impl<D, 1, NW>(a, p, s);
  if (hg <= 2) return launch_impl<D, 2, NW>(a, p, s);
  return launch_impl<D, 4, NW>(a, p, s);
}

}  // namespace

AttendPlan plan_attend(int Tq, long long nq, int n_keys_max, int H, int d) {
  // The split depends only on the queries per sequence and the key count, never
  // on the batch size or the GPU, so a sequence gives bit-identical results
  // alone or inside any batch.  Prefill-like calls (many queries per sequence)
  // fill the GPU with 4-warp CTAs over 64-key tiles, without splitting (up to
  // 8192 keys per CTA); decode-like calls use 8-warp CTAs over 128-key tiles
  // and split every query's keys over up to kMaxCluster CTAs.  Up to
  // kMaxCluster splits of a query run as one thread-block cluster and merge
  // through distributed shared memory; more splits (over kMaxCluster * 8192
  // keys) keep their partials in the workspace and merge in a second kernel.
  AttendPlan p;
  p.nw = Tq >= 16 ? 4 : 8;
  const int tile = 16 * p.nw;
  if (Tq < 16) {
    // decode kernel: ranges of about three 128-key tiles, up to kMaxCluster
    // ranges (64 tiles each at most) per (query, head group)
    const int n_tiles = (n_keys_max + tile - 1) / tile;
    int nr = (n_tiles + 2) / 3;
    nr = nr < 1 ? 1 : (nr > kMaxCluster ? kMaxCluster : nr);
    int tpr = (n_tiles + nr - 1) / nr;
    tpr = tpr < 1 ? 1 : tpr;
    if (tpr <= kMaxKeysPerCta / tile && nq <= 65535) {
      p.tiles_per_split = tpr;
      p.nsplit = n_tiles > 0 ? (n_tiles + tpr - 1) / tpr : 1;
      p.mode = 3;
      p.part_bytes = 0;
      return p;
    }
  }
  const int max_tps = kMaxKeysPerCta / tile;
  const int n_tiles = (n_keys_max + tile - 1) / tile;
  int tps;
  if (Tq >= 16) {
    tps = n_tiles < max_tps ? n_tiles : max_tps;
  } else {
    tps = (n_tiles + kMaxCluster - 1) / kMaxCluster;
    tps = tps > max_tps ? max_tps : tps;
  }
  if (tps > n_tiles) tps = n_tiles;
  if (tps < 1) tps = 1;
  p.tiles_per_split = tps;
  p.nsplit = n_tiles > 0 ? (n_tiles + tps - 1) / tps : 1;
  p.mode = p.nsplit == 1 ? 0 : (p.nsplit <= kMaxCluster ? 2 : 1);
  p.part_bytes = p.mode == 1 ? static_cast<size_t>(nq) * p.nsplit * H * (d + 1) * sizeof(float) : 0;
  return p;
}

cudaError_t launch_attend_combine(const AttendArgs& a, int nsplit, cudaStream_t s) {
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (nq * a.H == 0) return cudaSuccess;
  if (a.d == 128)
    return launch_k(attend_combine_kernel<128>, dim3(static_cast<unsigned>(nq * a.H)), dim3(128), 0, s, 1, a,
                    nsplit);
  if (a.d == 64)
    return launch_k(attend_combine_kernel<64>, dim3(static_cast<unsigned>(nq * a.H)), dim3(64), 0, s, 1, a,
                    nsplit);
  return cudaErrorNotSupported;
}

cudaError_t launch_attend(const AttendArgs& a, const AttendPlan& p, cudaStream_t s) {
  if (static_cast<long long>(a.B) * a.Tq == 0) return cudaSuccess;
  if (a.d == 128) return p.nw == 8 ? launch_d<128, 8>(a, p, s) : launch_d<128, 4>(a, p, s);
  if (a.d == 64) return p.nw == 8 ? launch_d<64, 8>(a, p, s) : launch_d<64, 4>(a, p, s);
  return cudaErrorNotSupported;
}

}  // namespace csa
