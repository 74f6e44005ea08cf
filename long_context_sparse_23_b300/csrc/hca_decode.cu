// (5) Dense HCA attention for decode-shaped calls, on the tcgen05 tensor cores.
// octagono "Hybrid Attention: CSA and HCA": HCA compresses every m' = 128
// tokens into one entry and attends to all of them densely, together with a
// window over the most recent raw tokens.  For query (n, j) at position t and
// head h, with K/V shared by all heads:
//   keys J = {k_cmp[b] : b < n_c}  ++  {k_raw[u - raw_base] : t-W < u <= t, u >= 0},
//   n_c = min(N, floor((t+1)/m')),
//   out[h] = sum_{x in J} softmax_x(scale * q[h] . K_x) V_x    (one softmax over J)
//
// Design.  Both key segments are contiguous rows, so a 128-key tile arrives
// by one TMA box per 64-column half (128-byte swizzle; rows past the segment
// or the buffer are masked).  A CTA owns one query and a range of up to
// kHcaTiles tiles (compressed tiles first, then the window tiles):
//   1. S^T = K Q^T on tcgen05 (M = 128 keys on the TMEM lanes, N = H heads,
//      K = d): every tile's scores stay in TMEM, kHcaTiles * H columns.  As
//      soon as a tile's MMAs finish, its K buffer is refilled with V.
//   2. Eight epilogue warps (four TMEM lane quarters x two halves of the
//      heads) take the exact per-head maximum over all of the CTA's keys
//      (warp butterfly reduce-scatter, then the four quarters in shared
//      memory), so the probabilities need no later rescaling; they write
//      P^T = 2^(s - max) as bf16 rows [key][head] (128-byte swizzle) and
//      sum them per head in fp32.
//   3. O^T = V^T P^T on tcgen05 (M = d = 128 lanes, N = H columns, K = keys),
//      both operands MN-major straight from the V tile and the P rows,
//      accumulated in TMEM over the tiles.
//   4. The epilogue divides by the sum and writes the output (one range) or
//      the range's partial (normalised O and log2-sum-exp) for the combine
//      kernel, which merges a query's ranges in range order.
// Every wait is bounded; a timeout raises the workspace error flag, and a
// window key outside the raw buffer raises the index flag and is skipped.
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kD = 128;            // head width handled here
constexpr int kHT = 128;           // keys per tile
constexpr int kHalfB = kHT * 128;  // one 64-column half of a tile: 128 rows x 128 bytes
constexpr int kThreads = 320;      // TMA producer, MMA issuer, 8 epilogue warps
constexpr long long kDrainBudget = 1LL << 31;

struct HParams {
  const int32_t* q_pos;
  const int32_t* raw_base;
  int Tq, N, T_raw, W, m;
  float sl2;  // scale * log2(e)
  int nsplit;
  void* out;
  int out_f32;
  float* lse;
  float* part;  // [nq][nsplit][H][D + 1], nsplit > 1
  uint32_t* errw;
  long long budget;
};

struct __align__(8) HBars {
  uint64_t q;
  uint64_t kfull[kHcaTiles];
  uint64_t sdone[kHcaTiles];
  uint64_t vfull[kHcaTiles];
  uint64_t pfull[kHcaTiles];
  uint64_t ofull;
};

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle
// layout: 64 consecutive M/N elements form one 128-byte row, 8 rows along K
// form a 1024-byte atom.  lbo = byte distance between 64-element M/N blocks,
// sbo = byte distance between 8-row K groups.  Other fields as for the
// K-major descriptor (version 1, base offset 0, layout type 2).
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Butterfly reduce-scatter over a warp: on return, v[0] of lane l holds the
// max (kMax) or the sum over all 32 lanes of the inputs' element l.  Fixed
// order, so sums are reproducible.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? v[i] : v[i + s];
      const float keep = up ? v[i + s] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, s);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// The query's key tiles: n_ct compressed tiles (rows 128 j ...), then the
// window tiles (window slots w = 128 (j - n_ct) + i, token u = t - W + 1 + w).
struct QTiles {
  int t, n_c, n_ct, n_tiles, raw_base;
};

__device__ __forceinline__ QTiles query_tiles(const HParams& p, long long qi, int b) {
  QTiles q;
  q.t = p.q_pos[qi];
  int nc = q.t >= 0 ? (q.t + 1) / p.m : 0;
  q.n_c = nc < p.N ? nc : p.N;
  q.n_ct = (q.n_c + kHT - 1) / kHT;
  q.n_tiles = q.n_ct + (p.W + kHT - 1) / kHT;
  q.raw_base = p.W > 0 ? p.raw_base[b] : 0;
  return q;
}

// Is key i of tile j attended?  *bad: a window key inside [0, t] whose row is
// outside the raw buffer (reported, then skipped).
__device__ __forceinline__ bool key_ok(const HParams& p, const QTiles& q, int j, int i, bool* bad) {
  if (j < q.n_ct) return j * kHT + i < q.n_c;
  const int w = (j - q.n_ct) * kHT + i;
  const long long u = static_cast<long long>(q.t) - p.W + 1 + w;
  if (w >= p.W || u < 0) return false;
  const long long r = u - q.raw_base;
  if (r < 0 || r >= p.T_raw) {
    *bad = true;
    return false;
  }
  return true;
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
    hca_decode_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tkc,
                      const __grid_constant__ CUtensorMap tvc, const __grid_constant__ CUtensorMap tkr,
                      const __grid_constant__ CUtensorMap tvr, HParams p) {
  static_assert(H == 64, "P^T rows are one 128-byte swizzle row of 64 heads");
  constexpr int HPG = H / 2;               // heads per epilogue warp
  constexpr int kQBytes = 2 * H * 128;     // two 64-column halves of the query rows
  constexpr int kTileB = 2 * kHalfB;       // K (then V) tile
  constexpr int kPB = kHT * 128;           // P^T rows of one tile
  constexpr uint32_t kTmemCols = 512;      // per tile: H score columns and H output columns
  constexpr uint32_t kOCol = kHcaTiles * H;
  static_assert(2 * kHcaTiles * H <= static_cast<int>(kTmemCols), "TMEM columns");
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  char* qs = smem;                             // [2][H][128 B]
  char* kv = qs + kQBytes;                     // [kHcaTiles][2][128][128 B]
  char* ps = kv + kHcaTiles * kTileB;          // [kHcaTiles][128][128 B]
  HBars* bars = reinterpret_cast<HBars*>(ps + kHcaTiles * kPB);
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  // per tile: the four lane quarters' per-head max of the raw scores and sum
  // of the probabilities, then per head the tile's exponent offset; at the
  // end per head the tiles' output coefficients
  __shared__ float m_part[kHcaTiles][4][H], l_part[kHcaTiles][4][H];
  __shared__ __align__(16) float r_s[kHcaTiles][H];  // per tile and head: the exponent offset
  __shared__ __align__(16) float coef[kHcaTiles][H];
  __shared__ float lse_s[H];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const long long qi = blockIdx.y;

  // ---- set-up that reads no input: it overlaps the previous kernel's tail
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bars->q, 1);
    for (int j = 0; j < kHcaTiles; ++j) {
      mbar_init(&bars->kfull[j], 1);
      mbar_init(&bars->sdone[j], 1);
      mbar_init(&bars->vfull[j], 1);
      mbar_init(&bars->pfull[j], 8);
    }
    mbar_init(&bars->ofull, 1);
    mbar_fence_init();
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tkc);
    tma_prefetch_desc(&tvc);
    tma_prefetch_desc(&tkr);
    tma_prefetch_desc(&tvr);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait_then_release();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  volatile int* abort_v = &abort_flag;

  const int b = static_cast<int>(qi / p.Tq);
  const QTiles qt = query_tiles(p, qi, b);
  const int j0 = split * kHcaTiles;
  int ntile = qt.n_tiles - j0;
  ntile = ntile < 0 ? 0 : (ntile > kHcaTiles ? kHcaTiles : ntile);

  if (ntile == 0) {
    // nothing of this query in this range: an empty partial, or (one range)
    // the output of an empty key set, 0 and lse = -inf
    for (int i = tid; i < H * kD; i += kThreads) {
      const int h = i / kD, c = i % kD;
      if (p.nsplit > 1) {
        float* pb = p.part + ((qi * p.nsplit + split) * H + h) * static_cast<long long>(kD + 1);
        pb[c] = 0.f;
        if (c == 0) pb[kD] = -INFINITY;
      } else {
        const long long o = (qi * H + h) * static_cast<long long>(kD) + c;
        if (p.out_f32)
          static_cast<float*>(p.out)[o] = 0.f;
        else
          static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
        if (p.lse && c == 0) p.lse[qi * H + h] = -INFINITY;
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // TMA coordinates of tile jj of this range (x = 64-column half)
      auto tile_src = [&](int jj, const CUtensorMap** kmap, const CUtensorMap** vmap, int* row) {
        const int j = j0 + jj;
        if (j < qt.n_ct) {
          *kmap = &tkc;
          *vmap = &tvc;
          *row = j * kHT;
        } else {
          *kmap = &tkr;
          *vmap = &tvr;
          long long r = static_cast<long long>(qt.t) - p.W + 1 + static_cast<long long>(j - qt.n_ct) * kHT -
                        qt.raw_base;
          r = r < -kHT ? -kHT : (r > p.T_raw ? p.T_raw : r);  // wholly outside: rows of fill, all masked
          *row = static_cast<int>(r);
        }
      };
      mbar_expect_tx(&bars->q, kQBytes);
      tma_load_2d(qs, &tmq, &bars->q, 0, static_cast<int>(qi * H));
      tma_load_2d(qs + H * 128, &tmq, &bars->q, 64, static_cast<int>(qi * H));
      for (int jj = 0; jj < ntile; ++jj) {
        const CUtensorMap *km, *vm;
        int row;
        tile_src(jj, &km, &vm, &row);
        mbar_expect_tx(&bars->kfull[jj], kTileB);
        tma_load_3d(kv + jj * kTileB, km, &bars->kfull[jj], 0, row, b);
        tma_load_3d(kv + jj * kTileB + kHalfB, km, &bars->kfull[jj], 64, row, b);
      }
      // a tile's buffer takes its V rows once the tile's score MMAs are done
      int v_issued = 0;
      for (int jj = 0; jj < ntile; ++jj) {
        if (!mbar_wait_sleep(&bars->sdone[jj], 0, p.budget, abort_v)) {
          if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
          *abort_v = 1;
          break;
        }
        const CUtensorMap *km, *vm;
        int row;
        tile_src(jj, &km, &vm, &row);
        mbar_expect_tx(&bars->vfull[jj], kTileB);
        tma_load_3d(kv + jj * kTileB, vm, &bars->vfull[jj], 0, row, b);
        tma_load_3d(kv + jj * kTileB + kHalfB, vm, &bars->vfull[jj], 64, row, b);
        v_issued = jj + 1;
      }
      // drain: every issued copy has landed before the CTA may exit
      mbar_wait_sleep(&bars->q, 0, kDrainBudget, nullptr);
      for (int jj = 0; jj < ntile; ++jj) mbar_wait_sleep(&bars->kfull[jj], 0, kDrainBudget, nullptr);
      for (int jj = 0; jj < v_issued; ++jj) mbar_wait_sleep(&bars->vfull[jj], 0, kDrainBudget, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, H);
      const uint32_t idesc_o = idesc_bf16_f32(128, H) | (1u << 15) | (1u << 16);  // A, B MN-major
      bool any = false, ok = mbar_wait_sleep(&bars->q, 0, p.budget, abort_v);
      for (int jj = 0; ok && jj < ntile; ++jj) {
        if (!mbar_wait_sleep(&bars->kfull[jj], 0, p.budget, abort_v)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(kv + jj * kTileB), b0 = smem_u32(qs);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int h = kk >> 2, w = kk & 3;
          umma_f16(tbase + static_cast<uint32_t>(jj * H), sdesc_kmajor_sw128(a0 + h * kHalfB + w * 32),
                   sdesc_kmajor_sw128(b0 + h * H * 128 + w * 32), idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->sdone[jj]);
        any = true;
      }
      for (int jj = 0; ok && jj < ntile; ++jj) {
        if (!mbar_wait_sleep(&bars->pfull[jj], 0, p.budget, abort_v) ||
            !mbar_wait_sleep(&bars->vfull[jj], 0, p.budget, abort_v)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(kv + jj * kTileB), b0 = smem_u32(ps + jj * kPB);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // 16 keys = two 8-row groups of the V tile (A = V^T, d on M) and of
          // the P^T rows (B = P^T, heads on N); tile jj accumulates alone
          umma_f16(tbase + kOCol + static_cast<uint32_t>(jj * H), sdesc_mnmajor_sw128(a0 + kk * 2048, kHalfB, 1024),
                   sdesc_mnmajor_sw128(b0 + kk * 2048, 1024, 1024), idesc_o, kk > 0 ? 1u : 0u);
        }
      }
      if (!ok) {
        if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
        *abort_v = 1;
      }
      // one commit for everything issued: the epilogue reads O after it, and
      // the CTA does not exit before the MMAs are done
      if (any) {
        umma_commit(&bars->ofull);
        mbar_wait_sleep(&bars->ofull, 0, kDrainBudget, nullptr);
      }
    }
  } else {
    // ---- epilogue: warp -> (TMEM lane quarter, half of the heads)
    const int quarter = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int etid = tid - 64;          // 0 .. 255
    const int i = quarter * 32 + lane;  // key row of every tile; d index of O
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true, bad = false;

    // per tile, as soon as its scores are in TMEM: the tile's per-head max,
    // P^T = 2^(s * sl2 - R) as bf16 rows, per-head sums in fp32
    for (int jj = 0; jj < ntile; ++jj) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bars->sdone[jj], 0, p.budget, abort_v));
      uint32_t r[2][16];
      const bool in = key_ok(p, qt, j0 + jj, i, &bad);
      float v[32];
      if (ok) {
        tc_fence_after();
        tmem_ld16(lane_addr + jj * H + grp * HPG, r[0]);
        tmem_ld16(lane_addr + jj * H + grp * HPG + 16, r[1]);
        tmem_ld_wait();
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = (ok && in) ? __uint_as_float(r[e >> 4][e & 15]) : -INFINITY;
      m_part[jj][quarter][grp * HPG + lane] = warp_reduce_scatter32<true>(v, lane);
      epi_bar();
      // one thread per head: the tile's exponent offset (log2 domain; no key -> 0)
      if (etid < H) {
        const float M = fmaxf(fmaxf(m_part[jj][0][etid], m_part[jj][1][etid]),
                              fmaxf(m_part[jj][2][etid], m_part[jj][3][etid]));
        r_s[jj][etid] = M == -INFINITY ? 0.f : M * p.sl2;
      }
      epi_bar();
      if (ok) {
        float R[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 q4 = *reinterpret_cast<const float4*>(&r_s[jj][grp * HPG + 4 * c4]);
          R[4 * c4] = q4.x;
          R[4 * c4 + 1] = q4.y;
          R[4 * c4 + 2] = q4.z;
          R[4 * c4 + 3] = q4.w;
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = in ? ex2(fmaf(__uint_as_float(r[e >> 4][e & 15]), p.sl2, -R[e])) : 0.f;
          const float p1 = in ? ex2(fmaf(__uint_as_float(r[e >> 4][(e & 15) + 1]), p.sl2, -R[e + 1])) : 0.f;
          pk[e / 2] = pack_bf16x2(p0, p1);
          v[e] = p0;
          v[e + 1] = p1;
        }
        char* row = ps + jj * kPB + i * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int ch = grp * 4 + cc;
          *reinterpret_cast<uint4*>(row + ((ch ^ (i & 7)) << 4)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        fence_proxy_async();  // the rows are read by the tensor cores
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->pfull[jj]);
      l_part[jj][quarter][grp * HPG + lane] = warp_reduce_scatter32<false>(v, lane);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(p.errw, kFlagIndex);
    epi_bar();
    // per head: the tiles' weights 2^(R_j - R) / L with R = max_j R_j and
    // L = sum_j 2^(R_j - R) L_j, and the log2-sum-exp R + log2 L
    if (etid < H) {
      const int h = etid;
      float Rj[kHcaTiles], Lj[kHcaTiles];
      float R = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kHcaTiles; ++jj) {
        const float M = jj < ntile ? fmaxf(fmaxf(m_part[jj][0][h], m_part[jj][1][h]),
                                           fmaxf(m_part[jj][2][h], m_part[jj][3][h]))
                                   : -INFINITY;
        Rj[jj] = M == -INFINITY ? -INFINITY : r_s[jj][h];
        Lj[jj] = jj < ntile ? (l_part[jj][0][h] + l_part[jj][1][h]) + (l_part[jj][2][h] + l_part[jj][3][h]) : 0.f;
        R = fmaxf(R, Rj[jj]);
      }
      float L = 0.f, w[kHcaTiles];
#pragma unroll
      for (int jj = 0; jj < kHcaTiles; ++jj) {
        w[jj] = Rj[jj] == -INFINITY ? 0.f : ex2(Rj[jj] - R);
        L = fmaf(w[jj], Lj[jj], L);
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int jj = 0; jj < kHcaTiles; ++jj) coef[jj][h] = w[jj] * inv;
      lse_s[h] = L > 0.f ? R + __log2f(L) : -INFINITY;
    }
    epi_bar();

    // O^T from TMEM: lane i = column d of the output, 32 heads per thread,
    // the tiles' accumulators weighted by coef
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bars->ofull, 0, p.budget, abort_v));
    if (ok) {
      float o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0.f;
      tc_fence_after();
      for (int jj = 0; jj < ntile; ++jj) {
        uint32_t r[2][16];
        tmem_ld16(lane_addr + kOCol + jj * H + grp * HPG, r[0]);
        tmem_ld16(lane_addr + kOCol + jj * H + grp * HPG + 16, r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 w4 = *reinterpret_cast<const float4*>(&coef[jj][grp * HPG + 4 * c4]);
          o[4 * c4] = fmaf(w4.x, __uint_as_float(r[c4 >> 2][(4 * c4) & 15]), o[4 * c4]);
          o[4 * c4 + 1] = fmaf(w4.y, __uint_as_float(r[c4 >> 2][(4 * c4 + 1) & 15]), o[4 * c4 + 1]);
          o[4 * c4 + 2] = fmaf(w4.z, __uint_as_float(r[c4 >> 2][(4 * c4 + 2) & 15]), o[4 * c4 + 2]);
          o[4 * c4 + 3] = fmaf(w4.w, __uint_as_float(r[c4 >> 2][(4 * c4 + 3) & 15]), o[4 * c4 + 3]);
        }
      }
      if (p.nsplit > 1) {
        float* pb = p.part + ((qi * p.nsplit + split) * H + grp * HPG) * static_cast<long long>(kD + 1) + i;
#pragma unroll
        for (int e = 0; e < 32; ++e) pb[e * (kD + 1)] = o[e];
        if (quarter == 0)
          p.part[((qi * p.nsplit + split) * H + grp * HPG + lane) * static_cast<long long>(kD + 1) + kD] =
              lse_s[grp * HPG + lane];
      } else {
        const long long ob = (qi * H + grp * HPG) * static_cast<long long>(kD) + i;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          if (p.out_f32)
            static_cast<float*>(p.out)[ob + e * kD] = o[e];
          else
            static_cast<__nv_bfloat16*>(p.out)[ob + e * kD] = __float2bfloat16_rn(o[e]);
        }
        if (quarter == 0 && p.lse) {
          const float l2 = lse_s[grp * HPG + lane];
          p.lse[qi * H + grp * HPG + lane] = l2 == -INFINITY ? -INFINITY : l2 * 0.6931471805599453f;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

int hca_decode_nsplit(int N, int W) {
  const long long tiles = (static_cast<long long>(N) + kHT - 1) / kHT + (static_cast<long long>(W) + kHT - 1) / kHT;
  const long long ns = (tiles + kHcaTiles - 1) / kHcaTiles;
  return static_cast<int>(ns < 1 ? 1 : ns);
}

bool hca_decode_supported(int Tq, long long nq, int N, int T_raw, int H, int d, int W) {
  // decode-shaped calls (the prefill shape keeps the mma.sync kernel, which
  // shares key tiles between the queries of a sequence)
  if (Tq >= 16 || nq <= 0 || nq > 65535) return false;
  if (H != 64 || d != kD || N <= 0) return false;
  if (W > 0 && T_raw <= 0) return false;
  return hca_decode_nsplit(N, W) <= 65535;
}

size_t hca_decode_part_bytes(long long nq, int N, int W, int H, int d) {
  const int ns = hca_decode_nsplit(N, W);
  return ns > 1 ? static_cast<size_t>(nq) * ns * H * (d + 1) * sizeof(float) : 0;
}

cudaError_t launch_hca_decode(const AttendArgs& a, long long budget, cudaStream_t s) {
  constexpr int H = 64;
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (nq == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmq, tkc, tvc, tkr, tvr;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(nq) * H};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(H)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto rows_map = [&](CUtensorMap* m, const void* base, int rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(a.B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(rows) * kD * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kHT), 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  if (!rows_map(&tkc, a.k_cmp, a.N) || !rows_map(&tvc, a.v_cmp, a.N)) return cudaErrorInvalidValue;
  if (a.W > 0) {
    if (!rows_map(&tkr, a.k_raw, a.T_raw) || !rows_map(&tvr, a.v_raw, a.T_raw)) return cudaErrorInvalidValue;
  } else {
    tkr = tkc;  // never read: no window tiles
    tvr = tvc;
  }
  HParams p;
  p.q_pos = a.q_pos;
  p.raw_base = a.raw_base;
  p.Tq = a.Tq;
  p.N = a.N;
  p.T_raw = a.T_raw;
  p.W = a.W;
  p.m = a.m;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.nsplit = hca_decode_nsplit(a.N, a.W);
  p.out = a.out;
  p.out_f32 = a.out_f32;
  p.lse = a.lse;
  p.part = a.part;
  p.errw = a.errw;
  p.budget = budget;
  const size_t smem = 1024 + 2 * H * 128 + kHcaTiles * (2 * kHalfB + kHT * 128) + sizeof(HBars);
  cudaError_t e = ensure_dyn_smem<hca_decode_kernel<H>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = launch_k(hca_decode_kernel<H>, dim3(static_cast<unsigned>(p.nsplit), static_cast<unsigned>(nq)),
               dim3(kThreads), smem, s, 1, tmq, tkc, tvc, tkr, tvr, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  return launch_attend_combine(a, p.nsplit, s);
}

}  // namespace csa
