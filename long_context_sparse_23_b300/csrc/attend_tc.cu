// (4)/(5) Decode attention on the tcgen05 tensor cores: the selected
// compressed entries plus the raw window (CSA), or every visible entry plus
// the window (dense HCA).
// "DeepSeek V4 technical review", section 2.1: attention runs only over the
// selected compressed blocks; octagono "Hybrid Attention: CSA and HCA": a
// window over the most recent raw tokens gives local context, and HCA attends
// to every entry compressed at m' = 128.  For query (n, j) at position t and
// head h, with K/V shared by all heads:
//   CSA  keys J = {k_cmp[idx[s]] : s < k, idx[s] >= 0} ++ window,
//   HCA  keys J = {k_cmp[b] : b < n_c}, n_c = min(N, floor((t+1)/m')) ++ window,
//   window = {k_raw[u - raw_base] : t-W < u <= t, u >= 0},
//   out[h] = sum_{x in J} softmax_x(scale * q[h] . K_x) V_x    (one softmax over J)
//
// Design.  A CTA owns one query and a range of up to kTcTiles (CSA; HCA:
// kTcTilesHca) tiles of 128 key slots, all 64 heads at once (the K/V rows are
// read once per range):
//   * keys: HCA tiles are contiguous rows, one TMA box per 64-column half
//     (128-byte swizzle); CSA tiles are gathered row by row with 16-byte
//     cp.async into the same swizzled layout by three producer warps, which
//     wait for their own copies and fence them for the tensor cores before
//     signalling (holes and rows outside their buffers are zero-filled and
//     masked);
//   1. S^T = K Q^T on tcgen05 (M = 128 keys on the TMEM lanes, N = 64 heads,
//      K = d): every tile's scores stay in TMEM.  Once a tile's MMAs finish,
//      its K buffer is refilled with V;
//   2. eight epilogue warps (four TMEM lane quarters x two halves of the
//      heads) take each tile's exact per-head max (warp butterfly
//      reduce-scatter, then the four quarters in shared memory) as soon as the
//      tile's scores are ready, write P^T = 2^(s - max) as bf16 rows
//      [key][head] (128-byte swizzle; two P buffers in turn, a buffer
//      rewritten once the MMAs that read it are done) and sum them per head
//      in fp32;
//   3. O_j^T = V^T P^T on tcgen05 per tile (M = d = 128 lanes, N = 64 heads,
//      K = keys), both operands MN-major straight from the V tile and the P
//      rows, each tile into its own TMEM accumulator: the columns of the
//      tile's scores, free once its P rows are written;
//   4. the epilogue weights the tiles by 2^(max_j - max) / L and writes the
//      output (one range) or the range's partial (normalised O and
//      log2-sum-exp).  Up to eight ranges of a query form a thread-block
//      cluster: each CTA keeps its partial in shared memory and, after a
//      cluster barrier, merges a share of the query's (head, column) outputs
//      from every range's partial over distributed shared memory, in range
//      order.  More ranges write their partials to the workspace for the
//      combine kernel, which merges them the same way.
// Every wait is bounded (and sleeps in hardware rather than polling); a
// timeout raises the workspace error flag, an index or window row outside its
// buffer raises the index flag and is skipped.
#include <cooperative_groups.h>

#include "attend_tile.cuh"
#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kH = 64;             // heads handled here
constexpr int kD = 128;            // head width handled here
constexpr int kHT = 128;           // key slots per tile
constexpr int kHalfB = kHT * 128;  // one 64-column half of a tile: 128 rows x 128 bytes
constexpr int kThreads = 384;      // MMA warp, three producer warps, eight epilogue warps
constexpr int kProducers = 96;
constexpr long long kDrainBudget = 1LL << 31;
constexpr int kPSlots = 2;         // P^T buffers, used by tiles in turn
constexpr int kTcClusterMax = 8;   // ranges of a query merged inside one cluster (portable size)
// cluster merge buffers in the K/V region (free once every MMA is done):
// the range's partial [H][kD] + [H] at 0, the shares received after it
constexpr int kRecvOff = 34 * 1024;
constexpr int kRecvBytes = 33 * 1024;  // >= ns * ceil(H * kD / 4 / ns) * 16 for 2 <= ns <= 8
static_assert(kRecvOff >= (kH * kD + kH) * 4, "partial before the receive buffers");
static_assert(kRecvOff + kRecvBytes + kTcClusterMax * kH * 4 <= kTcTiles * 2 * kHalfB,
              "merge buffers inside the K/V region");

// One bulk copy from this CTA's shared memory into CTA ``rank`` of the
// cluster, to the same offset as ``dst``, completing on that CTA's mbarrier
// at the offset of ``bar``.
__device__ __forceinline__ void bulk_to_rank(void* dst, const void* src, uint32_t bytes, uint64_t* bar, int rank) {
  uint32_t d, mb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(smem_u32(dst)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(mb) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
               "r"(smem_u32(src)), "r"(bytes), "r"(mb)
               : "memory");
}

struct TcParams {
  float sl2;  // scale * log2(e)
  int nsplit;
  int tpr;    // tiles per range
  int cluster;  // 1: the nsplit ranges of a query form a cluster and merge through DSMEM
  long long budget;
};

struct __align__(8) TcBars {
  uint64_t q;
  uint64_t kfull[kTcTiles];
  uint64_t sdone[kTcTiles];
  uint64_t vfull[kTcTiles];
  uint64_t pfull[kTcTiles];
  uint64_t pempty[2];  // P buffer read by the MMAs of its last tile
  uint64_t ofull;
  uint64_t mrecv;      // cluster merge: every range's share of the partial has landed
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
__device__ __forceinline__ void prod_bar() { asm volatile("bar.sync 2, 96;" ::: "memory"); }

// wait until at most n of this thread's cp.async groups are pending (n <= 3)
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  switch (n) {
    case 3: cp_async_wait<3>(); break;
    case 2: cp_async_wait<2>(); break;
    case 1: cp_async_wait<1>(); break;
    default: cp_async_wait<0>(); break;
  }
}

// A query's key tiles.  HCA: n_ct tiles of compressed rows 128 j ..., then the
// window tiles (window slot w = 128 (j - n_ct) + i).  CSA: the slots 0 .. k-1
// of the index list, then the W window slots, cut into tiles of 128.
struct QTiles {
  int t, n_c, n_ct, n_tiles, raw_base;
};

__device__ __forceinline__ QTiles query_tiles(const AttendArgs& a, long long qi, int b) {
  QTiles q;
  q.t = a.q_pos[qi];
  q.raw_base = a.W > 0 ? a.raw_base[b] : 0;
  if (a.idx) {
    q.n_c = a.k;
    q.n_ct = 0;
    q.n_tiles = (a.k + a.W + kHT - 1) / kHT;
  } else {
    const int nc = q.t >= 0 ? (q.t + 1) / a.m : 0;
    q.n_c = nc < a.N ? nc : a.N;
    q.n_ct = (q.n_c + kHT - 1) / kHT;
    q.n_tiles = q.n_ct + (a.W + kHT - 1) / kHT;
  }
  return q;
}

// HCA: is key i of tile j attended?  *bad: a window key inside [0, t] whose
// row is outside the raw buffer (reported, then skipped).
__device__ __forceinline__ bool hca_key_ok(const AttendArgs& a, const QTiles& q, int j, int i, bool* bad) {
  if (j < q.n_ct) return j * kHT + i < q.n_c;
  const int w = (j - q.n_ct) * kHT + i;
  const long long u = static_cast<long long>(q.t) - a.W + 1 + w;
  if (w >= a.W || u < 0) return false;
  const long long r = u - q.raw_base;
  if (r < 0 || r >= a.T_raw) {
    *bad = true;
    return false;
  }
  return true;
}

template <bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tkc,
                     const __grid_constant__ CUtensorMap tvc, const __grid_constant__ CUtensorMap tkr,
                     const __grid_constant__ CUtensorMap tvr, AttendArgs a, TcParams p) {
  constexpr int H = kH;
  constexpr int HPG = H / 2;               // heads per epilogue warp
  constexpr int kQBytes = 2 * H * 128;     // two 64-column halves of the query rows
  constexpr int kTileB = 2 * kHalfB;       // K (then V) tile
  constexpr int kPB = kHT * 128;           // P^T rows of one tile
  constexpr uint32_t kTmemCols = 512;      // per tile: H score columns, then the tile's H output columns
  static_assert(kTcTiles * H <= static_cast<int>(kTmemCols), "TMEM columns");
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  char* qs = smem;                             // [2][H][128 B]
  char* kv = qs + kQBytes;                     // [kTcTiles][2][128][128 B]
  char* ps = kv + kTcTiles * kTileB;           // [kPSlots][128][128 B]
  TcBars* bars = reinterpret_cast<TcBars*>(ps + kPSlots * kPB);
  // P^T rows of tile jj: a buffer per tile for ranges of up to four tiles
  // (ps, then the unused fifth K/V buffer); two buffers in turn for five
  const bool pring = p.tpr > kTcTilesHca;
  auto pbuf = [&](int jj) -> char* {
    if (pring) return ps + (jj % kPSlots) * kPB;
    return jj < kPSlots ? ps + jj * kPB : kv + (kTcTiles - 1) * kTileB + (jj - kPSlots) * kPB;
  };
  static_assert(kTcTilesHca - kPSlots <= kTileB / kPB, "P buffers of four tiles");
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  // per tile: the four lane quarters' per-head max of the raw scores and sum
  // of the probabilities, then per head the tile's exponent offset; at the
  // end per head the tiles' output coefficients
  __shared__ float m_part[kTcTiles][4][H], l_part[kTcTiles][4][H];
  __shared__ __align__(16) float r_s[kTcTiles][H];
  __shared__ __align__(16) float coef[kTcTiles][H];
  __shared__ float lse_s[H];
  __shared__ int codes_s[kGather ? kTcTiles : 1][kHT];  // gathered rows' codes (see slot_code)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const long long qi = blockIdx.y;

  // ---- set-up that reads no input: it overlaps the previous kernel's tail
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bars->q, 1);
    for (int j = 0; j < kTcTiles; ++j) {
      mbar_init(&bars->kfull[j], 1);
      mbar_init(&bars->sdone[j], 1);
      mbar_init(&bars->vfull[j], 1);
      mbar_init(&bars->pfull[j], 8);
    }
    for (int j = 0; j < kPSlots; ++j) mbar_init(&bars->pempty[j], 1);
    mbar_init(&bars->ofull, 1);
    mbar_init(&bars->mrecv, 1);
    mbar_fence_init();
    tma_prefetch_desc(&tmq);
    if (!kGather) {
      tma_prefetch_desc(&tkc);
      tma_prefetch_desc(&tvc);
      tma_prefetch_desc(&tkr);
      tma_prefetch_desc(&tvr);
    }
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait_then_release();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  volatile int* abort_v = &abort_flag;

  const int b = static_cast<int>(qi / a.Tq);
  const QTiles qt = query_tiles(a, qi, b);
  const int j0 = split * p.tpr;
  int ntile = qt.n_tiles - j0;
  ntile = ntile < 0 ? 0 : (ntile > p.tpr ? p.tpr : ntile);

  // the range's partial in shared memory when the ranges merge in the cluster:
  // [H][kD] normalised O, then [H] log2-sum-exp (the K/V buffers, free once
  // every MMA is done)
  float* part_s = reinterpret_cast<float*>(kv);
  if (ntile == 0) {
    // nothing of this query in this range: an empty partial, or (one range)
    // the output of an empty key set, 0 and lse = -inf
    for (int i = tid; i < H * kD; i += kThreads) {
      const int h = i / kD, c = i % kD;
      if (p.cluster) {
        part_s[i] = 0.f;
        if (c == 0) part_s[H * kD + h] = -INFINITY;
      } else if (p.nsplit > 1) {
        float* pb = a.part + ((qi * p.nsplit + split) * H + h) * static_cast<long long>(kD + 1);
        pb[c] = 0.f;
        if (c == 0) pb[kD] = -INFINITY;
      } else {
        const long long o = (qi * H + h) * static_cast<long long>(kD) + c;
        if (a.out_f32)
          static_cast<float*>(a.out)[o] = 0.f;
        else
          static_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(0.f);
        if (a.lse && c == 0) a.lse[qi * H + h] = -INFINITY;
      }
    }
  } else if (warp == 0) {
    // ---- MMA issuer
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
        const uint32_t a0 = smem_u32(kv + jj * kTileB), b0 = smem_u32(pbuf(jj));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // 16 keys = two 8-row groups of the V tile (A = V^T, d on M) and of
          // the P^T rows (B = P^T, heads on N); tile jj accumulates alone
          umma_f16(tbase + static_cast<uint32_t>(jj * H), sdesc_mnmajor_sw128(a0 + kk * 2048, kHalfB, 1024),
                   sdesc_mnmajor_sw128(b0 + kk * 2048, 1024, 1024), idesc_o, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->pempty[jj % kPSlots]);  // the P buffer is free once these MMAs are done
      }
      if (!ok) {
        if (!*abort_v) raise_flag(a.errw, kFlagTimeout);
        *abort_v = 1;
      }
      // one commit for everything issued: the epilogue reads O after it, and
      // the CTA does not exit before the MMAs are done
      if (any) {
        umma_commit(&bars->ofull);
        mbar_wait_sleep(&bars->ofull, 0, kDrainBudget, nullptr);
      }
    }
  } else if (warp < 4) {
    // ---- producers: the query rows (TMA), then the K and V tiles
    const int ptid = tid - 32;
    if (ptid == 0) {
      mbar_expect_tx(&bars->q, kQBytes);
      tma_load_2d(qs, &tmq, &bars->q, 0, static_cast<int>(qi * H));
      tma_load_2d(qs + H * 128, &tmq, &bars->q, 64, static_cast<int>(qi * H));
    }
    if constexpr (!kGather) {
      if (ptid == 0) {
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
            long long r = static_cast<long long>(qt.t) - a.W + 1 + static_cast<long long>(j - qt.n_ct) * kHT -
                          qt.raw_base;
            r = r < -kHT ? -kHT : (r > a.T_raw ? a.T_raw : r);  // wholly outside: rows of fill, all masked
            *row = static_cast<int>(r);
          }
        };
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
            if (!*abort_v) raise_flag(a.errw, kFlagTimeout);
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
    } else {
      // row codes of the range's slots, then 16-byte gathers into the
      // swizzled tile layout; a tile is signalled once every producer's
      // copies of it have landed and been fenced for the tensor cores
      bool bad = false;
      for (int s = ptid; s < ntile * kHT; s += kProducers)
        codes_s[s / kHT][s % kHT] = slot_code(a, qi, b, qt.t, qt.n_c, qt.raw_base, j0 * kHT + s, &bad);
      if (bad) raise_flag(a.errw, kFlagIndex);
      prod_bar();
      const size_t rowb = static_cast<size_t>(kD) * 2;
      auto gather = [&](int jj, bool v) {
        const char* cb = static_cast<const char*>(v ? a.v_cmp : a.k_cmp) + static_cast<size_t>(b) * a.N * rowb;
        const char* rb = static_cast<const char*>(v ? a.v_raw : a.k_raw) + static_cast<size_t>(b) * a.T_raw * rowb;
        char* dst0 = kv + jj * kTileB;
        for (int c = ptid; c < kHT * 16; c += kProducers) {
          const int r = c >> 4, ch = c & 15;
          const int code = codes_s[jj][r];
          const char* src = code >= 0 ? cb + code * rowb : (code <= -2 ? rb + (-code - 2) * rowb : cb);
          cp_async16(dst0 + (ch >> 3) * kHalfB + r * 128 + (((ch & 7) ^ (r & 7)) << 4), src + ch * 16, code != -1);
        }
        cp_async_commit();
      };
      for (int jj = 0; jj < ntile; ++jj) gather(jj, false);
      for (int jj = 0; jj < ntile; ++jj) {
        cp_async_wait_pending(ntile - 1 - jj);
        fence_proxy_async();  // the rows are read by the tensor cores
        prod_bar();
        if (ptid == 0) mbar_arrive(&bars->kfull[jj]);
      }
      bool ok = true;
      for (int jj = 0; jj < ntile; ++jj) {
        if (ok) ok = mbar_wait_sleep(&bars->sdone[jj], 0, p.budget, abort_v);
        if (ok) {
          gather(jj, true);
        } else {
          cp_async_commit();  // keep the group count
        }
      }
      for (int jj = 0; jj < ntile; ++jj) {
        cp_async_wait_pending(ntile - 1 - jj);
        fence_proxy_async();
        prod_bar();
        if (ptid == 0) mbar_arrive(&bars->vfull[jj]);
      }
      if (!ok && ptid == 0) {
        if (!*abort_v) raise_flag(a.errw, kFlagTimeout);
        *abort_v = 1;
      }
      cp_async_wait<0>();
      // the query rows' bulk copy has landed before the CTA may exit (the MMA
      // thread's own wait for it may have given up)
      if (ptid == 0) mbar_wait_sleep(&bars->q, 0, kDrainBudget, nullptr);
    }
  } else {
    // ---- epilogue: warp -> (TMEM lane quarter, half of the heads)
    const int quarter = warp & 3;
    const int grp = (warp - 4) >> 2;
    const int etid = tid - 128;         // 0 .. 255
    const int i = quarter * 32 + lane;  // key row of every tile; d index of O
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true, bad = false;
    // which of this thread's key rows are attended, one bit per tile
    uint32_t vmask = 0;
    for (int jj = 0; jj < ntile; ++jj) {
      bool in;
      if constexpr (kGather) {
        in = slot_code(a, qi, b, qt.t, qt.n_c, qt.raw_base, (j0 + jj) * kHT + i, &bad) != -1;
      } else {
        in = hca_key_ok(a, qt, j0 + jj, i, &bad);
      }
      vmask |= (in ? 1u : 0u) << jj;
    }
    if (!kGather && __any_sync(0xffffffffu, bad) && lane == 0) raise_flag(a.errw, kFlagIndex);

    // per tile, as soon as its scores are in TMEM: the tile's per-head max,
    // P^T = 2^(s * sl2 - R) as bf16 rows, per-head sums in fp32
    for (int jj = 0; jj < ntile; ++jj) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bars->sdone[jj], 0, p.budget, abort_v));
      uint32_t r[2][16];
      const bool in = (vmask >> jj) & 1u;
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
        // the P buffer's previous tile has been read by its MMAs
        if (pring && jj >= kPSlots)
          ok = __all_sync(0xffffffffu, mbar_wait_sleep(&bars->pempty[jj % kPSlots],
                                                       static_cast<uint32_t>(jj / kPSlots - 1) & 1u, p.budget,
                                                       abort_v));
        char* row = pbuf(jj) + i * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int ch = grp * 4 + cc;
          if (ok)
            *reinterpret_cast<uint4*>(row + ((ch ^ (i & 7)) << 4)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        fence_proxy_async();  // the rows are read by the tensor cores
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0.f;
      }
      // the tile's score columns are read: the MMAs may write its output there
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->pfull[jj]);
      l_part[jj][quarter][grp * HPG + lane] = warp_reduce_scatter32<false>(v, lane);
    }
    epi_bar();
    // per head: the tiles' weights 2^(R_j - R) / L with R = max_j R_j and
    // L = sum_j 2^(R_j - R) L_j, and the log2-sum-exp R + log2 L
    if (etid < H) {
      const int h = etid;
      float Rj[kTcTiles], Lj[kTcTiles];
      float R = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kTcTiles; ++jj) {
        const float M = jj < ntile ? fmaxf(fmaxf(m_part[jj][0][h], m_part[jj][1][h]),
                                           fmaxf(m_part[jj][2][h], m_part[jj][3][h]))
                                   : -INFINITY;
        Rj[jj] = M == -INFINITY ? -INFINITY : r_s[jj][h];
        Lj[jj] = jj < ntile ? (l_part[jj][0][h] + l_part[jj][1][h]) + (l_part[jj][2][h] + l_part[jj][3][h]) : 0.f;
        R = fmaxf(R, Rj[jj]);
      }
      float L = 0.f, w[kTcTiles];
#pragma unroll
      for (int jj = 0; jj < kTcTiles; ++jj) {
        w[jj] = Rj[jj] == -INFINITY ? 0.f : ex2(Rj[jj] - R);
        L = fmaf(w[jj], Lj[jj], L);
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int jj = 0; jj < kTcTiles; ++jj) coef[jj][h] = w[jj] * inv;
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
        tmem_ld16(lane_addr + jj * H + grp * HPG, r[0]);
        tmem_ld16(lane_addr + jj * H + grp * HPG + 16, r[1]);
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
      if (p.cluster) {
        float* ps_o = part_s + (grp * HPG) * kD + i;
#pragma unroll
        for (int e = 0; e < 32; ++e) ps_o[e * kD] = o[e];
        if (quarter == 0) part_s[H * kD + grp * HPG + lane] = lse_s[grp * HPG + lane];
      } else if (p.nsplit > 1) {
        float* pb = a.part + ((qi * p.nsplit + split) * H + grp * HPG) * static_cast<long long>(kD + 1) + i;
#pragma unroll
        for (int e = 0; e < 32; ++e) pb[e * (kD + 1)] = o[e];
        if (quarter == 0)
          a.part[((qi * p.nsplit + split) * H + grp * HPG + lane) * static_cast<long long>(kD + 1) + kD] =
              lse_s[grp * HPG + lane];
      } else {
        const long long ob = (qi * H + grp * HPG) * static_cast<long long>(kD) + i;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          if (a.out_f32)
            static_cast<float*>(a.out)[ob + e * kD] = o[e];
          else
            static_cast<__nv_bfloat16*>(a.out)[ob + e * kD] = __float2bfloat16_rn(o[e]);
        }
        if (quarter == 0 && a.lse) {
          const float l2 = lse_s[grp * HPG + lane];
          a.lse[qi * H + grp * HPG + lane] = l2 == -INFINITY ? -INFINITY : l2 * kLn2;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  if (p.cluster) {
    // merge of the query's ranges: the cluster rank (= range) r owns a
    // contiguous share [g_lo, g_hi) of the H x kD outputs in groups of four
    // columns.  Once every CTA of the cluster is past its main loop, each
    // pushes every share of its partial, and its log2-sum-exps, into the
    // owner's receive buffer by bulk copies completing on the owner's mrecv;
    // each owner folds the ranges' partials of its share in range order, as
    // the combine kernel does
    constexpr int kGroups = H * kD / 4;
    const int ns = p.nsplit;
    const int cap = (kGroups + ns - 1) / ns;  // groups of one share, at most
    const int g_lo = split * kGroups / ns, g_hi = (split + 1) * kGroups / ns;
    float4* recv = reinterpret_cast<float4*>(kv + kRecvOff);               // [ns][cap]
    float* recv_l = reinterpret_cast<float*>(kv + kRecvOff + kRecvBytes);  // [ns][H]
    fence_proxy_async();  // the partial, written by the threads, is read by bulk copies
    cg::this_cluster().sync();  // every receive buffer of the cluster is free
    if (tid == 0) {
      mbar_expect_tx(&bars->mrecv, static_cast<uint32_t>(ns * ((g_hi - g_lo) * 16 + H * 4)));
      for (int o = 0; o < ns; ++o) {
        const int olo = o * kGroups / ns, ohi = (o + 1) * kGroups / ns;
        bulk_to_rank(recv + split * cap, part_s + 4 * olo, static_cast<uint32_t>((ohi - olo) * 16), &bars->mrecv, o);
        bulk_to_rank(recv_l + split * H, part_s + H * kD, H * 4, &bars->mrecv, o);
      }
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    bool got = mbar_wait_sleep(&bars->mrecv, 0, p.budget, abort_v);
    if (!got) {
      // reported, then waited out: no copy may still be writing this CTA's
      // shared memory when it exits
      if (tid == 0) raise_flag(a.errw, kFlagTimeout);
      mbar_wait_sleep(&bars->mrecv, 0, kDrainBudget, nullptr);
    }
    // (loops over the ranges kept rolled: this code runs once per CTA, and a
    // short body is fetched sooner than eight unrolled copies)
    for (int g = g_lo + tid; got && g < g_hi; g += kThreads) {
      const int h = g / (kD / 4), c4 = (g % (kD / 4)) * 4;
      float M = -INFINITY;
#pragma unroll 1
      for (int r = 0; r < ns; ++r) M = fmaxf(M, recv_l[r * H + h]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 0.f;
      if (M != -INFINITY) {
#pragma unroll 1
        for (int r = 0; r < ns; ++r) {
          const float f = ex2(recv_l[r * H + h] - M);
          const float4 v = recv[r * cap + (g - g_lo)];
          den += f;
          acc.x = fmaf(f, v.x, acc.x);
          acc.y = fmaf(f, v.y, acc.y);
          acc.z = fmaf(f, v.z, acc.z);
          acc.w = fmaf(f, v.w, acc.w);
        }
      }
      const float val[4] = {den > 0.f ? acc.x / den : 0.f, den > 0.f ? acc.y / den : 0.f,
                            den > 0.f ? acc.z / den : 0.f, den > 0.f ? acc.w / den : 0.f};
      const long long o = (qi * H + h) * static_cast<long long>(kD) + c4;
      if (a.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o) = make_float4(val[0], val[1], val[2], val[3]);
      } else {
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + o) =
            make_uint2(pack_bf16x2(val[0], val[1]), pack_bf16x2(val[2], val[3]));
      }
      if (a.lse && c4 == 0) a.lse[qi * H + h] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
    }
    // this CTA's partial has been read by every copy before it exits
    if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
}

}  // namespace

int attend_tc_tiles(bool csa, int N, int k, int W) {
  const long long w = (static_cast<long long>(W) + kHT - 1) / kHT;
  const long long t = csa ? (static_cast<long long>(k) + W + kHT - 1) / kHT
                          : (static_cast<long long>(N) + kHT - 1) / kHT + w;
  return t > 0x7fffffffLL ? 0x7fffffff : static_cast<int>(t);
}

TcPlan attend_tc_plan(int n_tiles, bool csa) {
  // the split depends on the key count only (never on the batch), so a
  // sequence gives identical results alone or in any batch.  Gathered (CSA)
  // ranges take up to five tiles (decode at 128K: 1024 + 128 slots = 9 tiles
  // in two ranges, one wave of CTAs for 64 queries); contiguous (HCA) ranges
  // up to four (1M context: 65 tiles in 17 ranges of 4)
  const int mt = csa ? kTcTiles : kTcTilesHca;
  TcPlan p;
  p.nsplit = n_tiles > 0 ? (n_tiles + mt - 1) / mt : 1;
  p.tpr = n_tiles > 0 ? (n_tiles + p.nsplit - 1) / p.nsplit : 1;
  return p;
}

bool attend_tc_supported(bool csa, int Tq, long long nq, int N, int T_raw, int k, int H, int d, int W) {
  // decode-shaped calls (prefill keeps the mma.sync kernel, which shares key
  // tiles between the queries of a sequence)
  if (Tq >= 16 || nq <= 0 || nq > 65535) return false;
  if (H != kH || d != kD) return false;
  if (csa) {
    if (k < 0 || k + W <= 0) return false;
  } else {
    if (N <= 0 || (W > 0 && T_raw <= 0)) return false;
  }
  return attend_tc_plan(attend_tc_tiles(csa, N, k, W), csa).nsplit <= 65535;
}

size_t attend_tc_part_bytes(long long nq, int H, int d, const TcPlan& p) {
  // up to kTcClusterMax ranges merge inside their cluster: no partials
  return p.nsplit > kTcClusterMax ? static_cast<size_t>(nq) * p.nsplit * H * (d + 1) * sizeof(float) : 0;
}

cudaError_t launch_attend_tc(const AttendArgs& a, long long budget, cudaStream_t s) {
  const bool csa = a.idx != nullptr;
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (nq == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmq, tkc, tvc, tkr, tvr;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(nq) * kH};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kH)};
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
  tkc = tvc = tkr = tvr = tmq;  // CSA gathers its rows: the key maps are never read
  if (!csa) {
    if (!rows_map(&tkc, a.k_cmp, a.N) || !rows_map(&tvc, a.v_cmp, a.N)) return cudaErrorInvalidValue;
    if (a.W > 0 && (!rows_map(&tkr, a.k_raw, a.T_raw) || !rows_map(&tvr, a.v_raw, a.T_raw)))
      return cudaErrorInvalidValue;
  }
  const TcPlan pl = attend_tc_plan(attend_tc_tiles(csa, a.N, a.k, a.W), csa);
  TcParams p;
  p.sl2 = a.scale * 1.4426950408889634f;
  p.nsplit = pl.nsplit;
  p.tpr = pl.tpr;
  p.cluster = pl.nsplit > 1 && pl.nsplit <= kTcClusterMax ? 1 : 0;
  p.budget = budget;
  const size_t smem = 1024 + 2 * kH * 128 + kTcTiles * 2 * kHalfB + kPSlots * kHT * 128 + sizeof(TcBars);
  const dim3 grid(static_cast<unsigned>(p.nsplit), static_cast<unsigned>(nq));
  cudaError_t e;
  if (csa) {
    e = ensure_dyn_smem<attend_tc_kernel<true>>(static_cast<int>(smem));
    if (e == cudaSuccess)
      e = launch_k(attend_tc_kernel<true>, grid, dim3(kThreads), smem, s, p.cluster ? p.nsplit : 1, tmq, tkc, tvc,
                   tkr, tvr, a, p);
  } else {
    e = ensure_dyn_smem<attend_tc_kernel<false>>(static_cast<int>(smem));
    if (e == cudaSuccess)
      e = launch_k(attend_tc_kernel<false>, grid, dim3(kThreads), smem, s, p.cluster ? p.nsplit : 1, tmq, tkc, tvc,
                   tkr, tvr, a, p);
  }
  if (e != cudaSuccess || p.nsplit == 1 || p.cluster) return e;
  return launch_attend_combine(a, p.nsplit, s);
}

}  // namespace csa
