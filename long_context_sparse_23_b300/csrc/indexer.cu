// (2) Lightning Indexer scores on the tcgen05 tensor cores.
// Octagono "Hybrid Attention: CSA and HCA" and "DeepSeek V4 technical review"
// section 2.1: every query token gets its own indexer queries (64 heads of
// width 128), which are scored against the compressed indexer keys:
//   S[n, j, b] = sum_h w[h] * ReLU(q_idx[n, j, h, :] . k_idx[n, b, :]),
// for the blocks b visible at the query's position, b < floor((t+1)/m).
//
// Design: the contraction runs with keys on the MMA's M dimension (one
// 128-key tile = the 128 TMEM lanes) and (query, head) pairs on N (a group of
// G queries x H_I heads, N <= 256 columns), K = d_I.  So every epilogue thread
// owns one key row and reduces sum_h w_h * max(acc, 0) over its own TMEM
// columns -- no cross-thread reduction.  Warp roles per CTA (320 threads):
//   warp 0     TMA producer: the query group once, then key tiles into an
//              S-stage shared-memory ring (128-byte swizzle, OOB rows zero);
//   warp 1     allocates TMEM; one lane issues tcgen05.mma (kind::f16, bf16
//              operands, fp32 accumulators) into two TMEM accumulator buffers;
//   warps 2-9  epilogue, two groups of four alternating tiles (group e owns
//              TMEM accumulator buffer e): tcgen05.ld the tile's accumulators,
//              apply ReLU and the head weights, store fp32 scores (one
//              coalesced row per warp) and count them into the top-k bucket
//              histogram.
// mbarriers connect the stages (full/empty per smem stage, full/empty per
// TMEM buffer); every wait is bounded and reports CSA_FLAG_TIMEOUT instead of
// hanging.  Tiles past the group's last visible block are never loaded.
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kEpiGroups = 2;                      // epilogue warp groups, alternating tiles
constexpr int kEpiWarp0 = 3;                       // first epilogue warp
constexpr int kThreads = 32 * kEpiWarp0 + 128 * kEpiGroups;  // 3 role warps + 8 epilogue warps
constexpr int kTileKeys = 128;
constexpr int kHalfBytes = kTileKeys * 128;  // one 64-wide K half of a key tile
constexpr int kMaxG = 64;                    // queries per group (H_I >= 4, G * H_I <= 256)
constexpr int kSmemLimit = 227 * 1024;       // dynamic + static shared memory per CTA
constexpr int kStaticSmem = 4 * 1024;        // upper bound of the kernel's static shared memory
constexpr long long kDrainBudget = 1LL << 31;

struct KParams {
  const float* w;
  long long w_stride;  // 0: one [HI] vector for every query; else w[(n * Tq + j) * w_stride + h]
  const int32_t* q_pos;
  float* S;
  long long ld;
  int B, Tq, N, m;
  int G;        // queries per group
  int NC;       // MMA N (columns per accumulator), multiple of 16
  int kh;       // K halves of 64 elements (d_I / 64 rounded up)
  int stages;
  int n_groups;       // ceil(Tq / G)
  int items_per_group;
  int tiles_per_item;
  int items;          // B * n_groups * items_per_group
  int per_cta;        // > 0: CTA c owns the contiguous ranks [c * per_cta, (c + 1) * per_cta)
  int tmem_cols;
  uint32_t* errw;
  long long budget;
  uint32_t* hist;  // [B*Tq][kTopkBins] (G == 1 only), or nullptr
  int after_zero;  // see IndexerArgs::after_zero
  const void* q_base;  // the indexer queries (for the L2 prefetch of the next item's rows)
  int q_row_bytes;     // bytes of one query head's row
  const float* q_scale;  // FP8: [B * Tq * HI] scale of each query head's codes
};

struct __align__(8) Bars {
  uint64_t full[8];    // key stage loaded
  uint64_t empty[8];   // key stage consumed by the MMAs
  uint64_t tfull[2];   // accumulator buffer written by the MMAs
  uint64_t tempty[2];  // accumulator buffer read by its epilogue group
  uint64_t qfull;      // a query group's rows loaded (one phase per load)
  uint64_t qfree;      // a query group's MMAs done: the query buffer may be refilled
  uint64_t wfull[2];   // head weights / visibility of an item written
  uint64_t wfree[2];   // both epilogue groups are done with an item's weights
  uint64_t sfree[8];   // FP8: the key scales of a stage read by the epilogue
};

// One work item: a group of G queries of sequence b against the key tiles
// [tile_lo, tile_lo + ntile) (ntile <= 0: nothing of that range is visible).
struct Item {
  int b, j0, tile_lo, ntile;
};

// Item of rank r, rank 0 the heaviest: query groups from the last (longest
// visible prefix) to the first; the sequences and tile ranges of one group
// next to each other.
__device__ __forceinline__ Item item_of(const KParams& p, int r) {
  Item it;
  const int per_g = p.B * p.items_per_group;
  const int g = p.n_groups - 1 - r / per_g;
  const int rem = r % per_g;
  it.b = rem / p.items_per_group;
  const int sub = rem % p.items_per_group;
  it.j0 = g * p.G;
  const int jn = min(p.G, p.Tq - it.j0);
  int nv_max = 0;
  for (int jj = 0; jj < jn; ++jj) {
    const int t = p.q_pos[static_cast<long long>(it.b) * p.Tq + it.j0 + jj];
    const int nv = t >= 0 ? (t + 1) / p.m : 0;
    nv_max = max(nv_max, min(nv, p.N));
  }
  const int n_tiles_all = (p.N + kTileKeys - 1) / kTileKeys;
  const int tiles_vis = (nv_max + kTileKeys - 1) / kTileKeys;
  it.tile_lo = sub * p.tiles_per_item;
  it.ntile = min(min(it.tile_lo + p.tiles_per_item, n_tiles_all), tiles_vis) - it.tile_lo;
  return it;
}

// Key tile of the item's i-th step: the item's tiles rotated by the CTA
// index, so CTAs working on the same (L2-resident) keys at the same time read
// different tiles, not all the same one.
__device__ __forceinline__ int tile_at(const Item& I, int i) {
  const int rot = static_cast<int>(blockIdx.x) % I.ntile;
  const int j = i + rot;
  return I.tile_lo + (j >= I.ntile ? j - I.ntile : j);
}

// Rank of this CTA's k-th item, or -1.  Items of unequal weight (prefill:
// causal rows of every length) go in rounds of gridDim.x ranks taken in
// alternating direction (snake order), so every CTA gets a similar share of
// heavy and light items; items of equal weight (decode: one query group per
// sequence) go in contiguous blocks, so a CTA's consecutive items share
// their query rows and histogram.
__device__ __forceinline__ int rank_of(int k, const KParams& p) {
  const int n = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  long long r;
  if (p.per_cta > 0) {
    if (k >= p.per_cta) return -1;
    r = static_cast<long long>(c) * p.per_cta + k;
  } else {
    r = static_cast<long long>(k) * n + ((k & 1) ? n - 1 - c : c);
  }
  return r < p.items ? static_cast<int>(r) : -1;
}

__device__ __forceinline__ bool same_group(const Item& a, const Item& b) { return a.b == b.b && a.j0 == b.j0; }

// A CTA's walk over its items with visible tiles: k is the current item's
// index in the CTA's list (-1: no more).  The first one is found before the
// warp roles split, so no role waits on a fresh global read before its first
// copy or MMA; each later one is fetched once the current item's work is
// issued.
struct Cursor {
  int k;
  Item I;
};
// Consecutive items of one query group whose tile ranges adjoin (a decode
// CTA's contiguous block) are taken as one run, so the roles meet at item
// boundaries only where the query group changes.
__device__ __forceinline__ bool advance(const KParams& p, Cursor& c) {
  for (int kk = c.k + 1;; ++kk) {
    const int r = rank_of(kk, p);
    if (r < 0) {
      c.k = -1;
      return false;
    }
    Item J = item_of(p, r);
    if (J.ntile > 0) {
      for (;;) {
        const int rn = rank_of(kk + 1, p);
        if (rn < 0) break;
        const Item Jn = item_of(p, rn);
        if (!same_group(J, Jn) || Jn.tile_lo != J.tile_lo + J.ntile || Jn.ntile <= 0) break;
        J.ntile += Jn.ntile;
        ++kk;
      }
      c.k = kk;
      c.I = J;
      return true;
    }
  }
}

__device__ __forceinline__ void group_bar(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 3, 256;" ::: "memory"); }

// Persistent kernel: one CTA per SM walks its items; the key ring, the TMEM
// accumulator pair and the item buffers run on across item boundaries.
// Warp roles (352 threads):
//   warp 0      key producer: TMA key tiles into the S-stage ring;
//   warp 1      allocates TMEM; one lane issues the MMAs;
//   warp 2      item producer: per item, the head weights and visibility
//               (double-buffered) and the query rows (TMA, one buffer, loaded
//               once the previous item's MMAs are done; the next item's rows
//               are prefetched into L2 meanwhile);
//   warps 3-10  epilogue, two groups of four alternating tiles.
// F8: keys and queries are E4M3 codes (one 128-byte row per key / query head,
// one power-of-two scale per row); the MMAs are kind::f8f6f4 and the
// epilogue applies the scales: sum_h (w_h s_q,h) ReLU(acc_h) * s_k.
template <int HI, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tms, KParams p) {
  if (p.after_zero) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else {
    pdl_wait_then_release();
  }
  extern __shared__ __align__(1024) char smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  char* qs = smem;                                      // [kh][NC][128 B]
  char* ks = qs + p.kh * p.NC * 128;                    // [stages][kh][128][128 B]
  // FP8: [stages][128] scales of the stage's keys
  float* ksc = reinterpret_cast<float*>(ks + p.stages * p.kh * kHalfBytes);
  Bars* bars = reinterpret_cast<Bars*>(reinterpret_cast<char*>(ksc) + (F8 ? p.stages * kTileKeys * 4 : 0));
  // top-k bucket histogram of the current item's scores (one query per group)
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(bars) + sizeof(Bars));
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float w_s[2][256];      // [item parity][G][HI] head weights of each query of the item
  __shared__ int nvis_s[2][kMaxG];   // [item parity][G] visible blocks of each query

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (p.hist)
    for (int i = tid; i < kTopkBins; i += kThreads) hist_s[i] = 0u;
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->sfree[s], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 4);
      mbar_init(&bars->wfull[i], 1);
      mbar_init(&bars->wfree[i], kEpiGroups);
    }
    mbar_init(&bars->qfull, 1);
    mbar_init(&bars->qfree, 1);
    mbar_fence_init();
  }
  // this CTA's first item with visible tiles (the same answer in every
  // thread; none: nothing to do)
  Cursor first;
  first.k = -1;
  const bool any = advance(p, first);
  __syncthreads();
  if (!any) return;

  // the TMEM address reaches the MMA and epilogue warps over a named barrier;
  // the two producer warps need no TMEM and start copying at once
  uint32_t tbase = 0;
  if (warp != 0 && warp != 2) {
    if (warp == 1) {
      tmem_alloc(&tmem_base, p.tmem_cols);
      tmem_relinquish();
    }
    tc_fence_before();
    asm volatile("bar.sync 4, %0;" ::"r"(kThreads - 64) : "memory");
    tc_fence_after();
    tbase = tmem_base;
  }
  volatile int* abort_v = &abort_flag;
  auto fail = [&]() {
    if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
    *abort_v = 1;
  };

  if (warp == 0) {
    // ---- key producer
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      if (F8) tma_prefetch_desc(&tms);
      // the keys are read once per query group: evict-first, so the scores
      // this kernel writes stay in L2 for the top-k that reads them next
      const uint64_t key_policy = l2_policy_evict_first();
      int gt = 0;  // key tiles issued
      bool ok = true;
      for (Cursor c = first; ok && c.k >= 0; advance(p, c)) {
        const Item& I = c.I;
        for (int i = 0; i < I.ntile; ++i) {
          const int s = gt % p.stages;
          const uint32_t ph = (gt / p.stages) & 1;
          if (!mbar_wait(&bars->empty[s], ph ^ 1, p.budget, abort_v) ||
              (F8 && !mbar_wait(&bars->sfree[s], ph ^ 1, p.budget, abort_v))) {
            fail();
            ok = false;
            break;
          }
          mbar_expect_tx(&bars->full[s], p.kh * kHalfBytes + (F8 ? kTileKeys * 4 : 0));
          char* dst = ks + s * p.kh * kHalfBytes;
          for (int h = 0; h < p.kh; ++h)
            tma_load_3d_hint(dst + h * kHalfBytes, &tmk, &bars->full[s], h * 64, tile_at(I, i) * kTileKeys, I.b,
                             key_policy);
          if (F8) tma_load_2d(ksc + s * kTileKeys, &tms, &bars->full[s], tile_at(I, i) * kTileKeys, I.b);
          ++gt;
        }
      }
      // drain: every issued copy has landed before the CTA may exit
      for (int s = 0; s < p.stages && s < gt; ++s) {
        const int last = gt - 1 - ((gt - 1 - s) % p.stages);
        mbar_wait(&bars->full[s], (last / p.stages) & 1, kDrainBudget, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = F8 ? idesc_e4m3_f32(128, p.NC) : idesc_bf16_f32(128, p.NC);
      int gt = 0, nq = 0;
      bool ok = true;
      Item prev{-1, -1, 0, 0};
      for (Cursor c = first; ok && c.k >= 0; advance(p, c)) {
        const Item I = c.I;
        if (nq == 0 || !same_group(I, prev)) {
          // a new query group: the query buffer may be refilled once the
          // previous group's MMAs are done, and this group's rows must be in
          if (nq > 0) umma_commit(&bars->qfree);
          if (!mbar_wait(&bars->qfull, nq & 1, p.budget, abort_v)) {
            fail();
            break;
          }
          ++nq;
        }
        prev = I;
        for (int i = 0; i < I.ntile; ++i) {
          const int s = gt % p.stages;
          const uint32_t ph = (gt / p.stages) & 1;
          const int acc = gt & 1;
          const uint32_t aph = (gt >> 1) & 1;
          if (!mbar_wait(&bars->tempty[acc], aph ^ 1, p.budget, abort_v) ||
              !mbar_wait(&bars->full[s], ph, p.budget, abort_v)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(ks + s * p.kh * kHalfBytes);
          const uint32_t b0 = smem_u32(qs);
          const uint32_t d = tbase + static_cast<uint32_t>(acc * p.NC);
          for (int kk = 0; kk < p.kh * 4; ++kk) {
            const int h = kk >> 2, w = kk & 3;
            const uint64_t ad = sdesc_kmajor_sw128(a0 + h * kHalfBytes + w * 32);
            const uint64_t bd = sdesc_kmajor_sw128(b0 + h * p.NC * 128 + w * 32);
            if constexpr (F8)
              umma_f8(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
            else
              umma_f16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars->empty[s]);
          umma_commit(&bars->tfull[acc]);
          ++gt;
        }
        if (!ok) break;
      }
      // drain: the last MMAs have finished reading shared memory / writing TMEM
      if (gt > 0) mbar_wait(&bars->tfull[(gt - 1) & 1], ((gt - 1) >> 1) & 1, kDrainBudget, nullptr);
    }
  } else if (warp == 2) {
    // ---- item producer: query rows first (the MMAs wait for them), then the
    // head weights and visibility the epilogue needs
    if (lane == 0) tma_prefetch_desc(&tmq);
    int it = 0, nq = 0;
    Item prev{-1, -1, 0, 0};
    for (Cursor c = first; c.k >= 0; advance(p, c)) {
      const Item I = c.I;
      const int ib = it & 1;
      const bool new_group = nq == 0 || !same_group(I, prev);
      prev = I;
      bool ok = true;
      if (lane == 0 && new_group) {
        // the query rows, once the MMAs of the previous query group are done
        ok = nq == 0 || mbar_wait(&bars->qfree, (nq - 1) & 1, p.budget, abort_v);
        if (ok) {
          mbar_expect_tx(&bars->qfull, p.kh * p.NC * 128);
          const int qrow = (I.b * p.Tq + I.j0) * HI;
          for (int h = 0; h < p.kh; ++h) tma_load_2d(qs + h * p.NC * 128, &tmq, &bars->qfull, h * 64, qrow);
          // the next item's query rows into L2 while this item runs
          Cursor nx = c;
          if (advance(p, nx)) {
            const Item& J = nx.I;
            const int jn = min(p.G, p.Tq - J.j0);
            const uint32_t bytes = static_cast<uint32_t>(jn * HI * p.q_row_bytes);
            const char* src = static_cast<const char*>(p.q_base) +
                              (static_cast<size_t>(J.b) * p.Tq + J.j0) * HI * p.q_row_bytes;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
          }
        }
        if (!ok) fail();
      }
      if (lane == 0 && ok && it >= 2) {
        // the weight buffer of parity ib was last read for item it - 2
        ok = mbar_wait(&bars->wfree[ib], ((it - 2) >> 1) & 1, p.budget, abort_v);
        if (!ok) fail();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (new_group) ++nq;
      for (int i = lane; i < p.G * HI; i += 32) {
        const int jj = i / HI, h = i % HI;
        const long long qrow = static_cast<long long>(I.b) * p.Tq + I.j0 + jj;
        float wv = p.w_stride == 0 ? p.w[h] : (I.j0 + jj < p.Tq ? p.w[qrow * p.w_stride + h] : 0.f);
        // FP8: the query head's scale (a power of two) folds into its weight
        if (F8) wv = I.j0 + jj < p.Tq ? wv * p.q_scale[qrow * HI + h] : 0.f;
        w_s[ib][i] = wv;
      }
      for (int jj = lane; jj < p.G; jj += 32) {
        int nv = 0;
        if (I.j0 + jj < p.Tq) {
          const int t = p.q_pos[static_cast<long long>(I.b) * p.Tq + I.j0 + jj];
          nv = t >= 0 ? (t + 1) / p.m : 0;
          nv = nv < p.N ? nv : p.N;
        }
        nvis_s[ib][jj] = nv;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->wfull[ib]);
      ++it;
    }
    // drain: the last query copy has landed before the CTA may exit
    if (lane == 0 && nq > 0) mbar_wait(&bars->qfull, (nq - 1) & 1, kDrainBudget, nullptr);
  } else {
    // ---- epilogue warps: TMEM lane quarter = warp % 4; group e handles the
    // CTA's tiles gt = e (mod 2), i.e. TMEM accumulator buffer e
    const int ew = warp - kEpiWarp0;
    const int egroup = ew >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t col0 = lane_addr + static_cast<uint32_t>(egroup * p.NC);
    int gt = 0, it = 0;
    bool waited_zero = false;
    for (Cursor c = first; c.k >= 0; advance(p, c)) {
      const Item I = c.I;
      const int ib = it & 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->wfull[ib], (it >> 1) & 1, p.budget, abort_v));
      if (!ok && lane == 0) fail();
      const float* wi = w_s[ib];
      const int* nvi = nvis_s[ib];
      const long long srow0 = static_cast<long long>(I.b) * p.Tq + I.j0;
      for (int i = 0; i < I.ntile; ++i) {
        const int g2 = gt + i;
        if ((g2 & 1) != egroup) continue;
        const uint32_t aph = (g2 >> 1) & 1;
        const int st = g2 % p.stages;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->tfull[egroup], aph, p.budget, abort_v));
        // FP8: the key's scale, read before the stage's scale slot is released
        // (the stage's load phase is complete, so this wait returns at once and
        // makes the copy's writes visible to this thread)
        float kscale = 1.f;
        if (F8 && ok) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[st], (g2 / p.stages) & 1, p.budget, abort_v));
          if (ok) kscale = ksc[st * kTileKeys + row];
        }
        if (F8) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->sfree[st]);
        }
        if (!ok) {
          if (lane == 0) fail();
        } else {
          tc_fence_after();
          const int key = tile_at(I, i) * kTileKeys + row;
          if constexpr (HI >= 16) {
            for (int jj = 0; jj < p.G; ++jj) {
              // all of the query's head columns in flight at once, one wait
              uint32_t rr[HI / 16][16];
#pragma unroll
              for (int hc = 0; hc < HI / 16; ++hc) tmem_ld16(col0 + jj * HI + hc * 16, rr[hc]);
              tmem_ld_wait();
              const float* wq = wi + jj * HI;
              float sum = 0.f;
#pragma unroll
              for (int hc = 0; hc < HI / 16; ++hc)
#pragma unroll
                for (int e = 0; e < 16; ++e) sum = fmaf(wq[hc * 16 + e], fmaxf(__uint_as_float(rr[hc][e]), 0.f), sum);
              if (F8) sum *= kscale;
              const bool vis = key < nvi[jj];
              if (vis) p.S[(srow0 + jj) * p.ld + key] = sum;
              if (p.hist) {
                // bucket = top 12 bits of the order-preserving key of sum
                uint32_t u = __float_as_uint(sum);
                u = u == 0x80000000u ? 0u : u;
                u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
                const unsigned am = __ballot_sync(0xffffffffu, vis);
                if (vis) {
                  const unsigned peers = __match_any_sync(am, u >> 20);
                  if (lane == __ffs(peers) - 1) atomicAdd(&hist_s[u >> 20], static_cast<uint32_t>(__popc(peers)));
                }
              }
            }
          } else {
            constexpr int QPC = 16 / HI;  // queries per 16-column chunk
            for (int c0 = 0; c0 < p.NC; c0 += 16) {
              uint32_t rr[16];
              tmem_ld16(col0 + c0, rr);
              tmem_ld_wait();
#pragma unroll
              for (int qq = 0; qq < QPC; ++qq) {
                const int jj = c0 / HI + qq;
                const float* wq = wi + (jj < p.G ? jj : 0) * HI;
                float sum = 0.f;
#pragma unroll
                for (int e = 0; e < HI; ++e) sum = fmaf(wq[e], fmaxf(__uint_as_float(rr[qq * HI + e]), 0.f), sum);
                if (jj < p.G && key < nvi[jj]) p.S[(srow0 + jj) * p.ld + key] = sum;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tempty[egroup]);
      }
      gt += I.ntile;
      // this group is done with the item's weights and visibility
      group_bar(egroup);
      if ((ew & 3) == 0 && lane == 0) mbar_arrive(&bars->wfree[ib]);
      Cursor nx = c;
      if (p.hist && !(advance(p, nx) && same_group(I, nx.I))) {
        // both groups' counts of the query group are in: flush them (once
        // the histogram has been zeroed), then clear for the next group
        epi_bar();
        if (p.after_zero && !waited_zero) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          waited_zero = true;
        }
        uint32_t* g = p.hist + srow0 * kTopkBins;
        for (int i = ew * 32 + lane; i < kTopkBins; i += 32 * 4 * kEpiGroups) {
          const uint32_t v = hist_s[i];
          if (v) {
            atomicAdd(g + i, v);
            hist_s[i] = 0u;
          }
        }
        epi_bar();
      }
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, p.tmem_cols);
  }
}

template <int HI, bool F8>
cudaError_t launch_hi(const IndexerArgs& a, cudaStream_t s) {
  KParams p;
  p.w = a.w;
  p.w_stride = a.w_stride;
  p.q_pos = a.q_pos;
  p.S = a.scores;
  p.ld = a.ld;
  p.B = a.B;
  p.Tq = a.Tq;
  p.N = a.N;
  p.m = a.m;
  p.G = a.Tq < 256 / HI ? a.Tq : 256 / HI;
  p.NC = ((p.G * HI + 15) / 16) * 16;
  p.kh = F8 ? 1 : (a.d_I + 63) / 64;  // 128-byte rows: 64 bf16 or 128 E4M3 values
  p.n_groups = (a.Tq + p.G - 1) / p.G;
  int cols = 32;
  while (cols < 2 * p.NC) cols *= 2;
  p.tmem_cols = cols;
  const int q_bytes = p.kh * p.NC * 128;
  const int stage_bytes = p.kh * kHalfBytes;
  const bool fill_hist = a.hist != nullptr && p.G == 1 && HI >= 16;
  const int hist_bytes = fill_hist ? kTopkBins * 4 : 0;
  const int dyn_limit = kSmemLimit - kStaticSmem;
  int stages = (dyn_limit - 1024 - q_bytes - static_cast<int>(sizeof(Bars)) - hist_bytes) /
               (stage_bytes + (F8 ? kTileKeys * 4 : 0));
  stages = stages > 8 ? 8 : stages;
  if (stages < 2) return cudaErrorNotSupported;
  p.stages = stages;
  const int n_tiles_all = (a.N + kTileKeys - 1) / kTileKeys;
  const long long groups = static_cast<long long>(a.B) * p.n_groups;
  const int n_sm = sm_count();
  // tile ranges per group when the groups alone cannot fill the GPU: as many
  // that the item count is a multiple of the SM count (lcm(groups, SMs)
  // items), or failing that (too few tiles) one item per SM
  int ipg = 1;
  if (groups < n_sm) {
    long long g = groups, h = n_sm;
    while (h != 0) {
      const long long t = g % h;
      g = h;
      h = t;
    }
    ipg = static_cast<int>(n_sm / g);
    if (ipg > n_tiles_all) ipg = static_cast<int>(n_sm / groups);
    ipg = ipg < 1 ? 1 : (ipg > n_tiles_all ? n_tiles_all : ipg);
  }
  p.tiles_per_item = (n_tiles_all + ipg - 1) / ipg;
  p.items_per_group = (n_tiles_all + p.tiles_per_item - 1) / p.tiles_per_item;
  p.errw = a.errw;
  p.budget = a.budget;
  p.hist = fill_hist ? a.hist : nullptr;
  p.after_zero = p.hist != nullptr && a.after_zero;
  p.q_base = a.q_idx;
  p.q_row_bytes = a.d_I * (F8 ? 1 : 2);
  p.q_scale = a.q_scale;
  const long long items = groups * p.items_per_group;
  if (items == 0 || n_tiles_all == 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorNotSupported;
  p.items = static_cast<int>(items);
  const int grid = static_cast<int>(items < n_sm ? items : n_sm);
  // one query group per sequence (decode): items of equal weight, in
  // contiguous blocks per CTA; several groups per sequence (prefill, causal
  // rows of every length): snake order
  p.per_cta = p.n_groups == 1 ? static_cast<int>((items + grid - 1) / grid) : 0;

  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int esz = F8 ? 1 : 2;
  const cuuint32_t box_x = F8 ? 128 : 64;  // one 128-byte swizzle row
  CUtensorMap tmk, tmq, tms;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.d_I), static_cast<cuuint64_t>(a.N),
                          static_cast<cuuint64_t>(a.B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.d_I) * esz,
                             static_cast<cuuint64_t>(a.N) * a.d_I * esz};
    cuuint32_t box[3] = {box_x, static_cast<cuuint32_t>(kTileKeys), 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tmk, dt, 3, const_cast<void*>(a.k_idx), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.d_I),
                          static_cast<cuuint64_t>(a.B) * a.Tq * HI};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.d_I) * esz};
    cuuint32_t box[2] = {box_x, static_cast<cuuint32_t>(p.NC)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmq, dt, 2, const_cast<void*>(a.q_idx), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  tms = tmq;  // bf16: the key-scale map is never read
  if (F8) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.N), static_cast<cuuint64_t>(a.B)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.N) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileKeys), 1};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.k_scale), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const size_t smem = 1024 + q_bytes + static_cast<size_t>(stages) * (stage_bytes + (F8 ? kTileKeys * 4 : 0)) +
                     sizeof(Bars) + hist_bytes;
  cudaError_t e = ensure_dyn_smem<indexer_kernel<HI, F8>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_k(indexer_kernel<HI, F8>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), smem, s, 1, tmk, tmq,
                  tms, p);
}

}  // namespace

// ---- host: tensor maps -----------------------------------------------------
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

bool indexer_fills_hist(int Tq, int H_I) { return Tq == 1 && H_I >= 16; }

bool indexer_fp8_supported(int H_I, int d_I, int N) {
  return (H_I == 16 || H_I == 32 || H_I == 64 || H_I == 128) && d_I == 128 && N % 4 == 0;
}

cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s) {
  if (a.fp8) {
    if (!indexer_fp8_supported(a.H_I, a.d_I, a.N)) return cudaErrorNotSupported;
    switch (a.H_I) {
      case 16: return launch_hi<16, true>(a, s);
      case 32: return launch_hi<32, true>(a, s);
      case 64: return launch_hi<64, true>(a, s);
      default: return launch_hi<128, true>(a, s);
    }
  }
  switch (a.H_I) {
    case 4: return launch_hi<4, false>(a, s);
    case 8: return launch_hi<8, false>(a, s);
    case 16: return launch_hi<16, false>(a, s);
    case 32: return launch_hi<32, false>(a, s);
    case 64: return launch_hi<64, false>(a, s);
    case 128: return launch_hi<128, false>(a, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace csa
