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
// columns -- no cross-thread reduction.  A work item is one query group
// against a range of 128-key tiles; TMA feeds a 128-byte-swizzled shared-
// memory ring of key tiles, one thread issues tcgen05.mma into TMEM
// accumulators, and groups of four epilogue warps read them (tcgen05.ld,
// ReLU and the head weights, coalesced fp32 scores, the top-k bucket
// histogram).  Two kernels:
//   indexer_single_kernel  decode (one query group per sequence): one item
//                          per CTA; the query rows and the first key tile
//                          are requested before any global read;
//   indexer_kernel         prefill (query groups of every causal length):
//                          persistent, one CTA per SM walking its items
//                          (heavy first, snake order), an item producer warp
//                          loading each item's weights and query rows; every
//                          epilogue group on every tile, its share of the
//                          queries copied to registers before the reduction.
// mbarriers connect the stages (full/empty per smem stage, full/empty per
// TMEM buffer); every wait is bounded and reports CSA_FLAG_TIMEOUT instead of
// hanging.  Tiles past the group's last visible block are never loaded, but
// for the first ring stages of a decode item, which are requested before the
// visibility is read (such a tile lands and is left unread).
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kEpiGroups = 2;                      // epilogue warp groups
constexpr int kEpiWarp0 = 3;                       // first epilogue warp
// The persistent kernel's epilogue groups: four when a group's share of the
// 256 accumulator columns (64) holds whole queries (H_I <= 64), else two.
template <int HI>
constexpr int epi_groups_p() { return HI <= 64 ? 4 : 2; }
template <int HI>
constexpr int threads_p() { return 32 * kEpiWarp0 + 128 * epi_groups_p<HI>(); }
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
  int tmem_cols;
  int acc_shift;  // one-item kernel on E4M3 keys: 1 << acc_shift TMEM accumulators (2 or 4)
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
  uint64_t tfull[4];   // accumulator buffer written by the MMAs
  uint64_t tempty[4];  // accumulator buffer read by its epilogue group
  uint64_t qfull;      // the item's queries loaded
  uint64_t qfree;      // the item's MMAs done: the query buffer may be refilled
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

// Rank of this CTA's k-th item, or -1: rounds of gridDim.x ranks, taken in
// alternating direction (snake order), so every CTA gets a similar share of
// heavy and light items.
__device__ __forceinline__ int rank_of(int k, const KParams& p) {
  const int n = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const long long r = static_cast<long long>(k) * n + ((k & 1) ? n - 1 - c : c);
  return r < p.items ? static_cast<int>(r) : -1;
}

__device__ __forceinline__ void group_bar(int g) {
  asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
}
template <int NT>
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 5, %0;" ::"n"(NT) : "memory"); }

// Persistent kernel: one CTA per SM walks its items; the key ring, the TMEM
// accumulator pair and the item buffers run on across item boundaries.
// Warp roles (608 threads for H_I <= 64, 352 for H_I = 128):
//   warp 0      key producer: TMA key tiles into the S-stage ring;
//   warp 1      allocates TMEM; one lane issues the MMAs;
//   warp 2      item producer: per item, the head weights and visibility
//               (double-buffered) and the query rows (TMA, one buffer, loaded
//               once the previous item's MMAs are done; the next item's rows
//               are prefetched into L2 meanwhile);
//   warps 3..   epilogue, four groups of four (two for H_I = 128), all on
//               every tile, each group its share of the group's queries.
// F8: keys and queries are E4M3 codes (one 128-byte row per key / query head,
// one power-of-two scale per row); the MMAs are kind::f8f6f4 and the
// epilogue applies the scales: sum_h (w_h s_q,h) ReLU(acc_h) * s_k.
template <int HI, bool F8>
__global__ void __launch_bounds__(threads_p<HI>(), 1)
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
    for (int i = tid; i < kTopkBins; i += threads_p<HI>()) hist_s[i] = 0u;
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->sfree[s], 4 * epi_groups_p<HI>());
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 4 * epi_groups_p<HI>());
      mbar_init(&bars->wfull[i], 1);
      mbar_init(&bars->wfree[i], epi_groups_p<HI>());
    }
    mbar_init(&bars->qfull, 1);
    mbar_init(&bars->qfree, 1);
    mbar_fence_init();
  }
  // does this CTA own any item? (the same answer in every thread; an item
  // with nothing visible is skipped by every role, so its visibility, a
  // global read, is left to the roles rather than delaying the first copy)
  const bool any = rank_of(0, p) >= 0;
  __syncthreads();
  if (!any) return;

  if (warp == 1) {
    tmem_alloc(&tmem_base, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
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
      for (int k = 0; ok; ++k) {
        const int r = rank_of(k, p);
        if (r < 0) break;
        const Item I = item_of(p, r);
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
      int gt = 0, it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int r = rank_of(k, p);
        if (r < 0) break;
        const Item I = item_of(p, r);
        if (I.ntile <= 0) continue;
        if (!mbar_wait(&bars->qfull, it & 1, p.budget, abort_v)) {
          fail();
          break;
        }
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
        umma_commit(&bars->qfree);  // the query buffer is free once this item's MMAs are done
        ++it;
      }
      // drain: the last MMAs have finished reading shared memory / writing TMEM
      if (gt > 0) mbar_wait(&bars->tfull[(gt - 1) & 1], ((gt - 1) >> 1) & 1, kDrainBudget, nullptr);
    }
  } else if (warp == 2) {
    // ---- item producer: query rows first (the MMAs wait for them), then the
    // head weights and visibility the epilogue needs
    if (lane == 0) tma_prefetch_desc(&tmq);
    int it = 0, q_issued = 0;
    for (int k = 0;; ++k) {
      const int r = rank_of(k, p);
      if (r < 0) break;
      const Item I = item_of(p, r);
      if (I.ntile <= 0) continue;
      const int ib = it & 1;
      bool ok = true;
      if (lane == 0) {
        // the query rows, once the MMAs of the previous item are done
        ok = it == 0 || mbar_wait(&bars->qfree, (it - 1) & 1, p.budget, abort_v);
        if (ok) {
          mbar_expect_tx(&bars->qfull, p.kh * p.NC * 128);
          const int qrow = (I.b * p.Tq + I.j0) * HI;
          for (int h = 0; h < p.kh; ++h) tma_load_2d(qs + h * p.NC * 128, &tmq, &bars->qfull, h * 64, qrow);
          q_issued = it + 1;
          // the next item's query rows into L2 while this item runs
          const int rn = rank_of(k + 1, p);
          if (rn >= 0) {
            const Item J = item_of(p, rn);
            const int jn = min(p.G, p.Tq - J.j0);
            const uint32_t bytes = static_cast<uint32_t>(jn * HI * p.q_row_bytes);
            const char* src = static_cast<const char*>(p.q_base) +
                              (static_cast<size_t>(J.b) * p.Tq + J.j0) * HI * p.q_row_bytes;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
          }
          // the weight buffer of parity ib was last read for item it - 2
          if (it >= 2) ok = mbar_wait(&bars->wfree[ib], ((it - 2) >> 1) & 1, p.budget, abort_v);
        }
        if (!ok) fail();
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
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
    if (lane == 0 && q_issued > 0) mbar_wait(&bars->qfull, (q_issued - 1) & 1, kDrainBudget, nullptr);
  } else {
    // ---- epilogue warps: TMEM lane quarter = warp % 4; every group takes
    // every tile (TMEM accumulator gt mod 2), group e its share of the
    // group's queries (H_I >= 16) or of the 16-column chunks (H_I < 16), so
    // a tile's epilogue is split EG ways and the MMAs into the other
    // accumulator hide it
    const int ew = warp - kEpiWarp0;
    const int egroup = ew >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int EG = epi_groups_p<HI>();
    const int qh = (p.G + EG - 1) / EG;
    const int jlo = min(p.G, egroup * qh), jhi = min(p.G, jlo + qh);
    const int ch_h = (p.NC / 16 + EG - 1) / EG;
    const int clo = min(p.NC, egroup * ch_h * 16), chi = min(p.NC, (egroup + 1) * ch_h * 16);
    int gt = 0, it = 0;
    bool waited_zero = false;
    for (int k = 0;; ++k) {
      const int r = rank_of(k, p);
      if (r < 0) break;
      const Item I = item_of(p, r);
      if (I.ntile <= 0) continue;
      const int ib = it & 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->wfull[ib], (it >> 1) & 1, p.budget, abort_v));
      if (!ok && lane == 0) fail();
      const float* wi = w_s[ib];
      const int* nvi = nvis_s[ib];
      const long long srow0 = static_cast<long long>(I.b) * p.Tq + I.j0;
      for (int i = 0; i < I.ntile; ++i) {
        const int g2 = gt + i;
        const int acc = g2 & 1;
        const uint32_t aph = (g2 >> 1) & 1;
        const int st = g2 % p.stages;
        const uint32_t col0 = lane_addr + static_cast<uint32_t>(acc * p.NC);
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->tfull[acc], aph, p.budget, abort_v));
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
        bool released = false;
        if (!ok) {
          if (lane == 0) fail();
        } else {
          tc_fence_after();
          const int key = tile_at(I, i) * kTileKeys + row;
          if constexpr (HI >= 16) {
            // this group's share of the accumulator (G / EG queries x H_I
            // heads = 256 / EG columns: here G = 256 / H_I) into registers,
            // then the accumulator is released before the reduction, so the
            // MMAs of tile gt + 2 need not wait for it
            constexpr int NQ = 256 / EG / HI;
            constexpr int NCH = 256 / EG / 16;
            uint32_t rv[NCH][16];
#pragma unroll
            for (int c = 0; c < NCH; ++c) tmem_ld16(col0 + jlo * HI + c * 16, rv[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[acc]);
            released = true;
#pragma unroll
            for (int jq = 0; jq < NQ; ++jq) {
              const int jj = jlo + jq;
              const float* wq = wi + jj * HI;
              float sum = 0.f;
#pragma unroll
              for (int h = 0; h < HI; ++h)
                sum = fmaf(wq[h], fmaxf(__uint_as_float(rv[(jq * HI + h) >> 4][(jq * HI + h) & 15]), 0.f), sum);
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
            for (int c0 = clo; c0 < chi; c0 += 16) {
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
        if (!released) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->tempty[acc]);
        }
      }
      gt += I.ntile;
      // this group is done with the item's weights and visibility
      group_bar(egroup);
      if ((ew & 3) == 0 && lane == 0) mbar_arrive(&bars->wfree[ib]);
      if (p.hist) {
        // both groups' counts of the item are in: flush them (once the
        // histogram has been zeroed), then clear for the next item
        epi_bar<128 * EG>();
        if (p.after_zero && !waited_zero) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          waited_zero = true;
        }
        uint32_t* g = p.hist + srow0 * kTopkBins;
        for (int i = ew * 32 + lane; i < kTopkBins; i += 32 * 4 * EG) {
          const uint32_t v = hist_s[i];
          if (v) {
            atomicAdd(g + i, v);
            hist_s[i] = 0u;
          }
        }
        epi_bar<128 * EG>();
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

// One work item per CTA (decode: one query group per sequence, a range of
// its key tiles per CTA): 320 threads, no item loop.  Thread 0 initialises
// the barriers and at once requests the query rows and the first key tile
// (they need no global read: the item follows from the block index), while
// the other threads read the visibility and head weights; then the rest of
// the S-stage ring is requested, warp 0 keeps it filled, warp 1 issues the
// MMAs into two TMEM accumulators (four with E4M3 keys), warps 2-9 are the
// epilogue (two groups of four alternating tiles).  The same arithmetic as
// the persistent kernel.
constexpr int kThreads1 = 64 + 128 * kEpiGroups;

template <int HI, bool F8>
__global__ void __launch_bounds__(kThreads1, 1)
    indexer_single_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
                          const __grid_constant__ CUtensorMap tms, KParams p) {
  if (p.after_zero) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else {
    pdl_wait_then_release();
  }
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  char* qs = smem;                                      // [kh][NC][128 B]
  char* ks = qs + p.kh * p.NC * 128;                    // [stages][kh][128][128 B]
  float* ksc = reinterpret_cast<float*>(ks + p.stages * p.kh * kHalfBytes);  // FP8: [stages][128]
  Bars* bars = reinterpret_cast<Bars*>(reinterpret_cast<char*>(ksc) + (F8 ? p.stages * kTileKeys * 4 : 0));
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(bars) + sizeof(Bars));
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float w_s[256];      // [G][HI]
  __shared__ int nvis_s[kMaxG];   // [G]

  // TMEM accumulators: with E4M3 keys four when they fit in the 512 columns
  // (the MMAs run up to three tiles ahead of the epilogue, the longer stage
  // there), else two; two with bf16 keys
  const int acc_sh = F8 ? p.acc_shift : 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this CTA's (sequence, query group, tile range); heavy first
  const int item = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
  const int grp = item / p.items_per_group;
  const int sub = item % p.items_per_group;
  const int b = grp / p.n_groups;
  const int j0 = (grp % p.n_groups) * p.G;
  const int n_tiles_all = (p.N + kTileKeys - 1) / kTileKeys;
  const int tile_lo = sub * p.tiles_per_item;
  // the item's tiles before the visibility cut, of which the first n_pre are
  // requested at once
  const int tile_cap = min(tile_lo + p.tiles_per_item, n_tiles_all);
  const int n_pre = min(p.stages, max(tile_cap - tile_lo, 0));
  const uint32_t stage_tx = p.kh * kHalfBytes + (F8 ? kTileKeys * 4 : 0);
  char* const ks_c = ks;
  uint64_t key_policy = 0;
  auto issue_tile = [&](int i, int s) {  // key tile tile_lo + i into stage s (thread 0)
    mbar_expect_tx(&bars->full[s], stage_tx);
    char* dst = ks_c + s * p.kh * kHalfBytes;
    for (int h = 0; h < p.kh; ++h)
      tma_load_3d_hint(dst + h * kHalfBytes, &tmk, &bars->full[s], h * 64, (tile_lo + i) * kTileKeys, b,
                       key_policy);
    if (F8) tma_load_2d(ksc + s * kTileKeys, &tms, &bars->full[s], (tile_lo + i) * kTileKeys, b);
  };
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->sfree[s], 4);
    }
    for (int i = 0; i < (1 << acc_sh); ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 4);
    }
    mbar_init(&bars->qfull, 1);
    mbar_fence_init();
    // the query rows and the first key tile need no global read: they are
    // requested before the visibility, weights and TMEM are set up; the
    // next stages follow once those are (every stage is free at the start;
    // a tile that turns out invisible is loaded and left unread).  Alone in
    // flight at first, each CTA's first tile lands sooner, and the MMAs
    // start earlier.  The keys are read once: evict-first, so the scores
    // this kernel writes stay in L2 for the top-k that reads them next
    key_policy = l2_policy_evict_first();
    const int qrow = (b * p.Tq + j0) * HI;
    mbar_expect_tx(&bars->qfull, p.kh * p.NC * 128);
    for (int h = 0; h < p.kh; ++h) tma_load_2d(qs + h * p.NC * 128, &tmq, &bars->qfull, h * 64, qrow);
    if (n_pre > 0) issue_tile(0, 0);
  }
  for (int jj = tid; jj < p.G; jj += kThreads1) {
    int nv = 0;
    if (j0 + jj < p.Tq) {
      const int t = p.q_pos[static_cast<long long>(b) * p.Tq + j0 + jj];
      nv = t >= 0 ? (t + 1) / p.m : 0;
      nv = nv < p.N ? nv : p.N;
    }
    nvis_s[jj] = nv;
  }
  for (int i = tid; i < p.G * HI; i += kThreads1) {
    const int jj = i / HI, h = i % HI;
    const long long qrow = static_cast<long long>(b) * p.Tq + j0 + jj;
    float wv = p.w_stride == 0 ? p.w[h] : (j0 + jj < p.Tq ? p.w[qrow * p.w_stride + h] : 0.f);
    if (F8) wv = j0 + jj < p.Tq ? wv * p.q_scale[qrow * HI + h] : 0.f;
    w_s[i] = wv;
  }
  if (p.hist)
    for (int i = tid; i < kTopkBins; i += kThreads1) hist_s[i] = 0u;
  __syncthreads();
  if (tid == 0)
    for (int i = 1; i < n_pre; ++i) issue_tile(i, i);  // the rest of the first ring
  int nv_max = 0;
  for (int jj = 0; jj < p.G; ++jj) nv_max = max(nv_max, nvis_s[jj]);
  const int tiles_vis = (nv_max + kTileKeys - 1) / kTileKeys;
  const int tile_hi = min(tile_cap, tiles_vis);
  const int ntile = tile_hi - tile_lo;
  if (ntile <= 0) {
    // uniform: nothing visible in this range; the copies requested at the
    // start land before the CTA exits
    if (tid == 0) {
      for (int s = 0; s < n_pre; ++s) mbar_wait(&bars->full[s], 0, kDrainBudget, nullptr);
      mbar_wait(&bars->qfull, 0, kDrainBudget, nullptr);
    }
    return;
  }

  if (warp == 1) {
    tmem_alloc(&tmem_base, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  volatile int* abort_v = &abort_flag;
  auto fail = [&]() {
    if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
    *abort_v = 1;
  };

  if (warp == 0) {
    if (lane == 0) {
      int issued = n_pre;
      for (int i = n_pre; i < ntile; ++i) {
        const int s = i % p.stages;
        const uint32_t ph = (i / p.stages) & 1;
        if (!mbar_wait(&bars->empty[s], ph ^ 1, p.budget, abort_v) ||
            (F8 && !mbar_wait(&bars->sfree[s], ph ^ 1, p.budget, abort_v))) {
          fail();
          break;
        }
        issue_tile(i, s);
        issued = i + 1;
      }
      // drain: every issued copy has landed before the CTA may exit
      for (int s = 0; s < p.stages && s < issued; ++s) {
        const int last = issued - 1 - ((issued - 1 - s) % p.stages);
        mbar_wait(&bars->full[s], (last / p.stages) & 1, kDrainBudget, nullptr);
      }
      mbar_wait(&bars->qfull, 0, kDrainBudget, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = F8 ? idesc_e4m3_f32(128, p.NC) : idesc_bf16_f32(128, p.NC);
      int issued = 0;
      if (mbar_wait(&bars->qfull, 0, p.budget, abort_v)) {
        for (int i = 0; i < ntile; ++i) {
          const int s = i % p.stages;
          const uint32_t ph = (i / p.stages) & 1;
          const int acc = i & ((1 << acc_sh) - 1);
          const uint32_t aph = (i >> acc_sh) & 1;
          if (!mbar_wait(&bars->tempty[acc], aph ^ 1, p.budget, abort_v) ||
              !mbar_wait(&bars->full[s], ph, p.budget, abort_v)) {
            fail();
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
          issued = i + 1;
        }
      } else {
        fail();
      }
      // drain: the last MMAs have finished reading shared memory / writing TMEM
      if (issued > 0) {
        const int i = issued - 1;
        mbar_wait(&bars->tfull[i & ((1 << acc_sh) - 1)], (i >> acc_sh) & 1, kDrainBudget, nullptr);
      }
    }
  } else {
    // ---- epilogue warps 2..9: TMEM lane quarter = warp % 4; group e handles
    // the tiles i = e (mod 2), whose accumulators (i mod 2 or i mod 4) only
    // this group reads
    const int quarter = warp & 3;
    const int egroup = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    const long long srow0 = static_cast<long long>(b) * p.Tq + j0;
    for (int i = egroup; i < ntile; i += kEpiGroups) {
      const int acc = i & ((1 << acc_sh) - 1);
      const uint32_t aph = (i >> acc_sh) & 1;
      const uint32_t col0 = lane_addr + static_cast<uint32_t>(acc * p.NC);
      const int st = i % p.stages;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->tfull[acc], aph, p.budget, abort_v));
      float kscale = 1.f;
      if (F8 && ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[st], (i / p.stages) & 1, p.budget, abort_v));
        if (ok) kscale = ksc[st * kTileKeys + row];
      }
      if (F8) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->sfree[st]);
      }
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int key = (tile_lo + i) * kTileKeys + row;
      bool released = false;
      if constexpr (HI >= 16) {
        for (int jj = 0; jj < p.G; ++jj) {
          uint32_t rr[HI / 16][16];
#pragma unroll
          for (int hc = 0; hc < HI / 16; ++hc) tmem_ld16(col0 + jj * HI + hc * 16, rr[hc]);
          tmem_ld_wait();
          if (!F8 && p.G == 1) {
            // one query: its columns are in registers, the accumulator is
            // released before the reduction (measured with bf16 keys; the
            // E4M3 kernel keeps four accumulators instead)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[acc]);
            released = true;
          }
          const float* wq = w_s + jj * HI;
          float sum = 0.f;
#pragma unroll
          for (int hc = 0; hc < HI / 16; ++hc)
#pragma unroll
            for (int e = 0; e < 16; ++e) sum = fmaf(wq[hc * 16 + e], fmaxf(__uint_as_float(rr[hc][e]), 0.f), sum);
          if (F8) sum *= kscale;
          const bool vis = key < nvis_s[jj];
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
            const float* wq = w_s + (jj < p.G ? jj : 0) * HI;
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < HI; ++e) sum = fmaf(wq[e], fmaxf(__uint_as_float(rr[qq * HI + e]), 0.f), sum);
            if (jj < p.G && key < nvis_s[jj]) p.S[(srow0 + jj) * p.ld + key] = sum;
          }
        }
      }
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tempty[acc]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, p.tmem_cols);
  }
  if (p.after_zero) asm volatile("griddepcontrol.wait;" ::: "memory");  // the histogram is zeroed
  if (p.hist) {
    uint32_t* g = p.hist + (static_cast<long long>(b) * p.Tq + j0) * kTopkBins;
    for (int i = tid; i < kTopkBins; i += kThreads1)
      if (hist_s[i]) atomicAdd(g + i, hist_s[i]);
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
  // TMEM columns: two accumulators, four in the one-item kernel on E4M3 keys
  // when they fit in the 512 columns (NC = G * H_I rounded up: up to 256)
  const bool single = (a.Tq + p.G - 1) / p.G == 1;
  p.acc_shift = single && F8 && 4 * p.NC <= 512 ? 2 : 1;
  int cols = 32;
  while (cols < (1 << p.acc_shift) * p.NC) cols *= 2;
  if (cols > 512) return cudaErrorNotSupported;
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
  // tile ranges per group: one item per SM when the groups alone cannot fill the GPU
  int ipg = static_cast<int>(n_sm / (groups > 0 ? groups : 1));
  ipg = ipg < 1 ? 1 : (ipg > n_tiles_all ? n_tiles_all : ipg);
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
  if (p.n_groups == 1) {
    // decode (one query group per sequence): one item per CTA
    cudaError_t e = ensure_dyn_smem<indexer_single_kernel<HI, F8>>(static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(indexer_single_kernel<HI, F8>, dim3(static_cast<unsigned>(items)), dim3(kThreads1), smem, s, 1,
                    tmk, tmq, tms, p);
  }
  cudaError_t e = ensure_dyn_smem<indexer_kernel<HI, F8>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_k(indexer_kernel<HI, F8>, dim3(static_cast<unsigned>(grid)), dim3(threads_p<HI>()), smem, s, 1, tmk, tmq,
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
