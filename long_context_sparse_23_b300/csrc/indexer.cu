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

constexpr int kEpiGroups = 2;                       // epilogue warp groups, alternating tiles
constexpr int kThreads = 64 + 128 * kEpiGroups;    // producer, MMA, epilogue warps
constexpr int kTileKeys = 128;
constexpr int kHalfBytes = kTileKeys * 128;  // one 64-wide K half of a key tile
constexpr int kSmemBudget = 220 * 1024;
constexpr long long kDrainBudget = 1LL << 31;

struct KParams {
  const float* w;
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
  int tmem_cols;
  uint32_t* errw;
  long long budget;
  uint32_t* hist;  // [B*Tq][kTopkBins] (G == 1 only), or nullptr
  int after_zero;  // see IndexerArgs::after_zero
};

struct __align__(8) Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t qfull;
};

template <int HI>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
                   KParams p) {
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
  Bars* bars = reinterpret_cast<Bars*>(ks + p.stages * p.kh * kHalfBytes);
  // top-k bucket histogram of this CTA's scores (one query per group)
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(bars) + sizeof(Bars));
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float w_s[HI];
  __shared__ int nvis_s[256];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which (sequence, query group, tile range) this CTA owns; heavy first
  const int item = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);
  const int grp = item / p.items_per_group;
  const int sub = item % p.items_per_group;
  const int b = grp / p.n_groups;
  const int j0 = (grp % p.n_groups) * p.G;
  const int n_tiles_all = (p.N + kTileKeys - 1) / kTileKeys;

  for (int jj = tid; jj < p.G; jj += kThreads) {
    int nv = 0;
    if (j0 + jj < p.Tq) {
      const int t = p.q_pos[static_cast<long long>(b) * p.Tq + j0 + jj];
      nv = t >= 0 ? (t + 1) / p.m : 0;
      nv = nv < p.N ? nv : p.N;
    }
    nvis_s[jj] = nv;
  }
  for (int h = tid; h < HI; h += kThreads) w_s[h] = p.w[h];
  if (p.hist)
    for (int i = tid; i < kTopkBins; i += kThreads) hist_s[i] = 0u;
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 4);
    }
    mbar_init(&bars->qfull, 1);
    mbar_fence_init();
  }
  __syncthreads();
  int nv_max = 0;
  for (int jj = 0; jj < p.G; ++jj) nv_max = max(nv_max, nvis_s[jj]);
  const int tiles_vis = (nv_max + kTileKeys - 1) / kTileKeys;
  const int tile_lo = sub * p.tiles_per_item;
  const int tile_hi = min(min(tile_lo + p.tiles_per_item, n_tiles_all), tiles_vis);
  const int ntile = tile_hi - tile_lo;
  if (ntile <= 0) return;  // uniform: nothing visible in this range

  if (warp == 1) {
    tmem_alloc(&tmem_base, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  volatile int* abort_v = &abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmq);
      const int qrow = (b * p.Tq + j0) * HI;
      // the keys are read once: evict-first, so the scores this kernel writes
      // stay in L2 for the top-k that reads them next
      const uint64_t key_policy = l2_policy_evict_first();
      mbar_expect_tx(&bars->qfull, p.kh * p.NC * 128);
      for (int h = 0; h < p.kh; ++h) tma_load_2d(qs + h * p.NC * 128, &tmq, &bars->qfull, h * 64, qrow);
      int issued = 0;
      for (int i = 0; i < ntile; ++i) {
        const int s = i % p.stages;
        const uint32_t ph = (i / p.stages) & 1;
        if (!mbar_wait(&bars->empty[s], ph ^ 1, p.budget, abort_v)) {
          if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
          *abort_v = 1;
          break;
        }
        mbar_expect_tx(&bars->full[s], p.kh * kHalfBytes);
        char* dst = ks + s * p.kh * kHalfBytes;
        for (int h = 0; h < p.kh; ++h)
          tma_load_3d_hint(dst + h * kHalfBytes, &tmk, &bars->full[s], h * 64, (tile_lo + i) * kTileKeys, b,
                           key_policy);
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
      const uint32_t idesc = idesc_bf16_f32(128, p.NC);
      int issued = 0;
      if (mbar_wait(&bars->qfull, 0, p.budget, abort_v)) {
        for (int i = 0; i < ntile; ++i) {
          const int s = i % p.stages;
          const uint32_t ph = (i / p.stages) & 1;
          const int acc = i & 1;
          const uint32_t aph = (i >> 1) & 1;
          if (!mbar_wait(&bars->tempty[acc], aph ^ 1, p.budget, abort_v) ||
              !mbar_wait(&bars->full[s], ph, p.budget, abort_v)) {
            if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
            *abort_v = 1;
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
            umma_f16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars->empty[s]);
          umma_commit(&bars->tfull[acc]);
          issued = i + 1;
        }
      } else {
        if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
        *abort_v = 1;
      }
      // drain: the last MMAs have finished reading shared memory / writing TMEM
      if (issued > 0) {
        const int i = issued - 1;
        mbar_wait(&bars->tfull[i & 1], (i >> 1) & 1, kDrainBudget, nullptr);
      }
    }
  } else {
    // ---- epilogue warps 2..: TMEM lane quarter = warp % 4; group e handles
    // the tiles i = e (mod kEpiGroups), i.e. TMEM accumulator buffer e
    const int quarter = warp & 3;
    const int egroup = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tbase + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int i = egroup; i < ntile; i += kEpiGroups) {
      const int acc = i & 1;
      const uint32_t aph = (i >> 1) & 1;
      if (!mbar_wait(&bars->tfull[acc], aph, p.budget, abort_v)) {
        if (!*abort_v) raise_flag(p.errw, kFlagTimeout);
        *abort_v = 1;
        break;
      }
      tc_fence_after();
      const int key = (tile_lo + i) * kTileKeys + row;
      const uint32_t col0 = lane_addr + static_cast<uint32_t>(acc * p.NC);
      if constexpr (HI >= 16) {
        for (int jj = 0; jj < p.G; ++jj) {
          // all of the query's head columns in flight at once, one wait
          uint32_t r[HI / 16][16];
#pragma unroll
          for (int hc = 0; hc < HI / 16; ++hc) tmem_ld16(col0 + jj * HI + hc * 16, r[hc]);
          tmem_ld_wait();
          float sum = 0.f;
#pragma unroll
          for (int hc = 0; hc < HI / 16; ++hc)
#pragma unroll
            for (int e = 0; e < 16; ++e) sum = fmaf(w_s[hc * 16 + e], fmaxf(__uint_as_float(r[hc][e]), 0.f), sum);
          const bool vis = key < nvis_s[jj];
          if (vis) p.S[(static_cast<long long>(b) * p.Tq + j0 + jj) * p.ld + key] = sum;
          if (p.hist) {
            // bucket = top 12 bits of the order-preserving key of sum (sum >= 0 unless w < 0)
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
          uint32_t r[16];
          tmem_ld16(col0 + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int qq = 0; qq < QPC; ++qq) {
            const int jj = c0 / HI + qq;
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < HI; ++e) sum = fmaf(w_s[e], fmaxf(__uint_as_float(r[qq * HI + e]), 0.f), sum);
            if (jj < p.G && key < nvis_s[jj])
              p.S[(static_cast<long long>(b) * p.Tq + j0 + jj) * p.ld + key] = sum;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[acc]);
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
    for (int i = tid; i < kTopkBins; i += kThreads)
      if (hist_s[i]) atomicAdd(g + i, hist_s[i]);
  }
}

template <int HI>
cudaError_t launch_hi(const IndexerArgs& a, cudaStream_t s) {
  KParams p;
  p.w = a.w;
  p.q_pos = a.q_pos;
  p.S = a.scores;
  p.ld = a.ld;
  p.B = a.B;
  p.Tq = a.Tq;
  p.N = a.N;
  p.m = a.m;
  p.G = a.Tq < 256 / HI ? a.Tq : 256 / HI;
  p.NC = ((p.G * HI + 15) / 16) * 16;
  p.kh = (a.d_I + 63) / 64;
  p.n_groups = (a.Tq + p.G - 1) / p.G;
  int cols = 32;
  while (cols < 2 * p.NC) cols *= 2;
  p.tmem_cols = cols;
  const int q_bytes = p.kh * p.NC * 128;
  const int stage_bytes = p.kh * kHalfBytes;
  const int hist_bytes = (a.hist != nullptr && p.G == 1 && HI >= 16) ? kTopkBins * 4 : 0;
  int stages = (kSmemBudget - 1024 - q_bytes - static_cast<int>(sizeof(Bars)) - hist_bytes) / stage_bytes;
  stages = stages > 8 ? 8 : stages;
  if (stages < 2) return cudaErrorNotSupported;
  p.stages = stages;
  const int n_tiles_all = (a.N + kTileKeys - 1) / kTileKeys;
  const long long groups = static_cast<long long>(a.B) * p.n_groups;
  // one wave of one CTA per SM when the groups alone cannot fill the GPU
  int ipg = static_cast<int>(148 / (groups > 0 ? groups : 1));
  ipg = ipg < 1 ? 1 : (ipg > n_tiles_all ? n_tiles_all : ipg);
  p.tiles_per_item = (n_tiles_all + ipg - 1) / ipg;
  p.items_per_group = (n_tiles_all + p.tiles_per_item - 1) / p.tiles_per_item;
  p.errw = a.errw;
  p.budget = a.budget;
  p.hist = (a.hist != nullptr && p.G == 1 && HI >= 16) ? a.hist : nullptr;
  p.after_zero = p.hist != nullptr && a.after_zero;
  const long long items = groups * p.items_per_group;
  if (items == 0 || n_tiles_all == 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorNotSupported;

  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmk, tmq;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.d_I), static_cast<cuuint64_t>(a.N),
                          static_cast<cuuint64_t>(a.B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.d_I) * 2,
                             static_cast<cuuint64_t>(a.N) * a.d_I * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTileKeys), 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tmk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.k_idx), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.d_I),
                          static_cast<cuuint64_t>(a.B) * a.Tq * HI};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.d_I) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(p.NC)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.q_idx), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const size_t smem = 1024 + q_bytes + static_cast<size_t>(stages) * stage_bytes + sizeof(Bars) + hist_bytes;
  cudaError_t e = ensure_dyn_smem<indexer_kernel<HI>>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_k(indexer_kernel<HI>, dim3(static_cast<unsigned>(items)), dim3(kThreads), smem, s, 1, tmk, tmq,
                  p);
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

cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s) {
  switch (a.H_I) {
    case 4: return launch_hi<4>(a, s);
    case 8: return launch_hi<8>(a, s);
    case 16: return launch_hi<16>(a, s);
    case 32: return launch_hi<32>(a, s);
    case 64: return launch_hi<64>(a, s);
    case 128: return launch_hi<128>(a, s);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace csa
