// (3) Top-k selection.  "DeepSeek V4 technical review", section 2.1: every
// query keeps the top-k (k = 1024) compressed blocks by indexer score.  Among
// the n_vis visible scores the min(k, n_vis) largest are kept, equal scores
// going to the lower block index; indices are written in ascending order and
// padded with -1.
//
// Design: exact integer selection on order-preserving 32-bit keys (-0 folded
// onto +0).  One thread-block cluster of C CTAs (C = 1..16) owns one query;
// CTA r stages the contiguous index range [r*chunk, (r+1)*chunk) of the
// query's scores in its shared memory once.  The selection ends in a rule
// (prefix, mask, k_rem): keys whose masked bits exceed the prefix are kept,
// and of the keys equal to it the k_rem with the lowest indices.  A final
// warp-ballot compaction in index order writes the output; the CTAs' counts
// give each CTA its output offset.
//
// Two ways to find the rule:
//  * bucket path (long rows, C > 1): one 4096-bin histogram of the keys' top
//    12 bits, merged into rank 0 through distributed shared memory, names the
//    bucket holding the k-th key; only that bucket's keys (typically ~1k of
//    262k) travel to rank 0, which finishes the selection on them alone.
//    Four cluster barriers in total.
//  * digit path (short rows, or a bucket too full to gather): up to four
//    8-bit digit passes over all keys, histograms merged through rank 0.
// Counting uses integer shared-memory atomics only: exact and deterministic.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kMaxChunk = 40960;  // keys per CTA held in shared memory
constexpr int kBins = 4096;       // 12-bit buckets
constexpr int kCandCap = 4096;    // bucket keys gathered at rank 0
constexpr int kBucketBytes = 3 * kBins * 4 + kCandCap;  // local + merged histogram, keys, ranks

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

struct Rule {
  uint32_t prefix;
  uint32_t mask;
  int k_rem;
  int done;
};

struct BucketCtl {
  int beta;    // bucket holding the k-th largest key
  int above;   // keys in buckets above it
  int hb;      // keys in the bucket
  int pre_gt;  // keys kept above the rule in lower-ranked CTAs
  int pre_eq;  // keys equal to the rule in lower-ranked CTAs
  Rule rule;
};

// Warp-aggregated histogram increment (lanes with the same bin add once).
__device__ __forceinline__ void hist_add(uint32_t* hist, bool active, uint32_t bin) {
  const unsigned am = __ballot_sync(0xffffffffu, active);
  if (active) {
    const unsigned peers = __match_any_sync(am, bin);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
  }
}

// Inclusive scan of one value per thread over the whole block.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  uint32_t add = 0;
  for (int w = 0; w < warp; ++w) add += tmp[w];
  __syncthreads();
  return v + add;
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) tmp[warp] = v;
  __syncthreads();
  uint32_t s = 0;
  for (int w = 0; w < kWarps; ++w) s += tmp[w];
  __syncthreads();
  return s;
}

// Given a 256-bin histogram H of the digit at ``shift`` among the keys that
// match r, extend r by the digit holding the r.k_rem-th largest key.  The
// deciding thread writes the new rule to *dst in every CTA of the cluster
// (C = 1: its own copy).  All threads of the block call it.
__device__ __forceinline__ void pick_digit(const uint32_t* H, const Rule r, int shift, uint32_t* tmp,
                                           cg::cluster_group& cluster, int C, Rule* dst) {
  const int tid = threadIdx.x;
  const uint32_t v = tid < 256 ? H[255 - tid] : 0u;
  const uint32_t incl = block_scan(v, tmp);
  const uint32_t excl = incl - v;
  const uint32_t krem = static_cast<uint32_t>(r.k_rem);
  if (tid < 256 && excl < krem && krem <= incl) {
    const uint32_t digit = 255u - tid;
    Rule nr;
    nr.prefix = r.prefix | (digit << shift);
    nr.mask = r.mask | (255u << shift);
    nr.k_rem = static_cast<int>(krem - excl);
    nr.done = (v == krem - excl) || shift == 0;
    for (int q = 0; q < C; ++q) *cluster.map_shared_rank(dst, q) = nr;
  }
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a, int chunk, int bucket_path) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const long long qi = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(16) uint32_t dyn[];
  uint32_t* keys = dyn;             // [chunk]
  uint32_t* lhist = dyn + chunk;    // bucket path: [kBins]
  uint32_t* ghist = lhist + kBins;  // bucket path, rank 0: merged [kBins]
  uint32_t* cand = ghist + kBins;   // bucket path, rank 0: [kCandCap]
  uint8_t* cand_rank = reinterpret_cast<uint8_t*>(cand + kCandCap);
  __shared__ uint32_t hist[256];
  __shared__ uint32_t ghist8[256];
  __shared__ Rule rule;
  __shared__ BucketCtl bc;
  __shared__ uint32_t tmp[32];
  __shared__ uint32_t wcnt[2][kWarps];
  __shared__ uint32_t rcnt[2][kMaxCluster];
  __shared__ uint32_t cand_n;

  const int t = a.q_pos[qi];
  int n_vis = t >= 0 ? (t + 1) / a.m : 0;
  n_vis = n_vis < a.N ? n_vis : a.N;
  int32_t* out = a.idx_out + qi * a.k;
  float* sout = a.score_out ? a.score_out + qi * a.k : nullptr;
  const float* row = a.scores + qi * a.ld;

  if (n_vis <= a.k) {
    // every visible block is kept; index order == output order
    for (int p = rank * kThreads + tid; p < a.k; p += C * kThreads) {
      out[p] = p < n_vis ? p : -1;
      if (sout) sout[p] = p < n_vis ? row[p] : 0.f;
    }
    return;  // uniform over the cluster: no shared memory of another CTA is touched
  }

  const int lo = rank * chunk;
  const int cnt = max(0, min(lo + chunk, n_vis) - lo);
  for (int i = tid; i < cnt; i += kThreads) keys[i] = score_key(row[lo + i]);
  if (tid == 0) {
    rule = Rule{0u, 0u, a.k, 0};
    cand_n = 0;
  }
  if (tid < 256) ghist8[tid] = 0u;

  bool have_offsets = false;
  uint32_t pre_gt = 0, pre_eq = 0;
  bool bucket_ok = false;

  if (bucket_path) {
    for (int i = tid; i < kBins; i += kThreads) {
      lhist[i] = 0u;
      ghist[i] = 0u;
    }
    __syncthreads();
    for (int base = 0; base < cnt; base += kThreads) {
      const int i = base + tid;
      const uint32_t key = i < cnt ? keys[i] : 0u;
      hist_add(lhist, i < cnt, key >> 20);
    }
    cluster.sync();  // every local histogram done, rank 0's merged one zeroed
    for (int i = tid; i < kBins; i += kThreads)
      if (lhist[i]) atomicAdd(cluster.map_shared_rank(&ghist[i], 0), lhist[i]);
    cluster.sync();
    if (rank == 0) {
      // thread t owns buckets 4095-8t down to 4088-8t (descending order)
      uint32_t v = 0;
      const int top = kBins - 1 - 8 * tid;
#pragma unroll
      for (int j = 0; j < 8; ++j) v += ghist[top - j];
      const uint32_t incl = block_scan(v, tmp);
      uint32_t c = incl - v;
      const uint32_t k = static_cast<uint32_t>(a.k);
      if (c < k && k <= incl) {
        for (int j = 0; j < 8; ++j) {
          const uint32_t h = ghist[top - j];
          if (c + h >= k) {
            BucketCtl x;
            x.beta = top - j;
            x.above = static_cast<int>(c);
            x.hb = static_cast<int>(h);
            x.pre_gt = x.pre_eq = 0;
            x.rule = Rule{0u, 0u, 0, 0};
            for (int q = 0; q < C; ++q) *cluster.map_shared_rank(&bc, q) = x;
            break;
          }
          c += h;
        }
      }
    }
    cluster.sync();
    bucket_ok = bc.hb <= kCandCap;  // uniform over the cluster
    if (bucket_ok) {
      // keys above the bucket are kept; the bucket's keys go to rank 0
      const uint32_t beta = static_cast<uint32_t>(bc.beta);
      const unsigned lt = lanemask_lt();
      uint32_t n_above = 0;
      for (int base = 0; base < cnt; base += kThreads) {
        const int i = base + tid;
        const uint32_t key = i < cnt ? keys[i] : 0u;
        const uint32_t bin = key >> 20;
        n_above += (i < cnt && bin > beta) ? 1u : 0u;
        const bool eq = i < cnt && bin == beta;
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        if (beq) {
          uint32_t slot = 0;
          if (lane == __ffs(beq) - 1) slot = atomicAdd(cluster.map_shared_rank(&cand_n, 0), __popc(beq));
          slot = __shfl_sync(0xffffffffu, slot, __ffs(beq) - 1);
          if (eq) {
            const uint32_t pos = slot + __popc(beq & lt);
            *cluster.map_shared_rank(&cand[pos], 0) = key;
            *cluster.map_shared_rank(&cand_rank[pos], 0) = static_cast<uint8_t>(rank);
          }
        }
      }
      n_above = block_sum(n_above, tmp);
      if (tid == 0) *cluster.map_shared_rank(&rcnt[0][rank], 0) = n_above;
      cluster.sync();
      if (rank == 0) {
        // finish the selection among the bucket's keys
        const int n = static_cast<int>(cand_n);
        Rule r{static_cast<uint32_t>(bc.beta) << 20, 0xFFF00000u, a.k - bc.above, 0};
        if (r.k_rem == n) r.done = 1;
        const int shifts[3] = {12, 4, 0};
        for (int ps = 0; ps < 3 && !r.done; ++ps) {
          if (tid < 256) hist[tid] = 0u;
          __syncthreads();
          for (int base = 0; base < n; base += kThreads) {
            const int i = base + tid;
            const uint32_t key = i < n ? cand[i] : 0u;
            hist_add(hist, i < n && (key & r.mask) == r.prefix, (key >> shifts[ps]) & 255u);
          }
          __syncthreads();
          pick_digit(hist, r, shifts[ps], tmp, cluster, 1, &rule);
          __syncthreads();
          r = rule;
          __syncthreads();
        }
        // per-rank counts of bucket keys above / equal to the rule
        if (tid < kMaxCluster) {
          wcnt[0][tid] = 0u;
          wcnt[1][tid] = 0u;
        }
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t key = cand[i] & r.mask;
          if (key > r.prefix)
            atomicAdd(&wcnt[0][cand_rank[i]], 1u);
          else if (key == r.prefix)
            atomicAdd(&wcnt[1][cand_rank[i]], 1u);
        }
        __syncthreads();
        if (tid == 0) {
          uint32_t g = 0, e = 0;
          for (int q = 0; q < C; ++q) {
            BucketCtl x = bc;
            x.rule = r;
            x.pre_gt = static_cast<int>(g);
            x.pre_eq = static_cast<int>(e);
            *cluster.map_shared_rank(&bc, q) = x;
            g += rcnt[0][q] + wcnt[0][q];
            e += wcnt[1][q];
          }
        }
      }
      cluster.sync();
      if (tid == 0) rule = bc.rule;
      pre_gt = static_cast<uint32_t>(bc.pre_gt);
      pre_eq = static_cast<uint32_t>(bc.pre_eq);
      have_offsets = true;
      __syncthreads();
    }
  }

  if (!bucket_ok) {
    // digit path over all keys
    __syncthreads();
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (tid < 256) hist[tid] = 0u;
      __syncthreads();
      const Rule r = rule;  // read before anyone overwrites it below
      for (int base = 0; base < cnt; base += kThreads) {
        const int i = base + tid;
        const uint32_t key = i < cnt ? keys[i] : 0u;
        hist_add(hist, i < cnt && (key & r.mask) == r.prefix, (key >> shift) & 255u);
      }
      __syncthreads();
      uint32_t* H = hist;
      if (C > 1) {
        if (tid < 256 && hist[tid]) atomicAdd(cluster.map_shared_rank(&ghist8[tid], 0), hist[tid]);
        cluster.sync();
        H = ghist8;
      }
      if (rank == 0) {
        pick_digit(H, r, shift, tmp, cluster, C, &rule);
        if (C > 1) {
          __syncthreads();
          if (tid < 256) ghist8[tid] = 0u;
        }
      }
      cluster.sync();
      if (rule.done) break;
    }
  }

  // ---- compaction in index order -------------------------------------------
  const uint32_t prefix = rule.prefix, mask = rule.mask;
  const uint32_t krem = static_cast<uint32_t>(rule.k_rem);
  const int seg = ((cnt + kWarps - 1) / kWarps + 31) & ~31;
  const int s_lo = min(cnt, warp * seg), s_hi = min(cnt, s_lo + seg);
  uint32_t ngt = 0, neq = 0;
  for (int base = s_lo; base < s_hi; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < s_hi ? keys[i] & mask : 0u;
    ngt += __popc(__ballot_sync(0xffffffffu, i < s_hi && key > prefix));
    neq += __popc(__ballot_sync(0xffffffffu, i < s_hi && key == prefix));
  }
  if (lane == 0) {
    wcnt[0][warp] = ngt;
    wcnt[1][warp] = neq;
  }
  __syncthreads();
  uint32_t run_gt = 0, run_eq = 0, cta_gt = 0, cta_eq = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) {
      run_gt += wcnt[0][w];
      run_eq += wcnt[1][w];
    }
    cta_gt += wcnt[0][w];
    cta_eq += wcnt[1][w];
  }
  if (have_offsets) {
    run_gt += pre_gt;
    run_eq += pre_eq;
  } else if (C > 1) {
    if (tid == 0) {
      *cluster.map_shared_rank(&rcnt[0][rank], 0) = cta_gt;
      *cluster.map_shared_rank(&rcnt[1][rank], 0) = cta_eq;
    }
    cluster.sync();
    for (int q = 0; q < rank; ++q) {
      run_gt += *cluster.map_shared_rank(&rcnt[0][q], 0);
      run_eq += *cluster.map_shared_rank(&rcnt[1][q], 0);
    }
  }
  const unsigned lt = lanemask_lt();
  for (int base = s_lo; base < s_hi; base += 32) {
    const int i = base + lane;
    const uint32_t full = i < s_hi ? keys[i] : 0u;
    const uint32_t key = full & mask;
    const bool gt = i < s_hi && key > prefix;
    const bool eq = i < s_hi && key == prefix;
    const unsigned bgt = __ballot_sync(0xffffffffu, gt);
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const uint32_t gt_before = run_gt + __popc(bgt & lt);
    const uint32_t eq_before = run_eq + __popc(beq & lt);
    if (gt || (eq && eq_before < krem)) {
      const uint32_t pos = gt_before + min(eq_before, krem);
      out[pos] = lo + i;
      if (sout) sout[pos] = key_score(full);
    }
    run_gt += __popc(bgt);
    run_eq += __popc(beq);
  }
  if (!have_offsets && C > 1) cluster.sync();  // rank 0's counters stay alive until read
}

struct TopkConfig {
  bool init = false;
  int max_cluster = 8;
};

int max_cluster_for_device() {
  static TopkConfig cfg[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  TopkConfig& c = cfg[dev];
  if (!c.init) {
    c.max_cluster = 8;
    ensure_dyn_smem<topk_kernel>(kMaxChunk * 4 + kBucketBytes);
    if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t lc = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 16;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      lc.gridDim = dim3(16, 1, 1);
      lc.blockDim = dim3(kThreads, 1, 1);
      lc.dynamicSmemBytes = 16384 * 4 + kBucketBytes;
      lc.attrs = at;
      lc.numAttrs = 1;
      int nclusters = 0;
      if (cudaOccupancyMaxActiveClusters(&nclusters, topk_kernel, &lc) == cudaSuccess && nclusters > 0)
        c.max_cluster = 16;
    }
    cudaGetLastError();
    c.init = true;
  }
  return c.max_cluster;
}

}  // namespace

bool topk_supported(int N) { return N <= kMaxCluster * kMaxChunk; }

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (nq == 0) return cudaSuccess;
  const int cmax = max_cluster_for_device();
  int C = 1;
  while (C < cmax && (a.N + C - 1) / C > 16384) C *= 2;
  int chunk = (a.N + C - 1) / C;
  chunk = (chunk + 31) & ~31;
  if (chunk > kMaxChunk) return cudaErrorNotSupported;
  const int bucket_path = C > 1 ? 1 : 0;
  const size_t smem = static_cast<size_t>(chunk > 0 ? chunk : 32) * 4 + (bucket_path ? kBucketBytes : 0);
  cudaError_t e = ensure_dyn_smem<topk_kernel>(kMaxChunk * 4 + kBucketBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.gridDim = dim3(C, static_cast<unsigned>(nq), 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, topk_kernel, a, chunk, bucket_path);
}

}  // namespace csa
