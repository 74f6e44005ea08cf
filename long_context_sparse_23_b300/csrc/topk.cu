// (3) Top-k selection.  "DeepSeek V4 technical review", section 2.1: every
// query keeps the top-k (k = 1024) compressed blocks by indexer score.  Among
// the n_vis visible scores the min(k, n_vis) largest are kept, equal scores
// going to the lower block index; indices are written in ascending order and
// padded with -1.
//
// Design: exact integer radix selection.  Each fp32 score becomes an
// order-preserving 32-bit key (-0 folded onto +0).  One thread-block cluster
// of C CTAs (C = 1..16) owns one query; CTA r stages the contiguous index
// range [r*chunk, (r+1)*chunk) of that query's scores in its shared memory
// once, so the row is read from global memory exactly once.  Up to four 8-bit
// digit passes (most significant first) build a 256-bin histogram of the keys
// still matching the selected prefix; the CTAs add their histograms into rank
// 0's copy through distributed shared memory, rank 0 picks the digit where
// the running count from the top reaches the remaining k, and broadcasts the
// extended prefix.  The result is a (prefix, mask, k_rem) rule: keys above the
// prefix are kept, and of the keys equal to it the k_rem with the lowest
// indices.  A final warp-ballot compaction in index order, with the CTAs'
// counts exchanged through rank 0, writes the output.  Counting uses integer
// shared-memory atomics only, so the result is exact and deterministic.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kMaxChunk = 49152;  // keys per CTA held in shared memory (192 KB)

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

struct Ctl {
  uint32_t prefix;
  uint32_t mask;
  int k_rem;
  int done;
};

// Inclusive scan of one value per thread over threads 0..255 (others pass 0).
__device__ __forceinline__ uint32_t scan256(uint32_t v, uint32_t* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31 && warp < 8) tmp[warp] = v;
  __syncthreads();
  uint32_t add = 0;
  if (warp < 8)
    for (int w = 0; w < warp; ++w) add += tmp[w];
  __syncthreads();
  return v + add;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a, int chunk) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const long long qi = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t ghist[256];
  __shared__ Ctl ctl;
  __shared__ uint32_t tmp[32];
  __shared__ uint32_t wcnt[2][kWarps];
  __shared__ uint32_t rcnt[2][kMaxCluster];

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
  if (tid == 0) ctl = Ctl{0u, 0u, a.k, 0};
  if (tid < 256) ghist[tid] = 0u;
  cluster.sync();

  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
    // read the rule before any thread can overwrite it below
    const uint32_t prefix = ctl.prefix, mask = ctl.mask;
    const uint32_t krem = static_cast<uint32_t>(ctl.k_rem);
    for (int base = 0; base < cnt; base += kThreads) {
      const int i = base + tid;
      const uint32_t key = i < cnt ? keys[i] : 0u;
      const bool match = i < cnt && (key & mask) == prefix;
      const uint32_t digit = (key >> shift) & 255u;
      const unsigned am = __ballot_sync(0xffffffffu, match);
      if (match) {
        const unsigned peers = __match_any_sync(am, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
      }
    }
    __syncthreads();
    uint32_t* H = hist;
    if (C > 1) {
      if (tid < 256 && hist[tid]) atomicAdd(cluster.map_shared_rank(&ghist[tid], 0), hist[tid]);
      cluster.sync();
      H = ghist;
    }
    if (rank == 0) {
      // bins in descending digit order; find the digit holding the k_rem-th key
      const uint32_t v = tid < 256 ? H[255 - tid] : 0u;
      const uint32_t incl = scan256(v, tmp);
      const uint32_t excl = incl - v;
      if (tid < 256 && excl < krem && krem <= incl) {
        const uint32_t digit = 255u - tid;
        Ctl nc;
        nc.prefix = prefix | (digit << shift);
        nc.mask = mask | (255u << shift);
        nc.k_rem = static_cast<int>(krem - excl);
        nc.done = (v == krem - excl) || shift == 0;
        for (int r = 0; r < C; ++r) *cluster.map_shared_rank(&ctl, r) = nc;
      }
      if (C > 1) {
        __syncthreads();
        if (tid < 256) ghist[tid] = 0u;
      }
    }
    cluster.sync();
    if (ctl.done) break;
  }

  // ---- compaction in index order -------------------------------------------
  const uint32_t prefix = ctl.prefix, mask = ctl.mask;
  const int krem = ctl.k_rem;
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
  if (C > 1) {
    if (tid == 0) {
      *cluster.map_shared_rank(&rcnt[0][rank], 0) = cta_gt;
      *cluster.map_shared_rank(&rcnt[1][rank], 0) = cta_eq;
    }
    cluster.sync();
    for (int r = 0; r < rank; ++r) {
      run_gt += *cluster.map_shared_rank(&rcnt[0][r], 0);
      run_eq += *cluster.map_shared_rank(&rcnt[1][r], 0);
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
    if (gt || (eq && eq_before < static_cast<uint32_t>(krem))) {
      const uint32_t pos = gt_before + min(eq_before, static_cast<uint32_t>(krem));
      out[pos] = lo + i;
      if (sout) sout[pos] = key_score(full);
    }
    run_gt += __popc(bgt);
    run_eq += __popc(beq);
  }
  cluster.sync();  // rank 0's counters stay alive until every CTA has read them
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
      lc.dynamicSmemBytes = 16384 * 4;
      lc.attrs = at;
      lc.numAttrs = 1;
      int nclusters = 0;
      cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxChunk * 4);
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
  const size_t smem = static_cast<size_t>(chunk > 0 ? chunk : 32) * 4;
  // (the cluster-size attribute was set once by max_cluster_for_device)
  cudaError_t e = ensure_dyn_smem<topk_kernel>(kMaxChunk * 4);
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
  return cudaLaunchKernelEx(&lc, topk_kernel, a, chunk);
}

}  // namespace csa
