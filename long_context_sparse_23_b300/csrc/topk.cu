// (3) Top-k selection.  "DeepSeek V4 technical review", section 2.1: every
// query keeps the top-k (k = 1024) compressed blocks by indexer score.  Among
// the n_vis visible scores the min(k, n_vis) largest are kept, equal scores
// going to the lower block index; indices are written in ascending order and
// padded with -1.
//
// Exact integer selection on order-preserving 32-bit keys (-0 folded onto
// +0).  The selection ends in a rule (prefix, mask, k_rem): keys whose masked
// bits exceed the prefix are kept, and of the keys equal to it the k_rem with
// the lowest indices.  Counting uses integer atomics only, so the result is
// exact and does not depend on scheduling.
//
// Short rows (N <= 16384): one CTA per query stages the row's keys in shared
// memory and fixes the rule with up to four 8-bit digit passes; a warp-ballot
// compaction in index order writes the output.
//
// Mid rows (N <= 32768, e.g. decode at 128K context): the histogram below,
// then a cluster of two CTAs per query selects from it (topk_mid_kernel).
//
// Long rows (decode: few queries, up to ~10^6 keys each), three grid-wide
// steps instead of one CTA per query:
//  1. a 4096-bin histogram of every query's keys' top 12 bits, accumulated in
//     global memory (fused into the indexer's epilogue, or topk_hist_kernel
//     for given scores);
//  2. topk_select_kernel, (chunk, query) CTAs: each finds the bucket beta that
//     holds the k-th largest key from the histogram and appends every key of
//     its chunk whose bucket is >= beta (kept for sure, or undecided) to the
//     query's candidate list;
//  3. topk_finish_kernel, one CTA per query: digit passes over the candidates
//     of bucket beta fix the rule; kept candidates set bits in shared-memory
//     bitmaps over block indices, and a scan of the bitmaps writes the output
//     in index order.  When the candidates would not fit (a bucket holding
//     very many near-equal scores), the finish kernel selects from the whole
//     row in global memory instead (slower, same result).
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace cg = cooperative_groups;

namespace csa {

namespace {

constexpr int kShortThreads = 512;
constexpr int kSelThreads = 256;
constexpr int kSelPer = kTopkChunk / kSelThreads;   // keys per select thread (16)
constexpr int kFinThreads = 512;
constexpr int kFinSmemBudget = 200 * 1024;
static_assert(kSelPer == 16, "the select kernel packs four rounds of 4 keys per thread");

// n_vis <= k: every visible block is kept, in index order.
__device__ void keep_all(const TopkArgs& a, const float* row, int n_vis, int32_t* out, float* sout) {
  for (int p = threadIdx.x; p < a.k; p += blockDim.x) {
    out[p] = p < n_vis ? p : -1;
    if (sout) sout[p] = p < n_vis ? key_score(score_key(row[p])) : 0.f;
  }
}

__device__ __forceinline__ int visible(const TopkArgs& a, long long q) {
  const int t = a.q_pos[q];
  const int n = t >= 0 ? (t + 1) / a.m : 0;
  return n < a.N ? n : a.N;
}

// ---------------------------------------------------------------- short rows
__global__ void __launch_bounds__(kShortThreads) topk_short_kernel(TopkArgs a) {
  pdl_wait_then_release();
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t tmp[32];
  __shared__ uint32_t wgt[32], weq[32];
  __shared__ Rule rule;
  const long long q = blockIdx.x;
  const int n_vis = visible(a, q);
  int32_t* out = a.idx_out + q * a.k;
  float* sout = a.score_out ? a.score_out + q * a.k : nullptr;
  const float* row = a.scores + q * a.ld;
  if (n_vis <= a.k) {
    keep_all(a, row, n_vis, out, sout);
    return;
  }
  for (int i = threadIdx.x; i < n_vis; i += kShortThreads) keys[i] = score_key(row[i]);
  __syncthreads();
  const Rule r = digit_select<kShortThreads>(SmemKeys{keys}, n_vis, Rule{0u, 0u, static_cast<uint32_t>(a.k), 0u},
                                             24, hist, tmp, &rule);
  compact_row<kShortThreads>(SmemKeys{keys}, n_vis, r, out, sout, wgt, weq);
}

// ---------------------------------------------------------------- mid rows
// Rows of kTopkShortMax < N <= kTopkMidMax entries with the bucket histogram
// ready (decode at 128K context: 32768 blocks): a cluster of two CTAs per
// query instead of the select and finish passes, rank r holding the entries
// [r E, (r + 1) E), E = kTopkMidMax / 2, every step spread evenly over its
// threads:
//  1. the half row is copied to shared memory (cp.async) while the bucket
//     beta of the k-th largest key is found from the histogram;
//  2. candidates (bucket >= beta) by one float comparison per score against
//     the lowest score of bucket beta (the key map is order-preserving),
//     their indices appended to a list (warp-aggregated, any order);
//  3. per candidate: bucket above beta -> kept (bit in a bitmap over the
//     half row), bucket beta -> a second-level histogram of key bits 19..8;
//     each rank pushes its counts and second level into the other rank's
//     shared memory, and after a cluster barrier both hold the totals;
//  4. the sub-bucket holding the rest of the k-th largest, then at most one
//     8-bit pass (its histogram exchanged the same way), fix the exact rule,
//     identically in both ranks; the candidates of bucket beta set their
//     kept or tied bit;
//  5. rank 0 pushes its tie and kept counts to rank 1; thread t owns bitmap
//     word t (blocks 32t .. 32t + 31 of its half): a block scan of the words'
//     (kept, tied) counts keeps the k_rem lowest-index ties of the row and
//     gives each word's output position, and the kept indices are written in
//     ascending order.
// The candidate counts are checked against the histogram: a histogram that
// does not match the scores (an indexer that gave up, non-finite scores) or
// more candidates than a list holds (a row of near-equal scores) sends rank
// 0 to digit passes over the whole row in global memory instead, so the
// output is the exact selection of the given scores in every case.
constexpr int kMidRanks = 2;                      // CTAs per query (one cluster)
constexpr int kMidThreads = 512;
constexpr int kMidHalf = kTopkMidMax / kMidRanks;  // entries per CTA
constexpr int kMidWords = kMidHalf / 32;           // bitmap words, one per thread
constexpr int kMidList = 8192;                     // candidate indices staged per CTA
static_assert(kMidWords == kMidThreads && kMidHalf % (4 * kMidThreads) == 0, "mid rows: layout");

// dynamic shared memory of topk_mid_kernel, in 32-bit words
constexpr int kMidSmemWords = kMidHalf + 2 * kMidWords + 2 * kTopkBins + kMidList;

__global__ void __launch_bounds__(kMidThreads) topk_mid_kernel(TopkArgs a) {
  // every CTA of the cluster has started before any writes another's shared
  // memory (the wait is before the first such write)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  pdl_wait_then_release();
  extern __shared__ __align__(16) uint32_t msm[];
  float* sf = reinterpret_cast<float*>(msm);  // [kMidHalf] this half of the row's scores
  uint32_t* bm = msm + kMidHalf;              // [kMidWords] kept for sure
  uint32_t* eqm = bm + kMidWords;             // [kMidWords] equal to the rule's prefix
  uint32_t* h2 = eqm + kMidWords;             // [kTopkBins] bucket beta, key bits 19..8: this half's
  uint32_t* h2p = h2 + kTopkBins;             // [kTopkBins] ... the other half's, then both
  uint32_t* list = h2p + kTopkBins;           // [kMidList] candidate indices (in the half)
  __shared__ uint32_t h3[256], h3p[256], tmp[32], wgt[32], weq[32];
  __shared__ Rule rule;
  __shared__ Bucket sb, sb2;
  __shared__ uint32_t n_list, n_gt;
  __shared__ uint32_t peer_c, peer_g;    // the other rank's candidate and above-beta counts
  __shared__ uint32_t off_eq, off_kept;  // rank 1: rank 0's tied and kept-for-sure counts
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank()), peer = rank ^ 1;
  const long long q = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31;
  const int n_vis = visible(a, q);
  int32_t* out = a.idx_out + q * a.k;
  float* sout = a.score_out ? a.score_out + q * a.k : nullptr;
  const float* row = a.scores + q * a.ld;
  if (n_vis <= a.k) {  // both ranks (no cluster barrier follows)
    if (rank == 0) keep_all(a, row, n_vis, out, sout);
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    return;
  }
  const uint32_t k = static_cast<uint32_t>(a.k);
  const int base = rank * kMidHalf;
  const int n_loc = min(max(n_vis - base, 0), kMidHalf);  // entries of this half
  const float* rowl = row + base;
  constexpr int R = kMidHalf / (4 * kMidThreads);  // float4 rounds per thread
  // (1) the half row: whole vectors by cp.async (past it: zero-filled, never read as scores)
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = 4 * (tid + kMidThreads * r);
    cp_async16(sf + i, rowl + (i + 3 < n_loc ? i : 0), i + 3 < n_loc);
  }
  cp_async_commit();
  for (int i = tid; i < 2 * kMidWords + kTopkBins; i += kMidThreads) bm[i] = 0u;  // bm, eqm, h2
  if (tid == 0) {
    n_list = 0u;
    n_gt = 0u;
  }
  const Bucket bk = find_bucket<kMidThreads>(a.hist + q * kTopkBins, k, tmp, &sb);
  cp_async_wait<0>();
  if ((n_loc & 3) && ((n_loc >> 2) % kMidThreads) == tid) {
    const int i = n_loc & ~3;  // the partial last vector
    for (int e = 0; i + e < n_loc; ++e) sf[i + e] = rowl[i + e];
  }
  __syncthreads();
  const uint32_t beta = static_cast<uint32_t>(bk.beta);
  // lowest score of bucket beta (NaN -- nothing compares true -- when there
  // is no bucket or it holds no finite score)
  const float lo_b = bk.beta >= 0 ? key_score(beta << 20) : __uint_as_float(0x7fc00000u);
  // (2) candidates, each thread's in its own bit mask
  uint32_t mc = 0;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int i = 4 * (tid + kMidThreads * r);
    const float4 v = *reinterpret_cast<const float4*>(sf + i);
    mc |= (i < n_loc && v.x >= lo_b ? 1u : 0u) << (4 * r);
    mc |= (i + 1 < n_loc && v.y >= lo_b ? 1u : 0u) << (4 * r + 1);
    mc |= (i + 2 < n_loc && v.z >= lo_b ? 1u : 0u) << (4 * r + 2);
    mc |= (i + 3 < n_loc && v.w >= lo_b ? 1u : 0u) << (4 * r + 3);
  }
  {
    const uint32_t c = static_cast<uint32_t>(__popc(mc));
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    uint32_t b0 = 0;
    if (lane == 31) b0 = atomicAdd(&n_list, incl);
    uint32_t pos = __shfl_sync(0xffffffffu, b0, 31) + incl - c;
    while (mc) {
      const int j = __ffs(mc) - 1;
      mc &= mc - 1;
      if (pos < static_cast<uint32_t>(kMidList))
        list[pos] = static_cast<uint32_t>(4 * (tid + kMidThreads * (j >> 2)) + (j & 3));
      ++pos;
    }
  }
  __syncthreads();
  const uint32_t C = n_list;
  const bool fits = bk.beta >= 0 && C <= static_cast<uint32_t>(kMidList);
  if (fits) {
    // (3) keys above bucket beta are kept; bucket beta's keys feed the second level
    uint32_t g = 0;
    for (uint32_t e = tid; e < C; e += kMidThreads) {
      const uint32_t i = list[e];
      const uint32_t key = score_key(sf[i]);
      if ((key >> 20) > beta) {
        atomicOr(&bm[i >> 5], 1u << (i & 31));
        ++g;
      } else {
        atomicAdd(&h2[(key >> 8) & (kTopkBins - 1)], 1u);
      }
    }
    g = __reduce_add_sync(0xffffffffu, g);
    if (lane == 0 && g) atomicAdd(&n_gt, g);
  }
  __syncthreads();
  // push this half's counts and second level into the other rank
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  {
    uint32_t* rp = cl.map_shared_rank(h2p, peer);
    for (int i = tid; i < kTopkBins; i += kMidThreads) rp[i] = h2[i];
    if (tid == 0) {
      *cl.map_shared_rank(&peer_c, peer) = fits ? C : 0xffffffffu;  // a list that overflowed poisons the total
      *cl.map_shared_rank(&peer_g, peer) = n_gt;
    }
  }
  cl.sync();  // both halves' counts and second levels are here
  // the candidates must be exactly the histogram's keys in buckets >= beta
  const bool whole_row = !fits || peer_c == 0xffffffffu || n_gt + peer_g != bk.above ||
                         C + peer_c != bk.above + bk.hb;
  if (whole_row) {
    if (rank == 0) {
      const Rule r = digit_select<kMidThreads>(GlobalKeys{row}, n_vis, Rule{0u, 0u, k, 0u}, 24, h3, tmp, &rule);
      compact_row<kMidThreads>(GlobalKeys{row}, n_vis, r, out, sout, wgt, weq);
    }
    return;
  }
  for (int i = tid; i < kTopkBins; i += kMidThreads) h2p[i] += h2[i];
  __syncthreads();
  // (4) the rule: sub-bucket of bits 19..8 from the second level, then at most one 8-bit pass
  const Bucket b2 = find_bucket<kMidThreads>(h2p, k - bk.above, tmp, &sb2);
  Rule r{(beta << 20) | (static_cast<uint32_t>(b2.beta) << 8), 0xffffff00u, k - bk.above - b2.above,
         b2.hb == k - bk.above - b2.above ? 1u : 0u};
  if (!r.done) {  // the same in both ranks
    if (tid < 256) h3[tid] = 0u;
    __syncthreads();
    for (uint32_t e = tid; e < C; e += kMidThreads) {
      const uint32_t key = score_key(sf[list[e]]);
      if ((key & r.mask) == r.prefix) atomicAdd(&h3[key & 255u], 1u);
    }
    __syncthreads();
    if (tid < 256) cl.map_shared_rank(h3p, peer)[tid] = h3[tid];
    cl.sync();  // both halves' last digit counts are here
    if (tid < 256) h3p[tid] += h3[tid];
    __syncthreads();
    pick_digit<kMidThreads>(h3p, r, 0, tmp, &rule);
    r = rule;
  }
  for (uint32_t e = tid; e < C; e += kMidThreads) {
    const uint32_t i = list[e];
    const uint32_t key = score_key(sf[i]);
    if ((key >> 20) == beta) {
      const uint32_t mk = key & r.mask;
      if (mk > r.prefix) atomicOr(&bm[i >> 5], 1u << (i & 31));
      else if (mk == r.prefix) atomicOr(&eqm[i >> 5], 1u << (i & 31));
    }
  }
  __syncthreads();
  // (5) word tid: kept-for-sure and tied counts; prefix sums of both in one
  // scan (each total below 2^16)
  uint32_t wk = bm[tid], wq = eqm[tid];
  const uint32_t ng = static_cast<uint32_t>(__popc(wk)), ne = static_cast<uint32_t>(__popc(wq));
  const uint32_t incl = block_incl_scan<kMidThreads>(ng | (ne << 16), tmp);
  if (rank == 0 && tid == kMidThreads - 1) {  // rank 1's words follow rank 0's
    *cl.map_shared_rank(&off_kept, 1) = incl & 0xffffu;
    *cl.map_shared_rank(&off_eq, 1) = incl >> 16;
  }
  if (rank == 0 && tid == 0) {
    off_kept = 0u;
    off_eq = 0u;
  }
  cl.sync();  // rank 0's counts are in rank 1
  const uint32_t excl = incl - (ng | (ne << 16));
  const uint32_t eq_before = off_eq + (excl >> 16);  // ties in lower blocks of the whole row
  const uint32_t kept_before = off_kept + (excl & 0xffffu) + min(eq_before, r.k_rem);
  uint32_t take = r.k_rem > eq_before ? min(ne, r.k_rem - eq_before) : 0u;
  for (; take > 0; --take) {
    const uint32_t low = wq & (0u - wq);
    wk |= low;
    wq ^= low;
  }
  uint32_t pos = kept_before;
  while (wk) {
    const int bit = __ffs(wk) - 1;
    wk &= wk - 1;
    const int i = 32 * tid + bit;
    if (pos < k) {
      out[pos] = base + i;
      if (sout) sout[pos] = key_score(score_key(sf[i]));
    }
    ++pos;
  }
}

// ---------------------------------------------------------------- long rows
// (0) zero the histograms (the region the indexer / hist kernel accumulate into)
__global__ void __launch_bounds__(256) topk_zero_kernel(uint4* p, long long n16) {
  pdl_wait_then_release();
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n16; i += static_cast<long long>(gridDim.x) * 256)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// (1) histogram of given scores: (chunk, query) CTAs, flushed with integer atomics
__global__ void __launch_bounds__(kSelThreads) topk_hist_kernel(TopkArgs a) {
  pdl_wait_then_release();
  __shared__ uint32_t h[kTopkBins];
  const long long q = blockIdx.y;
  const int n_vis = visible(a, q);
  const int lo = static_cast<int>(blockIdx.x) * kTopkChunk;
  if (n_vis <= a.k || lo >= n_vis) return;
  const int hi = min(n_vis, lo + kTopkChunk);
  for (int i = threadIdx.x; i < kTopkBins; i += kSelThreads) h[i] = 0u;
  __syncthreads();
  const float* row = a.scores + q * a.ld;
  for (int base = lo; base < hi; base += kSelThreads) {
    const int i = base + static_cast<int>(threadIdx.x);
    hist_add(h, i < hi, i < hi ? score_key(row[i]) >> 20 : 0u);
  }
  __syncthreads();
  uint32_t* g = a.hist + q * kTopkBins;
  for (int i = threadIdx.x; i < kTopkBins; i += kSelThreads)
    if (h[i]) atomicAdd(g + i, h[i]);
}

// (2) candidates: the keys of one kTopkChunk-key chunk whose bucket is >=
// beta, written in index order to the chunk's own list; the keys of bucket
// beta also count into the second-level histogram of key bits 19..8.
__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(TopkArgs a) {
  pdl_wait_then_release();
  __shared__ unsigned long long tmp64[kSelThreads / 32];
  __shared__ uint32_t tmp[kSelThreads / 32];
  __shared__ Bucket sb;
  __shared__ unsigned long long tot_s;
  const long long q = blockIdx.y;
  const int c = blockIdx.x;
  const int n_vis = visible(a, q);
  const int lo = c * kTopkChunk;
  if (n_vis <= a.k || lo >= n_vis) return;
  const int hi = min(n_vis, lo + kTopkChunk);
  const int tid = threadIdx.x, lane = tid & 31;
  const long long nch = (a.N + kTopkChunk - 1) / kTopkChunk;
  // the chunk's scores first (they do not depend on the histogram):
  // thread t holds keys lo + 4*(t + 256*r) + e, r < kSelPer/4, e < 4
  const float* row = a.scores + q * a.ld;
  uint32_t key[kSelPer];
#pragma unroll
  for (int r = 0; r < kSelPer / 4; ++r) {
    const int i0 = lo + 4 * (tid + kSelThreads * r);
    float v[4];
    if (i0 + 3 < hi) {
      const float4 f = *reinterpret_cast<const float4*>(row + i0);  // lo, ld multiples of 4
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = i0 + e < hi ? row[i0 + e] : 0.f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) key[4 * r + e] = score_key(v[e]);
  }
  const Bucket bk = find_bucket<kSelThreads>(a.hist + q * kTopkBins, static_cast<uint32_t>(a.k), tmp, &sb);
  if (bk.beta < 0) {  // histogram holds fewer than k keys: the finish kernel reads the row instead
    if (tid == 0) a.ccount[q * nch + c] = 0u;
    return;
  }
  const uint32_t beta = static_cast<uint32_t>(bk.beta);
  uint32_t* hist2 = a.hist2 + q * kTopkBins;
  unsigned take = 0;
  unsigned long long packed = 0;
#pragma unroll
  for (int r = 0; r < kSelPer / 4; ++r) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 4 * r + e;
      const bool valid = lo + 4 * (tid + kSelThreads * r) + e < hi;
      const uint32_t bin = key[j] >> 20;
      if (valid && bin >= beta) {
        take |= 1u << j;
        packed += 1ull << (16 * r);
      }
      // second level: bits 19..8 of bucket beta's keys (warp-aggregated atomics)
      const bool inb = valid && bin == beta;
      const unsigned bal = __ballot_sync(0xffffffffu, inb);
      if (bal && inb) {
        const uint32_t b2 = (key[j] >> 8) & (kTopkBins - 1);
        const unsigned peers = __match_any_sync(bal, b2);
        if (lane == __ffs(peers) - 1) atomicAdd(hist2 + b2, static_cast<uint32_t>(__popc(peers)));
      }
    }
  }
  // index order within the chunk = (r, thread, e): scan the per-round counts
  const unsigned long long incl = block_incl_scan<kSelThreads>(packed, tmp64);
  if (tid == kSelThreads - 1) tot_s = incl;
  __syncthreads();
  const unsigned long long excl = incl - packed;
  const unsigned long long tot = tot_s;
  uint2* cand = a.cand + (q * nch + c) * kTopkChunk;
  uint32_t round_base = 0;
#pragma unroll
  for (int r = 0; r < kSelPer / 4; ++r) {
    uint32_t pos = round_base + static_cast<uint32_t>((excl >> (16 * r)) & 0xffffu);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 4 * r + e;
      if ((take >> j) & 1u) cand[pos++] = make_uint2(key[j], static_cast<uint32_t>(lo + 4 * (tid + kSelThreads * r) + e));
    }
    round_base += static_cast<uint32_t>((tot >> (16 * r)) & 0xffffu);
  }
  if (tid == 0) a.ccount[q * nch + c] = round_base;
}

// (3) the rule from the two histograms (and one last digit pass if needed),
// then the output: the chunks' candidate lists, concatenated in chunk order,
// are in index order, so one ordered compaction over them writes idx_out.
// The candidates are staged in shared memory when they fit (the usual case:
// a few thousand); otherwise the passes read them from global memory.
template <int T>
__device__ __forceinline__ void load_bins(const uint32_t* __restrict__ hist, uint32_t (&c)[kTopkBins / T]) {
  constexpr int P = kTopkBins / T;
  const int lo = kTopkBins - (static_cast<int>(threadIdx.x) + 1) * P;
#pragma unroll
  for (int i = 0; i < P; i += 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(hist + lo + i);
    c[i] = v.x;
    c[i + 1] = v.y;
    c[i + 2] = v.z;
    c[i + 3] = v.w;
  }
}

__global__ void __launch_bounds__(kFinThreads) topk_finish_kernel(TopkArgs a, int cap) {
  pdl_wait_then_release();
  // dynamic: per chunk count and start offset, then (cap) staged keys and indices
  extern __shared__ __align__(16) uint32_t fsm[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t tmp[32];
  __shared__ uint32_t wgt[32], weq[32];
  __shared__ Rule rule;
  __shared__ Bucket sb, sb2;
  __shared__ Tri tri_tmp[32];
  constexpr int NW = kFinThreads / 32;
  const long long q = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_vis = visible(a, q);
  int32_t* out = a.idx_out + q * a.k;
  float* sout = a.score_out ? a.score_out + q * a.k : nullptr;
  const float* row = a.scores + q * a.ld;
  if (n_vis <= a.k) {
    keep_all(a, row, n_vis, out, sout);
    return;
  }
  const uint32_t k = static_cast<uint32_t>(a.k);
  const long long nch_all = (a.N + kTopkChunk - 1) / kTopkChunk;
  const int nch = (n_vis + kTopkChunk - 1) / kTopkChunk;
  uint32_t* cnt_s = fsm;            // [nch]
  uint32_t* off_s = fsm + nch;      // [nch + 1]
  uint32_t* skey = fsm + 2 * nch + 4;
  uint32_t* sidx = skey + cap;
  const uint32_t* ccount = a.ccount + q * nch_all;
  const uint2* cand = a.cand + q * nch_all * kTopkChunk;
  // every independent load first: both histograms' bins and the chunk counts
  uint32_t c1[kTopkBins / kFinThreads], c2[kTopkBins / kFinThreads];
  load_bins<kFinThreads>(a.hist + q * kTopkBins, c1);
  load_bins<kFinThreads>(a.hist2 + q * kTopkBins, c2);
  const int per = (nch + kFinThreads - 1) / kFinThreads;  // chunks owned by a thread
  const int c_lo = min(nch, tid * per), c_hi = min(nch, c_lo + per);
  Tri v{0u, 0u, 0u};
  for (int c = c_lo; c < c_hi; ++c) {
    const uint32_t n = ccount[c];
    cnt_s[c] = n;
    v.z += n;
  }
#pragma unroll
  for (int i = 0; i < kTopkBins / kFinThreads; ++i) {
    v.x += c1[i];
    v.y += c2[i];
  }
  // one scan serves both bucket searches (thread order = descending buckets)
  // and the chunk offsets
  const Tri incl = block_incl_scan3<kFinThreads>(v, tri_tmp);
  if (tid == 0) {
    sb = Bucket{-1, 0u, 0u};
    sb2 = Bucket{-1, 0u, 0u};
  }
  {
    uint32_t run = incl.z - v.z;
    for (int c = c_lo; c < c_hi; ++c) {
      off_s[c] = run;
      run += cnt_s[c];
    }
    if (tid == kFinThreads - 1) off_s[nch] = incl.z;
  }
  __syncthreads();
  constexpr int P = kTopkBins / kFinThreads;
  const int bin_lo = kTopkBins - (tid + 1) * P;
  if (incl.x - v.x < k && k <= incl.x) {
    uint32_t run = incl.x - v.x;
#pragma unroll
    for (int i = P - 1; i >= 0; --i) {
      if (run + c1[i] >= k) {
        sb = Bucket{bin_lo + i, run, c1[i]};
        break;
      }
      run += c1[i];
    }
  }
  __syncthreads();
  const Bucket b1 = sb;
  if (b1.beta >= 0) {
    const uint32_t k2 = k - b1.above;
    if (incl.y - v.y < k2 && k2 <= incl.y) {
      uint32_t run = incl.y - v.y;
#pragma unroll
      for (int i = P - 1; i >= 0; --i) {
        if (run + c2[i] >= k2) {
          sb2 = Bucket{bin_lo + i, run, c2[i]};
          break;
        }
        run += c2[i];
      }
    }
  }
  __syncthreads();
  const Bucket b2 = sb2;
  if (b1.beta < 0 || b2.beta < 0) {
    // the histograms do not describe this row: select from the row itself
    const Rule r = digit_select<kFinThreads>(GlobalKeys{row}, n_vis, Rule{0u, 0u, k, 0u}, 24, hist, tmp, &rule);
    compact_row<kFinThreads>(GlobalKeys{row}, n_vis, r, out, sout, wgt, weq);
    return;
  }
  const int n_all = static_cast<int>(off_s[nch]);
  const bool staged = n_all <= cap;
  if (staged) {
    // each chunk's list is copied by tpc threads, eight loads in flight per thread
    int tpc = 1;
    while (tpc * 2 * nch <= kFinThreads && tpc < 32) tpc *= 2;
    const int groups = kFinThreads / tpc;
    for (int c = tid / tpc; c < nch; c += groups) {
      const int n = static_cast<int>(cnt_s[c]);
      const uint32_t dst = off_s[c];
      const uint2* cl = cand + static_cast<long long>(c) * kTopkChunk;
      for (int i0 = tid % tpc; i0 < n; i0 += 8 * tpc) {
        uint2 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * tpc;
          v[u] = i < n ? __ldcg(cl + i) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * tpc;
          if (i < n) {
            skey[dst + i] = v[u].x;
            sidx[dst + i] = v[u].y;
          }
        }
      }
    }
  }
  Rule r{(static_cast<uint32_t>(b1.beta) << 20) | (static_cast<uint32_t>(b2.beta) << 8), 0xFFFFFF00u,
         k - b1.above - b2.above, 0u};
  r.done = b2.hb == r.k_rem ? 1u : 0u;
  if (tid < 256) hist[tid] = 0u;
  __syncthreads();
  if (!r.done) {
    // last 8 bits among the candidates with this 24-bit prefix
    if (staged) {
      for (int base = 0; base < n_all; base += kFinThreads) {
        const int i = base + tid;
        const uint32_t key = i < n_all ? skey[i] : 0u;
        hist_add(hist, i < n_all && (key & r.mask) == r.prefix, key & 255u);
      }
    } else {
      for (int c = warp; c < nch; c += NW) {
        const uint2* cl = cand + static_cast<long long>(c) * kTopkChunk;
        const int n = static_cast<int>(cnt_s[c]);
        for (int base = 0; base < n; base += 32) {
          const int i = base + lane;
          const uint32_t key = i < n ? cl[i].x : 0u;
          hist_add(hist, i < n && (key & r.mask) == r.prefix, key & 255u);
        }
      }
    }
    __syncthreads();
    pick_digit<kFinThreads>(hist, r, 0, tmp, &rule);
    r = rule;
    __syncthreads();
  }
  // ordered compaction: each warp owns a contiguous segment of the list
  const int seg = ((n_all + NW - 1) / NW + 31) & ~31;
  const int s_lo = min(n_all, warp * seg), s_hi = min(n_all, s_lo + seg);
  auto cand_at = [&](int p) -> uint2 {
    if (staged) return make_uint2(skey[p], sidx[p]);
    int lo = 0, hi = nch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off_s[mid] <= static_cast<uint32_t>(p)) lo = mid; else hi = mid - 1;
    }
    return cand[static_cast<long long>(lo) * kTopkChunk + (p - off_s[lo])];
  };
  uint32_t ngt = 0, neq = 0;
  for (int base = s_lo; base < s_hi; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < s_hi ? cand_at(i).x & r.mask : 0u;
    ngt += __popc(__ballot_sync(0xffffffffu, i < s_hi && key > r.prefix));
    neq += __popc(__ballot_sync(0xffffffffu, i < s_hi && key == r.prefix));
  }
  if (lane == 0) {
    wgt[warp] = ngt;
    weq[warp] = neq;
  }
  __syncthreads();
  uint32_t run_gt = 0, run_eq = 0;
  for (int w = 0; w < warp; ++w) {
    run_gt += wgt[w];
    run_eq += weq[w];
  }
  const unsigned lt = lanemask_lt();
  for (int base = s_lo; base < s_hi; base += 32) {
    const int i = base + lane;
    const uint2 cv = i < s_hi ? cand_at(i) : make_uint2(0u, 0u);
    const uint32_t key = cv.x & r.mask;
    const bool gt = i < s_hi && key > r.prefix;
    const bool eq = i < s_hi && key == r.prefix;
    const unsigned bgt = __ballot_sync(0xffffffffu, gt);
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const uint32_t gt_before = run_gt + __popc(bgt & lt);
    const uint32_t eq_before = run_eq + __popc(beq & lt);
    if (gt || (eq && eq_before < r.k_rem)) {
      const uint32_t pos = gt_before + min(eq_before, r.k_rem);
      out[pos] = static_cast<int32_t>(cv.y);
      if (sout) sout[pos] = key_score(cv.x);
    }
    run_gt += __popc(bgt);
    run_eq += __popc(beq);
  }
}

}  // namespace

bool topk_supported(int N) { return N >= 0 && N <= kTopkMaxN; }

bool topk_long_rows(int N) { return N > kTopkShortMax; }

namespace {
inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }
inline long long n_chunks(int N) { return (static_cast<long long>(N) + kTopkChunk - 1) / kTopkChunk; }
}  // namespace

size_t topk_scratch_zero_bytes(long long nq) { return static_cast<size_t>(nq) * (kTopkBins * 2 + 256) * 4; }

// candidate bytes per query: the chunk lists of the select kernel, or the
// per-CTA lists of the fused decode tail, whichever is larger
size_t cand_bytes_per_query(int N) {
  const size_t a = static_cast<size_t>(n_chunks(N)) * kTopkChunk * 8;
  const size_t b = tail_cand_bytes_per_query(N);
  return a > b ? a : b;
}

size_t topk_scratch_bytes(long long nq, int N) {
  if (!topk_long_rows(N)) return 0;
  const long long nch = n_chunks(N);
  return topk_scratch_zero_bytes(nq) + al16(static_cast<size_t>(nq) * nch * 4) +
         static_cast<size_t>(nq) * cand_bytes_per_query(N);
}

void topk_scratch_carve(TopkArgs& a, void* base, long long nq) {
  char* p = static_cast<char*>(base);
  const long long nch = n_chunks(a.N);
  a.hist = reinterpret_cast<uint32_t*>(p);
  a.hist2 = reinterpret_cast<uint32_t*>(p + static_cast<size_t>(nq) * kTopkBins * 4);
  a.hist3 = reinterpret_cast<uint32_t*>(p + static_cast<size_t>(nq) * kTopkBins * 8);
  p += topk_scratch_zero_bytes(nq);
  a.ccount = reinterpret_cast<uint32_t*>(p);
  p += al16(static_cast<size_t>(nq) * nch * 4);
  a.cand = reinterpret_cast<uint2*>(p);
}

cudaError_t launch_topk_zero(const TopkArgs& a, long long nq, cudaStream_t s) {
  const long long n16 = static_cast<long long>(topk_scratch_zero_bytes(nq) / 16);
  long long blocks = (n16 + 255) / 256;
  blocks = blocks > 296 ? 296 : (blocks < 1 ? 1 : blocks);
  return launch_k(topk_zero_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, 1,
                  reinterpret_cast<uint4*>(a.hist), n16);
}

cudaError_t launch_topk_hist(const TopkArgs& a, cudaStream_t s) {
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (nq == 0) return cudaSuccess;
  if (nq > 65535) return cudaErrorNotSupported;
  cudaError_t e = launch_topk_zero(a, nq, s);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(n_chunks(a.N)), static_cast<unsigned>(nq));
  return launch_k(topk_hist_kernel, grid, dim3(kSelThreads), 0, s, 1, a);
}

cudaError_t launch_topk(const TopkArgs& a, bool hist_ready, cudaStream_t s) {
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (nq == 0) return cudaSuccess;
  if (nq > 0x7fffffffLL) return cudaErrorNotSupported;
  if (!topk_long_rows(a.N)) {
    const size_t smem = static_cast<size_t>(a.N > 0 ? a.N : 1) * 4;
    cudaError_t e = ensure_dyn_smem<topk_short_kernel>(kTopkShortMax * 4);
    if (e != cudaSuccess) return e;
    return launch_k(topk_short_kernel, dim3(static_cast<unsigned>(nq)), dim3(kShortThreads), smem, s, 1, a);
  }
  if (nq > 65535) return cudaErrorNotSupported;
  const dim3 grid(static_cast<unsigned>(n_chunks(a.N)), static_cast<unsigned>(nq));
  cudaError_t e;
  if (!hist_ready) {
    e = launch_topk_zero(a, nq, s);
    if (e != cudaSuccess) return e;
    e = launch_k(topk_hist_kernel, grid, dim3(kSelThreads), 0, s, 1, a);
    if (e != cudaSuccess) return e;
  }
  if (a.N <= kTopkMidMax) {
    // one CTA per query: the row's keys and bucket beta's keys in shared memory
    const size_t smem = static_cast<size_t>(kMidSmemWords) * 4;
    e = ensure_dyn_smem<topk_mid_kernel>(static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_k(topk_mid_kernel, dim3(kMidRanks, static_cast<unsigned>(nq)), dim3(kMidThreads), smem, s,
                    kMidRanks, a);
  }
  e = launch_k(topk_select_kernel, grid, dim3(kSelThreads), 0, s, 1, a);
  if (e != cudaSuccess) return e;
  // shared memory: per chunk a count and an offset, then up to ``cap`` staged
  // candidates (8 bytes each) within the budget
  const size_t head = (2 * static_cast<size_t>(n_chunks(a.N)) + 4) * 4;
  const int cap = static_cast<int>((kFinSmemBudget - head) / 8);
  e = ensure_dyn_smem<topk_finish_kernel>(kFinSmemBudget);
  if (e != cudaSuccess) return e;
  return launch_k(topk_finish_kernel, dim3(static_cast<unsigned>(nq)), dim3(kFinThreads), kFinSmemBudget, s, 1,
                  a, cap);
}

}  // namespace csa
