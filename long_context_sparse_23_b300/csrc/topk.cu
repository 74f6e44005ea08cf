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
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kShortThreads = 512;
constexpr int kSelThreads = 256;
constexpr int kSelPer = kTopkChunk / kSelThreads;   // keys per select thread (16)
constexpr int kFinThreads = 512;
constexpr int kFinSmemBudget = 200 * 1024;
static_assert(kSelPer == 16, "the select kernel packs four rounds of 4 keys per thread");

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
  uint32_t k_rem;
  uint32_t done;
};

struct Bucket {
  int beta;        // bucket of the k-th largest key, -1 if the histogram holds fewer than k keys
  uint32_t above;  // keys in higher buckets
  uint32_t hb;     // keys in the bucket
};

// Warp-aggregated shared-memory histogram increment (lanes with the same bin
// add once).  Every lane of the warp calls it.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool active, uint32_t bin) {
  const unsigned am = __ballot_sync(0xffffffffu, active);
  if (active) {
    const unsigned peers = __match_any_sync(am, bin);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
  }
}

// Inclusive scan of one value per thread over a block of T threads; tmp holds
// T/32 entries.  Every thread calls it.
template <int T, typename V>
__device__ __forceinline__ V block_incl_scan(V v, V* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    V w = lane < T / 32 ? tmp[lane] : V(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const V n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < T / 32) tmp[lane] = w;  // inclusive totals per warp
  }
  __syncthreads();
  const V add = warp > 0 ? tmp[warp - 1] : V(0);
  __syncthreads();
  return v + add;
}

// Inclusive scan of three counters per thread at once (one set of barriers).
struct Tri {
  uint32_t x, y, z;
};
template <int T>
__device__ __forceinline__ Tri block_incl_scan3(Tri v, Tri* tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t nx = __shfl_up_sync(0xffffffffu, v.x, o);
    const uint32_t ny = __shfl_up_sync(0xffffffffu, v.y, o);
    const uint32_t nz = __shfl_up_sync(0xffffffffu, v.z, o);
    if (lane >= o) {
      v.x += nx;
      v.y += ny;
      v.z += nz;
    }
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    Tri w = lane < T / 32 ? tmp[lane] : Tri{0u, 0u, 0u};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t nx = __shfl_up_sync(0xffffffffu, w.x, o);
      const uint32_t ny = __shfl_up_sync(0xffffffffu, w.y, o);
      const uint32_t nz = __shfl_up_sync(0xffffffffu, w.z, o);
      if (lane >= o) {
        w.x += nx;
        w.y += ny;
        w.z += nz;
      }
    }
    if (lane < T / 32) tmp[lane] = w;
  }
  __syncthreads();
  const Tri add = warp > 0 ? tmp[warp - 1] : Tri{0u, 0u, 0u};
  return Tri{v.x + add.x, v.y + add.y, v.z + add.z};
}

// The bucket holding the k-th largest key, from a 4096-bin histogram in
// global memory.  Thread t owns bins [4096 - (t+1)*P, 4096 - t*P), so a scan
// in thread order runs from the top bucket down.  All T threads call it.
template <int T>
__device__ Bucket find_bucket(const uint32_t* __restrict__ hist, uint32_t k, uint32_t* tmp, Bucket* sb) {
  constexpr int P = kTopkBins / T;
  static_assert(P % 4 == 0, "bins per thread must be a multiple of 4");
  const int lo = kTopkBins - (static_cast<int>(threadIdx.x) + 1) * P;
  uint32_t c[P];
#pragma unroll
  for (int i = 0; i < P; i += 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(hist + lo + i);
    c[i] = v.x;
    c[i + 1] = v.y;
    c[i + 2] = v.z;
    c[i + 3] = v.w;
  }
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < P; ++i) s += c[i];
  if (threadIdx.x == 0) *sb = Bucket{-1, 0u, 0u};
  const uint32_t incl = block_incl_scan<T>(s, tmp);
  const uint32_t excl = incl - s;
  if (excl < k && k <= incl) {
    uint32_t run = excl;
#pragma unroll
    for (int i = P - 1; i >= 0; --i) {
      if (run + c[i] >= k) {
        *sb = Bucket{lo + i, run, c[i]};
        break;
      }
      run += c[i];
    }
  }
  __syncthreads();
  const Bucket b = *sb;
  __syncthreads();
  return b;
}

// Given a 256-bin histogram H of the digit at ``shift`` among the keys that
// match r, extend r by the digit holding the r.k_rem-th largest key; the new
// rule is written to *dst.  All T threads call it; *dst is valid after it
// returns.
template <int T>
__device__ __forceinline__ void pick_digit(const uint32_t* H, const Rule r, int shift, uint32_t* tmp,
                                           Rule* dst) {
  const int tid = threadIdx.x;
  const uint32_t v = tid < 256 ? H[255 - tid] : 0u;
  const uint32_t incl = block_incl_scan<T>(v, tmp);
  const uint32_t excl = incl - v;
  if (tid < 256 && excl < r.k_rem && r.k_rem <= incl) {
    const uint32_t digit = 255u - static_cast<uint32_t>(tid);
    Rule nr;
    nr.prefix = r.prefix | (digit << shift);
    nr.mask = r.mask | (255u << shift);
    nr.k_rem = r.k_rem - excl;
    nr.done = (v == r.k_rem - excl) || shift == 0;
    *dst = nr;
  }
  __syncthreads();
}

// Keys of one query's row, read from shared memory (staged) or from the
// fp32 scores in global memory.
struct SmemKeys {
  const uint32_t* keys;
  __device__ uint32_t operator()(int i) const { return keys[i]; }
};
struct GlobalKeys {
  const float* row;
  __device__ uint32_t operator()(int i) const { return score_key(row[i]); }
};

// Fix the rule for the k largest of n keys by 8-bit digit passes (from bit
// 24 down), starting from ``r`` (prefix bits already fixed).  All T threads
// call it; returns the final rule.
template <int T, typename Keys>
__device__ Rule digit_select(Keys keys, int n, Rule r, int first_shift, uint32_t* hist, uint32_t* tmp,
                             Rule* sr) {
  for (int shift = first_shift; shift >= 0 && !r.done; shift -= 8) {
    if (threadIdx.x < 256) hist[threadIdx.x] = 0u;
    __syncthreads();
    for (int base = 0; base < n; base += T) {
      const int i = base + static_cast<int>(threadIdx.x);
      const uint32_t key = i < n ? keys(i) : 0u;
      hist_add(hist, i < n && (key & r.mask) == r.prefix, (key >> shift) & 255u);
    }
    __syncthreads();
    pick_digit<T>(hist, r, shift, tmp, sr);
    r = *sr;
    __syncthreads();
  }
  return r;
}

// Write the kept indices of a row in index order: each warp owns a
// contiguous segment, counts its kept keys, and after a scan over warps
// writes them with ballots.  All T threads call it.
template <int T, typename Keys>
__device__ void compact_row(Keys keys, int n, const Rule r, int32_t* out, float* sout, uint32_t* wgt,
                            uint32_t* weq) {
  constexpr int NW = T / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = ((n + NW - 1) / NW + 31) & ~31;
  const int s_lo = min(n, warp * seg), s_hi = min(n, s_lo + seg);
  uint32_t ngt = 0, neq = 0;
  for (int base = s_lo; base < s_hi; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < s_hi ? keys(i) & r.mask : 0u;
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
    const uint32_t full = i < s_hi ? keys(i) : 0u;
    const uint32_t key = full & r.mask;
    const bool gt = i < s_hi && key > r.prefix;
    const bool eq = i < s_hi && key == r.prefix;
    const unsigned bgt = __ballot_sync(0xffffffffu, gt);
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    const uint32_t gt_before = run_gt + __popc(bgt & lt);
    const uint32_t eq_before = run_eq + __popc(beq & lt);
    if (gt || (eq && eq_before < r.k_rem)) {
      const uint32_t pos = gt_before + min(eq_before, r.k_rem);
      out[pos] = i;
      if (sout) sout[pos] = key_score(full);
    }
    run_gt += __popc(bgt);
    run_eq += __popc(beq);
  }
  __syncthreads();
}

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

size_t topk_scratch_zero_bytes(long long nq) { return static_cast<size_t>(nq) * kTopkBins * 4 * 2; }

size_t topk_scratch_bytes(long long nq, int N) {
  if (!topk_long_rows(N)) return 0;
  const long long nch = n_chunks(N);
  return topk_scratch_zero_bytes(nq) + al16(static_cast<size_t>(nq) * nch * 4) +
         static_cast<size_t>(nq) * nch * kTopkChunk * 8;
}

void topk_scratch_carve(TopkArgs& a, void* base, long long nq) {
  char* p = static_cast<char*>(base);
  const long long nch = n_chunks(a.N);
  a.hist = reinterpret_cast<uint32_t*>(p);
  a.hist2 = reinterpret_cast<uint32_t*>(p + static_cast<size_t>(nq) * kTopkBins * 4);
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
