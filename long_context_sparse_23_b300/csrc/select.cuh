// Exact selection helpers shared by the top-k kernels and the fused decode
// tail: order-preserving 32-bit keys of fp32 scores (-0 folded onto +0),
// selection rules, warp-aggregated histograms, block-wide scans, digit passes
// and ordered compaction.  All integer arithmetic: exact and deterministic.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace csa {
namespace {

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

// The same for a histogram in global memory (integer reductions at L2).
__device__ __forceinline__ void hist_add_global(uint32_t* hist, bool active, uint32_t bin) {
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

// Position i of a row is block index i, or (a candidate list) the block index
// stored for it.
struct RowIndex {
  __device__ int operator()(int i) const { return i; }
};
struct ListIndex {
  const uint32_t* idx;
  __device__ int operator()(int i) const { return static_cast<int>(idx[i]); }
};

// Write the kept indices of a row (or of a candidate list in index order) in
// index order: each warp owns a contiguous segment, counts its kept keys, and
// after a scan over warps writes them with ballots.  All T threads call it.
template <int T, typename Keys, typename Index = RowIndex>
__device__ void compact_row(Keys keys, int n, const Rule r, int32_t* out, float* sout, uint32_t* wgt,
                            uint32_t* weq, Index index = Index{}) {
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
      out[pos] = index(i);
      if (sout) sout[pos] = key_score(full);
    }
    run_gt += __popc(bgt);
    run_eq += __popc(beq);
  }
  __syncthreads();
}

}  // namespace
}  // namespace csa
