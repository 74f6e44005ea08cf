// Fused decode tail of the CSA layer: top-k selection and window-merged
// sparse attention for decode-shaped calls, one thread-block cluster of 16
// CTAs per query.  "DeepSeek V4 technical review", section 2.1: the indexer's
// top-k blocks (k = 1024) are attended together with the sliding window of
// raw tokens (octagono "Hybrid Attention: CSA and HCA"); the selection and the
// attention compute exactly what topk_*_kernel and attend_*_kernel compute.
//
// Input: the indexer's fp32 scores of the query's n_vis visible blocks and a
// 4096-bin histogram of their order-preserving keys' top 12 bits.  Steps,
// with a cluster barrier between them:
//  1. CTA r scans its chunk [r*E, (r+1)*E) of the scores and keeps, in index
//     order, every key whose bucket is >= beta, the bucket holding the k-th
//     largest key (candidates: in global memory, and, when they fit, pushed
//     by one bulk copy per CTA into every CTA's shared memory before the
//     barrier);
//  2. every CTA reads the candidates of bucket beta and fixes the same exact
//     rule (prefix, mask, k_rem) with a histogram of key bits 19..8 and at
//     most one 8-bit pass: keys above the prefix are kept, and of the keys
//     equal to it the k_rem with the lowest indices;
//  3. each CTA counts its kept candidates, learns the counts of the CTAs
//     before it, and so the rank of each kept block in ascending order; it
//     writes idx_out and records (rank -> block) for the ranks it attends;
//  4. CTA r gathers the K/V rows of its virtual key slots [r*S_r, (r+1)*S_r)
//     (selected blocks by rank, then the window; all 256 threads, 16 bytes
//     each, consecutive threads on consecutive chunks of a row) and attends
//     them for every head (8 warps: 4 groups of 16 heads x 2 key halves,
//     mma.sync), merges the halves in registers (the two warps of a head
//     group meet at a named barrier), and sends each head's (O, max, sum)
//     to the CTA owning that head;
//  5. each CTA folds the partials of its heads in rank order and writes the
//     output.
// Everything merges in a fixed order: results do not depend on scheduling.
#include <cooperative_groups.h>

#include "attend_tile.cuh"
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace cg = cooperative_groups;

namespace csa {


namespace {

constexpr int kT = 256;         // threads per CTA
constexpr int kC = kTailCluster;  // CTAs per query (one cluster)
constexpr int kCandP = 256;     // candidates of one rank pushed to every CTA of the cluster
constexpr int kRun = 64;        // consecutive scores per thread in the candidate scan
constexpr int kBulk = 16384;    // bytes per bulk copy
// K/V tile rows: contiguous, 16 bytes of padding (conflict-free ldmatrix)
template <int D>
constexpr int kv_pitch() { return D * 2 + 16; }
// A wait that ran out of the call's budget is reported and then continued
// with this budget (about one second), so that no bulk copy is still writing
// this CTA's shared memory when the buffer is refilled or the CTA exits.
constexpr long long kDrainBudget = 1LL << 31;

// Shared-memory layout (bytes), the same on host and device.
struct TailLayout {
  int stage;      // step 1: a batch of scores
  int kv, codes;  // step 3: the K/V tile and slot codes
  int merge;      // step 3: the second key half's partials (overlap the above once consumed)
  int map, recv;  // persistent: rank -> block of this CTA's slots, partials of its heads
  int qs;         // persistent: the query's rows [H][D] bf16
  int own;        // this rank's first kCandP candidates (the source of its pushes)
  int plist;      // every rank's pushed candidates [kC][kCandP]
  int total;
  int hpc;        // heads owned per CTA
};

__host__ __device__ inline TailLayout tail_layout(int S_r, int H, int D, int E) {
  TailLayout L;
  const int ldo = D + 4;
  L.stage = 0;
  const int scores = (E < kT * kRun ? E : kT * kRun) * 4;
  const int sel_end = scores;
  L.kv = (sel_end + 127) / 128 * 128;
  L.codes = L.kv + 2 * S_r * (D * 2 + 16);
  const int kv_end = L.codes + S_r * 4;
  L.merge = 0;  // [H][ldo] o, then [H] m, [H] l of the second key half
  const int merge_end = L.merge + (H * ldo + 2 * H) * 4;
  const int a_end = kv_end > merge_end ? kv_end : merge_end;
  L.map = (a_end + 15) / 16 * 16;
  L.recv = L.map + (S_r * 4 + 15) / 16 * 16;
  L.hpc = (H + kC - 1) / kC;
  L.qs = L.recv + ((L.hpc * kC * ldo + 2 * L.hpc * kC) * 4 + 127) / 128 * 128;
  L.own = L.qs + H * D * 2;
  L.plist = L.own + kCandP * 8;
  L.total = L.plist + kC * kCandP * 8;
  return L;
}

// One-dimensional bulk copy (TMA) global -> this CTA's shared memory,
// completing on ``bar``; 16-byte aligned addresses, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// KH: keys per warp per tile step (the half of S_r a warp attends is walked
// in steps of KH keys; KH = S_r / 2 makes it one step).
template <int D, int KH>
__global__ void __launch_bounds__(kT, 1) decode_tail_kernel(TailArgs a, int E, int S_r) {
  constexpr int LDO = D + 4;
  constexpr int CH = D / 8, DT = D / 8;
  extern __shared__ __align__(128) char smem[];
  __shared__ uint32_t tmp[32];
  __shared__ Bucket sb;
  __shared__ Rule rule;
  __shared__ uint32_t tot32;

  cg::cluster_group cluster = cg::this_cluster();
  const int r = static_cast<int>(cluster.block_rank());
  const long long q = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const AttendArgs& at = a.at;
  const int H = at.H;
  const TailLayout L = tail_layout(S_r, H, D, E);
  int* map = reinterpret_cast<int*>(smem + L.map);
  float* recv = reinterpret_cast<float*>(smem + L.recv);  // [hpc][kC][LDO]
  float* recv_m = recv + L.hpc * kC * LDO;                // [hpc][kC]
  float* recv_l = recv_m + L.hpc * kC;                    // [hpc][kC]
  __shared__ __align__(8) uint64_t bar, bar_q, bar_l;
  __shared__ uint32_t rcnt[kC], wg[kT / 32], we[kT / 32];
  uint32_t bar_phase = 0;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&bar_q, 1);
    mbar_init(&bar_l, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // first half of a cluster barrier: every CTA of the cluster has started
  // before any writes another's shared memory (the wait is at the first
  // such write)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // wait for the bulk copies on ``bar``: bounded by the call's budget (a
  // timeout is reported), then drained, so the copies have landed before the
  // buffer is read, refilled or given up at exit
  auto bulk_wait = [&]() {
    if (!mbar_wait(&bar, bar_phase, a.budget, nullptr)) {
      raise_flag(at.errw, kFlagTimeout);
      mbar_wait(&bar, bar_phase, kDrainBudget, nullptr);
    }
    bar_phase ^= 1u;
  };

  const int b = static_cast<int>(q / at.Tq);
  const int t = a.q_pos[q];
  const int raw_base = at.W > 0 ? at.raw_base[b] : 0;  // read now: step 3's window slots need it
  int n_vis = t >= 0 ? (t + 1) / a.m : 0;
  n_vis = n_vis < a.N ? n_vis : a.N;
  const int k = a.k;
  const int K_total = k + at.W;
  const int A = (K_total + S_r - 1) / S_r;  // CTAs with key slots
  const bool all = n_vis <= k;              // every visible block is kept (uniform over the cluster)
  const float* row = a.scores + q * a.ld;
  uint2* gl_all = a.cand + q * static_cast<long long>(kC) * E;  // [kC][E]
  const int lo = r * E, hi = min(n_vis, lo + E);
  char* qs = smem + L.qs;  // the query's rows, used by step 3
  if (r < A && tid == 0) {
    mbar_expect_tx(&bar_q, static_cast<uint32_t>(H * D * 2));
    bulk_g2s(qs, static_cast<const char*>(at.q) + static_cast<size_t>(q) * H * D * 2,
             static_cast<uint32_t>(H * D * 2), &bar_q);
  }
  // K/V tile of this CTA's key slots (gathered in step 3)
  char* Ks = smem + L.kv;
  constexpr int PITCH = kv_pitch<D>();
  char* Vs = Ks + S_r * PITCH;
  const char* kc_base = static_cast<const char*>(at.k_cmp) + static_cast<size_t>(b) * at.N * D * 2;
  const char* vc_base = static_cast<const char*>(at.v_cmp) + static_cast<size_t>(b) * at.N * D * 2;

  // Everything above reads only the call's inputs (query positions, the
  // window's base position, the query rows), which no kernel of this call
  // writes; the kernel launched before
  // this one's predecessor has completed when this kernel starts (each
  // kernel releases its dependents after its own wait, the indexer after
  // the histogram-zeroing kernel's).  The scores and histograms below are
  // the indexer's: wait for it.
  pdl_wait_then_release();

  // the scores of this CTA's first batch to shared memory by bulk copy
  // (rounded up to 4 scores: the row holds ld >= N, a multiple of 4), issued
  // before the bucket search, which does not need them
  float* stage = reinterpret_cast<float*>(smem + L.stage);  // [kT * kRun] scores of a batch
  auto issue_batch = [&](int sub) {
    const uint32_t bytes = static_cast<uint32_t>(min(kT * kRun, ((hi - sub) + 3) & ~3)) * 4;
    if (tid == 0) {
      fence_proxy_async();  // the stage was read by the threads of the last batch
      mbar_expect_tx(&bar, bytes);
      for (uint32_t off = 0; off < bytes; off += kBulk)
        bulk_g2s(reinterpret_cast<char*>(stage) + off, reinterpret_cast<const char*>(row + sub) + off,
                 min(static_cast<uint32_t>(kBulk), bytes - off), &bar);
    }
  };
  if (!all && lo < hi) issue_batch(lo);
  Bucket b1{0, 0u, 0u};
  if (!all) {
    b1 = find_bucket<kT>(a.hist + q * kTopkBins, static_cast<uint32_t>(k), tmp, &sb);
    if (b1.beta < 0) {
      // the histogram does not describe the row (uniform): report and write
      // nothing, once this CTA's copy of the query has landed
      if (r == 0 && tid == 0) raise_flag(at.errw, kFlagIndex);
      if (r < A) mbar_wait(&bar_q, 0, kDrainBudget, nullptr);
      if (lo < hi) mbar_wait(&bar, 0, kDrainBudget, nullptr);
      return;
    }
  }

  // ---- 1. candidates of this CTA's chunk, in index order; the keys of
  // bucket beta also count into the second-level histogram (bits 19..8)
  uint32_t n_own = 0;
  if (!all) {
    const uint32_t beta = static_cast<uint32_t>(b1.beta);
    uint2* gl = gl_all + static_cast<long long>(r) * E;
    uint32_t* hist2 = a.hist2 + q * kTopkBins;
    uint2* own = reinterpret_cast<uint2*>(smem + L.own);
    // the lowest scores of buckets beta and beta + 1: the key map is
    // order-preserving (and folds -0 onto +0, as the float comparison does),
    // so a finite score is a candidate iff it compares >= tb and in bucket
    // beta iff also < tb1 (bucket 0 has no lowest value: every score is a
    // candidate then; above the top bucket nothing is)
    const float tb = beta == 0 ? -INFINITY : key_score(beta << 20);
    const float tb1 = beta >= kTopkBins - 1 ? INFINITY : key_score((beta + 1) << 20);
    for (int sub = lo; sub < hi; sub += kT * kRun) {
      if (sub != lo) issue_batch(sub);  // the first batch was requested before the bucket search
      bulk_wait();
      // thread tid owns the run [sub + kRun*tid, sub + kRun*(tid+1)); its 16
      // float4 reads start at a rotated position (fewer bank conflicts); the
      // marks are set at the read order's bit positions (constant shifts)
      // and rotated back to index order once
      const int i0 = sub + kRun * tid;
      const bool full_run = i0 + kRun <= hi;
      unsigned long long take_r = 0ull, inb_r = 0ull;
#pragma unroll
      for (int jr = 0; jr < kRun / 4; ++jr) {
        const int j = (jr + tid) & (kRun / 4 - 1);
        const float4 fv = *reinterpret_cast<const float4*>(stage + kRun * tid + 4 * j);
        const float v4[4] = {fv.x, fv.y, fv.z, fv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool c = (full_run || i0 + 4 * j + e < hi) && v4[e] >= tb;
          take_r |= static_cast<unsigned long long>(c) << (4 * jr + e);
          inb_r |= static_cast<unsigned long long>(c && v4[e] < tb1) << (4 * jr + e);
        }
      }
      // read position 4 jr + e holds element 4 ((jr + tid) mod 16) + e
      const int rot = 4 * (tid & (kRun / 4 - 1));
      unsigned long long take = rot ? (take_r << rot) | (take_r >> (64 - rot)) : take_r;
      const unsigned long long inb = rot ? (inb_r << rot) | (inb_r >> (64 - rot)) : inb_r;
      // bucket beta holds about k of the keys: one reduction per key of it
      for (unsigned long long m2 = inb; m2; m2 &= m2 - 1) {
        const int p = __ffsll(static_cast<long long>(m2)) - 1;
        atomicAdd(hist2 + ((score_key(stage[kRun * tid + p]) >> 8) & (kTopkBins - 1)), 1u);
      }
      const uint32_t mine = static_cast<uint32_t>(__popcll(take));
      const uint32_t incl = block_incl_scan<kT>(mine, tmp);
      if (tid == kT - 1) tot32 = incl;
      __syncthreads();
      uint32_t pos = n_own + incl - mine;
      while (take) {
        const int p = __ffsll(static_cast<long long>(take)) - 1;
        take &= take - 1;
        const uint2 cv = make_uint2(score_key(stage[kRun * tid + p]), static_cast<uint32_t>(i0 + p));
        if (pos < static_cast<uint32_t>(kCandP)) own[pos] = cv;
        gl[pos++] = cv;
      }
      n_own += tot32;
      __syncthreads();  // the stage and tot32 are rewritten by the next batch
    }
  }
  // this rank's candidate count into every CTA's table (read after the
  // barrier), and its candidates (when they fit) into every CTA's list
  // area by one bulk copy each, completing on that CTA's bar_l
  fence_proxy_async();  // the own list, written by the threads, is read by the bulk copies
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (tid < kC) {
    *cluster.map_shared_rank(&rcnt[r], tid) = n_own;
    if (n_own > 0 && n_own <= static_cast<uint32_t>(kCandP)) {
      uint32_t dst, mb;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                   : "=r"(dst)
                   : "r"(smem_u32(smem + L.plist + r * kCandP * 8)), "r"(tid));
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(mb) : "r"(smem_u32(&bar_l)), "r"(tid));
      asm volatile(
          "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
          "r"(smem_u32(smem + L.own)), "r"((n_own + 1) / 2 * 16), "r"(mb)
          : "memory");
    }
  }
  // no slot of this CTA holds a kept block until step 2 says so (with
  // consistent inputs step 2 fills every slot below k; with a histogram that
  // does not match the scores, unfilled slots stay empty instead of undefined)
  for (int j = tid; j < S_r; j += kT) map[j] = -1;
  cluster.sync();  // #1: every rank's candidates and bucket counts are written

  // ---- 2. the rule, and this CTA's ranks of the selection (every CTA reads
  // all candidates, so no further exchange is needed before the attention)
  if (all) {
    for (int j = tid; j < S_r; j += kT) {
      const int pos = r * S_r + j;
      map[j] = pos < n_vis ? pos : -1;
    }
    if (a.idx_out) {
      for (int p = r * kT + tid; p < k; p += kC * kT) {
        a.idx_out[q * k + p] = p < n_vis ? p : -1;
        if (a.score_out) a.score_out[q * k + p] = p < n_vis ? key_score(score_key(row[p])) : 0.f;
      }
    }
  } else {
    // the pushed lists: every rank whose candidates fit pushed them here
    // before the barrier; all pushes land before they are read (also when
    // another rank's did not fit and the lists are read from global memory)
    bool staged = true;
    uint32_t pushed = 0;
    for (int i = 0; i < kC; ++i) {
      const bool fits = rcnt[i] <= static_cast<uint32_t>(kCandP);
      staged = staged && fits;
      if (fits) pushed += (rcnt[i] + 1) / 2 * 16;
    }
    if (tid == 0) mbar_expect_tx(&bar_l, pushed);
    const uint2* lists = reinterpret_cast<const uint2*>(smem + L.plist);  // [kC][kCandP]
    // the rule's top 24 bits from the second-level histogram (global)
    const uint32_t beta = static_cast<uint32_t>(b1.beta);
    const uint32_t k2 = static_cast<uint32_t>(k) - b1.above;
    const Bucket b2 = find_bucket<kT>(a.hist2 + q * kTopkBins, k2, tmp, &sb);
    Rule rl{(beta << 20) | (static_cast<uint32_t>(b2.beta) << 8), 0xFFFFFF00u, k2 - b2.above, 0u};
    rl.done = (b2.beta >= 0 && b2.hb == rl.k_rem) ? 1u : 0u;
    if (!mbar_wait(&bar_l, 0, a.budget, nullptr)) {
      raise_flag(at.errw, kFlagTimeout);
      mbar_wait(&bar_l, 0, kDrainBudget, nullptr);
    }
    // candidate c of rank i
    auto cand_at = [&](int i, int c) -> uint2 {
      return staged ? lists[i * kCandP + c] : gl_all[static_cast<long long>(i) * E + c];
    };
    if (!rl.done) {
      // the last 8 bits among the keys with this 24-bit prefix (few keys)
      __shared__ uint32_t hbin[256];
      if (tid < 256) hbin[tid] = 0u;
      if (tid == 0) rule = rl;
      __syncthreads();
      for (int i = 0; i < kC; ++i) {
        const int n = static_cast<int>(rcnt[i]);
        for (int c = tid; c < n; c += kT) {
          const uint32_t key = cand_at(i, c).x;
          if ((key & rl.mask) == rl.prefix) atomicAdd(&hbin[key & 255u], 1u);
        }
      }
      __syncthreads();
      pick_digit<kT>(hbin, rl, 0, tmp, &rule);
      rl = rule;
      __syncthreads();
    }
    // ordered compaction: warp w walks ranks [w*RPW, (w+1)*RPW) (index order)
    constexpr int NW = kT / 32, RPW = kC / NW;
    uint32_t ngt = 0, neq = 0;
    for (int i = warp * RPW; i < (warp + 1) * RPW; ++i) {
      const int n = static_cast<int>(rcnt[i]);
      for (int base = 0; base < n; base += 32) {
        const int c = base + lane;
        const uint32_t key = c < n ? cand_at(i, c).x & rl.mask : 0u;
        ngt += __popc(__ballot_sync(0xffffffffu, c < n && key > rl.prefix));
        neq += __popc(__ballot_sync(0xffffffffu, c < n && key == rl.prefix));
      }
    }
    if (lane == 0) {
      wg[warp] = ngt;
      we[warp] = neq;
    }
    __syncthreads();
    uint32_t run_gt = 0, run_eq = 0;
    for (int w = 0; w < warp; ++w) {
      run_gt += wg[w];
      run_eq += we[w];
    }
    const unsigned ltm = lanemask_lt();
    const int p_lo = r * S_r, p_hi = p_lo + S_r;
    // this warp's kept candidates take the output positions [w_lo, w_hi)
    // (in index order); a warp whose range misses this CTA's slots has
    // nothing to write here
    const uint32_t w_lo = run_gt + min(run_eq, rl.k_rem);
    const uint32_t w_hi = run_gt + wg[warp] + min(run_eq + we[warp], rl.k_rem);
    const bool overlaps = w_lo < w_hi && static_cast<int>(w_lo) < p_hi && static_cast<int>(w_hi) > p_lo;
    for (int i = warp * RPW; overlaps && i < (warp + 1) * RPW; ++i) {
      const int n = static_cast<int>(rcnt[i]);
      for (int base = 0; base < n; base += 32) {
        const int c = base + lane;
        const uint2 cv = c < n ? cand_at(i, c) : make_uint2(0u, 0u);
        const uint32_t key = cv.x & rl.mask;
        const bool gt = c < n && key > rl.prefix;
        const bool eq = c < n && key == rl.prefix;
        const unsigned bgt = __ballot_sync(0xffffffffu, gt);
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        const uint32_t gt_b = run_gt + __popc(bgt & ltm);
        const uint32_t eq_b = run_eq + __popc(beq & ltm);
        if (gt || (eq && eq_b < rl.k_rem)) {
          const int pos = static_cast<int>(gt_b + min(eq_b, rl.k_rem));
          if (pos >= p_lo && pos < p_hi && pos < k) {  // this CTA attends that rank and reports it
            map[pos - p_lo] = static_cast<int>(cv.y);
            if (a.idx_out) a.idx_out[q * k + pos] = static_cast<int32_t>(cv.y);
            if (a.score_out) a.score_out[q * k + pos] = key_score(cv.x);
          }
        }
        run_gt += __popc(bgt);
        run_eq += __popc(beq);
      }
    }
  }
  __syncthreads();  // this CTA's map is complete

  // ---- 3. attention over this CTA's key slots
  if (r < A) {
    int* codes = reinterpret_cast<int*>(smem + L.codes);
    const int s0 = r * S_r;
    const char* kr_base = static_cast<const char*>(at.k_raw) + static_cast<size_t>(b) * at.T_raw * D * 2;
    const char* vr_base = static_cast<const char*>(at.v_raw) + static_cast<size_t>(b) * at.T_raw * D * 2;
    bool bad = false;
    // slot codes: kept blocks, then window rows, then nothing (one slot per
    // thread: S_r <= kT)
    int my_code = -1;
    if (tid < S_r) {
      const int s = s0 + tid;
      if (s < k) {
        my_code = all ? (s < n_vis ? s : -1) : map[tid];
      } else if (s < K_total) {
        const int u = t - at.W + 1 + (s - k);
        if (u >= 0) {
          const int rr = u - raw_base;
          if (rr < 0 || rr >= at.T_raw)
            bad = true;
          else
            my_code = -rr - 2;
        }
      }
      codes[tid] = my_code;
    }
    if (bad) raise_flag(at.errw, kFlagIndex);
    // each slot's K and V rows: all 256 threads load 16-byte chunks
    // (consecutive threads on consecutive chunks of a row; every load of a
    // thread issued before the first store) and store them into the padded
    // rows; an empty slot's rows are zeroed (its probability is 0, and
    // 0 * garbage could be NaN)
    __syncthreads();  // codes[] written
    {
      constexpr int NPT = (kTailMaxSlots * CH + kT - 1) / kT;  // chunks per thread at most
      uint4 kv[NPT][2];
#pragma unroll
      for (int u = 0; u < NPT; ++u) {
        const int i = tid + u * kT;
        kv[u][0] = kv[u][1] = make_uint4(0u, 0u, 0u, 0u);
        if (i < S_r * CH) {
          const int rw = i / CH, ch = i % CH;
          const int code = codes[rw];
          if (code != -1) {
            const char* kp = code >= 0 ? kc_base + static_cast<size_t>(code) * D * 2
                                       : kr_base + static_cast<size_t>(-code - 2) * D * 2;
            const char* vp = code >= 0 ? vc_base + static_cast<size_t>(code) * D * 2
                                       : vr_base + static_cast<size_t>(-code - 2) * D * 2;
            kv[u][0] = __ldg(reinterpret_cast<const uint4*>(kp + ch * 16));
            kv[u][1] = __ldg(reinterpret_cast<const uint4*>(vp + ch * 16));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < NPT; ++u) {
        const int i = tid + u * kT;
        if (i < S_r * CH) {
          const int rw = i / CH, ch = i % CH;
          *reinterpret_cast<uint4*>(Ks + rw * PITCH + ch * 16) = kv[u][0];
          *reinterpret_cast<uint4*>(Vs + rw * PITCH + ch * 16) = kv[u][1];
        }
      }
    }
    // Q fragments of head group hg (rows hg*16 + g and + 8) from shared memory
    const int hg = warp & 3, kh = warp >> 2;
    const int g = lane >> 2, c = lane & 3;
    const int h0 = hg * 16 + g, h1 = h0 + 8;
    if (!mbar_wait(&bar_q, 0, a.budget, nullptr)) {
      raise_flag(at.errw, kFlagTimeout);
      mbar_wait(&bar_q, 0, kDrainBudget, nullptr);
    }
    uint32_t qf[D / 16][4];
    {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(qs + static_cast<size_t>(h0) * D * 2);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(qs + static_cast<size_t>(h1) * D * 2);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qf[kk][0] = h0 < H ? q0[kk * 8 + c] : 0u;
        qf[kk][1] = h1 < H ? q1[kk * 8 + c] : 0u;
        qf[kk][2] = h0 < H ? q0[kk * 8 + 4 + c] : 0u;
        qf[kk][3] = h1 < H ? q1[kk * 8 + 4 + c] : 0u;
      }
    }
    float o[DT][4];
#pragma unroll
    for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl2 = at.scale * kLog2e;
    __syncthreads();  // every slot's rows stored
    if (hg * 16 < H) {
      const int half = S_r / 2;
      for (int kb = 0; kb < half; kb += KH)
        tile_step<D, KH, PITCH>(qf, Ks, Vs, kh * half + kb, codes + kh * half + kb, sl2, o, m0, m1, l0, l1);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();  // the K/V tile is consumed; the merge area overlaps it
    // the two key halves of head group hg merge in registers: the half-1
    // warp leaves its (o, m, l) in shared memory, the half-0 warp (named
    // barrier 1 + hg between the pair) merges them with its own and sends
    // its 16 heads' partials to their owner CTAs, one float4 per lane and
    // column block (a lane pair assembles it by one exchange)
    float* xo = reinterpret_cast<float*>(smem + L.merge);  // [H][LDO] half-1 partials
    float* xm = xo + H * LDO;                              // [H]
    float* xl = xm + H;                                    // [H]
    if (hg * 16 < H && kh == 1) {
#pragma unroll
      for (int i = 0; i < DT; ++i) {
        const int col = 8 * i + 2 * c;
        if (h0 < H) *reinterpret_cast<float2*>(xo + h0 * LDO + col) = make_float2(o[i][0], o[i][1]);
        if (h1 < H) *reinterpret_cast<float2*>(xo + h1 * LDO + col) = make_float2(o[i][2], o[i][3]);
      }
      if (c == 0) {
        if (h0 < H) {
          xm[h0] = m0;
          xl[h0] = l0;
        }
        if (h1 < H) {
          xm[h1] = m1;
          xl[h1] = l1;
        }
      }
    }
    if (hg * 16 < H) asm volatile("bar.sync %0, 64;" ::"r"(1 + hg) : "memory");
    if (hg * 16 < H && kh == 0) {
      // per row: the merged max, the halves' weights and the merged sum
      float fa[2], fb[2], Mx[2], Lx[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int h = hr == 0 ? h0 : h1;
        const float ma = hr == 0 ? m0 : m1, la = hr == 0 ? l0 : l1;
        const float mb = h < H ? xm[h] : -INFINITY, lb = h < H ? xl[h] : 0.f;
        const float M = fmaxf(ma, mb);
        const float R = M == -INFINITY ? 0.f : M;
        fa[hr] = ex2(ma - R);
        fb[hr] = ex2(mb - R);
        Mx[hr] = M;
        Lx[hr] = fa[hr] * la + fb[hr] * lb;
      }
      const bool even = (c & 1) == 0;
      // even lanes send row h0's column block 8i + 2c .. + 3, odd lanes row h1's
      const int hs = even ? h0 : h1;
      const int owner = hs / L.hpc, hl = hs - owner * L.hpc;
      float* dst = cluster.map_shared_rank(recv + (hl * kC + r) * LDO, owner);
#pragma unroll
      for (int i = 0; i < DT; ++i) {
        const int col = 8 * i + 2 * c;
        const float2 b0 = h0 < H ? *reinterpret_cast<const float2*>(xo + h0 * LDO + col) : make_float2(0.f, 0.f);
        const float2 b1 = h1 < H ? *reinterpret_cast<const float2*>(xo + h1 * LDO + col) : make_float2(0.f, 0.f);
        const float v0 = fa[0] * o[i][0] + fb[0] * b0.x, v1 = fa[0] * o[i][1] + fb[0] * b0.y;
        const float v2 = fa[1] * o[i][2] + fb[1] * b1.x, v3 = fa[1] * o[i][3] + fb[1] * b1.y;
        const float s0 = __shfl_xor_sync(0xffffffffu, even ? v2 : v0, 1);
        const float s1 = __shfl_xor_sync(0xffffffffu, even ? v3 : v1, 1);
        if (hs < H)
          *reinterpret_cast<float4*>(dst + (even ? col : col - 2)) =
              even ? make_float4(v0, v1, s0, s1) : make_float4(s0, s1, v2, v3);
      }
      if (c == 0) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int h = hr == 0 ? h0 : h1;
          if (h < H) {
            const int ow = h / L.hpc, hl2 = h - ow * L.hpc;
            *cluster.map_shared_rank(recv_m + hl2 * kC + r, ow) = Mx[hr];
            *cluster.map_shared_rank(recv_l + hl2 * kC + r, ow) = Lx[hr];
          }
        }
      }
    }
  }
  cluster.sync();  // #4: every partial has arrived

  // ---- 4. this CTA's heads, from the A partials in rank order
  const int h_lo = r * L.hpc;
  const int nh = max(0, min(H, h_lo + L.hpc) - h_lo);
  for (int it = tid; it < nh * (D / 4); it += kT) {
    const int hl = it / (D / 4), col = 4 * (it % (D / 4));
    const int h = h_lo + hl;
    float M = -INFINITY;
    for (int p = 0; p < A; ++p) M = fmaxf(M, recv_m[hl * kC + p]);
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      for (int p = 0; p < A; ++p) {
        const float f = ex2(recv_m[hl * kC + p] - M);
        den = fmaf(f, recv_l[hl * kC + p], den);
        const float4 v = *reinterpret_cast<const float4*>(recv + (hl * kC + p) * LDO + col);
        acc.x = fmaf(f, v.x, acc.x);
        acc.y = fmaf(f, v.y, acc.y);
        acc.z = fmaf(f, v.z, acc.z);
        acc.w = fmaf(f, v.w, acc.w);
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    const long long o0 = (q * H + h) * static_cast<long long>(D) + col;
    if (at.out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(at.out) + o0) = acc;
    } else {
      uint2 pk;
      pk.x = pack_bf16x2(acc.x, acc.y);
      pk.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(at.out) + o0) = pk;
    }
    if (at.lse && col == 0) at.lse[q * H + h] = den > 0.f ? (M + __log2f(den)) * kLn2 : -INFINITY;
  }
}

}  // namespace

int tail_chunk(int N) { return ((N + kC - 1) / kC + 1023) / 1024 * 1024; }

int tail_slots(int k, int W) {
  const int per = (k + W + kC - 1) / kC;
  return (per + 31) / 32 * 32;
}

bool tail_supported(int Tq, int N, int k, int W, int H, int d) {
  // Only the call's per-sequence shape decides (never B), so a sequence gives
  // the same bits alone or inside any batch.  Up to kTailMinEntries entries
  // the separate kernels (select, finish, decode attention) spread a batch
  // over more of the GPU.
  return Tq < 16 && N > kTailMinEntries && topk_long_rows(N) && H >= 1 && H <= 64 &&
         (d == 64 || d == 128) && tail_slots(k, W) <= kTailMaxSlots && k + W > 0 &&
         tail_layout(kTailMaxSlots, 64, d, kT * kRun).total <= 220 * 1024;
}

cudaError_t launch_decode_tail(const TailArgs& a, cudaStream_t s) {
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (nq == 0) return cudaSuccess;
  if (nq > 65535) return cudaErrorNotSupported;
  const int E = tail_chunk(a.N);
  const int S_r = tail_slots(a.k, a.at.W);
  const TailLayout L = tail_layout(S_r, a.at.H, a.at.d, E);
  static std::atomic<bool> attr_set[4][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  // one tile step of S_r / 2 keys per warp for the common slot count, else steps of 16
  const bool kh48 = S_r == 96;
  const int which = (a.at.d == 128 ? 0 : 2) + (kh48 ? 1 : 0);
  auto kern = a.at.d == 128 ? (kh48 ? decode_tail_kernel<128, 48> : decode_tail_kernel<128, 16>)
                            : (kh48 ? decode_tail_kernel<64, 48> : decode_tail_kernel<64, 16>);
  if (!attr_set[which][dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    const TailLayout Lmax = tail_layout(kTailMaxSlots, 64, a.at.d, kT * kRun);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lmax.total);
    if (e != cudaSuccess) return e;
    attr_set[which][dev].store(true, std::memory_order_release);
  }
  return launch_k(kern, dim3(kC, static_cast<unsigned>(nq)), dim3(kT), static_cast<size_t>(L.total), s, kC, a,
                  E, S_r);
}

size_t tail_cand_bytes_per_query(int N) { return static_cast<size_t>(kC) * tail_chunk(N) * 8; }

}  // namespace csa

