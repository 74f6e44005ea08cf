// Internal launch interface between the C ABI (csa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace csa {

// cuTensorMapEncodeTiled, resolved from the driver at run time (nullptr when
// the driver does not provide it)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// ---- (1) compression -------------------------------------------------------
struct CompressArgs {
  const void* x[3];
  const void* g[3];
  void* out[3];
  int D[3];
  int n_streams;
  int B, T, m;
  int out_f32;
};
cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s);

// decode-time append: the blocks completed by the queries' positions, from
// the raw window rows into the caches (bf16)
struct AppendArgs {
  const void* x[3];  // [B, T_raw, D[i]] raw window rows
  const void* g[3];  // [B, T_raw, D[i]] their gate logits
  void* out[3];      // [B, N, D[i]] caches
  int D[3];
  int n_streams;
  const int32_t* raw_base;  // [B]
  const int32_t* q_pos;     // [B, Tq]
  int B, Tq, T_raw, N, m;
  uint32_t* errw;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);

// ---- (2) indexer scores ----------------------------------------------------
struct IndexerArgs {
  const void* q_idx;  // [B, Tq, H_I, d_I] bf16
  const void* k_idx;  // [B, N, d_I] bf16
  const float* w;     // [H_I] (w_stride == 0) or per query: w[(n * Tq + j) * w_stride + h]
  const int32_t* q_pos;
  float* scores;
  long long ld;
  int B, Tq, N, H_I, d_I, m;
  uint32_t* errw;
  long long budget;
  uint32_t* hist;  // [B*Tq][kTopkBins] top-k bucket histogram to accumulate into, or nullptr
  // 1 when the launch directly follows the library's histogram-zeroing
  // kernel, which itself waited for every earlier kernel: the indexer then
  // streams at once and waits for the zeroing only before its histogram flush
  int after_zero;
  long long w_stride;
  // FP8 indexer: q_idx and k_idx hold E4M3 codes ([B, Tq, H_I, d_I] and
  // [B, N, d_I], one byte each), q_scale [B * Tq * H_I] and k_scale [B, N]
  // the power-of-two scale of each row (d_I == 128, N % 4 == 0)
  int fp8;
  const float* q_scale;
  const float* k_scale;
};
// rows [rows][D] bf16 -> E4M3 codes [rows][D] and one power-of-two scale per row
cudaError_t launch_quantize_fp8(const void* x, long long rows, int D, void* codes, float* scales, cudaStream_t s);
bool indexer_fp8_supported(int H_I, int d_I, int N);
// returns cudaErrorNotSupported for shapes outside the instantiated set
cudaError_t launch_indexer(const IndexerArgs& a, cudaStream_t s);
// whether launch_indexer fills IndexerArgs::hist for this shape (else it is ignored)
bool indexer_fills_hist(int Tq, int H_I);

// ---- (3) top-k --------------------------------------------------------------
constexpr int kTopkBins = 4096;        // buckets of 12 key bits (two levels: bits 31..20, 19..8)
constexpr int kTopkChunk = 4096;       // keys per candidate-select CTA (long rows)
constexpr int kTopkShortMax = 16384;   // rows up to this length are selected in shared memory
constexpr int kTopkMidMax = 32768;     // longer rows up to this length: one CTA per query from the histogram
constexpr int kTopkMaxN = 1 << 24;

struct TopkArgs {
  const float* scores;
  long long ld;
  const int32_t* q_pos;
  int B, Tq, N, m, k;
  int32_t* idx_out;
  float* score_out;
  // long-row scratch (topk_scratch_carve): the bucket histograms (key bits
  // 31..20, 19..8 and 7..0), and per chunk a candidate count and a candidate
  // list of (key, index) pairs
  uint32_t* hist;
  uint32_t* hist2;
  uint32_t* hist3;
  uint32_t* ccount;
  uint2* cand;
};
bool topk_supported(int N);
bool topk_long_rows(int N);
// bytes of long-row scratch for nq queries (0 for short rows), and of its
// leading part that must be zero before the histogram is accumulated
size_t topk_scratch_bytes(long long nq, int N);
size_t topk_scratch_zero_bytes(long long nq);
void topk_scratch_carve(TopkArgs& a, void* base, long long nq);
// hist_ready: the histogram was already accumulated (by the indexer) into a
// zeroed scratch; otherwise the scratch is zeroed and the histogram built here.
cudaError_t launch_topk(const TopkArgs& a, bool hist_ready, cudaStream_t s);
// zero the leading (histogram) part of the long-row scratch carved into ``a``
cudaError_t launch_topk_zero(const TopkArgs& a, long long nq, cudaStream_t s);

// ---- (4) attention ----------------------------------------------------------
struct AttendArgs {
  const void* q;
  const void* k_cmp;
  const void* v_cmp;
  const int32_t* idx;  // nullptr: HCA mode (every visible entry)
  const void* k_raw;
  const void* v_raw;
  const int32_t* raw_base;
  const int32_t* q_pos;
  int B, Tq, N, T_raw, H, d, k, W, m;
  float scale;
  void* out;
  int out_f32;
  float* lse;
  float* part;  // split partials (workspace), may be nullptr when nsplit == 1
  uint32_t* errw;
};
struct AttendPlan {
  int nsplit;
  int tiles_per_split;
  // 0: one split; 1: split partials in the workspace + combine kernel; 2: cluster merge;
  // 3: decode kernel (key ranges x 16-head groups, cluster merge)
  int mode;
  int nw;    // warps per CTA: 4 (64-key tiles) or 8 (128-key tiles)
  size_t part_bytes;
};
AttendPlan plan_attend(int Tq, long long nq, int n_keys_max, int H, int d);
cudaError_t launch_attend(const AttendArgs& a, const AttendPlan& plan, cudaStream_t s);
// merge nsplit partials per (query, head) from a.part, in split order, into a.out / a.lse
cudaError_t launch_attend_combine(const AttendArgs& a, int nsplit, cudaStream_t s);

// ---- decode attention on tcgen05 (H = 64, d = 128, Tq < 16) -----------------
// CSA (a.idx != nullptr): the k listed rows and the W window rows, gathered
// with cp.async; HCA (a.idx == nullptr): every visible entry and the window as
// TMA tiles.  One CTA per (query, range of up to kTcTiles (CSA) or
// kTcTilesHca (HCA) 128-key tiles); the ranges of a query merge inside their
// cluster (up to eight) or through workspace partials.
constexpr int kTcTiles = 5;
constexpr int kTcTilesHca = 4;
struct TcPlan {
  int nsplit;  // ranges per query
  int tpr;     // tiles per range
};
int attend_tc_tiles(bool csa, int N, int k, int W);  // tiles of the longest key list
TcPlan attend_tc_plan(int n_tiles, bool csa);
bool attend_tc_supported(bool csa, int Tq, long long nq, int N, int T_raw, int k, int H, int d, int W);
size_t attend_tc_part_bytes(long long nq, int H, int d, const TcPlan& p);
cudaError_t launch_attend_tc(const AttendArgs& a, long long wait_budget, cudaStream_t s);

// ---- fused decode tail: long-row top-k + attention, one cluster per query -------
constexpr int kTailCluster = 16;    // CTAs per query
constexpr int kTailMaxSlots = 128;  // key slots attended by one CTA
constexpr int kTailMinEntries = 65536;  // decode calls with more entries per sequence use the fused tail
struct TailArgs {
  const float* scores;  // [B*Tq][ld] indexer scores
  long long ld;
  const int32_t* q_pos;
  int B, Tq, N, m, k;
  const uint32_t* hist;  // [B*Tq][kTopkBins] bucket histogram of the visible scores
  uint32_t* hist2;       // [B*Tq][kTopkBins] zeroed: second level (key bits 19..8)
  uint32_t* hist3;       // [B*Tq][256] zeroed: third level (key bits 7..0)
  uint2* cand;           // [B*Tq][kTailCluster][tail_chunk(N)] candidate lists
  int32_t* idx_out;      // [B*Tq][k] or nullptr
  float* score_out;      // [B*Tq][k] or nullptr
  AttendArgs at;         // queries, caches, window, output (at.idx unused)
  long long budget;      // clock64 budget of each bounded wait
};
int tail_chunk(int N);
int tail_slots(int k, int W);
bool tail_supported(int Tq, int N, int k, int W, int H, int d);
size_t tail_cand_bytes_per_query(int N);
cudaError_t launch_decode_tail(const TailArgs& a, cudaStream_t s);
// the zeroing and histogram pass of the long-row top-k alone (for callers
// whose indexer did not accumulate the histogram)
cudaError_t launch_topk_hist(const TopkArgs& a, cudaStream_t s);

}  // namespace csa
