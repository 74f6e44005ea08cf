// C ABI of the CSA library (declared in include/csa.h): argument checks that
// run before anything is enqueued, workspace layout, and kernel dispatch.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/csa.h"
#include "common.cuh"
#include "kernels.h"

namespace {

long long g_wait_budget = 1LL << 31;  // clock64 cycles, about one second

// Instrumentation: events recorded around the next indexer launches of this
// host thread (csa_set_indexer_events).
thread_local cudaEvent_t t_idx_ev_begin = nullptr;
thread_local cudaEvent_t t_idx_ev_end = nullptr;

// (cudaEventRecordExternal: inside a stream capture the record becomes an
// event-record node of the graph, not a capture-internal dependency)
cudaError_t launch_indexer_marked(const csa::IndexerArgs& a, cudaStream_t s) {
  if (t_idx_ev_begin) {
    cudaError_t e = cudaEventRecordWithFlags(t_idx_ev_begin, s, cudaEventRecordExternal);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = csa::launch_indexer(a, s);
  if (e == cudaSuccess && t_idx_ev_end) e = cudaEventRecordWithFlags(t_idx_ev_end, s, cudaEventRecordExternal);
  return e;
}

constexpr size_t kAlignWs = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline csa_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CSA_OK;
  if (e == cudaErrorNotSupported) return CSA_ERR_UNSUPPORTED;
  return CSA_ERR_CUDA;
}

inline csa_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlignWs) != 0) return CSA_ERR_WORKSPACE;
  if (ws_bytes < need) return CSA_ERR_WORKSPACE;
  return CSA_OK;
}

inline uint32_t* err_word(void* ws) { return static_cast<uint32_t*>(ws); }

inline long long scores_ld(int N) { return (static_cast<long long>(N) + 3) / 4 * 4; }

inline size_t scores_bytes(int B, int Tq, int N) {
  return align_up(static_cast<size_t>(B) * Tq * scores_ld(N) * sizeof(float), kAlignWs);
}

bool hi_ok(int H_I) {
  return H_I == 4 || H_I == 8 || H_I == 16 || H_I == 32 || H_I == 64 || H_I == 128;
}
bool di_ok(int d_I) { return d_I == 32 || d_I == 64 || d_I == 128; }

csa_status check_index_args(const void* q_idx, const void* k_idx, const float* w,
                            const int32_t* q_pos, int B, int Tq, int N, int H_I, int d_I, int m) {
  if (!q_idx || !k_idx || !w || !q_pos) return CSA_ERR_INVALID;
  if (!al16(q_idx) || !al16(k_idx) || !al4(w) || !al4(q_pos)) return CSA_ERR_INVALID;
  if (B <= 0 || Tq <= 0 || N <= 0 || H_I <= 0 || d_I <= 0 || m <= 0) return CSA_ERR_INVALID;
  if (!hi_ok(H_I) || !di_ok(d_I)) return CSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Tq * H_I >= (1LL << 31)) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

csa_status check_topk_shape(const int32_t* q_pos, int B, int Tq, int N, int m, int k) {
  if (!q_pos || !al4(q_pos)) return CSA_ERR_INVALID;
  if (B <= 0 || Tq <= 0 || N <= 0 || m <= 0 || k <= 0) return CSA_ERR_INVALID;
  if (k > 4096) return CSA_ERR_UNSUPPORTED;
  if (!csa::topk_supported(N)) return CSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Tq >= (1LL << 31)) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

csa_status check_topk_args(const int32_t* q_pos, int B, int Tq, int N, int m, int k,
                           const int32_t* idx_out, const float* score_out) {
  if (!idx_out || !al4(idx_out) || (score_out && !al4(score_out))) return CSA_ERR_INVALID;
  return check_topk_shape(q_pos, B, Tq, N, m, k);
}

csa_status check_attend_args(const void* q, const void* k_cmp, const void* v_cmp, const void* k_raw,
                             const void* v_raw, const int32_t* raw_base, const int32_t* q_pos,
                             int B, int Tq, int N, int T_raw, int H, int d, int W, const void* out,
                             int out_dtype, const float* lse) {
  if (!q || !q_pos || !out) return CSA_ERR_INVALID;
  if (B <= 0 || Tq <= 0 || N < 0 || T_raw < 0 || H <= 0 || d <= 0 || W < 0) return CSA_ERR_INVALID;
  if (N > 0 && (!k_cmp || !v_cmp)) return CSA_ERR_INVALID;
  if (W > 0 && (!k_raw || !v_raw || !raw_base || T_raw <= 0)) return CSA_ERR_INVALID;
  if (!al16(q) || !al16(out) || (k_cmp && !al16(k_cmp)) || (v_cmp && !al16(v_cmp)) ||
      (k_raw && !al16(k_raw)) || (v_raw && !al16(v_raw)) || !al4(q_pos) ||
      (raw_base && !al4(raw_base)) || (lse && !al4(lse)))
    return CSA_ERR_INVALID;
  if (out_dtype != CSA_BF16 && out_dtype != CSA_F32) return CSA_ERR_INVALID;
  if (d != 64 && d != 128) return CSA_ERR_UNSUPPORTED;
  if (H > 64) return CSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Tq >= 65536LL * 1024) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

size_t topk_bytes(int B, int Tq, int N) {
  return align_up(csa::topk_scratch_bytes(static_cast<long long>(B) * Tq, N), kAlignWs);
}

// Indexer (optionally filling the top-k histogram) then top-k, with the
// long-row scratch at ``tk``.
csa_status index_then_topk(const csa::IndexerArgs& ia_in, const csa::TopkArgs& ta_in, void* tk,
                           cudaStream_t s) {
  csa::IndexerArgs ia = ia_in;
  csa::TopkArgs ta = ta_in;
  const long long nq = static_cast<long long>(ta.B) * ta.Tq;
  bool fused = false;
  if (csa::topk_long_rows(ta.N)) {
    csa::topk_scratch_carve(ta, tk, nq);
    fused = csa::indexer_fills_hist(ia.Tq, ia.H_I);
    if (fused) {
      cudaError_t e = csa::launch_topk_zero(ta, nq, s);
      if (e != cudaSuccess) return CSA_ERR_CUDA;
      ia.hist = ta.hist;
      ia.after_zero = 1;
    }
  }
  csa_status st = cuda_status(launch_indexer_marked(ia, s));
  if (st != CSA_OK) return st;
  return cuda_status(csa::launch_topk(ta, fused, s));
}

size_t attend_part_bytes(int B, int Tq, int n_keys_max, int H, int d) {
  const csa::AttendPlan p = csa::plan_attend(Tq, static_cast<long long>(B) * Tq, n_keys_max, H, d);
  return align_up(p.part_bytes, kAlignWs);
}

// Attention partials: the tcgen05 decode kernel's range partials or the
// general kernels' split partials, whichever is larger (the raw-buffer length
// that can also decide between them is not an argument of the size queries)
size_t attn_part_bytes(bool csa_mode, int B, int Tq, int N, int k, int W, int H, int d) {
  const size_t gen = attend_part_bytes(B, Tq, (csa_mode ? k : N) + W, H, d);
  const long long nq = static_cast<long long>(B) * Tq;
  if (!csa::attend_tc_supported(csa_mode, Tq, nq, N, 1, k, H, d, W)) return gen;
  const csa::TcPlan p = csa::attend_tc_plan(csa::attend_tc_tiles(csa_mode, N, k, W), csa_mode);
  const size_t tc = align_up(csa::attend_tc_part_bytes(nq, H, d, p), kAlignWs);
  return gen > tc ? gen : tc;
}

// The attention kernel for a's shape: tcgen05 for decode-shaped calls with
// H = 64 and d = 128, the mma.sync kernels otherwise.
cudaError_t launch_attention(const csa::AttendArgs& a, cudaStream_t s) {
  const bool csa_mode = a.idx != nullptr;
  const long long nq = static_cast<long long>(a.B) * a.Tq;
  if (csa::attend_tc_supported(csa_mode, a.Tq, nq, a.N, a.T_raw, a.k, a.H, a.d, a.W))
    return csa::launch_attend_tc(a, g_wait_budget, s);
  const csa::AttendPlan plan = csa::plan_attend(a.Tq, nq, (csa_mode ? a.k : a.N) + a.W, a.H, a.d);
  return csa::launch_attend(a, plan, s);
}

}  // namespace

extern "C" {

const char* csa_status_string(int s) {
  switch (s) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID: return "CSA_ERR_INVALID";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA";
    case CSA_ERR_TIMEOUT: return "CSA_ERR_TIMEOUT";
    case CSA_ERR_DEVICE_INDEX: return "CSA_ERR_DEVICE_INDEX";
    default: return "CSA_ERR_UNKNOWN";
  }
}

int csa_version(void) { return 100; }

void csa_set_wait_budget(long long cycles) { g_wait_budget = cycles > 0 ? cycles : (1LL << 31); }

void csa_set_indexer_events(void* ev_begin, void* ev_end) {
  t_idx_ev_begin = static_cast<cudaEvent_t>(ev_begin);
  t_idx_ev_end = static_cast<cudaEvent_t>(ev_end);
}

csa_status csa_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES) != CSA_OK) return CSA_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, CSA_WS_HEADER_BYTES, static_cast<cudaStream_t>(stream)));
}

csa_status csa_check_error(const void* ws, uint32_t* flags, int clear, void* stream) {
  if (check_ws(ws, CSA_WS_HEADER_BYTES, CSA_WS_HEADER_BYTES) != CSA_OK) return CSA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t f = 0;
  cudaError_t e = cudaMemcpyAsync(&f, ws, sizeof(f), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(const_cast<void*>(ws), 0, sizeof(f), s);
  if (e == cudaSuccess && clear) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return CSA_ERR_CUDA;
  if (flags) *flags = f;
  if (f & CSA_FLAG_TIMEOUT) return CSA_ERR_TIMEOUT;
  if (f & CSA_FLAG_INDEX) return CSA_ERR_DEVICE_INDEX;
  return CSA_OK;
}

// ---------------------------------------------------------------- (1)
csa_status csa_compress(int n_streams, const void* const* x, const void* const* g, void* const* out,
                        const int* D, int B, int T, int m, int out_dtype, void* stream) {
  if (n_streams < 1 || n_streams > 3 || !x || !g || !out || !D) return CSA_ERR_INVALID;
  if (B <= 0 || T < 0 || m < 1 || m > 4096) return CSA_ERR_INVALID;
  if (out_dtype != CSA_BF16 && out_dtype != CSA_F32) return CSA_ERR_INVALID;
  const bool empty = T / m == 0;  // no complete block: nothing is read or written
  csa::CompressArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int i = 0; i < n_streams; ++i) {
    if (D[i] <= 0 || D[i] % 8 != 0 || D[i] > 512) return CSA_ERR_INVALID;
    if (empty) continue;
    if (!x[i] || !g[i] || !out[i]) return CSA_ERR_INVALID;
    if (!al16(x[i]) || !al16(g[i]) || !al16(out[i])) return CSA_ERR_INVALID;
    a.x[i] = x[i];
    a.g[i] = g[i];
    a.out[i] = out[i];
    a.D[i] = D[i];
  }
  if (empty) return CSA_OK;
  a.n_streams = n_streams;
  a.B = B;
  a.T = T;
  a.m = m;
  a.out_f32 = out_dtype == CSA_F32;
  return cuda_status(csa::launch_compress(a, static_cast<cudaStream_t>(stream)));
}

csa_status csa_append(int n_streams, const void* const* x_win, const void* const* g_win, void* const* out,
                      const int* D, const int32_t* raw_base, const int32_t* q_pos, int B, int Tq, int T_raw,
                      int N, int m, void* ws, size_t ws_bytes, void* stream) {
  if (n_streams < 1 || n_streams > 3 || !x_win || !g_win || !out || !D) return CSA_ERR_INVALID;
  if (!raw_base || !q_pos || !al4(raw_base) || !al4(q_pos)) return CSA_ERR_INVALID;
  if (B <= 0 || Tq <= 0 || N <= 0 || m < 1 || m > 4096 || T_raw < m) return CSA_ERR_INVALID;
  csa::AppendArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int i = 0; i < n_streams; ++i) {
    if (D[i] <= 0 || D[i] % 8 != 0 || D[i] > 512) return CSA_ERR_INVALID;
    if (!x_win[i] || !g_win[i] || !out[i] || !al16(x_win[i]) || !al16(g_win[i]) || !al16(out[i]))
      return CSA_ERR_INVALID;
    a.x[i] = x_win[i];
    a.g[i] = g_win[i];
    a.out[i] = out[i];
    a.D[i] = D[i];
  }
  const csa_status st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES);
  if (st != CSA_OK) return st;
  a.n_streams = n_streams;
  a.raw_base = raw_base;
  a.q_pos = q_pos;
  a.B = B;
  a.Tq = Tq;
  a.T_raw = T_raw;
  a.N = N;
  a.m = m;
  a.errw = err_word(ws);
  return cuda_status(csa::launch_append(a, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- (2)
csa_status csa_index_scores(const void* q_idx, const void* k_idx, const float* w, int64_t w_stride,
                            const int32_t* q_pos, int B, int Tq, int N, int H_I, int d_I, int m,
                            float* scores, int64_t ld_scores, void* ws, size_t ws_bytes,
                            void* stream) {
  csa_status st = check_index_args(q_idx, k_idx, w, q_pos, B, Tq, N, H_I, d_I, m);
  if (st != CSA_OK) return st;
  if (w_stride != 0 && w_stride < H_I) return CSA_ERR_INVALID;
  if (!scores || !al16(scores) || ld_scores < N || ld_scores % 4 != 0) return CSA_ERR_INVALID;
  st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES);
  if (st != CSA_OK) return st;
  csa::IndexerArgs a{q_idx, k_idx, w, q_pos, scores, ld_scores, B, Tq, N, H_I, d_I, m,
                     err_word(ws), g_wait_budget, nullptr, 0, w_stride};
  return cuda_status(launch_indexer_marked(a, static_cast<cudaStream_t>(stream)));
}

csa_status csa_quantize_fp8(const void* x, int64_t rows, int D, void* codes, float* scales, void* stream) {
  if (!x || !codes || !scales || rows <= 0) return CSA_ERR_INVALID;
  if (D != 32 && D != 64 && D != 128 && D != 256) return CSA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) & 1u) || (reinterpret_cast<uintptr_t>(codes) & 1u) || !al4(scales))
    return CSA_ERR_INVALID;
  return cuda_status(csa::launch_quantize_fp8(x, rows, D, codes, scales, static_cast<cudaStream_t>(stream)));
}

csa_status csa_index_scores_fp8(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                                const float* w, int64_t w_stride, const int32_t* q_pos, int B, int Tq, int N,
                                int H_I, int d_I, int m, float* scores, int64_t ld_scores, void* ws,
                                size_t ws_bytes, void* stream) {
  csa_status st = check_index_args(q8, k8, w, q_pos, B, Tq, N, H_I, d_I, m);
  if (st != CSA_OK) return st;
  if (!q_scale || !k_scale || !al16(q_scale) || !al16(k_scale)) return CSA_ERR_INVALID;
  if (!csa::indexer_fp8_supported(H_I, d_I, N)) return CSA_ERR_UNSUPPORTED;
  if (w_stride != 0 && w_stride < H_I) return CSA_ERR_INVALID;
  if (!scores || !al16(scores) || ld_scores < N || ld_scores % 4 != 0) return CSA_ERR_INVALID;
  st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES);
  if (st != CSA_OK) return st;
  csa::IndexerArgs a{q8, k8, w, q_pos, scores, ld_scores, B, Tq, N, H_I, d_I, m,
                     err_word(ws), g_wait_budget, nullptr, 0, w_stride, 1, q_scale, k_scale};
  return cuda_status(launch_indexer_marked(a, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- (3)
csa_status csa_topk(const float* scores, int64_t ld_scores, const int32_t* q_pos, int B, int Tq,
                    int N, int m, int k, int32_t* idx_out, float* score_out, void* ws,
                    size_t ws_bytes, void* stream) {
  csa_status st = check_topk_args(q_pos, B, Tq, N, m, k, idx_out, score_out);
  if (st != CSA_OK) return st;
  if (!scores || !al16(scores) || ld_scores < N || ld_scores % 4 != 0) return CSA_ERR_INVALID;
  st = check_ws(ws, ws_bytes, CSA_WS_HEADER_BYTES + topk_bytes(B, Tq, N));
  if (st != CSA_OK) return st;
  csa::TopkArgs a{scores, ld_scores, q_pos, B, Tq, N, m, k, idx_out, score_out, nullptr, nullptr, nullptr, nullptr, nullptr};
  if (csa::topk_long_rows(N))
    csa::topk_scratch_carve(a, static_cast<char*>(ws) + CSA_WS_HEADER_BYTES, static_cast<long long>(B) * Tq);
  return cuda_status(csa::launch_topk(a, false, static_cast<cudaStream_t>(stream)));
}

csa_status csa_topk_workspace(int B, int Tq, int N, int k, size_t* bytes) {
  (void)k;
  if (!bytes || B <= 0 || Tq <= 0 || N <= 0) return CSA_ERR_INVALID;
  *bytes = CSA_WS_HEADER_BYTES + topk_bytes(B, Tq, N);
  return CSA_OK;
}

csa_status csa_index_topk_workspace(int B, int Tq, int N, int H_I, int d_I, int k, size_t* bytes) {
  (void)H_I;
  (void)d_I;
  (void)k;
  if (!bytes || B <= 0 || Tq <= 0 || N <= 0) return CSA_ERR_INVALID;
  *bytes = CSA_WS_HEADER_BYTES + scores_bytes(B, Tq, N) + topk_bytes(B, Tq, N);
  return CSA_OK;
}

csa_status csa_index_topk(const void* q_idx, const void* k_idx, const float* w, int64_t w_stride,
                          const int32_t* q_pos, int B, int Tq, int N, int H_I, int d_I, int m,
                          int k, int32_t* idx_out, float* score_out, void* ws, size_t ws_bytes,
                          void* stream) {
  csa_status st = check_index_args(q_idx, k_idx, w, q_pos, B, Tq, N, H_I, d_I, m);
  if (st != CSA_OK) return st;
  if (w_stride != 0 && w_stride < H_I) return CSA_ERR_INVALID;
  st = check_topk_args(q_pos, B, Tq, N, m, k, idx_out, score_out);
  if (st != CSA_OK) return st;
  size_t need = 0;
  csa_index_topk_workspace(B, Tq, N, H_I, d_I, k, &need);
  st = check_ws(ws, ws_bytes, need);
  if (st != CSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* S = reinterpret_cast<float*>(static_cast<char*>(ws) + CSA_WS_HEADER_BYTES);
  const long long ld = scores_ld(N);
  csa::IndexerArgs ia{q_idx, k_idx, w, q_pos, S, ld, B, Tq, N, H_I, d_I, m, err_word(ws), g_wait_budget, nullptr, 0,
                      w_stride};
  csa::TopkArgs ta{S, ld, q_pos, B, Tq, N, m, k, idx_out, score_out, nullptr, nullptr, nullptr, nullptr, nullptr};
  return index_then_topk(ia, ta, reinterpret_cast<char*>(S) + scores_bytes(B, Tq, N), s);
}

// ---------------------------------------------------------------- (4)
csa_status csa_attend_workspace(int B, int Tq, int H, int d, int k, int W, size_t* bytes) {
  if (!bytes || B <= 0 || Tq <= 0 || H <= 0 || d <= 0 || k < 0 || W < 0) return CSA_ERR_INVALID;
  *bytes = CSA_WS_HEADER_BYTES + attn_part_bytes(true, B, Tq, 1, k, W, H, d);
  return CSA_OK;
}

static csa_status attend_common(const void* q, const void* k_cmp, const void* v_cmp,
                                const int32_t* idx, const void* k_raw, const void* v_raw,
                                const int32_t* raw_base, const int32_t* q_pos, int B, int Tq, int N,
                                int T_raw, int H, int d, int k, int m, int W, float scale, void* out,
                                int out_dtype, float* lse, void* ws, size_t ws_bytes, void* stream) {
  const size_t need = CSA_WS_HEADER_BYTES + attn_part_bytes(idx != nullptr, B, Tq, N, k, W, H, d);
  csa_status st = check_ws(ws, ws_bytes, need);
  if (st != CSA_OK) return st;
  csa::AttendArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.k_cmp = k_cmp;
  a.v_cmp = v_cmp;
  a.idx = idx;
  a.k_raw = k_raw;
  a.v_raw = v_raw;
  a.raw_base = raw_base;
  a.q_pos = q_pos;
  a.B = B;
  a.Tq = Tq;
  a.N = N;
  a.T_raw = T_raw;
  a.H = H;
  a.d = d;
  a.k = k;
  a.W = W;
  a.m = m;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  a.out = out;
  a.out_f32 = out_dtype == CSA_F32;
  a.lse = lse;
  a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + CSA_WS_HEADER_BYTES);
  a.errw = err_word(ws);
  return cuda_status(launch_attention(a, static_cast<cudaStream_t>(stream)));
}

csa_status csa_attend(const void* q, const void* k_cmp, const void* v_cmp, const int32_t* idx,
                      const void* k_raw, const void* v_raw, const int32_t* raw_base,
                      const int32_t* q_pos, int B, int Tq, int N, int T_raw, int H, int d, int k,
                      int W, float scale, void* out, int out_dtype, float* lse, void* ws,
                      size_t ws_bytes, void* stream) {
  csa_status st = check_attend_args(q, k_cmp, v_cmp, k_raw, v_raw, raw_base, q_pos, B, Tq, N, T_raw,
                                    H, d, W, out, out_dtype, lse);
  if (st != CSA_OK) return st;
  if (k < 0 || (k > 0 && (!idx || !al4(idx)))) return CSA_ERR_INVALID;
  if (k > 0 && N <= 0) return CSA_ERR_INVALID;
  // k == 0 leaves only the window; any non-null pointer keeps the call in CSA
  // mode (the index list is empty and never read)
  return attend_common(q, k_cmp, v_cmp, idx ? idx : q_pos, k_raw,
                       v_raw, raw_base, q_pos, B, Tq, N, T_raw, H, d, k, 1, W, scale, out,
                       out_dtype, lse, ws, ws_bytes, stream);
}

csa_status hca_attend_workspace(int B, int Tq, int N, int H, int d, int W, size_t* bytes) {
  if (!bytes || B <= 0 || Tq <= 0 || N < 0 || H <= 0 || d <= 0 || W < 0) return CSA_ERR_INVALID;
  *bytes = CSA_WS_HEADER_BYTES + attn_part_bytes(false, B, Tq, N, 0, W, H, d);
  return CSA_OK;
}

csa_status hca_attend(const void* q, const void* k_cmp, const void* v_cmp, const void* k_raw,
                      const void* v_raw, const int32_t* raw_base, const int32_t* q_pos, int B,
                      int Tq, int N, int T_raw, int H, int d, int m, int W, float scale, void* out,
                      int out_dtype, float* lse, void* ws, size_t ws_bytes, void* stream) {
  csa_status st = check_attend_args(q, k_cmp, v_cmp, k_raw, v_raw, raw_base, q_pos, B, Tq, N, T_raw,
                                    H, d, W, out, out_dtype, lse);
  if (st != CSA_OK) return st;
  if (m <= 0) return CSA_ERR_INVALID;
  return attend_common(q, k_cmp, v_cmp, nullptr, k_raw, v_raw, raw_base, q_pos, B, Tq, N, T_raw, H,
                       d, 0, m, W, scale, out, out_dtype, lse, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- layer
// FP8 indexer: the step's indexer queries as E4M3 codes, then their scales
static size_t fp8_query_codes_bytes(const csa_layer_args* a) {
  return align_up(static_cast<size_t>(a->B) * a->Tq * a->H_I * a->d_I, kAlignWs);
}
static size_t fp8_query_bytes(const csa_layer_args* a) {
  return fp8_query_codes_bytes(a) + align_up(static_cast<size_t>(a->B) * a->Tq * a->H_I * 4, kAlignWs);
}

csa_status csa_layer_workspace(const csa_layer_args* a, size_t* bytes) {
  if (!a || !bytes || a->B <= 0 || a->Tq <= 0 || a->N <= 0 || a->k <= 0) return CSA_ERR_INVALID;
  size_t total = CSA_WS_HEADER_BYTES + scores_bytes(a->B, a->Tq, a->N) + topk_bytes(a->B, a->Tq, a->N);
  if (!a->idx_out) total += align_up(static_cast<size_t>(a->B) * a->Tq * a->k * 4, kAlignWs);
  if (a->i_scale) total += fp8_query_bytes(a);
  total += attn_part_bytes(true, a->B, a->Tq, a->N, a->k, a->W, a->H, a->d);
  *bytes = total;
  return CSA_OK;
}

// Every argument check of csa_layer (nothing is enqueued).
static bool layer_appends(const csa_layer_args* a) {
  return a->i_win || a->gk_win || a->gv_win || a->gi_win;
}

static csa_status layer_check(const csa_layer_args* a, const void* ws, size_t ws_bytes) {
  if (!a) return CSA_ERR_INVALID;
  const bool do_compress = a->g_k || a->g_v || a->g_i;
  if (a->i_scale) {
    // FP8 indexer keys: decode calls on given caches only
    if (do_compress || layer_appends(a)) return CSA_ERR_UNSUPPORTED;
    if (!al16(a->i_scale)) return CSA_ERR_INVALID;
    if (!csa::indexer_fp8_supported(a->H_I, a->d_I, a->N)) return CSA_ERR_UNSUPPORTED;
  }
  if (layer_appends(a)) {
    if (do_compress) return CSA_ERR_INVALID;  // a prefill compresses every block itself
    if (!a->i_win || !a->gk_win || !a->gv_win || !a->gi_win || !a->k_win || !a->v_win) return CSA_ERR_INVALID;
    if (!al16(a->i_win) || !al16(a->gk_win) || !al16(a->gv_win) || !al16(a->gi_win) || !a->k_cmp ||
        !a->v_cmp || !a->i_cmp || !al16(a->k_cmp) || !al16(a->v_cmp) || !al16(a->i_cmp))
      return CSA_ERR_INVALID;
    if (a->d % 8 != 0 || a->d_I % 8 != 0 || a->d > 512 || a->d_I > 512 || a->m < 1 || a->m > 4096 ||
        a->T_raw < a->m)
      return CSA_ERR_INVALID;
  }
  if (do_compress) {
    if (!a->g_k || !a->g_v || !a->g_i || !a->x_k || !a->x_v || !a->x_i) return CSA_ERR_INVALID;
    if (a->m <= 0 || a->T < 0 || a->T / a->m != a->N) return CSA_ERR_INVALID;
    if (!a->k_cmp || !a->v_cmp || !a->i_cmp) return CSA_ERR_INVALID;
  }
  csa_status st = check_index_args(a->q_idx, a->i_cmp, a->w, a->q_pos, a->B, a->Tq, a->N, a->H_I,
                                   a->d_I, a->m);
  if (st != CSA_OK) return st;
  if (a->w_stride != 0 && a->w_stride < a->H_I) return CSA_ERR_INVALID;
  int32_t* idx = a->idx_out;
  st = idx ? check_topk_args(a->q_pos, a->B, a->Tq, a->N, a->m, a->k, idx, nullptr)
           : check_topk_shape(a->q_pos, a->B, a->Tq, a->N, a->m, a->k);
  if (st != CSA_OK) return st;
  st = check_attend_args(a->q, a->k_cmp, a->v_cmp, a->k_win, a->v_win, a->raw_base, a->q_pos, a->B,
                         a->Tq, a->N, a->T_raw, a->H, a->d, a->W, a->out, a->out_dtype, a->lse);
  if (st != CSA_OK) return st;
  if (do_compress && (a->d % 8 != 0 || a->d_I % 8 != 0 || !al16(a->x_k) || !al16(a->x_v) ||
                      !al16(a->x_i) || !al16(a->g_k) || !al16(a->g_v) || !al16(a->g_i) ||
                      !al16(a->k_cmp) || !al16(a->v_cmp) || !al16(a->i_cmp)))
    return CSA_ERR_INVALID;
  size_t need = 0;
  csa_layer_workspace(a, &need);
  return check_ws(ws, ws_bytes, need);
}

// Enqueue steps (1)-(4) of an already checked call.
static csa_status layer_enqueue(const csa_layer_args* a, void* ws, cudaStream_t s) {
  const bool do_compress = a->g_k || a->g_v || a->g_i;
  int32_t* idx = a->idx_out;
  csa_status st = CSA_OK;
  if (layer_appends(a)) {
    // the blocks this step's positions complete enter the caches before the
    // indexer reads them (the next kernels start only after this one ends)
    csa::AppendArgs ap;
    std::memset(&ap, 0, sizeof(ap));
    ap.x[0] = a->k_win;
    ap.x[1] = a->v_win;
    ap.x[2] = a->i_win;
    ap.g[0] = a->gk_win;
    ap.g[1] = a->gv_win;
    ap.g[2] = a->gi_win;
    ap.out[0] = a->k_cmp;
    ap.out[1] = a->v_cmp;
    ap.out[2] = a->i_cmp;
    ap.D[0] = a->d;
    ap.D[1] = a->d;
    ap.D[2] = a->d_I;
    ap.n_streams = 3;
    ap.raw_base = a->raw_base;
    ap.q_pos = a->q_pos;
    ap.B = a->B;
    ap.Tq = a->Tq;
    ap.T_raw = a->T_raw;
    ap.N = a->N;
    ap.m = a->m;
    ap.errw = err_word(ws);
    st = cuda_status(csa::launch_append(ap, s));
    if (st != CSA_OK) return st;
  }
  char* base = static_cast<char*>(ws) + CSA_WS_HEADER_BYTES;
  float* S = reinterpret_cast<float*>(base);
  base += scores_bytes(a->B, a->Tq, a->N);
  void* tk = base;
  base += topk_bytes(a->B, a->Tq, a->N);
  if (!idx) {
    idx = reinterpret_cast<int32_t*>(base);
    base += align_up(static_cast<size_t>(a->B) * a->Tq * a->k * 4, kAlignWs);
  }
  void* q8 = nullptr;
  float* q8_scale = nullptr;
  if (a->i_scale) {
    q8 = base;
    q8_scale = reinterpret_cast<float*>(base + fp8_query_codes_bytes(a));
    base += fp8_query_bytes(a);
  }
  if (do_compress) {
    csa::CompressArgs c;
    std::memset(&c, 0, sizeof(c));
    c.x[0] = a->x_k;
    c.x[1] = a->x_v;
    c.x[2] = a->x_i;
    c.g[0] = a->g_k;
    c.g[1] = a->g_v;
    c.g[2] = a->g_i;
    c.out[0] = a->k_cmp;
    c.out[1] = a->v_cmp;
    c.out[2] = a->i_cmp;
    c.D[0] = a->d;
    c.D[1] = a->d;
    c.D[2] = a->d_I;
    c.n_streams = 3;
    c.B = a->B;
    c.T = a->T;
    c.m = a->m;
    c.out_f32 = 0;
    st = cuda_status(csa::launch_compress(c, s));
    if (st != CSA_OK) return st;
  }
  const long long ld = scores_ld(a->N);
  csa::IndexerArgs ia{a->q_idx, a->i_cmp, a->w, a->q_pos, S, ld, a->B, a->Tq, a->N, a->H_I, a->d_I,
                      a->m, err_word(ws), g_wait_budget, nullptr, 0, a->w_stride};
  if (a->i_scale) {
    // this step's indexer queries to E4M3 codes (one scale per head row)
    st = cuda_status(csa::launch_quantize_fp8(a->q_idx, static_cast<long long>(a->B) * a->Tq * a->H_I, a->d_I,
                                              q8, q8_scale, s));
    if (st != CSA_OK) return st;
    ia.q_idx = q8;
    ia.fp8 = 1;
    ia.q_scale = q8_scale;
    ia.k_scale = a->i_scale;
  }
  csa::TopkArgs ta{S, ld, a->q_pos, a->B, a->Tq, a->N, a->m, a->k, idx, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  if (!do_compress && csa::tail_supported(a->Tq, a->N, a->k, a->W, a->H, a->d)) {
    // decode: indexer (+ bucket histogram), then one fused top-k + attention kernel
    const long long nq = static_cast<long long>(a->B) * a->Tq;
    csa::topk_scratch_carve(ta, tk, nq);
    const bool fused = csa::indexer_fills_hist(a->Tq, a->H_I);
    if (fused) {
      st = cuda_status(csa::launch_topk_zero(ta, nq, s));
      if (st != CSA_OK) return st;
      ia.hist = ta.hist;
      ia.after_zero = 1;
    }
    st = cuda_status(launch_indexer_marked(ia, s));
    if (st != CSA_OK) return st;
    if (!fused) {
      st = cuda_status(csa::launch_topk_hist(ta, s));
      if (st != CSA_OK) return st;
    }
    csa::TailArgs tl;
    tl.scores = S;
    tl.ld = ld;
    tl.q_pos = a->q_pos;
    tl.B = a->B;
    tl.Tq = a->Tq;
    tl.N = a->N;
    tl.m = a->m;
    tl.k = a->k;
    tl.hist = ta.hist;
    tl.hist2 = ta.hist2;
    tl.hist3 = ta.hist3;
    tl.cand = ta.cand;
    tl.idx_out = a->idx_out;
    tl.score_out = nullptr;
    tl.budget = g_wait_budget;
    csa::AttendArgs& at = tl.at;
    at.q = a->q;
    at.k_cmp = a->k_cmp;
    at.v_cmp = a->v_cmp;
    at.idx = nullptr;
    at.k_raw = a->k_win;
    at.v_raw = a->v_win;
    at.raw_base = a->raw_base;
    at.q_pos = a->q_pos;
    at.B = a->B;
    at.Tq = a->Tq;
    at.N = a->N;
    at.T_raw = a->T_raw;
    at.H = a->H;
    at.d = a->d;
    at.k = a->k;
    at.W = a->W;
    at.m = a->m;
    at.scale = a->scale > 0.f ? a->scale : 1.0f / std::sqrt(static_cast<float>(a->d));
    at.out = a->out;
    at.out_f32 = a->out_dtype == CSA_F32;
    at.lse = a->lse;
    at.part = nullptr;
    at.errw = err_word(ws);
    return cuda_status(csa::launch_decode_tail(tl, s));
  }
  st = index_then_topk(ia, ta, tk, s);
  if (st != CSA_OK) return st;
  csa::AttendArgs at;
  std::memset(&at, 0, sizeof(at));
  at.q = a->q;
  at.k_cmp = a->k_cmp;
  at.v_cmp = a->v_cmp;
  at.idx = idx;
  at.k_raw = a->k_win;
  at.v_raw = a->v_win;
  at.raw_base = a->raw_base;
  at.q_pos = a->q_pos;
  at.B = a->B;
  at.Tq = a->Tq;
  at.N = a->N;
  at.T_raw = a->T_raw;
  at.H = a->H;
  at.d = a->d;
  at.k = a->k;
  at.W = a->W;
  at.m = a->m;
  at.scale = a->scale > 0.f ? a->scale : 1.0f / std::sqrt(static_cast<float>(a->d));
  at.out = a->out;
  at.out_f32 = a->out_dtype == CSA_F32;
  at.lse = a->lse;
  at.part = reinterpret_cast<float*>(base);
  at.errw = err_word(ws);
  return cuda_status(launch_attention(at, s));
}

csa_status csa_layer(const csa_layer_args* a, void* ws, size_t ws_bytes, void* stream) {
  const csa_status st = layer_check(a, ws, ws_bytes);
  if (st != CSA_OK) return st;
  return layer_enqueue(a, ws, static_cast<cudaStream_t>(stream));
}

csa_status csa_layer_host(const csa_layer_args* a, const void* q_host, const void* q_idx_host,
                          void* out_host, void* ws, size_t ws_bytes, void* stream) {
  csa_status st = layer_check(a, ws, ws_bytes);
  if (st != CSA_OK) return st;
  if (!q_host || !q_idx_host || !out_host) return CSA_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t nq = static_cast<size_t>(a->B) * a->Tq;
  const size_t q_bytes = nq * a->H * a->d * 2;
  const size_t qi_bytes = nq * a->H_I * a->d_I * 2;
  const size_t out_bytes = nq * a->H * a->d * (a->out_dtype == CSA_F32 ? 4 : 2);
  if (cudaMemcpyAsync(const_cast<void*>(a->q), q_host, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(const_cast<void*>(a->q_idx), q_idx_host, qi_bytes, cudaMemcpyHostToDevice, s) !=
          cudaSuccess)
    return CSA_ERR_CUDA;
  st = layer_enqueue(a, ws, s);
  if (st != CSA_OK) return st;
  return cuda_status(cudaMemcpyAsync(out_host, a->out, out_bytes, cudaMemcpyDeviceToHost, s));
}

// ---------------------------------------------------------------- stack
static size_t stack_act_bytes(const csa_stack_layer* l) {
  return align_up(static_cast<size_t>(l->a.B) * l->a.Tq * l->a.H * l->a.d * 2, kAlignWs);
}

// Layer i's arguments with its input and output activations filled in.
static csa_layer_args stack_args(const csa_stack_layer* l, const void* in, void* out, int out_dtype) {
  csa_layer_args a = l->a;
  a.q = in;
  a.q_idx = in;
  a.out = out;
  a.out_dtype = out_dtype;
  a.lse = nullptr;
  return a;
}

static size_t stack_layer_ws(const csa_stack_layer* l) {
  size_t need = 0;
  const csa_layer_args& a = l->a;
  if (l->kind == CSA_STACK_CSA) {
    csa_layer_workspace(&a, &need);
  } else if (l->kind == CSA_STACK_HCA) {
    hca_attend_workspace(a.B, a.Tq, a.N, a.H, a.d, a.W, &need);
  } else {
    csa_attend_workspace(a.B, a.Tq, a.H, a.d, 0, a.W, &need);
  }
  return need;
}

csa_status csa_stack_workspace(const csa_stack_layer* layers, int n_layers, size_t* bytes) {
  if (!layers || n_layers <= 0 || !bytes) return CSA_ERR_INVALID;
  size_t need = 0;
  for (int i = 0; i < n_layers; ++i) {
    const csa_layer_args& a = layers[i].a;
    if (a.B <= 0 || a.Tq <= 0 || a.H <= 0 || a.d <= 0) return CSA_ERR_INVALID;
    const size_t w = stack_layer_ws(&layers[i]);
    need = need > w ? need : w;
  }
  // the layer workspace, then two activation buffers (ping-pong)
  *bytes = align_up(need, kAlignWs) + 2 * stack_act_bytes(&layers[0]);
  return CSA_OK;
}

csa_status csa_stack_decode(const csa_stack_layer* layers, int n_layers, const void* x, void* y, int out_dtype,
                            void* ws, size_t ws_bytes, void* stream) {
  size_t need = 0;
  csa_status st = csa_stack_workspace(layers, n_layers, &need);
  if (st != CSA_OK) return st;
  if (!x || !y || !al16(x) || !al16(y)) return CSA_ERR_INVALID;
  if (out_dtype != CSA_BF16 && out_dtype != CSA_F32) return CSA_ERR_INVALID;
  st = check_ws(ws, ws_bytes, need);
  if (st != CSA_OK) return st;
  const csa_layer_args& a0 = layers[0].a;
  size_t layer_ws = 0;
  for (int i = 0; i < n_layers; ++i) {
    const size_t w = stack_layer_ws(&layers[i]);
    layer_ws = layer_ws > w ? layer_ws : w;
  }
  layer_ws = align_up(layer_ws, kAlignWs);
  char* act[2] = {static_cast<char*>(ws) + layer_ws, static_cast<char*>(ws) + layer_ws + stack_act_bytes(&layers[0])};
  // every layer's checks before anything is enqueued: same activation shape
  // throughout, and a CSA layer's indexer queries are its input activation
  for (int i = 0; i < n_layers; ++i) {
    const csa_stack_layer* l = &layers[i];
    const csa_layer_args& a = l->a;
    if (a.B != a0.B || a.Tq != a0.Tq || a.H != a0.H || a.d != a0.d) return CSA_ERR_INVALID;
    const void* in = i == 0 ? x : act[(i - 1) & 1];
    void* out = i == n_layers - 1 ? y : act[i & 1];
    const csa_layer_args la = stack_args(l, in, out, i == n_layers - 1 ? out_dtype : CSA_BF16);
    if (l->kind == CSA_STACK_CSA) {
      if (a.H_I * a.d_I != a.H * a.d) return CSA_ERR_INVALID;
      if (a.g_k || a.g_v || a.g_i) return CSA_ERR_INVALID;  // decode: the caches are given
      st = layer_check(&la, ws, layer_ws);
    } else if (l->kind == CSA_STACK_HCA || l->kind == CSA_STACK_SWA) {
      st = check_attend_args(la.q, la.k_cmp, la.v_cmp, la.k_win, la.v_win, la.raw_base, la.q_pos, la.B, la.Tq,
                             l->kind == CSA_STACK_HCA ? la.N : 0, la.T_raw, la.H, la.d, la.W, la.out,
                             la.out_dtype, nullptr);
      if (st == CSA_OK && l->kind == CSA_STACK_HCA && la.m <= 0) st = CSA_ERR_INVALID;
    } else {
      st = CSA_ERR_INVALID;
    }
    if (st != CSA_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < n_layers; ++i) {
    const csa_stack_layer* l = &layers[i];
    const void* in = i == 0 ? x : act[(i - 1) & 1];
    void* out = i == n_layers - 1 ? y : act[i & 1];
    const csa_layer_args la = stack_args(l, in, out, i == n_layers - 1 ? out_dtype : CSA_BF16);
    if (l->kind == CSA_STACK_CSA) {
      st = layer_enqueue(&la, ws, s);
    } else {
      // SWA: the window alone (no compressed entries); HCA: every visible entry + the window
      const bool hca = l->kind == CSA_STACK_HCA;
      st = attend_common(la.q, hca ? la.k_cmp : nullptr, hca ? la.v_cmp : nullptr, hca ? nullptr : la.q_pos,
                         la.k_win, la.v_win, la.raw_base, la.q_pos, la.B, la.Tq, hca ? la.N : 0, la.T_raw, la.H,
                         la.d, 0, hca ? la.m : 1, la.W, la.scale, la.out, la.out_dtype, nullptr, ws, layer_ws, s);
    }
    if (st != CSA_OK) return st;
  }
  return CSA_OK;
}

}  // extern "C"
