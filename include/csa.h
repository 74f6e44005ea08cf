/*
 * csa.h -- C ABI of the B300 (sm_103a) Compressed Sparse Attention library.
 *
 * The library computes the CSA layer of the DeepSeek-V4 descriptions and its
 * dense HCA mode on one GPU:
 *   (1) block compression of the raw K / V / indexer-key streams,
 *   (2) Lightning-Indexer scores of each query against the visible entries,
 *   (3) per-query top-k of those scores,
 *   (4) attention over the selected entries merged with a sliding window of
 *       raw tokens (CSA), or over every visible entry (HCA).
 *
 * Sources: "DeepSeek V4: Compressed Sparse Attention and the Million-Token
 * Context" (octagono.org), section "Hybrid Attention: CSA and HCA";
 * "DeepSeek V4 technical review" (takeshell.com), sections 2.1 CSA and
 * 2.2 HCA.  The accompanying workload specification fixes the compressor
 * (per-channel softmax of given gate logits times the raw vectors), the score
 * (sum_h w_h * ReLU(q_h . k)), the lowest-index tie rule, the visibility rule
 * (block b visible to position t iff (b+1)*m - 1 <= t), the scale 1/sqrt(d)
 * and the single shared K/V stream (MQA).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers named as tensors are DEVICE pointers owned by the caller; the
 *   library never allocates, frees or keeps them.  Arrays of pointers and
 *   size arrays (``x``, ``g``, ``out``, ``D`` of csa_compress, the args
 *   struct of csa_layer) are HOST memory, read during the call only.
 * - Tensors are dense row-major with the shapes given, bf16 unless stated.
 *   Every bf16 / fp32 tensor must start on a 16-byte boundary.
 * - ``stream`` is a cudaStream_t (NULL = legacy default stream).  Every call
 *   only enqueues work on it and returns; nothing synchronises except
 *   csa_check_error.
 * - Argument errors are found before anything is enqueued: a call that
 *   returns an error has written nothing.  CSA_ERR_CUDA reports a failed
 *   launch (cudaGetLastError).  Conditions found on the device (an index
 *   outside its buffer, a bounded wait that ran out) set bits in the error
 *   word at the start of the workspace; read them with csa_check_error.
 * - ``ws`` / ``ws_bytes``: caller-owned device scratch of at least the size
 *   the matching *_workspace call reports, 256-byte aligned, initialised once
 *   with csa_workspace_init.  One workspace must not be used by two calls
 *   that overlap on the GPU.
 * - Results do not depend on the GPU's SM count or on timing: no floating-
 *   point atomics are used and partial results are merged in a fixed order.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa_status {
    CSA_OK = 0,
    CSA_ERR_INVALID = 1,      /* null pointer, bad size, misaligned tensor       */
    CSA_ERR_UNSUPPORTED = 2,  /* valid, but a shape the library does not handle */
    CSA_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small      */
    CSA_ERR_CUDA = 4,         /* a CUDA call or kernel launch failed             */
    CSA_ERR_TIMEOUT = 5,      /* device: a bounded wait ran out                  */
    CSA_ERR_DEVICE_INDEX = 6  /* device: an index or window row outside its buffer */
} csa_status;

typedef enum csa_dtype { CSA_BF16 = 0, CSA_F32 = 1 } csa_dtype;

/* Device error-word bits (csa_check_error's *flags). */
#define CSA_FLAG_TIMEOUT 0x1u
#define CSA_FLAG_INDEX 0x2u

/* Bytes at the start of every workspace that hold the error word. */
#define CSA_WS_HEADER_BYTES 256

/* Human-readable name of a status code (static string, never NULL). */
const char* csa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int csa_version(void);

/* Zero the error word at the start of ``ws`` (stream-ordered memset).
 * Call once after allocating a workspace.  ws_bytes >= CSA_WS_HEADER_BYTES. */
csa_status csa_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Wait for ``stream`` and read the workspace error word.  *flags (nullable)
 * receives the raw bits; returns CSA_ERR_TIMEOUT / CSA_ERR_DEVICE_INDEX when a
 * bit is set, else CSA_OK.  clear != 0 zeroes the word after reading it. */
csa_status csa_check_error(const void* ws, uint32_t* flags, int clear, void* stream);

/* --------------------------------------------------------------------------
 * (1) Block compression.  "DeepSeek V4 technical review", section 2.1: each
 * compressed entry is a weighted sum of m consecutive tokens (section 2.2:
 * m' = 128 for HCA).  Entry b, channel c of stream i:
 *     out_i[n, b, c] = sum_{j<m} softmax_j(g_i[n, b*m+j, c]) * x_i[n, b*m+j, c]
 * n_streams (1..3) independent (x_i, g_i) -> out_i triples in one launch:
 *   x[i], g[i] : [B, T, D[i]] bf16          out[i] : [B, T/m, D[i]] out_dtype
 * T mod m trailing tokens are not compressed.  D[i] in {8, 16, ..., 512}
 * (multiple of 8); 1 <= m <= 4096; out_dtype CSA_BF16 (round to nearest
 * even) or CSA_F32.  Needs no workspace.
 * ------------------------------------------------------------------------ */
csa_status csa_compress(int n_streams, const void* const* x, const void* const* g,
                        void* const* out, const int* D, int B, int T, int m,
                        int out_dtype, void* stream);

/* --------------------------------------------------------------------------
 * (1') Decode-time compression and cache append.  Octagono "Hybrid Attention:
 * CSA and HCA" and the technical review, section 2.1: every m tokens become
 * one compressed entry.  During decoding the raw tokens of the newest
 * positions live in a window buffer; a query at position t = q_pos[n, j] with
 * (t + 1) % m == 0 completes block b = (t + 1) / m - 1 (tokens t-m+1 .. t),
 * and this call writes
 *     out_i[n, b, c] = sum_{j<m} softmax_j(g_i[n, r0+j, c]) * x_i[n, r0+j, c],
 *     r0 = t - m + 1 - raw_base[n],
 * exactly as csa_compress folds that block (bit-identical to compressing the
 * whole prefix).  Positions that complete no block leave the caches alone, so
 * the partial block stays raw in the window buffer.
 *   x_win[i], g_win[i] : [B, T_raw, D[i]] bf16 (row r holds token raw_base[n] + r)
 *   out[i]             : [B, N, D[i]] bf16 caches (capacity N entries)
 *   raw_base [B], q_pos [B, Tq] int32
 * A block whose rows are outside the window buffer, or whose entry is >= N,
 * is skipped and flagged with CSA_FLAG_INDEX.  D[i] multiple of 8, <= 512;
 * 1 <= m <= 4096; T_raw >= m.  Workspace: CSA_WS_HEADER_BYTES.
 * ------------------------------------------------------------------------ */
csa_status csa_append(int n_streams, const void* const* x_win, const void* const* g_win,
                      void* const* out, const int* D, const int32_t* raw_base,
                      const int32_t* q_pos, int B, int Tq, int T_raw, int N, int m,
                      void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * (2) Lightning Indexer scores.  Octagono "Hybrid Attention: CSA and HCA" and
 * the technical review, section 2.1: every query gets indexer queries that
 * are scored against the compressed entries; 64 heads of width 128.
 *     S[n, j, b] = sum_h w[n, j, h] * ReLU(q_idx[n, j, h, :] . k_idx[n, b, :])
 * for the visible blocks b < n_vis = min(N, floor((q_pos[n, j] + 1) / m)).
 *   q_idx  [B, Tq, H_I, d_I] bf16     k_idx [B, N, d_I] bf16
 *   q_pos  [B, Tq] int32 (absolute positions)
 *   w      fp32 head weights: w_stride == 0 -> one [H_I] vector shared by
 *          every query (w[n, j, h] = w[h]); w_stride >= H_I -> one vector per
 *          query, w[n, j, h] = w[(n * Tq + j) * w_stride + h] (produced per
 *          token, as the DSA-style indexer of the pages does; any sign)
 *   scores [B, Tq, ld_scores] fp32, ld_scores >= N and a multiple of 4;
 *          entries b >= n_vis are left untouched.
 * Computed on the tcgen05 tensor cores (bf16 products, fp32 accumulation).
 * H_I in {4, 8, 16, 32, 64, 128}; d_I in {32, 64, 128}.  Workspace:
 * CSA_WS_HEADER_BYTES.
 * ------------------------------------------------------------------------ */
csa_status csa_index_scores(const void* q_idx, const void* k_idx, const float* w,
                            int64_t w_stride, const int32_t* q_pos, int B, int Tq, int N, int H_I, int d_I,
                            int m, float* scores, int64_t ld_scores,
                            void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * (2') FP8 indexer.  "DeepSeek V4 technical review", section 5, and
 * dataforcee "Muon Optimizer and FP4 QAT": the indexer's QK product runs in
 * low precision.  Rows (one compressed indexer key, or one indexer query
 * head) are stored as OCP FP8 E4M3 codes with one power-of-two scale per row:
 * scale = 2^e, e the smallest integer with max|row| <= 448 * 2^e (in
 * [-126, 120]; an all-zero row gets 1), code = round-to-nearest-even of
 * row / scale.  The division is exact, so the code rounding is the only
 * inexact step and the result is fixed bit for bit.
 *
 * csa_quantize_fp8: x [rows, D] bf16 -> codes [rows, D] (one byte each),
 * scales [rows] fp32.  D in {32, 64, 128, 256}.
 *
 * csa_index_scores_fp8: the scores of (2) on the dequantised rows,
 *     S[n, j, b] = sum_h w[n, j, h] * ReLU((qs_h q8_h) . (ks_b k8_b))
 *                = ks_b * sum_h (w[n, j, h] qs_h) * ReLU(q8_h . k8_b),
 * computed as E4M3 x E4M3 products on the tcgen05 tensor cores (kind::f8f6f4,
 * fp32 accumulation) with the scales applied in the epilogue.
 *   q8 [B, Tq, H_I, d_I] codes, q_scale [B * Tq * H_I] fp32,
 *   k8 [B, N, d_I] codes, k_scale [B, N] fp32; the rest as csa_index_scores.
 * d_I = 128; N % 4 == 0; H_I in {16, 32, 64, 128}.  Workspace:
 * CSA_WS_HEADER_BYTES.  Keys take 128 + 4 bytes per entry instead of 256.
 * ------------------------------------------------------------------------ */
csa_status csa_quantize_fp8(const void* x, int64_t rows, int D, void* codes, float* scales,
                            void* stream);
csa_status csa_index_scores_fp8(const void* q8, const float* q_scale, const void* k8,
                                const float* k_scale, const float* w, int64_t w_stride,
                                const int32_t* q_pos, int B, int Tq, int N, int H_I, int d_I,
                                int m, float* scores, int64_t ld_scores, void* ws,
                                size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * (3) Top-k.  Technical review, section 2.1: keep the top-k compressed blocks
 * per query (k = 1024).  Among the n_vis visible scores of each query keep
 * the min(k, n_vis) largest; equal scores go to the lower block index.
 *   scores    [B, Tq, ld_scores] fp32 (only b < n_vis is read; -0 == +0)
 *   idx_out   [B, Tq, k] int32: kept block indices ascending, then -1
 *   score_out [B, Tq, k] fp32 (nullable): the kept scores, 0 in padding
 * Integer radix selection on order-preserving keys: exact, no tolerance.
 * 1 <= k <= 4096; N <= 2^24.  Rows longer than 16384 entries use a bucket
 * histogram and candidate list in the workspace: size from
 * csa_topk_workspace (CSA_WS_HEADER_BYTES alone when N <= 16384).
 * ------------------------------------------------------------------------ */
csa_status csa_topk_workspace(int B, int Tq, int N, int k, size_t* bytes);
csa_status csa_topk(const float* scores, int64_t ld_scores, const int32_t* q_pos,
                    int B, int Tq, int N, int m, int k, int32_t* idx_out, float* score_out,
                    void* ws, size_t ws_bytes, void* stream);

/* (2)+(3) in one call; the scores (and the long-row top-k scratch) live in
 * the workspace.  With Tq == 1 the indexer also accumulates the top-k bucket
 * histogram as it writes the scores. */
csa_status csa_index_topk_workspace(int B, int Tq, int N, int H_I, int d_I, int k,
                                    size_t* bytes);
csa_status csa_index_topk(const void* q_idx, const void* k_idx, const float* w,
                          int64_t w_stride, const int32_t* q_pos, int B, int Tq, int N, int H_I, int d_I,
                          int m, int k, int32_t* idx_out, float* score_out,
                          void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * (4) Sparse attention + sliding window (CSA).  Technical review, section
 * 2.1: attention runs only over the selected compressed blocks; octagono
 * "Hybrid Attention": a window over the most recent 128 raw tokens supplies
 * local context.  For query (n, j) at position t = q_pos[n, j] and head h:
 *     keys  J = { k_cmp[n, idx[n, j, i]] : idx >= 0 }
 *             ++ { k_raw[n, u - raw_base[n]] : max(0, t-W+1) <= u <= t }
 *     out[n, j, h] = sum_{x in J} softmax_x(scale * q[n, j, h] . K_x) V_x
 * one softmax over both parts (not de-duplicated); empty J gives 0 / -inf.
 *   q [B, Tq, H, d]; k_cmp, v_cmp [B, N, d]; idx [B, Tq, k] int32 (-1 = skip)
 *   k_raw, v_raw [B, T_raw, d] (row r holds token raw_base[n] + r)
 *   raw_base [B], q_pos [B, Tq] int32
 *   out [B, Tq, H, d] out_dtype;  lse [B, Tq, H] fp32 natural log (nullable)
 * scale <= 0 selects 1/sqrt(d).  d in {64, 128}; 1 <= H <= 64; W >= 0.
 * Indices >= N and window rows outside [0, T_raw) are skipped and flagged
 * with CSA_FLAG_INDEX.  bf16 MMAs, fp32 softmax and accumulation.
 * Workspace: the error word and the split partials of long key lists.
 * Decode-shaped calls (Tq < 16) with H = 64 and d = 128 run on the tcgen05
 * tensor cores and cut each query's k + W slots into n_r = ceil(n_t / 5)
 * ranges of 128-slot tiles, n_t = ceil((k + W) / 128); up to 8 ranges merge
 * inside a thread-block cluster (e.g. k = 1024, W = 128: 2 ranges, no
 * partials), more need B * Tq * n_r * H * (d + 1) * 4 bytes of partials
 * (e.g. k = 5200, W = 128: 9 ranges, 297 KB per query).  Other shapes need
 * partials only for k + W > 131072.  The split depends on k + W only, never
 * on B, so a sequence gives the same result alone or in any batch.
 * ------------------------------------------------------------------------ */
csa_status csa_attend_workspace(int B, int Tq, int H, int d, int k, int W, size_t* bytes);
csa_status csa_attend(const void* q, const void* k_cmp, const void* v_cmp, const int32_t* idx,
                      const void* k_raw, const void* v_raw, const int32_t* raw_base,
                      const int32_t* q_pos, int B, int Tq, int N, int T_raw, int H, int d,
                      int k, int W, float scale, void* out, int out_dtype, float* lse,
                      void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * csa_attend without a workspace, for callers that cannot allocate device
 * memory: operators hosted by a framework whose memory planner owns the
 * device and hands an operator only its inputs and outputs, and latency-bound
 * callers that must never reach cudaMalloc / cudaFree (both can synchronise
 * the device).  The pages describe no such call; it has no counterpart there.
 *
 * Arguments, layouts, results and the argument errors are those of
 * csa_attend; inputs and outputs are still caller-owned device memory.  Key
 * lists of up to 131072 keys (k + W) merge their split partials inside a
 * thread-block cluster and need no scratch at all; longer lists keep their
 * split partials in one fixed device array of CSA_NOALLOC_SCRATCH_BYTES
 * inside the library instead of a workspace.  Every GPU that loads the
 * library holds that array until the process exits, and no call allocates
 * or frees anything.
 * - Returns CSA_ERR_WORKSPACE when the call's partials would exceed
 *   CSA_NOALLOC_SCRATCH_BYTES: a list of k + W > 131072 keys is split into
 *   n_split = ceil((k + W) / 8192) ranges and needs
 *   B * Tq * n_split * H * (d + 1) * 4 bytes (for example k + W = 139392,
 *   H = 64, d = 128: 594 KB per query, at most 56 queries).
 * - The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 * - Every call on a device shares the one array, which keeps the last call's
 *   contents (each call writes every partial it reads, so nothing needs to
 *   start at zero).  Calls that overlap on the GPU -- on different streams,
 *   or from different host threads -- race on it: order them on one stream.
 * - There is no error word: indices >= N and window rows outside the buffer
 *   are skipped, as in csa_attend, but not reported.
 * ------------------------------------------------------------------------ */
#define CSA_NOALLOC_SCRATCH_BYTES (32u << 20)
csa_status csa_attend_noalloc(const void* q, const void* k_cmp, const void* v_cmp,
                              const int32_t* idx, const void* k_raw, const void* v_raw,
                              const int32_t* raw_base, const int32_t* q_pos, int B, int Tq,
                              int N, int T_raw, int H, int d, int k, int W, float scale,
                              void* out, int out_dtype, float* lse, void* stream);

/* --------------------------------------------------------------------------
 * HCA mode.  Octagono "Hybrid Attention: CSA and HCA" and the technical
 * review, section 2.2: entries compressed every m' (= 128) tokens, attended
 * densely with no selection, plus the same sliding window.  As csa_attend
 * with J's first part = every visible entry b < min(N, floor((t+1)/m)).
 * Decode-shaped calls with H = 64 and d = 128 load the entries as TMA tiles
 * on the tcgen05 path, in ranges of up to 4 tiles; there
 * n_t = ceil(N / 128) + ceil(W / 128) and n_r = ceil(n_t / 4) (e.g.
 * N = 8192, W = 128: 17 ranges, 561 KB of partials per query; up to 8
 * ranges merge inside a cluster and need none).
 * ------------------------------------------------------------------------ */
csa_status hca_attend_workspace(int B, int Tq, int N, int H, int d, int W, size_t* bytes);
csa_status hca_attend(const void* q, const void* k_cmp, const void* v_cmp,
                      const void* k_raw, const void* v_raw, const int32_t* raw_base,
                      const int32_t* q_pos, int B, int Tq, int N, int T_raw, int H, int d,
                      int m, int W, float scale, void* out, int out_dtype, float* lse,
                      void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * The whole CSA layer, steps (1) -> (2) -> (3) -> (4), enqueued on one stream.
 * If g_k, g_v and g_i are all non-NULL, step (1) compresses x_k, x_v, x_i
 * ([B, T, d], [B, T, d], [B, T, d_I]) at m into k_cmp, v_cmp, i_cmp
 * ([B, N, .] bf16, N = T / m); if all three are NULL the caches are read as
 * given (decode).  Steps (2)-(4) are csa_index_topk and csa_attend.
 * ------------------------------------------------------------------------ */
typedef struct csa_layer_args {
    int B, Tq, N, m, H, d, H_I, d_I, k, W;
    int T;                  /* raw tokens compressed (step 1 only)              */
    int T_raw;              /* rows of the window buffer k_win / v_win          */
    float scale;            /* <= 0: 1/sqrt(d)                                  */
    const void *x_k, *x_v, *x_i;   /* raw streams for step (1), or NULL         */
    const void *g_k, *g_v, *g_i;   /* gate logits for step (1), or NULL         */
    void *k_cmp, *v_cmp, *i_cmp;   /* compressed caches (written by step 1)     */
    const void *k_win, *v_win;     /* raw window buffer [B, T_raw, d]           */
    const int32_t* raw_base;       /* [B]                                       */
    const void* q;                 /* [B, Tq, H, d]                             */
    const void* q_idx;             /* [B, Tq, H_I, d_I]                         */
    const float* w;                /* [H_I], or per query (w_stride)            */
    const int32_t* q_pos;          /* [B, Tq]                                   */
    int32_t* idx_out;              /* [B, Tq, k] or NULL (kept in workspace)    */
    void* out;                     /* [B, Tq, H, d]                             */
    int out_dtype;
    float* lse;                    /* [B, Tq, H] or NULL                        */
    /* Decode-time append (all four non-NULL, or all NULL): before step (2)
     * every block that a query position completes ((t + 1) % m == 0) is
     * compressed into the caches from the window rows, as csa_append does
     * with the raw streams k_win, v_win, i_win and these gate logits.  Not
     * combined with step (1) (g_k, g_v, g_i must then be NULL). */
    const void* i_win;             /* raw indexer keys of the window rows [B, T_raw, d_I] */
    const void *gk_win, *gv_win, *gi_win;  /* their gate logits [B, T_raw, d / d / d_I] */
    long long w_stride;            /* 0: w is [H_I]; >= H_I: w is per query, see (2) */
    /* FP8 indexer keys (NULL: bf16): i_cmp holds E4M3 codes [B, N, d_I] made
     * by csa_quantize_fp8 and i_scale [B, N] their row scales; the step's
     * q_idx (bf16) is quantised the same way inside the call and step (2)
     * runs as csa_index_scores_fp8.  Decode calls on given caches only (no
     * step (1), no append); d_I = 128, N % 4 == 0, H_I in {16, 32, 64, 128}. */
    const float* i_scale;
} csa_layer_args;

csa_status csa_layer_workspace(const csa_layer_args* a, size_t* bytes);
csa_status csa_layer(const csa_layer_args* a, void* ws, size_t ws_bytes, void* stream);

/* csa_layer for a caller whose step inputs and result live in HOST memory:
 * on ``stream`` it copies q_host ([B, Tq, H, d] bf16) into a->q and
 * q_idx_host ([B, Tq, H_I, d_I] bf16) into a->q_idx, enqueues the layer
 * exactly as csa_layer does, then copies a->out into out_host
 * ([B, Tq, H, d] of a->out_dtype).  The compressed caches, the window buffer
 * and the weights stay resident on the device; a->q, a->q_idx and a->out are
 * the caller's device staging buffers.  The host buffers should be
 * page-locked (cudaHostAlloc, or torch's pin_memory) so that the copies are
 * asynchronous; out_host holds the result once the stream reaches the end
 * of the call (synchronise on it, or on an event recorded after the call).
 * All checks of csa_layer run before the first copy is enqueued; a NULL host
 * pointer is CSA_ERR_INVALID. */
csa_status csa_layer_host(const csa_layer_args* a, const void* q_host, const void* q_idx_host,
                          void* out_host, void* ws, size_t ws_bytes, void* stream);

/* --------------------------------------------------------------------------
 * The hybrid layer stack at decode time.  "DeepSeek V4 technical review",
 * section 2.3: the first two layers attend over a sliding window only, the
 * following layers alternate CSA and HCA.  The pages give no weights for
 * this path, so the stack carries the activations from layer to layer
 * unchanged (identity projections): layer i's output [B, Tq, H, d] is layer
 * i + 1's query, and for a CSA layer also its indexer query (H_I * d_I must
 * equal H * d; the same bytes read as [B, Tq, H_I, d_I]).  Each layer has
 * its own caches and window buffer.
 *   kind CSA_STACK_SWA: attention over the W newest raw tokens (k_win, v_win,
 *        T_raw, raw_base, W, q_pos, scale of ``a``);
 *   kind CSA_STACK_CSA: csa_layer on given caches (no step (1); ``a``'s q,
 *        q_idx, out and lse are ignored; idx_out, if set, receives the
 *        layer's kept indices);
 *   kind CSA_STACK_HCA: hca_attend on the layer's entries (k_cmp, v_cmp, N,
 *        m) and window.
 * x is layer 0's input, y receives the last layer's output (out_dtype); the
 * intermediate activations (bf16) live in the workspace.  Every layer has
 * the same B, Tq, H, d.  All checks run before anything is enqueued.
 * ------------------------------------------------------------------------ */
enum { CSA_STACK_SWA = 0, CSA_STACK_CSA = 1, CSA_STACK_HCA = 2 };
typedef struct csa_stack_layer {
    int kind;
    csa_layer_args a;
} csa_stack_layer;
csa_status csa_stack_workspace(const csa_stack_layer* layers, int n_layers, size_t* bytes);
csa_status csa_stack_decode(const csa_stack_layer* layers, int n_layers, const void* x, void* y,
                            int out_dtype, void* ws, size_t ws_bytes, void* stream);

/* Test hook: the clock64 budget of every bounded device-side wait issued by
 * later calls in this process (default ~2^31 cycles, about one second).
 * cycles <= 0 restores the default. */
void csa_set_wait_budget(long long cycles);

/* Instrumentation: until called again with NULLs, every call made from this
 * host thread that launches the indexer kernel (csa_index_scores,
 * csa_index_topk, csa_layer) records cudaEvent_t ev_begin on the call's
 * stream just before that launch and ev_end just after it, so the indexer can
 * be timed inside the fused calls (also inside a stream capture, where the
 * records become graph nodes).  Either may be NULL. */
void csa_set_indexer_events(void* ev_begin, void* ev_end);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H_ */
