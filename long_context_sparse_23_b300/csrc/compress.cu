// (1) Block compression.  "DeepSeek V4 technical review", section 2.1 (each
// compressed entry is a weighted sum over m tokens) and section 2.2 (m' = 128
// for HCA); the weights are the per-channel softmax of given gate logits:
//   out[n, b, c] = sum_{j<m} softmax_j(g[n, b*m+j, c]) * x[n, b*m+j, c]
//
// HBM-streaming design: one thread owns 8 channels (one 16-byte vector) of
// one block and walks the block's m rows in chunks of R (the largest of 8, 4,
// 2, 1 dividing m), keeping a running per-channel maximum, denominator and
// weighted sum in fp32 (one rescale per chunk, one exp2 per element).
// Consecutive threads own consecutive 16-byte vectors of a row, so every warp
// load covers whole 128-byte lines.  Up to three (x, g) -> out streams (K, V,
// indexer keys) share one launch via blockIdx.y.
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Fold R rows (one chunk) of 8 channels into the running (M, L, A) state.
template <int R>
__device__ __forceinline__ void fold_rows(const char* xp, const char* gp, size_t row_bytes,
                                          float (&M)[8], float (&L)[8], float (&A)[8]) {
  uint4 xv[R], gv[R];
#pragma unroll
  for (int j = 0; j < R; ++j) {
    xv[j] = ld_stream16(xp + static_cast<size_t>(j) * row_bytes);
    gv[j] = ld_stream16(gp + static_cast<size_t>(j) * row_bytes);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    // channels 2e, 2e+1 live in word e of every row
    float c0 = -INFINITY, c1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint32_t gw = (&gv[j].x)[e];
      c0 = fmaxf(c0, bf16lo(gw));
      c1 = fmaxf(c1, bf16hi(gw));
    }
    const float n0 = fmaxf(M[2 * e], c0 * kLog2e), n1 = fmaxf(M[2 * e + 1], c1 * kLog2e);
    const float s0 = ex2(M[2 * e] - n0), s1 = ex2(M[2 * e + 1] - n1);  // 0 while M = -inf
    float l0 = L[2 * e] * s0, l1 = L[2 * e + 1] * s1;
    float a0 = A[2 * e] * s0, a1 = A[2 * e + 1] * s1;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint32_t gw = (&gv[j].x)[e], xw = (&xv[j].x)[e];
      const float p0 = ex2(fmaf(bf16lo(gw), kLog2e, -n0));
      const float p1 = ex2(fmaf(bf16hi(gw), kLog2e, -n1));
      l0 += p0;
      l1 += p1;
      a0 = fmaf(p0, bf16lo(xw), a0);
      a1 = fmaf(p1, bf16hi(xw), a1);
    }
    M[2 * e] = n0;
    M[2 * e + 1] = n1;
    L[2 * e] = l0;
    L[2 * e + 1] = l1;
    A[2 * e] = a0;
    A[2 * e + 1] = a1;
  }
}

template <int R, bool kF32Out>
__global__ void __launch_bounds__(kThreads) compress_kernel(CompressArgs a) {
  pdl_wait_then_release();
  const int sidx = blockIdx.y;
  // select with constant indices so the argument block stays in param space
  const int D = sidx == 0 ? a.D[0] : (sidx == 1 ? a.D[1] : a.D[2]);
  const void* xsel = sidx == 0 ? a.x[0] : (sidx == 1 ? a.x[1] : a.x[2]);
  const void* gsel = sidx == 0 ? a.g[0] : (sidx == 1 ? a.g[1] : a.g[2]);
  void* osel = sidx == 0 ? a.out[0] : (sidx == 1 ? a.out[1] : a.out[2]);
  const int G = D >> 3;  // 16-byte vectors per row
  const int nb = a.T / a.m;
  const long long nwork = static_cast<long long>(a.B) * nb * G;
  const char* __restrict__ xs = static_cast<const char*>(xsel);
  const char* __restrict__ gs = static_cast<const char*>(gsel);
  const size_t row_bytes = static_cast<size_t>(D) * 2;

  for (long long wi = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; wi < nwork;
       wi += static_cast<long long>(gridDim.x) * kThreads) {
    const int cg = static_cast<int>(wi % G);
    const long long r = wi / G;
    const int blk = static_cast<int>(r % nb);
    const long long b = r / nb;
    const size_t off = (static_cast<size_t>(b) * a.T + static_cast<size_t>(blk) * a.m) * row_bytes +
                       static_cast<size_t>(cg) * 16;
    float M[8], L[8], A[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      M[c] = -INFINITY;
      L[c] = 0.f;
      A[c] = 0.f;
    }
    // m is a multiple of R (the launcher picks R)
    for (int j0 = 0; j0 < a.m; j0 += R)
      fold_rows<R>(xs + off + static_cast<size_t>(j0) * row_bytes,
                   gs + off + static_cast<size_t>(j0) * row_bytes, row_bytes, M, L, A);
    float o[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) o[c] = A[c] / L[c];

    const size_t oidx = (static_cast<size_t>(b) * nb + blk) * D + static_cast<size_t>(cg) * 8;
    if constexpr (kF32Out) {
      float4* op = reinterpret_cast<float4*>(static_cast<float*>(osel) + oidx);
      op[0] = make_float4(o[0], o[1], o[2], o[3]);
      op[1] = make_float4(o[4], o[5], o[6], o[7]);
    } else {
      uint4 v;
      v.x = pack_bf16x2(o[0], o[1]);
      v.y = pack_bf16x2(o[2], o[3]);
      v.z = pack_bf16x2(o[4], o[5]);
      v.w = pack_bf16x2(o[6], o[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(osel) + oidx) = v;
    }
  }
}

// Decode-time append: one thread per (query, 16-byte channel vector, stream).
// A query at position t with (t + 1) % m == 0 completes block (t + 1) / m - 1,
// whose m raw rows t - m + 1 .. t sit in the window buffer; they are folded
// exactly as compress_kernel folds a block (same chunks, same order), so the
// appended entry is bit-identical to the prefill compression of that block.
template <int R>
__global__ void __launch_bounds__(kThreads) append_kernel(AppendArgs a) {
  pdl_wait_then_release();
  const int sidx = blockIdx.y;
  const int D = sidx == 0 ? a.D[0] : (sidx == 1 ? a.D[1] : a.D[2]);
  const void* xsel = sidx == 0 ? a.x[0] : (sidx == 1 ? a.x[1] : a.x[2]);
  const void* gsel = sidx == 0 ? a.g[0] : (sidx == 1 ? a.g[1] : a.g[2]);
  void* osel = sidx == 0 ? a.out[0] : (sidx == 1 ? a.out[1] : a.out[2]);
  const int G = D >> 3;
  const long long nwork = static_cast<long long>(a.B) * a.Tq * G;
  const size_t row_bytes = static_cast<size_t>(D) * 2;
  for (long long wi = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; wi < nwork;
       wi += static_cast<long long>(gridDim.x) * kThreads) {
    const int cg = static_cast<int>(wi % G);
    const long long qi = wi / G;
    const int b = static_cast<int>(qi / a.Tq);
    const int t = a.q_pos[qi];
    if (t < 0 || (t + 1) % a.m != 0) continue;
    const int blk = (t + 1) / a.m - 1;
    const long long r0 = static_cast<long long>(t) - a.m + 1 - a.raw_base[b];
    if (blk >= a.N || r0 < 0 || r0 + a.m > a.T_raw) {
      if (cg == 0) raise_flag(a.errw, kFlagIndex);
      continue;
    }
    const size_t off = (static_cast<size_t>(b) * a.T_raw + static_cast<size_t>(r0)) * row_bytes +
                       static_cast<size_t>(cg) * 16;
    float M[8], L[8], A[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      M[c] = -INFINITY;
      L[c] = 0.f;
      A[c] = 0.f;
    }
    for (int j0 = 0; j0 < a.m; j0 += R)
      fold_rows<R>(static_cast<const char*>(xsel) + off + static_cast<size_t>(j0) * row_bytes,
                   static_cast<const char*>(gsel) + off + static_cast<size_t>(j0) * row_bytes, row_bytes, M, L, A);
    uint4 v;
    v.x = pack_bf16x2(A[0] / L[0], A[1] / L[1]);
    v.y = pack_bf16x2(A[2] / L[2], A[3] / L[3]);
    v.z = pack_bf16x2(A[4] / L[4], A[5] / L[5]);
    v.w = pack_bf16x2(A[6] / L[6], A[7] / L[7]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(osel) + (static_cast<size_t>(b) * a.N + blk) * D +
                              static_cast<size_t>(cg) * 8) = v;
  }
}

template <int R>
cudaError_t launch_r(const CompressArgs& a, dim3 grid, cudaStream_t s) {
  if (a.out_f32) return launch_k(compress_kernel<R, true>, grid, dim3(kThreads), 0, s, 1, a);
  return launch_k(compress_kernel<R, false>, grid, dim3(kThreads), 0, s, 1, a);
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t s) {
  long long maxwork = 0;
  for (int i = 0; i < a.n_streams; ++i) {
    const long long w = static_cast<long long>(a.B) * (a.T / a.m) * (a.D[i] / 8);
    maxwork = w > maxwork ? w : maxwork;
  }
  if (maxwork == 0) return cudaSuccess;
  long long blocks = (maxwork + kThreads - 1) / kThreads;
  const long long cap = 148LL * 8;  // grid-stride beyond eight resident blocks per SM
  if (blocks > cap) blocks = cap;
  dim3 grid(static_cast<unsigned>(blocks), a.n_streams);
  if (a.m % 8 == 0) return launch_r<8>(a, grid, s);
  if (a.m % 4 == 0) return launch_r<4>(a, grid, s);
  if (a.m % 2 == 0) return launch_r<2>(a, grid, s);
  return launch_r<1>(a, grid, s);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  long long maxwork = 0;
  for (int i = 0; i < a.n_streams; ++i) {
    const long long w = static_cast<long long>(a.B) * a.Tq * (a.D[i] / 8);
    maxwork = w > maxwork ? w : maxwork;
  }
  if (maxwork == 0) return cudaSuccess;
  long long blocks = (maxwork + kThreads - 1) / kThreads;
  if (blocks > 148LL * 8) blocks = 148LL * 8;
  const dim3 grid(static_cast<unsigned>(blocks), a.n_streams);
  if (a.m % 8 == 0) return launch_k(append_kernel<8>, grid, dim3(kThreads), 0, s, 1, a);
  if (a.m % 4 == 0) return launch_k(append_kernel<4>, grid, dim3(kThreads), 0, s, 1, a);
  if (a.m % 2 == 0) return launch_k(append_kernel<2>, grid, dim3(kThreads), 0, s, 1, a);
  return launch_k(append_kernel<1>, grid, dim3(kThreads), 0, s, 1, a);
}

}  // namespace csa
