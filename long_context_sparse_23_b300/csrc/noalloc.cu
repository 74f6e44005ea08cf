// csa_attend_noalloc: csa_attend for callers that cannot allocate device
// memory.  Some hosts hand a custom operator only its inputs and outputs --
// their memory planner owns the rest of the device and offers no scratch
// allocator -- and some latency-bound callers must never reach cudaMalloc /
// cudaFree, which can synchronise the whole device.  This entry point takes
// no workspace: the split-KV partials that csa_attend keeps in the caller's
// workspace live instead in one file-scope device array of fixed size, which
// every GPU that loads the library holds until the process exits.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/csa.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;

// Scratch for the split-KV partials (normalised O and log2-sum-exp per split).
static __device__ __align__(256) char g_noalloc_scratch[CSA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, per device.  In host code the array's
// name is only a host-side handle, so the address is asked for once per device
// (with that device current) and reused.
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" csa_status csa_attend_noalloc(const void* q, const void* k_cmp, const void* v_cmp,
                                         const int32_t* idx, const void* k_raw, const void* v_raw,
                                         const int32_t* raw_base, const int32_t* q_pos, int B,
                                         int Tq, int N, int T_raw, int H, int d, int k, int W,
                                         float scale, void* out, int out_dtype, float* lse,
                                         void* stream) {
  // the same argument rules as csa_attend
  if (!q || !q_pos || !out) return CSA_ERR_INVALID;
  if (B <= 0 || Tq <= 0 || N < 0 || T_raw < 0 || H <= 0 || d <= 0 || W < 0 || k < 0)
    return CSA_ERR_INVALID;
  if (N > 0 && (!k_cmp || !v_cmp)) return CSA_ERR_INVALID;
  if (W > 0 && (!k_raw || !v_raw || !raw_base || T_raw <= 0)) return CSA_ERR_INVALID;
  if (k > 0 && (!idx || !al4(idx) || N <= 0)) return CSA_ERR_INVALID;
  if (!al16(q) || !al16(out) || (k_cmp && !al16(k_cmp)) || (v_cmp && !al16(v_cmp)) ||
      (k_raw && !al16(k_raw)) || (v_raw && !al16(v_raw)) || !al4(q_pos) ||
      (raw_base && !al4(raw_base)) || (lse && !al4(lse)))
    return CSA_ERR_INVALID;
  if (out_dtype != CSA_BF16 && out_dtype != CSA_F32) return CSA_ERR_INVALID;
  if (d != 64 && d != 128) return CSA_ERR_UNSUPPORTED;
  if (H > 64) return CSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Tq >= 65536LL * 1024) return CSA_ERR_UNSUPPORTED;

  // the partials must fit the fixed scratch
  const long long nq = static_cast<long long>(B) * Tq;
  const csa::AttendPlan plan = csa::plan_attend(Tq, nq, k + W, H, d);
  if (plan.part_bytes > static_cast<size_t>(CSA_NOALLOC_SCRATCH_BYTES)) return CSA_ERR_WORKSPACE;

  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return CSA_ERR_CUDA;

  csa::AttendArgs a;
  a.q = q;
  a.k_cmp = k_cmp;
  a.v_cmp = v_cmp;
  a.idx = idx ? idx : q_pos;  // k == 0: the (empty) index list is never read
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
  a.m = 1;
  a.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(d));
  a.out = out;
  a.out_f32 = out_dtype == CSA_F32;
  a.lse = lse;
  a.part = static_cast<float*>(scratch);
  a.errw = nullptr;  // no error word: out-of-range indices are skipped unreported
  const cudaError_t e = csa::launch_attend(a, plan, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) return CSA_OK;
  return e == cudaErrorNotSupported ? CSA_ERR_UNSUPPORTED : CSA_ERR_CUDA;
}
