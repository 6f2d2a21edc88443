// Backward entry points over the FCP work list (the tile kernel is in fcp_bwd_tile.cu).
//
// The exact gradient of the attention of "Unleashing Scalable Context Parallelism for
// Foundation Models Pre-Training via FCP", Section 2.2 (the pages implement a backward but
// describe only the forward): with P = exp(S*scale - LSE) from the merged LSE,
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Di),  dQ = scale dS K,  dK = scale dS^T Q.
// fcp_block_attn_bwd runs the Di prologue (which also zeroes the float32 dQ accumulator),
// the tile kernel and the dQ conversion to bf16; the three parts are also exported alone,
// and an allocation-free variant keeps its scratch in a fixed device array.
#include <mutex>
#include <string>

#include "fcp_cuda_util.h"
#include "fcp_sm100.cuh"

namespace fcp {

fcp_status launch_prologue(int64_t T, const void* o, const void* dout, int hq, int D, float* di, float* dq_acc,
                           cudaStream_t s);
fcp_status launch_dq_convert(const float* dq_acc, void* dq, long long n, float scale, cudaStream_t s);
fcp_status launch_bwd_tiles(const fcp_plan* plan, const void* d_plan, const void* q, const void* k, const void* v,
                            const void* dout, const float* lse, const float* di, float* dq_acc, void* dk, void* dv,
                            int hq, int hkv, int head_dim, float* dk_acc, float* dv_acc, cudaStream_t stream);

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace fcp

using namespace fcp;

namespace {
fcp_status check_common(const fcp_plan* plan, const void* d_plan, int32_t hq, int32_t hkv, int32_t head_dim) {
  if (plan == nullptr || d_plan == nullptr) return FCP_ERR_INVALID;
  if (!plan->distributed) return FCP_ERR_STATE;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return FCP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return FCP_ERR_UNSUPPORTED;
  return FCP_OK;
}
}  // namespace

extern "C" fcp_status fcp_block_attn_bwd_tiles(const fcp_plan* plan, const void* d_plan, const void* q,
                                               const void* k, const void* v, const void* dout, const float* lse,
                                               const float* di, int32_t hq, int32_t hkv, int32_t head_dim,
                                               float* dq_acc, void* dk, void* dv, void* stream) {
  fcp_status st = check_common(plan, d_plan, hq, hkv, head_dim);
  if (st != FCP_OK) return st;
  if (plan->total_tokens == 0) return FCP_OK;
  if (!q || !k || !v || !dout || !lse || !di || !dq_acc || !dk || !dv) return FCP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(dq_acc))
    return FCP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_bwd_tiles(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, head_dim, nullptr, nullptr,
                          s);
}

extern "C" fcp_status fcp_block_attn_bwd_dq_convert(const fcp_plan* plan, const float* dq_acc, int32_t hq,
                                                    int32_t head_dim, void* dq, void* stream) {
  if (plan == nullptr || hq <= 0) return FCP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return FCP_ERR_UNSUPPORTED;
  if (plan->total_tokens == 0) return FCP_OK;
  if (!dq_acc || !dq || !aligned16(dq_acc) || !aligned16(dq)) return FCP_ERR_INVALID;
  return launch_dq_convert(dq_acc, dq, static_cast<long long>(hq) * plan->total_tokens * head_dim,
                           static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim))),
                           static_cast<cudaStream_t>(stream));
}

extern "C" fcp_status fcp_block_attn_bwd(const fcp_plan* plan, const void* d_plan, const void* q, const void* k,
                                         const void* v, const void* o, const void* dout, const float* lse,
                                         int32_t hq, int32_t hkv, int32_t head_dim, void* dq, void* dk, void* dv,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (plan == nullptr || d_plan == nullptr) return FCP_ERR_INVALID;
  if (!plan->distributed) return FCP_ERR_STATE;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return FCP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return FCP_ERR_UNSUPPORTED;
  const int64_t T = plan->total_tokens;
  if (T == 0) return FCP_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FCP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FCP_ERR_INVALID;
  if (workspace_bytes < fcp_bwd_workspace_bytes(plan, hq, head_dim)) return FCP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* dq_acc = static_cast<float*>(workspace);
  float* di = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                       align256(size_t(hq) * size_t(T) * size_t(head_dim) * sizeof(float)));
  fcp_status st = launch_prologue(T, o, dout, hq, head_dim, di, dq_acc, s);
  if (st != FCP_OK) return st;
  // query bands when the plan has them and the workspace holds their dK/dV sums
  const size_t base = fcp_bwd_workspace_bytes(plan, hq, head_dim);
  const size_t band = fcp_bwd_band_workspace_bytes(plan, hkv, head_dim);
  if (band > 0 && workspace_bytes >= base + band) {
    float* dkv_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + base);
    st = fcp_block_attn_bwd_tiles_banded(plan, d_plan, q, k, v, dout, lse, di, hq, hkv, head_dim, dq_acc, dkv_acc,
                                         dk, dv, stream);
  } else {
    st = launch_bwd_tiles(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, head_dim, nullptr, nullptr,
                          s);
  }
  if (st != FCP_OK) return st;
  return launch_dq_convert(dq_acc, dq, static_cast<long long>(hq) * T * head_dim,
                           static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim))), s);
}

extern "C" fcp_status fcp_block_attn_bwd_tiles_banded(const fcp_plan* plan, const void* d_plan, const void* q,
                                                      const void* k, const void* v, const void* dout,
                                                      const float* lse, const float* di, int32_t hq, int32_t hkv,
                                                      int32_t head_dim, float* dq_acc, float* dkv_acc, void* dk,
                                                      void* dv, void* stream) {
  fcp_status st = check_common(plan, d_plan, hq, hkv, head_dim);
  if (st != FCP_OK) return st;
  if (plan->layout.n_bands == 0) return FCP_ERR_STATE;
  const int64_t T = plan->total_tokens;
  if (T == 0) return FCP_OK;
  if (!q || !k || !v || !dout || !lse || !di || !dq_acc || !dkv_acc || !dk || !dv) return FCP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(dq_acc) || (reinterpret_cast<uintptr_t>(dkv_acc) & 255u) != 0)
    return FCP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t half = align256(size_t(hkv) * size_t(T) * size_t(head_dim) * sizeof(float));
  float* dk_acc = dkv_acc;
  float* dv_acc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dkv_acc) + half);
  FCP_CUDA_TRY(cudaMemsetAsync(dkv_acc, 0, 2 * half, s), "band accumulators");
  st = launch_bwd_tiles(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, head_dim, dk_acc, dv_acc, s);
  if (st != FCP_OK) return st;
  const long long n = static_cast<long long>(hkv) * T * head_dim;
  st = launch_dq_convert(dk_acc, dk, n, static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim))), s);
  if (st != FCP_OK) return st;
  return launch_dq_convert(dv_acc, dv, n, 1.0f, s);
}

// ---------------------------------------------------------------------------------------
// Backward without any allocation by the caller or the library.
//
// Some callers cannot call cudaMalloc at all: code that runs inside a memory pool or
// arena that owns every byte of the device (a framework that pre-reserved the GPU), code
// on a path where allocating would synchronise the device or break an allocation-free
// contract (real-time or inference-serving loops), or plain C hosts without a device
// allocator of their own. For them the backward's scratch (the float32 dQ accumulator and
// Di) lives in a fixed array in device memory that this library owns. Every GPU that
// loads the library holds this array until the process exits.
namespace fcp {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_bwd_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device. The host-side name of the array
// is only a stand-in, so the address is looked up once per device (with that device
// current) and cached for the life of the process; a cudaDeviceReset discards the array
// with the context, so the entry point is not for use on a device after a reset.
fcp_status static_scratch(void** out) {
  int dev = 0;
  FCP_CUDA_TRY(cudaGetDevice(&dev), "static scratch: current device");
  if (dev < 0 || dev >= kMaxDevices) return FCP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    FCP_CUDA_TRY(cudaGetSymbolAddress(&p, g_bwd_scratch), "static scratch: cudaGetSymbolAddress");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FCP_OK;
}

}  // namespace
}  // namespace fcp

extern "C" size_t fcp_bwd_static_scratch_bytes(void) { return fcp::kStaticScratchBytes; }

extern "C" fcp_status fcp_block_attn_bwd_static_scratch(const fcp_plan* plan, const void* d_plan, const void* q,
                                                        const void* k, const void* v, const void* o,
                                                        const void* dout, const float* lse, int32_t hq,
                                                        int32_t hkv, int32_t head_dim, void* dq, void* dk, void* dv,
                                                        void* stream) {
  if (plan == nullptr || hq <= 0 || head_dim <= 0) return FCP_ERR_INVALID;
  const size_t need = fcp_bwd_workspace_bytes(plan, hq, head_dim);
  if (need > fcp::kStaticScratchBytes) {
    fcp::set_last_error("backward scratch of " + std::to_string(need) + " bytes exceeds the library's static " +
                        std::to_string(fcp::kStaticScratchBytes) + "-byte array; use fcp_block_attn_bwd");
    return FCP_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  fcp_status st = fcp::static_scratch(&scratch);
  if (st != FCP_OK) return st;
  // The prologue rewrites the whole dQ accumulator with zeros and Di in full on every call,
  // so what the previous call left in the array does not matter.
  return fcp_block_attn_bwd(plan, d_plan, q, k, v, o, dout, lse, hq, hkv, head_dim, dq, dk, dv, scratch,
                            fcp::kStaticScratchBytes, stream);
}
