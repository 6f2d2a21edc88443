// Bandwidth-bound kernels of the hot path and the device-image entry points:
//   - the associative log-sum-exp merge of partial results ("Unleashing Scalable Context
//     Parallelism for Foundation Models Pre-Training via FCP", Section 2.3: partial results
//     over slices of L reduced to the final output);
//   - the backward prologue Di = rowsum(dO * O), fused with zeroing the dQ accumulator;
//   - the dQ conversion (scale, float32 -> bf16);
//   - fcp_plan_upload / fcp_device_error.
// One warp handles one (head, token) row of D channels: lane l owns channels
// [l*D/32, (l+1)*D/32), so every global access of a warp is one contiguous span.
#include <cuda_bf16.h>

#include <cmath>

#include "fcp_cuda_util.h"
#include "fcp_sm100.cuh"

namespace fcp {
namespace {

constexpr int kRowWarps = 8;  // warps (rows) per 256-thread block

template <int D>
struct Vec;
template <>
struct Vec<128> {
  using F = float4;
  static constexpr int N = 4;
};
template <>
struct Vec<64> {
  using F = float2;
  static constexpr int N = 2;
};

__device__ __forceinline__ void vload(const float4* p, float (&x)[4]) {
  const float4 v = __ldg(p);
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void vload(const float2* p, float (&x)[2]) {
  const float2 v = __ldg(p);
  x[0] = v.x; x[1] = v.y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kMergeRows = 8;  // consecutive tokens per warp

template <int N>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* dst, const float (&x)[N], float inv) {
  if constexpr (N == 4) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0] * inv, x[1] * inv);
    __nv_bfloat162 b = __floats2bfloat162_rn(x[2] * inv, x[3] * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&a);
    pk.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(x[0] * inv, x[1] * inv);
  }
}

// One row merged by the whole warp: partials at rows off + k * stride (k < nr), walked 32 at
// a time. Used when the warp's rows have more partials than the unrolled path holds.
template <int D>
__device__ __forceinline__ void merge_row_general(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                                  long long off, int stride, int nr, int lane, float (&acc)[D / 32],
                                                  float& m_out, float& wsum_out) {
  using V = Vec<D>;
  constexpr int N = V::N;
  float m = -INFINITY;
  for (int i = lane; i < nr; i += 32) m = fmaxf(m, __ldg(part_lse + off + static_cast<long long>(i) * stride));
  m = warp_max(m);
#pragma unroll
  for (int e = 0; e < N; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int base = 0; base < nr; base += 32) {
      float w_l = 0.f;
      if (base + lane < nr) w_l = __expf(__ldg(part_lse + off + static_cast<long long>(base + lane) * stride) - m);
      const int cnt = min(32, nr - base);
#pragma unroll 4
      for (int i = 0; i < cnt; ++i) {
        const float w = __shfl_sync(0xffffffffu, w_l, i);
        const long long pr = off + static_cast<long long>(base + i) * stride;
        float x[N];
        vload(reinterpret_cast<const typename V::F*>(part_o + pr * D) + lane, x);
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = fmaf(w, x[e], acc[e]);
        wsum += w;
      }
    }
  }
  m_out = m;
  wsum_out = wsum;
}

constexpr int kMergePairs = 8;  // (row, partial) pairs a warp fetches at once

// grid (ceil(T / (kRowWarps * kMergeRows)), Hq): warp w of block x merges tokens
// [(x*kRowWarps + w) * kMergeRows, +kMergeRows) of head y. Each token's partial rows come
// from one 16-byte record (base, stride, count), so the partial rows of all the warp's
// (row, partial) pairs are loaded at once, independently of their LSEs.
template <int D>
__global__ void __launch_bounds__(32 * kRowWarps)
    merge_kernel(const TokPart* __restrict__ tok2part, const float* __restrict__ part_o,
                 const float* __restrict__ part_lse, long long part_rows, long long T, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ lse) {
  using V = Vec<D>;
  constexpr int N = V::N;
  constexpr int R = kMergeRows;
  const int lane = threadIdx.x & 31;
  const long long t0 = (static_cast<long long>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5)) * R;
  if (t0 >= T) return;
  const long long hoff = static_cast<long long>(blockIdx.y) * part_rows;

  int4 info = make_int4(0, 0, 0, 0);
  if (lane < R && t0 + lane < T) info = __ldg(reinterpret_cast<const int4*>(tok2part + t0 + lane));
  int nr[R], stride[R], start[R + 1];
  long long off[R];
  start[0] = 0;
  bool single = true;  // no row has more than one partial (rows past T have none)
#pragma unroll
  for (int i = 0; i < R; ++i) {
    off[i] = hoff + __shfl_sync(0xffffffffu, info.x, i);
    stride[i] = __shfl_sync(0xffffffffu, info.y, i);
    nr[i] = __shfl_sync(0xffffffffu, info.z, i);
    start[i + 1] = start[i] + nr[i];
    single = single && nr[i] <= 1;
  }
  const int P = start[R];

  const long long obase = static_cast<long long>(blockIdx.y) * T;
  if (P <= kMergePairs) {
    // pair p = (row i, partial k): lane p knows its row and partial-row index
    int myrow = -1;
    long long prow = 0;
    if (lane < P) {
      int i = 0;
#pragma unroll
      for (int j = 1; j < R; ++j)
        if (lane >= start[j]) i = j;
      long long oi = off[0];
      int si = stride[0], sti = start[0];
#pragma unroll
      for (int j = 1; j < R; ++j)
        if (i == j) {
          oi = off[j];
          si = stride[j];
          sti = start[j];
        }
      myrow = i;
      prow = oi + static_cast<long long>(lane - sti) * si;
    }
    // all partial rows in flight first, then the LSEs
    float x[kMergePairs][N];
#pragma unroll
    for (int p = 0; p < kMergePairs; ++p) {
      const long long pr = __shfl_sync(0xffffffffu, prow, p);
      if (p < P) {
        vload(reinterpret_cast<const typename V::F*>(part_o + pr * D) + lane, x[p]);
      } else {
#pragma unroll
        for (int e = 0; e < N; ++e) x[p][e] = 0.f;
      }
    }
    const float l = lane < P ? __ldg(part_lse + prow) : -INFINITY;
    if (single) {
      // one partial per row (every row's range has a single run): the merge is the identity
      // for rows with a finite LSE; rows without any visible key give O = 0, LSE = -inf.
      // Rows past T (no partial) come last, so pair i is row i for every stored row.
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const long long t = t0 + i;
        const float li = __shfl_sync(0xffffffffu, l, i);
        if (t < T) {
          store_bf16<N>(o + (obase + t) * D + lane * N, x[i], li == -INFINITY ? 0.f : 1.f);
          if (lane == i) lse[obase + t] = li;
        }
      }
    } else {
      // per row: m = max lse, w = exp(lse - m), out = sum w x / sum w
      float m_mine = -INFINITY;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const float mi = warp_max(myrow == i ? l : -INFINITY);
        if (myrow == i) m_mine = mi;
      }
      const float w = (myrow >= 0 && l != -INFINITY) ? __expf(l - m_mine) : 0.f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const long long t = t0 + i;
        float acc[N];
#pragma unroll
        for (int e = 0; e < N; ++e) acc[e] = 0.f;
        float ws = 0.f;
#pragma unroll
        for (int p = 0; p < kMergePairs; ++p) {
          const float wp = __shfl_sync(0xffffffffu, w, p);
          const int rp = __shfl_sync(0xffffffffu, myrow, p);
          const float wi = (rp == i) ? wp : 0.f;
          ws += wi;
#pragma unroll
          for (int e = 0; e < N; ++e) acc[e] = fmaf(wi, x[p][e], acc[e]);
        }
        const float mi = __shfl_sync(0xffffffffu, m_mine, start[i] < 32 ? start[i] : 0);
        if (t < T) {
          store_bf16<N>(o + (obase + t) * D + lane * N, acc, ws > 0.f ? 1.f / ws : 0.f);
          if (lane == i) lse[obase + t] = ws > 0.f ? mi + logf(ws) : -INFINITY;
        }
      }
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < R; ++i) {
      const long long t = t0 + i;
      float acc[N];
      float mi, wsi;
      const long long oi = hoff + __shfl_sync(0xffffffffu, info.x, i);
      const int si = __shfl_sync(0xffffffffu, info.y, i);
      const int ni = __shfl_sync(0xffffffffu, info.z, i);
      merge_row_general<D>(part_o, part_lse, oi, si, ni, lane, acc, mi, wsi);
      if (t < T) {
        store_bf16<N>(o + (obase + t) * D + lane * N, acc, wsi > 0.f ? 1.f / wsi : 0.f);
        if (lane == 0) lse[obase + t] = wsi > 0.f ? mi + logf(wsi) : -INFINITY;
      }
    }
  }
}

// Di[h,t] = sum_d dO*O and dq_acc[h,t,:] = 0. grid (ceil(T / kRowWarps), Hq).
template <int D>
__global__ void __launch_bounds__(32 * kRowWarps)
    prologue_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout, long long T,
                    float* __restrict__ di, float* __restrict__ dq_acc) {
  constexpr int N = D / 32;
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const long long row = static_cast<long long>(blockIdx.y) * T + t;
  const __nv_bfloat16* po = o + row * D + lane * N;
  const __nv_bfloat16* pd = dout + row * D + lane * N;
  float s = 0.f;
  if constexpr (N == 4) {
    const uint2 a = *reinterpret_cast<const uint2*>(po);
    const uint2 b = *reinterpret_cast<const uint2*>(pd);
    const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.x));
    const float2 a1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a.y));
    const float2 b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.x));
    const float2 b1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.y));
    s = a0.x * b0.x + a0.y * b0.y + a1.x * b1.x + a1.y * b1.y;
    reinterpret_cast<float4*>(dq_acc + row * D)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(po));
    const float2 b0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(pd));
    s = a0.x * b0.x + a0.y * b0.y;
    reinterpret_cast<float2*>(dq_acc + row * D)[lane] = make_float2(0.f, 0.f);
  }
  s = warp_sum(s);
  if (lane == 0) di[row] = s;
}

// dq[i] = bf16(scale * dq_acc[i]), 8 elements per thread, grid-stride.
__global__ void __launch_bounds__(256)
    dq_convert_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, long long n8, float scale) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
    __nv_bfloat162 r0 = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    __nv_bfloat162 r1 = __floats2bfloat162_rn(a.z * scale, a.w * scale);
    __nv_bfloat162 r2 = __floats2bfloat162_rn(b.x * scale, b.y * scale);
    __nv_bfloat162 r3 = __floats2bfloat162_rn(b.z * scale, b.w * scale);
    uint4 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&r0);
    pk.y = *reinterpret_cast<uint32_t*>(&r1);
    pk.z = *reinterpret_cast<uint32_t*>(&r2);
    pk.w = *reinterpret_cast<uint32_t*>(&r3);
    reinterpret_cast<uint4*>(dq)[i] = pk;
  }
}

// Row permutation between the user's and the workers' token layouts. Thread u of head group
// blockIdx.y owns 16-byte chunk (u % chunks) of worker-layout row (u / chunks) in eight heads:
// the row's user index is read once and the eight copies go out together, so each thread
// keeps eight independent 16-byte loads in flight. Consecutive threads touch consecutive
// chunks of a row, so the gathered and the scattered side both move whole rows; splitting
// the heads over the grid's y dimension keeps the CTAs small enough that the SMs finish
// together.
template <bool kToWorkers>
__global__ void __launch_bounds__(256)
    reshuffle_kernel(const int* __restrict__ order, const uint4* __restrict__ src, uint4* __restrict__ dst,
                     long long T, int chunks, int heads) {
  const long long units = T * chunks;  // (row, chunk) pairs of one head; also the head stride
  const int groups = (heads + 7) / 8;
  for (int g = blockIdx.y; g < groups; g += gridDim.y) {
    const int h0 = g * 8;
    const int nh = heads - h0 < 8 ? heads - h0 : 8;
    const uint4* s = src + h0 * units;
    uint4* d = dst + h0 * units;
    for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
         u += static_cast<long long>(gridDim.x) * blockDim.x) {
      const long long i = u / chunks;
      const long long c = u - i * chunks;
      const long long ui = static_cast<long long>(order[i]) * chunks + c;
      const long long from = kToWorkers ? ui : u;
      const long long to = kToWorkers ? u : ui;
      if (nh == 8) {
        uint4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __ldg(s + j * units + from);
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j * units + to] = x[j];
      } else {
        for (int j = 0; j < nh; ++j) d[j * units + to] = __ldg(s + j * units + from);
      }
    }
  }
}

}  // namespace

fcp_status launch_dq_convert(const float* dq_acc, void* dq, long long n, float scale, cudaStream_t s) {
  if (n == 0) return FCP_OK;
  const long long n8 = n / 8;  // n = Hq*T*D with D in {64, 128}
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (n8 + 255) / 256;
  const unsigned grid = static_cast<unsigned>(want < 8LL * sms ? want : 8LL * sms);
  dq_convert_kernel<<<grid, 256, 0, s>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), n8, scale);
  FCP_CUDA_TRY(cudaGetLastError(), "dq convert launch");
  return FCP_OK;
}

fcp_status launch_prologue(int64_t T, const void* o, const void* dout, int hq, int D, float* di, float* dq_acc,
                           cudaStream_t s) {
  if (T == 0) return FCP_OK;
  const dim3 grid(static_cast<unsigned>((T + kRowWarps - 1) / kRowWarps), static_cast<unsigned>(hq));
  const auto* po = static_cast<const __nv_bfloat16*>(o);
  const auto* pd = static_cast<const __nv_bfloat16*>(dout);
  if (D == 128)
    prologue_kernel<128><<<grid, 32 * kRowWarps, 0, s>>>(po, pd, T, di, dq_acc);
  else
    prologue_kernel<64><<<grid, 32 * kRowWarps, 0, s>>>(po, pd, T, di, dq_acc);
  FCP_CUDA_TRY(cudaGetLastError(), "bwd prologue launch");
  return FCP_OK;
}

}  // namespace fcp

using namespace fcp;

namespace fcp {
namespace {

// Two threads wait on barriers that nothing ever completes, each with one of the kernels'
// bounded waits: thread 0 with the polling wait of the forward (it records kErrSelfTest in
// the error word), thread 32 with the poll-then-suspend wait of the backward (it records
// kErrSelfTest + 1 in the word after it). Each gives up after the wait limit and returns.
__global__ void bounded_wait_selftest_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int abort_flag[2];
  if (threadIdx.x == 0) {
    dev::mbar_init(dev::smem_u32(&bar[0]), 1);
    dev::mbar_init(dev::smem_u32(&bar[1]), 1);
    abort_flag[0] = 0;
    abort_flag[1] = 0;
    dev::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) dev::mbar_wait(dev::smem_u32(&bar[0]), 0, &abort_flag[0], err, kErrSelfTest);
  if (threadIdx.x == 32)
    dev::mbar_wait_backoff<64, 1000u>(dev::smem_u32(&bar[1]), 0, &abort_flag[1], err + 1, kErrSelfTest + 1);
}

}  // namespace
}  // namespace fcp

extern "C" {

fcp_status fcp_plan_upload(const fcp_plan* plan, void* d_plan, size_t bytes, void* stream) {
  if (plan == nullptr || d_plan == nullptr) return FCP_ERR_INVALID;
  if (!plan->distributed) return FCP_ERR_STATE;
  if (bytes < plan->layout.total || (reinterpret_cast<uintptr_t>(d_plan) & 255u) != 0) return FCP_ERR_INVALID;
  FCP_CUDA_TRY(cudaMemcpyAsync(d_plan, plan->image.data(), plan->layout.total, cudaMemcpyHostToDevice,
                               static_cast<cudaStream_t>(stream)),
               "plan upload");
  return FCP_OK;
}

fcp_status fcp_selftest_bounded_wait(void* d_plan, void* stream) {
  if (d_plan == nullptr || (reinterpret_cast<uintptr_t>(d_plan) & 255u) != 0) return FCP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fcp::bounded_wait_selftest_kernel<<<1, 64, 0, s>>>(fcp::dev_error_word(d_plan));
  FCP_CUDA_TRY(cudaGetLastError(), "bounded-wait self-test launch");
  return FCP_OK;
}

fcp_status fcp_device_error(const void* d_plan, int32_t* code, void* stream) {
  if (d_plan == nullptr || code == nullptr) return FCP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  FCP_CUDA_TRY(cudaMemcpyAsync(&v, d_plan, sizeof(v), cudaMemcpyDeviceToHost, s), "error word read");
  FCP_CUDA_TRY(cudaStreamSynchronize(s), "error word sync");
  *code = v;
  if (v != 0) {
    FCP_CUDA_TRY(cudaMemsetAsync(const_cast<void*>(d_plan), 0, sizeof(int32_t), s), "error word clear");
    FCP_CUDA_TRY(cudaStreamSynchronize(s), "error word clear sync");
    return FCP_ERR_DEVICE;
  }
  return FCP_OK;
}

fcp_status fcp_block_attn_merge(const fcp_plan* plan, const void* d_plan, const float* part_o, const float* part_lse,
                                int32_t hq, int32_t head_dim, void* o, float* lse, void* stream) {
  if (plan == nullptr || d_plan == nullptr) return FCP_ERR_INVALID;
  if (!plan->distributed) return FCP_ERR_STATE;
  if (hq <= 0) return FCP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return FCP_ERR_UNSUPPORTED;
  const int64_t T = plan->total_tokens;
  if (T == 0) return FCP_OK;
  if (!part_o || !part_lse || !o || !lse || !aligned16(part_o) || !aligned16(o)) return FCP_ERR_INVALID;
  const DevLayout& L = plan->layout;
  const long long rows_per_block = static_cast<long long>(kRowWarps) * kMergeRows;
  const dim3 grid(static_cast<unsigned>((T + rows_per_block - 1) / rows_per_block), static_cast<unsigned>(hq));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto* tok2 = dev_array<TokPart>(d_plan, L.tok2part);
  auto* out = static_cast<__nv_bfloat16*>(o);
  if (head_dim == 128)
    merge_kernel<128><<<grid, 32 * kRowWarps, 0, s>>>(tok2, part_o, part_lse, plan->partial_rows, T, out, lse);
  else
    merge_kernel<64><<<grid, 32 * kRowWarps, 0, s>>>(tok2, part_o, part_lse, plan->partial_rows, T, out, lse);
  FCP_CUDA_TRY(cudaGetLastError(), "merge launch");
  return FCP_OK;
}

fcp_status fcp_reshuffle(const fcp_plan* plan, const void* d_plan, const void* src, void* dst, int32_t heads,
                         int32_t row_bytes, int32_t direction, void* stream) {
  if (plan == nullptr || d_plan == nullptr || heads <= 0 || row_bytes <= 0 || (row_bytes & 15) != 0 ||
      (direction != 0 && direction != 1))
    return FCP_ERR_INVALID;
  if (!plan->distributed) return FCP_ERR_STATE;
  const int64_t T = plan->total_tokens;
  if (T == 0) return FCP_OK;
  if (!src || !dst || src == dst || !aligned16(src) || !aligned16(dst)) return FCP_ERR_INVALID;
  const int chunks = row_bytes / 16;
  const long long units = static_cast<long long>(T) * chunks;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (units + 255) / 256;
  const int groups = (heads + 7) / 8;
  const dim3 grid(static_cast<unsigned>(want < 64LL * sms ? want : 64LL * sms),
                  static_cast<unsigned>(groups < 65535 ? groups : 65535));
  const auto* order = dev_array<int>(d_plan, plan->layout.worker_order);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (direction == 0)
    reshuffle_kernel<true><<<grid, 256, 0, s>>>(order, static_cast<const uint4*>(src), static_cast<uint4*>(dst), T,
                                               chunks, heads);
  else
    reshuffle_kernel<false><<<grid, 256, 0, s>>>(order, static_cast<const uint4*>(src), static_cast<uint4*>(dst), T,
                                                chunks, heads);
  FCP_CUDA_TRY(cudaGetLastError(), "reshuffle launch");
  return FCP_OK;
}

fcp_status fcp_block_attn_bwd_prologue(const fcp_plan* plan, const void* o, const void* dout, int32_t hq,
                                       int32_t head_dim, float* di, float* dq_acc, void* stream) {
  if (plan == nullptr || hq <= 0) return FCP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return FCP_ERR_UNSUPPORTED;
  if (plan->total_tokens == 0) return FCP_OK;
  if (!o || !dout || !di || !dq_acc || !aligned16(o) || !aligned16(dout) || !aligned16(dq_acc))
    return FCP_ERR_INVALID;
  return launch_prologue(plan->total_tokens, o, dout, hq, head_dim, di, dq_acc, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
