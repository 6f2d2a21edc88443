// Backward block attention over the FCP work list on sm_103a (tcgen05 + TMEM + TMA).
//
// The exact gradient of the attention of "Unleashing Scalable Context Parallelism for
// Foundation Models Pre-Training via FCP", Section 2.2 (the pages implement a backward but
// describe only the forward): with P = exp(S*scale - LSE) from the merged LSE,
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Di),  dQ = scale dS K,  dK = scale dS^T Q.
//
// CTA = one 128-row key tile of one key range and one KV head. It walks the reversed work
// list -- every item whose key range is this one -- for each of the G query heads of the
// group and each query tile that sees this key tile, accumulating dK and dV in TMEM over all
// of them, so dK/dV are written once, in bf16, without atomics. dQ of each (query tile, head)
// is produced in TMEM and added to a float32 accumulator with vector atomics.
// 10 warps:
//   warps 0-3  compute: thread = key row = TMEM lane; P^T and dS^T from S^T and dP^T
//   warps 4-7  dQ drain: thread = query row = TMEM lane; TMEM -> atomics into dq_acc
//   warp  8    TMA producer: K, V once; Q, dO per step (2 stages); LSE/Di rows to smem
//   warp  9    TMEM allocator and single-thread tcgen05.mma issuer
// TMEM columns: [0,128) S^T = K Q^T, later P^T (bf16, first 64 cols), later dQ = dS K;
// [128,256) dP^T = V dO^T, later dS^T (bf16, first 64 cols); [256,384) dV; [384,512) dK.
// Per step the MMAs run S^T, dP^T | dV += P^T dO, dK += dS^T Q, dQ = dS K, all issued by
// one thread in that order, so each MMA that overwrites TMEM columns follows the MMA that
// last read them.
#include <mutex>
#include <string>

#include "fcp_cuda_util.h"
#include "fcp_sm100.cuh"

namespace fcp {

fcp_status launch_prologue(int64_t T, const void* o, const void* dout, int hq, int D, float* di, float* dq_acc,
                           cudaStream_t s);
fcp_status launch_dq_convert(const float* dq_acc, void* dq, long long n, float scale, cudaStream_t s);
fcp_status launch_bwd_d128(const fcp_plan* plan, const void* d_plan, const void* q, const void* k, const void* v,
                           const void* dout, const float* lse, const float* di, float* dq_acc, void* dk, void* dv,
                           int hq, int hkv, cudaStream_t stream);

namespace {

using namespace dev;

constexpr int kBwdThreads = 320;
constexpr int kPanelBytes = kTileM * 128;

struct BwdArgs {
  const fcp_item* items;
  const KvSeg* kvsegs;
  const int* kv_items;
  const BwdUnit* units;
  const float* lse;  // [Hq, T]
  const float* di;   // [Hq, T]
  float* dq_acc;     // [Hq, T, D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  long long T;
  int hq, hkv, group;
  float scale_log2, scale;
  int* err;
};

enum : int {
  B_KVFULL = 0,
  B_QFULL = 1,     // 2 stages (Q, dO, LSE, Di)
  B_QEMPTY = 3,    // 2 stages
  B_STFULL = 5,    // S^T and dP^T ready
  B_DSFULL = 6,    // P^T, dS^T written (TMEM + smem)
  B_DSEMPTY = 7,   // dS smem tile consumed (dQ MMA done)
  B_DQFULL = 8,    // dQ ready in TMEM
  B_DQEMPTY = 9,   // dQ drained from TMEM
  B_ACCDONE = 10,  // all dK/dV MMAs done
  B_COUNT = 11
};

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kPanels = D / 64;
  static constexpr int kK = 0;
  static constexpr int kV = kTileBytes;
  static constexpr int kQ = 2 * kTileBytes;             // 2 stages
  static constexpr int kDO = 4 * kTileBytes;            // 2 stages
  static constexpr int kDS = 6 * kTileBytes;            // [128 kv][128 q] bf16, 2 panels of 64 q
  static constexpr int kVec = kDS + kTileM * kTileN * 2;  // LSE*log2e and Di, 2 stages x 2 x 128 floats
  static constexpr int kBar = kVec + 2 * 2 * kTileM * 4;
  // at least half the SM's shared memory, so one CTA per SM holds all 512 TMEM columns
  static constexpr int kSmemBytes = (kBar + 128) > 118 * 1024 ? (kBar + 128) : 118 * 1024;
  static constexpr uint32_t kIdescST = idesc_bf16(kTileN, kTileM, false, false);  // M = keys, N = queries
  static constexpr uint32_t kIdescAcc = idesc_bf16(kTileN, D, false, true);      // dV, dK: B = dO/Q MN-major
  static constexpr uint32_t kIdescDQ = idesc_bf16(kTileM, D, true, true);        // A = dS (MN-major), B = K
};

// Query tiles of item `it` that see key tile kt: [first, end).
__device__ __forceinline__ int q_first(const fcp_item& it, int kt) {
  return it.mask == FCP_MASK_CAUSAL_DIAG ? kt : 0;
}
__device__ __forceinline__ int q_end(const fcp_item& it) { return (it.q_len + kTileM - 1) / kTileM; }

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte-swizzled TMA/MMA tiles need a 1024-byte aligned base; report, never fault
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(a.err, 0, kErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sb = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kBar + B_COUNT * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBar + B_COUNT * 8 + 4);
  float* vec = reinterpret_cast<float*>(smem + C::kVec);  // [stage][lse2 | di][128]
  auto bar = [&](int i) -> uint32_t { return sb + C::kBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int unit_idx = blockIdx.x / a.hkv;
  const int kvh = blockIdx.x - unit_idx * a.hkv;
  const BwdUnit unit = a.units[unit_idx];
  const KvSeg seg = a.kvsegs[unit.kvseg];
  const int kt = unit.kv_tile;
  const int kv_row0 = seg.tok0 + kt * kTileN;
  const int kv_valid = seg.len - kt * kTileN;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KVFULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL + s), 32);
      mbar_init(bar(B_QEMPTY + s), 1);
    }
    mbar_init(bar(B_STFULL), 1);
    mbar_init(bar(B_DSFULL), kTileN);
    mbar_init(bar(B_DSEMPTY), 1);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQEMPTY), kTileM);
    mbar_init(bar(B_ACCDONE), 1);
    *abort_flag = (*reinterpret_cast<volatile int*>(a.err) != 0) ? 1 : 0;
    mbar_fence_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  // The step sequence (head, item, query tile) is walked identically by every role; the
  // body returns false to stop (a wait gave up).
  auto for_each_step = [&](auto&& body) -> int {
    int step = 0;
    for (int hh = 0; hh < a.group; ++hh) {
      const int h = kvh * a.group + hh;
      for (int li = seg.list_begin; li < seg.list_end; ++li) {
        const fcp_item itm = a.items[a.kv_items[li]];
        const int qe = q_end(itm);
        for (int qt = q_first(itm, kt); qt < qe; ++qt, ++step)
          if (!body(step, h, itm, qt)) return step;
      }
    }
    return step;
  };

  int n_steps = 0;
  if (warp == 8) {
    // ------------------------------------------------------------ producer warp
    bool ok = !skip;
    if (ok && lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(bar(B_KVFULL), 2 * C::kTileBytes);
#pragma unroll
      for (int p = 0; p < C::kPanels; ++p) {
        tma_load_3d(sb + C::kK + p * kPanelBytes, &tmK, bar(B_KVFULL), p * 64, kv_row0, kvh);
        tma_load_3d(sb + C::kV + p * kPanelBytes, &tmV, bar(B_KVFULL), p * 64, kv_row0, kvh);
      }
    }
    n_steps = for_each_step([&](const int step, const int h, const fcp_item& itm, const int qt) -> bool {
      const int s = step & 1;
      const uint32_t ph = (step >> 1) & 1;
      ok = mbar_wait(bar(B_QEMPTY + s), ph ^ 1, abort_flag, a.err, kErrBwdWait + 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return false;
      const int qrow0 = itm.q_tok0 + qt * kTileM;
      const int q_valid = itm.q_len - qt * kTileM;
      if (lane == 0) {
        mbar_expect_tx(bar(B_QFULL + s), 2 * C::kTileBytes);
#pragma unroll
        for (int p = 0; p < C::kPanels; ++p) {
          tma_load_3d(sb + C::kQ + s * C::kTileBytes + p * kPanelBytes, &tmQ, bar(B_QFULL + s), p * 64, qrow0, h);
          tma_load_3d(sb + C::kDO + s * C::kTileBytes + p * kPanelBytes, &tmDO, bar(B_QFULL + s), p * 64, qrow0, h);
        }
      }
      // LSE (pre-scaled to log2 units) and Di of the tile's query rows; rows past the range
      // get LSE = +inf (P = 0) and Di = 0.
      float* v = vec + s * 2 * kTileM;
      const long long rowbase = static_cast<long long>(h) * a.T + qrow0;
#pragma unroll
      for (int i = 0; i < kTileM / 32; ++i) {
        const int c = i * 32 + lane;
        const bool in = c < q_valid;
        v[c] = in ? a.lse[rowbase + c] * 1.4426950408889634f : INFINITY;
        v[kTileM + c] = in ? a.di[rowbase + c] : 0.f;
      }
      mbar_arrive(bar(B_QFULL + s));
      return true;
    });
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = !skip;
    if (lane == 0) {
      if (ok) ok = mbar_wait(bar(B_KVFULL), 0, abort_flag, a.err, kErrBwdWait + 2);
      tc_fence_after();
      const uint32_t t_st = tmem, t_dpt = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 384;
      n_steps = for_each_step([&](const int step, const int h, const fcp_item& itm, const int qt) -> bool {
        const int s = step & 1;
        const uint32_t ph = (step >> 1) & 1;
        ok = mbar_wait(bar(B_QFULL + s), ph, abort_flag, a.err, kErrBwdWait + 3);
        if (ok && step > 0) ok = mbar_wait(bar(B_DQEMPTY), (step - 1) & 1, abort_flag, a.err, kErrBwdWait + 4);
        if (!ok) return false;
        tc_fence_after();
        const uint32_t qb = sb + C::kQ + s * C::kTileBytes;
        const uint32_t db = sb + C::kDO + s * C::kTileBytes;
        // S^T = K Q^T and dP^T = V dO^T (M = 128 keys, N = 128 queries, K = D)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
          mma_ss(t_st, sdesc_sw128(sb + C::kK + off, 16, 1024), sdesc_sw128(qb + off, 16, 1024), C::kIdescST, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
          mma_ss(t_dpt, sdesc_sw128(sb + C::kV + off, 16, 1024), sdesc_sw128(db + off, 16, 1024), C::kIdescST,
                 kk > 0);
        }
        tc_commit(bar(B_STFULL));
        ok = mbar_wait(bar(B_DSFULL), step & 1, abort_flag, a.err, kErrBwdWait + 5);
        if (!ok) return false;
        tc_fence_after();
        // dV += P^T dO, dK += dS^T Q (M = 128 keys, N = D, K = 128 queries; A from TMEM)
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {
          mma_ts(t_dv, t_st + kk * 8, sdesc_sw128(db + kk * 2048, kPanelBytes, 1024), C::kIdescAcc,
                 (step > 0 || kk > 0));
        }
#pragma unroll
        for (int kk = 0; kk < kTileM / 16; ++kk) {
          mma_ts(t_dk, t_dpt + kk * 8, sdesc_sw128(qb + kk * 2048, kPanelBytes, 1024), C::kIdescAcc,
                 (step > 0 || kk > 0));
        }
        // dQ = dS K (M = 128 queries, N = D, K = 128 keys): A = dS^T tile in smem read
        // MN-major, B = K tile read MN-major
#pragma unroll
        for (int kk = 0; kk < kTileN / 16; ++kk) {
          mma_ss(t_st, sdesc_sw128(sb + C::kDS + kk * 2048, kPanelBytes, 1024),
                 sdesc_sw128(sb + C::kK + kk * 2048, kPanelBytes, 1024), C::kIdescDQ, kk > 0);
        }
        tc_commit(bar(B_DQFULL));
        tc_commit(bar(B_DSEMPTY));
        tc_commit(bar(B_QEMPTY + s));
        return true;
    });
      tc_commit(bar(B_ACCDONE));
      // B_ACCDONE is also the drain: every MMA above has completed once it fires
      if (!ok) mbar_wait(bar(B_ACCDONE), 0, abort_flag, a.err, kErrBwdWait + 6);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ compute warps
    bool ok = !skip;
    const int r = warp * 32 + lane;  // key row in tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint8_t* ds_row = smem + C::kDS + (r >> 3) * 1024 + (r & 7) * 128;
    n_steps = for_each_step([&](const int step, const int h, const fcp_item& itm, const int qt) -> bool {
      const int s = step & 1;
      const bool diag = itm.mask == FCP_MASK_CAUSAL_DIAG && qt == kt;
      // visible query columns of this key row: [qmin, 128); rows past the key range see none
      const int qmin = (r >= kv_valid) ? kTileM : (diag ? r : 0);
      ok = mbar_wait(bar(B_QFULL + s), (step >> 1) & 1, abort_flag, a.err, kErrBwdWait + 7);
      if (ok) ok = mbar_wait(bar(B_STFULL), step & 1, abort_flag, a.err, kErrBwdWait + 8);
      if (ok && step > 0) ok = mbar_wait(bar(B_DSEMPTY), (step - 1) & 1, abort_flag, a.err, kErrBwdWait + 9);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return false;
      tc_fence_after();
      const float* lse2 = vec + s * 2 * kTileM;
      const float* dis = lse2 + kTileM;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sv[32], dv[32];
        tmem_ld32(lane_base + c * 32, sv);
        tmem_ld32(lane_base + 128 + c * 32, dv);
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int q0 = c * 32 + 2 * e;
          float p0 = 0.f, p1 = 0.f, d0 = 0.f, d1 = 0.f;
          if (q0 >= qmin) {
            p0 = fast_exp2(fmaf(__uint_as_float(sv[2 * e]), a.scale_log2, -lse2[q0]));
            d0 = p0 * (__uint_as_float(dv[2 * e]) - dis[q0]);
          }
          if (q0 + 1 >= qmin) {
            p1 = fast_exp2(fmaf(__uint_as_float(sv[2 * e + 1]), a.scale_log2, -lse2[q0 + 1]));
            d1 = p1 * (__uint_as_float(dv[2 * e + 1]) - dis[q0 + 1]);
          }
          pp[e] = pack_bf16(p0, p1);
          dd[e] = pack_bf16(d0, d1);
        }
        tmem_st16(lane_base + c * 16, pp);
        tmem_st16(lane_base + 128 + c * 16, dd);
        // dS^T row r, queries [32c, 32c+32) -> panel c/2, 16-byte chunks (c&1)*4 .. +3,
        // 128-byte swizzle: chunk index XOR (row & 7)
        uint8_t* prow = ds_row + (c >> 1) * (kTileN * 128);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int chunk = ((c & 1) * 4 + x) ^ (r & 7);
          *reinterpret_cast<uint4*>(prow + chunk * 16) = make_uint4(dd[4 * x], dd[4 * x + 1], dd[4 * x + 2], dd[4 * x + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_DSFULL));
      return true;
    });
    // epilogue: dV and scale * dK of this key tile, bf16
    if (ok) ok = mbar_wait(bar(B_ACCDONE), 0, abort_flag, a.err, kErrBwdWait + 10);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const bool store = r < kv_valid;
      const long long row = static_cast<long long>(kvh) * a.T + kv_row0 + r;
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = (which == 0 ? a.dv : a.dk) + row * D;
        const float f = which == 0 ? 1.f : a.scale;
        const uint32_t base = lane_base + (which == 0 ? 256 : 384);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32];
          if (n_steps > 0) {
            tmem_ld32(base + c * 32, x);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = 0u;
          }
          if (store) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 pk;
              pk.x = pack_bf16(__uint_as_float(x[8 * e + 0]) * f, __uint_as_float(x[8 * e + 1]) * f);
              pk.y = pack_bf16(__uint_as_float(x[8 * e + 2]) * f, __uint_as_float(x[8 * e + 3]) * f);
              pk.z = pack_bf16(__uint_as_float(x[8 * e + 4]) * f, __uint_as_float(x[8 * e + 5]) * f);
              pk.w = pack_bf16(__uint_as_float(x[8 * e + 6]) * f, __uint_as_float(x[8 * e + 7]) * f);
              reinterpret_cast<uint4*>(dst + c * 32)[e] = pk;
            }
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain warps (4-7)
    bool ok = !skip;
    const int r = (warp - 4) * 32 + lane;  // query row in tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp - 4) * 32) << 16);
    n_steps = for_each_step([&](const int step, const int h, const fcp_item& itm, const int qt) -> bool {
      ok = mbar_wait(bar(B_DQFULL), step & 1, abort_flag, a.err, kErrBwdWait + 11);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return false;
      tc_fence_after();
      const bool store = qt * kTileM + r < itm.q_len;
      float* dst = a.dq_acc + (static_cast<long long>(h) * a.T + itm.q_tok0 + qt * kTileM + r) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t x[32];
        tmem_ld32(lane_base + c * 32, x);
        if (store) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            atomicAdd(reinterpret_cast<float4*>(dst + c * 32) + e,
                      make_float4(__uint_as_float(x[4 * e]), __uint_as_float(x[4 * e + 1]),
                                  __uint_as_float(x[4 * e + 2]), __uint_as_float(x[4 * e + 3])));
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_DQEMPTY));
      return true;
    });
  }

  if (*abort_flag) {
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) __nanosleep(1000);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
fcp_status launch_bwd(const fcp_plan* plan, const void* d_plan, const void* q, const void* k, const void* v,
                      const void* dout, const float* lse, const float* di, float* dq_acc, void* dk, void* dv,
                      int hq, int hkv, cudaStream_t stream) {
  if constexpr (D == 128) {
    // head_dim 128 runs the pipelined kernel with 64-row query steps
    return launch_bwd_d128(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, stream);
  } else {
  using C = BwdCfg<D>;
  const DevLayout& L = plan->layout;
  if (L.n_bwd_units == 0) return FCP_OK;
  const int64_t T = plan->total_tokens;
  CUtensorMap mq, mk, mv, mdo;
  fcp_status st;
  if ((st = make_bf16_map(&mq, q, hq, T, D, kTileM)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mk, k, hkv, T, D, kTileN)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mv, v, hkv, T, D, kTileN)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mdo, dout, hq, T, D, kTileM)) != FCP_OK) return st;
  BwdArgs a;
  a.items = dev_array<fcp_item>(d_plan, L.items);
  a.kvsegs = dev_array<KvSeg>(d_plan, L.kvsegs);
  a.kv_items = dev_array<int>(d_plan, L.kv_items);
  a.units = dev_array<BwdUnit>(d_plan, L.bwd_units);
  a.lse = lse;
  a.di = di;
  a.dq_acc = dq_acc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.T = T;
  a.hq = hq;
  a.hkv = hkv;
  a.group = hq / hkv;
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  a.err = dev_error_word(d_plan);
  FCP_CUDA_TRY(cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes),
               "bwd smem attribute");
  const long long grid = static_cast<long long>(L.n_bwd_units) * hkv;
  if (grid > 0x7fffffffLL) return FCP_ERR_UNSUPPORTED;
  bwd_kernel<D><<<static_cast<unsigned>(grid), kBwdThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mdo, a);
  FCP_CUDA_TRY(cudaGetLastError(), "bwd launch");
  return FCP_OK;
  }
}

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
  if (head_dim == 128) return launch_bwd<128>(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, s);
  return launch_bwd<64>(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, s);
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
  if (head_dim == 128)
    st = launch_bwd<128>(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, s);
  else
    st = launch_bwd<64>(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, s);
  if (st != FCP_OK) return st;
  return launch_dq_convert(dq_acc, dq, static_cast<long long>(hq) * T * head_dim,
                           static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim))), s);
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
// current) and cached.
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
