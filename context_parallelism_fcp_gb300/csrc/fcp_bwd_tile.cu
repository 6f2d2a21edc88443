// Backward block attention on sm_103a (head_dim 64 or 128): a pipelined tile kernel.
//
// The exact gradient of the attention of "Unleashing Scalable Context Parallelism for
// Foundation Models Pre-Training via FCP" (Section 2.2) over the reversed work list: one CTA
// owns a 128-row key tile of one key range and one KV head, and walks every (query head of
// the group, item reading this key range, query step) accumulating dK and dV in TMEM.
//
// A query step is 64 rows, so the S^T/dP^T accumulators of a step need 128 TMEM columns and
// two steps fit beside dV and dK:
//   columns [128b, 128b+64)     S^T of buffer b (b = step & 1); P^T (bf16) overwrites
//                               [128b+16, 128b+48)
//   columns [128b+64, 128b+128) dP^T; dS^T (bf16) overwrites [128b+80, 128b+112); later
//                               dQ^T = K^T dS^T (128 lanes = channels x 64 queries)
//   columns [256, 256+D) dV, [384, 384+D) dK
// Each gradient warpgroup reads 32 columns of S^T and of dP^T and writes its packed half of
// P^T and dS^T inside the columns it has itself just read, so the two warpgroups never
// need to wait for each other. S^T of step i+2 may be issued before the drain of step i
// has read dQ^T (they occupy different halves of the buffer); only dP^T waits for it.
// The MMA warp issues S^T/dP^T of step i+1 before it waits for the gradient warps of step
// i, so the tensor core works on the next step while the current one is turned into P and
// dS. dQ^T is computed with the channels on TMEM lanes (M = 128: for D = 64 the upper 64
// channels read a zero panel and are never drained), so the drain warps stage it in shared
// memory with one 128-byte line per warp store and add it to the float32 accumulator with
// one TMA reduce per step, freeing the TMEM buffer as soon as the values are in registers.
// Warps: 0-7 gradient (two warpgroups, 32 query columns each; thread = key row = TMEM lane),
// 8-11 dQ drain (thread = channel = TMEM lane; D/32 of them active), 12 TMA producer
// (Q/dO/LSE/Di, 3 stages), 13 TMEM allocator and MMA issuer (warp-converged).
#include "fcp_cuda_util.h"
#include "fcp_sm100.cuh"

namespace fcp {
namespace {

using namespace dev;

constexpr int kBN = 128;  // key rows per CTA
constexpr int kBQ = 64;   // query rows per step
static_assert(kBQ == kBwdStepRows, "the plan's query bands count steps of this many rows");
constexpr int kStages = 3;
constexpr int kThreads = 448;

constexpr int kKVPanel = kBN * 128;        // 16384: [128 rows][64 ch]
constexpr int kQPanel = kBQ * 128;         // 8192: [64 rows][64 ch]
constexpr int kDSTile = kBN * kBQ * 2;     // 16384: [128 kv rows][64 q] bf16, one panel

// Shared-memory layout for head dimension D. The K region always holds two panels: the
// channels of K, then (D = 64) a zero panel, so that dQ^T = K^T dS^T is one M = 128
// instruction for either D.
template <int D>
struct TileCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kQTile = kBQ * D * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = 2 * kKVPanel;
  static constexpr int kOffQ = kOffV + kPanels * kKVPanel;   // kStages tiles
  static constexpr int kOffDO = kOffQ + kStages * kQTile;    // kStages tiles
  static constexpr int kOffDS = kOffDO + kStages * kQTile;   // 2 buffers
  static constexpr int kOffVec = kOffDS + 2 * kDSTile;       // kStages x (lse2[64], di[64])
  static constexpr int kOffStage = ((kOffVec + kStages * 2 * kBQ * 4) + 1023) & ~1023;  // dQ [64 q][D] float32
  static constexpr int kStageBytes = kBQ * D * 4;
  static constexpr int kOffBar = kOffStage + kStageBytes;
  static constexpr int kSmemBytes = kOffBar + 256;
  static constexpr int kDrainWarps = D / 32;  // drain warps holding real channels
  // dV, dK: M = 128 keys, N = D channels, A from TMEM, B (dO / Q) MN-major.
  static constexpr uint32_t kIdescAcc = idesc_bf16(kBN, D, false, true);
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  static_assert(kOffVec + kStages * 2 * kBQ * 4 <= kOffStage, "vector area");
};

// mbarrier indices, laid out from the stage count so that no two ever share a slot
enum : int {
  B_KVFULL = 0,
  B_QFULL = 1,                     // kStages
  B_QEMPTY = B_QFULL + kStages,    // kStages
  B_STFULL = B_QEMPTY + kStages,   // 2 buffers
  B_DSFULL = B_STFULL + 2,         // 2 buffers
  B_DSEMPTY = B_DSFULL + 2,        // 2 buffers
  B_DQFULL = B_DSEMPTY + 2,        // 2 buffers
  B_DQEMPTY = B_DQFULL + 2,        // 2 buffers
  B_ACCDONE = B_DQEMPTY + 2,
  B_STGFULL = B_ACCDONE + 1,       // the dQ staging tile is written
  B_STGFREE = B_STGFULL + 1,       // the previous reduce has read the staging tile
  B_DRAIN = B_STGFREE + 1,         // every MMA the CTA issued has completed
  B_COUNT = B_DRAIN + 1
};
static_assert(B_COUNT * 8 + 12 <= 256, "barrier area");

// S^T, dP^T: M = 128 keys, N = 64 queries, both operands K-major.
constexpr uint32_t kIdescST = idesc_bf16(kBN, kBQ, false, false);
// dQ^T = K^T dS^T: M = 128 channels, N = 64 queries, A (K read transposed) and B MN-major.
constexpr uint32_t kIdescDQ = idesc_bf16(128, kBQ, true, true);

// The backward's waits poll briefly and then suspend between polls (up to 1 us each): a step
// takes about 2500 cycles and most waits last hundreds of cycles, so spinning through them
// only spends issue slots and power, and under the power cap power is clock. Measured on the
// 32K causal step: 36.0 ms against 40.0 ms with plain polling (SM clock 1950 against 1820 MHz
// at the same board power); suspending from the first poll was slower (39.2 ms).
constexpr int kWaitSpin = 64;
constexpr uint32_t kWaitSuspendNs = 1000;
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err, int code) {
  return mbar_wait_backoff<kWaitSpin, kWaitSuspendNs>(bar, parity, abort_flag, err, code);
}

struct Args {
  const fcp_item* items;
  const KvSeg* kvsegs;
  const int* kv_items;
  const BwdUnit* units;
  const float* lse;
  const float* di;
  float* dq_acc;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  long long T;
  int hkv, group;
  float scale_log2, scale;
  int* err;
  // query bands: non-null band_units lists this launch's units (grid = units x KV heads); the
  // CTA walks only the query steps whose first row lies in [band_lo, band_hi) and adds its dK
  // and dV (unscaled, float32) into dk_acc / dv_acc instead of writing dk / dv
  const int* band_units;
  int band_lo, band_hi;
  float* dk_acc;
  float* dv_acc;
};

template <int D, bool kBanded>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tile_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const Args a) {
  using C = TileCfg<D>;
  constexpr int kD = D;
  constexpr int kOffK = C::kOffK, kOffV = C::kOffV, kOffQ = C::kOffQ, kOffDO = C::kOffDO, kOffDS = C::kOffDS;
  constexpr int kOffVec = C::kOffVec, kOffStage = C::kOffStage, kOffBar = C::kOffBar, kQTile = C::kQTile;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(a.err, 0, kErrSmemAlign);
    return;
  }
  const uint32_t sb = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + B_COUNT * 8 + 4);
  // set when an aborted CTA could not confirm that its issued copies or MMAs have finished
  volatile int* unquiesced = reinterpret_cast<volatile int*>(smem + kOffBar + B_COUNT * 8 + 8);
  float* vec = reinterpret_cast<float*>(smem + kOffVec);  // [stage][lse2[64] | di[64]]
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int slot = blockIdx.x / a.hkv;
  const int kvh = blockIdx.x - slot * a.hkv;
  // kBanded: one launch of a banded backward (a.band_units lists its units)
  const BwdUnit unit = a.units[kBanded ? a.band_units[slot] : slot];
  const KvSeg seg = a.kvsegs[unit.kvseg];
  const int kt = unit.kv_tile;
  const int kv_row0 = seg.tok0 + kt * kBN;
  const int kv_valid = seg.len - kt * kBN;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KVFULL), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_QFULL + s), 1);
      mbar_init(bar(B_QEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_STFULL + b), 1);
      mbar_init(bar(B_DSFULL + b), 8);
      mbar_init(bar(B_DSEMPTY + b), 1);
      mbar_init(bar(B_DQFULL + b), 1);
      mbar_init(bar(B_DQEMPTY + b), C::kDrainWarps);
    }
    mbar_init(bar(B_ACCDONE), 1);
    mbar_init(bar(B_STGFULL), C::kDrainWarps);
    mbar_init(bar(B_STGFREE), 1);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = (*reinterpret_cast<volatile int*>(a.err) != 0) ? 1 : 0;
    *unquiesced = 0;
    mbar_fence_init();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if constexpr (D < 128) {  // the zero panel beside K's channels (read as K^T rows D..127)
    uint4* zero = reinterpret_cast<uint4*>(smem + kOffK + C::kPanels * kKVPanel);
    for (int i = threadIdx.x; i < (2 - C::kPanels) * kKVPanel / 16; i += kThreads) zero[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  // Steps: for each query head of the group, each item whose key range is this one, each
  // 64-row query step that sees this key tile (a causal diagonal item starts at the step
  // holding the tile's first key). body(step, h, item, qs) returns false to stop.
  // (In a band every CTA still walks the group's heads in order: the CTAs of one KV head then
  // read the same Q/dO rows at about the same time, which measured 5-9% faster than starting
  // consecutive key tiles on different heads.)
  auto ceil_steps = [](int rows) { return rows > 0 ? (rows + kBQ - 1) / kBQ : -((-rows) / kBQ); };
  auto for_each_step = [&](auto&& body) -> int {
    int step = 0;
    for (int hh = 0; hh < a.group; ++hh) {
      const int h = kvh * a.group + hh;
      for (int li = seg.list_begin; li < seg.list_end; ++li) {
        const fcp_item itm = a.items[a.kv_items[li]];
        int q_end = (itm.q_len + kBQ - 1) / kBQ;
        int q_first = itm.mask == FCP_MASK_CAUSAL_DIAG ? (kt * kBN) / kBQ : 0;
        if constexpr (kBanded) {
          q_first = max(q_first, ceil_steps(a.band_lo - itm.q_tok0));
          q_end = min(q_end, ceil_steps(a.band_hi - itm.q_tok0));
        }
        for (int qs = q_first; qs < q_end; ++qs, ++step)
          if (!body(step, h, itm, qs)) return step;
      }
    }
    return step;
  };

  int n_steps = 0;
  if (warp == 12) {
    // ---------------------------------------------------------------- producer
    bool ok = !skip;
    int last_issued = -1;  // last step whose Q/dO loads went out
    if (ok && lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(bar(B_KVFULL), 2 * C::kPanels * kKVPanel);
#pragma unroll
      for (int p = 0; p < C::kPanels; ++p) {
        tma_load_3d(sb + kOffK + p * kKVPanel, &tmK, bar(B_KVFULL), p * 64, kv_row0, kvh);
        tma_load_3d(sb + kOffV + p * kKVPanel, &tmV, bar(B_KVFULL), p * 64, kv_row0, kvh);
      }
    }
    if (ok) {
      n_steps = for_each_step([&](const int step, const int h, const fcp_item& itm, const int qs) -> bool {
        const int s = step % kStages;
        const uint32_t ph = (step / kStages) & 1;
        ok = bwait(bar(B_QEMPTY + s), ph ^ 1, abort_flag, a.err, kErrBwdWait + 1);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        const int qrow0 = itm.q_tok0 + qs * kBQ;
        const int q_valid = itm.q_len - qs * kBQ;
        if (lane == 0) {
          mbar_expect_tx(bar(B_QFULL + s), 2 * kQTile);
#pragma unroll
          for (int p = 0; p < C::kPanels; ++p) {
            tma_load_3d(sb + kOffQ + s * kQTile + p * kQPanel, &tmQ, bar(B_QFULL + s), p * 64, qrow0, h);
            tma_load_3d(sb + kOffDO + s * kQTile + p * kQPanel, &tmDO, bar(B_QFULL + s), p * 64, qrow0, h);
          }
        }
        last_issued = step;
        // LSE in log2 units and Di of the step's query rows; rows past the range get
        // LSE = +inf (P = 0) and Di = 0
        float* v = vec + s * 2 * kBQ;
        const long long rowbase = static_cast<long long>(h) * a.T + qrow0;
#pragma unroll
        for (int i = 0; i < kBQ / 32; ++i) {
          const int c = i * 32 + lane;
          const bool in = c < q_valid;
          v[c] = in ? a.lse[rowbase + c] * 1.4426950408889634f : INFINITY;
          v[kBQ + c] = in ? a.di[rowbase + c] : 0.f;
        }
        mbar_arrive_warp(bar(B_QFULL + s));
        return true;
      });
    }
    if (!skip && *abort_flag && lane == 0) {
      // the loads already issued land in this CTA's shared memory: wait for them (bounded)
      // (a step's stage is reused only after that step's loads were consumed, so only the last
      // kStages steps can still be in flight)
      bool done = mbar_wait_quiesce(bar(B_KVFULL), 0, kWaitLimitNs);
      for (int j = last_issued - (kStages - 1) > 0 ? last_issued - (kStages - 1) : 0; j <= last_issued; ++j)
        done = mbar_wait_quiesce(bar(B_QFULL + j % kStages), (j / kStages) & 1, kWaitLimitNs) && done;
      if (!done) *unquiesced = 1;
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------------- MMA issuer
    // the whole warp runs this with uniform operands; one elected lane issues each MMA/commit
    bool ok = !skip;
    {
      auto wwait = [&](uint32_t bb, uint32_t parity, int code) -> bool {
        return __all_sync(0xffffffffu, bwait(bb, parity, abort_flag, a.err, code));
      };
      if (ok) ok = wwait(bar(B_KVFULL), 0, kErrBwdWait + 2);
      tc_fence_after();
      const uint32_t t_dv = tmem + 256, t_dk = tmem + 384;
      // number of steps, walked once without waiting
      const int total = ok ? for_each_step([](int, int, const fcp_item&, int) { return true; }) : 0;
      auto issue_sdp = [&](int j) -> bool {
        const int s = j % kStages, b = j & 1;
        if (!wwait(bar(B_QFULL + s), (j / kStages) & 1, kErrBwdWait + 3)) return false;
        tc_fence_after();
        const uint32_t qb = sb + kOffQ + s * kQTile, db = sb + kOffDO + s * kQTile;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * kKVPanel + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * kQPanel + (kk & 3) * 32;
          mma_ss_w(tmem + 128 * b, sdesc_sw128(sb + kOffK + ko, 16, 1024), sdesc_sw128(qb + qo, 16, 1024), kIdescST,
                 kk > 0);
        }
        // the dP^T half of buffer b is free once the dQ^T of step j-2 has been read out of it
        if (!wwait(bar(B_DQEMPTY + b), ((j >> 1) & 1) ^ 1, kErrBwdWait + 4)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * kKVPanel + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * kQPanel + (kk & 3) * 32;
          mma_ss_w(tmem + 128 * b + 64, sdesc_sw128(sb + kOffV + ko, 16, 1024), sdesc_sw128(db + qo, 16, 1024),
                 kIdescST, kk > 0);
        }
        tc_commit_w(bar(B_STFULL + b));
        return true;
      };
      if (ok && total > 0) ok = issue_sdp(0);
      for (int i = 0; i < total && ok; ++i) {
        if (i + 1 < total) {
          ok = issue_sdp(i + 1);
          if (!ok) break;
        }
        const int s = i % kStages, b = i & 1;
        ok = wwait(bar(B_DSFULL + b), (i >> 1) & 1, kErrBwdWait + 5);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qb = sb + kOffQ + s * kQTile, db = sb + kOffDO + s * kQTile;
        // dV += P^T dO and dK += dS^T Q: K = 64 queries in 4 steps of 16 (8 TMEM columns)
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_ts_w(t_dv, tmem + 128 * b + 16 + kk * 8, sdesc_sw128(db + kk * 2048, kQPanel, 1024), C::kIdescAcc,
                 (i > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk)
          mma_ts_w(t_dk, tmem + 128 * b + 80 + kk * 8, sdesc_sw128(qb + kk * 2048, kQPanel, 1024), C::kIdescAcc,
                 (i > 0 || kk > 0));
        // dQ^T = K^T dS^T: K = 128 keys in 8 steps of 16 rows (2048 bytes)
        const uint32_t dsb = sb + kOffDS + b * kDSTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ss_w(tmem + 128 * b + 64, sdesc_sw128(sb + kOffK + kk * 2048, kKVPanel, 1024),
                 sdesc_sw128(dsb + kk * 2048, kKVPanel, 1024), kIdescDQ, kk > 0);
        tc_commit_w(bar(B_DQFULL + b));
        tc_commit_w(bar(B_DSEMPTY + b));
        tc_commit_w(bar(B_QEMPTY + s));
      }
      n_steps = total;
      if (ok) tc_commit_w(bar(B_ACCDONE));
      // every issued MMA has completed once the drain barrier fires; wait for it also after
      // an abort (the wait ignores the abort flag) so that none still reads shared memory or
      // writes tensor memory when they are released
      tc_commit_w(bar(B_DRAIN));
      if (!__all_sync(0xffffffffu, mbar_wait_quiesce(bar(B_DRAIN), 0, kWaitLimitNs)) && lane == 0) {
        *abort_flag = 1;
        *unquiesced = 1;
        atomicCAS(a.err, 0, kErrBwdWait + 14);
      }
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- gradient warps
    bool ok = !skip;
    const int wg = warp >> 2;              // query columns [32 wg, 32 wg + 32) of a step
    const int r = (warp & 3) * 32 + lane;  // key row = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint8_t* ds_row = smem + kOffDS + r * 128;
    if (ok) {
      n_steps = for_each_step([&](const int step, const int h, const fcp_item& itm, const int qs) -> bool {
        const int s = step % kStages, b = step & 1;
        // visible query columns of this key row: c >= r + (key-tile start - step start) on a
        // causal diagonal item; none past the key range
        int qmin = 0;
        if (r >= kv_valid) {
          qmin = kBQ;
        } else if (itm.mask == FCP_MASK_CAUSAL_DIAG) {
          qmin = max(0, r + kt * kBN - qs * kBQ);
        }
        ok = bwait(bar(B_QFULL + s), (step / kStages) & 1, abort_flag, a.err, kErrBwdWait + 7);
        if (ok) ok = bwait(bar(B_STFULL + b), (step >> 1) & 1, abort_flag, a.err, kErrBwdWait + 8);
        // the dS^T tile of buffer b is free once the dQ^T MMA of step-2 has read it
        if (ok) ok = bwait(bar(B_DSEMPTY + b), ((step >> 1) & 1) ^ 1, abort_flag, a.err, kErrBwdWait + 9);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        tc_fence_after();
        const float* lse2 = vec + s * 2 * kBQ + 32 * wg;  // this warpgroup's 32 columns
        const float* dis = vec + s * 2 * kBQ + kBQ + 32 * wg;
        uint32_t sv[32], dv[32];
        tmem_ld32x2(lane_base + 128 * b + 32 * wg, lane_base + 128 * b + 64 + 32 * wg, sv, dv);
        uint32_t pp[16], dd[16];
        if (__all_sync(0xffffffffu, qmin <= 32 * wg)) {
          // every column visible: packed float32x2 arithmetic, LSE/Di as 16-byte loads
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 l4 = reinterpret_cast<const float4*>(lse2)[k];
            const float4 d4 = reinterpret_cast<const float4*>(dis)[k];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * k + h;
              const float l0 = h ? l4.z : l4.x, l1 = h ? l4.w : l4.y;
              const float i0 = h ? d4.z : d4.x, i1 = h ? d4.w : d4.y;
              const float2 x = ffma2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]), a.scale_log2,
                                     a.scale_log2, -l0, -l1);
              const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
              const float2 g = fsub2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1]), i0, i1);
              const float2 ds = fmul2(p0, p1, g.x, g.y);
              pp[e] = pack_bf16(p0, p1);
              dd[e] = pack_bf16(ds.x, ds.y);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = 32 * wg + 2 * e;
            float p0 = 0.f, p1 = 0.f, d0 = 0.f, d1 = 0.f;
            if (c0 >= qmin) {
              p0 = fast_exp2(fmaf(__uint_as_float(sv[2 * e]), a.scale_log2, -lse2[2 * e]));
              d0 = p0 * (__uint_as_float(dv[2 * e]) - dis[2 * e]);
            }
            if (c0 + 1 >= qmin) {
              p1 = fast_exp2(fmaf(__uint_as_float(sv[2 * e + 1]), a.scale_log2, -lse2[2 * e + 1]));
              d1 = p1 * (__uint_as_float(dv[2 * e + 1]) - dis[2 * e + 1]);
            }
            pp[e] = pack_bf16(p0, p1);
            dd[e] = pack_bf16(d0, d1);
          }
        }
        tmem_st16(lane_base + 128 * b + 16 + 16 * wg, pp);
        tmem_st16(lane_base + 128 * b + 80 + 16 * wg, dd);
        // dS^T row r, queries [32 wg, 32 wg + 32): 16-byte chunks 4 wg .. 4 wg + 3 of the
        // 128-byte row, 128-byte swizzle (chunk XOR row & 7)
        uint8_t* drow = ds_row + b * kDSTile;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int chunk = (4 * wg + x) ^ (r & 7);
          *reinterpret_cast<uint4*>(drow + chunk * 16) = make_uint4(dd[4 * x], dd[4 * x + 1], dd[4 * x + 2], dd[4 * x + 3]);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_warp(bar(B_DSFULL + b));
        return true;
      });
    }
    // epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK (bf16); in a band both
    // add their unscaled float32 sums into the band accumulators
    if (ok) ok = bwait(bar(B_ACCDONE), 0, abort_flag, a.err, kErrBwdWait + 10);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const bool store = r < kv_valid;
      const long long row = static_cast<long long>(kvh) * a.T + kv_row0 + r;
      __nv_bfloat16* dst = (wg == 0 ? a.dv : a.dk) + row * kD;
      const float f = wg == 0 ? 1.f : a.scale;
      const uint32_t base = lane_base + (wg == 0 ? 256 : 384);
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t x[32];
        if (n_steps > 0) {
          tmem_ld32(base + c * 32, x);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = 0u;
        }
        if (kBanded && store) {
          // float32 sums over the bands: this CTA owns these rows within the launch
          float4* acc = reinterpret_cast<float4*>((wg == 0 ? a.dv_acc : a.dk_acc) + row * kD + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float4 y = acc[e];
            y.x += __uint_as_float(x[4 * e + 0]);
            y.y += __uint_as_float(x[4 * e + 1]);
            y.z += __uint_as_float(x[4 * e + 2]);
            y.w += __uint_as_float(x[4 * e + 3]);
            acc[e] = y;
          }
        } else if (store) {
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
  } else if (warp - 8 < C::kDrainWarps) {
    // ---------------------------------------------------------------- dQ drain (warps 8..)
    // dQ^T (lane = channel) goes into a [64 q][D] float32 staging tile; one lane adds the
    // tile to the accumulator with a TMA reduce. Query rows past the item's range carry exact
    // zeros (their P and dS are 0), and rows past T are clipped by the tensor map.
    bool ok = !skip;
    const int d = (warp & 3) * 32 + lane;  // channel = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool issuer = threadIdx.x == 8 * 32;
    float* stage = reinterpret_cast<float*>(smem + kOffStage);
    if (ok) {
      if (issuer) tma_prefetch_desc(&tmDQ);
      n_steps = for_each_step([&](const int step, const int h, const fcp_item& itm, const int qs) -> bool {
        const int b = step & 1;
        ok = bwait(bar(B_DQFULL + b), (step >> 1) & 1, abort_flag, a.err, kErrBwdWait + 11);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        tc_fence_after();
        uint32_t x0[32], x1[32];
        tmem_ld32x2(lane_base + 128 * b + 64, lane_base + 128 * b + 96, x0, x1);
        tc_fence_before();
        mbar_arrive_warp(bar(B_DQEMPTY + b));  // TMEM buffer free
        // the previous step's reduce went out without a wait, so that the issuing warp could
        // read this dQ^T out of TMEM meanwhile; the staging tile is free once that reduce has
        // read it (the wait is a no-op on the lanes that issued nothing; warp-uniform branch)
        if (warp == 8 && step > 0) {
          bulk_wait_read_all();
          mbar_arrive_warp(bar(B_STGFREE));
        }
        ok = bwait(bar(B_STGFREE), (step & 1) ^ 1, abort_flag, a.err, kErrBwdWait + 12);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
#pragma unroll
        for (int q = 0; q < 32; ++q) stage[q * kD + d] = __uint_as_float(x0[q]);
#pragma unroll
        for (int q = 0; q < 32; ++q) stage[(32 + q) * kD + d] = __uint_as_float(x1[q]);
        fence_proxy_async_smem();
        mbar_arrive_warp(bar(B_STGFULL));
        if (warp == 8) {  // every drain warp has written its channels: one lane adds the tile
          ok = __all_sync(0xffffffffu, bwait(bar(B_STGFULL), step & 1, abort_flag, a.err, kErrBwdWait + 13));
          if (ok && issuer) {
            tma_reduce_add_3d(&tmDQ, sb + kOffStage, 0, itm.q_tok0 + qs * kBQ, h);
            bulk_commit_group();
          }
          __syncwarp();
        }
        return ok;
      });
      if (issuer) bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*unquiesced) {
    // fallback only: an issued copy or MMA did not report completion within the wait limit
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) __nanosleep(1000);
  }
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Launch of the backward tile kernel (same contract as fcp_block_attn_bwd_tiles). With dk_acc
// and dv_acc (zeroed float32 [Hkv, T, D]) the plan's query bands run as one launch each.
template <int D>
fcp_status launch_bwd_tile(const fcp_plan* plan, const void* d_plan, const void* q, const void* k, const void* v,
                           const void* dout, const float* lse, const float* di, float* dq_acc, void* dk, void* dv,
                           int hq, int hkv, float* dk_acc, float* dv_acc, cudaStream_t stream) {
  using C = TileCfg<D>;
  const DevLayout& L = plan->layout;
  if (L.n_bwd_units == 0) return FCP_OK;
  const int64_t T = plan->total_tokens;
  CUtensorMap mq, mk, mv, mdo, mdq;
  fcp_status st;
  if ((st = make_f32_map(&mdq, dq_acc, hq, T, D, kBQ)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mq, q, hq, T, D, kBQ)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mk, k, hkv, T, D, kBN)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mv, v, hkv, T, D, kBN)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mdo, dout, hq, T, D, kBQ)) != FCP_OK) return st;
  Args a;
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
  a.hkv = hkv;
  a.group = hq / hkv;
  a.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  a.err = dev_error_word(d_plan);
  a.band_units = nullptr;
  a.band_lo = a.band_hi = 0;
  a.dk_acc = dk_acc;
  a.dv_acc = dv_acc;
  FCP_CUDA_TRY(cudaFuncSetAttribute(bwd_tile_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmemBytes),
               "bwd smem attribute");
  FCP_CUDA_TRY(cudaFuncSetAttribute(bwd_tile_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmemBytes),
               "bwd smem attribute");
  if (dk_acc == nullptr) {
    const long long grid = static_cast<long long>(L.n_bwd_units) * hkv;
    if (grid > 0x7fffffffLL) return FCP_ERR_UNSUPPORTED;
    bwd_tile_kernel<D, false><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mdo,
                                                                                                 mdq, a);
    FCP_CUDA_TRY(cudaGetLastError(), "bwd launch");
    return FCP_OK;
  }
  if (L.n_bands == 0 || dv_acc == nullptr) return FCP_ERR_STATE;
  const int* band_units = dev_array<int>(d_plan, L.band_units);
  for (int32_t b = 0; b < L.n_bands; ++b) {
    const int32_t n = L.band_begin[b + 1] - L.band_begin[b];
    if (n == 0) continue;
    a.band_units = band_units + L.band_begin[b];
    a.band_lo = b * L.band_rows;
    a.band_hi = static_cast<int>(std::min<int64_t>(T, int64_t(b + 1) * L.band_rows));
    const long long grid = static_cast<long long>(n) * hkv;
    if (grid > 0x7fffffffLL) return FCP_ERR_UNSUPPORTED;
    bwd_tile_kernel<D, true><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mdo, mdq,
                                                                                                a);
    FCP_CUDA_TRY(cudaGetLastError(), "bwd band launch");
  }
  return FCP_OK;
}

}  // namespace

fcp_status launch_bwd_tiles(const fcp_plan* plan, const void* d_plan, const void* q, const void* k, const void* v,
                            const void* dout, const float* lse, const float* di, float* dq_acc, void* dk, void* dv,
                            int hq, int hkv, int head_dim, float* dk_acc, float* dv_acc, cudaStream_t stream) {
  if (head_dim == 128)
    return launch_bwd_tile<128>(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, dk_acc, dv_acc,
                                stream);
  return launch_bwd_tile<64>(plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, hq, hkv, dk_acc, dv_acc, stream);
}

}  // namespace fcp
