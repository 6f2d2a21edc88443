// Forward block attention over the FCP work list on sm_103a (tcgen05 + TMEM + TMA).
//
// Computes, for every run (a query range with up to c work items, "Unleashing Scalable
// Context Parallelism for Foundation Models Pre-Training via FCP", Section 4.2 coalescer) and
// every query head, the attention of Section 2.2 over the run's key ranges, written as a
// partial (O normalised over those keys, natural LSE) -- the per-slice partial results of
// Section 2.3 that the merge reduces.
//
// Work tile = one 128-row query tile of one run, for two query heads of the same KV group
// (two "heads" t = 0, 1 that share every K/V tile loaded into shared memory). The kernel is
// persistent: one CTA per SM takes tiles (sorted longest first) from a global counter, and
// the next tile's Q load, the K/V ring and the previous tile's partial stores overlap the
// current tile's MMAs. 10 warps:
//   warps 0-3  softmax of head 0: thread = query row = TMEM lane
//   warps 4-7  softmax of head 1
//   warp  8    tile scheduler and TMA producer: per tile the two Q tiles, then K and V tiles
//              through 2-stage rings counted across tiles
//   warp  9    TMEM allocator and MMA issuer (warp-converged, one elected lane issues)
// TMEM (512 columns x 128 lanes, fp32): S_t at columns [128t, 128t+128), O_t at
// [256+128t, 256+128t+D). Softmax overwrites S_t's first 64 columns with P_t as packed bf16,
// in two halves of 64 keys, each handed to the MMA warp as soon as it is stored; O_t += P_t V
// runs with A read from TMEM. Per key tile the issue order is PV(0,j-1), S(0,j), PV(1,j-1),
// S(1,j), so the tensor core works on one head while the other head's softmax runs. O is
// rescaled lazily: only when a row maximum grows by more than 2^8 (in exp2 units), keeping
// every P <= 256; the final normalisation uses the same stale maximum, so the result is
// exact up to rounding.
#include "fcp_cuda_util.h"
#include "fcp_sm100.cuh"

namespace fcp {
namespace {

using namespace dev;

constexpr int kFwdThreads = 320;
constexpr int kPanelBytes = kTileM * 128;  // one box: 128 rows x 64 bf16 channels
constexpr float kRescaleThreshold = 8.0f;   // log2 units

struct FwdArgs {
  const fcp_item* items;
  const fcp_run* runs;
  const FwdUnit* units;
  long long n_tiles;                 // units x KV heads x head pairs
  unsigned long long* next_tile;     // tile counter, zero at launch
  float* part_o;
  float* part_lse;
  long long part_rows;
  int hq, hkv, group, pairs_per_group;
  float scale_log2;
  int* err;
};

enum : int {
  B_QFULL = 0,
  B_QEMPTY = 1,  // the S MMAs of a tile have read Q
  B_KFULL = 2,   // 2 stages
  B_KEMPTY = 4,  // 2 stages
  B_VFULL = 6,
  B_VEMPTY = 8,
  B_SFULL = 10,  // per tile
  B_PFULL = 12,  // per tile and half: keys [0, 64) and [64, 128) of P are in TMEM
  B_ODONE = 16,  // per tile
  B_OFREE = 18,  // per tile: the epilogue has read O_t out of TMEM
  B_DRAIN = 20,
  B_TFULL = 21,   // 2 slots: the producer has published the next tile index
  B_TEMPTY = 23,  // 2 slots: the MMA warp and the 8 softmax warps have read it
  B_COUNT = 25
};

// barrier area: mbarriers, abort flag, TMEM base, then the 2-slot tile ring (48 bytes a slot)
constexpr int kTileSlotOff = 256;
constexpr int kBarArea = kTileSlotOff + 2 * 48;
static_assert(B_COUNT * 8 + 12 <= kTileSlotOff, "barrier area");

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = kTileM * D * 2;
  static constexpr int kPanels = D / 64;
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kTileBytes;
  static constexpr int kK = 2 * kTileBytes;
  static constexpr int kV = 4 * kTileBytes;
  static constexpr int kBar = 6 * kTileBytes;
  // epilogue staging: one [32 rows][32 float32] block per softmax warp
  static constexpr int kStage = kBar + kBarArea;
  static constexpr int kStageBytes = 8 * 32 * 32 * 4;
  static constexpr int kEnd = kStage + kStageBytes;
  // at least half the SM's shared memory, so one CTA per SM holds all 512 TMEM columns
  static constexpr int kSmemBytes = kEnd > 118 * 1024 ? kEnd : 118 * 1024;
  static_assert(kStage % 16 == 0, "16-byte aligned staging");
  static_assert(kSmemBytes <= 232448, "shared memory per block");
  static constexpr uint32_t kIdescS = idesc_bf16(kTileM, kTileN, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16(kTileM, D, false, true);
};

__device__ __forceinline__ int kv_tiles(const fcp_item& it, int q_tile) {
  int n = (it.kv_len + kTileN - 1) / kTileN;
  if (it.mask == FCP_MASK_CAUSAL_DIAG) n = min(n, q_tile + 1);
  return n;
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<D>;
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
  // set when an aborted CTA could not confirm that its issued copies or MMAs have finished
  volatile int* unquiesced = reinterpret_cast<volatile int*>(smem + C::kBar + B_COUNT * 8 + 8);
  auto bar = [&](int i) -> uint32_t { return sb + C::kBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int per_unit = a.hkv * a.pairs_per_group;

  // Tiles (unit, KV head, head pair), sorted longest first, are handed out dynamically: the
  // producer takes the next index from a global counter, decodes it and publishes it in a
  // 2-slot ring that the MMA warp and the softmax warps read (valid = 0: no tile left).
  struct Tile {
    int item_begin, item_end, q_tok0, q_len, part_row0, qt, kvh, h0, h1, has_h1, valid, pad;
  };
  Tile* tile_slot = reinterpret_cast<Tile*>(smem + C::kBar + kTileSlotOff);
  auto decode = [&](long long w) -> Tile {
    Tile t;
    const int unit_idx = static_cast<int>(w / per_unit);
    const int rem = static_cast<int>(w - static_cast<long long>(unit_idx) * per_unit);
    t.kvh = rem / a.pairs_per_group;
    const int pair = rem - t.kvh * a.pairs_per_group;
    t.h0 = t.kvh * a.group + 2 * pair;
    t.has_h1 = 2 * pair + 1 < a.group;
    t.h1 = t.has_h1 ? t.h0 + 1 : t.h0;
    const FwdUnit unit = a.units[unit_idx];
    const fcp_run run = a.runs[unit.run];
    t.item_begin = run.item_begin;
    t.item_end = run.item_end;
    t.q_tok0 = run.q_tok0;
    t.q_len = run.q_len;
    t.part_row0 = run.part_row0;
    t.qt = unit.q_tile;
    t.valid = 1;
    t.pad = 0;
    return t;
  };
  // consumer side: the tile of round u (valid = -1 when a wait gave up)
  auto next_tile = [&](int u, int code) -> Tile {
    Tile t;
    t.valid = -1;
    if (__all_sync(0xffffffffu, mbar_wait(bar(B_TFULL + (u & 1)), (u >> 1) & 1, abort_flag, a.err, code))) {
      const volatile Tile* src = tile_slot + (u & 1);
      t.item_begin = src->item_begin;
      t.item_end = src->item_end;
      t.q_tok0 = src->q_tok0;
      t.q_len = src->q_len;
      t.part_row0 = src->part_row0;
      t.qt = src->qt;
      t.kvh = src->kvh;
      t.h0 = src->h0;
      t.h1 = src->h1;
      t.has_h1 = src->has_h1;
      t.valid = src->valid;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_TEMPTY + (u & 1)));
    }
    return t;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + 2 * s), 4);  // one arrival per softmax warp of the head
      mbar_init(bar(B_PFULL + 2 * s + 1), 4);
      mbar_init(bar(B_ODONE + s), 1);
      mbar_init(bar(B_OFREE + s), 4);
    }
    mbar_init(bar(B_DRAIN), 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_TFULL + k), 1);
      mbar_init(bar(B_TEMPTY + k), 9);
    }
    *abort_flag = (*reinterpret_cast<volatile int*>(a.err) != 0) ? 1 : 0;
    *unquiesced = 0;
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

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // Q of tile u+1 is loaded as soon as the S MMAs of tile u have read Q; K and V stream
    // through 2-stage rings whose slots are counted across tiles (J).
    if (lane == 0 && !skip) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int J = 0;
      bool ok = true;
      int last_q = -1, last_kj = -1, last_vj = -1;  // tile of the last Q load, key tile of the last K, V loads
      for (int u = 0; ok; ++u) {
        const int k = u & 1;
        if (!mbar_wait(bar(B_TEMPTY + k), ((u >> 1) & 1) ^ 1, abort_flag, a.err, kErrFwdWait + 13)) break;
        unsigned long long got = atomicAdd(a.next_tile, 1ull);
        Tile T;
        T.valid = 0;
        if (got < static_cast<unsigned long long>(a.n_tiles)) T = decode(static_cast<long long>(got));
        {
          volatile Tile* dst = tile_slot + k;
          dst->item_begin = T.item_begin;
          dst->item_end = T.item_end;
          dst->q_tok0 = T.q_tok0;
          dst->q_len = T.q_len;
          dst->part_row0 = T.part_row0;
          dst->qt = T.qt;
          dst->kvh = T.kvh;
          dst->h0 = T.h0;
          dst->h1 = T.h1;
          dst->has_h1 = T.has_h1;
          dst->valid = T.valid;
        }
        mbar_arrive(bar(B_TFULL + k));
        if (!T.valid) break;
        if (!mbar_wait(bar(B_QEMPTY), (u & 1) ^ 1, abort_flag, a.err, kErrFwdWait + 11)) break;
        const int qrow = T.q_tok0 + T.qt * kTileM;
        mbar_arrive_expect_tx(bar(B_QFULL), 2 * C::kTileBytes);
#pragma unroll
        for (int p = 0; p < C::kPanels; ++p) {
          tma_load_3d(sb + C::kQ0 + p * kPanelBytes, &tmQ, bar(B_QFULL), p * 64, qrow, T.h0);
          tma_load_3d(sb + C::kQ1 + p * kPanelBytes, &tmQ, bar(B_QFULL), p * 64, qrow, T.h1);
        }
        last_q = u;
        for (int ii = T.item_begin; ii < T.item_end && ok; ++ii) {
          const fcp_item itm = a.items[ii];
          const int nkt = kv_tiles(itm, T.qt);
          for (int kt = 0; kt < nkt; ++kt, ++J) {
            const int s = J & 1;
            const uint32_t ph = (J >> 1) & 1;
            const int kvrow = itm.kv_tok0 + kt * kTileN;
            if (!mbar_wait(bar(B_KEMPTY + s), ph ^ 1, abort_flag, a.err, kErrFwdWait + 1)) { ok = false; break; }
            mbar_arrive_expect_tx(bar(B_KFULL + s), C::kTileBytes);
#pragma unroll
            for (int p = 0; p < C::kPanels; ++p)
              tma_load_3d(sb + C::kK + s * C::kTileBytes + p * kPanelBytes, &tmK, bar(B_KFULL + s), p * 64, kvrow,
                          T.kvh);
            last_kj = J;
            if (!mbar_wait(bar(B_VEMPTY + s), ph ^ 1, abort_flag, a.err, kErrFwdWait + 2)) { ok = false; break; }
            mbar_arrive_expect_tx(bar(B_VFULL + s), C::kTileBytes);
#pragma unroll
            for (int p = 0; p < C::kPanels; ++p)
              tma_load_3d(sb + C::kV + s * C::kTileBytes + p * kPanelBytes, &tmV, bar(B_VFULL + s), p * 64, kvrow,
                          T.kvh);
            last_vj = J;
          }
        }
      }
      if (*abort_flag) {
        // the loads already issued land in this CTA's shared memory: wait for them (bounded)
        // (a K/V stage is reused only after its previous tile was consumed, so only the last
        // two key tiles can still be in flight)
        bool done = last_q < 0 || mbar_wait_quiesce(bar(B_QFULL), last_q & 1, kWaitLimitNs);
        for (int j = last_kj > 0 ? last_kj - 1 : 0; j <= last_kj; ++j)
          done = mbar_wait_quiesce(bar(B_KFULL + (j & 1)), (j >> 1) & 1, kWaitLimitNs) && done;
        for (int j = last_vj > 0 ? last_vj - 1 : 0; j <= last_vj; ++j)
          done = mbar_wait_quiesce(bar(B_VFULL + (j & 1)), (j >> 1) & 1, kWaitLimitNs) && done;
        if (!done) *unquiesced = 1;
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs this with uniform operands; one elected lane issues each MMA/commit
    if (!skip) {
      auto wwait = [&](uint32_t bb, uint32_t parity, int code) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bb, parity, abort_flag, a.err, code));
      };
      auto issue_s = [&](int t, int s) {
        const uint32_t d = tmem + t * 128;
        const uint32_t qbase = sb + (t ? C::kQ1 : C::kQ0);
        const uint32_t kbase = sb + C::kK + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanelBytes + (kk & 3) * 32;
          mma_ss_w(d, sdesc_sw128(qbase + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), C::kIdescS, kk > 0);
        }
      };
      // O_t += P_t V for global key tile J-1, in two halves of 64 keys: each is issued as
      // soon as the softmax has stored that half of P
      auto issue_pv = [&](int t, int s, bool acc, int J) -> bool {
        const uint32_t d = tmem + 256 + t * 128;
        const uint32_t p = tmem + t * 128;
        const uint32_t vbase = sb + C::kV + s * C::kTileBytes;
        for (int half = 0; half < 2; ++half) {
          if (!wwait(bar(B_PFULL + 2 * t + half), (J - 1) & 1, kErrFwdWait + 6)) return false;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * half + k4;
            mma_ts_w(d, p + kk * 8, sdesc_sw128(vbase + kk * 2048, kPanelBytes, 1024), C::kIdescPV,
                     (acc || kk > 0));
          }
        }
        return true;
      };
      // PV of global key tile J-1 (local index jl-1) for both heads; the first PV of a tile
      // overwrites O_t, which the previous tile's epilogue must have read out first
      auto finish_pv = [&](int J, int jl, int u, bool last) -> bool {
        const int ps = (J - 1) & 1;
        if (!wwait(bar(B_VFULL + ps), ((J - 1) >> 1) & 1, kErrFwdWait + 5)) return false;
        for (int t = 0; t < 2; ++t) {
          if (jl == 1 && u > 0 && !wwait(bar(B_OFREE + t), (u - 1) & 1, kErrFwdWait + 12)) return false;
          if (!issue_pv(t, ps, jl - 1 > 0, J)) return false;
          tc_commit_w(bar(B_ODONE + t));
          if (t == 1 && last) tc_commit_w(bar(B_VEMPTY + ps));
        }
        return true;
      };
      bool ok = true;
      int J = 0;
      for (int u = 0; ok; ++u) {
        const Tile T = next_tile(u, kErrFwdWait + 14);
        if (T.valid <= 0) break;
        ok = wwait(bar(B_QFULL), u & 1, kErrFwdWait + 3);
        if (!ok) break;
        tc_fence_after();
        int jl = 0;
        for (int ii = T.item_begin; ii < T.item_end && ok; ++ii) {
          const fcp_item itm = a.items[ii];
          const int nkt = kv_tiles(itm, T.qt);
          for (int kt = 0; kt < nkt && ok; ++kt, ++J, ++jl) {
            const int s = J & 1;
            const uint32_t ph = (J >> 1) & 1;
            if (!wwait(bar(B_KFULL + s), ph, kErrFwdWait + 4)) { ok = false; break; }
            tc_fence_after();
            for (int t = 0; t < 2; ++t) {
              if (jl > 0) {
                const int ps = (J - 1) & 1;
                if (t == 0 && !wwait(bar(B_VFULL + ps), ((J - 1) >> 1) & 1, kErrFwdWait + 5)) { ok = false; break; }
                if (jl == 1 && u > 0 && !wwait(bar(B_OFREE + t), (u - 1) & 1, kErrFwdWait + 12)) {
                  ok = false;
                  break;
                }
                if (!issue_pv(t, ps, jl - 1 > 0, J)) { ok = false; break; }
                tc_commit_w(bar(B_ODONE + t));
                if (t == 1) tc_commit_w(bar(B_VEMPTY + ps));
              }
              issue_s(t, s);
              tc_commit_w(bar(B_SFULL + t));
            }
            if (ok) tc_commit_w(bar(B_KEMPTY + s));
          }
        }
        if (!ok) break;
        // every S of this tile has been issued: Q is free once they complete
        tc_commit_w(bar(B_QEMPTY));
        if (jl > 0) ok = finish_pv(J, jl, u, true);
      }
      // every issued MMA has completed once the drain barrier fires; wait for it also after
      // an abort (the wait ignores the abort flag), so that no MMA still reads shared memory
      // or writes tensor memory when they are released
      tc_commit_w(bar(B_DRAIN));
      if (!__all_sync(0xffffffffu, mbar_wait_quiesce(bar(B_DRAIN), 0, kWaitLimitNs)) && lane == 0) {
        *abort_flag = 1;
        *unquiesced = 1;
        atomicCAS(a.err, 0, kErrFwdWait + 7);
      }
    }
  } else if (!skip) {
    // ------------------------------------------------------------ softmax (warps 0-7)
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_addr = lane_base + t * 128;
    const uint32_t o_addr = lane_base + 256 + t * 128;
    bool ok = true;
    int J = 0;
    for (int u = 0; ok; ++u) {
      const Tile T = next_tile(u, kErrFwdWait + 15);
      if (T.valid <= 0) break;
      const int qt = T.qt;
      float m_used = -INFINITY;
      float l = 0.f;
      int jl = 0;
      for (int ii = T.item_begin; ii < T.item_end && ok; ++ii) {
        const fcp_item itm = a.items[ii];
        const int nkt = kv_tiles(itm, qt);
        for (int kt = 0; kt < nkt; ++kt, ++J, ++jl) {
          const int kv_valid = itm.kv_len - kt * kTileN;
          const bool diag = itm.mask == FCP_MASK_CAUSAL_DIAG && kt == qt;
          const int lim = diag ? min(r + 1, kv_valid) : kv_valid;  // visible key columns [0, lim)
          ok = mbar_wait(bar(B_SFULL + t), J & 1, abort_flag, a.err, kErrFwdWait + 8);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          uint32_t sv[128];
          tmem_ld128(s_addr, sv);
          // tiles with every column visible to every row of the warp take the short path
          // (packed float32x2 arithmetic, 3-input max); diagonal and ragged tiles mask
          const bool full = __all_sync(0xffffffffu, lim >= kTileN);
          float mx;
          if (full) {
            float mc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              mc[c] = __uint_as_float(sv[32 * c]);
#pragma unroll
              for (int e = 0; e < 15; ++e)
                mc[c] = max3f(mc[c], __uint_as_float(sv[32 * c + 1 + 2 * e]), __uint_as_float(sv[32 * c + 2 + 2 * e]));
              mc[c] = fmaxf(mc[c], __uint_as_float(sv[32 * c + 31]));
            }
            mx = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
          } else {
            mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (e < lim) mx = fmaxf(mx, __uint_as_float(sv[e]));
          }
          const float m_new = fmaxf(m_used, mx * a.scale_log2);
          float alpha = 1.f;
          const bool grow = m_new > m_used + kRescaleThreshold;
          if (grow) {
            alpha = fast_exp2(m_used - m_new);
            m_used = m_new;
          }
          const float mb = (m_used == -INFINITY) ? 0.f : m_used;
          // P in two halves of 64 keys, each handed to the MMA warp as soon as it is stored
          float rowsum = 0.f;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (full) {
              float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
              for (int c = 2 * half; c < 2 * half + 2; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const int i0 = 32 * c + 2 * e;
                  const float2 x = ffma2(__uint_as_float(sv[i0]), __uint_as_float(sv[i0 + 1]), a.scale_log2,
                                         a.scale_log2, -mb, -mb);
                  const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                  acc2 = fadd2(acc2.x, acc2.y, p0, p1);
                  pk[e] = pack_bf16(p0, p1);
                }
                tmem_st16(s_addr + c * 16, pk);
              }
              rowsum += acc2.x + acc2.y;
            } else {
#pragma unroll
              for (int c = 2 * half; c < 2 * half + 2; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const int c0 = c * 32 + 2 * e;
                  const float p0 = (c0 < lim) ? fast_exp2(fmaf(__uint_as_float(sv[c0]), a.scale_log2, -mb)) : 0.f;
                  const float p1 =
                      (c0 + 1 < lim) ? fast_exp2(fmaf(__uint_as_float(sv[c0 + 1]), a.scale_log2, -mb)) : 0.f;
                  rowsum += p0 + p1;
                  pk[e] = pack_bf16(p0, p1);
                }
                tmem_st16(s_addr + c * 16, pk);
              }
            }
            if (half == 0) {
              // O holds the sum through key tile jl-1 once PV(t, jl-1) completes; rows whose
              // maximum grew are rescaled before PV(t, jl) adds onto it (warp-uniform TMEM access).
              if (__any_sync(0xffffffffu, grow && jl > 0)) {
                ok = mbar_wait(bar(B_ODONE + t), (J - 1) & 1, abort_flag, a.err, kErrFwdWait + 9);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                  uint32_t ov[32];
                  tmem_ld32(o_addr + c * 32, ov);
#pragma unroll
                  for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                  tmem_st32(o_addr + c * 32, ov);
                }
              }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(bar(B_PFULL + 2 * t + half));
          }
          if (!ok) break;
          l = l * alpha + rowsum;
        }
      }
      if (!ok) break;
      if (jl == 0) {  // no key tile (not produced by the planner): O_t was never written
        tc_fence_before();
        mbar_arrive_warp(bar(B_OFREE + t));
        continue;
      }
      // epilogue: O_t is read out of TMEM (then released to the next tile's first PV) and
      // the normalised partial is stored
      ok = mbar_wait(bar(B_ODONE + t), (J - 1) & 1, abort_flag, a.err, kErrFwdWait + 10);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int qrow = qt * kTileM + r;
      const bool head_ok = t == 0 || T.has_h1;
      const bool store = qrow < T.q_len && head_ok;
      const int h = t ? T.h1 : T.h0;
      const long long prow = static_cast<long long>(h) * a.part_rows + T.part_row0 + qrow;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // Each 32-column slice of the warp's 32 rows goes through a shared [32][32] float32
      // block (16-byte slots XOR-swizzled by row, so neither side has bank conflicts) and
      // leaves as stores that write four whole 128-byte row segments per instruction, instead
      // of one 16-byte piece of 32 different rows.
      float4* stg = reinterpret_cast<float4*>(smem + C::kStage + warp * 4096);
      const int wrow0 = qt * kTileM + (warp & 3) * 32;   // the warp's first row in the run
      const int sub = lane >> 3, slot = lane & 7;        // store side: row sub + 4i, slot
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_addr + c * 32, ov);
        if (c == D / 32 - 1) {
          tc_fence_before();
          mbar_arrive_warp(bar(B_OFREE + t));
        }
        if (c > 0) __syncwarp();  // the previous slice has been read out of the block
#pragma unroll
        for (int e = 0; e < 8; ++e)
          stg[lane * 8 + (e ^ (lane & 7))] =
              make_float4(__uint_as_float(ov[4 * e]) * inv, __uint_as_float(ov[4 * e + 1]) * inv,
                          __uint_as_float(ov[4 * e + 2]) * inv, __uint_as_float(ov[4 * e + 3]) * inv);
        __syncwarp();
        if (head_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + sub;
            if (wrow0 + rr < T.q_len) {
              const long long orow = static_cast<long long>(h) * a.part_rows + T.part_row0 + wrow0 + rr;
              reinterpret_cast<float4*>(a.part_o + orow * D)[c * 8 + slot] = stg[rr * 8 + (slot ^ (rr & 7))];
            }
          }
        }
      }
      __syncwarp();  // the block is free for the next tile's epilogue
      if (store) a.part_lse[prow] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*unquiesced) {
    // fallback only: an issued copy or MMA did not report completion within the wait limit
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) __nanosleep(1000);
  }
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
fcp_status launch_fwd(const fcp_plan* plan, const void* d_plan, int32_t unit_begin, int32_t n_units,
                      const void* q, const void* k, const void* v, int hq, int hkv, float* part_o, float* part_lse,
                      cudaStream_t stream) {
  using C = FwdCfg<D>;
  const DevLayout& L = plan->layout;
  if (n_units == 0) return FCP_OK;
  const int64_t T = plan->total_tokens;
  CUtensorMap mq, mk, mv;
  fcp_status st;
  if ((st = make_bf16_map(&mq, q, hq, T, D, kTileM)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mk, k, hkv, T, D, kTileN)) != FCP_OK) return st;
  if ((st = make_bf16_map(&mv, v, hkv, T, D, kTileN)) != FCP_OK) return st;
  FwdArgs a;
  a.items = dev_array<fcp_item>(d_plan, L.items);
  a.runs = dev_array<fcp_run>(d_plan, L.runs);
  a.units = dev_array<FwdUnit>(d_plan, L.fwd_units) + unit_begin;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.part_rows = plan->partial_rows;
  a.hq = hq;
  a.hkv = hkv;
  a.group = hq / hkv;
  a.pairs_per_group = (a.group + 1) / 2;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  a.err = dev_error_word(d_plan);
  FCP_CUDA_TRY(cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes),
               "fwd smem attribute");
  a.n_tiles = static_cast<long long>(n_units) * hkv * a.pairs_per_group;
  a.next_tile = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(const_cast<void*>(d_plan)) +
                                                       kDevFwdTileOffset);
  FCP_CUDA_TRY(cudaMemsetAsync(a.next_tile, 0, sizeof(unsigned long long), stream), "fwd tile counter");
  // persistent: one CTA per SM (the kernel holds all 512 TMEM columns), each walking tiles
  int dev = 0, n_sm = 0;
  FCP_CUDA_TRY(cudaGetDevice(&dev), "fwd device");
  FCP_CUDA_TRY(cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev), "fwd SM count");
  const long long grid = std::min<long long>(a.n_tiles, std::max(n_sm, 1));
  fwd_kernel<D><<<static_cast<unsigned>(grid), kFwdThreads, C::kSmemBytes, stream>>>(mq, mk, mv, a);
  FCP_CUDA_TRY(cudaGetLastError(), "fwd launch");
  return FCP_OK;
}

}  // namespace
}  // namespace fcp

using namespace fcp;

namespace {
// The units [unit_begin, unit_begin + n_units) of the plan's forward unit list.
fcp_status fwd_units(const fcp_plan* plan, const void* d_plan, int32_t unit_begin, int32_t n_units, const void* q,
                     const void* k, const void* v, int32_t hq, int32_t hkv, int32_t head_dim, float* part_o,
                     float* part_lse, void* stream) {
  if (plan == nullptr || d_plan == nullptr) return FCP_ERR_INVALID;
  if (!plan->distributed) return FCP_ERR_STATE;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return FCP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return FCP_ERR_UNSUPPORTED;
  if (n_units == 0) return FCP_OK;
  if (!q || !k || !v || !part_o || !part_lse) return FCP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(part_o)) return FCP_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (head_dim == 128)
    return launch_fwd<128>(plan, d_plan, unit_begin, n_units, q, k, v, hq, hkv, part_o, part_lse, s);
  return launch_fwd<64>(plan, d_plan, unit_begin, n_units, q, k, v, hq, hkv, part_o, part_lse, s);
}
}  // namespace

extern "C" fcp_status fcp_block_attn_fwd(const fcp_plan* plan, const void* d_plan, const void* q, const void* k,
                                         const void* v, int32_t hq, int32_t hkv, int32_t head_dim, float* part_o,
                                         float* part_lse, void* stream) {
  if (plan == nullptr) return FCP_ERR_INVALID;
  return fwd_units(plan, d_plan, 0, plan->layout.n_fwd_units, q, k, v, hq, hkv, head_dim, part_o, part_lse, stream);
}

extern "C" fcp_status fcp_block_attn_fwd_stage(const fcp_plan* plan, const void* d_plan, int32_t stage,
                                               const void* q, const void* k, const void* v, int32_t hq, int32_t hkv,
                                               int32_t head_dim, float* part_o, float* part_lse, void* stream) {
  if (plan == nullptr) return FCP_ERR_INVALID;
  const std::vector<int32_t>& b = plan->layout.stage_unit_begin;
  if (stage < 0 || static_cast<size_t>(stage) + 1 >= b.size()) return FCP_ERR_INVALID;
  return fwd_units(plan, d_plan, b[stage], b[stage + 1] - b[stage], q, k, v, hq, hkv, head_dim, part_o, part_lse,
                   stream);
}
