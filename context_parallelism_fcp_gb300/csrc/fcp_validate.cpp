// Host-side validation of a distributed plan and of its device image: every index the
// kernels follow (items, runs, partial rows, token-to-partial records, forward and backward
// tile units, the reversed work list, the backward's query bands, the workers' token order)
// is checked against the token count, the sequence boundaries and the other arrays, so a
// plan that passes can be uploaded without any kernel reading or writing outside its buffers.
//
// The coverage check restates the work list's contract ("Unleashing Scalable Context
// Parallelism for Foundation Models Pre-Training via FCP", Section 2.2 with the block pairs
// of Section 4.1): the unmasked (query, key) pairs of the items add up to those of the
// whole batch, and a causal item either pairs a block with itself (masked diagonal) or
// with an earlier block of the same sequence.
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "fcp_internal.h"

namespace fcp {
namespace {

struct Fail {
  std::string msg;
};

template <class T>
std::vector<T> image_array(const fcp_plan* p, size_t offset, size_t count) {
  std::vector<T> out(count);
  if (count == 0) return out;
  if (offset + count * sizeof(T) > p->image.size()) throw Fail{"device image array past the end of the image"};
  std::memcpy(out.data(), p->image.data() + offset, count * sizeof(T));
  return out;
}

void require(bool ok, const std::string& what) {
  if (!ok) throw Fail{what};
}

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

void validate(const fcp_plan* p) {
  require(p->distributed, "plan not distributed");
  const int64_t T = p->total_tokens;
  const int32_t N = p->n_workers;
  const int64_t n_items = static_cast<int64_t>(p->items.size());
  const int64_t n_runs = static_cast<int64_t>(p->runs.size());

  // sequence of every token
  std::vector<int64_t> seq_start(p->seqlens.size() + 1, 0);
  for (size_t s = 0; s < p->seqlens.size(); ++s) seq_start[s + 1] = seq_start[s] + p->seqlens[s];
  require(seq_start.back() == T, "token count differs from the sum of the sequence lengths");
  auto seq_of = [&](int64_t tok) -> int64_t {
    return static_cast<int64_t>(std::upper_bound(seq_start.begin(), seq_start.end(), tok) - seq_start.begin()) - 1;
  };

  // items: ranges inside one sequence, masks, pair coverage
  int64_t pairs = 0;
  for (int64_t i = 0; i < n_items; ++i) {
    const fcp_item& it = p->items[i];
    const std::string at = "item " + std::to_string(i) + ": ";
    require(it.worker >= 0 && it.worker < N, at + "worker out of range");
    require(it.q_len > 0 && it.kv_len > 0, at + "empty range");
    require(it.q_tok0 >= 0 && it.q_tok0 + static_cast<int64_t>(it.q_len) <= T, at + "query range outside [0, T)");
    require(it.kv_tok0 >= 0 && it.kv_tok0 + static_cast<int64_t>(it.kv_len) <= T, at + "key range outside [0, T)");
    const int64_t sq = seq_of(it.q_tok0);
    require(seq_of(it.q_tok0 + it.q_len - 1) == sq, at + "query range crosses a sequence boundary");
    require(seq_of(it.kv_tok0) == sq && seq_of(it.kv_tok0 + it.kv_len - 1) == sq,
            at + "key range not in the query's sequence");
    require(it.run >= 0 && it.run < n_runs, at + "run index out of range");
    if (it.mask == FCP_MASK_CAUSAL_DIAG) {
      require(p->causal != 0, at + "diagonal mask in a full-mask plan");
      require(it.q_tok0 == it.kv_tok0 && it.q_len == it.kv_len, at + "diagonal item over different ranges");
      pairs += static_cast<int64_t>(it.q_len) * (it.q_len + 1) / 2;
    } else {
      require(it.mask == FCP_MASK_FULL, at + "unknown mask");
      if (p->causal != 0)
        require(it.kv_tok0 + static_cast<int64_t>(it.kv_len) <= it.q_tok0, at + "causal key block not before its query block");
      pairs += static_cast<int64_t>(it.q_len) * it.kv_len;
    }
  }
  require(pairs == p->total_pairs, "the items' unmasked pairs differ from the batch's");

  // runs: consecutive item ranges covering the work list, one query range and stage each,
  // disjoint partial rows inside [0, partial_rows)
  int64_t next = 0;
  std::vector<std::pair<int64_t, int64_t>> rows;
  for (int64_t r = 0; r < n_runs; ++r) {
    const fcp_run& rn = p->runs[r];
    const std::string at = "run " + std::to_string(r) + ": ";
    require(rn.item_begin == next && rn.item_end > rn.item_begin && rn.item_end <= n_items, at + "item range");
    for (int32_t i = rn.item_begin; i < rn.item_end; ++i) {
      const fcp_item& it = p->items[i];
      require(it.run == r, at + "item does not point back to its run");
      require(it.worker == rn.worker && it.q_tok0 == rn.q_tok0 && it.q_len == rn.q_len, at + "mixed query ranges");
      require(p->item_stage.empty() || p->item_stage[i] == rn.stage, at + "mixed execution stages");
    }
    require(rn.stage >= 0 && rn.stage < p->n_exec_stages, at + "stage out of range");
    require(rn.part_row0 >= 0 && rn.part_row0 + static_cast<int64_t>(rn.q_len) <= p->partial_rows,
            at + "partial rows outside the partial buffer");
    rows.push_back({rn.part_row0, rn.part_row0 + static_cast<int64_t>(rn.q_len)});
    next = rn.item_end;
  }
  require(next == n_items, "runs do not cover the work list");
  std::sort(rows.begin(), rows.end());
  for (size_t k = 1; k < rows.size(); ++k) require(rows[k].first >= rows[k - 1].second, "runs share partial rows");

  // device image
  const DevLayout& L = p->layout;
  require(p->image.size() >= L.total && L.total >= sizeof(DevHeader), "device image size");
  const auto img_items = image_array<fcp_item>(p, L.items, static_cast<size_t>(n_items));
  const auto img_runs = image_array<fcp_run>(p, L.runs, static_cast<size_t>(n_runs));
  require(n_items == 0 || std::memcmp(img_items.data(), p->items.data(), img_items.size() * sizeof(fcp_item)) == 0,
          "device items differ from the host work list");
  require(n_runs == 0 || std::memcmp(img_runs.data(), p->runs.data(), img_runs.size() * sizeof(fcp_run)) == 0,
          "device runs differ from the host runs");

  // token -> partial records: every token has at least one partial, all inside the buffer
  const auto tok2part = image_array<TokPart>(p, L.tok2part, static_cast<size_t>(T));
  std::vector<int32_t> parts_of_token(static_cast<size_t>(T), 0);
  for (const fcp_run& rn : p->runs)
    for (int32_t t = 0; t < rn.q_len; ++t) ++parts_of_token[static_cast<size_t>(rn.q_tok0) + t];
  for (int64_t t = 0; t < T; ++t) {
    const TokPart& tp = tok2part[t];
    const std::string at = "token " + std::to_string(t) + ": ";
    require(tp.count == parts_of_token[t] && tp.count >= 1, at + "partial count");
    require(tp.base >= 0 && tp.stride >= 1 &&
                tp.base + static_cast<int64_t>(tp.count - 1) * tp.stride < p->partial_rows,
            at + "partial rows outside the partial buffer");
  }

  // workers' token order: a permutation of [0, T)
  const auto order = image_array<int32_t>(p, L.worker_order, static_cast<size_t>(T));
  std::vector<uint8_t> seen(static_cast<size_t>(T), 0);
  for (int32_t t : order) {
    require(t >= 0 && t < T && !seen[t], "worker order is not a permutation");
    seen[t] = 1;
  }

  // forward units: every (run, query tile) once, grouped by stage as the stage offsets say
  const auto fwd = image_array<FwdUnit>(p, L.fwd_units, static_cast<size_t>(L.n_fwd_units));
  int64_t tiles = 0;
  for (const fcp_run& rn : p->runs) tiles += ceil_div64(rn.q_len, kTileM);
  require(static_cast<int64_t>(fwd.size()) == tiles, "forward unit count");
  std::vector<std::vector<uint8_t>> fwd_seen(static_cast<size_t>(n_runs));
  for (int64_t r = 0; r < n_runs; ++r) fwd_seen[r].assign(static_cast<size_t>(ceil_div64(p->runs[r].q_len, kTileM)), 0);
  const std::vector<int32_t>& sb = L.stage_unit_begin;
  require(static_cast<int32_t>(sb.size()) == p->n_exec_stages + 1 && sb.front() == 0 &&
              sb.back() == L.n_fwd_units,
          "stage offsets of the forward units");
  for (int32_t st = 0; st < p->n_exec_stages; ++st) {
    require(sb[st] <= sb[st + 1], "stage offsets of the forward units");
    for (int32_t u = sb[st]; u < sb[st + 1]; ++u) {
      const FwdUnit& fu = fwd[u];
      require(fu.run >= 0 && fu.run < n_runs, "forward unit run out of range");
      require(fu.q_tile >= 0 && fu.q_tile < static_cast<int32_t>(fwd_seen[fu.run].size()), "forward unit tile");
      require(p->runs[fu.run].stage == st, "forward unit in the wrong stage");
      require(!fwd_seen[fu.run][fu.q_tile], "forward unit listed twice");
      fwd_seen[fu.run][fu.q_tile] = 1;
    }
  }

  // reversed work list and backward units: every key range's items read exactly that range,
  // every item is listed once, every key tile once
  const auto kvsegs = image_array<KvSeg>(p, L.kvsegs, static_cast<size_t>(L.n_kvsegs));
  const auto kv_items = image_array<int32_t>(p, L.kv_items, static_cast<size_t>(L.n_kv_items));
  require(L.n_kv_items == n_items, "reversed work list size");
  std::vector<uint8_t> item_listed(static_cast<size_t>(n_items), 0);
  for (int32_t s = 0; s < L.n_kvsegs; ++s) {
    const KvSeg& ks = kvsegs[s];
    require(ks.list_begin >= 0 && ks.list_begin <= ks.list_end && ks.list_end <= L.n_kv_items, "key range list");
    require(ks.tok0 >= 0 && ks.len > 0 && ks.tok0 + static_cast<int64_t>(ks.len) <= T, "key range outside [0, T)");
    for (int32_t k = ks.list_begin; k < ks.list_end; ++k) {
      const int32_t i = kv_items[k];
      require(i >= 0 && i < n_items && !item_listed[i], "reversed work list entry");
      item_listed[i] = 1;
      require(p->items[i].kv_tok0 == ks.tok0 && p->items[i].kv_len == ks.len, "item in the wrong key range");
    }
  }
  const auto bwd = image_array<BwdUnit>(p, L.bwd_units, static_cast<size_t>(L.n_bwd_units));
  std::vector<std::vector<uint8_t>> bwd_seen(static_cast<size_t>(L.n_kvsegs));
  int64_t key_tiles = 0;
  for (int32_t s = 0; s < L.n_kvsegs; ++s) {
    bwd_seen[s].assign(static_cast<size_t>(ceil_div64(kvsegs[s].len, kTileN)), 0);
    key_tiles += static_cast<int64_t>(bwd_seen[s].size());
  }
  require(static_cast<int64_t>(bwd.size()) == key_tiles, "backward unit count");
  for (const BwdUnit& bu : bwd) {
    require(bu.kvseg >= 0 && bu.kvseg < L.n_kvsegs, "backward unit key range out of range");
    require(bu.kv_tile >= 0 && bu.kv_tile < static_cast<int32_t>(bwd_seen[bu.kvseg].size()), "backward unit tile");
    require(!bwd_seen[bu.kvseg][bu.kv_tile], "backward unit listed twice");
    bwd_seen[bu.kvseg][bu.kv_tile] = 1;
  }

  // query bands: every (unit, band) pair where the unit has a 64-row step starting in the band
  // is listed exactly once, and nothing else is
  if (L.n_bands == 0) {
    require(L.n_band_units == 0 && L.band_begin.empty(), "band lists without bands");
    return;
  }
  require(L.band_rows > 0 && L.band_rows % kBwdStepRows == 0, "band size");
  require(static_cast<int64_t>(L.n_bands) == ceil_div64(T, L.band_rows), "band count");
  const auto& bb = L.band_begin;
  require(static_cast<int32_t>(bb.size()) == L.n_bands + 1 && bb.front() == 0 && bb.back() == L.n_band_units,
          "band offsets");
  const auto band_units = image_array<int32_t>(p, L.band_units, static_cast<size_t>(L.n_band_units));
  std::vector<std::vector<int32_t>> want(static_cast<size_t>(L.n_bands));
  for (int32_t u = 0; u < L.n_bwd_units; ++u) {
    const KvSeg& ks = kvsegs[bwd[u].kvseg];
    for (int32_t li = ks.list_begin; li < ks.list_end; ++li) {
      const fcp_item& it = p->items[kv_items[li]];
      const int64_t first = it.mask == FCP_MASK_CAUSAL_DIAG ? (int64_t(bwd[u].kv_tile) * kTileN) / kBwdStepRows : 0;
      for (int64_t qs = first; qs < ceil_div64(it.q_len, kBwdStepRows); ++qs) {
        auto& w = want[(it.q_tok0 + qs * kBwdStepRows) / L.band_rows];
        if (w.empty() || w.back() != u) w.push_back(u);
      }
    }
  }
  for (int32_t b = 0; b < L.n_bands; ++b) {
    require(bb[b] <= bb[b + 1], "band offsets");
    std::vector<int32_t> got(band_units.begin() + bb[b], band_units.begin() + bb[b + 1]);
    for (int32_t u : got) require(u >= 0 && u < L.n_bwd_units, "band unit out of range");
    std::sort(got.begin(), got.end());
    require(std::adjacent_find(got.begin(), got.end()) == got.end(), "band unit listed twice");
    std::sort(want[b].begin(), want[b].end());
    require(got == want[b], "band unit list differs from the units with steps in the band");
  }
}

}  // namespace
}  // namespace fcp

using namespace fcp;

extern "C" fcp_status fcp_plan_validate(const fcp_plan* plan) {
  if (plan == nullptr) return FCP_ERR_INVALID;
  try {
    validate(plan);
  } catch (const Fail& f) {
    set_last_error("fcp_plan_validate: " + f.msg);
    return FCP_ERR_STATE;
  }
  return FCP_OK;
}
