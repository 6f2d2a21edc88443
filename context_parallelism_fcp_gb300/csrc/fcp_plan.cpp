// Host plan: sharding G, Zig-Zag partners, LPT assignment M under a token cap, the work
// list, coalesced runs and the device image with the kernels' tile schedules.
//
// "Unleashing Scalable Context Parallelism for Foundation Models Pre-Training via FCP":
// Section 3.3 (G, M, Comp(w)), Section 4.1 (fixed-size blocks, packing of short sequences,
// LPT to the least-loaded worker, O(K log N)), Section 3.2 (per-worker token limit; Zig-Zag,
// Figure 4), Section 4.2 (bottom-up coalescer).
#include <algorithm>
#include <cstring>
#include <map>
#include <numeric>
#include <set>
#include <utility>

#include "fcp_internal.h"

namespace fcp {

namespace {
thread_local std::string g_last_error;

// Unmasked score pairs of the queries at positions [start, start+len) of a sequence of
// length seq_len: causal sum_{i=start}^{start+len-1} (i+1), full len * seq_len.
int64_t segment_cost(int64_t start, int64_t len, int64_t seq_len, bool causal) {
  if (causal) return start * len + len * (len + 1) / 2;
  return len * seq_len;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

// Key tiles a query tile q_tile of item `it` visits: all of the key range, or up to and
// including the diagonal tile for a causal diagonal item (its query and key ranges coincide).
int32_t kv_tiles_of(const fcp_item& it, int32_t q_tile) {
  int32_t n = ceil_div(it.kv_len, kTileN);
  if (it.mask == FCP_MASK_CAUSAL_DIAG) n = std::min(n, q_tile + 1);
  return n;
}

// Query tiles that see key tile kv_tile of item `it`.
int32_t q_tiles_seeing(const fcp_item& it, int32_t kv_tile) {
  int32_t n = ceil_div(it.q_len, kTileM);
  if (it.mask == FCP_MASK_CAUSAL_DIAG) n = std::max(0, n - kv_tile);
  return n;
}

// Run ids grouped by query range (q_tok0, q_len), ranges in order of first appearance.
std::vector<std::vector<int32_t>> runs_by_range(const std::vector<fcp_run>& runs) {
  std::map<std::pair<int32_t, int32_t>, size_t> index;
  std::vector<std::vector<int32_t>> out;
  for (int32_t r = 0; r < static_cast<int32_t>(runs.size()); ++r) {
    auto ins = index.insert({{runs[r].q_tok0, runs[r].q_len}, out.size()});
    if (ins.second) out.emplace_back();
    out[ins.first->second].push_back(r);
  }
  return out;
}

// Runs: consecutive items of one worker over one query range (and one execution stage),
// at most `degree` items each (no limit when degree <= 0). Partial rows are allocated per
// query range, in order of first appearance, so the runs of a range own consecutive
// blocks of q_len rows.
void build_runs(fcp_plan* p, int32_t degree) {
  p->runs.clear();
  const size_t n = p->items.size();
  auto stage_of = [&](size_t i) { return p->item_stage.empty() ? 0 : p->item_stage[i]; };
  size_t i = 0;
  while (i < n) {
    const fcp_item& a = p->items[i];
    size_t j = i + 1;
    while (j < n && (degree <= 0 || static_cast<int32_t>(j - i) < degree) && p->items[j].worker == a.worker &&
           p->items[j].q_tok0 == a.q_tok0 && p->items[j].q_len == a.q_len && stage_of(j) == stage_of(i))
      ++j;
    fcp_run r{};
    r.worker = a.worker;
    r.q_block = a.q_block;
    r.q_tok0 = a.q_tok0;
    r.q_len = a.q_len;
    r.item_begin = static_cast<int32_t>(i);
    r.item_end = static_cast<int32_t>(j);
    r.part_row0 = -1;
    r.stage = stage_of(i);
    const int32_t run_id = static_cast<int32_t>(p->runs.size());
    for (size_t t = i; t < j; ++t) p->items[t].run = run_id;
    p->runs.push_back(r);
    i = j;
  }
  // partial rows per query range
  const auto ranges = runs_by_range(p->runs);
  int64_t row = 0;
  for (const auto& rg : ranges)
    for (int32_t r : rg) {
      p->runs[r].part_row0 = static_cast<int32_t>(row);
      row += p->runs[r].q_len;
    }
  p->partial_rows = row;
  p->coalesce = degree;
}

template <class T>
void put(std::vector<uint8_t>& img, size_t off, const std::vector<T>& v) {
  if (!v.empty()) std::memcpy(img.data() + off, v.data(), v.size() * sizeof(T));
}

// Device image: header, items, runs, query ranges with their runs, token -> partial rows,
// forward units (longest first), key ranges with their items, backward units (longest first).
// Device image of a distributed plan. FCP_ERR_UNSUPPORTED if its 32-bit indices would
// overflow, FCP_ERR_STATE if an internal invariant fails.
fcp_status build_image(fcp_plan* p) {
  // partial rows and item indices are 32-bit in the device image
  if (p->partial_rows > INT32_MAX || p->items.size() > static_cast<size_t>(INT32_MAX)) {
    set_last_error("plan too large: more than 2^31 - 1 partial rows or work items (raise the coalesce degree)");
    return FCP_ERR_UNSUPPORTED;
  }
  const auto ranges = runs_by_range(p->runs);
  std::vector<QSeg> qsegs;
  int32_t max_runs = 0;
  std::vector<TokPart> tok2part(static_cast<size_t>(p->total_tokens), TokPart{0, 0, 0, 0});
  for (const auto& rg : ranges) {
    const fcp_run& r0 = p->runs[rg.front()];
    const int32_t n = static_cast<int32_t>(rg.size());
    max_runs = std::max(max_runs, n);
    for (int32_t k = 0; k < n; ++k)
      if (p->runs[rg[k]].part_row0 != r0.part_row0 + k * r0.q_len) return FCP_ERR_STATE;  // contiguous rows
    qsegs.push_back(QSeg{r0.q_tok0, r0.q_len, n, r0.part_row0});
    for (int32_t t = 0; t < r0.q_len; ++t)
      tok2part[static_cast<size_t>(r0.q_tok0) + t] = TokPart{r0.part_row0 + t, r0.q_len, n, 0};
  }

  // forward units with their key-tile counts; longest first, ties in run/tile order
  std::vector<std::pair<int64_t, FwdUnit>> fu;
  for (int32_t r = 0; r < static_cast<int32_t>(p->runs.size()); ++r) {
    const fcp_run& run = p->runs[r];
    for (int32_t qt = 0; qt < ceil_div(run.q_len, kTileM); ++qt) {
      int64_t work = 0;
      for (int32_t i = run.item_begin; i < run.item_end; ++i) work += kv_tiles_of(p->items[i], qt);
      fu.push_back({work, FwdUnit{r, qt}});
    }
  }
  std::stable_sort(fu.begin(), fu.end(),
                   [&](const std::pair<int64_t, FwdUnit>& a, const std::pair<int64_t, FwdUnit>& b) {
                     const int32_t sa = p->runs[a.second.run].stage, sb = p->runs[b.second.run].stage;
                     if (sa != sb) return sa < sb;
                     return a.first > b.first;
                   });
  std::vector<FwdUnit> fwd_units;
  fwd_units.reserve(fu.size());
  for (auto& x : fu) fwd_units.push_back(x.second);
  std::vector<int32_t> stage_begin(static_cast<size_t>(p->n_exec_stages) + 1, 0);
  for (const FwdUnit& u : fwd_units) ++stage_begin[static_cast<size_t>(p->runs[u.run].stage) + 1];
  for (int32_t st = 0; st < p->n_exec_stages; ++st) stage_begin[st + 1] += stage_begin[st];

  // key ranges, each with the items that read it (ordered by query offset)
  std::vector<int32_t> order(p->items.size());
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    const fcp_item& x = p->items[a];
    const fcp_item& y = p->items[b];
    if (x.kv_tok0 != y.kv_tok0) return x.kv_tok0 < y.kv_tok0;
    if (x.kv_len != y.kv_len) return x.kv_len < y.kv_len;
    return x.q_tok0 < y.q_tok0;
  });
  std::vector<KvSeg> kvsegs;
  std::vector<int32_t> kv_items;
  for (int32_t idx : order) {
    const fcp_item& it = p->items[idx];
    if (kvsegs.empty() || kvsegs.back().tok0 != it.kv_tok0 || kvsegs.back().len != it.kv_len) {
      const int32_t at = static_cast<int32_t>(kv_items.size());
      kvsegs.push_back(KvSeg{it.kv_tok0, it.kv_len, at, at});
    }
    kv_items.push_back(idx);
    kvsegs.back().list_end = static_cast<int32_t>(kv_items.size());
  }
  std::vector<std::pair<int64_t, BwdUnit>> bu;
  for (int32_t s = 0; s < static_cast<int32_t>(kvsegs.size()); ++s) {
    for (int32_t kt = 0; kt < ceil_div(kvsegs[s].len, kTileN); ++kt) {
      int64_t work = 0;
      for (int32_t i = kvsegs[s].list_begin; i < kvsegs[s].list_end; ++i)
        work += q_tiles_seeing(p->items[kv_items[i]], kt);
      bu.push_back({work, BwdUnit{s, kt}});
    }
  }
  std::stable_sort(bu.begin(), bu.end(),
                   [](const std::pair<int64_t, BwdUnit>& a, const std::pair<int64_t, BwdUnit>& b) {
                     return a.first > b.first;
                   });
  std::vector<BwdUnit> bwd_units;
  bwd_units.reserve(bu.size());
  for (auto& x : bu) bwd_units.push_back(x.second);

  // Backward query bands: band k lists the units with a query step whose first row lies in
  // [k * R, (k + 1) * R). A unit's steps over one item are the 64-row steps from the one
  // holding the key tile's first key (causal diagonal) or 0 to the end of the item's rows.
  const int32_t R = p->bwd_band_rows > 0 ? p->bwd_band_rows
                    : (p->bwd_band_rows < 0 && p->total_tokens >= kAutoBandMinTokens ? kAutoBandRows : 0);
  std::vector<int32_t> band_begin, band_units;
  if (R > 0 && !bwd_units.empty()) {
    std::vector<std::vector<int32_t>> per(static_cast<size_t>(ceil_div(p->total_tokens, R)));
    for (int32_t u = 0; u < static_cast<int32_t>(bwd_units.size()); ++u) {
      const KvSeg& sg = kvsegs[bwd_units[u].kvseg];
      const int32_t kt = bwd_units[u].kv_tile;
      for (int32_t i = sg.list_begin; i < sg.list_end; ++i) {
        const fcp_item& it = p->items[kv_items[i]];
        const int32_t q_first = it.mask == FCP_MASK_CAUSAL_DIAG ? (kt * kTileN) / kBwdStepRows : 0;
        const int32_t q_end = ceil_div(it.q_len, kBwdStepRows);
        if (q_first >= q_end) continue;
        const int64_t b0 = (static_cast<int64_t>(it.q_tok0) + int64_t(q_first) * kBwdStepRows) / R;
        const int64_t b1 = (static_cast<int64_t>(it.q_tok0) + int64_t(q_end - 1) * kBwdStepRows) / R;
        for (int64_t b = b0; b <= b1; ++b)
          if (per[b].empty() || per[b].back() != u) per[b].push_back(u);
      }
    }
    band_begin.push_back(0);
    for (const auto& v : per) {
      band_units.insert(band_units.end(), v.begin(), v.end());
      band_begin.push_back(static_cast<int32_t>(band_units.size()));
    }
  }

  // workers' token layout: worker w's blocks in ascending id, their segments in order
  std::vector<int32_t> worker_order;
  worker_order.reserve(static_cast<size_t>(p->total_tokens));
  for (int32_t w = 0; w < p->n_workers; ++w)
    for (const fcp_block& B : p->blocks) {
      if (B.worker != w) continue;
      for (int32_t si = B.first_seg; si < B.first_seg + B.n_segs; ++si)
        for (int32_t t = 0; t < p->segs[si].len; ++t) worker_order.push_back(p->segs[si].tok0 + t);
    }
  if (static_cast<int64_t>(worker_order.size()) != p->total_tokens) return FCP_ERR_STATE;

  DevLayout L;
  size_t off = sizeof(DevHeader);
  L.items = off;
  off = align256(off + p->items.size() * sizeof(fcp_item));
  L.runs = off;
  off = align256(off + p->runs.size() * sizeof(fcp_run));
  L.qsegs = off;
  off = align256(off + qsegs.size() * sizeof(QSeg));
  L.tok2part = off;
  off = align256(off + tok2part.size() * sizeof(TokPart));
  L.worker_order = off;
  off = align256(off + worker_order.size() * sizeof(int32_t));
  L.fwd_units = off;
  off = align256(off + fwd_units.size() * sizeof(FwdUnit));
  L.kvsegs = off;
  off = align256(off + kvsegs.size() * sizeof(KvSeg));
  L.kv_items = off;
  off = align256(off + kv_items.size() * sizeof(int32_t));
  L.bwd_units = off;
  off = align256(off + bwd_units.size() * sizeof(BwdUnit));
  L.band_units = off;
  off = align256(off + band_units.size() * sizeof(int32_t));
  L.total = off;
  L.n_qsegs = static_cast<int32_t>(qsegs.size());
  L.n_fwd_units = static_cast<int32_t>(fwd_units.size());
  L.n_kvsegs = static_cast<int32_t>(kvsegs.size());
  L.n_kv_items = static_cast<int32_t>(kv_items.size());
  L.n_bwd_units = static_cast<int32_t>(bwd_units.size());
  L.max_runs_per_qseg = max_runs;
  L.stage_unit_begin = std::move(stage_begin);
  L.band_rows = band_begin.empty() ? 0 : R;
  L.n_bands = band_begin.empty() ? 0 : static_cast<int32_t>(band_begin.size()) - 1;
  L.n_band_units = static_cast<int32_t>(band_units.size());
  L.band_begin = std::move(band_begin);

  for (const TokPart& tp : tok2part)
    if (tp.count <= 0) return FCP_ERR_STATE;  // every token must belong to exactly one query range
  p->image.assign(L.total, 0);
  put(p->image, L.items, p->items);
  put(p->image, L.runs, p->runs);
  put(p->image, L.qsegs, qsegs);
  put(p->image, L.tok2part, tok2part);
  put(p->image, L.worker_order, worker_order);
  put(p->image, L.fwd_units, fwd_units);
  put(p->image, L.kvsegs, kvsegs);
  put(p->image, L.kv_items, kv_items);
  put(p->image, L.bwd_units, bwd_units);
  put(p->image, L.band_units, band_units);
  p->layout = L;
  return FCP_OK;
}

// Loads, tokens, work list, runs and device image of a plan whose blocks have owners.
// Work list: per worker, per owned block (ascending id), per segment; an unpacked causal
// block j of a sequence pairs with KV blocks 0..j of it (j: CAUSAL_DIAG), a full-mask block
// with every block of its sequence, a packed segment with itself.
fcp_status finish_distribution(fcp_plan* p, const std::vector<int32_t>& owner, int32_t n_workers, int64_t cap) {
  const int32_t K = static_cast<int32_t>(p->blocks.size());
  std::vector<int64_t> load(static_cast<size_t>(n_workers), 0), tokens(static_cast<size_t>(n_workers), 0);
  for (int32_t b = 0; b < K; ++b) {
    load[owner[b]] += p->blocks[b].cost;
    tokens[owner[b]] += p->blocks[b].tokens;
  }

  // blocks of each unpacked sequence, in position order (they were created in order)
  std::vector<std::vector<int32_t>> seq_blocks(p->seqlens.size());
  for (int32_t b = 0; b < K; ++b)
    if (p->blocks[b].seq >= 0) seq_blocks[p->blocks[b].seq].push_back(b);

  std::vector<std::vector<int32_t>> owned(static_cast<size_t>(n_workers));
  for (int32_t b = 0; b < K; ++b) owned[owner[b]].push_back(b);

  const bool c = p->causal != 0;
  p->items.clear();
  for (int32_t w = 0; w < n_workers; ++w) {
    for (int32_t qb : owned[w]) {
      const fcp_block& B = p->blocks[qb];
      for (int32_t si = B.first_seg; si < B.first_seg + B.n_segs; ++si) {
        const fcp_segment& qs = p->segs[si];
        if (B.seq < 0) {
          fcp_item it{w, qb, qb, qs.tok0, qs.len, qs.tok0, qs.len,
                      c ? FCP_MASK_CAUSAL_DIAG : FCP_MASK_FULL, -1, 0};
          p->items.push_back(it);
          continue;
        }
        const auto& kvs = seq_blocks[B.seq];
        const size_t nkv = c ? static_cast<size_t>(B.seq_block_idx) + 1 : kvs.size();
        for (size_t x = 0; x < nkv; ++x) {
          const int32_t kb = kvs[x];
          const fcp_segment& ks = p->segs[p->blocks[kb].first_seg];
          fcp_item it{w, qb, kb, qs.tok0, qs.len, ks.tok0, ks.len,
                      (c && kb == qb) ? FCP_MASK_CAUSAL_DIAG : FCP_MASK_FULL, -1, 0};
          p->items.push_back(it);
        }
      }
    }
  }
  p->n_workers = n_workers;
  p->token_cap = cap;
  p->load = std::move(load);
  p->tokens = std::move(tokens);
  p->work_list = p->items;
  p->distributed = true;
  p->solved = false;
  p->transfers.clear();
  p->n_stages = 0;
  p->item_stage.clear();
  p->n_exec_stages = 1;
  build_runs(p, 1);
  if (const fcp_status st = build_image(p); st != FCP_OK) {
    p->distributed = false;
    return st;
  }
  return FCP_OK;
}

}  // namespace

void set_last_error(const std::string& msg) { g_last_error = msg; }

}  // namespace fcp

using namespace fcp;

extern "C" {

fcp_status fcp_partition(const int32_t* seqlens, int32_t n_seqs, int32_t block_size, int32_t causal,
                         fcp_plan** out) {
  if (out == nullptr || n_seqs < 0 || block_size <= 0 || (n_seqs > 0 && seqlens == nullptr))
    return FCP_ERR_INVALID;
  *out = nullptr;
  int64_t T = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    if (seqlens[i] < 0) return FCP_ERR_INVALID;
    T += seqlens[i];
  }
  if (T >= (int64_t(1) << 31)) return FCP_ERR_INVALID;

  fcp_plan* p = new fcp_plan();
  p->seqlens.assign(seqlens, seqlens + n_seqs);
  p->block_size = block_size;
  p->causal = causal ? 1 : 0;
  p->total_tokens = T;
  const bool c = p->causal != 0;

  std::vector<int32_t> seq_start(static_cast<size_t>(n_seqs), 0);
  int64_t acc = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    seq_start[i] = static_cast<int32_t>(acc);
    acc += seqlens[i];
    p->total_pairs += c ? int64_t(seqlens[i]) * (seqlens[i] + 1) / 2 : int64_t(seqlens[i]) * seqlens[i];
  }

  // sequences of at least one block: ceil(L/b) blocks from the start, in input order
  for (int32_t i = 0; i < n_seqs; ++i) {
    const int32_t L = seqlens[i];
    if (L < block_size) continue;
    const int32_t k = ceil_div(L, block_size);
    for (int32_t j = 0; j < k; ++j) {
      const int32_t start = j * block_size;
      const int32_t len = std::min(block_size, L - start);
      fcp_block b{};
      b.first_seg = static_cast<int32_t>(p->segs.size());
      b.n_segs = 1;
      b.tokens = len;
      b.seq = i;
      b.seq_block_idx = j;
      b.seq_nblocks = k;
      b.zz_partner = (c && k - 1 - j != j) ? k - 1 - j : -1;
      b.worker = -1;
      b.cost = segment_cost(start, len, L, c);
      p->blocks.push_back(b);
      p->segs.push_back(fcp_segment{i, start, len, seq_start[i] + start});
    }
  }

  // shorter sequences: first-fit-decreasing into block_size-token bins
  std::vector<int32_t> shorts;
  for (int32_t i = 0; i < n_seqs; ++i)
    if (seqlens[i] > 0 && seqlens[i] < block_size) shorts.push_back(i);
  std::stable_sort(shorts.begin(), shorts.end(),
                   [&](int32_t a, int32_t b) { return seqlens[a] > seqlens[b]; });
  std::vector<std::vector<int32_t>> bins;
  std::vector<int32_t> room;
  for (int32_t i : shorts) {
    size_t bi = 0;
    while (bi < bins.size() && room[bi] < seqlens[i]) ++bi;
    if (bi == bins.size()) {
      bins.emplace_back();
      room.push_back(block_size);
    }
    bins[bi].push_back(i);
    room[bi] -= seqlens[i];
  }
  for (const auto& members : bins) {
    fcp_block b{};
    b.first_seg = static_cast<int32_t>(p->segs.size());
    b.n_segs = static_cast<int32_t>(members.size());
    b.seq = -1;
    b.seq_block_idx = 0;
    b.seq_nblocks = 1;
    b.zz_partner = -1;
    b.worker = -1;
    for (int32_t i : members) {
      p->segs.push_back(fcp_segment{i, 0, seqlens[i], seq_start[i]});
      b.tokens += seqlens[i];
      b.cost += segment_cost(0, seqlens[i], seqlens[i], c);
    }
    p->blocks.push_back(b);
  }
  *out = p;
  return FCP_OK;
}

fcp_status fcp_distribute(fcp_plan* p, int32_t n_workers, int64_t token_cap) {
  if (p == nullptr || n_workers <= 0) return FCP_ERR_INVALID;
  const int32_t K = static_cast<int32_t>(p->blocks.size());
  const int64_t cap =
      token_cap > 0 ? token_cap : int64_t(p->block_size) * (K > 0 ? ceil_div(K, n_workers) : 1);

  std::vector<int32_t> order(static_cast<size_t>(K));
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return p->blocks[a].cost > p->blocks[b].cost; });

  // Workers ordered by (load, id); the first with room under the cap takes the block.
  std::vector<int64_t> load(static_cast<size_t>(n_workers), 0), tokens(static_cast<size_t>(n_workers), 0);
  std::set<std::pair<int64_t, int32_t>> by_load;
  for (int32_t w = 0; w < n_workers; ++w) by_load.insert({0, w});
  std::vector<int32_t> owner(static_cast<size_t>(K), -1);
  for (int32_t b : order) {
    const int64_t need = p->blocks[b].tokens;
    int32_t chosen = -1;
    for (auto it = by_load.begin(); it != by_load.end(); ++it) {
      if (tokens[it->second] + need <= cap) {
        chosen = it->second;
        by_load.erase(it);
        break;
      }
    }
    if (chosen < 0) {
      for (auto& blk : p->blocks) blk.worker = -1;
      p->distributed = false;
      return FCP_ERR_CAPACITY;
    }
    owner[b] = chosen;
    load[chosen] += p->blocks[b].cost;
    tokens[chosen] += need;
    by_load.insert({load[chosen], chosen});
  }
  for (int32_t b = 0; b < K; ++b) p->blocks[b].worker = owner[b];
  return finish_distribution(p, owner, n_workers, cap);
}

fcp_status fcp_partition_ring(const int32_t* seqlens, int32_t n_seqs, int32_t n_workers, int32_t causal,
                              fcp_plan** out) {
  if (out == nullptr || n_seqs < 0 || n_workers <= 0 || (n_seqs > 0 && seqlens == nullptr)) return FCP_ERR_INVALID;
  *out = nullptr;
  int64_t T = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    if (seqlens[i] < 0) return FCP_ERR_INVALID;
    T += seqlens[i];
  }
  if (T >= (int64_t(1) << 31)) return FCP_ERR_INVALID;
  fcp_plan* p = new fcp_plan();
  p->seqlens.assign(seqlens, seqlens + n_seqs);
  p->causal = causal ? 1 : 0;
  p->total_tokens = T;
  const bool c = p->causal != 0;
  const int64_t two_n = 2 * int64_t(n_workers);
  std::vector<int32_t> owner;
  int32_t max_len = 1;
  int64_t acc = 0;
  for (int32_t i = 0; i < n_seqs; ++i) {
    const int64_t L = seqlens[i];
    const int32_t tok0 = static_cast<int32_t>(acc);
    acc += L;
    p->total_pairs += c ? L * (L + 1) / 2 : L * L;
    std::vector<int32_t> grid(static_cast<size_t>(two_n), -1);
    const int32_t first = static_cast<int32_t>(p->blocks.size());
    int32_t dense = 0;
    for (int64_t j = 0; j < two_n; ++j) {
      const int64_t a = j * L / two_n, e = (j + 1) * L / two_n;
      if (e == a) continue;
      fcp_block b{};
      b.first_seg = static_cast<int32_t>(p->segs.size());
      b.n_segs = 1;
      b.tokens = static_cast<int32_t>(e - a);
      b.seq = i;
      b.seq_block_idx = dense++;
      b.worker = static_cast<int32_t>(j < n_workers ? j : two_n - 1 - j);
      b.cost = segment_cost(a, e - a, L, c);
      grid[static_cast<size_t>(j)] = static_cast<int32_t>(p->blocks.size());
      owner.push_back(b.worker);
      max_len = std::max(max_len, b.tokens);
      p->blocks.push_back(b);
      p->segs.push_back(fcp_segment{i, static_cast<int32_t>(a), static_cast<int32_t>(e - a), tok0 + static_cast<int32_t>(a)});
    }
    for (int64_t j = 0; j < two_n; ++j) {
      const int32_t id = grid[static_cast<size_t>(j)];
      if (id < 0) continue;
      p->blocks[id].seq_nblocks = dense;
      const int32_t partner = grid[static_cast<size_t>(two_n - 1 - j)];
      p->blocks[id].zz_partner = (c && partner >= 0 && partner != id) ? partner : -1;
    }
    (void)first;
  }
  p->block_size = max_len;
  fcp_status st = finish_distribution(p, owner, n_workers, 0);
  if (st != FCP_OK) {
    delete p;
    return st;
  }
  p->token_cap = *std::max_element(p->tokens.begin(), p->tokens.end());
  *out = p;
  return FCP_OK;
}

fcp_status fcp_coalesce(fcp_plan* p, int32_t degree) {
  if (p == nullptr || degree <= 0) return FCP_ERR_INVALID;
  if (!p->distributed) return FCP_ERR_STATE;
  if (!p->item_stage.empty()) {  // back to the work-list order of fcp_distribute
    p->items = p->work_list;
    p->item_stage.clear();
    p->n_exec_stages = 1;
  }
  build_runs(p, degree);
  if (const fcp_status st = build_image(p); st != FCP_OK) {
    p->distributed = false;
    return st;
  }
  return FCP_OK;
}

fcp_status fcp_schedule(fcp_plan* p, int32_t degree, int32_t* n_stages) {
  if (p == nullptr || degree <= 0) return FCP_ERR_INVALID;
  if (!p->distributed) return FCP_ERR_STATE;
  if (!p->solved) {
    fcp_status st = fcp_solve_stages(p);
    if (st != FCP_OK) return st;
  }
  // sub-stage of each remote (KV block, receiver) pair
  std::vector<std::vector<std::pair<int32_t, int32_t>>> arrive(static_cast<size_t>(p->n_workers));
  for (const fcp_transfer& t : p->transfers) arrive[t.dst].push_back({t.kv_block, t.stage});
  p->items = p->work_list;
  const size_t n = p->items.size();
  std::vector<int32_t> stage(n, 0);
  int32_t n_exec = 1;
  for (size_t i = 0; i < n; ++i) {
    const fcp_item& it = p->items[i];
    if (p->blocks[it.kv_block].worker == it.worker) continue;  // local: stage 0
    int32_t sub = -1;
    for (const auto& a : arrive[it.worker])
      if (a.first == it.kv_block) sub = a.second;
    if (sub < 0) return FCP_ERR_STATE;  // every remote pair has a transfer
    stage[i] = 1 + sub / degree;
    n_exec = std::max(n_exec, stage[i] + 1);
  }
  std::vector<size_t> order(n);
  std::iota(order.begin(), order.end(), size_t(0));
  std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) {
    if (p->items[a].worker != p->items[b].worker) return p->items[a].worker < p->items[b].worker;
    return stage[a] < stage[b];
  });
  std::vector<fcp_item> items(n);
  std::vector<int32_t> item_stage(n);
  for (size_t k = 0; k < n; ++k) {
    items[k] = p->items[order[k]];
    item_stage[k] = stage[order[k]];
  }
  p->items = std::move(items);
  p->item_stage = std::move(item_stage);
  p->n_exec_stages = n_exec;
  build_runs(p, 0);
  if (const fcp_status st = build_image(p); st != FCP_OK) {
    p->distributed = false;
    return st;
  }
  p->coalesce = degree;
  if (n_stages != nullptr) *n_stages = n_exec;
  return FCP_OK;
}

fcp_status fcp_plan_query(const fcp_plan* p, fcp_plan_view* v) {
  if (p == nullptr || v == nullptr) return FCP_ERR_INVALID;
  std::memset(v, 0, sizeof(*v));
  v->n_seqs = static_cast<int32_t>(p->seqlens.size());
  v->n_blocks = static_cast<int32_t>(p->blocks.size());
  v->n_segs = static_cast<int32_t>(p->segs.size());
  v->n_items = static_cast<int32_t>(p->items.size());
  v->n_runs = static_cast<int32_t>(p->runs.size());
  v->n_workers = p->n_workers;
  v->block_size = p->block_size;
  v->causal = p->causal;
  v->coalesce = p->coalesce;
  v->distributed = p->distributed ? 1 : 0;
  v->n_exec_stages = p->n_exec_stages;
  v->total_tokens = p->total_tokens;
  v->token_cap = p->token_cap;
  v->total_pairs = p->total_pairs;
  v->partial_rows = p->partial_rows;
  v->seqlens = p->seqlens.data();
  v->blocks = p->blocks.data();
  v->segs = p->segs.data();
  v->items = p->items.data();
  v->runs = p->runs.data();
  v->worker_load = p->load.data();
  v->worker_tokens = p->tokens.data();
  return FCP_OK;
}

fcp_status fcp_plan_set_bwd_band(fcp_plan* p, int32_t band_rows) {
  if (p == nullptr || band_rows < -1 || (band_rows > 0 && band_rows % kBwdStepRows != 0)) return FCP_ERR_INVALID;
  p->bwd_band_rows = band_rows;
  if (!p->distributed) return FCP_OK;  // applied when the plan is distributed
  if (const fcp_status st = build_image(p); st != FCP_OK) {
    p->distributed = false;
    return st;
  }
  return FCP_OK;
}

fcp_status fcp_plan_bwd_bands(const fcp_plan* p, int32_t* n_bands, int32_t* band_rows) {
  if (p == nullptr || n_bands == nullptr || band_rows == nullptr) return FCP_ERR_INVALID;
  if (!p->distributed) return FCP_ERR_STATE;
  *n_bands = p->layout.n_bands;
  *band_rows = p->layout.band_rows;
  return FCP_OK;
}

size_t fcp_plan_device_bytes(const fcp_plan* p) {
  if (p == nullptr || !p->distributed) return 0;
  return p->layout.total;
}

fcp_status fcp_partial_sizes(const fcp_plan* p, int32_t hq, int32_t head_dim, size_t* o_bytes,
                             size_t* lse_bytes) {
  if (p == nullptr || o_bytes == nullptr || lse_bytes == nullptr || hq <= 0 || head_dim <= 0)
    return FCP_ERR_INVALID;
  if (!p->distributed) return FCP_ERR_STATE;
  *o_bytes = size_t(hq) * size_t(p->partial_rows) * size_t(head_dim) * sizeof(float);
  *lse_bytes = size_t(hq) * size_t(p->partial_rows) * sizeof(float);
  return FCP_OK;
}

size_t fcp_bwd_workspace_bytes(const fcp_plan* p, int32_t hq, int32_t head_dim) {
  if (p == nullptr || hq <= 0 || head_dim <= 0) return 0;
  const size_t T = size_t(p->total_tokens);
  return align256(size_t(hq) * T * size_t(head_dim) * sizeof(float)) + align256(size_t(hq) * T * sizeof(float));
}

size_t fcp_bwd_band_workspace_bytes(const fcp_plan* p, int32_t hkv, int32_t head_dim) {
  if (p == nullptr || hkv <= 0 || head_dim <= 0 || !p->distributed || p->layout.n_bands == 0) return 0;
  return 2 * align256(size_t(hkv) * size_t(p->total_tokens) * size_t(head_dim) * sizeof(float));
}

void fcp_plan_free(fcp_plan* p) { delete p; }

const char* fcp_status_string(fcp_status s) {
  switch (s) {
    case FCP_OK: return "ok";
    case FCP_ERR_INVALID: return "invalid argument";
    case FCP_ERR_CAPACITY: return "a block fits no worker under the token cap";
    case FCP_ERR_UNSUPPORTED: return "unsupported shape";
    case FCP_ERR_CUDA: return "CUDA error";
    case FCP_ERR_STATE: return "plan not in the required state";
    case FCP_ERR_DEVICE: return "device-side error (a bounded wait gave up)";
  }
  return "unknown status";
}

const char* fcp_last_error(void) { return fcp::g_last_error.c_str(); }

}  // extern "C"
