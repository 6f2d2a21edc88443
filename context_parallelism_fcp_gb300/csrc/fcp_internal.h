// Internal definitions shared by the host plan (fcp_plan.cpp) and the device entry points
// (*.cu): the host plan object and the layout of its device image.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "fcp.h"

namespace fcp {

// Tile shape of the attention kernels: 128 query rows x 128 key rows. 128 is the M of one
// single-CTA tcgen05.mma and the number of TMEM lanes, so one thread owns one row.
constexpr int kTileM = 128;
constexpr int kTileN = 128;
// Query rows of one backward step (the N of the backward's S^T and dP^T MMAs).
constexpr int kBwdStepRows = 64;
// Query bands of the backward: off below this many tokens unless a plan asks for them, and
// this many rows per band when on by default.
constexpr int64_t kAutoBandMinTokens = 131072;
constexpr int32_t kAutoBandRows = 16384;

// A query range with its runs (consecutive in the run list): what the merge reduces.
// A query range: its tokens, how many runs reduce it and the first of its partial rows.
struct QSeg {
  int32_t tok0, len, n_runs, part_row0;
};
// Where the partials of one query token are: its k-th partial (k < count) is partial row
// base + k * stride. The runs of a query range own consecutive blocks of q_len partial
// rows, so stride is the range's length.
struct TokPart {
  int32_t base, stride, count, reserved;
};
// One forward CTA's work: query tile q_tile of run `run`.
struct FwdUnit {
  int32_t run, q_tile;
};
// A key range with the items that read it (indices into kv_items[list_begin, list_end)).
struct KvSeg {
  int32_t tok0, len, list_begin, list_end;
};
// One backward CTA's work: key tile kv_tile of key range `kvseg`.
struct BwdUnit {
  int32_t kvseg, kv_tile;
};

// Header at offset 0 of the device image. error: 0, or the code of the first device-side
// failure (a bounded wait that gave up); see fcp_device_error.
struct DevHeader {
  int32_t error;
  int32_t error_info;
  int32_t reserved0[14];
  unsigned long long fwd_next_tile;  // tile counter of the persistent forward, zeroed per launch
  int32_t reserved[46];
};
constexpr size_t kDevFwdTileOffset = 64;
static_assert(sizeof(DevHeader) == 256, "header is one 256-byte line");
static_assert(offsetof(DevHeader, fwd_next_tile) == kDevFwdTileOffset, "tile counter offset");

// Byte offsets of the arrays in the device image and their lengths.
struct DevLayout {
  size_t items = 0, runs = 0, qsegs = 0, tok2part = 0, worker_order = 0, fwd_units = 0, kvsegs = 0, kv_items = 0,
         bwd_units = 0, total = 0;
  int32_t n_qsegs = 0, n_fwd_units = 0, n_kvsegs = 0, n_kv_items = 0, n_bwd_units = 0;
  int32_t max_runs_per_qseg = 0;
  // forward units of execution stage s: [stage_unit_begin[s], stage_unit_begin[s + 1])
  std::vector<int32_t> stage_unit_begin;
  // Backward query bands (0 rows: none). Band k covers the query steps whose first row lies
  // in [k * band_rows, (k + 1) * band_rows); its units are band_units[band_begin[k],
  // band_begin[k + 1]) (indices into bwd_units, in their order).
  size_t band_units = 0;
  int32_t band_rows = 0, n_bands = 0, n_band_units = 0;
  std::vector<int32_t> band_begin;
};

// Device error codes written into DevHeader::error (kernel id * 16 + wait id).
enum DevError : int32_t {
  kErrSmemAlign = 0x01,
  kErrFwdWait = 0x10,
  kErrBwdWait = 0x20,
  kErrSelfTest = 0x40,  // the bounded-wait self-test gave up, as it must (0x41: its second wait)
};

void set_last_error(const std::string& msg);

}  // namespace fcp

struct fcp_plan {
  std::vector<int32_t> seqlens;
  int32_t block_size = 0;
  int32_t causal = 0;
  int64_t total_tokens = 0;
  int64_t total_pairs = 0;
  std::vector<fcp_block> blocks;
  std::vector<fcp_segment> segs;

  bool distributed = false;
  int32_t n_workers = 0;
  int64_t token_cap = 0;
  int32_t coalesce = 1;
  std::vector<int64_t> load, tokens;
  std::vector<fcp_item> items;
  std::vector<fcp_run> runs;
  int64_t partial_rows = 0;

  // The work list in fcp_distribute's order (items holds it too unless fcp_schedule
  // reordered them).
  std::vector<fcp_item> work_list;
  // Execution stage per item (fcp_schedule); empty: every item in stage 0.
  std::vector<int32_t> item_stage;
  int32_t n_exec_stages = 1;

  // Congestion-free solver output (fcp_solve_stages).
  bool solved = false;
  std::vector<fcp_transfer> transfers;
  int32_t n_stages = 0;

  // Backward query bands: -1 chooses (on for long batches), 0 off, > 0 rows per band.
  int32_t bwd_band_rows = -1;

  // Host copy of the device image, rebuilt after distribute/coalesce.
  std::vector<uint8_t> image;
  fcp::DevLayout layout;
};
