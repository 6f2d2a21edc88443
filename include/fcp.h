/*
 * fcp.h -- C ABI of the block-wise variable-length attention library (FCP hot path).
 *
 * The operations follow "Unleashing Scalable Context Parallelism for Foundation
 * Models Pre-Training via FCP" (arXiv 2605.08524):
 *   - Section 3.3 (problem formulation): sequences S = {s_1..s_tau}, workers
 *     W = {w_1..w_N}, a sharding function G: s_i -> {B_i1..B_ik_i} and an
 *     assignment function M: B -> w; worker load Comp(w) = sum of f(B) over its blocks.
 *   - Section 4.1 (block distributor): fixed-size blocks, short sequences packed into
 *     the fewest blocks; LPT assignment to the least-loaded worker under a strict
 *     per-worker token limit (Section 3.2, "Memory").
 *   - Section 3.2 / Figure 4: Zig-Zag pairing of a causal sequence's blocks.
 *   - Section 2.2: attention O = Softmax(Q K^T / sqrt(D) (+) M) V over [H, L, D]
 *     tensors; Section 2.3: associativity, partial results over slices of L reduced
 *     to the final output (here: the log-sum-exp merge).
 *   - Section 4.2 (bottom-up coalescer): c consecutive block sub-stages of a worker
 *     executed as one stage; block-level pipelining and the congestion-free solver
 *     (the transfers of remote KV blocks split into Delta matchings).
 *   - Section 4.3 (transparent reshuffler): the permutation between the user's token
 *     order and the workers' order.
 *
 * Conventions for every call:
 *   - Device tensors are packed over tokens in input order: Q, O, dO, dQ are
 *     [Hq, T, D] bf16, K, V, dK, dV are [Hkv, T, D] bf16, LSE is [Hq, T] float32
 *     (natural log), all contiguous, row-major, D innermost. T is the sum of the
 *     sequence lengths given to fcp_partition. Base addresses must be 16-byte aligned.
 *   - Query head h reads KV head h / (Hq / Hkv). Scale is 1/sqrt(D). D is 64 or 128.
 *   - "stream" is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Device calls are asynchronous on that stream and only enqueue work.
 *   - The caller owns every device buffer. The library owns only the host plan
 *     (released by fcp_plan_free) and allocates no device memory.
 *   - No call asserts, traps or exits. Errors are returned as fcp_status; on
 *     FCP_ERR_CUDA, fcp_last_error() gives the CUDA error text. A kernel that gives
 *     up a bounded wait sets an error word in the device plan image; read it with
 *     fcp_device_error().
 *   - A host plan is not thread-safe; distinct plans are independent.
 */
#ifndef FCP_H_
#define FCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FCP_OK = 0,
  FCP_ERR_INVALID = 1,     /* a malformed argument (null pointer, negative length, bad shape) */
  FCP_ERR_CAPACITY = 2,    /* a block fits no worker under the token cap */
  FCP_ERR_UNSUPPORTED = 3, /* a valid but unsupported shape (e.g. D not in {64,128}) */
  FCP_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed */
  FCP_ERR_STATE = 5,       /* calls out of order (e.g. upload before distribute) */
  FCP_ERR_DEVICE = 6       /* a kernel reported a device-side error (bounded wait gave up) */
} fcp_status;

typedef enum { FCP_MASK_FULL = 0, FCP_MASK_CAUSAL_DIAG = 1 } fcp_mask_kind;

/* One block B of the sharding G. A packed block (seq = -1) holds several short
 * sequences as consecutive segments. zz_partner is the Zig-Zag partner of block
 * seq_block_idx in a causal sequence of seq_nblocks blocks (seq_nblocks-1-idx), or -1.
 * cost is f(B): the unmasked (query, key) score pairs whose query lies in B. */
typedef struct {
  int32_t first_seg, n_segs, tokens, seq, seq_block_idx, seq_nblocks, zz_partner, worker;
  int64_t cost;
} fcp_block;

/* A contiguous token range of one sequence inside a block; tok0 is its offset in T. */
typedef struct {
  int32_t seq, start_in_seq, len, tok0;
} fcp_segment;

/* A work item: the query range [q_tok0, q_tok0+q_len) against the key range
 * [kv_tok0, kv_tok0+kv_len). FULL: every key visible. CAUSAL_DIAG: the two ranges are
 * the same and key j is visible to query i iff j <= i. run: its partial-result slot. */
typedef struct {
  int32_t worker, q_block, kv_block, q_tok0, q_len, kv_tok0, kv_len, mask, run, reserved;
} fcp_item;

/* A run: items [item_begin, item_end) of one worker over one query range, reduced into
 * one partial (O, LSE) at rows [part_row0, part_row0 + q_len) of the partial buffers.
 * stage: the execution stage the run belongs to (0 unless fcp_schedule ordered the plan).
 * The runs of one query range own consecutive partial rows, q_len apart. */
typedef struct {
  int32_t worker, q_block, q_tok0, q_len, item_begin, item_end, part_row0, stage;
} fcp_run;

/* One block transfer of the communication plan: KV block kv_block moves from its owner
 * src to worker dst (which owns a Q block that attends to it), in congestion-free
 * sub-stage `stage`. tokens is the block's length. */
typedef struct {
  int32_t kv_block, src, dst, stage, tokens, reserved;
} fcp_transfer;

typedef struct fcp_plan fcp_plan;

/* Read-only view of a host plan. Pointers stay valid until the next mutating call on
 * the plan (fcp_distribute, fcp_coalesce, fcp_schedule) or fcp_plan_free.
 * n_exec_stages: execution stages of the forward (1 unless fcp_schedule ran). */
typedef struct {
  int32_t n_seqs, n_blocks, n_segs, n_items, n_runs, n_workers, block_size, causal, coalesce;
  int32_t distributed, n_exec_stages;
  int64_t total_tokens, token_cap, total_pairs, partial_rows;
  const int32_t* seqlens;
  const fcp_block* blocks;
  const fcp_segment* segs;
  const fcp_item* items;
  const fcp_run* runs;
  const int64_t* worker_load;   /* Comp(w): sum of block costs, n_workers entries */
  const int64_t* worker_tokens; /* sum of len(B) per worker, n_workers entries */
} fcp_plan_view;

/* Sharding G (Section 4.1, "Sharding Policy"; Zig-Zag of Section 3.2, Figure 4).
 * seqlens: n_seqs lengths >= 0 (host memory, copied). A sequence of length >= block_size
 * becomes ceil(L/block_size) blocks aligned at its start (the last may be short); the
 * shorter ones are packed first-fit-decreasing (ties: lower sequence index) into
 * block_size-token blocks. Block ids: unpacked sequences in input order, then packed
 * blocks. causal != 0 selects the causal mask for every sequence. On success *out
 * receives a new plan owned by the caller (fcp_plan_free). Errors: FCP_ERR_INVALID for a
 * null pointer, n_seqs < 0, block_size <= 0, a negative length or T >= 2^31. */
fcp_status fcp_partition(const int32_t* seqlens, int32_t n_seqs, int32_t block_size, int32_t causal,
                         fcp_plan** out);

/* Assignment M (Section 4.1, "Assignment Policy"; token limit of Section 3.2): blocks in
 * decreasing cost (ties: lower id) each go to the least-loaded worker (ties: lower id)
 * whose tokens + len(B) <= token_cap; token_cap <= 0 selects block_size*ceil(K/N). Then
 * builds the work list: per worker, per owned block (ascending id), per segment; an
 * unpacked causal block j of a sequence pairs with KV blocks 0..j (j: CAUSAL_DIAG, others
 * FULL), a full-mask block with every block of its sequence, a packed segment with itself.
 * Runs are rebuilt with coalesce degree 1 (one partial per item). Errors: FCP_ERR_INVALID
 * (null plan, n_workers <= 0), FCP_ERR_CAPACITY (the plan is left undistributed),
 * FCP_ERR_UNSUPPORTED (more than 2^31 - 1 partial rows or work items; also from
 * fcp_coalesce and fcp_schedule). */
fcp_status fcp_distribute(fcp_plan* plan, int32_t n_workers, int64_t token_cap);

/* The ring-attention baseline the pages compare against (Section 3.4, "Balance-optimized",
 * Figure 5a; Zig-Zag of Figure 4), as a distributed plan: every sequence of length L is cut
 * into 2N equal blocks, block j covering [j*L/(2N), (j+1)*L/(2N)) (integer division; empty
 * blocks are skipped, so a sequence shorter than 2N tokens has fewer blocks), and worker w
 * takes blocks w and 2N-1-w of every sequence. Block ids follow the sequences in input order;
 * the work list, runs, device image and token_cap (= the largest worker's tokens) are built
 * as in fcp_distribute, so every other call (fcp_coalesce, fcp_solve_stages, the kernels)
 * accepts the result. Errors: FCP_ERR_INVALID as fcp_partition, or n_workers <= 0. */
fcp_status fcp_partition_ring(const int32_t* seqlens, int32_t n_seqs, int32_t n_workers, int32_t causal,
                              fcp_plan** out);

/* Bottom-up coalescing (Section 4.2): rebuild runs so that up to `degree` consecutive
 * items of one worker over the same query range share one partial result. degree = 1
 * gives one partial per (Q-block, KV-block) pair. A plan that fcp_schedule ordered returns
 * to the work-list order first. Errors: FCP_ERR_INVALID (degree <= 0), FCP_ERR_STATE (not
 * distributed). */
fcp_status fcp_coalesce(fcp_plan* plan, int32_t degree);

/* Congestion-free solver (Section 4.2, "Congestion-free solver"; Lemmas 1 and 2; Figure 8):
 * builds the data-flow bipartite multigraph of a distributed plan -- one edge S(src) ->
 * R(dst) per distinct (KV block, receiving worker) whose block is owned elsewhere, in
 * work-list order -- and partitions its edges into Delta disjoint matchings, Delta being
 * the maximum number of blocks any worker sends or receives (the optimum: a stage is a
 * matching, Lemma 1, and the busiest worker needs Delta stages, Lemma 2). The graph is
 * padded to Delta-regular with dummy edges and perfect matchings are peeled off with
 * Hopcroft-Karp. Results: fcp_plan_transfers. Errors: FCP_ERR_INVALID, FCP_ERR_STATE (not
 * distributed). Recomputed by each call; cleared by fcp_distribute. */
fcp_status fcp_solve_stages(fcp_plan* plan);

/* A caller-supplied congestion-free plan in place of the solver's (the pages note that the
 * plan may be pre-computed elsewhere, Section 4.2): stages[i] is the sub-stage of the i-th
 * edge of the plan's data-flow graph, the edges taken in the order fcp_solve_stages lists
 * them (distinct (KV block, receiver) pairs, work-list order). n_transfers must equal the
 * number of edges; every sub-stage must be a matching (each worker sends at most one block
 * and receives at most one), each in [0, 2^24). The number of sub-stages becomes
 * max(stages) + 1, which may exceed Delta. Errors: FCP_ERR_INVALID (count mismatch, a stage
 * out of range, a sub-stage that is not a matching; the plan is left unsolved),
 * FCP_ERR_STATE (not distributed). */
fcp_status fcp_set_stages(fcp_plan* plan, const int32_t* stages, int32_t n_transfers);

/* Read-only access to the solver's result: *transfers (n_transfers entries, valid until
 * the next mutating call) and the number of sub-stages. FCP_ERR_STATE if not solved. */
fcp_status fcp_plan_transfers(const fcp_plan* plan, const fcp_transfer** transfers, int32_t* n_transfers,
                              int32_t* n_stages);

/* Block-level pipeline with the bottom-up coalescer (Section 4.2, "Block-level pipelining",
 * "Bottom-up coalescer", Figure 7): runs the solver if needed, then gives every work item
 * the execution stage in which its KV block is available -- stage 0 for blocks the worker
 * owns (local computation first, Section 4.3), 1 + s / degree for a block pulled in
 * congestion-free sub-stage s, i.e. `degree` consecutive sub-stages merged into one stage
 * -- reorders each worker's items by stage (stable, keeping the work-list order within a
 * stage) and rebuilds the runs so that none crosses a stage; in each stage a worker
 * receives at most `degree` blocks. *n_stages receives the number of execution stages.
 * fcp_block_attn_fwd_stage then runs one stage at a time; fcp_block_attn_fwd runs them all.
 * Errors: FCP_ERR_INVALID (degree <= 0), FCP_ERR_STATE (not distributed). */
fcp_status fcp_schedule(fcp_plan* plan, int32_t degree, int32_t* n_stages);
/* (fcp_schedule starts from the work list of fcp_distribute and uses the sub-stages in
 * place when it is called; after fcp_solve_stages or fcp_set_stages, call it again.
 * fcp_coalesce returns the plan to the unscheduled work-list order.) */

/* Host-side check of a distributed plan and its device image (no counterpart on the pages;
 * the defence that stands in for a device-side bounds checker): every item's query and key
 * ranges lie inside [0, T) and inside one sequence; a causal item pairs a block with itself
 * or with an earlier block; the items' unmasked pairs add up to the batch's; runs cover the
 * work list with disjoint partial rows inside the partial buffer; every token's partial
 * records, the forward units (per execution stage), the reversed work list, the backward
 * units and the workers' token order are complete and in range. FCP_OK, or FCP_ERR_STATE
 * with the first violation in fcp_last_error(). Plans built by this library always pass. */
fcp_status fcp_plan_validate(const fcp_plan* plan);

/* Fill *view with read-only pointers into the plan. */
fcp_status fcp_plan_query(const fcp_plan* plan, fcp_plan_view* view);

/* Bytes of the device image of a distributed plan (work list, runs, tile schedules,
 * token-to-range map, error word); 0 if not distributed. */
size_t fcp_plan_device_bytes(const fcp_plan* plan);

/* Copy the device image into caller-owned device memory d_plan (>= fcp_plan_device_bytes,
 * 256-byte aligned) on `stream`, clearing its error word. The host plan must stay alive
 * and unmodified while kernels that use d_plan run. Errors: FCP_ERR_STATE, FCP_ERR_INVALID
 * (too small or misaligned), FCP_ERR_CUDA. */
fcp_status fcp_plan_upload(const fcp_plan* plan, void* d_plan, size_t bytes, void* stream);

/* Sizes of the partial buffers for (Hq, D): part_o float32 [Hq, partial_rows, D] and
 * part_lse float32 [Hq, partial_rows]. */
fcp_status fcp_partial_sizes(const fcp_plan* plan, int32_t hq, int32_t head_dim, size_t* o_bytes,
                             size_t* lse_bytes);

/* Forward over the work list (Section 2.2 attention per item; Section 2.3 partial results):
 * for every run r, query head h and query row i of the run's range, the softmax of the
 * scaled masked scores over the keys of the run's items, giving part_o[h, part_row0 + i, :]
 * (normalised over those keys) and part_lse[h, part_row0 + i] (natural log-sum-exp).
 * Inputs q, k, v bf16 device tensors as above; outputs float32 device buffers sized by
 * fcp_partial_sizes. The kernel is persistent and takes its tiles from a counter kept in
 * d_plan (reset on `stream` before the launch), so forward launches that share one d_plan
 * must be ordered on one stream. Errors: FCP_ERR_INVALID (nulls, Hq % Hkv != 0),
 * FCP_ERR_UNSUPPORTED (D), FCP_ERR_STATE, FCP_ERR_CUDA. */
fcp_status fcp_block_attn_fwd(const fcp_plan* plan, const void* d_plan, const void* q, const void* k,
                              const void* v, int32_t hq, int32_t hkv, int32_t head_dim, float* part_o,
                              float* part_lse, void* stream);

/* The forward of one execution stage only (the runs whose stage field is `stage`), with
 * the arguments of fcp_block_attn_fwd. Running every stage and then the merge gives the
 * same result as fcp_block_attn_fwd + merge. Errors as fcp_block_attn_fwd, and
 * FCP_ERR_INVALID for a stage outside [0, n_stages). */
fcp_status fcp_block_attn_fwd_stage(const fcp_plan* plan, const void* d_plan, int32_t stage, const void* q,
                                    const void* k, const void* v, int32_t hq, int32_t hkv, int32_t head_dim,
                                    float* part_o, float* part_lse, void* stream);

/* Associative log-sum-exp merge (Section 2.3) of every run's partial into the final
 * output: per (h, token) with partials s over its query range, m = max lse_s,
 * w_s = exp(lse_s - m), o = sum w_s O_s / sum w_s (bf16), lse = m + log sum w_s (float32).
 * o is [Hq, T, D] bf16, lse [Hq, T] float32. */
fcp_status fcp_block_attn_merge(const fcp_plan* plan, const void* d_plan, const float* part_o,
                                const float* part_lse, int32_t hq, int32_t head_dim, void* o, float* lse,
                                void* stream);

/* Backward prologue: di[h, t] = sum_d dO[h,t,d] * O[h,t,d] (float32 [Hq, T]) and
 * dq_acc[h, t, :] = 0 (float32 [Hq, T, D]). */
fcp_status fcp_block_attn_bwd_prologue(const fcp_plan* plan, const void* o, const void* dout, int32_t hq,
                                       int32_t head_dim, float* di, float* dq_acc, void* stream);

/* Workspace bytes for fcp_block_attn_bwd: a float32 dQ accumulator [Hq, T, D] followed by
 * the float32 Di [Hq, T] (each 256-byte aligned). */
size_t fcp_bwd_workspace_bytes(const fcp_plan* plan, int32_t hq, int32_t head_dim);

/* Query bands of the backward (no counterpart on the pages; a schedule of the backward on one
 * GPU). With bands, the backward runs as one launch per band of band_rows query rows: each
 * launch walks only the query steps whose first row lies in its band, so the CTAs running
 * together walk the same slice of query rows head by head and share, while they are in L2, the
 * dQ rows they add into and the Q/dO/LSE/Di rows they read; dK and dV are summed over the bands in float32 scratch (fcp_bwd_band_workspace_bytes) and
 * written as bf16 at the end. band_rows: -1 lets the plan choose (16384 for batches of at least
 * 131072 tokens, else none; the default), 0 none, > 0 rows per band (a multiple of 64).
 * Measured on one causal sequence, 64/8 heads, D = 128 (backward ms, one box per row):
 * 524288 tokens 13664 with none, 12181 / 10813 / 10234 with 2048 / 4096 / 8192-row bands, and
 * on another box 10397 / 9969 / 11082 with 8192 / 16384 / 32768; 131072 tokens 761-791 with
 * none, 615-617 with 8192 and 605-606 with 16384; 65536 tokens 150.0-150.2 with none and
 * 148.9-149.0 with 16384; 32768 tokens 36.74-36.80 with none and 36.66-36.88 with 16384.
 * May be called before or after fcp_distribute; a distributed plan's device image is rebuilt
 * (upload it again). Errors: FCP_ERR_INVALID. */
fcp_status fcp_plan_set_bwd_band(fcp_plan* plan, int32_t band_rows);

/* The bands of a distributed plan: *n_bands (0: none) and *band_rows. FCP_ERR_STATE if the
 * plan is not distributed. */
fcp_status fcp_plan_bwd_bands(const fcp_plan* plan, int32_t* n_bands, int32_t* band_rows);

/* Float32 scratch for dK and dV summed over the query bands ([2][Hkv, T, D], each half
 * 256-byte aligned), 0 if the plan has no bands. fcp_block_attn_bwd runs banded when the plan
 * has bands and its workspace holds fcp_bwd_workspace_bytes + this many bytes. */
size_t fcp_bwd_band_workspace_bytes(const fcp_plan* plan, int32_t hkv, int32_t head_dim);

/* Backward over the same work list (the exact gradient of the Section 2.2 attention; the
 * pages implement a backward but describe only the forward): with P = exp(S*scale - lse),
 * dV = sum P^T dO, dP = dO V^T, dS = P * (dP - Di), dQ = scale dS K, dK = scale dS^T Q,
 * KV gradients summed over the query heads of their group. lse is the merged LSE from
 * fcp_block_attn_merge, o the merged output. Launches the prologue, the tile kernel and
 * the dQ conversion on `stream`. dq [Hq,T,D], dk and dv [Hkv,T,D] bf16 outputs; workspace
 * of fcp_bwd_workspace_bytes, 256-byte aligned, to which a plan with query bands adds
 * fcp_bwd_band_workspace_bytes to run banded (with less it runs in one launch). */
fcp_status fcp_block_attn_bwd(const fcp_plan* plan, const void* d_plan, const void* q, const void* k,
                              const void* v, const void* o, const void* dout, const float* lse, int32_t hq,
                              int32_t hkv, int32_t head_dim, void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, void* stream);

/* The tile kernel of fcp_block_attn_bwd alone: given di and a dq_acc zeroed by the prologue,
 * accumulates float32 dQ / scale into dq_acc [Hq, T, D] (atomically) and writes dk, dv
 * [Hkv, T, D] bf16. dq_acc is caller-owned scratch (256-byte aligned). */
fcp_status fcp_block_attn_bwd_tiles(const fcp_plan* plan, const void* d_plan, const void* q, const void* k,
                                    const void* v, const void* dout, const float* lse, const float* di,
                                    int32_t hq, int32_t hkv, int32_t head_dim, float* dq_acc, void* dk, void* dv,
                                    void* stream);

/* The banded tile kernels of fcp_block_attn_bwd alone (a plan with query bands): zeroes
 * dkv_acc (float32 [2][Hkv, T, D] of fcp_bwd_band_workspace_bytes, 256-byte aligned), launches
 * the tile kernel once per band, accumulating dQ / scale into dq_acc as
 * fcp_block_attn_bwd_tiles does and dK, dV into dkv_acc, then writes dk, dv [Hkv, T, D] bf16.
 * FCP_ERR_STATE if the plan has no bands. */
fcp_status fcp_block_attn_bwd_tiles_banded(const fcp_plan* plan, const void* d_plan, const void* q, const void* k,
                                           const void* v, const void* dout, const float* lse, const float* di,
                                           int32_t hq, int32_t hkv, int32_t head_dim, float* dq_acc,
                                           float* dkv_acc, void* dk, void* dv, void* stream);

/* The last step of fcp_block_attn_bwd alone: dq = bf16(dq_acc / sqrt(D)) over [Hq, T, D]. */
fcp_status fcp_block_attn_bwd_dq_convert(const fcp_plan* plan, const float* dq_acc, int32_t hq, int32_t head_dim,
                                         void* dq, void* stream);

/* Backward that allocates nothing (the paper has no counterpart; this serves callers that
 * cannot call cudaMalloc -- code running inside a memory pool that owns the whole device, an
 * allocation-free serving or real-time loop, or a C host without a device allocator). Same
 * arguments, results and errors as fcp_block_attn_bwd, without the workspace: the scratch
 * (float32 dQ accumulator and Di, fcp_bwd_workspace_bytes) lives in a fixed device array
 * of fcp_bwd_static_scratch_bytes() = 32 MiB inside the library, which every GPU that loads
 * the library holds until the process exits. A larger requirement returns
 * FCP_ERR_UNSUPPORTED with the sizes in fcp_last_error(). The first call on a device looks
 * up the array's device address with that device current and keeps it for the life of the
 * process; make that first call before any stream capture, and do not use this entry point
 * on a device after cudaDeviceReset (the reset discards the array, and the kept address
 * would be stale). All calls share the one array: calls whose work overlaps on the GPU (other
 * streams, other threads) race on it and must be serialised by the caller. Each call
 * re-zeroes the accumulator itself, so nothing needs clearing between calls. */
size_t fcp_bwd_static_scratch_bytes(void);
fcp_status fcp_block_attn_bwd_static_scratch(const fcp_plan* plan, const void* d_plan, const void* q,
                                             const void* k, const void* v, const void* o, const void* dout,
                                             const float* lse, int32_t hq, int32_t hkv, int32_t head_dim, void* dq,
                                             void* dk, void* dv, void* stream);

/* Transparent reshuffle (Section 4.3): the two all-to-alls around attention become, on one
 * GPU, a permutation of token rows between the user's layout (tokens in input order) and
 * the workers' layout (worker 0's blocks in ascending id -- each block's segments in order
 * -- then worker 1's, ...). For every head h < heads and row i < T:
 *   direction 0 (to workers):  dst[h, i, :] = src[h, user_token(i), :]
 *   direction 1 (to users):    dst[h, user_token(i), :] = src[h, i, :]
 * where user_token(i) is the input position of worker-layout row i. src and dst are
 * distinct device buffers of heads * T * row_bytes bytes; row_bytes is a multiple of 16
 * (e.g. 256 for bf16 rows of D = 128). Errors: FCP_ERR_INVALID, FCP_ERR_STATE, FCP_ERR_CUDA. */
fcp_status fcp_reshuffle(const fcp_plan* plan, const void* d_plan, const void* src, void* dst, int32_t heads,
                         int32_t row_bytes, int32_t direction, void* stream);

/* Synchronise `stream`, copy the device plan's error word to *code (0 = none; else the
 * kernel and wait that gave up) and clear it. Returns FCP_ERR_DEVICE if it was set. */
fcp_status fcp_device_error(const void* d_plan, int32_t* code, void* stream);

/* Self-test of the device-side failure path (no counterpart on the pages): two threads wait,
 * each with one of the bounded mbarrier waits the tile kernels use (the polling wait of the
 * forward, the poll-then-suspend wait of the backward), on barriers that nothing ever
 * completes. After the waits' 2-second limit the first records code 0x40 in the error word of
 * d_plan (int32 word 0) and the second code 0x41 in int32 word 1, and the kernel exits; the
 * context stays usable. d_plan is a device buffer of at least 256 bytes, 256-byte aligned,
 * whose first two words should be clear. Read word 0 with fcp_device_error. Errors:
 * FCP_ERR_INVALID, FCP_ERR_CUDA. */
fcp_status fcp_selftest_bounded_wait(void* d_plan, void* stream);

void fcp_plan_free(fcp_plan* plan);
const char* fcp_status_string(fcp_status status);
/* Detail of the last FCP_ERR_CUDA in this thread ("" if none). */
const char* fcp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FCP_H_ */
