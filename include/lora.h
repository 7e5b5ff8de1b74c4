/*
 * lora.h -- C ABI of the GB300 (sm_103a) multi-adapter LoRA library.
 *
 * For a batch of tokens, each tagged with an adapter id (-1 = none), the
 * library adds the low-rank delta of each token's own adapter to the base
 * layer output without merging weights:
 *
 *     y[t] = y_base[t] + scale_i * ((x[t] A_i^T) B_i^T),   i = lora_id_map[t] >= 0
 *
 * ("vLLM-Ascend dynamic LoRA fused operator", section 1.1 for the two-matmul
 * definition, section 2.1 for the operator inputs and outputs).  Adapters may
 * have different ranks (1..64).  The MoE variant adds the gate/up and down
 * deltas of an expert block ("[SGLang] LoRA + MoE fusion", stages 1.5/3.5).
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are plain host memory.  bf16 means IEEE bfloat16 bit patterns.
 *   - Matrices are row-major with a leading dimension in elements.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work: none of lora_pack_weights' successors blocks the
 *     host, except lora_get_status, which synchronises `stream`.
 *   - Argument errors are reported synchronously and launch nothing.  Errors
 *     found on the device (bad ids, a bounded wait that ran out) set a sticky
 *     word in the workspace that lora_get_status reads and clears.  No call
 *     traps or aborts the GPU context.
 *   - The same inputs give bit-identical outputs on every call.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *lora_stream_t; /* == cudaStream_t */

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,      /* bad pointer, size, alignment or handle; nothing launched */
    LORA_ERR_CUDA = 2,             /* a CUDA runtime call failed */
    LORA_ERR_OOM = 3,              /* table allocation failed */
    LORA_ERR_BAD_ADAPTER_ID = 4,   /* an id >= L or < -1 was seen (those rows were left unchanged) */
    LORA_ERR_BAD_EXPERT_ID = 5,    /* a top-k expert id outside [0, E) was seen (pair skipped) */
    LORA_ERR_TIMEOUT = 6,          /* a bounded in-kernel wait ran out; rebuild segments before reuse */
    LORA_ERR_WORKSPACE = 7,        /* the workspace is too small for this call's work list */
    LORA_ERR_UNSUPPORTED = 8       /* shape outside the supported range */
} lora_status;

/* Opaque handle to a packed, immutable adapter weight table (library-owned device memory). */
typedef struct lora_table_s *lora_table;

/*
 * One adapter of one projection.
 *   rank : true rank r, 1..64.  Stored rank is r rounded up to a multiple of 16
 *          with zero rows/columns ("vLLM-Ascend dynamic LoRA fused operator",
 *          section 4.3); the padding never changes a result.
 *   scale: multiplies the expand result (use 1.0 for the plain definition).
 *   A    : bf16 device, [E_A][n_a * rank][K] row-major (row block s of A is the
 *          shrink weight of slice s, "[SGLang] LoRA Layers", A = (3r, in) for QKV).
 *   B    : bf16 device, [E_B][N][rank] row-major, N = sum of slice widths
 *          (B = (q + 2kv, r) for QKV).
 */
typedef struct {
    int32_t rank;
    float scale;
    const void *A;
    const void *B;
} lora_adapter_desc;

/*
 * Shape of one LoRA-wrapped projection.
 *   K        : in-features, a multiple of 8, at most 2^20.
 *   n_slices : 1..4 output slices ("[SGLang] LoRA Layers": q/k/v, gate/up).
 *   slice_n  : slice widths, each a multiple of 8; N = sum; slice s occupies
 *              output columns [off_s, off_s + slice_n[s]).
 *   n_a      : row blocks of A: n_slices (slice s uses block s) or 1 (every
 *              slice uses the one block, e.g. the MoE gate/up A shared by gate
 *              and up).
 *   E_A, E_B : expert dimension of A and of B: 1 (shared by all experts, or a
 *              dense layer) or the MoE expert count ("[SGLang] LoRA + MoE
 *              fusion", LoRAInfo: gate_up A [L, 1, r, hidden] when
 *              experts_shared_outer_loras, B [L, E, gate_up_dim, r]).
 */
typedef struct {
    int32_t K;
    int32_t n_slices;
    int32_t slice_n[4];
    int32_t n_a;
    int32_t E_A;
    int32_t E_B;
} lora_proj_shape;

/*
 * Build a rank-grouped contiguous weight table from L adapters
 * ("vLLM-Ascend dynamic LoRA fused operator", section 2.1: adapters of equal
 * rank are stored in one contiguous run, A and B alike, and each adapter's
 * start is found by a lookup on its id; laid out once at load time, section
 * 3.1).  The table owns one device allocation per stored rank; A is kept
 * K-major and B pre-laid for the expand, so no step transposes on the device
 * (section 2.2).
 *
 * The copies run on `stream`; the caller's A/B buffers must stay valid until
 * that work completes, after which they may be freed.  *out receives the
 * handle.  Errors: LORA_ERR_INVALID_ARG (L < 1, rank outside 1..64, K or a
 * slice width not a multiple of 8, n_a not 1 or n_slices, NULL pointers),
 * LORA_ERR_OOM, LORA_ERR_CUDA.
 */
lora_status lora_pack_weights(const lora_adapter_desc *adapters, int32_t L, const lora_proj_shape *shape,
                              lora_stream_t stream, lora_table *out);

/*
 * Hot-swap one adapter of a live table ("vLLM-Ascend dynamic LoRA fused
 * operator", section 3.1: a fixed-size device pool per rank group, blocks
 * taken on load and returned whole on unload instead of frequent allocation;
 * section 4.3: replacing an adapter while steps run needs a version lock or a
 * double buffer).  The new weights (any rank 1..64; `adapter` as in
 * lora_pack_weights, same K, slices and expert counts as the table) are packed
 * on `stream` into a free block of the pool of their stored rank, then the
 * adapter's lookup entries are rewritten on `stream`: launches enqueued on
 * `stream` before this call read the old adapter, launches after it the new
 * one, and none reads a mix.  The replaced block returns to the pool once
 * `stream` has passed the new entries.  A pool with no free block of that
 * rank grows by one chunk of 4 blocks (a device allocation: not during stream
 * capture).  Work on other streams that uses the table must be ordered with
 * `stream` by the caller.  Not thread-safe against other calls on the same
 * table.  Errors: LORA_ERR_INVALID_ARG (index outside [0, L), rank outside
 * 1..64, NULL pointers), LORA_ERR_OOM, LORA_ERR_CUDA.
 */
lora_status lora_table_set_adapter(lora_table table, int32_t index, const lora_adapter_desc *adapter,
                                   lora_stream_t stream);

/* Free a table.  The caller must ensure no enqueued work still uses it. */
lora_status lora_table_destroy(lora_table table);

/* Host-visible facts about a packed table (for inspection and tests). */
typedef struct {
    int32_t L, K, N, n_slices, n_a, E_A, E_B;
    int32_t num_rank_groups;      /* distinct stored ranks */
    int64_t device_bytes;         /* bytes of packed A and B, pool blocks included */
    int32_t stored_rank_of_max;   /* stored rank of the largest adapter */
} lora_table_info_t;
lora_status lora_table_info(lora_table table, lora_table_info_t *info);

/* Stored (padded) rank of one adapter of `table`, or -1 on a bad argument. */
int32_t lora_table_stored_rank(lora_table table, int32_t adapter);

/*
 * Caller-owned device workspace for one stream.  Holds the segment table built
 * by lora_build_segments (an input of lora_apply / lora_moe_delta) plus the
 * scratch those kernels use to hand rank-sized partial results between thread
 * blocks.  Size it with lora_workspace_bytes; fill the fields; the library
 * never frees d_ptr.  One workspace serves every projection of a forward pass
 * (any table with the same adapter count L), as long as its calls are ordered
 * on one stream: calls that share a workspace must not overlap on the GPU.
 *   max_M       : the largest token count passed to lora_build_segments.
 *   L           : adapter count (must equal the tables' L).
 *   topk, num_experts, block_m : MoE alignment parameters; block_m = 0 means
 *                 dense only ("[SGLang] LoRA + MoE fusion": block_size_m).
 * d_ptr must be 256-byte aligned (any cudaMalloc / torch allocation is).
 */
typedef struct {
    void *d_ptr;
    size_t bytes;
    int32_t max_M;
    int32_t L;
    int32_t topk;
    int32_t num_experts;
    int32_t block_m;
} lora_workspace;

/* Bytes a workspace with these parameters needs (0 on a bad argument). */
size_t lora_workspace_bytes(int32_t max_M, int32_t L, int32_t topk, int32_t num_experts, int32_t block_m);

/*
 * Byte offsets, inside the workspace, of the arrays lora_build_segments writes,
 * so callers can read them back.  All arrays are int32.
 *   header         : [16]  M, num_segments, num_valid, num_moe_groups, topk,
 *                          E, block_m, P_max, B_max, reserved...
 *   perm           : [max_M] token index at each sorted position; tokens of
 *                    adapter 0 first (ascending), then adapter 1, ...; -1,
 *                    disabled and bad-id tokens last.
 *   segments       : [seg_capacity][4] (adapter, expert=0, start in perm, count)
 *                    for every adapter with tokens, ascending adapter id.
 *   sorted_ids     : [L][P_max] MoE pair ids p = t*topk + k grouped by ascending
 *                    expert, each group padded to a multiple of block_m with the
 *                    sentinel M*topk ("moe_lora_align_block_size" output).
 *   expert_ids     : [L][B_max] expert of each block_m block, -1 if unused.
 *   ntpp           : [L] num_tokens_post_padded per adapter.
 *   moe_groups     : [moe_group_capacity][4] (adapter, expert, index into
 *                    sorted_ids, count) for every non-empty (adapter, expert).
 * P_max = roundup(M*topk + E*(block_m-1), block_m) for the M of the last build
 * (the row stride of sorted_ids), B_max = P_max / block_m.
 */
typedef struct {
    size_t header, perm, segments, sorted_ids, expert_ids, ntpp, moe_groups, scratch;
    int32_t seg_capacity, moe_group_capacity;
} lora_workspace_layout_t;
lora_status lora_workspace_layout(const lora_workspace *ws, lora_workspace_layout_t *out);

/*
 * Segment table by bucketing tokens on their adapter id ("vLLM-Ascend dynamic
 * LoRA fused operator", section 2.3; work per core fixed before the compute
 * starts, section 2.4), built on the device so the step needs no host sync.
 * A stable counting sort of d_lora_id_map (int32 [M], device) into perm and
 * the segment list.  With d_topk_ids (int32 [M][topk], device) it also builds
 * the (adapter, expert) block alignment of the MoE variant ("[SGLang] LoRA +
 * MoE fusion", moe_lora_align_block_size).  d_adapter_enabled (uint8 [L],
 * device, NULL = all enabled) drops disabled adapters as if their tokens had
 * id -1 ("[SGLang] LoRA + MoE fusion", adapter_enabled under graph capture).
 * M may be 0.  Out-of-range ids are treated as -1 and raise
 * LORA_ERR_BAD_ADAPTER_ID / LORA_ERR_BAD_EXPERT_ID through lora_get_status.
 * Also resets the workspace scratch.  Errors (synchronous):
 * LORA_ERR_INVALID_ARG, LORA_ERR_WORKSPACE (bytes too small, M > max_M).
 */
lora_status lora_build_segments(const lora_workspace *ws, const int32_t *d_lora_id_map, int32_t M,
                                const int32_t *d_topk_ids, const uint8_t *d_adapter_enabled, lora_stream_t stream);

/*
 * Fused shrink -> expand -> add for every segment ("vLLM-Ascend dynamic LoRA
 * fused operator", section 2.3: per segment X_seg A_i^T, then times B_i^T,
 * added to the base rows, all segments in one operator instance; section 4.2:
 * the rank-sized intermediate accumulates in fp32).  Reads the segment table
 * of the last lora_build_segments on `ws`.  Workspaces of at most 32 tokens
 * take one launch of the persistent engine (small tiles, the shrink-to-expand
 * hand-off in L2); larger ones take the streaming path: a shrink kernel and an
 * expand kernel chained with programmatic dependent launch (64-row tiles,
 * tcgen05 shrink and expand).  LORA_OPT_PATH overrides the choice.
 *   d_x : bf16 [M][ldx] device, the layer input (K columns used).
 *   d_y : bf16 [M][ldy] device, in: the base output y_base, out: y (N columns).
 *         Rows of tokens without an adapter are not touched.
 * ldx >= K and ldy >= N, both multiples of 8; d_x and d_y 16-byte aligned.
 * Errors (synchronous): LORA_ERR_INVALID_ARG (also table L != ws->L).
 * Device-side: LORA_ERR_TIMEOUT, LORA_ERR_WORKSPACE via lora_get_status.
 */
lora_status lora_apply(lora_table table, const lora_workspace *ws, const void *d_x, int64_t ldx, void *d_y,
                       int64_t ldy, lora_stream_t stream);

/*
 * lora_build_segments(ws, d_lora_id_map, M, NULL, NULL) followed by
 * lora_apply(table, ws, d_x, ldx, d_y, ldy): the same results, bit for bit,
 * and the same segment table left in `ws` for later lora_apply calls.  When
 * every group is sure to run on small tiles (dense, M <= 32, M at most
 * LORA_OPT_TC_MIN_ROWS, or half of it when the table's largest A block has
 * more than 128 rows, or LORA_OPT_PATH = 1) both run in one launch: each
 * thread block sorts the ids itself, and one of them writes the table.  That
 * launch does not reset the workspace scratch; it needs the scratch as every
 * launch that completed without error leaves it (a fresh zero-filled
 * workspace, or one that lora_build_segments has reset, after an error).
 * Otherwise it makes the two calls.  Errors: those of the two calls.
 */
lora_status lora_build_and_apply(lora_table table, const lora_workspace *ws, const int32_t *d_lora_id_map, int32_t M,
                                 const void *d_x, int64_t ldx, void *d_y, int64_t ldy, lora_stream_t stream);

typedef enum { LORA_MOE_GATE_UP = 0, LORA_MOE_DOWN = 1 } lora_moe_stage;

/*
 * LoRA delta inside an MoE block ("[SGLang] LoRA + MoE fusion"), over the
 * (adapter, expert) alignment of the last lora_build_segments on `ws`.
 *   LORA_MOE_GATE_UP: d_in = hidden states bf16 [M][ld_in] (per token);
 *       d_cache = gate/up base output bf16 [M*topk][ld_cache] (per pair
 *       p = t*topk + k), updated in place before SiLU-mul (stage 1.5).  The
 *       table's A is usually shared by the experts (E_A = 1), B per expert.
 *   LORA_MOE_DOWN: d_in = SiLU-mul output bf16 [M*topk][ld_in] (per pair);
 *       d_cache = down base output bf16 [M*topk][ld_cache], updated in place
 *       before the top-k reduce (stage 3.5).  A per expert, B usually shared.
 *   d_topk_weights: NULL adds the unweighted delta (for caches the reduce
 *       weights later); else float [M*topk] multiplies each pair's delta.
 * Same alignment, error and determinism rules as lora_apply.
 */
lora_status lora_moe_delta(lora_table table, int32_t stage, const lora_workspace *ws, const void *d_in,
                           int64_t ld_in, void *d_cache, int64_t ld_cache, const float *d_topk_weights,
                           lora_stream_t stream);

/*
 * A LoRA linear layer in one kernel ("vLLM-Ascend dynamic LoRA fused
 * operator", section 3.3: the custom linear layer runs the base matmul and
 * the LoRA operator, merged into one fused operator):
 *   y[t] = x[t] W^T + scale_i (x[t] A_i^T) B_i^T   for tokens with adapter i,
 *   y[t] = x[t] W^T                                 for tokens without one,
 * over the segment table of the last lora_build_segments on `ws` (dense).
 *   d_x : bf16 [M][ldx] device, the layer input (K columns used).
 *   d_w : bf16 [N][ldw] device, the base weight (row n = output column n, K
 *         columns used; N = the table's sum of slice widths).
 *   d_y : bf16 [M][ldy] device, out: y (N columns).  It is written, not read:
 *         no base output is needed.  Rows of tokens past the last build's M
 *         are not touched.
 * The base product and S = x A_i^T accumulate in fp32 in one pass over x; S
 * is scaled and rounded once to bf16, and S B_i^T is added to the fp32
 * accumulator before the one rounding of y to bf16.
 * ldx, ldw >= K and ldy >= N, all multiples of 8; d_x, d_w and d_y 16-byte
 * aligned.  Errors (synchronous): LORA_ERR_INVALID_ARG (also a MoE table or
 * table L != ws->L), LORA_ERR_UNSUPPORTED (more than 65535 token tiles).
 * Device-side: LORA_ERR_TIMEOUT via lora_get_status.
 */
lora_status lora_linear(lora_table table, const lora_workspace *ws, const void *d_x, int64_t ldx, const void *d_w,
                        int64_t ldw, void *d_y, int64_t ldy, lora_stream_t stream);

/*
 * Embedding LoRA ("[SGLang] LoRA Layers", VocabParallelEmbeddingWithLoRA: the
 * LoRA A matrix acts as an embedding lookup over the vocabulary and B as a
 * plain matmul added to the base embedding), over the segment table of the
 * last lora_build_segments on `ws` (adapter per token):
 *   y[t] += scale_i * B_i A_i[:, vocab[t]]
 * `table`: packed with K = the vocabulary size V (a multiple of 8; A_i given as
 * [r_i][V]), one A block for all slices (n_a = 1), N = the embedding width.
 *   d_vocab : int32 [M] device, the tokens' vocabulary ids.
 *   d_y     : bf16 [M][ldy] device, in: the base embedding rows, out: + delta.
 *             Rows of tokens without an adapter are not touched.
 * Vocabulary ids outside [0, V) leave the row unchanged and raise
 * LORA_ERR_BAD_ADAPTER_ID through lora_get_status.  The LM-head LoRA of the
 * same page (hidden @ A^T @ B^T added to the logits, B cut by vocabulary for
 * a tensor-parallel shard) is lora_apply with a table of K = the hidden size
 * and N = the vocabulary (or the shard's rows of B).
 * ldy >= N, a multiple of 8; d_y 16-byte aligned.  Errors (synchronous):
 * LORA_ERR_INVALID_ARG (also n_a != 1 or a MoE table), LORA_ERR_UNSUPPORTED.
 */
lora_status lora_embedding_apply(lora_table table, const lora_workspace *ws, const int32_t *d_vocab, void *d_y,
                                 int64_t ldy, lora_stream_t stream);

/* Synchronise `stream`, read and clear the workspace's sticky device error
 * word, and return the most severe error seen since the last call (LORA_OK if
 * none). */
lora_status lora_get_status(const lora_workspace *ws, lora_stream_t stream);

const char *lora_status_string(lora_status status);

/*
 * Process-wide tuning knobs (not thread-safe against concurrent calls).
 *   LORA_OPT_PATH            : 0 auto: dense workspaces of at most 32 tokens
 *                              on the persistent engine (groups of at most
 *                              LORA_OPT_TC_MIN_ROWS rows on small 16-row tiles
 *                              with warp-level MMAs, the rest on 128-row
 *                              tcgen05 tiles), larger ones and every MoE delta
 *                              on the streaming path (64-row tiles); 1 the
 *                              engine, every group on small tiles; 2 the
 *                              engine, every group on 128-row tiles; 3 the
 *                              streaming path on 16-row tiles.
 *   LORA_OPT_TC_MIN_ROWS     : engine groups with more rows take 128-row tiles
 *                              (default 32; groups whose A block has more than
 *                              128 rows, n_a * stored rank, switch at half).
 *   LORA_OPT_WAIT_TIMEOUT_NS : limit of every in-kernel wait (default 1 s).
 *   LORA_OPT_GRID_CTAS       : grid size of the engine and of both streaming
 *                              kernels (0 = one block per SM).
 *   LORA_OPT_TEST_WITHHOLD_HANDOFF : test hook; nonzero makes the next launches
 *                              skip the shrink-to-expand hand-off (the engine
 *                              does not publish its partials, the streaming
 *                              expand never loads S), so the waits of the
 *                              expand work run out (checks the timeout path).
 *   LORA_OPT_PDL             : 1 (default) launches the one-warp segment
 *                              build (dense, at most 32 tokens), the engine
 *                              when its workspace holds at most 32 tokens
 *                              (dense) and both streaming kernels with
 *                              programmatic stream serialization: such a kernel
 *                              may be scheduled while the kernel before it on
 *                              the stream finishes, and waits on the device
 *                              (griddepcontrol) before it reads anything; 0
 *                              launches every kernel in plain stream order.
 * Returns LORA_ERR_INVALID_ARG for an unknown option or value.
 */
typedef enum {
    LORA_OPT_PATH = 0,
    LORA_OPT_TC_MIN_ROWS = 1,
    LORA_OPT_WAIT_TIMEOUT_NS = 2,
    LORA_OPT_GRID_CTAS = 3,
    LORA_OPT_TEST_WITHHOLD_HANDOFF = 4,
    LORA_OPT_PDL = 5
} lora_option;
lora_status lora_set_option(int32_t option, int64_t value);
int64_t lora_get_option(int32_t option);

/*
 * Phase tracing (off by default).  With a non-NULL device buffer, every later
 * lora_apply / lora_moe_delta launch writes uint64 %globaltimer stamps (ns,
 * 0 = phase not reached).  Persistent engine: 32 per thread block, 0 entry,
 * 24 group records loaded, 25 launch plan made, 1 work list ready, 2 first
 * shrink item started, 3..10 its pipeline stages issued (small tiles: 3 =
 * operands landed, 30 = partial computed), 11 its MMAs done, 12 its partial
 * stored, 13 it was published, 29 shrink items done, 26 first finish item
 * started, 27 its tile's partials all in, 28 its S stored, 14 first expand
 * item's tile ready, 15 its S in place, 16..23 the first four expand units
 * (operands landed, output written), 31 exit; blocks past bytes/256 are not
 * traced.  Streaming path: [kernel][block][32] with kernel 0 the shrink and 1
 * the expand, over bytes/768 blocks.  Shrink: 0 entry, 1 past its wait on
 * the kernel before, 10 and 11 the plan's two passes over the groups done,
 * 2 the block's share planned, 12..19 its first eight stages issued, 20..27
 * the same stages landed, 3..6 its first four chunks done, 8 all its chunks
 * done, 31 exit.  Expand: 0 entry, 1 the launch's tile records out, 29 the
 * shrink grid ended (the block's S sums start), 30 its S sums out, 3 every
 * block's S sums out (S loader starts), 4 first S in place, 2 the MMA issuer
 * found the first B landed, 5..8 the B of units 8..11 landed, 25..28 and their
 * accumulators free, 13..16 those units' B copies issued, 17..20 their y
 * gathers issued, 31 exit.  Pass NULL to switch tracing off.  Process-wide.
 */
lora_status lora_set_trace(void *d_trace, size_t bytes);

/*
 * One step without any caller-provided device scratch: builds the segment
 * table of d_lora_id_map (int32 [M], device) and applies the LoRA delta of
 * `table` to d_y exactly as lora_build_segments + lora_apply would.  The
 * pages have no counterpart; it exists for callers that cannot allocate
 * device memory (code running inside another allocator's arena, under a
 * no-allocation policy on a serving hot path, or in a process that only
 * receives pre-made buffers), who can still pass their inputs and outputs.
 *
 * Every byte of scratch (segment table, hand-off partials and counters) is a
 * fixed array in this library, about 32.2 MiB, that each GPU which loads the
 * library holds until the process exits.  Limits, checked before anything is
 * launched: the table's adapters L + 1 <= 16000 (the segment build's key
 * limit, else LORA_ERR_UNSUPPORTED); M <= 4096 tokens, and
 * M * R * (ceil(K / 64) + 1) + 64 * R * min(M, L) <= 2^23 partial floats,
 * where R is the table's largest A block (n_a * stored rank) and 64 the
 * shortest K-chunk the engine cuts (else LORA_ERR_WORKSPACE).  Same argument
 * rules as lora_apply (dense tables only).  The delta runs on the persistent
 * engine (the streaming path of lora_apply needs the workspace's plan area).
 *
 * The first call on a device looks the array up (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  All
 * calls share the one array and it keeps the last call's contents: the call
 * clears what must start at zero itself, and calls that overlap on the GPU
 * (different streams, or different host threads) race on it.  Device-side
 * conditions (ids out of range are left unchanged as in lora_apply; a wait
 * that ran out) are not reported by this entry point.
 */
lora_status lora_apply_static_scratch(lora_table table, const int32_t *d_lora_id_map, int32_t M, const void *d_x,
                                      int64_t ldx, void *d_y, int64_t ldy, lora_stream_t stream);

/* Stored rank for a true rank: rounded up to a multiple of 16 ("vLLM-Ascend
 * dynamic LoRA fused operator", section 4.3: 16 stays 16, 20 becomes 32).
 * Host-only; returns -1 outside 1..64. */
int32_t lora_rank_padded(int32_t rank);

#ifdef __cplusplus
}
#endif
#endif /* LORA_GB300_H */
