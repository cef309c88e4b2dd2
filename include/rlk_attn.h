/*
 * rlk_attn.h -- C ABI of librlk_attn.so: batch-invariant, split-order-
 * invariant causal GQA attention for sm_103a (GB300).
 *
 * What the library computes.  For every query row and every global KV block
 * b of its sequence, a partial state
 *     state_b = (o_b, lse_b, global_block_index = b)
 * with FP32 accumulation; the states of a row are merged in ascending
 * global_block_index order, whatever logical context-parallel (CP) rank or
 * arrival order produced them, and the result is downcast to BF16 only at the
 * final write.  Source pages:
 *   [P1] "WS2 Attention PR5 Drift Benchmark" (design doc): Scope (Qwen3-8B
 *        heads Hq=32, Hkv=8, D=128; CP sweep; full and chunked prefill; BF16
 *        path vs FP32), Transformer Engine Reuse (state tuple; sort by
 *        global_block_index, then online-softmax correction), Report Contract
 *        (merge order global_block_index, downcast_at final_write, block
 *        metadata hash).
 *   [P3] "[WS2][Attention] H100 validation and reproduction guide for #235
 *        PR1-PR8": Status (FP32 accumulation, Split-KV disabled, fixed merge
 *        order, full-KV arithmetic retained), PR stack (decode KV-cache replay,
 *        paged-KV adapter, dQ/dK/dV backward), Acceptance (Out/LSE/dQ/dK/dV
 *        max abs 0.0 across 2/4/8 ranks; fallback=false).
 *   [P4] "[WS2][Cross-config][Attention] Integrate the Qwen3-8B TP=2 CP=2
 *        BF16 Attention setting ..." (PR #263): the attention-contract knobs
 *        (reduction order, split-KV policy with its supported k values, batch
 *        size, dtype).
 *
 * Conventions (every entry point):
 *   - Tensors are packed varlen ("THD"), row-major, contiguous:
 *       q [Tq, Hq, 128] BF16, k/v [Tk, Hkv, 128] BF16,
 *       out [Tq, Hq, 128] FP32 and/or BF16, lse [Tq, Hq] FP32.
 *     Query head h reads KV head h / (Hq / Hkv).  softmax scale is given.
 *   - Device pointers are CUDA device memory of the current device, 16-byte
 *     aligned.  Arrays documented as HOST are read on the host during the
 *     call and not retained.
 *   - The caller owns every buffer (outputs, state table, workspace).  The
 *     library never allocates, frees or synchronises in these calls; work is
 *     enqueued on `stream` (NULL = legacy default stream).
 *   - Arguments are validated before anything is launched.  On failure the
 *     call returns a status, launches nothing and sets rlk_attn_last_error().
 *     There is no fallback: an unsupported shape returns RLK_ERR_UNSUPPORTED.
 *   - Faults detected on the device (a wait that timed out, a bad page id, a
 *     duplicate or missing block in a state table) set the device error word;
 *     read it with rlk_attn_check_device_error().
 *   - A batch may hold up to 2^20 sequences.  One launch's sequence tables
 *     ride in kernel parameters and take 128 sequences, so a larger batch
 *     runs as consecutive ranges of 128 sequences on `stream`, each range a
 *     complete call on its own rows (every range is validated before the
 *     first launch).  A sequence's arithmetic does not depend on the other
 *     sequences of its batch, so the results are those of one launch.
 *   - Causal masking is bottom-right aligned: query row i of a sequence with
 *     q_len queries and kv_len keys sits at key position kv_len - q_len + i
 *     (q_len <= kv_len), so chunked-prefill replay passes the chunk's queries
 *     and the KV cache up to the chunk's end.
 */
#ifndef RLK_ATTN_H
#define RLK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* rlk_stream_t; /* a cudaStream_t */

typedef enum {
  RLK_OK = 0,
  RLK_ERR_INVALID_ARGUMENT = 1,
  RLK_ERR_UNSUPPORTED = 2,
  RLK_ERR_WORKSPACE_TOO_SMALL = 3,
  RLK_ERR_DUPLICATE_BLOCK = 4,
  RLK_ERR_MISSING_BLOCK = 5,
  RLK_ERR_DEVICE_TIMEOUT = 6,
  RLK_ERR_CUDA = 7,
  RLK_ERR_BAD_PAGE = 8,
  RLK_ERR_BAD_STATE_TABLE = 9
} rlk_status;

/* Problem description shared by the entry points. */
typedef struct {
  int32_t num_seqs;      /* sequences in the batch, 1..1048576 */
  int32_t num_q_heads;   /* Hq */
  int32_t num_kv_heads;  /* Hkv, divides Hq */
  int32_t head_dim;      /* must be 128 */
  float softmax_scale;   /* e.g. 1/sqrt(128) */
  int32_t causal;        /* must be 1 */
  int32_t kv_block_size; /* global KV block size B: 64 or 128 */
  int32_t cp_size;       /* logical context-parallel ranks, 1..8 */
  int32_t cp_layout;     /* 0 = contiguous chunks, 1 = zigzag (2*cp chunks, rank r owns r and 2cp-1-r) */
} rlk_attn_params;

/*
 * One slab of the partial-state table: the states of global block `block`
 * of sequence `seq` for the query rows [row_begin, row_begin + row_count)
 * (relative to the sequence's first query row) -- exactly the rows whose
 * causal window reaches the block.  Storage, for query head h and row i:
 *     pair  = offset + h * row_count + (i - row_begin)
 *     o_b   = state_o[pair * 128 .. pair * 128 + 127]   (FP32)
 *     lse_b = state_lse[pair]                            (FP32, natural log)
 * `producer` is the logical CP rank that produced the slab (provenance).
 * [P1] Transformer Engine Reuse: state_i = (out_i, lse_i, global_block_index_i).
 */
typedef struct {
  int32_t seq;
  int32_t block;
  int32_t row_begin;
  int32_t row_count;
  int64_t offset;
  int32_t producer;
  int32_t reserved;
} rlk_attn_slab;

/*
 * Block plan (host only, no device work).  Lists the slabs that logical rank
 * `cp_rank` produces (cp_rank = -1: every rank's), in ascending (seq, block)
 * order, with storage offsets starting at `pair_base`.  Global block b of a
 * sequence holds keys [b*B, (b+1)*B) counted from the sequence's first key;
 * its producer is the rank that owns key b*B under the cp_layout partition of
 * the sequence's kv_len keys ([P3] Status: full-KV deterministic arithmetic
 * retained, so a state always covers a whole global block).
 *   cu_seqlens_q, cu_seqlens_k: HOST [num_seqs + 1], prefix sums, q_len <= kv_len.
 *   slabs: HOST output of max_slabs entries, or NULL to only count.
 *   *n_slabs, *n_pairs: slabs listed and (row, head) pairs they hold.
 * Returns RLK_ERR_INVALID_ARGUMENT for bad lengths / ranks, and
 * RLK_ERR_WORKSPACE_TOO_SMALL when max_slabs is too small (counts still set).
 */
rlk_status rlk_attn_plan_states(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                const int32_t* cu_seqlens_k, int32_t cp_rank, int64_t pair_base,
                                rlk_attn_slab* slabs, int64_t max_slabs, int64_t* n_slabs,
                                int64_t* n_pairs);

/*
 * Block-manifest hash (host only): FNV-1a 64 over (seq, block, first key,
 * last key, producer) of every global block, in ascending (seq, block)
 * order.  Two runs agree on it iff they use the same block decomposition and
 * producer assignment ([P1] Report Contract: block metadata hash).
 */
rlk_status rlk_attn_block_manifest_hash(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                        const int32_t* cu_seqlens_k, uint64_t* hash);

/*
 * Partial states of logical rank `cp_rank` (-1: all ranks): writes, for every
 * slab rlk_attn_plan_states(params, cu_seqlens_q, cu_seqlens_k, cp_rank,
 * pair_base, ...) lists, o_b and lse_b into state_o / state_lse at the
 * slab's offsets.  q, k, v: device BF16 as in the conventions;
 * cu_seqlens_q/_k: HOST.  state_o: device FP32 [>= (pair_base + n_pairs) * 128],
 * state_lse: device FP32 [>= pair_base + n_pairs].
 */
rlk_status rlk_attn_prefill_states(const rlk_attn_params* params, const void* q, const void* k,
                                   const void* v, const int32_t* cu_seqlens_q,
                                   const int32_t* cu_seqlens_k, int32_t cp_rank, int64_t pair_base,
                                   float* state_o, float* state_lse, rlk_stream_t stream);

/*
 * Canonical merge of a state table whose slabs arrive in ANY order: sorts by
 * global_block_index per (sequence, block), then folds each (row, head) left
 * to right with the canonical FP32 fold, writing out_f32 (device FP32
 * [Tq,Hq,128], nullable), out_bf16 (device BF16, nullable; not both NULL)
 * and lse (device FP32 [Tq,Hq]).  slabs: DEVICE array of n_slabs entries
 * (e.g. several ranks' plans concatenated in any order), offsets into
 * state_o / state_lse.  n_state_pairs: the number of (row, head) pairs the
 * table holds (state_o: device FP32 [n_state_pairs, 128], state_lse: device
 * FP32 [n_state_pairs]).  workspace: device, >= rlk_attn_workspace_size(...,
 * RLK_OP_MERGE, ...) bytes.  Every block of every row must be present exactly
 * once: a duplicate sets RLK_ERR_DUPLICATE_BLOCK, a missing one
 * RLK_ERR_MISSING_BLOCK (and NaN rows) on the device error word.  A slab
 * whose rows do not fit the table (offset + Hq * row_count > n_state_pairs),
 * or whose sequence, block or row range disagrees with cu_seqlens, is not
 * read: it sets RLK_ERR_BAD_STATE_TABLE, and its block then counts as
 * missing.
 * [P1] Transformer Engine Reuse; the drift-class table (merge_order_probe:
 * reversed arrival equals the sorted merge).
 */
rlk_status rlk_attn_merge_states(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                 const int32_t* cu_seqlens_k, const rlk_attn_slab* slabs,
                                 int64_t n_slabs, const float* state_o, const float* state_lse,
                                 int64_t n_state_pairs, float* out_f32, void* out_bf16, float* lse,
                                 void* workspace, size_t workspace_bytes, rlk_stream_t stream);

/*
 * Fused causal prefill (full or chunked replay): for each query row, the
 * block states of blocks 0..last are computed and folded on chip in
 * ascending order -- bit-identical to rlk_attn_prefill_states followed by
 * rlk_attn_merge_states.  cp_rank >= 0 computes only the query rows that
 * logical rank owns under the cp_layout partition of each sequence's q_len
 * rows (other rows are left untouched); -1 computes every row.  Outputs as
 * in rlk_attn_merge_states.  cu_seqlens_q/_k: HOST.
 * [P1] Scope: full prefill and chunked-prefill replay; [P3] Acceptance.
 */
rlk_status rlk_attn_prefill(const rlk_attn_params* params, const void* q, const void* k,
                            const void* v, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int32_t cp_rank, float* out_f32, void* out_bf16, float* lse,
                            rlk_stream_t stream);

/*
 * rlk_attn_prefill with the queries' RoPE applied by the call: q is the
 * PRE-RoPE query (left unchanged); each query row is rotated at its absolute
 * position kv_len - q_len + i (the sequence's token index) in the FP32 form
 * of rlk_attn_rope, so the result is bit-identical to rlk_attn_rope on q
 * followed by rlk_attn_prefill.  k is post-RoPE, as stored in a KV cache.
 * With cp_rank -1 one pass writes the rotated rows into the output buffer
 * (out_bf16 if given, else the first half of each out_f32 row), each row into
 * its own (token, head) slot, and the prefill reads them from there before it
 * overwrites the slot with the result; with cp_rank >= 0 the kernel rotates
 * each tile in shared memory after it lands (the other rows of the buffer
 * belong to the other ranks' calls).  The outputs must not overlap q, k or v.
 *   rope_table: device FP32 [rope_max_pos][128] from rlk_attn_rope_table;
 *   every sequence with queries needs kv_len <= rope_max_pos.
 * Other arguments and outputs as in rlk_attn_prefill.
 * [P1] Scope: optional RoPE composition before Attention (CP attention still
 * consumes post-RoPE Q/K); [P3] PR stack: cache/position/RoPE identity.
 */
rlk_status rlk_attn_prefill_rope(const rlk_attn_params* params, const void* q, const void* k,
                                 const void* v, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                 int32_t cp_rank, const float* rope_table, int32_t rope_max_pos,
                                 float* out_f32, void* out_bf16, float* lse, rlk_stream_t stream);

/*
 * Paged-KV decode: one query token per sequence, at the last position of its
 * context, against keys stored in pages of page_size tokens:
 *   q: device BF16 [num_seqs, Hq, 128]
 *   k_pool, v_pool: device BF16 [n_pages, page_size, Hkv, 128]
 *   page_table: device int32 [num_seqs, max_pages]; key t of sequence s is
 *     slot t % page_size of page page_table[s * max_pages + t / page_size]
 *   seqlens: HOST int32 [num_seqs], context lengths, 1 .. max_pages*page_size
 *   out_f32 / out_bf16 / lse: device, [num_seqs, Hq, 128] / [num_seqs, Hq].
 * page_size must divide kv_block_size and be >= 8: page_size-token pages
 * are addressing only; the arithmetic blocks are the same kv_block_size
 * global blocks as prefill, so the result equals the last row of the
 * equivalent full prefill bit for bit.  A page id outside [0, n_pages) is
 * read as zeros and sets RLK_ERR_BAD_PAGE on the device error word.
 * [P3] PR stack: decode KV-cache replay, paged-KV adapter; Acceptance.
 */
rlk_status rlk_attn_decode_paged(const rlk_attn_params* params, const void* q, const void* k_pool,
                                 const void* v_pool, int32_t n_pages, int32_t page_size,
                                 const int32_t* page_table, int32_t max_pages,
                                 const int32_t* seqlens, float* out_f32, void* out_bf16, float* lse,
                                 rlk_stream_t stream);

/*
 * RoPE table for rlk_attn_rope and rlk_attn_decode_paged_rope (host only):
 * table[p * 128 + i] = (float)cos(p * theta^(-2i/128)) and
 * table[p * 128 + 64 + i] = (float)sin(...) for p < max_pos, i < 64, the
 * angle in double and rounded once.  The caller copies it to the device.
 *   theta: base, finite and > 1 (Qwen3: 1e6); table: HOST, max_pos * 128 floats.
 * RLK_ERR_INVALID_ARGUMENT for theta <= 1, max_pos < 1 or a NULL table.
 * [P1] Scope: optional RoPE composition before Attention.
 */
rlk_status rlk_attn_rope_table(double theta, int32_t max_pos, float* table);

/*
 * Rotary position embedding of packed BF16 rows, rotate-half convention
 * (pairs (i, i + 64) of the 128 dimensions), in the one FP32 form every
 * RoPE path of the library uses:
 *   y_i      = bf16_rn(fmaf(x_i, c, -(x_{i+64} * s)))
 *   y_{i+64} = bf16_rn(fmaf(x_{i+64}, c, x_i * s))     (products rounded to FP32)
 * with c, s the table's entries at the row's position -- so a row's result
 * depends only on its values and its position (cache / position / RoPE
 * identity between prefill, chunked replay and decode).
 *   x, y: device BF16 [T, num_heads, 128], T = cu_seqlens[num_seqs]; y may
 *     equal x (in place) but must not otherwise overlap it;
 *   cu_seqlens: HOST [num_seqs + 1]; pos_offset: HOST [num_seqs] or NULL
 *     (0): row i of sequence s is at position pos_offset[s] + i (a chunk of
 *     q_len queries over a cache of kv_len keys: kv_len - q_len);
 *   table: device, from rlk_attn_rope_table, max_pos positions.
 * Only params->num_seqs and head_dim are read.  Every position must be
 * < max_pos (RLK_ERR_INVALID_ARGUMENT otherwise, before any launch).
 * [P1] Scope: RoPE before Attention, Attention consuming post-RoPE Q/K.
 */
rlk_status rlk_attn_rope(const rlk_attn_params* params, const void* x, void* y, int32_t num_heads,
                         const int32_t* cu_seqlens, const int32_t* pos_offset, const float* table,
                         int32_t max_pos, rlk_stream_t stream);

/*
 * rlk_attn_rope over the queries and keys of the same tokens in one launch:
 * q [T, Hq, 128] -> q_out and k [T, Hkv, 128] -> k_out (BF16, device; an
 * output may equal its input), Hq and Hkv from params, every token of
 * sequence s at position pos_offset[s] + its index (pos_offset HOST or
 * NULL).  Bit-identical to rlk_attn_rope on q and on k.
 * [P1] Scope: RoPE composed before Attention; [P3] PR stack:
 * cache/position/RoPE identity.
 */
rlk_status rlk_attn_rope_qk(const rlk_attn_params* params, const void* q, void* q_out, const void* k,
                            void* k_out, const int32_t* cu_seqlens, const int32_t* pos_offset,
                            const float* table, int32_t max_pos, rlk_stream_t stream);

/*
 * rlk_attn_decode_paged with the query's RoPE applied inside the decode
 * kernel: q holds the pre-RoPE query of each sequence, rotated at position
 * seqlens[s] - 1 right after it lands in shared memory (the form of
 * rlk_attn_rope, so the result equals rlk_attn_rope + rlk_attn_decode_paged
 * bit for bit); the pools hold post-RoPE K (rotated once, when the token
 * entered the cache) and V.
 *   rope_table: device, from rlk_attn_rope_table, rope_max_pos positions
 *     (every seqlens[s] <= rope_max_pos).
 * Needs kv_block_size 128 and at most 8 query heads per KV head
 * (RLK_ERR_UNSUPPORTED otherwise).
 * [P3] PR stack: decode KV-cache replay and cache/position/RoPE identity.
 */
rlk_status rlk_attn_decode_paged_rope(const rlk_attn_params* params, const void* q, const void* k_pool,
                                      const void* v_pool, int32_t n_pages, int32_t page_size,
                                      const int32_t* page_table, int32_t max_pages,
                                      const int32_t* seqlens, const float* rope_table,
                                      int32_t rope_max_pos, float* out_f32, void* out_bf16,
                                      float* lse, rlk_stream_t stream);

/*
 * Paged-KV decode with each (sequence, KV head)'s KV blocks split over
 * split_k fixed work items that different SMs process.  Every item writes
 * the block states (o_b, lse_b) of its blocks to a state table in the
 * workspace, and each (sequence, query head) is folded in ascending block
 * order with the canonical fold.  Two schedules, with the same bits:
 *   - when the num_seqs * num_kv_heads * split_k items and the fold CTAs
 *     (one warp per (sequence, query head), 16 a CTA) fit on the device at
 *     once (one CTA per SM), item r takes the blocks b = r (mod split_k) and
 *     the whole call is one cooperative launch whose fold CTAs, on SMs the
 *     items leave free, fold the states as the items write them (the fold
 *     hides behind the producers).  Each item first marks its table slots
 *     unwritten and then sets its flag in the workspace to a value new to
 *     the call; inside a CUDA graph capture a fill of the table precedes
 *     the launch instead (a replay repeats the launch's arguments);
 *   - otherwise item r takes the contiguous blocks floor(r*nb/k) up to
 *     floor((r+1)*nb/k) (nb = the sequence's blocks) and a second kernel
 *     folds the table.
 * The arithmetic is the single-pass decode's step for step, so the result
 * equals rlk_attn_decode_paged (and the last row of the equivalent prefill)
 * bit for bit whatever split_k; it spreads few long sequences over all SMs.
 *   Arguments as rlk_attn_decode_paged, plus
 *   split_k: 1 .. 64 items per (sequence, KV head), or 0 to let the library
 *     pick k from the context lengths and the SM count (few pairs: the
 *     largest k whose items fit on the device at once, with the fold on
 *     chip; otherwise a model of the busiest SM's blocks plus the fold; k = 1
 *     runs the single-pass decode) -- the result is the same for every k;
 *   workspace: device, >= rlk_attn_workspace_size(params,
 *     RLK_OP_DECODE_SPLIT, NULL, seqlens) bytes (the state table: 516 bytes
 *     per (sequence, block, query head), rounded up to 256, then 512 bytes
 *     of item flags per (sequence, KV head)); its contents need no
 *     initialisation, and calls on one workspace must not overlap.
 * Needs kv_block_size 128 and at most 8 query heads per KV head
 * (RLK_ERR_UNSUPPORTED otherwise).
 * [P3] PR stack: decode KV-cache replay; Status: fixed global_block_index
 * merge; [P4] split-KV policy as an explicit, fixed knob.
 */
rlk_status rlk_attn_decode_paged_splitk(const rlk_attn_params* params, const void* q, const void* k_pool,
                                        const void* v_pool, int32_t n_pages, int32_t page_size,
                                        const int32_t* page_table, int32_t max_pages,
                                        const int32_t* seqlens, int32_t split_k, float* out_f32,
                                        void* out_bf16, float* lse, void* workspace,
                                        size_t workspace_bytes, rlk_stream_t stream);

/*
 * rlk_attn_decode_paged_splitk with the query's RoPE applied inside the
 * decode kernel, as in rlk_attn_decode_paged_rope (q pre-RoPE, rotated at
 * position seqlens[s] - 1; the pools hold post-RoPE K): the result equals
 * rlk_attn_decode_paged_rope bit for bit whatever split_k.
 *   rope_table, rope_max_pos: as for rlk_attn_decode_paged_rope (NULL table:
 *     RLK_ERR_INVALID_ARGUMENT); the other arguments as for
 *     rlk_attn_decode_paged_splitk.
 * [P3] PR stack: decode KV-cache replay and cache/position/RoPE identity;
 * [P4] split-KV policy as an explicit, fixed knob.
 */
rlk_status rlk_attn_decode_paged_splitk_rope(const rlk_attn_params* params, const void* q, const void* k_pool,
                                             const void* v_pool, int32_t n_pages, int32_t page_size,
                                             const int32_t* page_table, int32_t max_pages,
                                             const int32_t* seqlens, int32_t split_k, const float* rope_table,
                                             int32_t rope_max_pos, float* out_f32, void* out_bf16,
                                             float* lse, void* workspace, size_t workspace_bytes,
                                             rlk_stream_t stream);

/*
 * The split factor rlk_attn_decode_paged_splitk uses for split_k == 0 on a
 * device with num_sms SMs (host only, no device work): 1 .. 64, or -1 for
 * invalid params, a NULL seqlens, a context length < 1 or num_sms < 1.
 *   seqlens: HOST [num_seqs] context lengths.
 * [P4] split-KV policy as an explicit, fixed knob.
 */
int32_t rlk_attn_decode_auto_split(const rlk_attn_params* params, const int32_t* seqlens, int32_t num_sms);

/*
 * Deterministic backward of causal prefill (q_len == kv_len per sequence):
 *   q, k, v, dout: device BF16; out_f32: device FP32 forward output;
 *   lse: device FP32 forward lse; cu_seqlens: HOST [num_seqs + 1];
 *   dq [Tq,Hq,128], dk, dv [Tk,Hkv,128]: device FP32 outputs.
 * Delta_i = sum_d dout_id * out_id; P = exp(S - lse); dS = P (dP - Delta).
 * dK/dV of a KV block accumulate over query blocks in ascending order, and
 * within a query block over the Hq/Hkv query heads of the group in ascending
 * order; dQ accumulates over KV blocks in ascending order; no atomics.
 * cp_rank >= 0 computes the dK/dV rows of the KV blocks that rank produces
 * and the dQ rows it owns (other rows untouched); -1 computes all.
 * workspace: device, >= rlk_attn_workspace_size(..., RLK_OP_BACKWARD, ...).
 * [P1] Scope: optional backward dq, dk, dv; [P3] Acceptance: dQ/dK/dV max
 * abs 0.0 across ranks.
 */
rlk_status rlk_attn_backward(const rlk_attn_params* params, const void* q, const void* k,
                             const void* v, const float* out_f32, const void* dout,
                             const float* lse, const int32_t* cu_seqlens, int32_t cp_rank,
                             float* dq, float* dk, float* dv, void* workspace,
                             size_t workspace_bytes, rlk_stream_t stream);

/*
 * rlk_attn_merge_states without a workspace, for callers that cannot
 * allocate device memory -- for instance code that runs inside a CUDA graph
 * being captured, under an allocator that must not grow, or behind an API
 * that hands out only its input and output buffers.  The pages have no
 * counterpart: this is a convenience of this library.
 *   Arguments, results and device errors are those of rlk_attn_merge_states;
 *   the caller still passes the state table and the outputs.
 *   Scratch: the (sequence, block) index lives in a file-scope device array
 *   of 65,536 int32 entries (256 KB) that every GPU loading the library
 *   holds until the process exits.  num_seqs times the largest number of KV
 *   blocks of a sequence must not exceed 65,536; larger problems return
 *   RLK_ERR_UNSUPPORTED with a message.  Nothing is allocated or freed.
 *   The first call of any entry point on a device sets the library up
 *   there (with that device current), which includes looking up the array's
 *   device address; make that first call before any stream capture.
 *   Every call reuses the same array and initialises it itself, so calls in
 *   sequence are independent, but calls that overlap on the GPU (different
 *   streams, or different host threads on one device) race on it.
 */
rlk_status rlk_attn_merge_states_noalloc(const rlk_attn_params* params, const int32_t* cu_seqlens_q,
                                         const int32_t* cu_seqlens_k, const rlk_attn_slab* slabs,
                                         int64_t n_slabs, const float* state_o, const float* state_lse,
                                         int64_t n_state_pairs, float* out_f32, void* out_bf16, float* lse,
                                         rlk_stream_t stream);

enum { RLK_OP_MERGE = 1, RLK_OP_BACKWARD = 2, RLK_OP_DECODE_SPLIT = 3 };

/* Workspace bytes an entry point needs (HOST cu_seqlens; 0 on bad input).
 * RLK_OP_DECODE_SPLIT takes the decode context lengths (seqlens) as
 * cu_seqlens_k and ignores cu_seqlens_q. */
size_t rlk_attn_workspace_size(const rlk_attn_params* params, int32_t op,
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k);

/* Synchronises `stream`, reads and clears the device error word of the
 * current device; returns RLK_OK or the status of the first fault class. */
rlk_status rlk_attn_check_device_error(rlk_stream_t stream);

/*
 * Diagnostic of the failure-detection path: launches one warp that waits on
 * a barrier nothing completes, through the bounded wait every kernel uses
 * (limit 1 s); the kernel then records a device timeout (site 0x7e1) in the
 * error word and returns, so the next rlk_attn_check_device_error on the
 * stream reports RLK_ERR_DEVICE_TIMEOUT and clears the word.  No fault, no
 * trap: the context stays usable.  Returns the launch status.
 */
rlk_status rlk_attn_selftest_wait_timeout(rlk_stream_t stream);

/* Message of the last failing call on this thread ("" if none). */
const char* rlk_attn_last_error(void);

/* Provenance of the arithmetic core and merge order. */
const char* rlk_attn_core_id(void);

#ifdef __cplusplus
}
#endif

#endif /* RLK_ATTN_H */
