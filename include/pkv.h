/*
 * pkv.h - C ABI of the paged-KV attention library (GB300, sm_103a).
 *
 * The operations follow the paged-KV rollout engine described in the
 * scripts/benchmarks commit log ("Why this works": one contiguous page pool
 * plus a page table mapping (sequence, logical block) -> physical page;
 * "Files": new K/V rows are written in-kernel to their physical slot before
 * attention reads them) and the varlen interface of the cb_sync_driver.py
 * commit message (phase-2 fixes: cu_seq_lens_q on every paged forward) and
 * the README "Integration notes" (max_seqlen_q / max_seqlen_k).  The sliding
 * window rule (causal AND q_pos - kv_pos < window, strict) is the Gemma-4
 * sliding-window commit of the same log.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller; the
 *   library never allocates, frees, synchronises the host, or keeps a
 *   pointer after returning.  Work is enqueued on `stream` (a cudaStream_t
 *   passed as void*; NULL = legacy default stream) and runs asynchronously.
 * - bf16 means IEEE bfloat16 (2 bytes).  Every tensor is dense and
 *   row-major (C order) with the shape given below.
 * - Page pools: k_cache and v_cache are separate tensors of shape
 *   [num_pages, num_kv_heads, page_size, head_dim] bf16.  Token position p
 *   of a sequence with block-table row T lives in page T[p / page_size],
 *   row p % page_size.  A slot is page * page_size + row.
 * - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 * - Supported shapes of the attention calls: head_dim in {64, 128, 256,
 *   512} (paged_attn_decode_shared_prefix and paged_attn_mixed: see there);
 *   page_size a multiple of 16 (decode tests use 16 and 64, varlen tests 16
 *   to 256), and for varlen a divisor or a multiple of its key tile (128
 *   keys for head_dim 64 and 128, 64 for 256, 32 for 512); num_q_heads a
 *   multiple of num_kv_heads with a group of at most 8 for decode and
 *   dividing 128 for varlen; decode batch <= 4096 and varlen batch <= 1024
 *   (their schedules live in shared memory; varlen at head_dim 512, whose
 *   Q tile takes 128 KB of it, up to 64).
 *   Anything else returns PKV_ERR_UNSUPPORTED.  The append calls take any
 *   page_size >= 1; paged_kv_append any head_dim that is a multiple of 8,
 *   paged_kv_append_rope head_dim in {64, 128, 256}.
 * - Host-detectable argument errors return PKV_ERR_INVALID before anything
 *   is enqueued.  CUDA launch errors return PKV_ERR_CUDA (message from
 *   pkv_last_cuda_error()).
 * - Data-dependent errors never fault and never trap: the offending row or
 *   page is skipped (masked out) and, if `err_flag` is non-NULL, the bits
 *   below are OR-ed into that device int32.  The caller clears it.
 * - Base pointers must be 16-byte aligned (k_cache/v_cache/q/out/k_new/
 *   v_new); otherwise PKV_ERR_INVALID.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID = 1,     /* bad argument detected on the host; nothing enqueued */
  PKV_ERR_UNSUPPORTED = 2, /* well-formed but outside the supported shapes */
  PKV_ERR_CUDA = 3         /* a CUDA runtime/driver call failed */
} pkv_status;

/* Bits OR-ed into *err_flag by the kernels. */
#define PKV_DEVERR_SLOT    1  /* slot >= num_pages*page_size: that row was not written */
#define PKV_DEVERR_PAGE    2  /* block-table entry outside [0, num_pages): its keys masked */
#define PKV_DEVERR_LEN     4  /* a length exceeded max_blocks_per_seq*page_size or the
                                 declared maximum: clamped */
#define PKV_DEVERR_TIMEOUT 8  /* an internal pipeline wait gave up (never expected) */
#define PKV_DEVERR_POS     16 /* a position outside [0, max_position) of the rotary
                                 table: that token was skipped */

/*
 * paged_kv_append - scatter this step's new K/V rows into the page pools.
 *
 * Source: scripts/benchmarks commit log, "Files" paragraph of the flex
 * paged-KV engine commit (in-kernel k_cache[addr] = k_val write of each new
 * row to its physical address; one reserved no-op slot for padded rows).
 *
 *   k_new, v_new   [num_tokens, num_kv_heads, head_dim] bf16 (read)
 *   k_cache,v_cache[num_pages, num_kv_heads, page_size, head_dim] bf16 (written)
 *   slot_mapping   [num_tokens] int64: destination slot of row t; a negative
 *                  slot means "skip this row" (padding)
 *
 * Rows are copied bit-exactly.  Slots must be distinct within one call
 * (duplicates race; the winner is unspecified).  num_tokens == 0 is a no-op.
 * num_tokens * num_kv_heads * head_dim / 8 must be below 2^31 (else
 * PKV_ERR_UNSUPPORTED).
 */
pkv_status paged_kv_append(const void* k_new, const void* v_new,
                           void* k_cache, void* v_cache,
                           const int64_t* slot_mapping, int32_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim,
                           int32_t page_size, int64_t num_pages,
                           int32_t* err_flag, void* stream);

/*
 * paged_attn_decode_workspace_size - bytes of device scratch that
 * paged_attn_decode needs for this batch shape (on the current device).
 */
size_t paged_attn_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim);

/*
 * paged_attn_decode - one query token per sequence attends its whole paged
 * prefix (the decode step of the rollout engine: scripts/benchmarks commit
 * log, "Why this works", page-table routing of every decode query).
 *
 *   out          [batch, num_q_heads, head_dim] bf16 (written)
 *   q            [batch, num_q_heads, head_dim] bf16
 *   block_table  [batch, max_blocks_per_seq] int32 physical page ids;
 *                entries past ceil(seq_len/page_size) are never read
 *   seq_lens     [batch] int32: keys of sequence b (its new token included,
 *                i.e. append first); the query sits at position seq_len-1.
 *                seq_len 0 gives a zero output row.
 *   scale        multiplier of q.k (typically 1/sqrt(head_dim))
 *   window       > 0: only keys with (seq_len-1) - pos < window are read;
 *                <= 0: no window
 *   max_seq_len  an upper bound on seq_lens (sizes the launch; larger
 *                lengths are clamped to max_blocks_per_seq*page_size and
 *                flagged)
 *   workspace    device scratch of paged_attn_decode_workspace_size() bytes,
 *                256-byte aligned.  Zero-fill it once before its first use
 *                (e.g. cudaMemsetAsync); every call leaves it zero-filled
 *                again, so it can be reused by later calls in stream order.
 *                A workspace may be shared by calls with the same head
 *                shapes and any batch up to the one it was sized for.
 *                Calls that overlap on the GPU need separate workspaces.
 *                After a call that raised PKV_DEVERR_TIMEOUT, zero it again.
 *
 * One persistent kernel launch: one CTA per SM takes (sequence, kv head)
 * segments from a longest-first queue kept in the workspace; a segment
 * longer than half of a CTA's fair share is cut into chunks whose partial
 * outputs are merged (log-sum-exp weights) by whichever CTA delivers the
 * last chunk, found with an arrival counter kept in the workspace.
 */
pkv_status paged_attn_decode(void* out, const void* q,
                             const void* k_cache, const void* v_cache,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, int32_t batch,
                             int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t page_size, int64_t num_pages,
                             int32_t max_seq_len, float scale, int32_t window,
                             void* workspace, size_t workspace_bytes,
                             int32_t* err_flag, void* stream);

/*
 * paged_attn_decode_append - the decode step with its append fused in: the
 * same result as paged_kv_append of each sequence's newest token (slot =
 * block_table[b][(seq_lens[b]-1) / page_size] * page_size +
 * (seq_lens[b]-1) % page_size) followed by paged_attn_decode, in one launch
 * (the decode step of the rollout engine: scripts/benchmarks commit log,
 * "Files", the in-kernel k_cache[addr] = k_val write, and "Why this works").
 *
 *   k_new, v_new  [batch, num_kv_heads, head_dim] bf16: sequence b's new
 *                 token (read), 16-byte aligned
 *   k_cache, v_cache  the pools, written at each sequence's position
 *                 seq_lens[b]-1 (a sequence of length 0 writes nothing)
 *   every other argument as paged_attn_decode (same workspace).
 *
 * The row is written by the CTA that reads the tile holding that position,
 * before its TMA copies of the tile; no other work of the call reads it.
 * An out-of-range page id of that position skips the write and raises
 * PKV_DEVERR_PAGE.
 */
pkv_status paged_attn_decode_append(void* out, const void* q, const void* k_new,
                                    const void* v_new, void* k_cache, void* v_cache,
                                    const int32_t* block_table, int32_t max_blocks_per_seq,
                                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                    int64_t num_pages, int32_t max_seq_len, float scale,
                                    int32_t window, void* workspace, size_t workspace_bytes,
                                    int32_t* err_flag, void* stream);

/*
 * paged_attn_decode_shared_prefix - paged_attn_decode for batches whose
 * sequences come in groups that share their leading pages (cascade
 * decode).  Source: the grpo_equivalence page (num_generations = 4
 * completions decoded per prompt) and the flex paged-KV engine's page
 * table of the scripts/benchmarks commit log (block tables may point at the
 * same physical pages).
 *
 * Sequences b = j*group_size .. j*group_size + group_size - 1 (the last
 * group may be shorter) form group j.  prefix_lens [ceil(batch /
 * group_size)] int32 (device): the group's shared prefix in keys, a
 * multiple of page_size; the first prefix_lens[j] / page_size block-table
 * entries of every member of group j must be the same pages (the caller's
 * contract; not checked).  0 means no sharing.  A length that is negative,
 * not a multiple of page_size or longer than a block-table row is treated
 * as 0 and flagged PKV_DEVERR_LEN.
 *
 * The result is paged_attn_decode's (every query attends all of its keys,
 * full causal attention: there is no window argument), computed in two
 * launches on `stream`: a prefix pass reads each group's prefix pages once
 * per kv head for the query rows of all members whose length exceeds the
 * prefix, then the split-KV decode reads only those members' suffixes and
 * merges them with the prefix partials (log-sum-exp weights).  Members no
 * longer than their prefix are decoded whole.
 *
 *   workspace  paged_attn_decode_shared_prefix_workspace_size() bytes,
 *              256-byte aligned, zero-filled before its first use, with the
 *              reuse rules of paged_attn_decode's workspace.
 * Limits: head_dim in {64, 128, 256}; group_size * num_q_heads /
 * num_kv_heads query rows per group and kv head at most 32 (head_dim 64),
 * 16 (128) or 8 (256); else PKV_ERR_UNSUPPORTED.
 */
size_t paged_attn_decode_shared_prefix_workspace_size(int32_t batch, int32_t num_q_heads,
                                                      int32_t num_kv_heads, int32_t head_dim);
pkv_status paged_attn_decode_shared_prefix(void* out, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_table,
                                           int32_t max_blocks_per_seq,
                                           const int32_t* seq_lens, int32_t batch,
                                           int32_t group_size, const int32_t* prefix_lens,
                                           int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t page_size,
                                           int64_t num_pages, int32_t max_seq_len, float scale,
                                           void* workspace, size_t workspace_bytes,
                                           int32_t* err_flag, void* stream);

/*
 * paged_attn_varlen - packed variable-length attention over the paged cache
 * (prefill chunks of the continuous-batching step).  Source: the
 * cb_sync_driver.py commit message (cu_seq_lens_q on every paged forward),
 * README "Integration notes" (max_seqlen_q / max_seqlen_k), and the
 * document-causal / sliding-window masks of the scripts/benchmarks log.
 *
 *   out            [total_q, num_q_heads, head_dim] bf16 (written)
 *   q              [total_q, num_q_heads, head_dim] bf16
 *   cu_seq_lens_q  [batch+1] int32, non-decreasing, cu_seq_lens_q[0] = 0,
 *                  cu_seq_lens_q[batch] = total_q
 *   cu_seq_lens_k  [batch+1] int32: k_len of chunk b is
 *                  cu_seq_lens_k[b+1]-cu_seq_lens_k[b] (cached prefix plus
 *                  the chunk, already appended) and must be >= its q_len
 *   block_table    [batch, max_blocks_per_seq] int32
 *   max_seqlen_q, max_seqlen_k  upper bounds of q_len / k_len (size the
 *                  launch; longer chunks are clamped and flagged)
 *   scale          >= 0 (negative or NaN: PKV_ERR_INVALID)
 *   causal         1: query i of a chunk sits at position k_len - q_len + i
 *                  (bottom-right) and sees keys <= its position;
 *                  0: every key of the chunk (window must then be <= 0)
 *   window         > 0 (causal only): also require q_pos - k_pos < window
 *
 * Runs QK^T and PV on the tcgen05 tensor cores with TMEM accumulators in
 * one persistent launch (one CTA per SM).  Limits: batch <= 1024 chunks;
 * page_size as above, else PKV_ERR_UNSUPPORTED.
 */
pkv_status paged_attn_varlen(void* out, const void* q,
                             const void* k_cache, const void* v_cache,
                             const int32_t* cu_seq_lens_q, const int32_t* cu_seq_lens_k,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             int32_t batch, int32_t max_seqlen_q, int32_t max_seqlen_k,
                             int32_t total_q,
                             int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t page_size, int64_t num_pages,
                             float scale, int32_t causal, int32_t window,
                             int32_t* err_flag, void* stream);

/*
 * paged_attn_mixed - the attention of one continuous-batching step in a
 * single persistent launch: decode rows (as paged_attn_decode) and causal
 * prefill chunks (as paged_attn_varlen with causal = 1) over the same page
 * pools.  Source: scripts/benchmarks commit log, batch-sweep commit (vLLM's
 * chunked prefill packs a step's prefill and decode into the same kernels);
 * README, "Why continuous batching is still slower than vLLM on this
 * workload" (separate prefill and decode passes per step).
 *
 *   dec_*        the decode half, meaning as paged_attn_decode (dec_batch 0:
 *                no decode rows)
 *   pre_*, cu_seq_lens_q/k, max_seqlen_q/k, total_q
 *                the prefill half, meaning as paged_attn_varlen (pre_batch
 *                or total_q 0: no prefill)
 *   window       applies to both halves (<= 0: none)
 *   decode_ctas  CTAs (one per SM) that start with decode while the others
 *                run the prefill; those join the decode queue when their
 *                prefill work is done.  <= 0: chosen from the shapes.
 *   workspace    as paged_attn_decode, for dec_batch rows
 *                (paged_attn_decode_workspace_size(dec_batch, ...) bytes)
 *
 * Results equal those of the two separate calls (decode may differ in
 * rounding with the split, like paged_attn_decode between batch shapes).
 * Supported: head_dim 128, the decode and prefill limits of the separate
 * calls (group <= 8 dividing 128, page_size a divisor or multiple of 128,
 * pre_batch <= 1024); else PKV_ERR_UNSUPPORTED.  The prefill half must not
 * write rows that the decode half reads (distinct out tensors).
 */
pkv_status paged_attn_mixed(void* dec_out, const void* dec_q,
                            const int32_t* dec_block_table, int32_t dec_max_blocks_per_seq,
                            const int32_t* dec_seq_lens, int32_t dec_batch,
                            int32_t dec_max_seq_len,
                            void* pre_out, const void* pre_q,
                            const int32_t* cu_seq_lens_q, const int32_t* cu_seq_lens_k,
                            const int32_t* pre_block_table, int32_t pre_max_blocks_per_seq,
                            int32_t pre_batch, int32_t max_seqlen_q, int32_t max_seqlen_k,
                            int32_t total_q,
                            const void* k_cache, const void* v_cache,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t page_size, int64_t num_pages, float scale, int32_t window,
                            int32_t decode_ctas, void* workspace, size_t workspace_bytes,
                            int32_t* err_flag, void* stream);

/*
 * paged_attn_mixed_append - paged_attn_mixed with the step's append fused
 * in: the same result as paged_kv_append(k_new, v_new, slot_mapping)
 * followed by paged_attn_mixed, in one launch (the engine's in-kernel
 * k_cache[addr] = k_val write: scripts/benchmarks commit log, "Files").
 *
 *   k_new, v_new    [num_new_tokens, num_kv_heads, head_dim] bf16 (read),
 *                   16-byte aligned: the step's new rows (decode rows' and
 *                   prefill chunks' tokens alike)
 *   slot_mapping    [num_new_tokens] int64 (device): page * page_size + row;
 *                   negative: skip; past the pool: skipped, PKV_DEVERR_SLOT
 *   k_cache, v_cache  the pools, written at the slots, then read
 *   workspace       required whenever num_new_tokens > 0 (the launch's grid
 *                   barrier keeps two counters in it), at least
 *                   paged_attn_decode_workspace_size(dec_batch, ...) bytes
 *   every other argument as paged_attn_mixed.
 *
 * Every CTA of the launch appends a slice of the rows, then all CTAs meet
 * at a grid barrier (one CTA per SM, all resident; a wait that does not
 * end within 2 s raises PKV_DEVERR_TIMEOUT) before any of them reads a
 * pool.  Slots must be distinct, as for paged_kv_append.
 */
pkv_status paged_attn_mixed_append(
    void* dec_out, const void* dec_q, const int32_t* dec_block_table,
    int32_t dec_max_blocks_per_seq, const int32_t* dec_seq_lens, int32_t dec_batch,
    int32_t dec_max_seq_len, void* pre_out, const void* pre_q, const int32_t* cu_seq_lens_q,
    const int32_t* cu_seq_lens_k, const int32_t* pre_block_table, int32_t pre_max_blocks_per_seq,
    int32_t pre_batch, int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t total_q,
    const void* k_new, const void* v_new, const int64_t* slot_mapping, int32_t num_new_tokens,
    void* k_cache, void* v_cache, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t page_size, int64_t num_pages, float scale, int32_t window, int32_t decode_ctas,
    void* workspace, size_t workspace_bytes, int32_t* err_flag, void* stream);

/*
 * paged_attn_decode_static - paged_attn_decode for callers that cannot
 * allocate device memory.  (Not an operation of the pages: it exists for
 * callers of this library that may not call cudaMalloc on the attention
 * path -- an engine that has already given all free HBM to its KV page
 * pool, or a plugin host that hands a kernel only its inputs and outputs.)
 *
 * Same arguments, semantics and results as paged_attn_decode, minus the
 * workspace: the scratch lives in one fixed 8 MiB (8388608-byte) array of
 * device memory inside the library, which a device holds from the time the
 * array is placed there (below) until the process exits.  A batch whose
 * paged_attn_decode_workspace_size() exceeds 8 MiB is rejected with
 * PKV_ERR_UNSUPPORTED (message in pkv_last_cuda_error()).
 *
 * CUDA places the array on a device when the library's module holding it
 * is loaded there: under the default lazy module loading that is the
 * first call of this entry point on the device, which also looks up the
 * array's device address (once per device and CUDA context, with that
 * device current).  Make that first call before handing the remaining free
 * HBM to a page pool, and before any stream capture.  All host-side checks
 * run first: a rejected call enqueues nothing.  Every accepted call clears
 * the array's arrival counters on `stream` before its kernel runs.  All
 * calls share the one array: calls whose work may overlap on the GPU
 * (different streams or host threads) race and must be serialised by the
 * caller.  No allocation and no free is made.
 */
pkv_status paged_attn_decode_static(void* out, const void* q,
                                    const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, int32_t max_blocks_per_seq,
                                    const int32_t* seq_lens, int32_t batch,
                                    int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t page_size, int64_t num_pages,
                                    int32_t max_seq_len, float scale, int32_t window,
                                    int32_t* err_flag, void* stream);

/*
 * pkv_rope_table - fill the rotary (cos, sin) table that
 * paged_kv_append_rope reads.  Source: scripts/benchmarks commit log,
 * Gemma-4 engine commit ("Dual attention regimes": (cos, sin) pairs
 * precomputed per position and per attention regime, rope_theta 1e6 for
 * full attention).
 *
 *   cos_sin       [max_position, head_dim] float32 (written), 16-byte
 *                 aligned.  Row p, column i < head_dim/2 holds
 *                 cos(p * theta^(-2i/head_dim)); column head_dim/2 + i the
 *                 sine of the same angle.
 *   theta         the rotary base (> 0 and finite)
 *
 * Each entry is computed in double precision on the device and rounded
 * once to float.  Call it once per (max_position, head_dim, theta); the
 * table is the caller's.  head_dim must be even; max_position == 0 is a
 * no-op.
 */
pkv_status pkv_rope_table(float* cos_sin, int32_t max_position, int32_t head_dim,
                          double theta, void* stream);

/*
 * paged_kv_append_rope - paged_kv_append with the attention's input
 * transform fused in: per-head RMSNorm of q and k, then the rotary
 * embedding, for the same tokens whose K/V rows are appended.  Sources:
 * scripts/benchmarks commit log -- Llama-3.2 support commit (Qwen3's
 * per-head QK RMSNorm over head_dim of [B, S, H, D]), Gemma-4 shared-KV
 * commit (the cache keeps post-rotary K and V as projected).
 *
 *   q              [num_tokens, num_q_heads, head_dim] bf16, transformed in
 *                  place; NULL: no q (num_q_heads is then ignored)
 *   k_new, v_new   [num_tokens, num_kv_heads, head_dim] bf16 (read)
 *   k_cache,v_cache,slot_mapping, page_size, num_pages: as paged_kv_append
 *   positions      [num_tokens] int32: the token's position in its sequence
 *                  (the row of cos_sin)
 *   cos_sin        [max_position, head_dim] float32, as pkv_rope_table
 *                  writes it (16-byte aligned)
 *   q_norm_weight, k_norm_weight
 *                  [head_dim] bf16 RMSNorm weights, 16-byte aligned; NULL
 *                  means no norm on that side
 *   norm_eps       the RMSNorm epsilon (>= 0, finite)
 *
 * For each token t and head, with x the row as float:
 *   x <- x * w / sqrt(mean(x^2) + norm_eps)        (when a weight is given)
 *   for i < head_dim/2, with c, s = cos_sin[positions[t]][i], [head_dim/2 + i]:
 *     x'[i] = x[i] c - x[i + head_dim/2] s,  x'[i + head_dim/2] = x[i + head_dim/2] c + x[i] s
 * computed in float with one rounding to bf16 (nearest-even).  q rows are
 * written back; k rows go to slot_mapping[t] and v rows are copied there
 * bit-exactly.  A negative slot skips the append of that token (its q rows
 * are still transformed).  A position outside [0, max_position) skips the
 * token whole and raises PKV_DEVERR_POS.  head_dim in {64, 128, 256};
 * num_tokens * (num_q_heads + num_kv_heads) * head_dim / 8 < 2^30.
 * q must not overlap k_new, v_new or the pools.
 */
pkv_status paged_kv_append_rope(void* q, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache,
                                const int64_t* slot_mapping, const int32_t* positions,
                                const float* cos_sin, int32_t max_position,
                                const void* q_norm_weight, const void* k_norm_weight,
                                float norm_eps, int32_t num_tokens,
                                int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t page_size, int64_t num_pages,
                                int32_t* err_flag, void* stream);

/*
 * pkv_copy - copy `bytes` bytes from src to dst with the GPU's SMs, on
 * `stream`, for the small per-step transfers between pinned host memory
 * and the device: a decode step's inputs going in, its output rows coming
 * back.  The pages have no counterpart; it serves the step's host
 * transfers, whose fixed cost on the copy engines (11-14 us for 0.5-0.8 MB
 * on a GB300) is a fifth of the decode kernel's time.
 *
 *   dst, src  16-byte aligned; each is either device memory of the current
 *             device or host memory pinned through CUDA (cudaHostAlloc,
 *             cudaHostRegister, torch's pin_memory) and mapped at the same
 *             address on the device (unified addressing); the two ranges
 *             must not overlap
 *   bytes     a multiple of 16 (0: no-op)
 *
 * Each call checks both pointers with cudaPointerGetAttributes and rejects
 * other memory (pageable host memory, another device's memory) with
 * PKV_ERR_UNSUPPORTED; bad alignment, sizes or overlap give
 * PKV_ERR_INVALID.  Nothing is enqueued on a rejected call.  The copy is
 * asynchronous and allocates nothing.  It waits for the previous kernel in
 * the stream before its first load (programmatic dependent launch), so it
 * may read a kernel's output directly.  The data are in place when the
 * stream reaches the next operation (for host memory, after the stream has
 * been synchronised or an event waited on).
 */
pkv_status pkv_copy(void* dst, const void* src, size_t bytes, void* stream);

/* Human-readable name of a pkv_status value (static string). */
const char* pkv_status_string(int32_t status);

/* Message of the last CUDA error seen by this library on the calling host
 * thread ("" if none). */
const char* pkv_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */
