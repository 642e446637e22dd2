/*
 * pkv.h -- C ABI of libpkv.so: batched paged decode attention over a shared
 * bf16 KV page pool, with the one-token KV append (rotate-half RoPE), for
 * NVIDIA GB300 (sm_103a).
 *
 * Source of the operations: the Tiny-vLLM README translation "Hours of YouTube
 * and 85 handtyped pages of notes on LLM Inference - Start here", section
 * "これまでの進捗" (progress so far): a shared BF16 KV page pool whose pages
 * each hold K and V for 16 tokens, one block table per (sequence, layer);
 * decode adds one new token per sequence at its absolute RoPE position; paged
 * decode attention streams each sequence's cached pages with an FP32 online
 * softmax, never gathering a contiguous prefix and never storing scores; the
 * batched decode packs one token per active sequence and each sequence's
 * attention reads only its own cache.  The model dimensions (32 query heads,
 * 8 kv heads, head dim 64) are the fixed Llama 3.2 1B ones of section
 * "現在のスコープ" (scope).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - bf16 values are passed as pkv_bf16 (the raw 16-bit pattern).
 *  - Every tensor pointer is DEVICE memory owned by the caller, unless the
 *    comment says otherwise.  The library never allocates, frees or
 *    synchronizes; all work is enqueued on `stream` (NULL = the legacy
 *    default stream) and returns before it runs.  Calls are thread-safe,
 *    also across streams.  State kept between calls: a per-thread cache of
 *    TMA descriptors and of the wait limit (pkv_set_wait_limit_ns), the
 *    device's SM count, and per device up to four RoPE cos/sin tables for
 *    positions below 2048 (6 MiB of static device memory).  The first call
 *    with a rope_theta not seen before on a device builds a table for it in
 *    a free slot, on the calling stream, and tags the slot afterwards; a
 *    tagged slot is never rewritten.  Kernels read a table only once they
 *    have read its tag, and otherwise (table not built yet, or all four
 *    slots taken by other thetas) evaluate sincos themselves.  So calls with
 *    different thetas may run concurrently on any streams.  The library's
 *    device state (these tables, the static scratch buffer below) belongs to
 *    the CUDA context it was set up in: do not reset a device
 *    (cudaDeviceReset) between calls.
 *  - RoPE bit-exactness: keys are rotated in FP64 and rounded once to bf16,
 *    as the oracle does.  cos and sin come from CUDA's FP64 sincos on the
 *    device and from the C library on the oracle's side; where the two
 *    libraries differ in the last FP64 bit, a bf16 rounding could flip (about
 *    2^-44 per element, never observed over every position below 4096 for
 *    the thetas tested).  "Bit-exact" below is relative to that.
 *  - Pool layout: [num_pages][2 (K, V)][page_size][num_kv_heads][head_dim]
 *    bf16, i.e. element ((page*2 + kv)*page_size + slot)*Hkv*D + h*D + d.
 *    The pool must be 16-byte aligned.
 *  - Block table of one layer: int32 [batch][max_blocks]; entry k of row b is
 *    the physical page of tokens [16k, 16k+16) of sequence b.  Entries past
 *    the sequence's last block are never read (any value, -1 by convention).
 *  - Query head j uses kv head j / (num_q_heads / num_kv_heads).
 *  - Supported sizes: num_q_heads = 32, num_kv_heads = 8, head_dim = 64,
 *    page_size = 16 (other values return PKV_EUNSUPPORTED).
 *  - Kernels are launched with programmatic dependent launch: a kernel may
 *    start while the previous kernel on `stream` is still running, and waits
 *    for it (griddepcontrol.wait) before it reads anything it uses.  Before
 *    that wait the attention kernels only prefetch pool pages into L2, with
 *    addresses taken from the plan, lengths and block tables as they stand
 *    (every index range-checked); those words are read again after the wait,
 *    so a caller's kernel that writes them just before a call is safe.
 *  - Return value: PKV_OK or a PKV_E* code (see pkv_strerror).  Argument
 *    errors are detected on the host before anything is enqueued.  Bad DEVICE
 *    data (a page id outside [0, num_pages), a length or position outside the
 *    block table) never traps: the offending access is skipped and the
 *    matching PKV_DEVERR_* bit is OR-ed into *dev_err when dev_err is not NULL.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef uint16_t pkv_bf16;
typedef struct CUstream_st* pkv_stream_t; /* same type as cudaStream_t */

/* Host-side status codes. */
#define PKV_OK 0
#define PKV_EINVAL 1        /* NULL pointer, non-positive size, bad scale ... */
#define PKV_EUNSUPPORTED 2  /* head counts / dims / page size not compiled in */
#define PKV_EWORKSPACE 3    /* workspace missing or smaller than required */
#define PKV_ECUDA 4         /* a CUDA runtime call or launch failed */
#define PKV_EALIGN 5        /* a pointer violates the alignment stated above */
#define PKV_ESCRATCH 6      /* split partials exceed PKV_STATIC_SCRATCH_BYTES */

/* Device-side error bits OR-ed into *dev_err. */
#define PKV_DEVERR_PAGE 1u      /* block-table entry outside [0, num_pages) */
#define PKV_DEVERR_SEQLEN 2u    /* seq_lens[b] < 0 or > max_blocks*page_size */
#define PKV_DEVERR_POSITION 4u  /* positions[b] < 0 or >= max_blocks*page_size */
#define PKV_DEVERR_TIMEOUT 8u   /* an in-kernel wait for a page copy gave up */
#define PKV_DEVERR_OFFSETS 16u  /* a token outside the ranges of token_offsets */
#define PKV_DEVERR_PLAN 32u     /* seq_lens[b] differs from the length a work plan holds */

/* Library ABI version (bumped when a signature changes). */
PKV_API int pkv_abi_version(void);

/*
 * Limit, in nanoseconds, of each wait a kernel makes on its own progress (a
 * page copy landing, another warp role's hand-off, an MMA completing) for the
 * kernels that the CALLING THREAD launches from now on; returns the previous
 * value.  The default is 2,000,000,000 (2 s).  Past the limit a kernel stops
 * waiting, ORs PKV_DEVERR_TIMEOUT into *dev_err, lets every copy and MMA it
 * has started finish (those waits always take the full 2 s limit, so nothing
 * it started is still running when it exits), frees what it holds and
 * returns, so a stalled copy never hangs the stream; the outputs of a call
 * that timed out are finite but not the attention result.  0 means a single
 * look: a copy that has not landed when first waited for counts as a
 * timeout (useful to exercise that path on normal inputs).  A CUDA graph
 * keeps the value its captured launches were made with.  Host code only.
 * (The source pages have no counterpart: failure handling of this library.)
 */
PKV_API unsigned long long pkv_set_wait_limit_ns(unsigned long long ns);

/* Static description of a status code; never NULL. */
PKV_API const char* pkv_strerror(int status);

/*
 * pkv_kv_append -- decode-time KV append ("これまでの進捗", KV page pool item:
 * one new token per sequence at its absolute RoPE position).
 *
 * For every sequence b and kv head h, with pos = positions[b],
 * page = block_table[b*max_blocks + pos/page_size], slot = pos % page_size:
 *   pool[page][K][slot][h][:] = RoPE(k_new[b][h][:], pos)
 *   pool[page][V][slot][h][:] = v_new[b][h][:]
 * RoPE is rotate-half: for i < D/2 the pair (x_i, x_{i+D/2}) turns by the
 * angle pos * rope_theta^(-2i/D); the rotation is evaluated in FP64 and
 * rounded once to bf16 (round to nearest even), so results are bit-exact.
 * If q_in and q_out are both non-NULL the same rotation is applied out of
 * place to the queries: q_out[b][j] = RoPE(q_in[b][j], positions[b]) for
 * j < num_q_heads (q_in/q_out: [batch][num_q_heads][head_dim]); otherwise
 * both must be NULL.
 *
 *   k_new, v_new  [batch][num_kv_heads][head_dim] bf16, read only
 *   pool          the shared page pool (layout above); written in place at
 *                 one slot per sequence
 *   positions     int32 [batch]
 *   dev_err       optional int32, bits PKV_DEVERR_PAGE / _POSITION
 * A sequence with a bad position or page is skipped (its query rotation is
 * still written).  Two sequences must not name the same (page, slot).
 */
PKV_API int pkv_kv_append(const pkv_bf16* k_new, const pkv_bf16* v_new,
                          pkv_bf16* pool, int64_t num_pages,
                          const int32_t* block_table, int max_blocks,
                          const int32_t* positions, int batch,
                          int num_kv_heads, int head_dim, int page_size,
                          double rope_theta, const pkv_bf16* q_in,
                          pkv_bf16* q_out, int num_q_heads, int32_t* dev_err,
                          pkv_stream_t stream);

/*
 * pkv_kv_write_prefill -- paged prefill write ("これまでの進捗", KV page pool
 * item: prefill fills the prompt pages).  Writes a ragged batch of new tokens
 * into the pool through the block tables, each exactly as pkv_kv_append
 * would write it at its position.
 *
 * Sequence b owns tokens [token_offsets[b], token_offsets[b+1]) of k and v
 * ([num_tokens][num_kv_heads][head_dim] bf16); its i-th token goes to
 * position start_positions[b] + i, i.e. slot (pos % page_size) of page
 * block_table[b*max_blocks + pos/page_size], K rotated by RoPE at pos (FP64,
 * one rounding to bf16) and V unchanged.
 *
 *   k, v             16-byte aligned
 *   token_offsets    int32 [batch + 1], non-decreasing, token_offsets[0] = 0,
 *                    token_offsets[batch] = num_tokens
 *   start_positions  int32 [batch]
 *   dev_err          optional int32, bits PKV_DEVERR_PAGE / _POSITION /
 *                    _OFFSETS (a token whose offsets do not bracket it)
 * A token with a bad position, page or offset is skipped.  No two tokens may
 * name the same (page, slot).
 */
PKV_API int pkv_kv_write_prefill(const pkv_bf16* k, const pkv_bf16* v,
                                 int num_tokens, const int32_t* token_offsets,
                                 const int32_t* start_positions,
                                 pkv_bf16* pool, int64_t num_pages,
                                 const int32_t* block_table, int max_blocks,
                                 int batch, int num_kv_heads, int head_dim,
                                 int page_size, double rope_theta,
                                 int32_t* dev_err, pkv_stream_t stream);

/*
 * pkv_paged_decode_attention -- paged decode attention with an FP32 online
 * softmax ("これまでの進捗", paged decode attention item).
 *
 * For every sequence b and query head j, with g = j / (Hq/Hkv) and
 * L = seq_lens[b]:
 *   out[b][j][:] = sum_{t<L} softmax_t(scale * q[b][j] . K_t) V_t
 * where K_t, V_t are row (t % page_size) of kv head g in page
 * block_table[b*max_blocks + t/page_size].  L counts the token appended in
 * the same step.  L = 0 gives a zero row.  Scores and the softmax are FP32;
 * the output is rounded to bf16 (nearest even).
 *
 *   q          [batch][num_q_heads][head_dim] bf16 (already rotated)
 *   seq_lens   int32 [batch]
 *   out        [batch][num_q_heads][head_dim] bf16, written
 *   workspace  device scratch for split-K partials, at least
 *              pkv_workspace_bytes(...) bytes, 16-byte aligned; may be NULL
 *              when that size is 0.  Its contents need no initialisation and
 *              are garbage afterwards.
 *   num_splits 0 = choose automatically; S > 0 = split each sequence's pages
 *              into at most S contiguous logical ranges, combined by a merge
 *              kernel.  The same inputs and num_splits give bit-identical
 *              outputs on every run.
 *   dev_err    optional int32, bits PKV_DEVERR_PAGE / _SEQLEN / _TIMEOUT
 * Pages of a sequence with a bad id are skipped; a length outside the block
 * table is clamped to [0, max_blocks*page_size].
 */
PKV_API int pkv_paged_decode_attention(
    const pkv_bf16* q, const pkv_bf16* pool, int64_t num_pages,
    const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
    int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
    float scale, pkv_bf16* out, void* workspace, size_t workspace_bytes,
    int num_splits, int32_t* dev_err, pkv_stream_t stream);

/*
 * pkv_decode_step -- one whole decode step of one layer in a single kernel:
 * the KV append of pkv_kv_append at position seq_lens[b] - 1 followed by the
 * attention of pkv_paged_decode_attention over seq_lens[b] tokens ("これまで
 * の進捗": decode adds one token per sequence at its absolute RoPE position,
 * then every query head streams its sequence's pages).
 *
 * Results are the same as calling pkv_kv_append(positions = seq_lens - 1)
 * and then pkv_paged_decode_attention with the same arguments: the pool slot
 * receives the same bits and `out` is bit-identical.  The CTA that processes
 * a sequence's last page computes the new K/V row itself, writes it to the
 * pool and uses it directly, so no second launch and no global round trip
 * separate the two stages.  Sequences with seq_lens[b] == 0 append nothing
 * and give a zero row.  The pool is written at one slot per sequence.
 * Workspace, num_splits and dev_err are as for pkv_paged_decode_attention
 * (dev_err additionally reports PKV_DEVERR_PAGE for the appended block).
 */
PKV_API int pkv_decode_step(const pkv_bf16* q, const pkv_bf16* k_new,
                            const pkv_bf16* v_new, pkv_bf16* pool,
                            int64_t num_pages, const int32_t* block_table,
                            int max_blocks, const int32_t* seq_lens, int batch,
                            int num_q_heads, int num_kv_heads, int head_dim,
                            int page_size, double rope_theta, float scale,
                            pkv_bf16* out, void* workspace,
                            size_t workspace_bytes, int num_splits,
                            int32_t* dev_err, pkv_stream_t stream);

/*
 * Bytes of workspace pkv_paged_decode_attention needs for these sizes and
 * num_splits (0 = the automatic choice on the current device).  Returns 0
 * when no split is needed, and (size_t)-1 for invalid sizes.
 */
PKV_API size_t pkv_workspace_bytes(int batch, int num_q_heads,
                                   int num_kv_heads, int head_dim,
                                   int max_blocks, int num_splits);

/*
 * The number of logical page ranges per sequence that
 * pkv_paged_decode_attention will use for these sizes (resolving
 * num_splits = 0 on the current device), or -1 for invalid sizes.
 */
PKV_API int pkv_plan_splits(int batch, int num_kv_heads, int max_blocks,
                            int num_splits);

/*
 * Host-side check of a batch's block tables and lengths, for callers that
 * want bad entries found before a launch (the kernels themselves skip them
 * and report PKV_DEVERR_* bits): every seq_lens[b] in [0, max_blocks *
 * page_size], and every live table entry (block < ceil(seq_lens[b] /
 * page_size)) in [0, num_pages).  block_table [batch][max_blocks] and
 * seq_lens [batch] are host memory.  Returns PKV_OK, or PKV_EINVAL with
 * *bad_seq and *bad_block (either may be NULL) set to the first offending
 * sequence and block (*bad_block = -1 for a bad length, and both -1 for bad
 * sizes or pointers).  Pure host code.
 */
PKV_API int pkv_check_tables(const int32_t* block_table, int max_blocks,
                             const int32_t* seq_lens, int batch, int64_t num_pages,
                             int page_size, int* bad_seq, int* bad_block);

/*
 * Work plans: split a ragged batch on the host, run it on the device.
 *
 * The automatic split plan of the calls above cannot see the lengths (they
 * live on the device), so a batch that mixes a few long sequences with many
 * short ones waits on its long sequences.  A caller that holds the lengths
 * on the host -- a scheduler always does -- can build a work plan instead
 * and pass it to the _planned entry points.  A plan is sized by a work unit
 * of U pages per warp: ranges of R = clamp(4 U, 8, min(max_blocks, 1024))
 * pages, and
 *   - sequences of more than R pages are cut into ceil(p / R) ranges of
 *     near-equal size, one CTA per (range, kv head), combined afterwards by
 *     a merge kernel; sequences of up to R pages get one such CTA;
 *   - sequences of at most min(R / 4, 16) pages (and empty ones) are packed
 *     four to a CTA, one warp each, so a warp again streams about U pages;
 *   - CTAs run in order of the pages their busiest warp streams, most first.
 * U is the smallest unit, from ceil(P / (2 SMs)) up (P: the batch's pages),
 * whose plan fits in one wave of four CTAs per SM; when none does, the
 * ranges take the whole table width (a batch of long sequences then gets
 * one range each, as with num_splits = 1).
 * Larger layers (P >= 16 x SMs) get a segment plan instead when its bins
 * hold at least 16 pages: the pages are cut into pieces (a sequence of more
 * than T pages into ceil(p / T) near-equal pieces) and packed best-fit,
 * largest first, into bins of at most T pages and 4 segments, T the smallest
 * bin size whose bins fit in one wave of two CTAs per SM; one CTA of all 8 kv
 * heads streams each bin, each page one 32 KiB box.  A sequence in several
 * pieces is combined by the merge kernel.
 * The plan is plain data: 12 header words
 *   {PKV_PLAN_MAGIC, batch, max_blocks, num_items, num_merges, num_slots,
 *    range_pages, bytes_used, num_shared, shared_pages, num_segs, layout},
 * then num_items items of 16 int32 words, all of kinds 0 and 1 or all of
 * kind 2:
 *   kind 0 (range), 1 (packed): {kind, slot (-1: not split), p_begin, n,
 *     seq[4], len[4], 0, 0, 0, 0} -- a range item repeats its sequence in all
 *     four seq/len words; a packed item holds one sequence per warp, -1 for
 *     none;
 *   kind 2 (segment CTA): {2, first segment, segments, pages, 0 x 12};
 * then num_merges entries {b, first slot, pieces, 0}, then num_shared
 * shared-prefix items of 36 words {members, p_begin, n, 0, seq[16],
 * slot[16]} (plans from pkv_plan_build_shared only; shared_pages is the
 * longest one's n), then num_segs segments of 8 words {b, L, p_begin, n,
 * slot (-1: writes the output), fold, fold_slot, 0}: a segment with fold > 0
 * writes the output of its sequence's pages [p_begin, p_begin + n) combined
 * with the partials of slots [fold_slot, fold_slot + fold), which the
 * shared-prefix items wrote (a group member whose own pages are one segment
 * needs no merge entry).  range_pages is the longest range or bin.
 * layout 0: the shared-prefix CTAs (if any) run first, two per SM, and the
 * other kernels after them.  layout 1 (a shared-prefix plan whose
 * shared-prefix CTAs fit one per SM; pkv_plan_build_shared makes it whenever
 * they do): the other attention CTAs run beside the shared-prefix CTAs,
 * streaming their own pages from the start, and wait for the shared-prefix
 * grid only to fold its partials and before they end -- segment CTAs sized
 * for one per SM when bins of one CTA per SM reach 16 pages (whatever P),
 * else per-(item, kv head) CTAs sized for two per SM next to each
 * shared-prefix CTA.  Any other layout value is refused.  The results follow the same numerics as the
 * calls above (same tolerance, bit-identical on repeated runs of a plan).
 */
#define PKV_PLAN_MAGIC 0x32564b50 /* "PKV2" */

/* Bytes a plan for this batch and table width can take (host buffer). */
PKV_API size_t pkv_plan_bytes(int batch, int max_blocks);

/*
 * Build a plan from the host copy of the lengths (after this step's append,
 * as seq_lens), for a device with num_sms SMs (0 = the current device).
 * plan: host memory, 16-byte aligned, at least pkv_plan_bytes() bytes.
 * Returns PKV_OK, PKV_EINVAL (a length outside [0, max_blocks * page_size],
 * bad sizes or buffer), PKV_EALIGN, PKV_EUNSUPPORTED (more than 65535 work
 * items) or PKV_ECUDA (no device to size it for).  Pure host code; thread-safe.
 * The planner keeps its working buffers per calling thread and reuses them
 * from one call to the next (a few MB for the largest batches), so a
 * serving loop that plans every step allocates nothing once warm; they are
 * freed when the thread exits.
 */
PKV_API int pkv_plan_build(const int32_t* seq_lens_host, int batch, int max_blocks,
                           int num_sms, void* plan, size_t plan_bytes);

/*
 * A plan for a batch whose sequences share prompt prefixes (block tables
 * naming the same physical pages; "Tiny-vLLMでゼロから構築する高性能LLM推論
 * エンジン", section "KV Cache").  block_tables_host: the host copy of this
 * layer's tables, int32 [batch][max_blocks].  Runs of up to 16 consecutive
 * sequences whose tables start with the same min_shared_pages or more page
 * ids form a group; its common pages (never a member's last page) become
 * shared-prefix items, each attended once for all members by
 * paged_decode_shared_kernel, which writes one partial per member.  Each
 * member's own pages become ranges writing partials too, and one merge
 * combines a member's partials.  Sequences in no group are planned as by
 * pkv_plan_build.  Same returns as pkv_plan_build (PKV_EUNSUPPORTED also for
 * more than 65535 shared-prefix items).  Pure host code.
 */
PKV_API int pkv_plan_build_shared(const int32_t* seq_lens_host, const int32_t* block_tables_host,
                                  int batch, int max_blocks, int num_sms, int min_shared_pages,
                                  void* plan, size_t plan_bytes);

/* Device workspace bytes a built plan needs (0 when nothing is split). */
PKV_API size_t pkv_plan_workspace_bytes(const void* plan);

/*
 * pkv_paged_decode_attention / pkv_decode_step under a work plan.
 * plan_host: the built plan (read on the host for the grid sizes);
 * plan_dev: a device copy of its first bytes_used bytes, 16-byte aligned,
 * which must stay unchanged until the call's kernels have run.  The kernels
 * read plan_dev as soon as they start, which may be before the kernel queued
 * just ahead of the call has finished (programmatic dependent launch): fill
 * it with a copy (cudaMemcpyAsync, as the Python binding's Plan.to does) or
 * earlier work, not with a kernel launched right before the call.  The kernels
 * take every length from the plan; seq_lens is only compared with it, and a
 * difference sets PKV_DEVERR_PLAN (the outputs then follow the plan's
 * lengths).  workspace: at least pkv_plan_workspace_bytes(plan_host).
 * Other arguments as for the calls above.
 */
PKV_API int pkv_paged_decode_attention_planned(
    const pkv_bf16* q, const pkv_bf16* pool, int64_t num_pages,
    const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
    int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
    float scale, pkv_bf16* out, const void* plan_host, const void* plan_dev,
    void* workspace, size_t workspace_bytes, int32_t* dev_err, pkv_stream_t stream);

PKV_API int pkv_decode_step_planned(
    const pkv_bf16* q, const pkv_bf16* k_new, const pkv_bf16* v_new, pkv_bf16* pool,
    int64_t num_pages, const int32_t* block_table, int max_blocks,
    const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
    int head_dim, int page_size, double rope_theta, float scale, pkv_bf16* out,
    const void* plan_host, const void* plan_dev, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, pkv_stream_t stream);

/*
 * pkv_decode_step_planned for `layers` layers of one decode step in one call:
 * layer l takes q + l*batch*Hq*D, k_new / v_new + l*batch*Hkv*D, block_tables
 * + l*batch*max_blocks and writes out + l*batch*Hq*D (every array holding the
 * layers back to back), with the same lengths, plan and workspace; the layers
 * are launched in order on `stream`, exactly as `layers` separate calls would
 * be.  Arguments are checked once, before anything is enqueued.
 */
PKV_API int pkv_decode_steps_planned(
    int layers, const pkv_bf16* q, const pkv_bf16* k_new, const pkv_bf16* v_new,
    pkv_bf16* pool, int64_t num_pages, const int32_t* block_tables, int max_blocks,
    const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
    int page_size, double rope_theta, float scale, pkv_bf16* out, const void* plan_host,
    const void* plan_dev, void* workspace, size_t workspace_bytes, int32_t* dev_err,
    pkv_stream_t stream);

/*
 * pkv_kv_write_prefill for `layers` layers of the same prompts in one call:
 * layer l writes k + l*num_tokens*Hkv*D and v + l*num_tokens*Hkv*D through
 * block_tables + l*batch*max_blocks (the arrays holding the layers back to
 * back), with the same offsets and positions; launched in layer order on
 * `stream`.  Arguments are checked once, before anything is enqueued.
 */
PKV_API int pkv_kv_write_prefill_layers(int layers, const pkv_bf16* k, const pkv_bf16* v,
                                        int num_tokens, const int32_t* token_offsets,
                                        const int32_t* start_positions, pkv_bf16* pool,
                                        int64_t num_pages, const int32_t* block_tables,
                                        int max_blocks, int batch, int num_kv_heads,
                                        int head_dim, int page_size, double rope_theta,
                                        int32_t* dev_err, pkv_stream_t stream);

/*
 * The kernels pkv_paged_decode_attention (plan == NULL, with num_splits as
 * given) or the _planned calls (plan = a built plan; num_splits ignored) launch
 * for this batch on the current device, joined by '+': the attention kernel
 * ("paged_decode_pagebox_kernel", one CTA per sequence range covering all kv
 * heads, for batches that fill the SMs; else "paged_decode_kernel", one CTA
 * per (sequence range, kv head)), then the split merge when one runs.  The
 * fused steps launch the same kernels.  Static strings; NULL for invalid sizes.
 */
PKV_API const char* pkv_attention_kernels(int batch, int max_blocks, int num_splits,
                                          const void* plan);

/*
 * pkv_paged_decode_attention_static_ws -- the same computation as
 * pkv_paged_decode_attention, for callers that cannot allocate device memory.
 * (The source pages have no counterpart to this entry point.)
 *
 * Who needs it: code that runs where cudaMalloc is not an option -- for
 * example inside a host callback or an allocator hook, in a process whose
 * device memory is entirely owned by another framework's caching allocator,
 * or in a tight real-time loop that must never enter the driver's allocator.
 * Such a caller still owns and passes every input and the output; only the
 * split-K partials move from a caller workspace to a fixed scratch buffer
 * that the library holds in device memory (a file-scope __device__ array of
 * PKV_STATIC_SCRATCH_BYTES bytes, present on every GPU that loads libpkv
 * until the process exits).  This entry point calls no cudaMalloc, cudaFree
 * or other allocating routine.
 *
 * Arguments and results are those of pkv_paged_decode_attention without the
 * workspace pair.  If the chosen split plan would need more than
 * PKV_STATIC_SCRATCH_BYTES of partials (pkv_workspace_bytes() > that size),
 * the call returns PKV_ESCRATCH before enqueuing anything; pass a smaller
 * num_splits (1 needs no scratch at all) or use the workspace entry point.
 *
 * The first call on each device looks up the device address of the scratch
 * buffer with that device current (cudaGetSymbolAddress) and caches it; with
 * lazy module loading that first call may also be the one that loads the
 * library's device code and places the buffer.  So make one call on each
 * device before any stream capture, and do not reset the device
 * (cudaDeviceReset) or destroy its primary context between calls: the
 * cached address belongs to the context it was taken in.  All calls on a device share
 * the one buffer: two calls whose kernels overlap in time on the GPU (for
 * example on two streams without an ordering between them) race on it and
 * produce garbage.  Calls ordered on one stream are safe.  The buffer keeps
 * the previous call's partials; nothing in it has to start at zero, because
 * every partial the merge reads is written earlier in the same call.
 */
#define PKV_STATIC_SCRATCH_BYTES (4u << 20)

PKV_API int pkv_paged_decode_attention_static_ws(
    const pkv_bf16* q, const pkv_bf16* pool, int64_t num_pages,
    const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
    int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
    float scale, pkv_bf16* out, int num_splits, int32_t* dev_err,
    pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
