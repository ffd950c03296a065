/*
 * tf.h -- C ABI of the segmented speculative-verify step (LFM2 shared-round
 * decode with drafts) for NVIDIA GB300 (sm_103a).
 *
 * What the step computes comes from the TensorFold pages:
 *   [SRD]   PR #1377 "LFM2: shared-round decode"
 *           - commit "a shared round runs each layer's conv and attention once
 *             over all its streams" (segment table of cache addresses, row
 *             offsets and key counts; one launch per layer over every row;
 *             per-stream attention partials; float64 attention and a host
 *             replay of the conv steps as the checks);
 *           - commit "a verify's greedy rows take the GPU's pick of their
 *             logits" (the largest logit, the lowest id among equal ones,
 *             nonfinite rows flagged);
 *           - commit "the conv, qk, attention and merge kernels' bodies as
 *             inline functions" (qk, attention, merge);
 *           - section "Failures the tests catch" (a scratch too small for
 *             per-stream partials; a table reaching memory it did not declare).
 *   [DSP]   PR #1391 "lfm2: draft with LiquidAI's DSpark drafter (--drafter)":
 *           every draft is verified by the target; the target's attention
 *           stays causal; the drafter's block attention (the same kernels
 *           with a FULL flag, under which every row of a block sees all of
 *           its stream's keys), its Markov head (each draft row adds the
 *           product of W2 with the W1 row of the previous pick to its logits
 *           and takes the argmax, the rows in sequence; the step as the
 *           argmax of bf16(base + bf16(W2 . W1[prev])), lowest token on a
 *           tie, a NaN score flagged) and the held path's kernel that fills
 *           the verify's ids from the drafter's picks (a bad pick raises a
 *           flag for the verify instead of becoming a token).
 *
 * Conventions for every call:
 *   - All tensors are dense, row-major, in DEVICE memory owned by the caller,
 *     and start on a 16-byte boundary. bf16 tensors are passed as `void*`.
 *   - Every call is asynchronous on the caller's CUDA stream `stream` (a
 *     cudaStream_t; NULL is the legacy default stream) and never synchronises.
 *   - Every call returns a tf_status. Invalid arguments are refused on the host
 *     before anything is launched; nothing aborts. A nonfinite logit is data,
 *     reported in the flags, never an error.
 *   - Model widths are fixed (LFM2.5-24B-A2B): TF_H conv channels, conv input
 *     TF_CIN = 3*TF_H as the consecutive slices (B, C, x), kernel width TF_KW,
 *     TF_NQ query heads sharing TF_NKV KV heads of width TF_D.
 */
#ifndef TF_H_INCLUDED
#define TF_H_INCLUDED

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TF_H        2048
#define TF_CIN      6144
#define TF_KW       3
#define TF_NQ       32
#define TF_NKV      8
#define TF_D        64
#define TF_MAX_ROWS 16          /* window rows per stream (1 + drafts) */
#define TF_MAX_KEYS (1 << 22)   /* cache rows per stream */
#define TF_MAX_PROMPT_ROWS 65536  /* rows of one prompt call (tf_prompt_build) */
#define TF_PROMPT_WINDOW_ROWS 32  /* a prompt call's attention window (tf_prompt_build) */
#define TF_MAX_STREAMS 65536
#define TF_MK       256         /* width of the drafter's Markov head rows (W1, W2) */

typedef enum {
    TF_OK = 0,
    TF_EINVAL = 1,   /* null pointer, bad shape, unpacked rows, aliasing, misalignment */
    TF_ERANGE = 2,   /* a size beyond the limits above */
    TF_ENOMEM = 3,   /* the library's own table allocation failed */
    TF_ECUDA = 4,    /* a CUDA call or launch failed (see tf_last_cuda_error) */
    TF_ETIMEOUT = 5  /* a kernel gave up a bounded device wait (tf_segments_status) */
} tf_status;

struct CUstream_st;                       /* cudaStream_t is struct CUstream_st* */
typedef struct CUstream_st* tf_cuda_stream;

/* One stream of a shared round ([SRD]: the table lists each stream's cache
 * addresses, row offset and key count).
 *   rows        window rows r_s = 1 + drafts, 1..TF_MAX_ROWS
 *   row_offset  first row of the stream in every [R][...] tensor; streams are
 *               packed in order: row_offset_0 = 0, row_offset_{s+1} =
 *               row_offset_s + rows_s
 *   keys        k_s, cache entries INCLUDING the window's own rows (their K/V
 *               are already written); window row i sees keys
 *               [0, keys - rows + i + 1) (causal, [DSP]); rows <= keys
 *   kv_capacity cache rows allocated per KV head, keys <= kv_capacity */
typedef struct {
    int32_t rows;
    int32_t row_offset;
    int32_t keys;
    int32_t kv_capacity;
} tf_stream;

/* Host-side sizes of a table, from tf_segments_plan (no GPU needed). */
typedef struct {
    int32_t n_streams;
    int32_t n_rows;           /* R = sum of rows */
    int32_t max_rows;
    int32_t n_conv_tiles;     /* conv tiles of at most 8 rows ([SRD]) */
    int32_t n_attn_items;     /* (stream, key chunk) work items per KV head */
    int32_t attn_kernels;     /* partial-kernel launches per attention layer (1 or 2) */
    int32_t attn_merge_launch;/* 1 if tf_attn also launches the merge kernel */
    int32_t reserved;
    int64_t n_partials;       /* partial records: sum_s rows_s * 32 * chunks_s */
    int64_t partials_bytes;   /* scratch tf_attn_partials needs (see below) */
} tf_plan;

/* The library's own device copy of a segment table. Immutable once built. */
typedef struct tf_segments tf_segments;

/* Split-K chunk of a stream: keys [c*chunk, (c+1)*chunk). The chunk length is
 * 256 * max(rows, 4) keys (partial records stay near 1/64 of the K/V bytes),
 * and 512 * rows for windows of 9 to 16 rows (the tensor-core kernel: fewer,
 * longer units measured faster there); it depends on the stream alone, so a
 * stream's results do not depend on which other streams share the round. */
int32_t tf_chunk_keys(int32_t rows);

/* Validate `streams` and compute the table's sizes. Host only; touches no GPU.
 * Errors: TF_EINVAL (null, rows < 1, unpacked offsets, keys < rows,
 * keys > kv_capacity), TF_ERANGE (beyond TF_MAX_*). n_streams == 0 is an
 * empty round (every call on its table is a no-op). */
int tf_segments_plan(const tf_stream* streams, int n_streams, tf_plan* out);

/* Build the segment table on the device ([SRD] segments.zig).
 *   streams      host array [n_streams]
 *   conv_state   host array [n_conv][n_streams] of device pointers, each to a
 *                bf16 [2][TF_H] rolling conv state (oldest row first), read
 *                and rewritten in place by tf_conv_rows / tf_accept
 *   conv_hist    NULL, or host array [n_conv][n_streams] of device pointers,
 *                each to a bf16 [rows+2][TF_H] history written by
 *                tf_conv_rows (the state before the window, then every row's
 *                gate); entries of one-row streams may be NULL. NULL disables
 *                the conv rewind in tf_accept.
 *   k_cache, v_cache  host arrays [n_attn][n_streams] of device pointers, each
 *                to a bf16 [TF_NKV][kv_capacity][TF_D] cache (head-major)
 * Refuses (TF_EINVAL) null or misaligned pointers and any two buffers of the
 * table that overlap (conv states and histories across every stream and
 * layer; K and V caches likewise) -- the bug class of [SRD]'s planted controls,
 * in which every stream reads or writes stream 0's conv state or KV cache.
 * The table is copied to the device on `stream` before the call returns; the
 * host arrays may be freed at once. *out is owned by the caller and released
 * with tf_segments_free. */
int tf_segments_build(const tf_stream* streams, int n_streams,
                      const void* const* conv_state, const void* const* conv_hist,
                      const void* const* k_cache, const void* const* v_cache,
                      int n_conv, int n_attn, tf_cuda_stream stream,
                      tf_segments** out);

/* Free a table (synchronises the device through cudaFree). NULL is a no-op. */
int tf_segments_free(tf_segments* seg);

/* Sizes of a built table (same as tf_segments_plan's). */
int tf_segments_query(const tf_segments* seg, tf_plan* out);

/* Bytes of partial scratch tf_attn_partials writes and tf_attn_merge reads
 * ([SRD]: each stream keeps its own partials in the scratch).
 * Layout: float o[n_partials][TF_D], then float2 ml[n_partials] (m, l).
 * 0 for a NULL table. */
size_t tf_partials_bytes(const tf_segments* seg);

/* a1. LFM2 gated short conv of one conv layer over every row of every stream
 * ([SRD]: the 30 short-conv layers, each run once over every row).
 *   bcx  bf16 [R][TF_CIN], row = (B, C, x)
 *   w    bf16 [TF_H][TF_KW] depthwise taps; w[c][0] multiplies the oldest row
 *   y    float [R][TF_H] output, y = C * conv
 * Per stream, row by row: bx = bf16_rne(B*x); seq = [state0, state1, bx_0..];
 * conv_i = w0*seq[i] + w1*seq[i+1] + w2*seq[i+2] (fp32). Afterwards the
 * stream's state holds the last two entries of seq and its history (if any)
 * all of them; both are bit-exact. Errors: TF_EINVAL (null/misaligned,
 * conv_layer out of range). */
int tf_conv_rows(const tf_segments* seg, int conv_layer, const void* bcx,
                 const void* w, float* y, tf_cuda_stream stream);

/* a2. Causal GQA attention partials of one attention layer: for every stream,
 * KV head, key chunk, window row and query head, (m, l, o) over the chunk's
 * visible keys ([SRD]: the qk, attention and merge of the 10 attention
 * layers). Streams with windows of 9 rows or more run on the tcgen05
 * tensor-core kernel, the others
 * on the mma.sync kernel; the choice depends on the stream alone (so a
 * stream's bits do not depend on its round), and a round holding both kinds
 * makes one launch of each (tf_plan.attn_kernels). The environment variable
 * TF_ATTN_PATH=mma|tc, read by tf_segments_build, forces one kernel for every
 * window of at most 16 rows (a prompt table's wider windows always run on the
 * tensor cores); the mma.sync kernel takes a window as items of at most 8
 * rows. P.V runs with P and V in fp16 and fp32 accumulation; a piece of work
 * whose fp16 result holds a partial sum that is not finite (a V of 65,536 or
 * more has no fp16 value) or whose partial outputs |o|/l all lie below 2^-10
 * is computed again with V in bf16 and P split into a bf16 high part and a
 * bf16 remainder (the mma.sync kernel per item, the tensor-core kernel per
 * unit of one chunk and KV head, in the launch's last CTA). So every finite
 * V is supported; in an fp16 result only values of V below 2^-14 round, by
 * at most 2^-25 each. Sums of P.V must stay within fp32's range.
 *   q         bf16 [R][TF_NQ][TF_D]
 *   partials  device scratch of tf_partials_bytes(seg) bytes. Record of
 *             stream s, chunk c, KV head g, row i, head 4g+hh:
 *             pbase_s + ((c*8 + g)*rows_s + i)*4 + hh, pbase_s = sum over
 *             earlier streams of rows * 32 * chunks.
 *             m = (largest score) * log2(e), l = sum 2^(s*log2(e) - m),
 *             o[d] = sum 2^(s*log2(e) - m) * v[d]; a chunk without a visible
 *             key has m = -inf, l = 0, o = 0.
 * Score = (q . k) / 8; query head h reads KV head h / 4. Errors: TF_EINVAL. */
int tf_attn_partials(const tf_segments* seg, int attn_layer, const void* q,
                     void* partials, tf_cuda_stream stream);

/* a2+a3 in one call: the attention output of one layer. One launch of the
 * partials kernel(s) in which a stream with a single key chunk writes its
 * output directly and a stream with few partial records (4 * rows * chunks
 * <= 512) is merged by the last CTA to finish each of its KV heads (counted
 * by per-layer counters in the table that reset themselves); streams with
 * more records are merged by one merge launch. ([SRD]: each layer runs once
 * over every row.) A round holding both kinds of window runs the mma.sync
 * launch on a stream of the table's own, forked from `stream` and joined
 * back to it before the call returns, so that the two launches run side by
 * side; work queued on `stream` after the call waits for both. Same
 * arguments as tf_attn_partials plus `out`
 * (float [R][TF_NQ][TF_D]); `partials` is the scratch of tf_partials_bytes.
 * Calls on the same table and layer must not overlap on the GPU.
 * Errors: TF_EINVAL. */
int tf_attn(const tf_segments* seg, int attn_layer, const void* q, void* partials, float* out,
            tf_cuda_stream stream);

/* The drafter's non-causal block attention ([DSP] lfm2_attn_block: the
 * target's attention kernels with a FULL flag, under which every row of a
 * block sees the keys [0, len + 1)). Reading: len + 1 is the stream's key
 * count including
 * the block's own rows, so every window row sees all `keys` keys of its
 * stream (what the last row sees under the causal count). Same arguments,
 * records, kernels, chunking and errors as tf_attn_partials / tf_attn; the
 * merge (tf_attn_merge) is shared. */
int tf_attn_block_partials(const tf_segments* seg, int attn_layer, const void* q,
                           void* partials, tf_cuda_stream stream);
int tf_attn_block(const tf_segments* seg, int attn_layer, const void* q, void* partials,
                  float* out, tf_cuda_stream stream);

/* a3. Log-sum-exp merge of the partials into the attention output
 * ([SRD] lfm2_merge_row): out = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c,
 * M = max_c m_c, empty chunks skipped.
 *   out  float [R][TF_NQ][TF_D]. Errors: TF_EINVAL. */
int tf_attn_merge(const tf_segments* seg, const void* partials, float* out,
                  tf_cuda_stream stream);

/* Attention of one layer (tf_attn_partials then tf_attn_merge) that allocates
 * nothing: the partial scratch is a fixed array of TF_STATIC_SCRATCH_BYTES
 * compiled into the library (no counterpart on the pages; it exists for
 * callers that cannot call cudaMalloc or any allocating routine, such as code
 * under a strict memory budget or an allocator it does not own).
 *   q    bf16 [R][TF_NQ][TF_D], out float [R][TF_NQ][TF_D], as above.
 * Every GPU that loads the library holds the array until the process exits.
 * The first call on a device looks the array's device address up (with that
 * device current); make that first call before any stream capture. The
 * address is kept for the life of the process: a cudaDeviceReset (or
 * anything else that unloads the library's module from a device) leaves it
 * stale, so do not call tf_attn_static after one. Calls
 * share the one array: calls whose launches overlap on the GPU (different
 * streams at once) race and give wrong results. Nothing in the array has to
 * start at zero; each call writes every record it reads.
 * Errors: TF_ERANGE when tf_partials_bytes(seg) > TF_STATIC_SCRATCH_BYTES
 * (nothing is launched), TF_EINVAL as tf_attn_partials. Calls no cudaMalloc,
 * cudaFree or other allocating routine. */
#define TF_STATIC_SCRATCH_BYTES (16u << 20)
int tf_attn_static(const tf_segments* seg, int attn_layer, const void* q, float* out,
                   tf_cuda_stream stream);

/* a4. Greedy pick of each row of bf16 logits ([SRD] lfm2_argmax: the largest
 * logit, the lowest id among equal largest values, and a flag on any row
 * holding a nonfinite value).
 *   logits      bf16, row r at logits + r*row_stride (elements), V per row
 *   pick        int32 [R]: lowest id holding the row's largest value (-0 and
 *               +0 are equal); -1 when the row is flagged
 *   flag        uint8 [R]: 1 if the row holds a NaN, +Inf or -Inf, else 0
 * Needs no table. R == 0 is a no-op. Errors: TF_EINVAL (null, V < 1,
 * row_stride < V), TF_ERANGE (V > 2^30, R > 2^24). Rows are read with 16-byte
 * vector loads when logits and row_stride allow it. One launch takes at most
 * 65,535 rows (the grid's y extent); larger R runs as several launches. */
int tf_argmax_rows(const void* logits, int R, int V, int64_t row_stride,
                   int32_t* pick, uint8_t* flag, tf_cuda_stream stream);

/* a5. Greedy verify of every stream: the accepted-draft prefix length
 * ([DSP]: the target verifies every draft; [SRD] verifyFn takes the pick
 * for greedy rows, flagged rows are drawn on the host).
 *   ids         int32 [R]: row 0 of a window is the pending token, rows 1..
 *               the drafts
 *   pick, flag  from tf_argmax_rows
 *   vocab       draft ids outside [0, vocab) never match
 *   accept_len  int32 [S]: a = leading drafts j+1 with pick[j] == ids[j+1]
 *               and row j unflagged (0 <= a <= rows-1)
 *   next_token  int32 [S]: pick of row a, or -1 when row a is flagged
 *   new_keys    int32 [S]: keys - rows + a + 1
 *   sflag       uint8 [S]: bit 0 row a flagged (host draws), bit 1 a draft id
 *               of the window lies outside [0, vocab)
 *   rewind_conv nonzero: rewrite every conv layer's state of every stream with
 *               rows > 1 to history rows a+1, a+2 (the state after row a);
 *               needs the table's conv_hist
 * Errors: TF_EINVAL (null outputs; rewind without histories). */
int tf_accept(const tf_segments* seg, const int32_t* ids, const int32_t* pick,
              const uint8_t* flag, int vocab, int32_t* accept_len,
              int32_t* next_token, int32_t* new_keys, uint8_t* sflag,
              int rewind_conv, tf_cuda_stream stream);

/* The drafter's Markov head over the draft rows of a verify table ([DSP]
 * lfm2_markov_scan / lfm2_markov_pick). Stream s drafts rows_s - 1 tokens;
 * its block rows are packed stream after stream at draft row o_s - s (o_s its
 * window's row offset), R - S rows in all. Block row j of stream s scores
 *   score[v] = bf16(base[v] + bf16(W2[v] . W1[tok]))     (v < vocab)
 * with tok = prev[s] for j = 0 and the pick of row j-1 after that (the rows in
 * sequence); the dot accumulates in fp32 on the tensor cores and is
 * rounded to nearest even, as is the sum. The pick is the lowest token with
 * the largest score.
 *   W1, W2      bf16 [vocab][TF_MK]
 *   base        bf16 logits, draft row k at base + k*base_stride (elements)
 *   prev        int32 [S]: each stream's pending token
 *   pick        int32 [R - S]: the row's pick, -1 when flagged
 *   flag        uint8 [R - S]: bit 0 a nonfinite score in the row, or no
 *               valid previous token (outside [0, vocab), e.g. a flagged row
 *               before it); bit 1 the kernel gave up waiting for its own
 *               copies or MMAs (more than 2 s; the row is not computed)
 * Tables of at most 128 streams run the whole chain in one cooperative launch
 * (one CTA per SM, all resident; the CTAs meet between steps, every wait
 * bounded) after a 16-byte memset of the table's step barrier; larger tables
 * (or TF_MARKOV_PATH=step) take one launch per step (rows_max - 1 launches).
 * Either way W2 is read once a step for up to 128 streams. The table holds the
 * cross-CTA scratch: calls on one table must not overlap on the GPU. Errors: TF_EINVAL (null, misaligned W2 or base,
 * base_stride < vocab or not a multiple of 8, vocab < 1), TF_ERANGE
 * (vocab > 2^24). */
int tf_markov_chain(const tf_segments* seg, const void* W1, const void* W2, int vocab,
                    const void* base, int64_t base_stride, const int32_t* prev,
                    int32_t* pick, uint8_t* flag, tf_cuda_stream stream);

/* The next verify's ids from each stream's pending token and the drafter's
 * picks ([DSP] lfm2_draft_ids, on the GPU so that the host reads no pick
 * between the drafter and the verify). Window row 0 of stream s is prev[s];
 * window row j >= 1 is the draft at packed draft row o_s - s + j - 1 (the
 * layout tf_markov_chain writes). A token outside [0, vocab), or a draft whose
 * draft_flag is nonzero, is written as -1 (the verify never accepts it).
 *   prev        int32 [S] (e.g. tf_accept's next_token)
 *   drafts      int32 [R - S]; may be NULL when every window has one row
 *   draft_flag  uint8 [R - S] or NULL
 *   ids         int32 [R]: the verify's ids
 *   dflag       uint8 [S]: bit 0 (TF_DFLAG_BAD_PENDING) the pending token was
 *               bad, bit 1 (TF_DFLAG_BAD_DRAFT) a draft was bad
 * Errors: TF_EINVAL (null, vocab < 1). */
#define TF_DFLAG_BAD_PENDING 1
#define TF_DFLAG_BAD_DRAFT   2
int tf_draft_ids(const tf_segments* seg, const int32_t* prev, const int32_t* drafts,
                 const uint8_t* draft_flag, int vocab, int32_t* ids, uint8_t* dflag,
                 tf_cuda_stream stream);

/* A prompt (prefill) call of one stream ([SRD]: prompt calls and windows of a
 * single stream still take the per-stream launches; those kernels run them in their own
 * 16-row tiles, here 32-row windows, which fill a 128-lane tensor-core tile
 * with their 4 query heads per KV head):
 * `rows` new rows (row 0 first) whose K/V are already in the cache, so the
 * cache holds `keys` entries in all (keys >= rows). The returned table serves
 * tf_conv_rows (the rows in order with the stream's conv state; no history)
 * and the attention calls (tf_attn, tf_attn_partials + tf_attn_merge,
 * tf_attn_static, tf_partials_bytes): the rows run as windows of
 * W = TF_PROMPT_WINDOW_ROWS rows (the last may be shorter), window t seeing
 * its causal count keys - rows + W*t + i + 1 for its row i, all reading the
 * one cache.
 *   conv_state  [n_conv] -> bf16 [2][TF_H], updated in place
 *   k_cache, v_cache [n_attn] -> bf16 [TF_NKV][kv_capacity][TF_D]
 * The conv input, queries and outputs are [rows][...] as in the verify calls.
 * tf_accept, tf_draft_ids and tf_markov_chain refuse a prompt table.
 * Errors: TF_EINVAL (null/misaligned/overlapping buffers, rows < 1,
 * keys < rows, kv_capacity < keys), TF_ERANGE (rows > TF_MAX_PROMPT_ROWS,
 * kv_capacity > TF_MAX_KEYS), TF_ENOMEM, TF_ECUDA. Free with tf_segments_free. */
int tf_prompt_build(int32_t rows, int32_t keys, int32_t kv_capacity,
                    const void* const* conv_state, const void* const* k_cache,
                    const void* const* v_cache, int n_conv, int n_attn,
                    tf_cuda_stream stream, tf_segments** out);

/* ---- failures on the device ------------------------------------------------
 * The tensor-core attention kernel (tf_attn*, streams of 9 rows or more and
 * prompt windows) and the Markov chain (tf_markov_chain) wait on barriers
 * that other warps or CTAs of the same launch complete. Every such wait is
 * bounded by the wait limit below. A CTA whose wait runs out gives up: it
 * lets its own copies and MMAs in flight land, writes NaN in place of the
 * results it could not compute (attention records; Markov rows get pick -1
 * and flag bit 1), sets a bit in the table's status word and returns. Nothing
 * faults and the context stays usable; the launch itself still reports
 * success, so the failure is read with tf_segments_status (the review of
 * the drafter's held path asks that a failure flag of asynchronous work
 * reach the host: PR #1391, its review of the held path).
 *
 * tf_set_wait_limit_ns sets the limit (process-wide) for every later launch;
 * a launch captured in a CUDA graph keeps the limit it was captured with.
 * Default TF_WAIT_LIMIT_DEFAULT_NS (2 s), at most TF_WAIT_LIMIT_MAX_NS
 * (TF_ERANGE beyond). 0 makes a kernel give up at the first wait that is
 * not already complete when first tested: a way to exercise the failure
 * path, not a setting for real work. tf_wait_limit_ns returns the current
 * limit. */
#define TF_WAIT_LIMIT_DEFAULT_NS 2000000000ull
#define TF_WAIT_LIMIT_MAX_NS 60000000000ull
int tf_set_wait_limit_ns(uint64_t ns);
uint64_t tf_wait_limit_ns(void);

/* Status word bits of a table. */
#define TF_STATUS_ATTN_TIMEOUT   1u   /* the tensor-core attention kernel gave up a wait */
#define TF_STATUS_MARKOV_TIMEOUT 2u   /* the Markov chain gave up a wait */

/* Read and clear a table's status word. Synchronises `stream` (so it must not
 * be called during stream capture), copies the word to *bits (if bits is not
 * NULL) and, when it is nonzero, zeroes the table's cross-CTA scratch
 * (attention merge counters, work counters, Markov step keys and barrier) and
 * the word itself, so the next calls on the table start clean. No call on the
 * table may be in flight on another stream meanwhile.
 * Returns TF_OK (no kernel gave up since the last check), TF_ETIMEOUT (one
 * did: every result the table's calls wrote since the last check is invalid),
 * TF_EINVAL (NULL table) or TF_ECUDA. */
int tf_segments_status(tf_segments* seg, tf_cuda_stream stream, uint32_t* bits);

/* Name of a status code. */
const char* tf_strerror(int status);

/* The CUDA error code behind the last TF_ECUDA of this thread (0 if none). */
int tf_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TF_H_INCLUDED */
