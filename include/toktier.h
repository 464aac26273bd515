/*
 * toktier.h - C ABI of the exact full-context BPE tokenizer for GB300 (sm_103a).
 *
 * The library computes, for every request of a batch, the token IDs of
 * GPT-family regex pre-tokenization followed by byte-level BPE, bit-identical
 * to a sequential reference tokenizer.  It is the GPU full path for session
 * initialisation / rebuild described in "TokTier: Exact Stateful CPU+GPU
 * Tokenization for Agentic LLM Serving" (arXiv 2607.29678):
 *   - §4.1 run decomposition: UTF-8 decode, four character classes, maximal
 *     same-class runs, and a per-character piece-start predicate from run
 *     offset, bounded lookback and per-run aggregates obtained by prefix
 *     scans;
 *   - §4.2 segmented BPE: per-piece merging by lowest rank, the whole-piece
 *     vocabulary shortcut (ignore_merges), length-dispatched execution units;
 *   - §4.3 batching: documents are concatenated and runs are cut at document
 *     boundaries; counts stay in device memory; output compaction.
 *
 * Conventions for every call:
 *   - Device pointers ("d_" prefix) are CUDA global-memory addresses on the
 *     current device; host pointers are ordinary memory.  The library never
 *     takes ownership of a caller's buffer and never keeps a pointer to one
 *     after the call returns (device buffers are used by work enqueued on
 *     `stream`, so they must stay valid until that work completes).
 *   - A batch is `n_requests` UTF-8 byte strings stored back to back:
 *     request r is bytes [byte_offsets[r], byte_offsets[r+1]) of the byte
 *     buffer.  byte_offsets has n_requests + 1 non-decreasing entries, the
 *     first >= 0.  Empty requests are allowed.  A batch holds fewer than
 *     2^29 - 64 bytes (byte_offsets[n] - byte_offsets[0]); larger batches are
 *     rejected with TT_ERR_CAPACITY.
 *   - Output IDs are int32, concatenated per request: request r owns
 *     out_ids[out_id_offsets[r] - out_id_offsets[0] ...).  out_id_offsets is
 *     int64 with n_requests + 1 entries and out_id_offsets[0] = 0.  A request
 *     never yields more IDs than bytes, so an output buffer of
 *     byte_offsets[n] - byte_offsets[0] entries is always large enough.
 *   - A request that is not valid UTF-8 (RFC 3629: no overlongs, surrogates,
 *     code points above U+10FFFF, stray or missing continuation bytes) is
 *     rejected: it yields zero IDs, and the batch's device status records
 *     TT_ERR_INVALID_UTF8 with the lowest rejected request index (read it with
 *     tt_get_status).  Other requests are unaffected.
 *   - Calls are asynchronous with respect to the host unless stated: they
 *     enqueue work on `stream` and return.  Argument errors are returned
 *     immediately; errors found by the kernels (invalid UTF-8, a capacity
 *     bound exceeded, a bounded device wait that ran out) are recorded in a
 *     device status word owned by the handle and read with tt_get_status.
 *     A batch larger than its stated bound, or one whose bounded device wait
 *     ran out, yields zero IDs for every request (out_id_offsets all 0) and
 *     writes nothing to out_ids: IDs are exact or absent, never approximate
 *     (the paper's output contract, TokTier §4.1 and §4.4: a fallback may
 *     change latency, never the returned IDs).
 *   - A handle may be used from several host threads on different streams;
 *     each stream gets its own device workspace.  Calls on the same stream
 *     are ordered by the stream.
 */
#ifndef TOKTIER_H
#define TOKTIER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tt_stream_t;   /* the same type as cudaStream_t; NULL = legacy default stream */
typedef struct tt_tokenizer tt_tokenizer;

typedef enum {
  TT_OK = 0,
  TT_ERR_INVALID_ARG = 1,   /* a pointer, size or offset array violates this header */
  TT_ERR_BAD_VOCAB = 2,     /* vocabulary / merge list rejected by tt_create (see there) */
  TT_ERR_BAD_FAMILY = 3,    /* unknown pattern family */
  TT_ERR_INVALID_UTF8 = 4,  /* at least one request was not valid UTF-8 (device status) */
  TT_ERR_CAPACITY = 5,      /* the batch exceeds a stated bound (device status or immediate) */
  TT_ERR_OOM = 6,           /* a device or host allocation failed */
  TT_ERR_CUDA = 7,          /* a CUDA runtime call failed */
  TT_ERR_TIMEOUT = 8        /* a bounded device-side wait ran out (device status) */
} tt_status;

typedef enum {
  /* letters / numbers 1..3 / other / whitespace with lookahead; contractions
   * 's 't 're 've 'm 'll 'd (ASCII case-insensitive) as their own pieces */
  TT_FAMILY_CL100K_STYLE = 1,
  /* letter pieces split on case (upper* lower+ | upper+ lower*), marks count
   * as letters, contractions attach to the preceding letters */
  TT_FAMILY_O200K_STYLE = 2,
  /* three splitters in sequence, each re-splitting every piece of the one
   * before and keeping the text between its matches as pieces (TokTier §4.1
   * on DeepSeek-family tokenizers): digit groups of 1..3, then runs of
   * Hiragana / Katakana / CJK Unified Ideographs (U+3040-U+30FF,
   * U+4E00-U+9FFF), then the cl100k-style alternatives without the digit one,
   * with each piece as the whole text (a blank run's lookahead ends at the
   * piece end) */
  TT_FAMILY_DEEPSEEK_STYLE = 3
} tt_pattern_family;

/*
 * tt_create - build a tokenizer handle (synchronous; uses the current device).
 *
 *   merge_pairs   host, int32 [n_merges][2]: merge k joins (left_id, right_id);
 *                 its rank is k (lower rank = applied first).
 *   vocab_bytes   host, the byte strings of all token IDs back to back;
 *   vocab_offsets host, int64 [n_vocab + 1]: token id i is
 *                 vocab_bytes[vocab_offsets[i] .. vocab_offsets[i+1]).
 *   pattern_family one of tt_pattern_family.
 *   out           receives the handle (NULL on failure).
 *
 * The arrays are copied; the caller keeps ownership.  The vocabulary is
 * rejected (TT_ERR_BAD_VOCAB) unless:
 *   - every single byte 0..255 is a token and all byte strings are distinct
 *     and non-empty;
 *   - every merge's operands are valid IDs, the concatenation of their bytes
 *     is a token (the merge's result), no pair appears twice and no result is
 *     produced by two merges;
 *   - the list is well-ordered: a token produced by merge j is used as an
 *     operand only by merges of rank > j.  (Merging every leftmost
 *     non-overlapping occurrence of the lowest-ranked pair in one round equals
 *     iterated single merges only under this condition; §4.2.)
 *   - limits: n_vocab <= 2^20, n_merges <= 2^24 - 1, token length <= 4095.
 * The whole-piece shortcut is always on: a piece whose bytes are a token is
 * emitted as that one ID (ignore_merges, §4.2).
 */
tt_status tt_create(const int32_t *merge_pairs, int64_t n_merges,
                    const uint8_t *vocab_bytes, const int64_t *vocab_offsets, int64_t n_vocab,
                    int32_t pattern_family, tt_tokenizer **out);

/*
 * tt_set_added_tokens - reserve literal strings as single IDs (added and
 * special tokens such as "<|endoftext|>").
 *
 * TokTier §4.4: a leftmost-longest literal pass extracts them before the
 * pattern family handles the remaining segments.  Every later encode of the
 * handle does the same: scanning each request left to right, at the leftmost
 * position where a literal occurs, the longest literal occurring there is cut
 * out as one piece with its ID; the text between literals is pre-tokenized as
 * separate documents (runs are cut at literal boundaries, as at request
 * boundaries) and encoded as usual.  A literal never spans two requests.
 *
 *   literal_bytes    host, the literals concatenated;
 *   literal_offsets  host, int64 [n_literals + 1]: literal k is
 *                    literal_bytes[offsets[k] .. offsets[k+1]);
 *   literal_ids      host, int32 [n_literals]: its reserved ID, distinct,
 *                    >= the handle's n_vocab and < 2^20;
 *   n_literals       0 .. 4095; 0 removes the set.
 * Each literal is 1 .. 255 bytes of valid UTF-8 and no two are equal; else
 * TT_ERR_BAD_VOCAB and the previous set stays.  The arrays are copied.  Call
 * it while no encode of the handle is in flight; the next encode on each
 * stream captures its graph again.  Spans of a literal ID cover its bytes.
 */
tt_status tt_set_added_tokens(tt_tokenizer *h, const uint8_t *literal_bytes, const int64_t *literal_offsets,
                              const int32_t *literal_ids, int64_t n_literals);

/* tt_destroy - release the handle and every device buffer it owns (waits for
 * the handle's outstanding work).  NULL is ignored.  The pages say only that
 * tokenizer entries are immutable after registration (TokTier §4.4), so a
 * handle keeps its tables unchanged from tt_create to this call. */
void tt_destroy(tt_tokenizer *h);

/*
 * tt_encode_batch - tokenize a batch held in device memory.
 *
 * The state-miss full path of TokTier §4.1-§4.3: per request, pre-tokenization
 * by the run rules (§4.1), each piece encoded independently by BPE (§4.2),
 * requests concatenated with runs cut at their boundaries and the IDs
 * compacted in device memory (§4.3).  IDs are delivered as a device array,
 * the delivery the paper's Figure 10(b) measures against Python lists.
 *
 *   d_utf8          device, the batch bytes (see the batch convention above).
 *   d_byte_offsets  device, int64 [n_requests + 1].
 *   n_requests      >= 0; with 0 the call only writes d_out_id_offsets[0] = 0.
 *   d_out_ids       device, int32, capacity >= total bytes of the batch.
 *   d_out_id_offsets device, int64 [n_requests + 1].
 *   stream          CUDA stream for all work.
 *
 * This entry point reads byte_offsets[0] and byte_offsets[n] back to the host
 * (one 16-byte copy and a wait on `stream`) to size the launch; use
 * tt_encode_batch_bounded to stay fully asynchronous.
 */
tt_status tt_encode_batch(tt_tokenizer *h,
                          const uint8_t *d_utf8, const int64_t *d_byte_offsets, int64_t n_requests,
                          int32_t *d_out_ids, int64_t *d_out_id_offsets, tt_stream_t stream);

/*
 * tt_encode_batch_bounded - as tt_encode_batch, without any host wait.
 *
 *   max_total_bytes  host-known upper bound on byte_offsets[n] -
 *                    byte_offsets[0]; the launch geometry and the workspace
 *                    are sized from it, the kernels read the true sizes from
 *                    device memory.  If the batch is larger than this bound
 *                    (even if it would fit the workspace's size bucket),
 *                    nothing is written except a zeroed d_out_id_offsets and
 *                    the device status TT_ERR_CAPACITY, so d_out_ids needs
 *                    room for max_total_bytes IDs only.
 * Work is launched as one CUDA graph per (stream, size bucket): the first
 * call of a bucket captures it (on a private stream), later calls replay it.
 * Buckets are powers of two of max_total_bytes (at least 64 KiB); each
 * (stream, bucket) keeps its own device workspace, about 31 bytes per byte of
 * bucket capacity, until tt_destroy.
 * d_utf8 and d_out_ids may be NULL only if max_total_bytes is 0.
 */
tt_status tt_encode_batch_bounded(tt_tokenizer *h,
                                  const uint8_t *d_utf8, const int64_t *d_byte_offsets, int64_t n_requests,
                                  int64_t max_total_bytes,
                                  int32_t *d_out_ids, int64_t *d_out_id_offsets, tt_stream_t stream);

/*
 * tt_encode_batch_spans - as tt_encode_batch_bounded, and for every ID the
 * source bytes it covers.
 *
 * The paper's session state holds, beside each token ID, the byte span of the
 * text it encodes (TokTier §3, the per-session store; §5.7, Figure 14a: 4 bytes of
 * ID and 8 bytes of span per token), and its GPU full path returns IDs
 * without spans, so a state miss that must build that state falls back to the
 * CPU (§4.4).  This call returns both.
 *
 *   d_out_spans  device, int32 [2 * capacity], capacity as d_out_ids (>= the
 *                batch bytes).  ID i gets (start, end) = d_out_spans[2i],
 *                d_out_spans[2i + 1]: the half-open range of batch bytes it
 *                encodes, as offsets from d_byte_offsets[0] (the batch
 *                start; subtract d_byte_offsets[r] - d_byte_offsets[0] for
 *                offsets within request r).  A request's spans tile its bytes
 *                in order; a rejected request has no IDs and no spans.
 *   other arguments, the graph and the errors as tt_encode_batch_bounded;
 *   d_out_spans may be NULL only if max_total_bytes is 0 (else
 *   TT_ERR_INVALID_ARG).  The caller owns every buffer.
 */
tt_status tt_encode_batch_spans(tt_tokenizer *h,
                                const uint8_t *d_utf8, const int64_t *d_byte_offsets, int64_t n_requests,
                                int64_t max_total_bytes,
                                int32_t *d_out_ids, int64_t *d_out_id_offsets, int32_t *d_out_spans,
                                tt_stream_t stream);

/*
 * tt_encode_batch_noalloc - tokenize a small device batch without allocating.
 *
 * The paper has no counterpart: this exists for callers that must not
 * allocate device memory while they run, e.g. code inside a fixed memory
 * budget or a custom allocator that forbids cudaMalloc/cudaFree after
 * start-up, or latency-critical paths where an allocation would
 * synchronise the device.  tt_encode_batch_bounded may allocate a
 * per-stream workspace on first use or when a batch outgrows it; this entry
 * point never does: its scratch is one fixed array compiled into the
 * library (about 6.4 MB, held on every device that loads the library until
 * the process exits).
 *
 *   Arguments and outputs as tt_encode_batch_bounded; the limits are
 *   max_total_bytes <= TT_NOALLOC_MAX_BYTES and
 *   n_requests <= TT_NOALLOC_MAX_REQUESTS.  Larger values are rejected with
 *   TT_ERR_CAPACITY before anything is enqueued.  A batch whose true size
 *   exceeds max_total_bytes is caught on the device as in the bounded call:
 *   zeroed d_out_id_offsets, nothing written to d_out_ids, device status
 *   TT_ERR_CAPACITY.  The current device must be the handle's.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call on a device shares the one array and leaves its contents
 * behind (each call clears what must start at zero), so calls that overlap
 * on the GPU race: serialise them, e.g. issue them on one stream.  The
 * handle's status word is shared with the other entry points.
 */
#define TT_NOALLOC_MAX_BYTES (256 * 1024)
#define TT_NOALLOC_MAX_REQUESTS 1024
tt_status tt_encode_batch_noalloc(tt_tokenizer *h,
                                  const uint8_t *d_utf8, const int64_t *d_byte_offsets, int64_t n_requests,
                                  int64_t max_total_bytes,
                                  int32_t *d_out_ids, int64_t *d_out_id_offsets, tt_stream_t stream);

/*
 * tt_encode_host - tokenize a batch held in HOST memory (synchronous).
 *
 *   utf8, byte_offsets  host; the batch (byte_offsets[0] may be > 0).
 *   out_ids             host, int32, capacity out_capacity entries.
 *   out_id_offsets      host, int64 [n_requests + 1].
 * Copies the batch to device buffers owned by the handle, encodes it on
 * `stream`, copies the IDs back and waits.  Returns the device status of the
 * batch (TT_OK, TT_ERR_INVALID_UTF8, ...), or TT_ERR_CAPACITY if the IDs do
 * not fit in out_capacity (out_id_offsets is then still filled).  Any host
 * memory works.  When out_ids and out_id_offsets are both page-locked (or
 * managed) memory and out_capacity >= the batch bytes, the kernels write the
 * IDs and offsets into them directly and the call waits once; otherwise the
 * IDs are staged on the device and copied back after the count is read (two
 * waits).  The input is always copied to the device first (page-locked input
 * makes that a plain DMA).
 */
tt_status tt_encode_host(tt_tokenizer *h,
                         const uint8_t *utf8, const int64_t *byte_offsets, int64_t n_requests,
                         int32_t *out_ids, int64_t out_capacity, int64_t *out_id_offsets,
                         tt_stream_t stream);

/*
 * tt_get_status - wait for `stream`, then return and clear the device status
 * recorded by the handle's kernels since the last call (TT_OK if none).
 * *bad_request (may be NULL) receives the lowest rejected request index for
 * TT_ERR_INVALID_UTF8, else -1.  The pages define no status interface; this
 * call carries the paper's output contract (TokTier §4.4: requests that fail
 * a check change latency, never the IDs returned) to a device pipeline whose
 * checks run in the kernels: a failed request has zero IDs and its cause is
 * reported here.
 */
tt_status tt_get_status(tt_tokenizer *h, tt_stream_t stream, int64_t *bad_request);

/*
 * tt_pretokenize_batch - test hook: pre-tokenizer piece boundaries only.
 *
 * TokTier §4.1 checks an implementation at two levels, piece boundaries and
 * final IDs, because a boundary fault can leave the IDs unchanged; this call
 * exposes the first level (the kernels of tt_encode_batch up to the piece
 * table, then a copy of the boundaries).
 *
 *   d_piece_starts   device, int64, capacity >= total bytes of the batch:
 *                    the absolute byte offset (in d_utf8) of every piece
 *                    start, in order.
 *   d_piece_offsets  device, int64 [n_requests + 1]: request r owns entries
 *                    [d_piece_offsets[r], d_piece_offsets[r+1]).
 * A rejected request (invalid UTF-8) reports no pieces.  Same waiting
 * behaviour as tt_encode_batch.
 */
tt_status tt_pretokenize_batch(tt_tokenizer *h,
                               const uint8_t *d_utf8, const int64_t *d_byte_offsets, int64_t n_requests,
                               int64_t *d_piece_starts, int64_t *d_piece_offsets, tt_stream_t stream);

/* tt_status_string - static English text for a status code. */
const char *tt_status_string(tt_status s);

/*
 * tt_profile - per-kernel timing (tracing aid).  enable != 0 makes later
 * encode calls on any stream record CUDA events around each kernel;
 * tt_profile_read waits for the handle's work and returns, per kernel name,
 * the summed milliseconds and launch counts since the last read:
 *   names     host, receives up to `cap` pointers to static kernel names;
 *   ms        host, double [cap];   launches host, int64 [cap].
 * Returns the number of kernels written.  Profiling adds event records
 * between launches and disables graph replay while enabled.
 */
void tt_profile(tt_tokenizer *h, int enable);
int tt_profile_read(tt_tokenizer *h, const char **names, double *ms, int64_t *launches, int cap);

/* tt_launch_count - total kernels launched (directly or inside replayed
 * graphs) by this handle since creation, the argument-staging kernel of
 * tt_encode_batch_noalloc included. */
int64_t tt_launch_count(tt_tokenizer *h);

/* tt_table_digest - SHA-256 (hex, 64 chars + NUL) of the frozen character
 * class table compiled into the library. */
const char *tt_table_digest(void);

/*
 * tt_debug_lookback - test setting for the pre-tokenizer's bounded waits.
 *
 * The pages describe no such setting; it exists so that tests can make a
 * device wait run out without faulting or hanging anything.  The two
 * decoupled look-backs of the pre-tokenizer poll their predecessors' flags at
 * most `spin_limit` times per window (0 restores the default, 2^22); with
 * withhold_tile >= 0, that tile of every later batch publishes nothing, so
 * its successors' waits run out: the batch then yields zero IDs and the
 * device status TT_ERR_TIMEOUT.  withhold_tile = -1 turns this off.  Waits
 * for the handle's outstanding work; later encodes capture their graphs
 * again.  Returns TT_ERR_INVALID_ARG for spin_limit < 0 or withhold_tile < -1.
 */
tt_status tt_debug_lookback(tt_tokenizer *h, int32_t spin_limit, int32_t withhold_tile);

#ifdef __cplusplus
}
#endif

#endif /* TOKTIER_H */
