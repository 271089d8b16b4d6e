/*
 * ctcpb.h -- C ABI of the GB300-native batched CTC prefix beam search decoder.
 *
 * What it computes ("GPU CTC Prefix Beam Search Decoder", OASR docs):
 *   log_prob[B, T, V] (float32 log-probabilities, label 'blank_id' is the CTC
 *   blank) -> per row the N best collapsed label sequences and their CTC
 *   posterior log-scores, by prefix beam search (section 3): each hypothesis
 *   keeps a blank-ending and a non-blank-ending log-probability (3.1), extends
 *   by every non-blank label through the two paths of 3.2 / 3.4.1, keeps its
 *   blank/stay slot (3.4.2), merges a shorter hypothesis' extension into the
 *   longer hypothesis it equals (3.4.3) and keeps the best `beam` candidates
 *   (3.4.4-3.4.5).  Offline decoding may skip blank-dominant frames (3.5);
 *   streaming decoding carries the beam state across chunks (section 8).
 *
 * Conventions (all calls):
 *   - Every buffer pointer is a DEVICE pointer, allocated and owned by the
 *     caller; the library never allocates or frees memory (section 5).
 *   - log_prob rows are float32 with V contiguous; stride_b / stride_t are in
 *     elements (64-bit, so offsets past 2^31 elements are fine, section 13).
 *   - Calls are asynchronous on `stream` and never synchronise with the host.
 *   - Return value: CTCPB_OK (0) or a negative status for argument errors
 *     found on the host (nothing is launched then).  Conditions found on the
 *     device set bits in a status word inside the workspace / state, read with
 *     ctcpb_read_status().
 *   - Workspace and state buffers must be 256-byte aligned.
 *
 * Arithmetic: float32 with a fixed operation order and the library's own
 * logsumexp, max(a, b) + F(|a - b|) with F(d) = log(1 + e^-d) evaluated from a
 * table of degree-5 Taylor polynomials (96 segments of width 1/4; F = 0 from
 * d = 24 on), so results are reproducible bit for bit on any launch shape.
 */
#ifndef CTCPB_H
#define CTCPB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* ctcpb_stream_t;

/* Host-side status codes. */
#define CTCPB_OK 0
#define CTCPB_EINVAL (-1)   /* a dimension or configuration value is out of range */
#define CTCPB_ENULL (-2)    /* a required pointer is NULL */
#define CTCPB_EALIGN (-3)   /* workspace/state pointer not 256-byte aligned */
#define CTCPB_ESIZE (-4)    /* workspace/state buffer smaller than the size query */
#define CTCPB_ECUDA (-5)    /* a CUDA launch failed (the runtime error is pending) */

/*
 * The coefficient table of the library's logsumexp ("GPU CTC Prefix Beam
 * Search Decoder", section 3: logsumexp(a, b) = max + log(1 + exp(-|a - b|))).
 * log(1 + e^-d) is evaluated on 96 segments [k/4, (k+1)/4) by the degree-5
 * Taylor polynomial about the segment midpoint k/4 + 1/8 (zero for d >= 24);
 * entry 6k + n is the n-th coefficient of segment k, the float32 rounding of
 * the n-th derivative over n!.  Writes the first min(n, 576) entries to the
 * HOST buffer `out` and returns 576 (the table's size), so callers and tests
 * can check the arithmetic the kernels use; negative on a bad argument.
 */
int ctcpb_lse_table(float* out, int n);

/* Device-side status bits (ctcpb_read_status). */
#define CTCPB_DEV_HEADER 0x1u   /* state header does not match the call's dims/config: call skipped */
#define CTCPB_DEV_PAGES 0x2u    /* paged token pool exhausted: the beam kept its prefix (section 13) */
#define CTCPB_DEV_TIMEOUT 0x4u  /* a bounded inter-block wait gave up: results of the call are invalid */
#define CTCPB_DEV_OVERFLOW 0x8u /* an internal candidate buffer overflowed: results are invalid */
#define CTCPB_DEV_BOOST 0x10u   /* a label-boost entry was rejected and ignored (see ctcpb_boost) */

/*
 * Decoder configuration (section 11).
 *   beam             beam width, 1..128 (MAX_BEAM_SIZE of section 11).
 *   nbest            hypotheses returned per row, 1..beam.
 *   blank_id         CTC blank label, 0..V-1.
 *   max_seq_len      cap on labels per hypothesis; a hypothesis at the cap has
 *                    no non-blank extension (section 11).  <= 0 selects the
 *                    default: T offline (never binds), 4096 when streaming.
 *   blank_threshold  offline frame skip (section 3.5): frame t is decoded iff
 *                    log_prob[b,t,blank] < log(blank_threshold); >= 1 keeps all
 *                    frames, <= 0 keeps none (section 13).  Ignored when
 *                    streaming.  Must not be NaN.
 *   paged            0: flat double-buffered token rows (section 7, "Flat");
 *                    1: paged, prefix-shared, reference-counted pages (4.2, 7).
 *   page_size        labels per page in paged mode, 1..1024 (section 11: 16).
 *   list_len         labels ranked per frame by the vocabulary pre-pass; 0
 *                    selects min(2*beam+2, V-1) (section 3.4.7).  Any value in
 *                    1..V-1 gives the same decode: when a frame's list cannot
 *                    prove the selection, that step re-ranks the whole frame.
 *   word_boundary    0: no word-boundary label (a zero-initialised config);
 *                    1: space_id is the model's word-boundary ("space") label
 *                    (sections 3.4.1/3.4.2): its extension always takes
 *                    lp[space] + lse(pb, pnb), so every space frame is a token
 *                    of its own, and a space-ending beam has no stay path.
 *   space_id         the word-boundary label, 0..V-1 (no effect when it equals
 *                    blank_id); ignored when word_boundary is 0.
 *   max_boost        0: no label boosting.  1..4096: every row (utterance or
 *                    stream) may boost up to max_boost labels (ctcpb_boost);
 *                    the workspace / state then holds a label-boost hash table
 *                    per row, and the decode runs kernel instantiations that
 *                    read it (the plain ones carry no boosting code).
 */
typedef struct ctcpb_config {
  int32_t beam;
  int32_t nbest;
  int32_t blank_id;
  int32_t max_seq_len;
  float blank_threshold;
  int32_t paged;
  int32_t page_size;
  int32_t list_len;
  int32_t word_boundary;
  int32_t space_id;
  int32_t max_boost;
} ctcpb_config;

/*
 * Label boosting: the per-utterance word-boosting table of "GPU-Accelerated
 * WFST Beam Search Decoder for CTC-based Speech Recognition" (one hash table
 * per utterance, consulted whenever an output label is emitted), applied to
 * CTC labels at the extension point the decoder page names in section 15
 * (scores added to the extension table before the top-K).  A label c that an
 * extension emits -- including the repeat after a blank -- scores
 * lp'[c] = lp[c] + bonus[c] (float32, clamped at -FLT_MAX) in place of
 * lp[c]: in the per-frame label ranking (so step 0 seeds by lp'), in the
 * section 3.4.1 extensions and in the 3.4.3 merge folds.  The blank and the
 * stay path emit no label and keep lp.  Without pruning a prefix scores its
 * CTC log-posterior plus the sum of its labels' bonuses; a positive bonus
 * favours the label, a negative one penalises it.
 *
 * The table of every row is given in compressed-row form, all DEVICE arrays:
 *   row_ptr  [B + 1] int32: row b's entries are [row_ptr[b], row_ptr[b+1])
 *   tokens   [row_ptr[B]] int32: the boosted labels
 *   bonus    [row_ptr[B]] float32: their bonuses
 * Entries are taken in order.  One is rejected -- ignored, with
 * CTCPB_DEV_BOOST set in the device status -- when its label is outside
 * [0, V) or is the blank, repeats an earlier label of the row, its bonus is
 * not finite or exceeds 1e6 in magnitude, or the row already holds max_boost
 * labels; a row whose offsets decrease is ignored whole.
 */
typedef struct ctcpb_boost {
  const int32_t* row_ptr;
  const int32_t* tokens;
  const float* bonus;
} ctcpb_boost;

/*
 * Diagnostic counters of the last call on a workspace or state (synchronises
 * the device): [0] decode steps, [1] steps whose first candidate set could not
 * prove the selection, [2] steps that fell back to an exhaustive selection
 * (warp kernel: over the frame's list; block kernel: the chunked sort of every
 * candidate), [3] steps that also scored every unlisted label of the frame,
 * [4] merges proposed by prefix hashes and confirmed on stored tokens, [5]
 * launches that ran the pre-pass and the steps of a tile as one cooperative
 * kernel (CTCPB_NO_FUSE=1 in the environment makes every call use two kernels
 * instead).
 */
int ctcpb_read_counters(const void* ws_or_state, uint32_t counters[6]);

/* Human-readable text for a host status code. */
const char* ctcpb_status_string(int status);

/*
 * Workspace bytes for ctcpb_decode_offline on [B, T, V] (section 5,
 * calculate_[paged_]workspace_size).  Writes *bytes; returns a status.
 */
int ctcpb_workspace_size(const ctcpb_config* cfg, int B, int T, int V, size_t* bytes);

/*
 * Offline decode (section 3.7 / 12.1, ctc_beam_search_decode[_paged]).
 *   log_prob      [B, T, V] float32, element strides stride_b, stride_t (>= V).
 *   seq_lengths   [B] int32 valid frames per row (values clamped to [0, T]);
 *                 NULL means T for every row.  Frames t >= len_b are never read.
 *   ws, ws_bytes  workspace of at least ctcpb_workspace_size() bytes; its
 *                 contents need no initialisation and are overwritten.
 *   out_tokens    [B, nbest, out_len] int32: labels of each hypothesis, padded
 *                 with -1; a hypothesis longer than out_len is cut (its length
 *                 still reports the full count, section 13).
 *   out_lengths   [B, nbest] int32;  out_scores [B, nbest] float32.
 *   Hypotheses are ordered by score (descending); a row with fewer live
 *   hypotheses than nbest has dead slots (length 0, score -FLT_MAX, tokens -1);
 *   a row with no decoded frame returns the empty hypothesis with score 0 in
 *   slot 0 (section 13).  B == 0 is a no-op.
 */
int ctcpb_decode_offline(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                         const int32_t* seq_lengths, int B, int T, int V, void* ws, size_t ws_bytes,
                         int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                         ctcpb_stream_t stream);

/*
 * ctcpb_decode_offline with label boosting (ctcpb_boost): row b of the batch
 * boosts the labels of boost's row b.  Requires cfg->max_boost >= 1.  A NULL
 * boost is ctcpb_decode_offline.  Errors: CTCPB_EINVAL when max_boost is 0,
 * CTCPB_ENULL for a NULL row_ptr, tokens or bonus, otherwise as
 * ctcpb_decode_offline.
 */
int ctcpb_decode_offline_boosted(const ctcpb_config* cfg, const ctcpb_boost* boost, const float* log_prob,
                                 int64_t stride_b, int64_t stride_t, const int32_t* seq_lengths, int B, int T,
                                 int V, void* ws, size_t ws_bytes, int32_t* out_tokens, int32_t* out_lengths,
                                 float* out_scores, int out_len, ctcpb_stream_t stream);

/*
 * Offline decode of a batch that lives in HOST memory, results written to
 * host memory: the only call of this header whose data pointers are host
 * pointers (the workspace is device memory, as everywhere).  The frames go
 * to the device in chunks (whole 64-frame tiles, at least 1 MB of each row)
 * on the library's own copy stream (valid frames only: row b's first
 * seq_lengths[b]), while `stream` decodes every chunk already there; the
 * results come back on `stream`.  The output
 * is exactly ctcpb_decode_offline's on the same frames.
 *   log_prob      host [B, T, V] float32, element strides stride_b, stride_t.
 *   seq_lengths   host [B] int32, or NULL (T for every row).
 *   ws, ws_bytes  DEVICE workspace of ctcpb_host_workspace_size() bytes
 *                 (its size depends on out_len).
 *   out_tokens / out_lengths / out_scores   host, the layout of
 *                 ctcpb_decode_offline.
 * Asynchrony: with page-locked log_prob, seq_lengths and outputs the call
 * returns once everything is enqueued and completes on `stream` (synchronise
 * it before reading the outputs); pageable buffers make CUDA stage the copies
 * and the call may block.  The host buffers must stay valid until `stream`
 * completes.  Calls are serialised on each device (a lock guards the copy
 * stream and its events).
 */
int ctcpb_host_workspace_size(const ctcpb_config* cfg, int B, int T, int V, int out_len, size_t* bytes);
int ctcpb_decode_offline_host(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                              const int32_t* seq_lengths, int B, int T, int V, void* ws, size_t ws_bytes,
                              int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                              ctcpb_stream_t stream);

/* The same with label boosting (ctcpb_boost: DEVICE arrays, as in
 * ctcpb_decode_offline_boosted; requires cfg->max_boost >= 1). */
int ctcpb_decode_offline_host_boosted(const ctcpb_config* cfg, const ctcpb_boost* boost, const float* log_prob,
                                      int64_t stride_b, int64_t stride_t, const int32_t* seq_lengths, int B, int T,
                                      int V, void* ws, size_t ws_bytes, int32_t* out_tokens, int32_t* out_lengths,
                                      float* out_scores, int out_len, ctcpb_stream_t stream);

/*
 * Offline decode for callers that cannot allocate device memory.  The pages
 * have no counterpart.  It is for code that may not call cudaMalloc: a plugin
 * of an engine that owns the device heap and forbids allocations from outside
 * it, or a real-time path that must not block in the allocator.  Same
 * arguments and results as ctcpb_decode_offline without the workspace: the
 * workspace is a fixed device array of CTCPB_NOALLOC_SCRATCH_BYTES inside this
 * library, held by every device that loads the library until the process
 * exits.
 *   - Returns CTCPB_ESIZE when the problem's workspace (ctcpb_workspace_size)
 *     exceeds CTCPB_NOALLOC_SCRATCH_BYTES; nothing is launched then.
 *   - Calls no allocator.  The first call on each device looks up the array's
 *     device address (cudaGetSymbolAddress) with that device current, and
 *     keeps it for the process.  The kept address does not survive
 *     cudaDeviceReset: do not use this call on a device after resetting it.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents (each call resets what it reads before reading it).  Calls
 *     whose work overlaps on the GPU (different streams, or several host
 *     threads) race and corrupt each other's results.  Serialise them, e.g. on
 *     one stream.
 *   - ctcpb_noalloc_read_status reads the array's device status word (the
 *     CTCPB_DEV_* bits of the last call on the current device, as
 *     ctcpb_read_status does for a workspace).  It synchronises the device.
 */
#define CTCPB_NOALLOC_SCRATCH_BYTES (32u << 20)
int ctcpb_decode_offline_noalloc(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                                 const int32_t* seq_lengths, int B, int T, int V, int32_t* out_tokens,
                                 int32_t* out_lengths, float* out_scores, int out_len, ctcpb_stream_t stream);
int ctcpb_noalloc_read_status(uint32_t* device_status);

/*
 * Streaming state bytes for B independent streams of vocabulary V (section 5,
 * calculate_[paged_]state_buffer_size).  The state holds each stream's beam,
 * its label storage and its step/frame counters (section 4.3).
 */
int ctcpb_state_size(const ctcpb_config* cfg, int B, int V, size_t* bytes);

/*
 * Reset a streaming state (section 8, init_streaming_state[_paged]): every
 * stream starts before its first frame.  The state is position independent
 * (offsets, not pointers), so it may be copied with cudaMemcpy and resumed.
 */
int ctcpb_stream_init(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                      ctcpb_stream_t stream);

/*
 * Set the label boosts of every stream of a state (ctcpb_boost; requires
 * cfg->max_boost >= 1): they replace the streams' previous boosts and apply
 * from the next decoded frame on (ctcpb_stream_init clears them).  Errors:
 * CTCPB_EINVAL when max_boost is 0, CTCPB_ENULL for a NULL boost, row_ptr,
 * tokens or bonus, otherwise as ctcpb_stream_step_chunk.
 */
int ctcpb_stream_set_boost(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                           const ctcpb_boost* boost, ctcpb_stream_t stream);

/*
 * Decode one chunk of frames for every stream (section 8, ctc_beam_search_chunk).
 *   lp_chunk   [B, chunk_T, V] float32 with element strides stride_b, stride_t.
 *   n_frames   [B] int32 device array: stream b decodes its first n_frames[b]
 *              rows of the chunk (values clamped to [0, chunk_T]); NULL means
 *              chunk_T for every stream.
 * Streaming never skips frames (section 3.5).  The step and frame counters
 * live in the state on the device.  Decoding a stream in any chunking gives
 * the same result as decoding its frames offline without skipping.
 */
int ctcpb_stream_step_chunk(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                            const float* lp_chunk, int64_t stride_b, int64_t stride_t, const int32_t* n_frames,
                            int chunk_T, ctcpb_stream_t stream);

/*
 * ctcpb_stream_step_chunk with a speech mask (section 8's is_speech_mask of
 * ctc_beam_search_chunk; sections 14 and 15: frames marked as non-speech
 * bypass the decoder).
 *   is_speech    [B, chunk_T] uint8 device array, row stride mask_stride
 *                (>= chunk_T): frame j of stream b is decoded iff
 *                is_speech[b * mask_stride + j] != 0.
 * A masked frame still advances the stream's frame counter; the decoder
 * treats it like a frame skipped by the blank threshold (section 3.5): the
 * next decoded frame collapses the beam's blank-ending residue (section 3.4).
 * Decoding a stream in any chunking gives the same result as decoding its
 * frames offline with the same mask.  Errors: CTCPB_ENULL for a null mask,
 * CTCPB_EINVAL for mask_stride < chunk_T, otherwise as ctcpb_stream_step_chunk.
 */
int ctcpb_stream_step_chunk_masked(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                                   const float* lp_chunk, int64_t stride_b, int64_t stride_t,
                                   const int32_t* n_frames, const uint8_t* is_speech, int64_t mask_stride,
                                   int chunk_T, ctcpb_stream_t stream);

/*
 * Decode one frame for every stream (section 9, ctc_beam_search_step: one
 * streaming frame).
 *   lp_frame   [B, V] float32, row stride stride_b (>= V) elements.
 *   is_speech  [B] uint8 device array or NULL: stream b decodes the frame iff
 *              is_speech[b] != 0; NULL decodes it for every stream.  A stream
 *              whose flag is 0 still advances its frame counter, like a masked
 *              frame of ctcpb_stream_step_chunk_masked: this is how a caller
 *              that drops frames marks the gap that the pages' step call takes
 *              as actual_frame_index.
 * The same as ctcpb_stream_step_chunk (ctcpb_stream_step_chunk_masked when
 * is_speech is given) with chunk_T = 1, and with the same errors.
 */
int ctcpb_stream_step(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                      const float* lp_frame, int64_t stride_b, const uint8_t* is_speech, ctcpb_stream_t stream);

/*
 * Write the current N best of every stream (section 8, read_streaming_results)
 * in the output layout of ctcpb_decode_offline.  Does not modify the state.
 */
int ctcpb_read_state(const ctcpb_config* cfg, const void* state, size_t state_bytes, int B, int V,
                     int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                     ctcpb_stream_t stream);

/*
 * Self-test of the bounded waits (failure detection without a GPU fault).
 * One warp runs the two forms of wait the kernels use against conditions
 * that never complete, and gives up as the kernels do:
 *   flags      [nflags] uint32 device array: ready flags acquired up to 32 at
 *              a time, as the fused launch waits for ranked records; the wait
 *              stops at the first flag still 0 after max_spins tries
 *              (1 <= max_spins <= 2^20, about 100 ns a try);
 *   then an mbarrier phase that expects two arrivals and gets one, waited on
 *   with the pre-pass's bounded barrier wait (under a second).
 *   out        [3] uint32 device array: out[0] = flags found set in order,
 *              out[1] = CTCPB_DEV_TIMEOUT if the flag wait gave up, out[2] =
 *              CTCPB_DEV_TIMEOUT if the barrier wait gave up (it always does).
 * Asynchronous on `stream`; the context stays usable.  Errors: CTCPB_EINVAL
 * for nflags < 0 or max_spins out of range, CTCPB_ENULL for a NULL out (or
 * NULL flags with nflags > 0), CTCPB_ECUDA for a failed launch.
 */
int ctcpb_selftest_waits(const uint32_t* flags, int nflags, long long max_spins, uint32_t* out,
                         ctcpb_stream_t stream);

/*
 * Copy the device status word of a workspace or state to *device_status.
 * Synchronises the device (for tests and error reporting, not the hot path).
 */
int ctcpb_read_status(const void* ws_or_state, uint32_t* device_status);

/* ---- Stage entry points (the steps of the hot path, exposed for testing
 * and per-kernel timing). */

/* Stages of ctcpb_decode_offline, in launch order. */
#define CTCPB_STAGE_INIT 0x1u    /* reset the workspace's per-row state (section 3.7) */
#define CTCPB_STAGE_SELECT 0x2u  /* frame selection (section 3.5) */
#define CTCPB_STAGE_RANK 0x4u    /* vocabulary pre-pass of every kept frame (section 3.4.7) */
#define CTCPB_STAGE_STEPS 0x8u   /* all decode steps of every row (sections 3.3-3.4) */
#define CTCPB_STAGE_OUTPUT 0x10u /* N-best gather (section 3.6) */
#define CTCPB_STAGE_ALL 0x1fu

/*
 * ctcpb_decode_offline restricted to the stages in stage_mask, on the same
 * workspace and with the same arguments.  Running the five stages in order,
 * in one call or several, is exactly ctcpb_decode_offline; a stage reads what
 * the earlier stages left in the workspace.
 */
int ctcpb_decode_offline_staged(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                                const int32_t* seq_lengths, int B, int T, int V, void* ws, size_t ws_bytes,
                                int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                                uint32_t stage_mask, ctcpb_stream_t stream);

/* Number of labels the pre-pass ranks per frame for this config and V (>= 1),
 * or a negative status for an invalid config. */
int ctcpb_list_len(const ctcpb_config* cfg, int V);

/*
 * Frame selection (section 3.5): sel [B, T] int32 receives the kept frames of
 * each row in order (the rest of the row is -1), nsel [B] their count.  The
 * frames, lengths and threshold are read as in ctcpb_decode_offline.  Errors:
 * CTCPB_EINVAL for B or T < 0 or a stride below V, CTCPB_ENULL for a NULL
 * nsel (or log_prob or sel with T > 0); B == 0 is a no-op.
 */
int ctcpb_select_frames(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                        const int32_t* seq_lengths, int B, int T, int V, int32_t* sel, int32_t* nsel,
                        ctcpb_stream_t stream);

/*
 * Vocabulary pre-pass (section 3.4.7) over R frame rows (row r at
 * log_prob + r * stride_r): the first L = list_len non-blank live labels by
 * (log-prob desc, label asc) -> ids [R, L] int32 / lps [R, L] float32 (padded
 * with -1 / -FLT_MAX), cnt [R], the blank log-prob lpb [R], and the next
 * ranked label after the list (front_id [R], front_lp [R]; -1 / -FLT_MAX when
 * none).  A label is live iff its log-prob is > -FLT_MAX (NaN and -inf are
 * read as -FLT_MAX).  Errors: CTCPB_EINVAL for R < 0 or stride_r < V,
 * CTCPB_ENULL for any NULL array; R == 0 is a no-op.
 */
int ctcpb_topk_prepass(const ctcpb_config* cfg, const float* log_prob, int64_t stride_r, int R, int V,
                       int32_t* ids, float* lps, int32_t* cnt, float* lpb, float* front_lp, int32_t* front_id,
                       ctcpb_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CTCPB_H */
