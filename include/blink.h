/*
 * blink.h -- C ABI of the GB300 (sm_103a) library for the shared-prefix one-pass decision path.
 *
 * Many questions share one prefix (a system prompt plus the evidence).  The prefix KV is held
 * once in a contiguous arena; each question runs only its tail, which attends to the prefix
 * without a mask and to its own tail causally.  The answer is read from the next-token
 * distribution restricted to the offered option labels: the last-token hidden state against
 * the unembedding rows of those labels, then a temperature softmax.  No tokens are generated.
 *
 * Sources (the pages this library restates):
 *   blink.py   -- the "blink-4b" serving module: `_batches`, `_padded`, `_forward`,
 *                 `_forward_shared`, `_read`, `_read_batched`, `softmax`, the limits
 *                 MAX_OPTIONS / MAX_QUESTIONS / MAX_INPUT_TOKENS / TOKEN_BUDGET and the
 *                 PREFIX_CACHE note;
 *   engine.py  -- "simit" backends/mot: the contiguous KV arena and its varlen attention
 *                 metadata (cu_seqlens, per-request region start, keys used).
 *
 * Conventions for every entry point:
 *   - Pointers named d_* and all tensor pointers are DEVICE pointers; h_* are HOST pointers
 *     (pinned memory for asynchronous copies).  The caller owns every buffer; the library
 *     allocates nothing and keeps no state between calls.
 *   - bf16 tensors are passed as `blink_bf16` (16-bit storage of bfloat16 values), row-major.
 *   - Calls are asynchronous on `stream` unless a host output is requested, in which case the
 *     call synchronises the stream before returning.
 *   - Arguments are checked on the host first (BLINK_INVALID_ARG / BLINK_OUT_OF_RANGE, nothing
 *     launched).  Problems only visible on the device (a bad length or label id inside a
 *     device array, a bounded wait that ran out) are latched in a device error word, read back
 *     by the host-output path or by blink_read_device_status().  No kernel traps.
 */
#ifndef BLINK_H
#define BLINK_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t blink_bf16;
typedef int32_t blink_status;

#define BLINK_OK 0
#define BLINK_INVALID_ARG 1          /* malformed argument (null pointer, bad shape, T <= 0 ...) */
#define BLINK_OUT_OF_RANGE 2         /* a limit of the pages is exceeded (options, questions, context) */
#define BLINK_WORKSPACE_TOO_SMALL 3  /* ws_bytes below what the *_workspace() query returned */
#define BLINK_CUDA_ERROR 4           /* a CUDA runtime call failed; cudaGetLastError() has the detail */
#define BLINK_DEVICE_FLAG 5          /* a device-side check failed (bad length, label id, CSR offsets) */
#define BLINK_DEVICE_TIMEOUT 6       /* a bounded wait inside a kernel ran out; outputs are invalid */

/* Limits from blink.py: MAX_OPTIONS, MAX_QUESTIONS, MAX_INPUT_TOKENS.  The planner also takes
 * up to 64 requests of 512 questions at once (blink.py `Batcher.MAX_REQUESTS` packs every
 * question of every request into the same forwards). */
#define BLINK_MAX_OPTIONS 255
#define BLINK_MAX_QUESTIONS 512
#define BLINK_MAX_INPUT_TOKENS 131072
#define BLINK_MAX_PLAN_SEQUENCES 32768

/* A short English description of a status code (a static string). */
const char *blink_status_string(blink_status s);

/* Reads (and, if `clear` != 0, resets) the device error word at the start of a workspace
 * passed to blink_prefix_tail_attention or blink_label_readout.  Synchronises `stream`.
 * Returns BLINK_OK, BLINK_DEVICE_FLAG or BLINK_DEVICE_TIMEOUT (or BLINK_CUDA_ERROR). */
blink_status blink_read_device_status(void *d_ws, int32_t clear, cudaStream_t stream);

/* Self-test of the failure path every kernel relies on (no counterpart on the pages): one
 * thread waits, with the library's bounded wait, on a barrier that nothing arrives at; after
 * limit_us microseconds (1..1000000) the wait gives up and latches BLINK_DEVICE_TIMEOUT in the
 * workspace's error word, exactly as a kernel whose copy or peer never arrived would.  Returns
 * that status (BLINK_DEVICE_TIMEOUT when the path works), after clearing the word.  Nothing
 * faults or traps and the context stays usable.  d_ws: a workspace of at least 256 bytes.
 * Synchronises `stream`. */
blink_status blink_selftest_wait_timeout(uint32_t limit_us, void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Pack plan -- blink.py `_batches` (token-budget packing, shortest first, a forward closes when
 * (longest x count) would pass the padded-token budget or at the row cap; a sequence longer
 * than the budget runs alone) and `_padded` (right padding to each forward's longest).
 *
 * d_lengths [n]        sequence lengths (tails, or whole prompts on the plain path), 1..131072
 * n                    1..BLINK_MAX_PLAN_SEQUENCES
 * budget               padded tokens per forward (blink.py TOKEN_BUDGET = 32768), >= 1
 * max_rows             row cap per forward, 0 = none (blink.py caps rows on the prefix path)
 * Outputs (device, int32; slot s = the s-th sequence in the stable ascending length order):
 *   d_order [n]            sequence index held by slot s
 *   d_slot_of [n]          the inverse: slot holding sequence i (d_slot_of[d_order[s]] == s)
 *   d_fwd_of_slot [n]      forward of slot s
 *   d_fwd_slot_start [n+1] first slot of forward f for f <= n_forwards; n beyond
 *   d_fwd_width [n]        padded width (longest length) of forward f; 0 beyond n_forwards
 *   d_cu_seqlens [n+1]     varlen token offsets of the slots (cu[0] = 0)
 *   d_last_varlen [n]      last token of slot s in the varlen packing: cu[s+1] - 1
 *   d_last_padded [n]      last token of slot s in its forward's padded [rows, width] batch:
 *                          row * width + len - 1
 *   d_n_forwards [1]       number of forwards, or -1 if a length was outside 1..131072
 *   h_n_forwards           optional (may be NULL): the same count copied to pinned host memory;
 *                          when given, the call synchronises the stream.
 * Errors: BLINK_INVALID_ARG (null output, budget < 1, max_rows < 0), BLINK_OUT_OF_RANGE (n),
 * BLINK_DEVICE_FLAG (only with h_n_forwards: a length out of range), BLINK_CUDA_ERROR.
 * Up to 2048 lengths the whole plan is one thread block.  Above that, the stable sort runs over
 * the whole GPU first (blocks sort runs of 1024 keys, then merge rounds), with d_fwd_of_slot and
 * d_last_padded as its two ping-pong buffers; the one-block plan kernel reads the sorted keys
 * before it writes those outputs.  So the planner needs no workspace of its own:
 * blink_pack_plan_workspace() returns 0 for every n.
 * ------------------------------------------------------------------------------------------ */
size_t blink_pack_plan_workspace(int32_t n);

blink_status blink_pack_plan(const int32_t *d_lengths, int32_t n, int32_t budget, int32_t max_rows,
                             int32_t *d_order, int32_t *d_slot_of, int32_t *d_fwd_of_slot, int32_t *d_fwd_slot_start,
                             int32_t *d_fwd_width, int32_t *d_cu_seqlens, int32_t *d_last_varlen,
                             int32_t *d_last_padded, int32_t *d_n_forwards, int32_t *h_n_forwards,
                             cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Shared-prefix length -- blink.py `_shared_prefix_len`: the number of leading tokens common to
 * every sequence, leaving each sequence at least one token of its own (its answer position is
 * computed in the per-question pass); 0 for fewer than two sequences.  blink.py `_forward` takes
 * the shared path only when this is at least PREFIX_MIN_TOKENS (256), a host decision.
 *
 * d_tokens, n_tokens  int32 token ids of all sequences back to back (n_tokens of them); sequence i
 *                     at d_tokens + (d_cu[i] - d_cu[0]) with length d_cu[i+1] - d_cu[i] (>= 1)
 * d_cu [n+1], n       1..BLINK_MAX_PLAN_SEQUENCES sequences
 * d_len [1]           output (device); h_len optional pinned host copy (the call then synchronises)
 * d_ws, ws_bytes      workspace of blink_shared_prefix_len_workspace() bytes (error word)
 * A length below 1 or a sequence past n_tokens latches BLINK_DEVICE_FLAG.
 * ------------------------------------------------------------------------------------------ */
size_t blink_shared_prefix_len_workspace(void);

blink_status blink_shared_prefix_len(const int32_t *d_tokens, int64_t n_tokens, const int32_t *d_cu, int32_t n,
                                     int32_t *d_len, int32_t *h_len, void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * KV rows into the arena -- simit engine.py: one contiguous KV arena with a region per request
 * (`KVArena`, `arena.copy`): the prefix's K/V, computed once, are written into its region, and a
 * cached prefix region can be copied into another request's region.
 *
 * Copies n_rows token rows of row_elems (= Hkv * d, a multiple of 8) bf16 values, for K and V,
 * from k_src / v_src (rows src_row_stride elements apart) to arena rows
 * [dst_slot, dst_slot + n_rows) (rows arena_row_stride elements apart, arena_slots rows in all).
 * Source and destination must not overlap.  Asynchronous on `stream`.
 * Errors: BLINK_INVALID_ARG (null, alignment, strides), BLINK_OUT_OF_RANGE (rows past the arena).
 * ------------------------------------------------------------------------------------------ */
blink_status blink_kv_to_arena(const blink_bf16 *k_src, const blink_bf16 *v_src, int64_t src_row_stride,
                               int64_t n_rows, int32_t row_elems, blink_bf16 *k_arena, blink_bf16 *v_arena,
                               int64_t arena_row_stride, int64_t arena_slots, int64_t dst_slot, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Prefix-tail attention -- blink.py PREFIX_CACHE note and `_forward_shared` (the prefix is
 * encoded once; every tail runs against it: same tokens, same positions, only the
 * floating-point order differs), with the arena layout of simit engine.py.
 *
 * For question b, query head h (kv head h / (Hq/Hkv)) and tail row i:
 *   O = softmax(scale * q . [K_pre ; K_tail_b[0..i]]^T) [V_pre ; V_tail_b[0..i]]
 * i.e. every prefix key without a mask and the question's own tail causally.  The prefix part
 * and the tail part are merged by log-sum-exp.
 *
 * q      [rows, Hq, d]   bf16; question b's tail at rows start_b .. start_b + len_b - 1
 * k_pre  [P, Hkv, d]     bf16; position p's keys at k_pre + p * pre_row_stride (elements), so
 * v_pre                  the prefix may be a region of a wider KV arena; pre_row_stride >= Hkv*d
 *                        and a multiple of 8; 16-byte aligned base.  Unused when P == 0.
 * k_tail, v_tail [rows, Hkv, d] bf16, same rows as q
 * d_cu_seqlens [B+1]     len_b = cu[b+1] - cu[b]; in the varlen layout (d_seq_start == NULL)
 *                        start_b = cu[b] - cu[0], so a slice of a larger cu array can be passed
 *                        together with pointers offset by cu[0] rows
 * d_seq_start [B]        right-padded layout: start_b, strictly increasing, rows not shared;
 *                        rows owned by no question get O = 0 and LSE = -inf
 * B                      1..BLINK_MAX_PLAN_SEQUENCES questions
 * rows                   token rows of q / k_tail / v_tail / out (>= 1)
 * P                      prefix length, 0 (plain causal path) .. 131072
 * max_tail               upper bound of len_b, checked on the device; P and max_tail are each at
 *                        most 131072 (blink.py MAX_INPUT_TOKENS bounds one rendered prompt; the
 *                        largest request keeps a full 131072-token prefix plus its tails)
 * Hq, Hkv, d             Hq % Hkv == 0, Hq/Hkv <= 128, d in {64, 128}
 * scale                  softmax scale; <= 0 selects 1/sqrt(d)
 * out   [rows, Hq, d]    bf16 (round to nearest even)
 * lse   [Hq, rows]       optional (may be NULL): fp32 natural-log log-sum-exp of each row
 * d_ws, ws_bytes         workspace of at least blink_attention_workspace(...) bytes, zero-filled
 *                        before its first use; the first word is the device error word
 * Prefix chunks (one request with a prefix; the work units are (row pair, kv head)): when a
 * launch-time model predicts a clear gain, units run their prefix in chunks of key tiles on
 * separate blocks whose partial outputs are merged by LSE in a second kernel (the merge of the
 * prefix and tail parts, applied again), launched as the attention launch's programmatic
 * dependent on `stream`.  Either every unit is cut (a small grid, e.g. a few questions against
 * a long prefix: chunks of at least 4 tiles), or whole waves of units run unsplit and only the
 * units of the last, partial wave are cut, into chunks that run, in the same launch, on the SMs
 * the whole units free first.  The last chunk of a unit, which also runs its tail tiles, takes
 * fewer prefix tiles.  blink_attention_workspace then includes room for the fp32 partials (it
 * sizes them for the current device); with a smaller workspace the call runs unsplit.  Results
 * agree with the unsplit path within the rounding of the merge.
 * Errors: BLINK_INVALID_ARG, BLINK_OUT_OF_RANGE, BLINK_WORKSPACE_TOO_SMALL, BLINK_CUDA_ERROR;
 * device-side: BLINK_DEVICE_FLAG (a length outside 1..max_tail or past `rows`),
 * BLINK_DEVICE_TIMEOUT.
 * ------------------------------------------------------------------------------------------ */
size_t blink_attention_workspace(int32_t rows, int32_t B, int32_t P, int32_t Hq, int32_t Hkv, int32_t d);

/* The prefix-chunk plan blink_prefix_tail_attention uses for one request of `rows` tail rows
 * against a prefix of P tokens, on a GPU with `sms` SMs, when the workspace has room for it (no
 * device call: for inspection and tests).  Units are (row pair, kv head): with g = Hq / Hkv and
 * 128 / g tokens per 128-row tile, ceil(ceil(rows / (128 / g)) / 2) * Hkv of them.
 * *whole_units  units [0, *whole_units) run whole (all units when nothing is cut)
 * *chunks       chunks each remaining unit is cut into (1: nothing is cut)
 * *chunk_tiles  prefix key tiles (128 keys each) of chunks 0 .. chunks-2; the last chunk takes the
 *               remaining 0 .. *chunk_tiles tiles and the unit's tail tiles (with *chunks = 1:
 *               the whole prefix in tiles)
 * Errors: BLINK_INVALID_ARG (a null output, sms < 1, or a shape the attention call rejects). */
blink_status blink_attention_split_plan(int32_t rows, int32_t P, int32_t Hq, int32_t Hkv, int32_t d, int32_t sms,
                                        int64_t *whole_units, int32_t *chunks, int32_t *chunk_tiles);

blink_status blink_prefix_tail_attention(const blink_bf16 *q, const blink_bf16 *k_pre, const blink_bf16 *v_pre,
                                         int64_t pre_row_stride, const blink_bf16 *k_tail,
                                         const blink_bf16 *v_tail, const int32_t *d_cu_seqlens,
                                         const int32_t *d_seq_start, int32_t B, int32_t rows, int32_t P,
                                         int32_t max_tail, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                         blink_bf16 *out, float *lse, void *d_ws, size_t ws_bytes,
                                         cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Prefix-tail attention over several requests in one launch -- blink.py `logits_many` /
 * `Batcher` (every question of up to 64 requests packed into the same forwards, each request's
 * rows taken only from its own prompts) with simit engine.py's arena (one arena, a region per
 * request).  Request r owns the tail rows [h_req_rows[r], h_req_rows[r+1]) (whole questions
 * only) and attends to its own prefix of h_req_prefix_len[r] tokens at arena slots
 * [h_req_prefix_start[r], + h_req_prefix_len[r]).  Per row the result is exactly that of
 * blink_prefix_tail_attention with the request's prefix.
 *
 * k_arena, v_arena  [arena_slots, Hkv, d] bf16 rows arena_row_stride elements apart
 * n_req             1..64
 * h_req_rows        host [n_req+1], h_req_rows[0] = 0, non-decreasing, h_req_rows[n_req] = rows
 * h_req_prefix_*    host [n_req]; a request with prefix length 0 runs the plain causal path
 * Other arguments and errors as blink_prefix_tail_attention; a question that starts before its
 * request's first row latches BLINK_DEVICE_FLAG.
 * ------------------------------------------------------------------------------------------ */
blink_status blink_prefix_tail_attention_multi(const blink_bf16 *q, const blink_bf16 *k_arena, const blink_bf16 *v_arena,
                                               int64_t arena_row_stride, int64_t arena_slots, const blink_bf16 *k_tail,
                                               const blink_bf16 *v_tail, const int32_t *d_cu_seqlens,
                                               const int32_t *d_seq_start, int32_t B, int32_t rows, int32_t n_req,
                                               const int32_t *h_req_rows, const int32_t *h_req_prefix_start,
                                               const int32_t *h_req_prefix_len, int32_t max_tail, int32_t Hq,
                                               int32_t Hkv, int32_t d, float scale, blink_bf16 *out, float *lse,
                                               void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Label readout -- blink.py `_read` / `_read_batched` (the last hidden state of each question
 * against the lm_head rows of its offered labels only, in FP32), `softmax` (z / T, minus the
 * max, exp, normalise), `decide` (the temperature must be positive) and, optionally,
 * `answer_for` (the typed answer per question).
 *
 * hidden [hidden_rows, H] bf16, row r at hidden + r * hidden_row_stride (elements; multiple of 8)
 * d_last_idx              hidden row of each last token (0 <= idx < hidden_rows): indexed by
 *                         question (d_slot_of == NULL) or by slot (question b reads
 *                         d_last_idx[d_slot_of[b]]), so the plan's d_last_varlen / d_slot_of
 *                         can be passed straight through
 * unembed [V, H]          bf16 row-major; H a multiple of 8, 16-byte aligned
 * d_label_off [B+1], d_label_ids [sum_k]  CSR, request order: question b offers
 *                         label_ids[off[b] .. off[b+1]), 1..255 labels each, ids in [0, V)
 * temperature             > 0 and finite
 * d_probs [sum_k]         fp32 output probabilities (CSR like the ids)
 * h_probs                 optional pinned host copy of d_probs; when given the call copies once
 *                         and synchronises the stream, and reports device-side errors
 * d_logits [sum_k]        optional fp32 raw logits (before the temperature)
 * d_qtype [B], d_answers [B][3], h_answers   optional, together: blink.py `answer_for` on the device.
 *                         d_qtype[b] is 0 (choice), 1 (noul: first label = "yes") or 2 (score:
 *                         label i = level i); d_answers[b] = {index, confidence, value} as fp32:
 *                         the chosen label (first of equal probabilities), for a choice
 *                         (p_best - 1/K)/(1 - 1/K) and p_best, for a score the same confidence
 *                         clamped to [0, 1] and the expected level sum_i i p_i, for a noul NaN and
 *                         p_yes (probabilities renormalised first).  h_answers (pinned) receives a
 *                         copy in the same synchronising host transfer as h_probs.
 * d_ws, ws_bytes          workspace of blink_label_readout_workspace(B) bytes, zero-filled before
 *                         its first use; the call leaves its counters at zero
 * A label id outside [0, V) makes that question's probabilities NaN and latches
 * BLINK_DEVICE_FLAG; so do malformed offsets (then no probability is written).
 * ------------------------------------------------------------------------------------------ */
size_t blink_label_readout_workspace(int32_t B);

blink_status blink_label_readout(const blink_bf16 *hidden, int64_t hidden_row_stride, int32_t hidden_rows,
                                 const int32_t *d_last_idx, const int32_t *d_slot_of, const blink_bf16 *unembed,
                                 int32_t V, int32_t H,
                                 const int32_t *d_label_off, const int32_t *d_label_ids, int32_t B,
                                 int32_t sum_k, float temperature, float *d_probs, float *h_probs,
                                 float *d_logits, const int32_t *d_qtype, float *d_answers, float *h_answers,
                                 void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Log-space readout over several option orders -- the ruling engine (engine.py `_score_plain`,
 * `_prior`, `answer`): each question is scored in passes, one per order of its options; per
 * pass the answer codes' logits z (from blink_label_readout's d_logits) give
 *   lp_j = z_j - logsumexp(z) - prior_K[j]          (position j of the pass)
 * and option i's raw score is the mean of lp over the passes, taken at the position each pass
 * showed option i in.  Then p = softmax(raw / T) and, optionally, the typed answer (as in
 * blink_label_readout).
 *
 * d_logits [..]          pass p's K logits at d_logits[d_pass_off[p] .. d_pass_off[p+1])
 * d_key_of_pos [..]      same layout: the option index (0..K-1) pass p shows at each position;
 *                        each pass's entries must be a permutation of 0..K-1
 * n_pass, d_pass_off [n_pass+1]
 * d_question_pass [B+1]  question q's passes are [d_question_pass[q], d_question_pass[q+1]) (>= 1)
 * d_raw_off [B+1], sum_k question q's options at [d_raw_off[q], d_raw_off[q+1]) of d_raw/d_probs;
 *                        every pass of q has that many positions (1..255)
 * d_prior                optional [255][255] fp32: row K-1 holds the content-free log-probability
 *                        of each position for K options (NULL: no prior subtracted)
 * temperature            > 0 and finite
 * d_raw [sum_k]          optional output: the mean debiased log-probabilities
 * d_probs [sum_k]        output: softmax(raw / T); h_probs optional pinned copy
 * d_qtype, d_answers, h_answers  optional typed answers, as for blink_label_readout
 * d_ws, ws_bytes         blink_rotation_debias_workspace() bytes (error word)
 * A malformed table (a pass of the wrong size, an option index out of range) latches
 * BLINK_DEVICE_FLAG and makes that question's probabilities NaN.
 * ------------------------------------------------------------------------------------------ */
size_t blink_rotation_debias_workspace(void);

blink_status blink_rotation_debias(const float *d_logits, const int32_t *d_pass_off, const int32_t *d_key_of_pos,
                                   int32_t n_pass, const int32_t *d_question_pass, const int32_t *d_raw_off, int32_t B,
                                   int32_t sum_k, const float *d_prior, float temperature, float *d_raw,
                                   float *d_probs, float *h_probs, const int32_t *d_qtype, float *d_answers,
                                   float *h_answers, void *d_ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------------------------
 * Label readout that allocates nothing.  The pages have no counterpart: this entry point is an
 * addition of this library for callers that cannot hand it a workspace.
 *
 * Who needs it: code embedded in a host that gives it only its input and output buffers and
 * owns every other byte of device memory (a serving runtime with a fixed memory plan made at
 * start-up), and latency-critical loops that must never call cudaMalloc, which may synchronise
 * the whole device.  Such callers cannot provide the `d_ws` that blink_label_readout needs.
 *
 * Arguments and results are those of blink_label_readout without d_ws / ws_bytes and without the
 * answer outputs.  The scratch
 * (an error word and one ticket per question) is a static device array of
 * 256 + 4 * BLINK_STATIC_SCRATCH_QUESTIONS bytes (128.25 KiB) that every GPU which loads this
 * library keeps until the process exits.
 *   - B above BLINK_STATIC_SCRATCH_QUESTIONS returns BLINK_OUT_OF_RANGE; nothing is launched.
 *   - The first call on a device looks up the array's device address with that device current
 *     (cudaGetSymbolAddress); make that first call before any stream capture on the device.  The
 *     address is kept per device and context: after a device reset (a new context, so a new copy
 *     of the array) the next call looks it up again, and that call too should come before any
 *     capture.
 *   - From 8192 labels on, the softmaxes run in a second launch (as in blink_label_readout), so
 *     only the error word is used; below that, one ticket per question as well.
 *   - Every call first clears the array's error word and tickets on `stream`.  All calls share
 *     the one array, which keeps the last call's contents: calls whose work can overlap on the
 *     GPU (different streams with no ordering between them) race, and must not be made.
 *   - Device-side errors are reported only through the host-output path (h_probs != NULL).
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 * ------------------------------------------------------------------------------------------ */
#define BLINK_STATIC_SCRATCH_QUESTIONS 32768

blink_status blink_label_readout_noalloc(const blink_bf16 *hidden, int64_t hidden_row_stride, int32_t hidden_rows,
                                         const int32_t *d_last_idx, const int32_t *d_slot_of,
                                         const blink_bf16 *unembed, int32_t V, int32_t H, const int32_t *d_label_off,
                                         const int32_t *d_label_ids, int32_t B, int32_t sum_k, float temperature,
                                         float *d_probs, float *h_probs, float *d_logits, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BLINK_H */
