/*
 * strata_sample.h -- C ABI of the GB300 decode-time token sampler.
 *
 * One library call samples one token for each of B head-logit rows (verify-window positions or
 * batch slots) in a single kernel launch, and optionally reports raw-logit log-probabilities.
 * Definitions follow the pages of the engine this library serves:
 *   [P19]   "#19 serve: per-request temperature/top_p/top_k/min_p/penalties sampling",
 *           section "What changed" (paragraphs "min_p and the penalties", "The sampled chain is
 *           one block per token", "A persistent per-request draw counter; sampled requests
 *           default top_k=20", "server.py forwards the block to the engine").
 *   [P3200] "#3200 [Engine] OpenAI logprobs / top_logprobs / allowed_token_ids for the CUDA/HIP
 *           engine", sections "Problem and result" and "Approach".
 *   [P1916] "#1916 OpenAI logprobs on /v1/chat/completions for the CUDA/HIP engine",
 *           section "What changed".
 *   [P559]  "#559 Several conversations at once: batch slots, a pipelined layer split, per-stage
 *           dense weights", section "What it adds", item 1 (one row per slot, per-slot keys,
 *           Philox(seed, position)).
 *
 * Conventions for every call:
 *   - Device pointers are plain CUDA device addresses owned by the caller; the library reads and
 *     writes them only from work it enqueues on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream).  Host pointers are read before the call returns.
 *   - Calls that take a stream are asynchronous unless stated otherwise: outputs are valid once
 *     the stream has reached the call's work.
 *   - Every call returns STRATA_OK (0) or a negative STRATA_E* code; strata_last_error() then
 *     holds a one-line message for the calling thread.  Argument checks run before any work is
 *     enqueued, so a call that returns an error has launched nothing and written nothing.
 *   - A context serves one stream at a time: calls on one context must be ordered (one stream,
 *     or synchronised streams).  Calls on different contexts are independent.
 *   - The calling thread's current CUDA device must be the context's device.
 *   - With STRATA_SAMPLE_DEBUG set to a value other than "0" in the environment (read once per
 *     process), every sampling or logprobs call that passes its argument checks prints one line
 *     to stderr before it launches: the entry point, B, V, the logit type, the flags and the
 *     launch shape chosen (split, chunk, ring slots, warp-maxima per warp, hash capacity, dynamic
 *     shared memory, grid).  Unset, the library prints nothing.
 */
#ifndef STRATA_SAMPLE_H
#define STRATA_SAMPLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---------------------------------------------------------------------- */
#define STRATA_OK        0
#define STRATA_EINVAL  (-1)   /* a parameter or shape is invalid                                 */
#define STRATA_EALIGN  (-2)   /* a logit pointer or row stride is not 16-byte aligned            */
#define STRATA_ERANGE  (-3)   /* slot, rows or vocabulary above the limits given at create time  */
#define STRATA_ECUDA   (-4)   /* a CUDA runtime call failed (message in strata_last_error)       */
#define STRATA_ENOMEM  (-5)   /* device or host allocation failed at create time                 */

/* ---- logit element types ----------------------------------------------------------------- */
#define STRATA_DTYPE_F32   0  /* IEEE float32 rows                                               */
#define STRATA_DTYPE_BF16  1  /* bfloat16 rows; widened to float32 exactly                       */

/* ---- limits ------------------------------------------------------------------------------ */
#define STRATA_MAX_TOP_K           64   /* [P19]: the sampled path requires top_k in 1..64       */
#define STRATA_DEFAULT_TOP_K       20   /* [P19]: sampled requests default to top_k=20           */
#define STRATA_MAX_TOP_N           20   /* [P3200]: top_logprobs 0..20                           */
#define STRATA_DEFAULT_LAST_N      64   /* [P19]: a penalty without a window uses 64 tokens      */
#define STRATA_MAX_PENALTY_LAST_N  4096 /* library limit on the penalty history window           */
#define STRATA_MAX_VOCAB           524288 /* library limit on V (per-row split over <= 16 SMs)   */
#define STRATA_HISTORY_CAP         4096 /* ids a slot's kept history holds (its newest ids)      */
#define STRATA_MAX_SHARDS          16   /* vocabulary slices one strata_merge_shards call merges  */
#define STRATA_SHARD_RECORD_BYTES  1280 /* bytes of one row's record from one vocabulary slice    */

/* ---- launch flags (strata_sample_rows / strata_logprobs_rows `flags`) --------------------- */
/* Launch with programmatic dependent launch: the kernel may be scheduled while the previous
 * kernel on the stream finishes; it waits for that kernel before reading any input.            */
#define STRATA_FLAG_PDL         0x1u
/* With STRATA_FLAG_PDL: the caller asserts that every input the call reads (logit rows, row
 * slots, positions, drafts, history rows, allowed lists) was complete before the previous kernel
 * on the stream started (none of it is that kernel's output).  The kernel then starts its loads
 * before waiting for the previous kernel; draw counters, the slots' kept histories
 * (STRATA_FLAG_HISTORY_RING) and every output are still read or written after the wait (draw
 * counters and outputs without any wait under STRATA_FLAG_OWN_OUTPUTS, below).                  */
#define STRATA_FLAG_EARLY_LOAD  0x2u
/* strata_sample_rows with allowed/allowed_off: a row that names allowed ids samples only among
 * them (allowed_token_ids as a sampling mask for constrained decoding [P3200, "Problem and result"
 * names the client use]): penalties, top_k, min_p, top_p, temperature and the draw run over the
 * named ids (a repeat counts once, ids outside [0, V) are ignored).  A row with an empty list is
 * not restricted; a row whose ids are all outside [0, V) gets id -1 and STRATA_DEVERR_NOCAND.
 * The log-probability outputs still describe the row's full raw distribution.                  */
#define STRATA_FLAG_ALLOWED_MASK 0x4u
/* strata_sample_rows / strata_sample_verify: take each row's penalty window from its slot's kept
 * history in the context (strata_history_enable) instead of hist/hist_off, which must then be
 * NULL.  [P19, "min_p and the penalties": the serve loop uploads the request's last
 * penalty_last_n tokens before every window.]  Every row of a slot counts over the same window,
 * the last min(penalty_last_n, length) ids as they stood before the call; in the same launch
 * the slot's history then grows by its rows' picks in row order (strata_sample_verify: only the
 * rows it keeps), a pick of -1 appending nothing.  Slots that no row names are not touched.  The
 * update happens on the device, so a captured call carries the history forward on every replay.
 * Ignored by strata_logprobs_rows.                                                              */
#define STRATA_FLAG_HISTORY_RING 0x8u
/* With STRATA_FLAG_PDL | STRATA_FLAG_EARLY_LOAD, for strata_sample_rows and strata_logprobs_rows
 * (not verify windows, not kept histories: STRATA_EINVAL): the caller asserts that no call that
 * may still be running when this one starts (the previous calls on the stream) writes or reads
 * this call's output buffers, for instance because consecutive calls write different buffers.
 * The call then never waits for the previous one: it takes its draw counters at its start, before
 * the next call on the stream may launch, so counters still advance in call order (each sampled
 * slot by one per call, every row of a slot seeing the value from before the call), and it writes
 * its outputs when they are ready.  Results are the same as without the flag.  A sampling call
 * without the flag takes its counters late (after waiting for its predecessor, or during its
 * run), so once the context has launched such a call, its later calls (sampling or logprobs)
 * ignore this flag and wait as usual, until a call without STRATA_FLAG_PDL that takes no late
 * counters, or strata_read_errors, has drained the stream.  Keep a stream that carries flagged
 * calls to one context: another context's flagged call would break the chain of waits that this
 * context's waiting calls rely on.  The next call's
 * launch then waits for this call's counter atomics (a few memory round trips at its start), so
 * one stream of calls alone can run slower with the flag; it pays when independent request groups
 * (other contexts, other streams) keep the GPU busy meanwhile (see STRATA_FLAG_CONCURRENT).     */
#define STRATA_FLAG_OWN_OUTPUTS 0x20u
/* A launch-shape hint: calls on other streams (of other contexts) run on the GPU at the same time
 * as this one, so whole-GPU throughput matters more than this call's latency.  The call then gives
 * each row one block per STRATA_CONCURRENT_ROW_BYTES of logits (two blocks for a full fp32 row of
 * 248,320 ids, one for a bf16 row): fewer blocks per byte and a small exchange between them, at
 * the price of a longer call.  Calls with STRATA_FLAG_HISTORY_RING (which wait for the previous
 * call before their penalties) take one block per 128 KiB.  Results are the same as without the
 * flag.  A forced split (STRATA_FLAG_SPLIT) takes precedence.                                    */
#define STRATA_FLAG_CONCURRENT  0x10u
#define STRATA_CONCURRENT_ROW_BYTES (1u << 19)
/* A launch-shape choice: hold each block's chunk whole in shared memory (at most 64 KiB of logits:
 * up to 16 blocks per row) instead of streaming it through a ring of shared-memory slots, with a
 * row threshold exchanged across the row's blocks and candidates read from shared memory.  A row
 * too large for 16 such blocks streams as usual.  Results are the same either way.  Measured on
 * GB300 slower than streaming for every workload (the post-pass dominates a block's life), so it
 * is off by default.                                                                           */
#define STRATA_FLAG_RESIDENT    0x40u
/* Testing aid: the row leaders also wait for one arrival that nothing sends, so that their bounded
 * device wait (about two seconds) runs out: the call sets STRATA_DEVERR_TIMEOUT, its outputs are
 * undefined, and the context stays usable.  It exercises the failure path without a GPU fault.  */
#define STRATA_FLAG_TEST_STALL  0x10000u
/* Testing aid: force the number of thread blocks (1..16) that split each row; 0 = automatic.  A
 * forced split whose blocks would not fit their shared memory is STRATA_ERANGE.                */
#define STRATA_FLAG_SPLIT(n)    (((uint32_t)(n) & 0x1Fu) << 8)

/* ---- device error bits (strata_read_errors) ---------------------------------------------- */
#define STRATA_DEVERR_SLOT      0x01u  /* a row named a slot outside [0, max_slots): out id -1  */
#define STRATA_DEVERR_ALLOWED   0x02u  /* an allowed id outside [0, V): its output is NaN       */
#define STRATA_DEVERR_CHOSEN    0x04u  /* a chosen id outside [0, V): its logprob is NaN        */
#define STRATA_DEVERR_TIMEOUT   0x08u  /* a bounded device wait ran out (outputs of that call
                                          are not valid)                                        */
#define STRATA_DEVERR_NOCAND    0x10u  /* a row had no orderable logit (all NaN): out id -1     */
#define STRATA_DEVERR_HISTORY   0x20u  /* the history table of a row overflowed (not expected)  */
#define STRATA_DEVERR_SHAPE     0x40u  /* a slot's top_k exceeded the launch shape: a call captured
                                          in a CUDA graph before the slot's keys grew; the row kept
                                          fewer survivors.  Re-capture after raising top_k.      */

typedef struct strata_ctx strata_ctx;

/*
 * A request's sampling keys [P19, "What changed": the GEN keys temperature=, top_p=, top_k=,
 * min_p=, penalty_repeat=, penalty_freq=, penalty_present=, penalty_last_n=, seed=].
 * Plain data; `struct_size` must be at least sizeof(strata_sampling_params) as defined here
 * (a larger value from a newer caller is accepted and the unknown tail is ignored).
 */
typedef struct strata_sampling_params {
  uint32_t struct_size;
  float    temperature;      /* > 0: sampled row.  <= 0: greedy argmax of the penalised logits
                                ([P19]: absent temperature and temperature=0 both mean greedy)   */
  int32_t  top_k;            /* sampled rows: 1..64 survivors; 0 means 20 [P19]; else EINVAL     */
  float    top_p;            /* nucleus mass over the min_p survivors; >= 1 disables; <= 0 keeps
                                the head only                                                     */
  float    min_p;            /* >= 0; 0 disables; keep sel_logit >= sel_logit[0] + logf(min_p),
                                the head always kept [P19]                                        */
  float    penalty_repeat;   /* > 0; 1 is neutral.  l <= 0: l*r, l > 0: l/r [P19]                 */
  float    penalty_freq;     /* finite; 0 is neutral.  subtract freq * count [P19]                */
  float    penalty_present;  /* finite; 0 is neutral.  subtract present if count > 0 [P19]        */
  int32_t  penalty_last_n;   /* 0..4096 history tokens counted; 0 disables the penalties          */
  uint32_t reserved;         /* must be 0                                                         */
  uint64_t seed;             /* Philox key [P19], [P559]                                          */
} strata_sampling_params;

/* Library version: major*10000 + minor*100 + patch. */
int strata_version(void);

/* Message of the calling thread's last failed call ("" if none).  Owned by the library. */
const char *strata_last_error(void);

/* Fill *p with the neutral greedy defaults: temperature 0, top_k 0, top_p 1, min_p 0, repeat 1,
 * freq 0, present 0, penalty_last_n 64, seed 0, struct_size set.  Host only. */
void strata_default_params(strata_sampling_params *p);

/* Check keys without a context: STRATA_OK or STRATA_EINVAL (reason in strata_last_error).
 * An invalid key is rejected, never silently adjusted [P19, "server.py forwards the block to
 * the engine"].  Host only, no CUDA call. */
int strata_validate_params(const strata_sampling_params *p);

/*
 * Create a context on `device` (must be the calling thread's current device) for up to
 * `max_slots` request slots (1..65536), vocabularies up to `max_vocab` (1..STRATA_MAX_VOCAB)
 * and up to `max_rows` rows per call (1..65535).  Allocates the device slot table (keys and
 * 48-bit draw counters, all slots greedy-neutral with counter 0) and a device error word.
 * Synchronous.  Returns STRATA_ECUDA when no usable device is present.
 */
int strata_create(strata_ctx **out, int device, int max_slots, int max_vocab, int max_rows);

/* Free a context and its device memory.  Synchronises the device first.  NULL is a no-op. */
void strata_destroy(strata_ctx *ctx);

/*
 * Set a slot's keys (validated as strata_validate_params) and, with reset_counter != 0, its
 * draw counter to 0.  The device copy is updated by a copy enqueued on `stream`, so sample calls
 * enqueued later on that stream see the new keys.  Without reset the counter keeps counting
 * [P19: the draw counter persists across a request's verify windows].
 */
int strata_set_slot_params(strata_ctx *ctx, int slot, const strata_sampling_params *p,
                           int reset_counter, void *stream);

/* Read a slot's keys and its current draw counter.  Synchronises `stream` (counters live on the
 * device and advance inside sample calls).  Either output pointer may be NULL. */
int strata_get_slot_state(strata_ctx *ctx, int slot, strata_sampling_params *p,
                          uint64_t *counter, void *stream);

/* Restore a slot's keys and counter exactly (checkpoint/resume of a request); asynchronous on
 * `stream` like strata_set_slot_params.  Counters are 48-bit: a value >= 2^48 is STRATA_ERANGE. */
int strata_set_slot_state(strata_ctx *ctx, int slot, const strata_sampling_params *p,
                          uint64_t counter, void *stream);

/*
 * Sample one token per row: penalties over the slot's history window -> top_k (value
 * descending, ties to the lowest index) -> min_p -> top_p -> temperature -> one draw from
 * Philox(seed, position) at the slot's draw counter [P19]; greedy rows take the first entry of
 * the penalised order.  One kernel launch on `stream`.
 *
 *   logits      device, [B][ld] elements of `dtype`, row b at logits + b*ld; base address and
 *               ld*sizeof(element) must be multiples of 16 bytes (else STRATA_EALIGN); ld >= V.
 *               Logits must be finite or -inf; NaN is outside the contract.
 *   row_slot    device int32[B]: the slot whose keys, history and counter row b uses.
 *   row_pos     device int64[B]: row b's absolute token position (the Philox counter word).
 *   hist        device int32[]: concatenated history ids of slots 0..n_hist_slots-1;
 *   hist_off    device int32[n_hist_slots+1]: slot s owns hist[hist_off[s] .. hist_off[s+1]).
 *               The penalties count the last min(penalty_last_n, length) ids of the slot's run;
 *               ids outside [0, V) are ignored.  hist/hist_off NULL (or a slot >= n_hist_slots)
 *               means no history: the penalty stage is skipped and the logits are used unchanged [P19].
 *               With STRATA_FLAG_HISTORY_RING both must be NULL (else STRATA_EINVAL) and the
 *               window comes from the slot's kept history; without strata_history_enable first
 *               that flag is STRATA_EINVAL.
 *   out_ids     device int32[B]: the sampled id of each row (always written; -1 for a row whose
 *               slot is out of range, with STRATA_DEVERR_SLOT).
 *   Optional fused logprobs of the raw (pre-penalty, pre-temperature) logits [P3200, P1916];
 *   every NULL output switches its part off at no cost:
 *   top_n       0..20 alternatives per row.
 *   chosen_lp   device float[B]: log-probability of out_ids[b] under the raw softmax.
 *   top_ids     device int32[B][top_n] and top_lps float[B][top_n]: the top_n raw logits
 *               (ties to the lowest index) and their log-probabilities; rows with V < top_n are
 *               padded with id -1 and -inf.
 *   allowed     device int32[]: concatenated allowed_token_ids of rows 0..B-1;
 *   allowed_off device int32[B+1]: row b names allowed[allowed_off[b] .. allowed_off[b+1]);
 *   allowed_lps device float[allowed_off[B]]: log-probabilities normalised over only the
 *               named ids, in the caller's order (a repeated id counts once in the normaliser).
 *   Optional debug outputs (NULL = off): topk_ids int32[B][64] and topk_vals float[B][64] (the
 *   ordered survivors of top_k and their penalised logits, padded with -1 / NaN), kept
 *   int32[B][2] (survivors after min_p, after top_p).
 *   flags       STRATA_FLAG_* bits.
 *
 * Counter rule: each slot that has at least one sampled row in the call advances its draw
 * counter by exactly 1; all rows of the call read the counter as it was before the call (rows of
 * one slot differ by position).  The advance happens on the device inside the launch, so the
 * call can be captured in a CUDA graph and every replay draws fresh numbers.
 */
int strata_sample_rows(strata_ctx *ctx, const void *logits, int dtype, int B, int V, int64_t ld,
                       const int32_t *row_slot, const int64_t *row_pos,
                       const int32_t *hist, const int32_t *hist_off, int n_hist_slots,
                       int32_t *out_ids,
                       int top_n, float *chosen_lp, int32_t *top_ids, float *top_lps,
                       const int32_t *allowed, const int32_t *allowed_off, float *allowed_lps,
                       int32_t *topk_ids, float *topk_vals, int32_t *kept,
                       uint32_t flags, void *stream);

/*
 * Sample verify windows and count the rows each slot keeps [P19, "What changed": the emitted
 * tokens are always the target's own samples, the drafts only fill the verified window; P559,
 * "Not done (yet)": a sampled row is accepted when its pick equals the draft].  Samples exactly as
 * strata_sample_rows (same keys, history, counter rule, fused chosen/top-N logprobs; no allowed
 * subsets or debug outputs) and, in the same launch, compares each row's pick with its draft:
 *
 *   row_draft  device int32[B]: the draft placed right after row b's position in its slot's
 *              window, or -1 for the window's last row.  The rows of a slot, in row order, are
 *              that slot's window.
 *   slot_keep  device int32[max_slots]: for every slot named by a row, the number of its rows to
 *              keep = 1 + the leading rows whose pick equals their draft (a pick of -1 never
 *              matches).  The entries of slots no row names are not written.
 *
 * The count is taken on the device by the last row of each slot to finish (a per-slot arrival
 * word in the context, cleared by that row), so the call can be captured in a CUDA graph.
 * Errors as strata_sample_rows; row_draft and slot_keep are required (STRATA_EINVAL).
 */
int strata_sample_verify(strata_ctx *ctx, const void *logits, int dtype, int B, int V, int64_t ld,
                         const int32_t *row_slot, const int64_t *row_pos, const int32_t *row_draft,
                         const int32_t *hist, const int32_t *hist_off, int n_hist_slots,
                         int32_t *out_ids, int32_t *slot_keep,
                         int top_n, float *chosen_lp, int32_t *top_ids, float *top_lps,
                         uint32_t flags, void *stream);

/*
 * Logprobs without sampling [P3200, "Approach": the head logits before sampling, penalties and
 * temperature; P1916, "What changed"].  Same layouts as above; `chosen` (device int32[B], or
 * NULL) names the id whose log-probability goes to chosen_lp[b] (NaN and STRATA_DEVERR_CHOSEN
 * for an id outside [0, V)).  No slot state is read or changed.
 */
int strata_logprobs_rows(strata_ctx *ctx, const void *logits, int dtype, int B, int V, int64_t ld,
                         const int32_t *chosen, float *chosen_lp,
                         int top_n, int32_t *top_ids, float *top_lps,
                         const int32_t *allowed, const int32_t *allowed_off, float *allowed_lps,
                         uint32_t flags, void *stream);

/*
 * Vocabulary-sliced sampling: each row's V ids are split into disjoint slices (for instance one per
 * GPU holding that slice of the head's output), each slice is reduced to a small record, the
 * records are exchanged, and a merge of every slice's record gives what strata_sample_rows gives on
 * the whole row.  The pages split a model across GPUs only by layers, with sampling on the last
 * stage [P559, "What it adds"]; this pair is a library addition whose result is defined by the
 * whole-row chain [P19, "min_p and the penalties", "The sampled chain is one block per token"]
 * and the raw-logit logprobs [P3200, "Approach"]: the row's top_k list is among the union of its
 * slices' own top_k lists, its top_n raw alternatives among the union of theirs, and its
 * log-sum-exp is the log of the summed exponentials of theirs.
 *
 * strata_shard_rows: one slice of B rows.  logits/dtype/ld as in strata_sample_rows, with V_shard
 * columns that hold the ids id_offset .. id_offset + V_shard - 1 (id_offset >= 0).  row_slot,
 * hist, hist_off and n_hist_slots as in strata_sample_rows; history ids are the row's own (whole
 * vocabulary) ids and the slice counts those inside it.  top_n (0..20) alternatives are kept per
 * record.  records: device, [B][STRATA_SHARD_RECORD_BYTES], 16-byte aligned (else
 * STRATA_EALIGN).  Record layout (little-endian 32-bit words):
 *   word 0: n_pen, entries in the penalised list (<= the row's top_k, 1 for a greedy row,
 *           0 for a row whose slot is out of range)
 *   word 1: n_raw, entries in the raw list (<= top_n)
 *   word 2: float, log of the sum of exp(raw logit) over the slice's ids
 *   word 3: 0
 *   bytes 16 .. 16 + 16*64: penalised entries, best first: key low word, key high word, raw logit
 *           (float), 0
 *   bytes 1040 .. 1040 + 8*20: raw entries, best first: key low word, key high word
 *   the rest: unused.
 * A key is (ord(v) << 32) | (0xFFFFFFFF - id), larger is better: v the entry's (penalised or raw)
 * logit, ord the order-preserving map of a float to uint32 (sign bit clear: bits | 0x80000000;
 * set: ~bits; -0.0 as +0.0), id the whole-vocabulary id, so equal values order by lower id.  No
 * slot state changes: the counters move only in the merge.
 * flags: STRATA_FLAG_CONCURRENT and STRATA_FLAG_SPLIT only (else STRATA_EINVAL).
 *
 * strata_merge_shards: records device, [n_shards][B][STRATA_SHARD_RECORD_BYTES] (slice-major: the
 * concatenation of every slice's strata_shard_rows output for the same B rows, in any slice
 * order), 1 <= n_shards <= STRATA_MAX_SHARDS.  The slices must be disjoint and made with the same
 * context state (slot keys) and the same top_n.  Runs top_k, min_p, top_p, temperature and the
 * Philox draw on the merged list of each row and writes out_ids, chosen_lp, top_ids/top_lps
 * (top_n as given to the slices) and the debug outputs topk_ids/topk_vals/kept exactly as
 * strata_sample_rows does, with row_pos the rows' positions; the counter rule is that of
 * strata_sample_rows (each slot with a sampled row advances by 1 in this call).  Every GPU that
 * merges the same records with the same slot state writes the same outputs.  flags: 0 (else
 * STRATA_EINVAL).  The allowed-subset logprobs, STRATA_FLAG_ALLOWED_MASK, verify windows and kept
 * histories are not available on sliced rows.
 */
int strata_shard_rows(strata_ctx *ctx, const void *logits, int dtype, int B, int V_shard, int64_t ld,
                      int id_offset, const int32_t *row_slot,
                      const int32_t *hist, const int32_t *hist_off, int n_hist_slots,
                      int top_n, void *records, uint32_t flags, void *stream);
int strata_merge_shards(strata_ctx *ctx, const void *records, int n_shards, int B,
                        const int32_t *row_slot, const int64_t *row_pos, int32_t *out_ids,
                        int top_n, float *chosen_lp, int32_t *top_ids, float *top_lps,
                        int32_t *topk_ids, float *topk_vals, int32_t *kept,
                        uint32_t flags, void *stream);

/*
 * Kept per-slot histories (STRATA_FLAG_HISTORY_RING).  A slot's history is the ids of its run so
 * far; the context keeps its newest STRATA_HISTORY_CAP ids (a ring per slot, enough for every
 * penalty window) and its total length.
 *
 * strata_history_enable: allocate the histories of all max_slots slots (4 * STRATA_HISTORY_CAP
 * bytes per slot plus an 8-byte length), every one empty.  Synchronous; a second call is a no-op.
 * STRATA_ENOMEM when the device allocation fails.
 *
 * strata_history_set: replace slot `slot`'s history by the n ids of host array `ids` (the
 * prompt, or a run restored from a checkpoint); only the newest min(n, STRATA_HISTORY_CAP) are
 * read, n becomes the length.  ids outside [0, V) are kept but never penalise.  Asynchronous on
 * `stream` like strata_set_slot_params (the host array is read before the call returns).
 *
 * strata_history_get: synchronise `stream`, then write the newest min(length,
 * STRATA_HISTORY_CAP, max_n) ids of the slot, oldest first, to host array `ids`, their count to
 * *n_out and the total length to *length (either pointer may be NULL).
 *
 * All three: STRATA_EINVAL for a null context, STRATA_ERANGE for a slot outside [0, max_slots);
 * set/get before enable, or n < 0 / max_n < 0, is STRATA_EINVAL.
 */
int strata_history_enable(strata_ctx *ctx);
int strata_history_set(strata_ctx *ctx, int slot, const int32_t *ids, int64_t n, void *stream);
int strata_history_get(strata_ctx *ctx, int slot, int32_t *ids, int max_n, int *n_out, int64_t *length,
                       void *stream);

/* Synchronise `stream`, return the accumulated STRATA_DEVERR_* bits in *bits and clear them. */
int strata_read_errors(strata_ctx *ctx, uint32_t *bits, void *stream);

/*
 * The launch shape a call with these arguments would use (host only, nothing enqueued):
 * blocks per row (the thread-block cluster size), elements per block, dynamic shared memory
 * bytes and the total grid size.  mode 0 = strata_sample_rows, 1 = strata_logprobs_rows,
 * 2 = strata_sample_verify.  The shape is that of a call without allowed lists.  Allowed
 * lists need a bitmap of the block's ids, which shares the block's copy ring and changes nothing
 * unless it is larger than the ring; STRATA_FLAG_ALLOWED_MASK adds a second bitmap of that size.
 */
int strata_launch_shape(strata_ctx *ctx, int mode, int dtype, int B, int V, int top_n,
                        uint32_t flags, int *split, int *chunk_elems, int *smem_bytes, int *grid);

/*
 * Allocation-free sampling, for callers that cannot call cudaMalloc (code running inside a
 * framework whose allocator owns all device memory, or a process that must not grow its device
 * footprint once serving has started).  The pages have no counterpart of this call; it is a
 * library addition.
 *
 * Same chain and kernel as strata_sample_rows, with no context: row b is its own request slot,
 * its keys come from the host array row_params[b] and its draw counter value from the host array
 * row_counters[b] (< 2^48).  The caller owns the counters: after a call, advance every sampled
 * row's counter by one itself (greedy rows draw nothing).  hist/hist_off is CSR per row
 * ([B+1] offsets; NULL = no history).  Outputs as in strata_sample_rows (no allowed subsets, no
 * debug outputs).  B is at most STRATA_NOALLOC_MAX_ROWS; more rows is STRATA_ERANGE.
 *
 * Memory: nothing is allocated on the device.  The per-row key records, counter words, the
 * row-to-slot table and the device error word live in one static device array of about 60 KiB
 * that every GPU loading this library holds until the process exits.  Every call shares that
 * array and it keeps the last call's contents; each call rewrites (and zeroes) what it reads, but
 * calls that overlap on the GPU race, so issue them on one stream.  Device error bits of these
 * calls are not reported.  On the host, each call prepares the keys and counters in one static
 * buffer of the library and copies them to the device array with cudaMemcpyAsync on `stream`;
 * host threads take turns on that buffer (a lock), and a copy from such pageable memory returns
 * once the CUDA runtime holds the bytes, which can mean waiting for work already queued on the
 * stream.  The first call on each device sets that device up synchronously (finds the array's
 * device address, sets kernel attributes, uploads the row table); make that first call before
 * capturing any stream.
 */
#define STRATA_NOALLOC_MAX_ROWS 1024
int strata_sample_rows_noalloc(const void *logits, int dtype, int B, int V, int64_t ld,
                               const strata_sampling_params *row_params, const uint64_t *row_counters,
                               const int64_t *row_pos, const int32_t *hist, const int32_t *hist_off,
                               int32_t *out_ids, int top_n, float *chosen_lp, int32_t *top_ids,
                               float *top_lps, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* STRATA_SAMPLE_H */
