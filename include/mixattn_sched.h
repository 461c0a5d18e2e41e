/*
 * mixattn_sched.h -- the fair batch builder: the host step that turns a set of
 * requests into the row arrays (row_kinds, seq_lens, q_offsets) of one
 * ForwardBatch for mixattn_plan_create / mixattn_plan_update.  Plain C++ on
 * the host; no GPU, no allocation of device memory, no attention arithmetic.
 *
 * Source: reference page "自研RDNA高併發推論引擎 以AI Max+ 395為範例",
 * §1 "公平性：排隊不插隊（SRTF＋飢餓 decode 優先搶佔＋near-done 閘門）" and the
 * "排程器保證什麼" (scheduler guarantees) table.  The rules, in this order:
 *
 *   1. Decode first.  Due decoders are served before any prefill: a chunk
 *      joins a step only when every due decoder fits in that step (nothing
 *      due is left waiting behind a prefill); otherwise the step is
 *      decode-only.  (Guarantees table, row 1.)
 *   2. Bounded chunk.  A step carries at most one prefill slice of at most
 *      prefill_chunk tokens (default 512), so a 250k-token prompt is fed one
 *      slice per step.  (Row 3.)
 *   3. SRTF prefill choice.  Resident prefills with at most one chunk left
 *      (near-done) go before continuation slices of long prefills; FIFO by
 *      admission within a class.  (§1, first bullet.)
 *   4. Starvation preemption behind the near-done gate.  While requests wait
 *      for a session slot and some resident decoder is within near_done_tokens
 *      (default 64) of its token limit, long-prefill slices yield (near-done
 *      prefills still run), so resident decodes drain and the slot frees
 *      sooner.  With only long-output decoders resident there is no
 *      preemption.  (§1, second and third bullets.)
 *   5. MarkAllDecodersDue.  After every step that carried a chunk, all
 *      resident decoders are due again, so the next step serves them all.
 *      (Row 2.)
 *   6. PopDecoder rotation.  The decoders a step serves move to the back of
 *      the decode queue, so with a cap on decode rows no session keeps
 *      winning the front places.  (Row 4.)
 *   7. Per-client admission.  A client may have at most
 *      max_pending_per_client requests waiting for a slot (submit returns
 *      MIXATTN_ERR_CLIENT_QUOTA beyond that), and admission to free slots
 *      takes the clients in turn, oldest request of each first.  (Row 5.)
 *
 * Readings where the page is silent: "pending" per client counts requests
 * waiting for a session slot (not resident ones); a decoder that was served by
 * a decode-only step is not due again until the next step with a chunk, or
 * until no step could run otherwise (then all are marked due); the step that
 * completes a prompt yields its first output token, and that request joins the
 * decode queue at the back, due.
 *
 * Positions follow the attention ABI: a prefill slice of n tokens of a request
 * with c tokens cached is a chunk row (seq_len c + n, q_offset c); a decoder
 * with g generated tokens (the last one not yet in the cache) is a decode row
 * at seq_len prompt + g, q_offset prompt + g - 1.  The caller appends the
 * rows' new K/V (mixattn_kv_append_quant) before the attention, maps pages,
 * and reports the step done with mixattn_sched_complete.
 *
 * Every call returns a mixattn_status (0 = OK) unless stated; a scheduler is
 * not thread-safe (one owner thread).
 */
#ifndef MIXATTN_SCHED_H
#define MIXATTN_SCHED_H

#include <stdint.h>

#include "mixattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Status of a submit refused by the per-client cap (the page's client_quota). */
#define MIXATTN_ERR_CLIENT_QUOTA (-6)

/* Kind of step a batch is. */
typedef enum {
  MIXATTN_STEP_IDLE = 0,    /* nothing to run                               */
  MIXATTN_STEP_DECODE = 1,  /* decode rows only                             */
  MIXATTN_STEP_MERGED = 2,  /* decode rows and one prefill slice            */
  MIXATTN_STEP_PREFILL = 3  /* one prefill slice, no decoder is resident or due */
} mixattn_step_kind;

/* Request states (mixattn_sched_request_info). */
typedef enum {
  MIXATTN_REQ_WAITING = 0,  /* submitted, waiting for a session slot */
  MIXATTN_REQ_PREFILL = 1,  /* resident, prompt not fully cached      */
  MIXATTN_REQ_DECODE = 2,   /* resident, generating                   */
  MIXATTN_REQ_DONE = 3      /* finished; its slot is free             */
} mixattn_req_state;

typedef struct {
  int32_t max_sessions;           /* resident request slots, >= 1                         */
  int32_t prefill_chunk;          /* tokens per prefill slice, >= 1 (the page: 512)       */
  int32_t max_pending_per_client; /* requests waiting per client, 0 = no cap              */
  int32_t near_done_tokens;       /* near-done gate, >= 0 (the page: 64)                  */
  int32_t max_decode_rows;        /* decode rows per step, 0 = no cap (all residents)     */
} mixattn_sched_config;

typedef struct mixattn_sched mixattn_sched;

/* Fills the page's defaults: 16 sessions, 512-token chunk, no per-client cap,
 * a 64-token near-done gate, no decode-row cap. */
void mixattn_sched_default_config(mixattn_sched_config* cfg);

int mixattn_sched_create(mixattn_sched** out, const mixattn_sched_config* cfg);
void mixattn_sched_destroy(mixattn_sched* s);

/* A new request: prompt_len >= 1 prompt tokens, at most max_new_tokens >= 1
 * output tokens (its token limit).  request_id must be unused.  Returns
 * MIXATTN_ERR_CLIENT_QUOTA when the client already has max_pending_per_client
 * requests waiting (nothing is queued then). */
int mixattn_sched_submit(mixattn_sched* s, int64_t request_id, int32_t client_id, int32_t prompt_len,
                         int32_t max_new_tokens);

/* Builds the next step: admits waiting requests to free slots, picks the rows
 * and writes them to the host arrays (capacity `cap`, which must be at least
 * max_sessions + 1): decode rows first (queue order), then the chunk row if
 * any.  request_ids (may be NULL) receives the request of each row.  Returns
 * the number of rows (0 when idle) or a negative status; *kind_out (may be
 * NULL) receives the mixattn_step_kind.  A built step must be completed with
 * mixattn_sched_complete before the next one is built (otherwise
 * MIXATTN_ERR_INVALID_ARG). */
int32_t mixattn_sched_next_batch(mixattn_sched* s, int32_t cap, int32_t* row_kinds, int32_t* seq_lens,
                                 int32_t* q_offsets, int64_t* request_ids, int32_t* kind_out);

/* Reports the built step as run: every row's tokens are in the cache, every
 * decode row and every chunk row that completed its prompt produced one
 * token.  Requests that reached their token limit, or are listed in
 * stop_ids (e.g. they emitted an end-of-sequence token this step; n_stop >= 0,
 * ids not in the step are ignored), finish and free their slot. */
int mixattn_sched_complete(mixattn_sched* s, const int64_t* stop_ids, int32_t n_stop);

/* State of a request: any output pointer may be NULL.  cached = tokens in the
 * cache, generated = output tokens so far, first_token_step = index of the
 * step that produced its first token (-1 before), done_step likewise. */
int mixattn_sched_request_info(const mixattn_sched* s, int64_t request_id, int32_t* state, int32_t* cached,
                               int32_t* generated, int64_t* first_token_step, int64_t* done_step);

/* Counts: waiting, resident prefills, resident decoders, completed steps. */
int mixattn_sched_counts(const mixattn_sched* s, int32_t* waiting, int32_t* prefills, int32_t* decoders,
                         int64_t* steps);

#ifdef __cplusplus
}
#endif

#endif /* MIXATTN_SCHED_H */
