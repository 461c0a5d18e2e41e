// scheduler.cc -- the fair batch builder behind include/mixattn_sched.h.
//
// Page "自研RDNA高併發推論引擎 以AI Max+ 395為範例", §1 "公平性：排隊不插隊" and
// the "排程器保證什麼" table: decode first, one bounded prefill slice per step,
// SRTF among prefills, starvation preemption behind the near-done gate,
// MarkAllDecodersDue after every step with a chunk, PopDecoder rotation, and
// per-client admission with a pending cap.  The header states each rule and
// the readings taken where the page is silent.  Host code only: it produces the
// row arrays the attention ABI takes and holds no attention arithmetic.
#include <stdint.h>

#include <algorithm>
#include <deque>
#include <map>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/mixattn_sched.h"

namespace {

struct Request {
  int64_t id = 0;
  int32_t client = 0;
  int32_t prompt = 0;     // prompt tokens
  int32_t limit = 0;      // token limit (output tokens at most)
  int32_t state = MIXATTN_REQ_WAITING;
  int32_t cached = 0;     // tokens in the cache
  int32_t generated = 0;  // output tokens so far
  bool due = false;       // decoders: must be served before the next prefill slice
  int64_t admitted = -1;  // admission order (FIFO within an SRTF class)
  int64_t first_token_step = -1;
  int64_t done_step = -1;
};

}  // namespace

struct mixattn_sched {
  mixattn_sched_config cfg{};
  std::unordered_map<int64_t, Request> reqs;
  std::map<int32_t, std::deque<int64_t>> waiting;  // per client, oldest first
  std::deque<int32_t> client_turn;                 // clients with waiting requests, in turn
  int32_t n_waiting = 0;
  std::deque<int64_t> decoders;  // the decode queue (PopDecoder order)
  std::vector<int64_t> prefills; // resident prefills, in admission order
  int32_t resident = 0;
  int64_t admit_seq = 0;
  int64_t steps = 0;
  // the step built and not yet completed
  bool built = false;
  std::vector<int64_t> step_decode;
  int64_t step_chunk = -1;
  int32_t step_chunk_len = 0;
};

namespace {

void admit(mixattn_sched* s) {
  while (s->resident < s->cfg.max_sessions && !s->client_turn.empty()) {
    const int32_t c = s->client_turn.front();
    s->client_turn.pop_front();
    std::deque<int64_t>& q = s->waiting[c];
    const int64_t id = q.front();
    q.pop_front();
    if (!q.empty()) s->client_turn.push_back(c);  // the client's next request waits its turn
    --s->n_waiting;
    Request& r = s->reqs[id];
    r.state = MIXATTN_REQ_PREFILL;
    r.admitted = s->admit_seq++;
    s->prefills.push_back(id);
    ++s->resident;
  }
}

// The prefill slice to run next, or -1: near-done prefills (at most one chunk
// left) first, then long ones unless starvation preemption holds them back;
// FIFO by admission within a class.
int64_t pick_prefill(const mixattn_sched* s) {
  bool preempt = false;
  if (s->n_waiting > 0) {
    for (int64_t id : s->decoders) {
      const Request& r = s->reqs.at(id);
      if (r.limit - r.generated <= s->cfg.near_done_tokens) {
        preempt = true;
        break;
      }
    }
  }
  int64_t near = -1, far = -1;
  int64_t near_seq = INT64_MAX, far_seq = INT64_MAX;
  for (int64_t id : s->prefills) {
    const Request& r = s->reqs.at(id);
    const bool near_done = r.prompt - r.cached <= s->cfg.prefill_chunk;
    if (near_done && r.admitted < near_seq) {
      near = id;
      near_seq = r.admitted;
    } else if (!near_done && r.admitted < far_seq) {
      far = id;
      far_seq = r.admitted;
    }
  }
  if (near >= 0 || (near == -1 && far == -1)) return near;
  return preempt ? -1 : far;
}

}  // namespace

extern "C" {

void mixattn_sched_default_config(mixattn_sched_config* cfg) {
  if (!cfg) return;
  cfg->max_sessions = 16;
  cfg->prefill_chunk = 512;
  cfg->max_pending_per_client = 0;
  cfg->near_done_tokens = 64;
  cfg->max_decode_rows = 0;
}

int mixattn_sched_create(mixattn_sched** out, const mixattn_sched_config* cfg) {
  if (!out || !cfg) return MIXATTN_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->max_sessions < 1 || cfg->prefill_chunk < 1 || cfg->max_pending_per_client < 0 ||
      cfg->near_done_tokens < 0 || cfg->max_decode_rows < 0)
    return MIXATTN_ERR_INVALID_ARG;
  mixattn_sched* s = new (std::nothrow) mixattn_sched();
  if (!s) return MIXATTN_ERR_INVALID_ARG;
  s->cfg = *cfg;
  *out = s;
  return MIXATTN_OK;
}

void mixattn_sched_destroy(mixattn_sched* s) { delete s; }

int mixattn_sched_submit(mixattn_sched* s, int64_t request_id, int32_t client_id, int32_t prompt_len,
                         int32_t max_new_tokens) {
  if (!s || prompt_len < 1 || max_new_tokens < 1) return MIXATTN_ERR_INVALID_ARG;
  if ((int64_t)prompt_len + max_new_tokens > INT32_MAX) return MIXATTN_ERR_INVALID_ARG;
  if (s->reqs.count(request_id)) return MIXATTN_ERR_INVALID_ARG;
  std::deque<int64_t>& q = s->waiting[client_id];
  if (s->cfg.max_pending_per_client > 0 && (int32_t)q.size() >= s->cfg.max_pending_per_client)
    return MIXATTN_ERR_CLIENT_QUOTA;
  Request r;
  r.id = request_id;
  r.client = client_id;
  r.prompt = prompt_len;
  r.limit = max_new_tokens;
  s->reqs[request_id] = r;
  if (q.empty()) s->client_turn.push_back(client_id);
  q.push_back(request_id);
  ++s->n_waiting;
  return MIXATTN_OK;
}

int32_t mixattn_sched_next_batch(mixattn_sched* s, int32_t cap, int32_t* row_kinds, int32_t* seq_lens,
                                 int32_t* q_offsets, int64_t* request_ids, int32_t* kind_out) {
  if (!s || s->built || !row_kinds || !seq_lens || !q_offsets) return MIXATTN_ERR_INVALID_ARG;
  if (cap < s->cfg.max_sessions + 1) return MIXATTN_ERR_INVALID_ARG;
  admit(s);
  std::vector<int64_t> due;
  for (int64_t id : s->decoders)
    if (s->reqs.at(id).due) due.push_back(id);
  int64_t chunk = pick_prefill(s);
  if (due.empty() && chunk < 0 && !s->decoders.empty()) {
    // nothing due and no slice may run: every resident decoder is due again
    for (int64_t id : s->decoders) s->reqs.at(id).due = true;
    due.assign(s->decoders.begin(), s->decoders.end());
  }
  const size_t cap_dec = s->cfg.max_decode_rows > 0 ? (size_t)s->cfg.max_decode_rows : due.size();
  const size_t n_dec = std::min(due.size(), cap_dec);
  // decode first: a slice joins only when every due decoder is served in this step
  if (n_dec < due.size()) chunk = -1;

  s->step_decode.assign(due.begin(), due.begin() + n_dec);
  s->step_chunk = chunk;
  s->step_chunk_len = 0;
  int32_t n = 0;
  for (int64_t id : s->step_decode) {
    Request& r = s->reqs.at(id);
    row_kinds[n] = MIXATTN_ROW_DECODE;
    seq_lens[n] = r.prompt + r.generated;  // the newest output token joins the cache
    q_offsets[n] = seq_lens[n] - 1;
    if (request_ids) request_ids[n] = id;
    ++n;
    r.due = false;
  }
  // PopDecoder: the served decoders move to the back of the queue, in the order served
  if (n_dec > 0) {
    std::deque<int64_t> rest;
    for (int64_t id : s->decoders)
      if (std::find(s->step_decode.begin(), s->step_decode.end(), id) == s->step_decode.end()) rest.push_back(id);
    for (int64_t id : s->step_decode) rest.push_back(id);
    s->decoders.swap(rest);
  }
  if (chunk >= 0) {
    const Request& r = s->reqs.at(chunk);
    s->step_chunk_len = std::min(s->cfg.prefill_chunk, r.prompt - r.cached);
    row_kinds[n] = MIXATTN_ROW_CHUNK;
    seq_lens[n] = r.cached + s->step_chunk_len;
    q_offsets[n] = r.cached;
    if (request_ids) request_ids[n] = chunk;
    ++n;
  }
  int32_t kind = MIXATTN_STEP_IDLE;
  if (n_dec > 0) kind = chunk >= 0 ? MIXATTN_STEP_MERGED : MIXATTN_STEP_DECODE;
  else if (chunk >= 0) kind = MIXATTN_STEP_PREFILL;
  if (kind_out) *kind_out = kind;
  s->built = n > 0;
  return n;
}

int mixattn_sched_complete(mixattn_sched* s, const int64_t* stop_ids, int32_t n_stop) {
  if (!s || !s->built || n_stop < 0 || (n_stop > 0 && !stop_ids)) return MIXATTN_ERR_INVALID_ARG;
  auto stopped = [&](int64_t id) { return std::find(stop_ids, stop_ids + n_stop, id) != stop_ids + n_stop; };
  auto finish = [&](Request& r) {
    r.state = MIXATTN_REQ_DONE;
    r.done_step = s->steps;
    --s->resident;
  };
  for (int64_t id : s->step_decode) {
    Request& r = s->reqs.at(id);
    r.cached += 1;
    r.generated += 1;
    if (r.generated >= r.limit || stopped(id)) {
      finish(r);
      s->decoders.erase(std::find(s->decoders.begin(), s->decoders.end(), id));
    }
  }
  if (s->step_chunk >= 0) {
    Request& r = s->reqs.at(s->step_chunk);
    r.cached += s->step_chunk_len;
    if (r.cached == r.prompt) {  // the prompt is complete: its first output token
      r.generated = 1;
      r.first_token_step = s->steps;
      s->prefills.erase(std::find(s->prefills.begin(), s->prefills.end(), r.id));
      if (r.limit <= 1 || stopped(r.id)) {
        finish(r);
      } else {
        r.state = MIXATTN_REQ_DECODE;
        s->decoders.push_back(r.id);
      }
    }
    // MarkAllDecodersDue: after a step with a chunk every resident decoder is due
    for (int64_t id : s->decoders) s->reqs.at(id).due = true;
  }
  ++s->steps;
  s->built = false;
  s->step_decode.clear();
  s->step_chunk = -1;
  s->step_chunk_len = 0;
  return MIXATTN_OK;
}

int mixattn_sched_request_info(const mixattn_sched* s, int64_t request_id, int32_t* state, int32_t* cached,
                               int32_t* generated, int64_t* first_token_step, int64_t* done_step) {
  if (!s) return MIXATTN_ERR_INVALID_ARG;
  auto it = s->reqs.find(request_id);
  if (it == s->reqs.end()) return MIXATTN_ERR_INVALID_ARG;
  const Request& r = it->second;
  if (state) *state = r.state;
  if (cached) *cached = r.cached;
  if (generated) *generated = r.generated;
  if (first_token_step) *first_token_step = r.first_token_step;
  if (done_step) *done_step = r.done_step;
  return MIXATTN_OK;
}

int mixattn_sched_counts(const mixattn_sched* s, int32_t* waiting, int32_t* prefills, int32_t* decoders,
                         int64_t* steps) {
  if (!s) return MIXATTN_ERR_INVALID_ARG;
  if (waiting) *waiting = s->n_waiting;
  if (prefills) *prefills = (int32_t)s->prefills.size();
  if (decoders) *decoders = (int32_t)s->decoders.size();
  if (steps) *steps = s->steps;
  return MIXATTN_OK;
}

}  // extern "C"
