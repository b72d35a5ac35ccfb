/*
 * fs_sched.h — host scheduler around decode_step_batch (continuous batching).
 *
 * Sources (page title, section):
 *   - "Fat-station continuous batching — the live-path integration",
 *     "Components", item 3: the decode thread loops fill (a free lane takes
 *     a pending job: lane reset, position 0), gather (one input token per
 *     live lane: the next prompt token while the prompt lasts, else the last
 *     sampled token), one batched step, fold (feed count + 1; inside the
 *     prompt nothing is sampled; otherwise sample with the lane's
 *     temperature and seed, append, retire on the stop token or
 *     max_new_tokens and free the lane for the next fill).
 *   - "DGR-012 — Continuous batching and bounded admission: evidence",
 *     "Summary": decode first, then bounded prefill — in-flight decodes
 *     always run; prompt work per tick is capped by
 *     max_prefill_tokens_per_tick, with at least one so a long prompt still
 *     progresses; a full queue is refused (backpressure). "Summary",
 *     bounded admission: a session is admitted only if it fits the KV budget
 *     (it must be able to hold its whole generation, prompt + new tokens, on
 *     its own); what cannot fit is rejected up front with its reason; what
 *     fits but finds no room waits in the bounded queue; KV growth stays
 *     within the budget and returns to zero as sessions complete. Telemetry:
 *     active sessions, queue depth, occupancy (last/avg/max), KV pressure,
 *     prefill/decode totals and rates, rejections by reason.
 *
 * Policy (the readings taken where the pages leave it open):
 *   - fill: at the start of a step each free lane, in lane order, takes the
 *     oldest pending job; a lane freed in step t is refilled in step t+1;
 *   - gather: every lane past its prompt is in the step (one row each);
 *     lanes still in their prompt are added oldest-admitted first, each with
 *     up to prefill_chunk of its next prompt tokens (chunked prefill,
 *     "Fat-station continuous batching", "What /generate does today"), until
 *     max_prefill_tokens_per_tick prompt tokens (at least 1) or `lanes` rows
 *     in all; the rows list lanes in lane order and a lane's positions in
 *     ascending order; a step with a lane on several rows runs through
 *     fs_step_batch_chunked, any other through fs_decode_step_batch;
 *   - admission: a job reserves prompt_len + max_new_tokens tokens of KV.
 *     Submit refuses it (FS_ERR_KV_BUDGET) when that exceeds kv_budget_tokens
 *     or the engine's tokens per lane; fill admits the oldest pending job
 *     into a free lane only while the reservations of the lanes' jobs plus
 *     its own stay within kv_budget_tokens, else the queue waits (oldest
 *     first, no overtaking); a retired job releases its reservation. A
 *     session has no external key here, so there is no duplicate check, and
 *     activation scratch is preallocated per lane, so `lanes` is the scratch
 *     bound;
 *   - prefix reuse (prefix_reuse_min > 0; "MODEL-BATCHING-RESULTS", "Why
 *     in-kernel batching, not vLLM": Clone for prefix reuse): when fill
 *     admits a job into lane k, the busy lane whose fed history shares the
 *     longest prefix with the job's prompt (ties: the lowest lane), capped
 *     at prompt_len - 1 tokens, is cloned into k and the clone's history
 *     past that prefix is evicted (fs_lane_clone, fs_lane_evict), provided
 *     the prefix has at least prefix_reuse_min tokens; the job then feeds
 *     only the rest of its prompt. A lane's history is the tokens its job
 *     fed (prompt, then generated tokens fed back). The job's tokens are
 *     those it gives alone: a position's K and V depend only on the tokens
 *     up to it. Its KV reservation is unchanged;
 *   - fold: the step that consumes a prompt's last token yields the job's
 *     first generated token (from that lane's last row); the job's t-th generated token is sampled with
 *     (seed, counter = t), so a job's tokens do not depend on its lane, its
 *     step or its neighbours.
 *
 * Conventions as in fs.h: FS_OK or a negative FS_ERR_* code; a scheduler is
 * used by one host thread at a time; pointers are host pointers.
 */
#ifndef FS_SCHED_H_
#define FS_SCHED_H_

#include "fs.h"

#ifdef __cplusplus
extern "C" {
#endif

#define FS_ERR_QUEUE_FULL (-12) /* bounded pending queue is full (backpressure) */
#define FS_ERR_KV_BUDGET (-13)  /* a job's prompt + new tokens can never fit   */

/* Job states (fs_sched_status). */
#define FS_JOB_UNKNOWN (-1)     /* never submitted, or already taken          */
#define FS_JOB_QUEUED 0         /* waiting for a lane                         */
#define FS_JOB_RUNNING 1        /* on a lane                                  */
#define FS_JOB_DONE_LENGTH 2    /* finished: max_new_tokens generated         */
#define FS_JOB_DONE_STOP 3      /* finished: sampled its stop token           */
#define FS_JOB_CANCELLED 4      /* cancelled (fs_sched_cancel)                */

typedef struct fs_sched fs_sched;

typedef struct fs_sched_config {
  int32_t lanes;                       /* lanes used: 1 .. engine capacity   */
  int32_t max_prefill_tokens_per_tick; /* prompt tokens per step (>= 1)      */
  int32_t max_queue;                   /* pending jobs allowed, 0 = no bound */
  int32_t prefill_chunk;               /* prompt tokens per lane per step;
                                          0 or 1: one (no chunking)         */
  int64_t kv_budget_tokens;            /* KV tokens reserved by the lanes'
                                          jobs at most; 0 = no bound        */
  int32_t prefix_reuse_min;            /* shortest prompt prefix taken from
                                          a running lane; 0 = no reuse      */
} fs_sched_config;

typedef struct fs_job {
  const int32_t* prompt;   /* prompt_len tokens (copied at submit)           */
  int32_t prompt_len;      /* >= 1                                            */
  int32_t max_new_tokens;  /* >= 1                                            */
  float temperature;       /* 0: greedy                                       */
  uint64_t seed;           /* per-job sampling seed                           */
  int32_t stop_token;      /* retire after sampling this token; -1: none      */
} fs_job;

typedef struct fs_sched_stats {
  int64_t steps;           /* batched steps run                               */
  int64_t prefill_tokens;  /* prompt tokens consumed                          */
  int64_t decode_tokens;   /* generated tokens fed back                       */
  int64_t jobs_submitted;
  int64_t jobs_done;
  int64_t rejected;        /* submits refused (all reasons)                   */
  int32_t active;          /* lanes holding a job                             */
  int32_t queued;          /* pending jobs                                    */
  int32_t occupancy_last;  /* lanes in the last step                          */
  int32_t occupancy_max;
  double occupancy_avg;    /* mean rows per step                              */
  int64_t rejected_queue_full;  /* refused: pending queue full               */
  int64_t rejected_kv_budget;   /* refused: prompt + new tokens cannot fit   */
  int64_t kv_reserved_tokens;   /* KV tokens reserved by the lanes' jobs     */
  int64_t kv_reserved_max;      /* the largest reservation so far            */
  int64_t kv_budget_tokens;     /* the configured budget (0 = no bound)      */
  int64_t kv_wait_steps;        /* steps where a free lane waited on the KV
                                   budget                                    */
  double seconds;               /* host time from the first step to the last */
  double prefill_tok_s;         /* prefill_tokens / seconds                  */
  double decode_tok_s;          /* decode_tokens / seconds                   */
  int64_t prefix_hits;          /* admissions that cloned a running lane     */
  int64_t prefix_tokens;        /* prompt tokens taken from clones, not fed  */
  int64_t jobs_cancelled;
} fs_sched_stats;

/* Scheduler over a decode handle: each step is one fs_decode_step_batch
 * (logits kept inside the handle) and one fs_sample over the step's lanes.
 * cfg->lanes must not exceed the handle's max_lanes. The handle must outlive
 * the scheduler. Errors: FS_ERR_ARG. */
int fs_sched_create(fs_handle* h, const fs_sched_config* cfg, fs_sched** out);

/* Scheduler over a model-free engine (no GPU): a lane's "model" keeps a
 * running 64-bit hash of the tokens it consumed; after a step, greedy lanes
 * draw hash % vocab and sampled lanes (hash ^ mix(seed, counter)) % vocab,
 * where mix is the splitmix64 finaliser of seed + 0x9E3779B97F4A7C15 *
 * (counter + 1) and the hash update is h = (h ^ token) * 0x100000001B3 over
 * an initial 0xCBF29CE484222325 at lane reset. A clone copies a lane's
 * hashes; an evict of a suffix returns to the hash after the kept tokens
 * (only suffixes can be evicted). For testing the policy. */
int fs_sched_create_model_free(const fs_sched_config* cfg, int32_t vocab,
                               fs_sched** out);

/* Host-side fault injection for tests of the policy (the pages have no
 * counterpart): the model-free engine of s fails its next n lane resets with
 * FS_ERR_CUDA, as a GPU engine would on a failed CUDA call. A step whose fill
 * meets such a failure returns that error with the job still pending and
 * the KV reservation not taken. Errors: FS_ERR_ARG (n < 0), FS_ERR_STATE (s
 * is not over the model-free engine). */
int fs_sched_model_free_fail_resets(fs_sched* s, int32_t n);

int fs_sched_destroy(fs_sched* s);

/* Queues a job (FIFO). *job_id_out receives its id (0, 1, ... in submit
 * order). Errors: FS_ERR_ARG, FS_ERR_QUEUE_FULL (nothing queued). */
int fs_sched_submit(fs_sched* s, const fs_job* job, int64_t* job_id_out);

/* One fill / gather / step / fold. *n_retired_out (optional) receives the
 * number of jobs that finished in this step. Idle (no lane, no job) is a
 * no-op. Errors: those of the engine (the scheduler state is then
 * undefined). */
int fs_sched_step(fs_sched* s, int32_t* n_retired_out);

/* Steps until no job is queued or running, at most max_steps steps. */
int fs_sched_run(fs_sched* s, int64_t max_steps, int64_t* steps_out);

/* Copies a finished or cancelled job's generated tokens (up to cap) and
 * their count, then forgets the job. Errors: FS_ERR_STATE (unknown job, or
 * one still queued or running). */
int fs_sched_take(fs_sched* s, int64_t job_id, int32_t* tokens_out,
                  int32_t cap, int32_t* n_out);

int fs_sched_get_stats(const fs_sched* s, fs_sched_stats* out);

/* State of a job: one of FS_JOB_* (a taken job is unknown again). */
int fs_sched_status(const fs_sched* s, int64_t job_id, int32_t* state_out);

/* Cancels a queued or running job between steps (failure and cancellation
 * handling of "DGR-012", "Summary": the KV is released when a session ends):
 * a queued job leaves the queue; a running job's lane is reset (its pages go
 * back to the pool), its KV reservation is released and the lane is free for
 * the next fill. The tokens generated so far stay for fs_sched_take; the
 * job's state becomes FS_JOB_CANCELLED. Errors: FS_ERR_STATE (unknown or
 * already finished job), the engine's (lane reset). */
int fs_sched_cancel(fs_sched* s, int64_t job_id);

/* Lanes of the last step in batch order (inspection hook). */
int fs_sched_last_batch(const fs_sched* s, int32_t* lanes_out, int32_t cap,
                        int32_t* n_out);

/* Message of the last failure on s. */
const char* fs_sched_last_error(const fs_sched* s);

#ifdef __cplusplus
}
#endif
#endif /* FS_SCHED_H_ */
