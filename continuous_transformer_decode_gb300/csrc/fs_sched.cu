// Host scheduler around decode_step_batch: fill / gather / step / fold with
// decode-first, bounded prefill ("Fat-station continuous batching",
// "Components" item 3; "DGR-012", "Summary"). Policy details are stated in
// include/fs_sched.h. Host code only.

#include <algorithm>
#include <chrono>
#include <cstring>
#include <deque>
#include <map>
#include <memory>
#include <string>
#include <vector>

#include "../../include/fs.h"
#include "../../include/fs_sched.h"

namespace {

// What one batched step needs from a model.
struct Engine {
  virtual ~Engine() = default;
  virtual int capacity() const = 0;
  virtual int64_t lane_tokens() const = 0;  // KV tokens one lane can hold; 0 = no bound
  virtual int reset(int lane) = 0;
  virtual int clone(int src, int dst) = 0;            // dst (empty) takes src's history
  virtual int evict(int lane, int start, int end) = 0;  // positions [start, end) leave
  // n rows (lane, position, token); a lane on several rows has them at its
  // next consecutive positions (chunked); positions advanced on success
  virtual int step(const int32_t* lanes, int32_t* positions, const int32_t* tokens, int n,
                   bool chunked) = 0;
  virtual int sample(int n, const float* temps, const uint64_t* seeds,
                     const uint64_t* counters, int32_t* out) = 0;
  virtual std::string error() const = 0;
};

struct GpuEngine : Engine {
  fs_handle* h;
  int cap;
  explicit GpuEngine(fs_handle* hh, int c) : h(hh), cap(c) {}
  int capacity() const override { return cap; }
  int64_t lane_tokens() const override {
    int32_t t = 0;
    return fs_lane_capacity(h, &t) == FS_OK ? t : 0;
  }
  int reset(int lane) override { return fs_lane_reset(h, lane); }
  int clone(int src, int dst) override { return fs_lane_clone(h, src, dst); }
  int evict(int lane, int start, int end) override { return fs_lane_evict(h, lane, start, end); }
  int step(const int32_t* lanes, int32_t* positions, const int32_t* tokens, int n,
           bool chunked) override {
    return chunked ? fs_step_batch_chunked(h, lanes, positions, tokens, n, nullptr)
                   : fs_decode_step_batch(h, lanes, positions, tokens, n, nullptr);
  }
  int sample(int n, const float* temps, const uint64_t* seeds, const uint64_t* counters,
             int32_t* out) override {
    return fs_sample(h, n, temps, seeds, counters, out);
  }
  std::string error() const override { return fs_last_error(h); }
};

uint64_t mix64(uint64_t z) {  // splitmix64 finaliser
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Deterministic stand-in for a model: each lane hashes the tokens it consumed
// (the running hash after every token is kept, so a suffix can be evicted).
struct ModelFreeEngine : Engine {
  static constexpr uint64_t kInit = 0xCBF29CE484222325ull;
  int cap, vocab;
  std::vector<std::vector<uint64_t>> hist;  // per lane: the hash after each token
  std::vector<int32_t> last_lanes;
  ModelFreeEngine(int c, int v) : cap(c), vocab(v), hist(c) {}
  int capacity() const override { return cap; }
  int64_t lane_tokens() const override { return 0; }
  uint64_t hash(int lane) const { return hist[lane].empty() ? kInit : hist[lane].back(); }
  int fail_resets = 0;  // host-side fault injection: the next n resets fail
  int reset(int lane) override {
    if (lane < 0 || lane >= cap) return FS_ERR_LANE;
    if (fail_resets > 0) {
      --fail_resets;
      return FS_ERR_CUDA;
    }
    hist[lane].clear();
    return FS_OK;
  }
  int clone(int src, int dst) override {
    if (src < 0 || src >= cap || dst < 0 || dst >= cap) return FS_ERR_LANE;
    if (src == dst || !hist[dst].empty()) return FS_ERR_STATE;
    hist[dst] = hist[src];
    return FS_OK;
  }
  int evict(int lane, int start, int end) override {
    if (lane < 0 || lane >= cap) return FS_ERR_LANE;
    if (start < 0 || start > end || end != (int)hist[lane].size()) return FS_ERR_ARG;
    hist[lane].resize(start);
    return FS_OK;
  }
  int step(const int32_t* lanes, int32_t* positions, const int32_t* tokens, int n,
           bool) override {
    // rows in order; a lane's rows at its next consecutive positions
    std::vector<int32_t> at(cap);
    for (int k = 0; k < cap; ++k) at[k] = (int32_t)hist[k].size();
    for (int i = 0; i < n; ++i) {
      if (lanes[i] < 0 || lanes[i] >= cap) return FS_ERR_LANE;
      if (positions[i] != at[lanes[i]]) return FS_ERR_POSITION;
      if (tokens[i] < 0 || tokens[i] >= vocab) return FS_ERR_TOKEN;
      at[lanes[i]] += 1;
    }
    last_lanes.assign(lanes, lanes + n);
    for (int i = 0; i < n; ++i) {
      const uint64_t hh = (hash(lanes[i]) ^ (uint64_t)(uint32_t)tokens[i]) * 0x100000001B3ull;
      hist[lanes[i]].push_back(hh);
      positions[i] += 1;
    }
    return FS_OK;
  }
  int sample(int n, const float* temps, const uint64_t* seeds, const uint64_t* counters,
             int32_t* out) override {
    if (n != (int)last_lanes.size()) return FS_ERR_STATE;
    for (int i = 0; i < n; ++i) {
      const uint64_t hh = hash(last_lanes[i]);
      uint64_t v = hh;
      if (temps[i] != 0.0f) v = hh ^ mix64(seeds[i] + 0x9E3779B97F4A7C15ull * (counters[i] + 1));
      out[i] = (int32_t)(v % (uint64_t)vocab);
    }
    return FS_OK;
  }
  std::string error() const override { return "model-free engine"; }
};

struct Job {
  int64_t id;
  int64_t need;  // KV tokens reserved: prompt + max_new
  std::vector<int32_t> prompt;
  int32_t max_new;
  float temp;
  uint64_t seed;
  int32_t stop;
};

struct Lane {
  bool busy = false;
  Job job;
  int32_t feed = 0;
  std::vector<int32_t> gen;
  int32_t last = 0;
  int64_t seq = 0;
  int32_t pos = 0;
};

}  // namespace

struct fs_sched {
  std::unique_ptr<Engine> eng;
  fs_sched_config cfg{};
  std::deque<Job> pending;
  std::vector<Lane> lanes;
  std::map<int64_t, std::vector<int32_t>> done;
  std::map<int64_t, int32_t> done_state;  // FS_JOB_DONE_* or FS_JOB_CANCELLED
  int64_t next_id = 0, admit_seq = 0;
  int64_t reserved = 0;  // KV tokens reserved by the lanes' jobs
  bool clock_started = false;
  std::chrono::steady_clock::time_point t_first, t_last;
  fs_sched_stats st{};
  double occ_sum = 0.0;
  std::vector<int32_t> last_batch;
  std::string err;
  // per-step buffers
  std::vector<int32_t> b_lanes, b_pos, b_tok, b_out;
  std::vector<float> b_temp;
  std::vector<uint64_t> b_seed, b_ctr;

  int fail(int code, const std::string& m) {
    err = m;
    return code;
  }
};

namespace {

int make(std::unique_ptr<Engine> eng, const fs_sched_config* cfg, fs_sched** out) {
  if (!cfg || !out) return FS_ERR_ARG;
  if (cfg->lanes < 1 || cfg->lanes > eng->capacity() || cfg->max_prefill_tokens_per_tick < 1 ||
      cfg->max_queue < 0 || cfg->prefill_chunk < 0 || cfg->kv_budget_tokens < 0 ||
      cfg->prefix_reuse_min < 0)
    return FS_ERR_ARG;
  fs_sched* s = new fs_sched();
  s->eng = std::move(eng);
  s->cfg = *cfg;
  s->st.kv_budget_tokens = cfg->kv_budget_tokens;
  s->lanes.resize(cfg->lanes);
  *out = s;
  return FS_OK;
}

}  // namespace

namespace {
// Token a lane fed at position p (p < its position): its prompt, then its
// generated tokens fed back.
int32_t fed_token(const Lane& l, int p) {
  const int P = (int)l.job.prompt.size();
  return p < P ? l.job.prompt[p] : l.gen[p - P];
}

// Prefix reuse for the job just admitted into lane k (see fs_sched.h).
int reuse_prefix(fs_sched* s, int k) {
  Lane& ln = s->lanes[k];
  const int cap = (int)ln.job.prompt.size() - 1;
  int best = 0, src = -1;
  for (int j = 0; j < s->cfg.lanes; ++j) {
    const Lane& o = s->lanes[j];
    if (j == k || !o.busy) continue;
    const int lim = std::min(cap, o.pos);
    int c = 0;
    while (c < lim && fed_token(o, c) == ln.job.prompt[c]) ++c;
    if (c > best) {
      best = c;
      src = j;
    }
  }
  if (src < 0 || best < s->cfg.prefix_reuse_min) return FS_OK;
  int rc = s->eng->clone(src, k);
  if (rc) return s->fail(rc, "prefix clone: " + s->eng->error());
  rc = s->eng->evict(k, best, s->lanes[src].pos);
  if (rc) return s->fail(rc, "prefix evict: " + s->eng->error());
  ln.pos = best;
  ln.feed = best;
  s->st.prefix_hits += 1;
  s->st.prefix_tokens += best;
  return FS_OK;
}
}  // namespace

extern "C" {

int fs_sched_create(fs_handle* h, const fs_sched_config* cfg, fs_sched** out) {
  if (!h || !cfg || cfg->lanes < 1) return FS_ERR_ARG;
  int32_t len = 0;  // the handle must address lanes 0 .. cfg->lanes - 1
  if (fs_lane_length(h, cfg->lanes - 1, &len) != FS_OK) return FS_ERR_ARG;
  return make(std::unique_ptr<Engine>(new GpuEngine(h, cfg->lanes)), cfg, out);
}

int fs_sched_create_model_free(const fs_sched_config* cfg, int32_t vocab, fs_sched** out) {
  if (!cfg || vocab < 1) return FS_ERR_ARG;
  return make(std::unique_ptr<Engine>(new ModelFreeEngine(cfg->lanes, vocab)), cfg, out);
}

int fs_sched_model_free_fail_resets(fs_sched* s, int32_t n) {
  if (!s || n < 0) return FS_ERR_ARG;
  ModelFreeEngine* e = dynamic_cast<ModelFreeEngine*>(s->eng.get());
  if (!e) return s->fail(FS_ERR_STATE, "not a model-free scheduler");
  e->fail_resets = n;
  return FS_OK;
}

int fs_sched_destroy(fs_sched* s) {
  delete s;
  return FS_OK;
}

int fs_sched_submit(fs_sched* s, const fs_job* j, int64_t* job_id_out) {
  if (!s || !j) return FS_ERR_ARG;
  if (!j->prompt || j->prompt_len < 1 || j->max_new_tokens < 1 || !(j->temperature >= 0.0f))
    return s->fail(FS_ERR_ARG, "job needs a prompt, max_new_tokens >= 1, temperature >= 0");
  const int64_t need = (int64_t)j->prompt_len + j->max_new_tokens;
  const int64_t lane_cap = s->eng->lane_tokens();
  if ((s->cfg.kv_budget_tokens > 0 && need > s->cfg.kv_budget_tokens) ||
      (lane_cap > 0 && need > lane_cap)) {
    s->st.rejected += 1;
    s->st.rejected_kv_budget += 1;
    return s->fail(FS_ERR_KV_BUDGET, "prompt + new tokens exceed the KV budget");
  }
  if (s->cfg.max_queue > 0 && (int)s->pending.size() >= s->cfg.max_queue) {
    s->st.rejected += 1;
    s->st.rejected_queue_full += 1;
    return s->fail(FS_ERR_QUEUE_FULL, "pending queue is full");
  }
  Job job;
  job.id = s->next_id++;
  job.need = need;
  job.prompt.assign(j->prompt, j->prompt + j->prompt_len);
  job.max_new = j->max_new_tokens;
  job.temp = j->temperature;
  job.seed = j->seed;
  job.stop = j->stop_token;
  s->pending.push_back(std::move(job));
  s->st.jobs_submitted += 1;
  if (job_id_out) *job_id_out = s->next_id - 1;
  return FS_OK;
}

int fs_sched_step(fs_sched* s, int32_t* n_retired_out) {
  if (!s) return FS_ERR_ARG;
  if (n_retired_out) *n_retired_out = 0;
  const int L = s->cfg.lanes;
  // ---- fill: free lanes in lane order take the oldest pending jobs while
  // their KV reservations fit the budget (no overtaking)
  const int64_t budget_kv = s->cfg.kv_budget_tokens;
  for (int k = 0; k < L && !s->pending.empty(); ++k) {
    Lane& ln = s->lanes[k];
    if (ln.busy) continue;
    if (budget_kv > 0 && s->reserved + s->pending.front().need > budget_kv) {
      s->st.kv_wait_steps += 1;
      break;
    }
    // the reservation is taken only once the lane is reset: a failed reset
    // leaves the job pending and the reserved count unchanged
    int rc = s->eng->reset(k);
    if (rc) return s->fail(rc, "lane reset: " + s->eng->error());
    s->reserved += s->pending.front().need;
    s->st.kv_reserved_max = std::max(s->st.kv_reserved_max, s->reserved);
    ln.busy = true;
    ln.job = std::move(s->pending.front());
    s->pending.pop_front();
    ln.feed = 0;
    ln.gen.clear();
    ln.last = 0;
    ln.pos = 0;
    ln.seq = s->admit_seq++;
    if (s->cfg.prefix_reuse_min > 0) {
      rc = reuse_prefix(s, k);
      if (rc) return rc;
    }
  }
  // ---- gather: decode lanes always (one row each); prompt lanes oldest
  // first, each up to prefill_chunk tokens, within the prompt-token budget
  // and within L rows in all
  std::vector<int> prompt_lanes;
  std::vector<int32_t> take(L, 0);
  int rows_left = L;
  for (int k = 0; k < L; ++k) {
    const Lane& ln = s->lanes[k];
    if (!ln.busy) continue;
    if (ln.feed >= (int)ln.job.prompt.size()) {
      take[k] = 1;
      --rows_left;
    } else {
      prompt_lanes.push_back(k);
    }
  }
  std::sort(prompt_lanes.begin(), prompt_lanes.end(),
            [&](int a, int b) { return s->lanes[a].seq < s->lanes[b].seq; });
  int left = std::max(1, s->cfg.max_prefill_tokens_per_tick);
  const int chunk = std::max(1, s->cfg.prefill_chunk);
  for (int k : prompt_lanes) {
    const Lane& ln = s->lanes[k];
    const int t = std::min(std::min((int)ln.job.prompt.size() - ln.feed, chunk),
                           std::min(left, rows_left));
    if (t <= 0) break;
    take[k] = t;
    left -= t;
    rows_left -= t;
  }
  s->b_lanes.clear();
  s->b_pos.clear();
  s->b_tok.clear();
  bool chunked = false;
  for (int k = 0; k < L; ++k) {
    const Lane& ln = s->lanes[k];
    chunked = chunked || take[k] > 1;
    for (int r = 0; r < take[k]; ++r) {
      const int f = ln.feed + r;
      s->b_lanes.push_back(k);
      s->b_pos.push_back(ln.pos + r);
      s->b_tok.push_back(f < (int)ln.job.prompt.size() ? ln.job.prompt[f] : ln.last);
    }
  }
  const int n = (int)s->b_lanes.size();
  if (n == 0) return FS_OK;
  if (!s->clock_started) {
    s->clock_started = true;
    s->t_first = std::chrono::steady_clock::now();
  }
  // ---- one batched step, then one sample over the step's rows
  int rc = s->eng->step(s->b_lanes.data(), s->b_pos.data(), s->b_tok.data(), n, chunked);
  if (rc) return s->fail(rc, "decode step: " + s->eng->error());
  s->b_temp.resize(n);
  s->b_seed.resize(n);
  s->b_ctr.resize(n);
  s->b_out.resize(n);
  for (int i = 0; i < n; ++i) {
    const Lane& ln = s->lanes[s->b_lanes[i]];
    s->b_temp[i] = ln.job.temp;
    s->b_seed[i] = ln.job.seed;
    s->b_ctr[i] = (uint64_t)ln.gen.size();
  }
  rc = s->eng->sample(n, s->b_temp.data(), s->b_seed.data(), s->b_ctr.data(), s->b_out.data());
  if (rc) return s->fail(rc, "sample: " + s->eng->error());
  s->last_batch = s->b_lanes;
  s->t_last = std::chrono::steady_clock::now();
  s->st.steps += 1;
  s->st.occupancy_last = n;
  s->st.occupancy_max = std::max(s->st.occupancy_max, n);
  s->occ_sum += n;
  // ---- fold: a lane's rows advance its feed; its last row's token counts
  // once the prompt is consumed
  int retired = 0;
  for (int i = 0; i < n;) {
    const int k = s->b_lanes[i];
    Lane& ln = s->lanes[k];
    const int last = i + take[k] - 1;
    for (; i <= last; ++i) {
      ln.pos += 1;
      if (ln.feed < (int)ln.job.prompt.size())
        s->st.prefill_tokens += 1;
      else
        s->st.decode_tokens += 1;
      ln.feed += 1;
    }
    if (ln.feed < (int)ln.job.prompt.size()) continue;
    const int32_t t = s->b_out[last];
    ln.gen.push_back(t);
    ln.last = t;
    if ((int)ln.gen.size() >= ln.job.max_new || (ln.job.stop >= 0 && t == ln.job.stop)) {
      s->done[ln.job.id] = ln.gen;
      s->done_state[ln.job.id] =
          (ln.job.stop >= 0 && t == ln.job.stop) ? FS_JOB_DONE_STOP : FS_JOB_DONE_LENGTH;
      s->reserved -= ln.job.need;
      ln.busy = false;
      s->st.jobs_done += 1;
      ++retired;
    }
  }
  if (n_retired_out) *n_retired_out = retired;
  return FS_OK;
}

int fs_sched_run(fs_sched* s, int64_t max_steps, int64_t* steps_out) {
  if (!s) return FS_ERR_ARG;
  int64_t k = 0;
  auto busy = [&] {
    if (!s->pending.empty()) return true;
    for (const Lane& l : s->lanes)
      if (l.busy) return true;
    return false;
  };
  while (busy() && k < max_steps) {
    int rc = fs_sched_step(s, nullptr);
    if (rc) return rc;
    ++k;
  }
  if (steps_out) *steps_out = k;
  return FS_OK;
}

int fs_sched_take(fs_sched* s, int64_t job_id, int32_t* tokens_out, int32_t cap,
                  int32_t* n_out) {
  if (!s || !n_out || cap < 0 || (cap > 0 && !tokens_out)) return FS_ERR_ARG;
  auto it = s->done.find(job_id);
  if (it == s->done.end()) return s->fail(FS_ERR_STATE, "job unknown or not finished");
  const int n = (int)it->second.size();
  std::memcpy(tokens_out, it->second.data(), (size_t)std::min(n, cap) * 4);
  *n_out = n;
  s->done.erase(it);
  s->done_state.erase(job_id);
  return FS_OK;
}

int fs_sched_status(const fs_sched* s, int64_t job_id, int32_t* state_out) {
  if (!s || !state_out) return FS_ERR_ARG;
  *state_out = FS_JOB_UNKNOWN;
  for (const Job& j : s->pending)
    if (j.id == job_id) *state_out = FS_JOB_QUEUED;
  for (const Lane& l : s->lanes)
    if (l.busy && l.job.id == job_id) *state_out = FS_JOB_RUNNING;
  auto it = s->done_state.find(job_id);
  if (it != s->done_state.end()) *state_out = it->second;
  return FS_OK;
}

int fs_sched_cancel(fs_sched* s, int64_t job_id) {
  if (!s) return FS_ERR_ARG;
  for (auto it = s->pending.begin(); it != s->pending.end(); ++it)
    if (it->id == job_id) {
      s->pending.erase(it);
      s->done[job_id] = {};
      s->done_state[job_id] = FS_JOB_CANCELLED;
      s->st.jobs_cancelled += 1;
      return FS_OK;
    }
  for (int k = 0; k < s->cfg.lanes; ++k) {
    Lane& ln = s->lanes[k];
    if (!ln.busy || ln.job.id != job_id) continue;
    const int rc = s->eng->reset(k);
    if (rc) return s->fail(rc, "lane reset: " + s->eng->error());
    s->done[job_id] = ln.gen;
    s->done_state[job_id] = FS_JOB_CANCELLED;
    s->reserved -= ln.job.need;
    ln.busy = false;
    s->st.jobs_cancelled += 1;
    return FS_OK;
  }
  return s->fail(FS_ERR_STATE, "job unknown or already finished");
}

int fs_sched_get_stats(const fs_sched* s, fs_sched_stats* out) {
  if (!s || !out) return FS_ERR_ARG;
  *out = s->st;
  int active = 0;
  for (const Lane& l : s->lanes) active += l.busy ? 1 : 0;
  out->active = active;
  out->queued = (int32_t)s->pending.size();
  out->occupancy_avg = s->st.steps ? s->occ_sum / (double)s->st.steps : 0.0;
  out->kv_reserved_tokens = s->reserved;
  out->seconds = s->clock_started
                     ? std::chrono::duration<double>(s->t_last - s->t_first).count()
                     : 0.0;
  out->prefill_tok_s = out->seconds > 0 ? (double)s->st.prefill_tokens / out->seconds : 0.0;
  out->decode_tok_s = out->seconds > 0 ? (double)s->st.decode_tokens / out->seconds : 0.0;
  return FS_OK;
}

int fs_sched_last_batch(const fs_sched* s, int32_t* lanes_out, int32_t cap, int32_t* n_out) {
  if (!s || !n_out || cap < 0 || (cap > 0 && !lanes_out)) return FS_ERR_ARG;
  const int n = (int)s->last_batch.size();
  std::memcpy(lanes_out, s->last_batch.data(), (size_t)std::min(n, cap) * 4);
  *n_out = n;
  return FS_OK;
}

const char* fs_sched_last_error(const fs_sched* s) { return s ? s->err.c_str() : ""; }

}  // extern "C"
