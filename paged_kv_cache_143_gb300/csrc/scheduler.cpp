// scheduler.cpp — the host scheduler and block manager (pa_sched_*), host C++.
//
// [V1-blog "고정 예산 기반 청크 분할 알고리즘"]: a per-step token budget; one
// token for every running decode first, the rest in prefill chunks of
// min(remaining prompt, remaining budget, cap). [vLLM-wiki "블록 테이블"]:
// blocks are taken when a token lands past the last one. [vLLM-wiki "블록
// 공유와 쓰기 시 복사"]: reference counts, copy before writing into a shared
// block. [vLLM-wiki "스케줄링과 선점"]: first come, first served; when blocks
// run out the latest arrival is preempted and later recomputed. [vLLM-wiki
// "엔진 구조와 주요 기능", automatic prefix caching]: full blocks keyed by
// (previous key, tokens, salt), reused by matching prefixes, unreferenced
// ones evicted in LRU order. [MRV2 "재설계 1", "재설계 3"]: persistent slots,
// table diffs.
//
// Data structures: blocks are a reference-count array, a free stack (lowest
// id on top initially) and an LRU list of cached unreferenced blocks (O(1)
// unlink through stored iterators); the prefix cache is a hash map from a
// 64-bit chained key to its block; requests live in a map by id, the waiting
// queue is ordered by arrival and the running list by admission; free slots
// are an ordered set. Every step reuses the same output vectors.
#include <algorithm>
#include <list>
#include <memory>
#include <set>
#include <unordered_map>
#include <vector>

#include "../../include/pa_sched.h"

namespace {

// splitmix64 finaliser: a 64-bit mixer for the prefix keys
inline uint64_t mix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

enum class State { kWaiting, kRunning, kDone };

struct Req {
  int64_t id = 0;
  std::vector<int32_t> tokens;
  int32_t prompt_len = 0, max_new = 0;
  uint64_t salt = 0;
  int64_t arrival = 0;
  int32_t slot = -1;
  std::vector<int32_t> blocks;
  int32_t num_computed = 0, generated = 0;
  bool caught_up = false;     // its last step computed all of its tokens
  int32_t dirty_from = 0;     // first table entry the device row lacks
  std::vector<uint64_t> keys; // keys of its full blocks, in order
  State state = State::kWaiting;
};

}  // namespace

struct pa_sched {
  pa_sched_config cfg{};
  // ---- blocks
  std::vector<int32_t> ref;
  std::vector<int32_t> free_stack;  // back = next taken
  std::list<int32_t> lru;           // front = released longest ago
  std::vector<std::list<int32_t>::iterator> lru_pos;
  std::vector<char> in_lru;
  std::vector<char> has_key;
  std::vector<uint64_t> key_of;
  std::unordered_map<uint64_t, int32_t> cache;
  // ---- requests
  std::unordered_map<int64_t, std::unique_ptr<Req>> reqs;
  std::vector<Req*> waiting;  // by arrival
  std::vector<Req*> running;  // by admission
  std::set<int32_t> free_slots;
  int64_t arrivals = 0;
  bool pending = false;       // a step awaits its commit
  std::vector<Req*> last;     // entries of the pending step
  std::vector<char> last_done;
  pa_sched_stats st{};
  // ---- output of the last step
  std::vector<int64_t> o_ids, o_slots64;
  std::vector<int32_t> o_idx, o_q, o_qsl, o_seq, o_pos, o_tok, o_rows, o_starts, o_offs, o_vals,
      o_src, o_dst;

  // ------------------------------------------------------------ allocator
  int32_t available() const { return (int32_t)(free_stack.size() + lru.size()); }

  int32_t take() {
    int32_t b;
    if (!free_stack.empty()) {
      b = free_stack.back();
      free_stack.pop_back();
    } else {
      b = lru.front();
      lru.pop_front();
      in_lru[b] = 0;
      cache.erase(key_of[b]);
      has_key[b] = 0;
    }
    ref[b] = 1;
    return b;
  }

  void incref(int32_t b) {
    if (ref[b] == 0 && in_lru[b]) {
      lru.erase(lru_pos[b]);
      in_lru[b] = 0;
    }
    ++ref[b];
  }

  void release(int32_t b) {
    if (--ref[b] == 0) {
      if (has_key[b]) {
        lru.push_back(b);
        lru_pos[b] = std::prev(lru.end());
        in_lru[b] = 1;
      } else {
        free_stack.push_back(b);
      }
    }
  }

  void release_all(Req* r) {
    for (auto it = r->blocks.rbegin(); it != r->blocks.rend(); ++it) release(*it);
    r->blocks.clear();
  }

  void free_slot(Req* r) {
    free_slots.insert(r->slot);
    r->slot = -1;
  }

  void remove_running(Req* r) {
    running.erase(std::find(running.begin(), running.end(), r));
  }

  void insert_waiting(Req* r) {
    auto it = std::find_if(waiting.begin(), waiting.end(),
                           [&](Req* w) { return w->arrival > r->arrival; });
    waiting.insert(it, r);
  }

  void preempt(Req* r) {
    remove_running(r);
    release_all(r);
    free_slot(r);
    r->num_computed = 0;
    r->caught_up = false;
    r->keys.clear();
    r->dirty_from = 0;
    r->state = State::kWaiting;
    insert_waiting(r);
    ++st.preemptions;
  }

  // blocks a step of q tokens needs (new ones plus a copy), and whether the
  // block at the first written position is shared
  int32_t needed(const Req* r, int32_t q, bool* cow) const {
    const int32_t B = cfg.block_size, nc = r->num_computed;
    const int32_t total = (nc + q + B - 1) / B;
    const int32_t fresh = std::max(0, total - (int32_t)r->blocks.size());
    *cow = nc % B != 0 && nc / B < (int32_t)r->blocks.size() && ref[r->blocks[nc / B]] > 1;
    return fresh + (*cow ? 1 : 0);
  }

  int32_t fit(const Req* r, int32_t q) const {
    bool cow;
    needed(r, q, &cow);
    const int64_t avail = (int64_t)available() - (cow ? 1 : 0);
    if (avail < 0) return 0;
    const int64_t most = ((int64_t)r->blocks.size() + avail) * cfg.block_size - r->num_computed;
    return (int32_t)std::max<int64_t>(0, std::min<int64_t>(q, most));
  }

  void ensure(Req* r, int32_t q) {
    bool cow;
    needed(r, q, &cow);
    const int32_t B = cfg.block_size;
    if (cow) {
      const int32_t i = r->num_computed / B;
      const int32_t old = r->blocks[i];
      const int32_t fresh = take();
      release(old);
      r->blocks[i] = fresh;
      o_src.push_back(old);
      o_dst.push_back(fresh);
      r->dirty_from = std::min(r->dirty_from, i);
    }
    while ((int64_t)r->blocks.size() * B < (int64_t)r->num_computed + q) r->blocks.push_back(take());
  }

  uint64_t block_key(const Req* r, int32_t i, uint64_t prev, bool has_prev) const {
    const int32_t B = cfg.block_size;
    uint64_t h = mix64(has_prev ? prev ^ 0x5bd1e9955bd1e995ull : 0x2545F4914F6CDD1Dull);
    for (int32_t k = 0; k < B; ++k) h = mix64(h ^ (uint64_t)(uint32_t)r->tokens[i * B + k]);
    return mix64(h ^ r->salt);
  }

  // ------------------------------------------------------------------ step
  void step(pa_sched_batch* out) {
    const int32_t B = cfg.block_size;
    int32_t budget = cfg.token_budget;
    std::vector<std::pair<Req*, int32_t>> entries;
    std::set<int64_t> scheduled, preempted_now;
    o_src.clear();
    o_dst.clear();
    // 1. one token for every running decode, first
    const std::vector<Req*> snapshot = running;
    for (Req* r : snapshot) {
      if (r->state != State::kRunning) continue;
      if (!(r->caught_up && (int32_t)r->tokens.size() - r->num_computed == 1)) continue;
      if (budget < 1) break;
      bool cow;
      while (needed(r, 1, &cow) > available()) {
        Req* victim = nullptr;
        for (Req* x : running)
          if (!scheduled.count(x->id) && (!victim || x->arrival > victim->arrival)) victim = x;
        preempt(victim);
        preempted_now.insert(victim->id);
        if (victim == r) break;
      }
      if (r->state != State::kRunning) continue;
      ensure(r, 1);
      entries.emplace_back(r, 1);
      scheduled.insert(r->id);
      budget -= 1;
    }
    const int32_t num_decode = (int32_t)entries.size();
    // 2. prefill chunks: running requests first, then admissions in arrival order
    for (Req* r : std::vector<Req*>(running)) {
      if (budget <= 0) break;
      if (scheduled.count(r->id) || r->caught_up) continue;
      const int32_t want = std::min({(int32_t)r->tokens.size() - r->num_computed, budget,
                                     cfg.chunk_cap});
      const int32_t q = fit(r, want);
      if (q <= 0) continue;
      ensure(r, q);
      entries.emplace_back(r, q);
      scheduled.insert(r->id);
      budget -= q;
    }
    while (!waiting.empty() && budget > 0 && !free_slots.empty()) {
      Req* r = waiting.front();
      if (preempted_now.count(r->id)) break;
      std::vector<int32_t> hits;
      std::vector<uint64_t> keys;
      if (cfg.prefix_caching) {
        const int32_t full = ((int32_t)r->tokens.size() - 1) / B;
        for (int32_t i = 0; i < full; ++i) {
          const uint64_t key = block_key(r, i, keys.empty() ? 0 : keys.back(), !keys.empty());
          auto it = cache.find(key);
          if (it == cache.end()) break;
          hits.push_back(it->second);
          keys.push_back(key);
        }
      }
      for (int32_t b : hits) incref(b);
      r->blocks = hits;
      r->keys = keys;
      r->num_computed = (int32_t)hits.size() * B;
      const int32_t want = std::min({(int32_t)r->tokens.size() - r->num_computed, budget,
                                     cfg.chunk_cap});
      const int32_t q = fit(r, want);
      if (q <= 0) {
        release_all(r);
        r->keys.clear();
        r->num_computed = 0;
        break;
      }
      waiting.erase(waiting.begin());
      r->slot = *free_slots.begin();
      free_slots.erase(free_slots.begin());
      r->state = State::kRunning;
      r->dirty_from = 0;
      running.push_back(r);
      st.prefix_hit_tokens += r->num_computed;
      ensure(r, q);
      entries.emplace_back(r, q);
      scheduled.insert(r->id);
      budget -= q;
    }
    // 3. the batch
    o_ids.clear(); o_idx.clear(); o_q.clear(); o_qsl.assign(1, 0); o_seq.clear();
    o_pos.clear(); o_tok.clear(); o_slots64.clear();
    o_rows.clear(); o_starts.clear(); o_offs.assign(1, 0); o_vals.clear();
    last.clear();
    for (auto& [r, q] : entries) {
      const int32_t nc = r->num_computed;
      o_ids.push_back(r->id);
      o_idx.push_back(r->slot);
      o_q.push_back(q);
      o_qsl.push_back(o_qsl.back() + q);
      o_seq.push_back(nc + q);
      for (int32_t p = nc; p < nc + q; ++p) {
        o_pos.push_back(p);
        o_tok.push_back(r->tokens[p]);
        o_slots64.push_back((int64_t)r->blocks[p / B] * B + p % B);
      }
      r->num_computed = nc + q;
      r->caught_up = r->num_computed == (int32_t)r->tokens.size();
      if (cfg.prefix_caching) {
        for (int32_t i = (int32_t)r->keys.size(); i < r->num_computed / B; ++i) {
          const uint64_t key =
              block_key(r, i, r->keys.empty() ? 0 : r->keys.back(), !r->keys.empty());
          r->keys.push_back(key);
          const int32_t blk = r->blocks[i];
          if (!cache.count(key) && !has_key[blk]) {
            cache.emplace(key, blk);
            key_of[blk] = key;
            has_key[blk] = 1;
          }
        }
      }
      if (r->dirty_from < (int32_t)r->blocks.size()) {
        o_rows.push_back(r->slot);
        o_starts.push_back(r->dirty_from);
        o_vals.insert(o_vals.end(), r->blocks.begin() + r->dirty_from, r->blocks.end());
        o_offs.push_back((int32_t)o_vals.size());
        r->dirty_from = (int32_t)r->blocks.size();
      }
      last.push_back(r);
    }
    pending = true;
    ++st.steps;
    st.scheduled_tokens += o_qsl.back();
    out->num_reqs = (int32_t)o_ids.size();
    out->num_tokens = o_qsl.back();
    out->num_decode = num_decode;
    out->req_ids = o_ids.data();
    out->idx_mapping = o_idx.data();
    out->num_scheduled = o_q.data();
    out->query_start_loc = o_qsl.data();
    out->seq_lens = o_seq.data();
    out->positions = o_pos.data();
    out->token_ids = o_tok.data();
    out->slot_mapping = o_slots64.data();
    out->num_diffs = (int32_t)o_rows.size();
    out->diff_rows = o_rows.data();
    out->diff_starts = o_starts.data();
    out->diff_val_offsets = o_offs.data();
    out->diff_vals = o_vals.data();
    out->num_copies = (int32_t)o_src.size();
    out->copy_src = o_src.data();
    out->copy_dst = o_dst.data();
  }

  void finish(Req* r) {
    remove_running(r);
    release_all(r);
    free_slot(r);
    r->state = State::kDone;
  }

  int32_t commit(const int32_t* sampled, int64_t* ids, int32_t cap) {
    int32_t done = 0;
    for (size_t i = 0; i < last.size(); ++i) {
      Req* r = last[i];
      if (!r || r->state != State::kRunning || !r->caught_up) continue;
      r->tokens.push_back(sampled[i]);
      if (++r->generated >= r->max_new) {
        finish(r);
        if (done < cap && ids) ids[done] = r->id;
        ++done;
        ++st.finished;
        reqs.erase(r->id);
      }
    }
    last.clear();
    pending = false;
    return done;
  }
};

extern "C" pa_status pa_sched_create(const pa_sched_config* c, pa_sched** out) {
  if (!c || !out) return PA_ERR_INVALID;
  *out = nullptr;
  if (c->num_blocks <= 0 || c->block_size <= 0 || c->max_reqs <= 0 ||
      c->max_blocks_per_req <= 0 || c->token_budget <= 0 || c->chunk_cap <= 0 ||
      (c->prefix_caching != 0 && c->prefix_caching != 1))
    return PA_ERR_INVALID;
  auto* s = new pa_sched();
  s->cfg = *c;
  const size_t n = (size_t)c->num_blocks;
  s->ref.assign(n, 0);
  s->free_stack.resize(n);
  for (size_t i = 0; i < n; ++i) s->free_stack[i] = (int32_t)(n - 1 - i);
  s->lru_pos.resize(n);
  s->in_lru.assign(n, 0);
  s->has_key.assign(n, 0);
  s->key_of.assign(n, 0);
  for (int32_t i = 0; i < c->max_reqs; ++i) s->free_slots.insert(i);
  *out = s;
  return PA_OK;
}

extern "C" void pa_sched_destroy(pa_sched* s) { delete s; }

extern "C" pa_status pa_sched_add_request(pa_sched* s, int64_t id, const int32_t* prompt,
                                          int32_t prompt_len, int32_t max_new, uint64_t salt) {
  if (!s || !prompt || prompt_len < 1 || max_new < 1 || s->reqs.count(id)) return PA_ERR_INVALID;
  if ((int64_t)prompt_len + max_new >
      (int64_t)s->cfg.max_blocks_per_req * s->cfg.block_size)
    return PA_ERR_INVALID;
  auto r = std::make_unique<Req>();
  r->id = id;
  r->tokens.assign(prompt, prompt + prompt_len);
  r->prompt_len = prompt_len;
  r->max_new = max_new;
  r->salt = salt;
  r->arrival = s->arrivals++;
  s->waiting.push_back(r.get());
  s->reqs.emplace(id, std::move(r));
  return PA_OK;
}

extern "C" pa_status pa_sched_fork(pa_sched* s, int64_t parent, int64_t child, int32_t max_new) {
  if (!s || max_new < 1 || s->reqs.count(child)) return PA_ERR_INVALID;
  auto it = s->reqs.find(parent);
  if (it == s->reqs.end() || it->second->state != State::kRunning) return PA_ERR_INVALID;
  if (s->free_slots.empty()) return PA_ERR_UNSUPPORTED;
  const Req* p = it->second.get();
  auto c = std::make_unique<Req>();
  c->id = child;
  c->tokens = p->tokens;
  c->prompt_len = p->prompt_len;
  c->max_new = max_new;
  c->salt = p->salt;
  c->arrival = s->arrivals++;
  c->blocks = p->blocks;
  for (int32_t b : c->blocks) s->incref(b);
  c->num_computed = p->num_computed;
  c->generated = p->generated;
  c->caught_up = p->caught_up;
  c->keys = p->keys;
  c->slot = *s->free_slots.begin();
  s->free_slots.erase(s->free_slots.begin());
  c->state = State::kRunning;
  s->running.push_back(c.get());
  s->reqs.emplace(child, std::move(c));
  return PA_OK;
}

extern "C" pa_status pa_sched_abort(pa_sched* s, int64_t id) {
  if (!s) return PA_ERR_INVALID;
  auto it = s->reqs.find(id);
  if (it == s->reqs.end()) return PA_ERR_INVALID;
  Req* r = it->second.get();
  if (r->state == State::kRunning) {
    s->finish(r);
  } else {
    s->waiting.erase(std::find(s->waiting.begin(), s->waiting.end(), r));
  }
  for (auto& e : s->last)
    if (e == r) e = nullptr;  // a pending step no longer hands it a token
  s->reqs.erase(it);
  return PA_OK;
}

extern "C" pa_status pa_sched_step(pa_sched* s, pa_sched_batch* batch) {
  if (!s || !batch || s->pending) return PA_ERR_INVALID;
  s->step(batch);
  return PA_OK;
}

extern "C" pa_status pa_sched_commit(pa_sched* s, const int32_t* sampled, int32_t n,
                                     int64_t* finished_ids, int32_t finished_cap,
                                     int32_t* num_finished) {
  if (!s || !s->pending || n != (int32_t)s->last.size() || (n > 0 && !sampled) ||
      finished_cap < 0 || (finished_cap > 0 && !finished_ids))
    return PA_ERR_INVALID;
  const int32_t done = s->commit(sampled, finished_ids, finished_cap);
  if (num_finished) *num_finished = done;
  return PA_OK;
}

extern "C" pa_status pa_sched_get_stats(const pa_sched* s, pa_sched_stats* out) {
  if (!s || !out) return PA_ERR_INVALID;
  *out = s->st;
  out->running = (int32_t)s->running.size();
  out->waiting = (int32_t)s->waiting.size();
  out->free_blocks = (int32_t)s->free_stack.size();
  out->cached_free_blocks = (int32_t)s->lru.size();
  // fill of every referenced block: the most tokens any holder stores in it
  std::unordered_map<int32_t, int32_t> fill;
  const int32_t B = s->cfg.block_size;
  for (const Req* r : s->running)
    for (size_t i = 0; i < r->blocks.size(); ++i) {
      const int32_t n = std::max(0, std::min(B, r->num_computed - (int32_t)i * B));
      int32_t& f = fill[r->blocks[i]];
      f = std::max(f, n);
    }
  int64_t stored = 0;
  for (auto& kv : fill) stored += kv.second;
  out->used_blocks = (int32_t)fill.size();
  out->stored_tokens = stored;
  out->wasted_slots = (int64_t)fill.size() * B - stored;
  return PA_OK;
}

extern "C" pa_status pa_sched_block_table(const pa_sched* s, int64_t id, int32_t* blocks,
                                          int32_t cap, int32_t* n) {
  if (!s || !n || cap < 0 || (cap > 0 && !blocks)) return PA_ERR_INVALID;
  auto it = s->reqs.find(id);
  if (it == s->reqs.end()) return PA_ERR_INVALID;
  const auto& b = it->second->blocks;
  *n = (int32_t)b.size();
  for (int32_t i = 0; i < cap && i < (int32_t)b.size(); ++i) blocks[i] = b[i];
  return PA_OK;
}
