/*
 * pa_sched.h — C ABI of the host scheduler and block manager of libpa (host
 * code only: no call here touches the GPU).
 *
 * Each step the scheduler decides which requests run and how many tokens
 * each computes, keeps every request's block table, and emits what the
 * device calls of pa.h need for that step: the (row, start, values) diffs for
 * pa_apply_staged_writes, the copy-on-write pairs for pa_copy_blocks, the
 * persistent slots and counts for pa_prepare_inputs, and the host mirrors
 * (query_start_loc, seq_lens) and slot mapping for pa_forward / pa_write_kv.
 *
 * Rules (source pages as in pa.h):
 *  - [V1-blog, "고정 예산 기반 청크 분할 알고리즘"]: a step has a token budget;
 *    every running decode gets its one token first (in admission order); the
 *    rest goes to prefill chunks of min(remaining prompt, remaining budget,
 *    chunk_cap) tokens, first for requests already running, then for waiting
 *    ones in arrival order (first come, first served).
 *  - [vLLM-wiki, "블록 테이블"]: a physical block is taken only when a token
 *    lands past the request's last block.
 *  - [vLLM-wiki, "블록 공유와 쓰기 시 복사"]: blocks carry reference counts
 *    (pa_sched_fork shares all blocks of a running request); a request that
 *    writes into a shared block first copies it (a pair in copy_src/copy_dst).
 *  - [vLLM-wiki, "스케줄링과 선점"]: when a decode finds no free block, the
 *    running request that arrived last (and is not yet in this step) is
 *    preempted: all of its blocks are released and it is recomputed from its
 *    first token when it is admitted again (never in the same step).
 *  - [vLLM-wiki, "엔진 구조와 주요 기능", automatic prefix caching]: with
 *    prefix_caching, every full block is keyed by a 64-bit hash of (the
 *    previous block's key, its tokens, the request's salt); an admitted
 *    request reuses the blocks of its longest cached prefix of full blocks
 *    (never its whole prompt: the last prompt token is computed); blocks that
 *    no request references stay cached and are evicted least recently
 *    released first, only when no free block is left.
 *  - [MRV2, "재설계 1"]: a running request holds a persistent slot (the
 *    lowest free one) until it finishes, aborts or is preempted.
 *  - [MRV2, "재설계 3"]: the device table receives only diffs.
 * Choices the pages leave open: free blocks form a stack whose lowest id
 * comes out first; a request's blocks are released last block first; the
 * copy of a shared block is taken before a step's new blocks.
 *
 * Ownership: the scheduler object is created by pa_sched_create and released
 * by pa_sched_destroy. Arrays in pa_sched_batch belong to the scheduler and
 * stay valid until its next pa_sched_step or pa_sched_destroy. Calls on one
 * scheduler must not overlap (it is not thread-safe); distinct schedulers are
 * independent. Errors: PA_ERR_INVALID for a bad argument or call order (the
 * scheduler is left unchanged), PA_ERR_UNSUPPORTED when a fork finds no free
 * slot.
 */
#ifndef PA_SCHED_H_
#define PA_SCHED_H_

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_sched pa_sched;

typedef struct {
  int32_t num_blocks;          /* physical blocks of the pool                      */
  int32_t block_size;          /* tokens per block (B)                             */
  int32_t max_reqs;            /* persistent slots = rows of the device table      */
  int32_t max_blocks_per_req;  /* columns of the device table                      */
  int32_t token_budget;        /* tokens per step                                  */
  int32_t chunk_cap;           /* largest prefill chunk                            */
  int32_t prefix_caching;      /* 1: reuse cached full blocks of matching prefixes */
} pa_sched_config;

/* One step. Entry i (0 <= i < num_reqs) is request req_ids[i] in slot
 * idx_mapping[i], computing num_scheduled[i] tokens at positions
 * seq_lens[i] - num_scheduled[i] .. seq_lens[i] - 1; decodes come first
 * (entries 0 .. num_decode-1, one token each). */
typedef struct {
  int32_t num_reqs;
  int32_t num_tokens;
  int32_t num_decode;
  const int64_t* req_ids;           /* [R]                                        */
  const int32_t* idx_mapping;       /* [R]                                        */
  const int32_t* num_scheduled;     /* [R]                                        */
  const int32_t* query_start_loc;   /* [R+1]                                      */
  const int32_t* seq_lens;          /* [R]                                        */
  const int32_t* positions;         /* [T]                                        */
  const int32_t* token_ids;         /* [T] the tokens whose K/V this step computes */
  const int64_t* slot_mapping;      /* [T] pool slot = block * B + offset         */
  int32_t num_diffs;                /* W: table diffs, in record order            */
  const int32_t* diff_rows;         /* [W]                                        */
  const int32_t* diff_starts;       /* [W]                                        */
  const int32_t* diff_val_offsets;  /* [W+1]                                      */
  const int32_t* diff_vals;         /* [diff_val_offsets[W]]                      */
  int32_t num_copies;               /* copy-on-write pairs, before the KV writes  */
  const int32_t* copy_src;          /* [num_copies]                               */
  const int32_t* copy_dst;          /* [num_copies]                               */
} pa_sched_batch;

typedef struct {
  int64_t steps;
  int64_t scheduled_tokens;   /* summed over steps                               */
  int64_t preemptions;
  int64_t prefix_hit_tokens;  /* tokens served from cached blocks at admission   */
  int64_t finished;
  int32_t running;
  int32_t waiting;
  int32_t free_blocks;        /* never used or released uncached                */
  int32_t cached_free_blocks; /* unreferenced but kept for prefix reuse          */
  int32_t used_blocks;        /* referenced by a running request                 */
  int64_t stored_tokens;      /* slots of used blocks holding K/V (once each)    */
  int64_t wasted_slots;       /* used_blocks * B - stored_tokens                 */
} pa_sched_stats;

pa_status pa_sched_create(const pa_sched_config* config, pa_sched** sched);
void pa_sched_destroy(pa_sched* sched);

/* Queues a request (waiting). prompt: host int32 [prompt_len], copied;
 * prompt_len >= 1, max_new_tokens >= 1, prompt_len + max_new_tokens <=
 * max_blocks_per_req * block_size, req_id not live. */
pa_status pa_sched_add_request(pa_sched* sched, int64_t req_id, const int32_t* prompt,
                               int32_t prompt_len, int32_t max_new_tokens, uint64_t salt);

/* The running request parent_id gets a child that shares all of its blocks
 * and tokens (parallel sampling) and a slot of its own; the child runs next
 * to the parent from the next step on. */
pa_status pa_sched_fork(pa_sched* sched, int64_t parent_id, int64_t child_id,
                        int32_t max_new_tokens);

/* Drops a live request (waiting or running) and releases its blocks. */
pa_status pa_sched_abort(pa_sched* sched, int64_t req_id);

/* Schedules the next step into *batch. A step must be committed before the
 * next one. */
pa_status pa_sched_step(pa_sched* sched, pa_sched_batch* batch);

/* Closes the last step: sampled[i] (host int32 [n], n = that step's
 * num_reqs) is appended to entry i's request if the entry computed all of
 * its tokens (a decode, or the last chunk of a prompt); other entries ignore
 * it. Requests that reached max_new_tokens finish and release their blocks
 * and slot; their ids go to finished_ids (up to finished_cap; *num_finished
 * is the total, may exceed the cap). finished_ids may be NULL if cap is 0. */
pa_status pa_sched_commit(pa_sched* sched, const int32_t* sampled, int32_t n,
                          int64_t* finished_ids, int32_t finished_cap, int32_t* num_finished);

pa_status pa_sched_get_stats(const pa_sched* sched, pa_sched_stats* stats);

/* Copies the block table of a live request (up to cap entries) into
 * blocks[]; *n = its length. */
pa_status pa_sched_block_table(const pa_sched* sched, int64_t req_id, int32_t* blocks,
                               int32_t cap, int32_t* n);

#ifdef __cplusplus
}
#endif

#endif /* PA_SCHED_H_ */
