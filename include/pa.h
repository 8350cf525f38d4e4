/*
 * pa.h — C ABI of libpa, the hot path of a paged-KV-cache attention engine
 * for one NVIDIA GB300 (sm_103a).
 *
 * Source pages (cited by title and section throughout this library):
 *   [vLLM-wiki] itwiki.kr, "vLLM"
 *   [MRV2]      llm-wiki.hwlabs.dev, "vLLM 0.25 Model Runner V2: 비동기 추론 경로의
 *               재설계와 마이그레이션"
 *   [V1-blog]   techknowgenie.com, "vLLM V1 코어 리팩토링 아키텍처: Zero-overhead C++
 *               스케줄러와 Dynamic Chunked Prefill, PagedAttention v3 심층 분석"
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Ownership: every buffer is allocated and owned by the caller. The library
 *    never allocates, frees or keeps a pointer after the call returns, except
 *    through work that it has enqueued on `stream`.
 *  - Execution: every call enqueues kernels on `stream` (a cudaStream_t passed
 *    as void*; NULL is the legacy default stream) and returns without waiting.
 *    Only pa_get_error() synchronises.
 *  - Host-side argument errors (NULL pointers, negative sizes, misaligned
 *    pointers, inconsistent host mirrors) return PA_ERR_INVALID before any
 *    launch; unsupported shapes return PA_ERR_UNSUPPORTED. A failed launch
 *    returns PA_ERR_CUDA.
 *  - Device-side range errors (a block id, slot or table row that points
 *    outside its buffer) never fault: the kernel skips or clamps the offending
 *    access and sets a sticky bit in a per-device error word, which
 *    pa_get_error() reports and clears. Outputs of a call that raised a device
 *    error are unspecified.
 *  - All pointers marked "dev" are device pointers on the current device; "host"
 *    pointers are read synchronously during the call only.
 *  - The library looks up the device addresses of its own device variables
 *    (the error word, the scratch array of pa_forward_noalloc) once per device,
 *    on first use, and keeps them for the life of the process. They do not
 *    survive cudaDeviceReset: after a reset of a device, make no further call
 *    of this library on that device in the same process.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* pa_stream_t; /* a cudaStream_t */

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID = 1,       /* bad argument, detected on the host before launch   */
  PA_ERR_UNSUPPORTED = 2,   /* shape or dtype outside the supported set           */
  PA_ERR_CUDA = 3,          /* a CUDA runtime call failed                         */
  PA_ERR_DEVICE_BOUNDS = 4, /* a kernel met an out-of-range index (pa_get_error)  */
  PA_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (pa_get_error)  */
} pa_status;

typedef enum pa_kv_dtype {
  PA_KV_BF16 = 0,     /* K/V stored as bfloat16                                  */
  PA_KV_FP8_E4M3 = 1  /* K/V stored as OCP FP8 E4M3 codes with per-tensor scales */
} pa_kv_dtype;

/*
 * The physical KV block pool.
 * [vLLM-wiki, "블록 테이블"]: device memory is split ahead of time into equal-size
 * physical blocks of `block_size` tokens; a request's logical blocks map to
 * physical blocks that need not be contiguous.
 *
 * Layout (caller-owned device memory, 16-byte aligned), for K and V separately:
 *     pool[num_blocks][num_kv_heads][block_size][head_dim]
 * so the `block_size` tokens of one (block, kv-head) pair are one contiguous
 * chunk of block_size*head_dim elements. Element type is bf16 (2 bytes) or an
 * E4M3 code (1 byte) according to `dtype`.
 *
 * FP8 [vLLM-wiki, "엔진 구조와 주요 기능", quantisation bullet; V1-blog, "FP8 KV 캐시
 * 양자화의 네이티브 통합"]: a stored code c represents decode(c) * k_scale (or
 * v_scale). Scales are ignored for bf16 pools.
 *
 * Supported: head_dim in {64, 128}; block_size in {16, 32, 64}.
 */
typedef struct pa_kv_pool {
  void* k_pool;          /* dev */
  void* v_pool;          /* dev */
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype;         /* pa_kv_dtype */
  float k_scale;
  float v_scale;
} pa_kv_pool;

/*
 * pa_write_kv — scatter this step's new keys and values into the pool.
 * [vLLM-wiki, "블록 테이블"] (slot = physical_block * block_size + offset) and
 * [MRV2, "재설계 4"] (slot_mapping is prepared per token before the forward).
 *
 *   k_new, v_new   dev bf16 [T][num_kv_heads][head_dim], 16-byte aligned
 *   slot_mapping   dev int64 [T]; slot < 0 marks a padding token (skipped)
 *   T              number of tokens (0 is a no-op)
 *
 * For token t with s = slot_mapping[t] >= 0: blk = s / block_size,
 * off = s % block_size, and for every kv head h and dim d
 *     K[blk][h][off][d] = k_new[t][h][d]   (and the same for V).
 * bf16 pools copy the bits. FP8 pools store e4m3(float(x) / scale), the
 * quotient correctly rounded in fp32, then rounded to nearest-even with
 * saturation to +-448; NaN stores 0x7F.
 * A slot >= num_blocks*block_size sets PA_ERR_DEVICE_BOUNDS and is skipped.
 * Duplicate slots within one call: which token wins is unspecified.
 */
pa_status pa_write_kv(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                      const int64_t* slot_mapping, int32_t T, pa_stream_t stream);

/*
 * pa_forward_workspace_size — bytes of optional scratch that lets pa_forward
 * split long decode requests across CTAs (split-KV, merged by log-sum-exp).
 * `max_splits` is the largest number of splits the caller wants per request.
 * pa_forward works with any workspace size, including 0 (then each decode
 * request is handled by one CTA per kv head).
 */
size_t pa_forward_workspace_size(int32_t num_reqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_splits);

/*
 * pa_forward — paged attention over a mixed batch of decode tokens and prefill
 * chunks.
 * [vLLM-wiki, "블록 단위 어텐션 계산", equation for A_ij and o_i]: the softmax runs
 * across every visible key of every block of the request; the result equals
 * ordinary attention, only the memory layout differs.
 * [V1-blog, "고정 예산 기반 청크 분할 알고리즘"] and [vLLM-wiki, "엔진 구조와 주요 기능"
 * unified-scheduler bullet]: one step packs one token per running decode next to
 * prefill chunks.
 * [MRV2, "재설계 4"]: query_start_loc and seq_lens describe the batch.
 *
 *   q                 dev bf16 [T][num_q_heads][head_dim], 16-byte aligned
 *   out               dev bf16 [T][num_q_heads][head_dim], 16-byte aligned
 *   query_start_loc   dev int32 [R+1], qsl[0]=0, non-decreasing, qsl[R]=T
 *   seq_lens          dev int32 [R], all tokens of request r including this
 *                     step's query tokens (whose K/V must already be written)
 *   qsl_host, seq_lens_host
 *                     host mirrors of the two arrays above (same values); used
 *                     to plan grids without a device sync
 *   block_tables      dev int32 [R][max_blocks]: physical block of logical
 *                     block i of request r; entries past ceil(seq_len/B) unread
 *   num_q_heads       Hq; must be a multiple of pool->num_kv_heads. Query head
 *                     h reads kv head h / (Hq / Hkv) (contiguous GQA groups).
 *   scale             softmax scale (e.g. 1/sqrt(head_dim))
 *   causal            1: query j of request r (absolute position
 *                     p = seq_len - q_len + j) sees keys 0..p. 0: every query
 *                     sees keys 0..seq_len-1. A decode query (q_len == 1)
 *                     sees all seq_len keys either way.
 *   workspace         dev scratch of workspace_bytes (may be NULL/0)
 *
 * out[t][h][:] = sum_n softmax_n(scale * q[t][h] . k_n) v_n over the visible
 * keys, computed in fp32 and rounded to bf16 (nearest-even). Rows of requests
 * with q_len == 0 are not touched. Requests may appear in any order.
 * Host checks: qsl_host must be non-decreasing with qsl_host[R] == T, and
 * 1 <= q_len <= seq_len <= max_blocks * block_size for every request with
 * q_len > 0, and a pool with at least one block when any request has
 * q_len > 0; otherwise PA_ERR_INVALID.
 * Device checks: the grids are planned from the host mirrors. A device
 * query_start_loc or seq_lens that disagrees with them so that a request's
 * rows would leave [0, T), or its keys or query tiles would need more CTAs
 * or workspace slots than were planned, sets PA_ERR_DEVICE_BOUNDS; nothing is
 * read or written outside q, out, the pool and the workspace.
 */
pa_status pa_forward(const void* q, void* out, const int32_t* query_start_loc,
                     const int32_t* seq_lens, const int32_t* qsl_host,
                     const int32_t* seq_lens_host, const int32_t* block_tables,
                     int32_t max_blocks, int32_t num_reqs, int32_t num_tokens,
                     int32_t num_q_heads, const pa_kv_pool* pool, float scale,
                     int32_t causal, void* workspace, size_t workspace_bytes,
                     pa_stream_t stream);

/*
 * pa_forward_shared_prefix — pa_forward for a batch in which groups of decode
 * requests share the physical blocks of a common prefix (parallel sampling,
 * beam candidates, a shared system prompt).
 * [vLLM-wiki, "블록 공유와 쓰기 시 복사"]:
 * the samples of one prompt map the prompt's logical blocks to the same
 * physical blocks (reference-counted, copied on write); only the tails differ.
 * The result is the attention pa_forward computes (the same bounds against
 * exact arithmetic; the fp32 summation order differs): the softmax over the
 * union of the prefix keys and the tail keys is taken in parts, the prefix
 * pieces and the tail splits, merged by log-sum-exp. Each group's prefix K/V
 * is read once for every 64 of its (member, GQA head) rows (four warps share
 * each staged K/V chunk) instead of once per member; any GQA width.
 *
 * Arguments as pa_forward, plus:
 *   num_groups          G, 0 <= G <= 64 (more: PA_ERR_UNSUPPORTED). G == 0
 *                       behaves as pa_forward.
 *   group_first_host    host int32 [G]: group k is the group_size_host[k]
 *   group_size_host     host int32 [G]  consecutive requests from
 *                       group_first_host[k]; groups in increasing order and
 *                       disjoint, within [0, num_reqs); other requests may sit
 *                       before, between and after them
 *   prefix_blocks_host  host int32 [G]: the first prefix_blocks_host[k]
 *                       entries of every member's block-table row are the
 *                       same physical blocks (the caller's contract: the
 *                       prefix is read through the first member's row)
 *   workspace           required: at least pa_forward_workspace_size(R, Hq,
 *                       head_dim, 2) bytes (one prefix piece and one tail
 *                       split per member); more lets the call cut prefixes and
 *                       tails into more pieces that run in parallel
 *
 * Host checks (PA_ERR_INVALID): every member is a decode request (q_len 1)
 * with seq_len > prefix_blocks * block_size, 1 <= prefix_blocks <=
 * max_blocks, groups non-empty and in range, workspace large enough.
 * Requests outside every group, and prefill chunks, are handled exactly as by
 * pa_forward. If members' rows differ on the prefix, the result is
 * unspecified but every block id read is still bounds-checked.
 */
pa_status pa_forward_shared_prefix(const void* q, void* out, const int32_t* query_start_loc,
                                   const int32_t* seq_lens, const int32_t* qsl_host,
                                   const int32_t* seq_lens_host, const int32_t* block_tables,
                                   int32_t max_blocks, int32_t num_reqs, int32_t num_tokens,
                                   int32_t num_q_heads, const pa_kv_pool* pool, float scale,
                                   int32_t causal, int32_t num_groups,
                                   const int32_t* group_first_host,
                                   const int32_t* group_size_host,
                                   const int32_t* prefix_blocks_host, void* workspace,
                                   size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_prepare_inputs — one step's attention inputs built on the device from
 * per-slot state, so that the host sends only (slot, token count) per request
 * and the block-table diffs.
 * [MRV2, "재설계 1"]: a live request keeps a fixed persistent slot; entry i of
 * the step is slot idx_mapping[i]. [MRV2, "재설계 4"]: query_start_loc,
 * positions, seq_lens and the slot mapping are prepared on the GPU.
 * [vLLM-wiki, "블록 테이블"]: position p lives in logical block p / B at offset
 * p % B; its pool slot is physical_block * B + offset.
 *
 *   num_computed     dev int32 [max_reqs]: tokens of each slot whose K/V are
 *                    stored; read, then advanced by the step's counts
 *   table            dev int32 [max_reqs][max_blocks]: the persistent block
 *                    table (after pa_apply_staged_writes)
 *   idx_mapping      dev int32 [R]: slot of entry i (each slot at most once)
 *   num_scheduled    dev int32 [R]: tokens of entry i this step (>= 0);
 *                    NULL: one token per entry (a decode step)
 *   token_capacity   entries of positions / slot_mapping
 *   query_start_loc  dev int32 [R+1]  out: running sum of num_scheduled
 *   seq_lens         dev int32 [R]    out: num_computed[slot] + num_scheduled
 *   positions        dev int32 [T]    out: the tokens' positions
 *   slot_mapping     dev int64 [T]    out: the tokens' pool slots (input of
 *                                     pa_write_kv)
 *
 * One launch on `stream`. Integer work: exactly the definition above. A slot
 * outside [0, max_reqs), a negative count, a total above token_capacity, a
 * position past the table row or a block outside [0, num_blocks) sets
 * PA_ERR_DEVICE_BOUNDS (read by pa_get_error); such slots are written as -1
 * (pa_write_kv skips them) and nothing is written outside the buffers. A slot
 * listed twice gives unspecified counts. Host checks: PA_ERR_INVALID for
 * negative sizes or NULL buffers that the sizes require.
 */
pa_status pa_prepare_inputs(int32_t* num_computed, int32_t max_reqs, const int32_t* table,
                            int32_t max_blocks, int32_t block_size, int32_t num_blocks,
                            const int32_t* idx_mapping, const int32_t* num_scheduled,
                            int32_t num_reqs, int32_t token_capacity, int32_t* query_start_loc,
                            int32_t* seq_lens, int32_t* positions, int64_t* slot_mapping,
                            pa_stream_t stream);

/*
 * pa_decode_graph_* — several decode steps of the same requests captured once
 * into a CUDA graph and replayed with one launch.
 * [V1-blog, "PagedAttention V3 커널 아키텍처와 하드웨어 레벨 메모리 정렬",
 * multi-step scheduling bullet]: N decode steps (4 to 8, say) run from a CUDA
 * graph without a host round trip per token. [MRV2, "재설계 4"]: graphs are
 * managed explicitly; each captured shape costs capture time and memory.
 *
 * Step s of the graph (s = 0 .. num_steps-1) is exactly this eager sequence:
 *   pa_prepare_inputs(num_computed, ..., idx_mapping, NULL (one token each),
 *                     num_reqs, num_reqs, query_start_loc, seq_lens, positions,
 *                     slot_mapping)
 *   pa_write_kv(pool, k_new + s * R*Hkv*D, v_new + s * R*Hkv*D, slot_mapping, R)
 *   pa_forward(q + s * R*Hq*D, out + s * R*Hq*D, query_start_loc, seq_lens,
 *              {0, 1, .., R}, seq_len_bound_host, block_tables, max_blocks, R, R,
 *              num_q_heads, pool, scale, 1, workspace, workspace_bytes)
 * so every output equals that of the eager calls made with the same bound.
 * The forward plan is fixed at creation from seq_len_bound_host; every launch
 * should keep each request's sequence length (num_computed + 1 at each step)
 * at or below its bound. A length past its bound is either still covered by
 * the plan, with exact results (the persistent GQA decode of pa_forward cuts
 * the device-side lengths into its CTA ranges at every launch, within the
 * workspace's split slots), or refused with PA_ERR_DEVICE_BOUNDS; nothing is
 * ever read out of range. The table must already hold the blocks of every
 * position the steps write; block_tables holds the rows table[idx_mapping[i]].
 *
 * The pool struct, pointers and sizes are read at creation and baked into the
 * graph: the buffers must stay allocated and in place until destroy. The
 * graph object is created (host and driver memory) by create and released by
 * destroy; the library allocates no device memory. Launches of one graph must
 * not overlap (they share the scratch buffers); launch returns without
 * waiting. Errors: PA_ERR_INVALID (NULL or non-positive sizes), the status of
 * the first captured call that fails, PA_ERR_CUDA if capture or instantiation
 * fails.
 */
typedef struct pa_decode_graph pa_decode_graph;

typedef struct {
  const pa_kv_pool* pool;
  float scale;
  int32_t num_q_heads;
  int32_t num_reqs;                    /* R: decode requests, one token per step  */
  int32_t num_steps;                   /* N                                        */
  int32_t* num_computed;               /* dev int32 [max_reqs] (advanced N / launch) */
  int32_t max_reqs;
  const int32_t* table;                /* dev int32 [max_reqs][max_blocks]         */
  int32_t max_blocks;
  const int32_t* idx_mapping;          /* dev int32 [R]                            */
  const int32_t* block_tables;         /* dev int32 [R][max_blocks]                */
  const int32_t* seq_len_bound_host;   /* host int32 [R]                           */
  const void* q;                       /* dev bf16 [N][R][Hq][D]                   */
  const void* k_new;                   /* dev bf16 [N][R][Hkv][D]                  */
  const void* v_new;                   /* dev bf16 [N][R][Hkv][D]                  */
  void* out;                           /* dev bf16 [N][R][Hq][D]                   */
  int32_t* query_start_loc;            /* dev scratch int32 [R+1]                  */
  int32_t* seq_lens;                   /* dev scratch int32 [R]                    */
  int32_t* positions;                  /* dev scratch int32 [R]                    */
  int64_t* slot_mapping;               /* dev scratch int64 [R]                    */
  void* workspace;                     /* as pa_forward (may be NULL / 0)          */
  size_t workspace_bytes;
} pa_decode_graph_desc;

pa_status pa_decode_graph_create(const pa_decode_graph_desc* desc, pa_decode_graph** graph);
pa_status pa_decode_graph_launch(pa_decode_graph* graph, pa_stream_t stream);
void pa_decode_graph_destroy(pa_decode_graph* graph);
/* Kernel launches one pa_decode_graph_launch performs (0 for NULL). */
uint32_t pa_decode_graph_kernels(const pa_decode_graph* graph);

/*
 * pa_apply_staged_writes — apply packed block-table diffs, then gather the
 * rows of this step.
 * [MRV2, "재설계 3: 큰 block table은 staged diff만 보낸다"]: the device copy of the
 * block table is the reference copy; the host records (row, start, values)
 * diffs, uploads them in one small staging buffer, and one kernel applies them;
 * the rows needed this step are then gathered by idx_mapping.
 * [MRV2, "재설계 1"]: a request keeps a fixed persistent slot (row) while live;
 * idx_mapping[i] is the slot of the i-th request of this batch.
 * [MRV2, "재설계 2"]: the staging buffers must not be modified by the caller until
 * the stream has consumed them.
 *
 *   table          dev int32 [max_reqs][max_blocks], updated in place
 *   rows, starts   dev int32 [W]
 *   val_offsets    dev int32 [W+1], non-decreasing from val_offsets[0] >= 0;
 *                  diff w writes len_w = val_offsets[w+1] - val_offsets[w]
 *                  values
 *   vals           dev int32 [val_offsets[W]]
 *   idx_mapping    dev int32 [R]
 *   gathered       dev int32 [R][max_blocks]
 *
 * For w = 0..W-1 in record order: table[rows[w]][starts[w] + k] =
 * vals[val_offsets[w] + k], k < len_w (a later diff overwrites an earlier one
 * on the same cell: last writer wins). Then gathered[i][c] =
 * table[idx_mapping[i]][c] for every c < max_blocks. A diff whose row or
 * column range leaves the table, whose value run leaves [0, val_offsets[W]),
 * or an idx_mapping entry outside
 * [0, max_reqs), sets PA_ERR_DEVICE_BOUNDS and is skipped (gathered row left
 * untouched). W == 0 performs only the gather; R == 0 only the writes.
 */
pa_status pa_apply_staged_writes(int32_t* table, int32_t max_reqs, int32_t max_blocks,
                                 const int32_t* rows, const int32_t* starts,
                                 const int32_t* val_offsets, const int32_t* vals,
                                 int32_t W, const int32_t* idx_mapping, int32_t R,
                                 int32_t* gathered, pa_stream_t stream);

/*
 * pa_copy_blocks — copy whole physical blocks (K and V, every kv head), the
 * device half of copy-on-write.
 * [vLLM-wiki, "블록 공유와 쓰기 시 복사"]: a block shared by several sequences is
 * copied only when one of them must write a new token into it.
 *
 *   src, dst   dev int32 [n]; block src[i] is copied to block dst[i]
 * The dst blocks must be distinct from each other and from every src block
 * (then the copies are order-independent). An id outside [0, num_blocks) sets
 * PA_ERR_DEVICE_BOUNDS and that pair is skipped.
 */
pa_status pa_copy_blocks(const pa_kv_pool* pool, const int32_t* src, const int32_t* dst,
                         int32_t n, pa_stream_t stream);

/*
 * pa_gather_rows — dst row i = src row rows[i], for i < n: the rows a step
 * hands on (each request's last query token, whose output the sampler
 * needs) gathered by index, as [MRV2, "재설계 1"] gathers the persistent
 * batch's rows by idx_mapping.
 *
 *   src        dev, src_rows rows of row_bytes bytes (16-byte aligned)
 *   row_bytes  a positive multiple of 16
 *   rows       dev int32 [n]
 *   dst        dev, n rows of row_bytes bytes (16-byte aligned), not
 *              overlapping src
 * A row index outside [0, src_rows) sets PA_ERR_DEVICE_BOUNDS and that dst
 * row is left unchanged. n == 0 is a no-op. Argument errors: PA_ERR_INVALID.
 */
pa_status pa_gather_rows(const void* src, int64_t src_rows, int64_t row_bytes,
                         const int32_t* rows, int32_t n, void* dst, pa_stream_t stream);

/*
 * pa_get_error — synchronise `stream`, then return and clear the sticky
 * device error word of the current device: PA_ERR_TIMEOUT if a bounded wait
 * gave up, else PA_ERR_DEVICE_BOUNDS if an index was out of range, else
 * PA_OK. Returns PA_ERR_CUDA if the synchronisation itself failed.
 * The word is read and cleared in one atomic exchange (a one-thread kernel on
 * `stream`, counted by pa_kernel_launches), so a bit that a kernel on another
 * stream sets meanwhile is returned by this call or by the next one, never
 * cleared unseen. Not callable during stream capture (it synchronises).
 */
pa_status pa_get_error(pa_stream_t stream);

/* pa_status_string — a static, human-readable name for a status code. */
const char* pa_status_string(pa_status status);

/*
 * pa_forward_noalloc — pa_forward for callers that cannot allocate device
 * memory. The pages have no counterpart of this call.
 *
 * Some callers may not call cudaMalloc (or any allocator) where they run
 * attention: a plugin inside a host runtime that has reserved the device
 * memory through its own pool and gives plugins no allocator, or a serving
 * loop that forbids allocation after start-up because cudaMalloc can
 * synchronise the device. This call takes the same arguments as pa_forward
 * except the workspace: its split-KV scratch comes from a fixed array that
 * the library keeps in device memory, PA_NOALLOC_SCRATCH_BYTES on every GPU
 * that loads the library, held until the process exits.
 *
 *   max_splits   as in pa_forward_workspace_size; the scratch it needs,
 *                pa_forward_workspace_size(num_reqs, num_q_heads, head_dim,
 *                max_splits), must not exceed PA_NOALLOC_SCRATCH_BYTES, else
 *                the call returns PA_ERR_UNSUPPORTED before any launch.
 *                0 uses no scratch (one split per decode request).
 *
 * The call allocates nothing and frees nothing. The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress) and caches it;
 * make that first call before any stream capture. The cached address does not
 * survive cudaDeviceReset (see the conventions above). Every call shares the same
 * array: calls that may run at the same time on the GPU (different streams,
 * or several host threads) race on it and must be serialised by the caller.
 * The array keeps the previous call's contents; nothing needs clearing,
 * because every cell a call reads is written earlier in that call.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)

pa_status pa_forward_noalloc(const void* q, void* out, const int32_t* query_start_loc,
                             const int32_t* seq_lens, const int32_t* qsl_host,
                             const int32_t* seq_lens_host, const int32_t* block_tables,
                             int32_t max_blocks, int32_t num_reqs, int32_t num_tokens,
                             int32_t num_q_heads, const pa_kv_pool* pool, float scale,
                             int32_t causal, int32_t max_splits, pa_stream_t stream);

/*
 * pa_selftest_wait_timeout — diagnostics, not part of the method on the pages.
 * Launches one small kernel that waits on a device barrier which nothing will
 * complete, through the same bounded wait that every kernel of this library
 * uses. The wait gives up after its limit (about 2 seconds), records the
 * timeout in the error word and returns: afterwards pa_get_error() reports
 * PA_ERR_TIMEOUT. Lets callers and tests check the no-hang error path.
 */
pa_status pa_selftest_wait_timeout(pa_stream_t stream);

/*
 * pa_kernel_launches — number of CUDA kernels this library has launched in
 * this process (all devices, all streams), for launch accounting in
 * benchmarks and tests. Not part of the method on the pages; never fails.
 */
uint64_t pa_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
