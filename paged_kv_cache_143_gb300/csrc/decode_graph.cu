// decode_graph.cu — several decode steps captured once into a CUDA graph and
// replayed with one launch (pa_decode_graph_*).
//
// [V1-blog "PagedAttention V3 커널 아키텍처와 하드웨어 레벨 메모리 정렬",
// multi-step scheduling]: N decode steps (4 to 8, say) run back to back from a
// CUDA graph instead of a host round trip per token, which removes the launch
// overhead; [MRV2 "재설계 4"]: graphs are managed explicitly, and each captured
// shape costs capture time and memory. Small decode batches are bound by the
// cost of launching their kernels, not by the GPU. Each captured step is exactly the eager sequence:
//   pa_prepare_inputs (one token per request: seq_lens, positions and the
//   slot mapping from the per-slot state, which it advances),
//   pa_write_kv (the step's new K/V at those slots),
//   pa_forward (decode attention into the step's output rows).
// The forward plan (split size, grid, merge) is fixed at capture from an upper
// bound of every sequence length the graph will see; the kernels read the
// actual lengths from device memory each step (CTAs past a request's splits
// return at once), so one plan serves every step while the bound holds. A
// longer sequence is caught on the device (PA_ERR_DEVICE_BOUNDS), never read
// out of range.
#include <vector>

#include "pa_internal.h"

struct pa_decode_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  unsigned kernels = 0;  // kernel launches per graph launch
};

namespace {

pa_status capture_steps(const pa_decode_graph_desc& d, cudaStream_t s) {
  const int R = d.num_reqs, Hq = d.num_q_heads;
  const int Hkv = d.pool->num_kv_heads, D = d.pool->head_dim;
  std::vector<int32_t> qsl_host(R + 1);
  for (int i = 0; i <= R; ++i) qsl_host[i] = i;
  const size_t q_step = (size_t)R * Hq * D * 2, kv_step = (size_t)R * Hkv * D * 2;
  for (int step = 0; step < d.num_steps; ++step) {
    pa_status st = pa_prepare_inputs(d.num_computed, d.max_reqs, d.table, d.max_blocks,
                                     d.pool->block_size, d.pool->num_blocks, d.idx_mapping,
                                     nullptr, R, R, d.query_start_loc, d.seq_lens, d.positions,
                                     d.slot_mapping, s);
    if (st != PA_OK) return st;
    st = pa_write_kv(d.pool, static_cast<const uint8_t*>(d.k_new) + step * kv_step,
                     static_cast<const uint8_t*>(d.v_new) + step * kv_step, d.slot_mapping, R, s);
    if (st != PA_OK) return st;
    st = pa_forward(static_cast<const uint8_t*>(d.q) + step * q_step,
                    static_cast<uint8_t*>(d.out) + step * q_step, d.query_start_loc, d.seq_lens,
                    qsl_host.data(), d.seq_len_bound_host, d.block_tables, d.max_blocks, R, R,
                    Hq, d.pool, d.scale, 1, d.workspace, d.workspace_bytes, s);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_graph_create(const pa_decode_graph_desc* d,
                                            pa_decode_graph** graph) {
  if (!d || !graph) return PA_ERR_INVALID;
  *graph = nullptr;
  pa_status st = pa::check_pool(d->pool);
  if (st != PA_OK) return st;
  if (d->num_reqs <= 0 || d->num_steps <= 0 || d->num_q_heads <= 0 || d->max_reqs <= 0 ||
      d->max_blocks <= 0 || !d->seq_len_bound_host)
    return PA_ERR_INVALID;
  if (!d->num_computed || !d->table || !d->idx_mapping || !d->block_tables || !d->q ||
      !d->k_new || !d->v_new || !d->out || !d->query_start_loc || !d->seq_lens ||
      !d->positions || !d->slot_mapping)
    return PA_ERR_INVALID;
  // per-device state is set up before the capture (it calls the runtime)
  if (!pa::error_word() || pa::num_sms() <= 0) return PA_ERR_CUDA;
  cudaStream_t s;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return PA_ERR_CUDA;
  auto* g = new pa_decode_graph();
  const unsigned long long before = pa::launches_so_far();
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(s);
    delete g;
    return PA_ERR_CUDA;
  }
  st = capture_steps(*d, s);
  const cudaError_t end = cudaStreamEndCapture(s, &g->graph);
  g->kernels = (unsigned)(pa::launches_so_far() - before);
  pa::uncount_launches(g->kernels);  // counted when the graph runs
  cudaStreamDestroy(s);
  if (st == PA_OK && end != cudaSuccess) st = PA_ERR_CUDA;
  if (st == PA_OK && cudaGraphInstantiate(&g->exec, g->graph, 0) != cudaSuccess) st = PA_ERR_CUDA;
  if (st != PA_OK) {
    cudaGetLastError();
    pa_decode_graph_destroy(g);
    return st;
  }
  *graph = g;
  return PA_OK;
}

extern "C" pa_status pa_decode_graph_launch(pa_decode_graph* graph, pa_stream_t stream) {
  if (!graph || !graph->exec) return PA_ERR_INVALID;
  if (cudaGraphLaunch(graph->exec, pa::as_stream(stream)) != cudaSuccess) return PA_ERR_CUDA;
  pa::count_launches(graph->kernels);
  return PA_OK;
}

extern "C" void pa_decode_graph_destroy(pa_decode_graph* graph) {
  if (!graph) return;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
}

extern "C" uint32_t pa_decode_graph_kernels(const pa_decode_graph* graph) {
  return graph ? graph->kernels : 0u;
}
