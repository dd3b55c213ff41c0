// One layer's decode step, enqueued on one stream in the order of the review page's
// "Decode: predict the transfer, then recall exactly": write-back of the new token,
// prefetch budget, indexer scoring with fused threshold prefetch, exact top-k with
// the EMA update, recall of every missing selected token, sparse MLA attention.
// The prefetch budget is computed by the write-back's launch and the exact prefetch
// cap is deferred from the indexer into the top-k launch, so prefetch adds no launch
// of its own to the step.
// Host code only: it launches the kernels of the other translation units; every
// count it depends on stays in device memory, so the sequence can be captured in a
// CUDA Graph and replayed step after step.

#include "common.cuh"

extern "C" echo_status_t echo_decode_layer_step(const echo_cache_layer_t *layer, const echo_step_args_t *a,
                                                echo_stream_t stream) {
  if (!layer || !a) return ECHO_ERR_INVALID_ARG;
  // block granularity or another row width: the entry points in order
  if (layer->block_tokens > 1 || echo::kv_row_elems(*layer) != echo::KV_W) return ECHO_ERR_UNSUPPORTED;
  const bool pf = a->prefetch != 0 && a->cap_max > 0;
  // write-back, and in the same launch the step's prefetch budget
  echo_status_t st = echo::cache_writeback_reserve(layer, a->new_kv, a->new_ik, a->idx_k, a->D, a->Lmax, a->idx_dtype,
                                                   a->host_base, a->seq_len, a->B, a->cap_max, a->cap_div,
                                                   pf ? a->cap : nullptr, a->pf_count, stream);
  if (st != ECHO_OK) return st;
  cudaStream_t cs = (cudaStream_t)stream;
  if (a->index_events[0]) ECHO_CUDA_OK(cudaEventRecordWithFlags((cudaEvent_t)a->index_events[0], cs, cudaEventRecordExternal));
  st = echo_index_prefetch(a->q_idx, a->w_idx, a->idx_k, a->seq_len, a->B, a->H, a->D, a->Lmax, a->idx_dtype,
                           a->theta, pf ? a->cap : nullptr, a->cap_max, a->host_base, layer, a->scores, a->pf_list,
                           a->pf_count, a->stage_kv, pf ? ECHO_PF_DEFER_CAP : 0, stream);
  if (st != ECHO_OK) return st;
  if (a->index_events[1]) ECHO_CUDA_OK(cudaEventRecordWithFlags((cudaEvent_t)a->index_events[1], cs, cudaEventRecordExternal));
  st = pf ? echo_topk_prefetch(a->scores, a->seq_len, a->B, a->Lmax, a->k, a->sel, a->kth, a->theta, a->alpha,
                               a->cap, a->cap_max, a->host_base, layer, a->pf_list, a->pf_count, a->stage_kv, stream)
          : echo_topk(a->scores, a->seq_len, a->B, a->Lmax, a->k, a->sel, a->kth, a->theta, a->alpha, stream);
  if (st != ECHO_OK) return st;
  st = echo_cache_recall(layer, a->sel, a->host_base, a->B, a->k, pf ? a->pf_list : nullptr,
                         pf ? a->pf_count : nullptr, a->cap_max, a->stage_kv, a->miss_list, a->n_miss, a->slot_idx,
                         stream);
  if (st != ECHO_OK) return st;
  return echo_sparse_mla_decode(a->q_mla, layer->gpu_kv, layer->n_gpu, layer->kv_dtype, a->slot_idx, a->B, a->Hq,
                                a->k, a->scale, a->out, a->lse, a->mla_workspace, a->mla_workspace_bytes, stream);
}
