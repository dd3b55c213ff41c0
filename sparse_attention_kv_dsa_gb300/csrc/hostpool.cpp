// Model-wide host pool (N1): one pinned buffer holds every layer's host rows, and a
// request's context takes the same row range in every layer.  "ECHO: Efficient KV
// Cache Offloading with Lossless Prefetching ..." review page, section "In-graph
// per-layer cache management": the GPU cache of each layer is managed in the graph,
// the host pool for the whole model.  First-fit row ranges from a sorted, coalesced
// free list kept in the caller's struct.  Host code only.

#include <cuda_runtime.h>

#include <cstring>

#include "echo.h"

namespace {

size_t row_bytes(int32_t kv_dtype) { return (size_t)ECHO_KV_WIDTH * (kv_dtype == ECHO_F32 ? 4 : 2); }

bool dtype_ok(int32_t kv_dtype) { return kv_dtype == ECHO_F32 || kv_dtype == ECHO_BF16; }

}  // namespace

extern "C" size_t echo_host_pool_bytes(int32_t n_layers, int64_t rows_per_layer, int32_t kv_dtype) {
  if (n_layers <= 0 || rows_per_layer <= 0 || !dtype_ok(kv_dtype)) return 0;
  return (size_t)n_layers * (size_t)rows_per_layer * row_bytes(kv_dtype);
}

extern "C" echo_status_t echo_host_pool_init(echo_host_pool_t *pool, void *base, int32_t n_layers,
                                             int64_t rows_per_layer, int32_t kv_dtype) {
  if (!pool || !base || n_layers <= 0 || rows_per_layer <= 0 || !dtype_ok(kv_dtype)) return ECHO_ERR_INVALID_ARG;
  std::memset(pool, 0, sizeof(*pool));
  pool->base = base;
  pool->n_layers = n_layers;
  pool->kv_dtype = kv_dtype;
  pool->rows_per_layer = rows_per_layer;
  pool->n_free = 1;
  pool->free_first[0] = 0;
  pool->free_rows[0] = rows_per_layer;
  return ECHO_OK;
}

extern "C" echo_status_t echo_host_pool_alloc(echo_host_pool_t *pool, int64_t rows, int64_t *first_row) {
  if (!pool || !first_row || rows <= 0) return ECHO_ERR_INVALID_ARG;
  for (int i = 0; i < pool->n_free; ++i) {
    if (pool->free_rows[i] < rows) continue;
    *first_row = pool->free_first[i];                   // the low end of the first range that fits
    pool->free_first[i] += rows;
    pool->free_rows[i] -= rows;
    if (pool->free_rows[i] == 0) {                      // range used up: close the gap
      for (int j = i; j + 1 < pool->n_free; ++j) {
        pool->free_first[j] = pool->free_first[j + 1];
        pool->free_rows[j] = pool->free_rows[j + 1];
      }
      --pool->n_free;
    }
    pool->rows_in_use += rows;
    return ECHO_OK;
  }
  return ECHO_ERR_POOL_EXHAUSTED;
}

extern "C" echo_status_t echo_host_pool_free(echo_host_pool_t *pool, int64_t first_row, int64_t rows) {
  if (!pool || rows <= 0 || first_row < 0 || first_row > pool->rows_per_layer - rows) return ECHO_ERR_INVALID_ARG;
  const int64_t end = first_row + rows;
  int i = 0;                                            // first free range that starts after the block
  while (i < pool->n_free && pool->free_first[i] < first_row) ++i;
  // a double free overlaps the free range before it or the one at i
  if (i > 0 && pool->free_first[i - 1] + pool->free_rows[i - 1] > first_row) return ECHO_ERR_INVALID_ARG;
  if (i < pool->n_free && pool->free_first[i] < end) return ECHO_ERR_INVALID_ARG;
  const bool join_prev = i > 0 && pool->free_first[i - 1] + pool->free_rows[i - 1] == first_row;
  const bool join_next = i < pool->n_free && pool->free_first[i] == end;
  if (join_prev && join_next) {                         // the block fills a gap: three ranges become one
    pool->free_rows[i - 1] += rows + pool->free_rows[i];
    for (int j = i; j + 1 < pool->n_free; ++j) {
      pool->free_first[j] = pool->free_first[j + 1];
      pool->free_rows[j] = pool->free_rows[j + 1];
    }
    --pool->n_free;
  } else if (join_prev) {
    pool->free_rows[i - 1] += rows;
  } else if (join_next) {
    pool->free_first[i] = first_row;
    pool->free_rows[i] += rows;
  } else {
    if (pool->n_free >= ECHO_HOST_POOL_MAX_RANGES) return ECHO_ERR_UNSUPPORTED;
    for (int j = pool->n_free; j > i; --j) {
      pool->free_first[j] = pool->free_first[j - 1];
      pool->free_rows[j] = pool->free_rows[j - 1];
    }
    pool->free_first[i] = first_row;
    pool->free_rows[i] = rows;
    ++pool->n_free;
  }
  pool->rows_in_use -= rows;
  return ECHO_OK;
}

extern "C" echo_status_t echo_host_pool_layer(const echo_host_pool_t *pool, int32_t layer, void **host_rows,
                                              void **host_rows_dev) {
  if (!pool || !pool->base || layer < 0 || layer >= pool->n_layers) return ECHO_ERR_INVALID_ARG;
  char *p = static_cast<char *>(pool->base) + (size_t)layer * (size_t)pool->rows_per_layer * row_bytes(pool->kv_dtype);
  if (host_rows) *host_rows = p;
  if (host_rows_dev) {
    void *d = nullptr;
    if (cudaHostGetDevicePointer(&d, p, 0) != cudaSuccess || !d) return ECHO_ERR_CUDA;
    *host_rows_dev = d;
  }
  return ECHO_OK;
}
