/*
 * echo.h -- C ABI of the ECHO per-layer decode hot path on one GB300 (sm_103a).
 *
 * Sources, cited by page and section:
 *   [REV]   "ECHO: Efficient KV Cache Offloading with Lossless Prefetching for Serving
 *           Native Sparse Attention LLMs (OSDI 2026)", review page (awesome-system-papers).
 *   [NOTES] "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs", podcast show notes.
 *   [DSA]   DeepSeek-V3.2-Exp report (listed in the show notes' sources): lightning indexer.
 *
 * Conventions shared by every call
 *   - Ownership: the caller allocates every buffer (device memory, and pinned host
 *     memory made device-visible with echo_host_device_pointer).  The library
 *     allocates nothing and never synchronises the stream, except
 *     echo_cache_status / echo_cache_read_counters, which do.  It keeps no global
 *     state, with one exception: echo_sparse_mla_decode_noalloc uses a scratch
 *     array compiled into the library (one per GPU that loads it) and caches that
 *     array's device address per device.
 *   - Every data-dependent count (misses, prefetched rows, the step number, context
 *     lengths, the EMA threshold) lives in device memory, so a sequence of calls can
 *     be captured into one CUDA Graph and replayed step after step [REV] "In-graph
 *     per-layer cache management"; [NOTES] fixed-size integer tensors on the GPU.
 *   - Errors: a call returns ECHO_ERR_INVALID_ARG for a null pointer or a bad size,
 *     ECHO_ERR_UNSUPPORTED for a dtype/shape the kernels do not handle, ECHO_ERR_CUDA
 *     when a launch fails.  Conditions found on the device set a sticky status word
 *     (counters[ECHO_CTR_STATUS], first error wins) and the kernels skip the bad
 *     access instead of trapping; read it with echo_cache_status.
 *   - Host index of token t of request b is host_base[b] + t: each request owns a
 *     contiguous range of the model-wide host pool ([REV] "In-graph per-layer cache
 *     management": the host pool is managed for the whole model).
 *   - Latent rows are 576 wide (ECHO_KV_WIDTH); attention values are the first 512.
 */
#ifndef ECHO_H
#define ECHO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *echo_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef int32_t echo_status_t;
enum {
  ECHO_OK = 0,
  ECHO_ERR_INVALID_ARG = 1,
  ECHO_ERR_UNSUPPORTED = 2,
  ECHO_ERR_CUDA = 3,
  ECHO_ERR_TIMEOUT = 4,        /* device: a bounded wait gave up                        */
  ECHO_ERR_POOL_EXHAUSTED = 5, /* device: not enough evictable slots for the tokens    */
  ECHO_ERR_HOST_INDEX = 6,     /* device: a host index fell outside [0, n_host)        */
  ECHO_ERR_STAGING = 7,        /* device: a request's prefetch cap exceeds its staging  */
  ECHO_ERR_SCRATCH_LIMIT = 8,  /* host: the call needs more than the library's built-in
                                  scratch (echo_sparse_mla_decode_noalloc only)         */
  ECHO_ERR_NOT_RESIDENT = 9    /* device: a token to attend over has no GPU slot        */
};

enum { ECHO_F32 = 0, ECHO_BF16 = 1, ECHO_E4M3 = 2 };

enum { ECHO_KV_WIDTH = 576, ECHO_V_WIDTH = 512 };

/* Indices into the per-layer counters block (int32[ECHO_NUM_COUNTERS], device). */
enum {
  ECHO_CTR_STEP = 0,        /* current decode step s (a write-back begins a step)       */
  ECHO_CTR_N_FREE = 1,      /* number of free GPU slots                                 */
  ECHO_CTR_STATUS = 2,      /* sticky device status (ECHO_OK or an ECHO_ERR_*)           */
  ECHO_CTR_NEED = 3,        /* tokens the current recall must bind to slots             */
  ECHO_CTR_CURSOR = 4,      /* allocation cursor (scratch)                              */
  ECHO_CTR_EVICT_M = 5,     /* victims requested by the last eviction                   */
  ECHO_CTR_HITS = 8,        /* stats, cleared by echo_cache_writeback as a step begins:  */
  ECHO_CTR_STAGED_HITS = 9, /*   selected & resident / selected & prefetched this step  */
  ECHO_CTR_MISSES = 10,     /*   selected & copied from the host after the top-k        */
  ECHO_CTR_EVICTED = 11,    /*   tokens evicted by the recall                           */
  ECHO_CTR_STAGED = 12,     /*   rows prefetched (staged) during scoring                */
  ECHO_CTR_WB_EVICTED = 13, /*   tokens evicted by the write-back                       */
  ECHO_CTR_BOUND = 14,      /*   tokens bound to slots by the recall                    */
  ECHO_CTR_QUALIFIED = 15,  /*   tokens that met the prefetch rule (before the cap)     */
                            /* 16..31: the manager's own words (grid barrier, cursors,   */
                            /*   the pending victim list's count and step); set to zero  */
                            /*   by echo_cache_reset                                     */
  ECHO_NUM_COUNTERS = 32
};

/*
 * One layer's GPU cache ([REV] "In-graph per-layer cache management": a
 * preallocated free bitmap, eviction priorities, index buffers and a bidirectional
 * host<->GPU map).  Every pointer is caller-owned device memory, except host_kv,
 * which is the device-visible pointer of a pinned host buffer.
 *   host2gpu[n_host] : slot of each host token; -1 = not resident; <= -2 = staged in
 *                      this step at staging row (-2 - value), until the recall binds it
 *   gpu2host[n_gpu]  : host token in each slot; -1 = free
 *   priority[n_gpu]  : step of the slot's last touch (LRU key with the host index)
 *   index_buf[n_gpu] : the manager's scratch (victim-selection histograms, at most
 *                      3 x 2048 words; pools under 6 slots use counter words 24..29);
 *                      zero between calls, except, in pools of at least
 *                      ECHO_PENDING_LIST_MIN_SLOTS slots, its last 768 words: the
 *                      pending victim list that a recall leaves for the next
 *                      write-back (the recall ranks the B least recently used slots
 *                      it does not evict; the write-back evicts them in one CTA if
 *                      every slot still holds its recorded key, and otherwise runs
 *                      the full selection)
 *   free_map[n_gpu]  : one byte per slot, 1 = free
 * Metadata = 4*n_host + 13*n_gpu bytes (echo_cache_metadata_bytes) plus the fixed
 * 128-byte counters block.  gpu2host, priority and counters must be 16-byte aligned
 * (read as vectors); calls reject other layers with ECHO_ERR_INVALID_ARG.
 * The manager calls (write-back, recall, alloc, evict) are cooperative launches over
 * the whole device, one CTA per SM (a write-back on a pool of at least
 * ECHO_PENDING_LIST_MIN_SLOTS slots first launches one CTA that uses the pending
 * list; the cooperative launch then returns at once if that CTA did the work); calls
 * on one layer must not run concurrently, and only the library writes the layer's
 * arrays between calls.
 * A manager call whose grid barrier waited more than ~1 s sets ECHO_ERR_TIMEOUT and
 * leaves the layer undefined until echo_cache_reset.
 */
/* Pools of at least this many slots keep the pending victim list in index_buf: two
 * sets of three 2048-word histograms, 1024 miss counters and 3 x 256 list words. */
#define ECHO_PENDING_LIST_MIN_SLOTS 14080

typedef struct {
  int32_t n_gpu;
  int32_t n_host;
  int32_t *host2gpu;
  int32_t *gpu2host;
  int32_t *priority;
  int32_t *index_buf;
  uint8_t *free_map;
  int32_t *counters;   /* [ECHO_NUM_COUNTERS] */
  void *gpu_kv;        /* [n_gpu, 576], kv_dtype                                  */
  void *host_kv;       /* [n_host, 576], kv_dtype, pinned host memory (device view) */
  int32_t kv_dtype;    /* ECHO_F32 or ECHO_BF16                                    */
  /* Adaptive prefetch cap, optional (NULL pf_new_rows: the cap follows the context
   * alone).  [REV] "Decode: predict the transfer, then recall exactly" (the cap
   * limits the predicted transfer; the critique asks for its prediction error).
   * Per request b of the calls on this layer:
   *   pf_new_rows[b] tokens of its last exact selection that were not resident when
   *                  that step began (prefetched hits + misses); -1 = no step yet.
   *                  The step's budget (echo_cache_writeback inside
   *                  echo_decode_layer_step, or echo_cache_reserve) reads it and sets
   *                  it to 0; echo_cache_recall adds this step's rows to it.
   *   pf_pred_err[b] |theta - kth| / |kth| of the last step (float; 0 when either is
   *                  not finite or kth = 0), written by echo_topk_prefetch.
   *   cap_b = min(context cap, ceil(min((1 + pf_pred_err[b]) * pf_new_rows[b], 1e9))
   *               + cap_slack) once pf_new_rows[b] >= 0, the context cap before. */
  int32_t *pf_new_rows; /* [B] or NULL                                              */
  float *pf_pred_err;   /* [B] (with pf_new_rows)                                   */
  int32_t cap_slack;
  /* Block granularity, optional ([REV] critique: block-sparse / GQA models keep the
   * metadata per block of tokens).  0 or 1: every host index and slot is one token.
   * T > 1: one host index / slot holds T consecutive tokens of a request (host_kv
   * [n_host * T, 576], gpu_kv [n_gpu * T, 576], metadata 4*n_host + 13*n_gpu bytes
   * over blocks).  The write-back (host_base in tokens, a multiple of T per request)
   * writes each new token to its host row.  A token that starts a block that is not
   * resident takes a slot for it like a new token (victims: the LRU-smallest slots
   * not touched in this step); one in the middle of a block that is not resident
   * takes none.  After these binds, a token whose block is resident is written to the
   * block's GPU row and touches the block (priority = this step).  The recall (host_base in blocks: host_base / T) binds and copies
   * whole blocks; slot_idx holds block slots (echo_expand_block_slots makes the
   * token slots attention reads).  No fused prefetch: echo_index_prefetch with a cap
   * and echo_cache_recall with prefetched rows are rejected on such a layer, and so
   * is echo_decode_layer_step (ECHO_ERR_UNSUPPORTED). */
  int32_t block_tokens;
  /* Values per token row of host_kv and gpu_kv (and of the write-back's new_kv):
   * 0 means ECHO_KV_WIDTH (576, the MLA latent).  Otherwise a positive width whose
   * bytes are a multiple of 16, e.g. 2*d for one KV head's key and value of a GQA
   * layer (several KV heads, [REV] critique: a KV-head dimension; reading R26: each
   * (request, KV head) pair is a request of its own to the cache).  Layers with a
   * width other than 576 take no fused prefetch and no echo_decode_layer_step
   * (ECHO_ERR_UNSUPPORTED). */
  int32_t row_elems;
} echo_cache_layer_t;

/* sizeof of the structs this header declares (echo_cache_layer_t, echo_step_args_t,
 * echo_host_pool_t), in that order, written to out[0..2]: lets a binding check its
 * own copy of the layouts.  Pure host function. */
void echo_abi_struct_sizes(size_t out[3]);

/* Closed form of the per-layer metadata, 4*N_H + 13*N_G bytes
 * ([REV] "In-graph per-layer cache management": 2M host / 200K GPU slots give
 * about 10 MB per layer).  Pure host function. */
size_t echo_cache_metadata_bytes(int64_t n_host, int64_t n_gpu);

/* Device-visible address of pinned host memory (cudaHostGetDevicePointer).
 * host_ptr must come from cudaHostAlloc / pinned torch memory. */
echo_status_t echo_host_device_pointer(void *host_ptr, void **dev_ptr);

/* Number of SMs of the current device (for callers sizing persistent work). */
int32_t echo_device_sm_count(void);

/* Empty cache: every slot free, both maps -1, priorities 0, step 0, counters 0,
 * n_free = n_gpu.  The cache starts cold. */
echo_status_t echo_cache_reset(const echo_cache_layer_t *layer, echo_stream_t stream);

/*
 * A1 -- write-back of each request's new token ([REV] "In-graph per-layer cache
 * management": KV is backed up to the host when generated, so eviction needs no
 * copy back; "Trade-offs": every new token is written back).
 * Begins step s = counters[STEP] + 1.  For b = 0..B-1: h = host_base[b] + seq_len[b];
 * new_kv[b] (one row: 576 values, or the layer's row_elems; kv_dtype) is stored to host_kv[h] and to a GPU slot (a free
 * one, else the resident token with the smallest (priority, host index) among those
 * with priority < s is evicted); the slot's priority becomes s; new_ik[b] (D values,
 * ik_dtype) is appended to idx_k[b, seq_len[b]]; seq_len[b] += 1.
 *   new_kv [B,row] device; new_ik [B,D] device; idx_k [B,Lmax,D] device (in/out);
 *   host_base [B], seq_len [B] device int32 (seq_len in/out).
 * Device errors: HOST_INDEX if h >= n_host; POOL_EXHAUSTED if no slot can be freed;
 * a token whose seq_len has reached Lmax is not appended (INVALID_ARG status).
 */
echo_status_t echo_cache_writeback(const echo_cache_layer_t *layer, const void *new_kv,
                                   const void *new_ik, void *idx_k, int32_t D, int32_t Lmax,
                                   int32_t ik_dtype, const int32_t *host_base, int32_t *seq_len,
                                   int32_t B, echo_stream_t stream);

/*
 * A2 -- reserve the prefetch budget of this step before scoring ([REV] "Decode:
 * predict the transfer, then recall exactly": a global counter caps the prefetch
 * volume, and the cap grows with the context).  For each request:
 * cap[b] = min(cap_max, ceil(seq_len[b] / cap_div)) (cap_div > 0) or cap_max
 * (cap_div == 0); pf_count[b] = 0.  The per-request staging area holds cap_max rows,
 * so cap[b] rows of it are reserved.
 *   seq_len [B], cap [B] (out), pf_count [B] (out) device int32.
 */
echo_status_t echo_cache_reserve(const echo_cache_layer_t *layer, const int32_t *seq_len,
                                 int32_t B, int32_t cap_max, int32_t cap_div, int32_t *cap,
                                 int32_t *pf_count, echo_stream_t stream);

/*
 * A3 + A4 -- lightning-indexer scoring with fused threshold prefetch
 * ([REV] "Problem and motivation": the DSA indexer scores every past token;
 *  [DSA] score_b(t) = sum_h w[b,h] * ReLU(q[b,h,:] . idx_k[b,t,:]);
 *  [REV] "Decode: predict the transfer, then recall exactly" and "Fusing prefetch
 *  into the indexer pipeline": as soon as a block of scores exists, tokens above the
 *  EMA threshold that are not cached are fetched, without waiting for the top-k).
 *   q      [B,H,D]  dtype (ECHO_E4M3 with H=64, D=128, or ECHO_F32 with D % 4 == 0)
 *   w      [B,H]    float32 head weights
 *   idx_k  [B,Lmax,D] dtype: GPU-resident indexer keys (never offloaded)
 *   seq_len[B]      device int32, tokens 0..seq_len[b]-1 are scored
 *   scores [B,Lmax] float32 out (entries >= seq_len[b] untouched)
 *   theta  [B]      float32 EMA threshold; +inf marks nothing
 *   cap    [B]      device int32 from echo_cache_reserve, or NULL for no prefetch
 *   pf_list[B,cap_max] int32 out: prefetched token indices of request b in rows
 *                   0..pf_count[b]-1 (any order); staging row of pf_list[b,i] is b*cap_max+i
 *   pf_count[B]     int32 in/out (zeroed by echo_cache_reserve): rows staged
 *   stage_kv[B*cap_max, 576] kv_dtype out: staged latent rows (host -> GPU copies)
 * Prefetch rule: t is staged iff score > theta[b] (strict), host2gpu[h] == -1, and t is
 * among the first cap[b] such tokens by ascending t.  Staged tokens get
 * host2gpu[h] = -2 - staging_row until echo_cache_recall binds them.
 *   flags  0, or ECHO_PF_DEFER_CAP: rows are claimed in arrival order and, when a
 *          request's qualifying tokens outnumber its cap, the "first cap by t" rule
 *          is restored by a later call: pf_count[b] then holds the number of
 *          qualifying tokens (staged rows = min(pf_count[b], cap)) until
 *          echo_topk_prefetch, which must run next on the same stream with the same
 *          scores, theta (before its update), cap and layer.  Without the flag the
 *          rule is restored by a small extra launch before this call returns.
 * Device errors: STAGING if cap[b] > cap_max; TIMEOUT if a bounded wait gave up.
 */
#define ECHO_PF_DEFER_CAP 1
echo_status_t echo_index_prefetch(const void *q, const float *w, const void *idx_k,
                                  const int32_t *seq_len, int32_t B, int32_t H, int32_t D,
                                  int32_t Lmax, int32_t dtype, const float *theta,
                                  const int32_t *cap, int32_t cap_max, const int32_t *host_base,
                                  const echo_cache_layer_t *layer, float *scores, int32_t *pf_list,
                                  int32_t *pf_count, void *stage_kv, int32_t flags,
                                  echo_stream_t stream);

/*
 * A5 -- exact top-k with the EMA threshold update ([REV] "Problem and motivation":
 * the 2048 highest-scoring tokens; "Decode: ...": exact top-k after the indexer;
 * "Key observations" Obs. 2: EMA of the k-th score with smoothing 0.5).
 * For each b: out_idx[b, 0..k) = the k tokens of largest score (equal scores: lower
 * token index first), any order; if seq_len[b] < k all tokens are selected and the
 * rest of the row is -1.  kth[b] = the smallest selected score (-inf if none);
 * theta[b] <- kth[b] if theta[b] == +inf, else alpha*kth[b] + (1-alpha)*theta[b]
 * (float32, each operation rounded, no fused multiply-add).
 *   scores [B,Lmax] float32; seq_len [B]; out_idx [B,k] int32; kth [B]; theta [B] in/out.
 * kth's contents on entry (the previous step's k-th scores when the caller keeps the
 * buffer) only size the search around theta: any value gives the same results.
 */
echo_status_t echo_topk(const float *scores, const int32_t *seq_len, int32_t B, int32_t Lmax,
                        int32_t k, int32_t *out_idx, float *kth, float *theta, float alpha,
                        echo_stream_t stream);

/*
 * A5 + the deferred end of A4 -- echo_topk, and in the same launch the exact prefetch
 * cap of an echo_index_prefetch call made with ECHO_PF_DEFER_CAP ([REV] "Decode:
 * ...": a counter caps the prefetch volume; "Fusing prefetch into the indexer
 * pipeline": prefetch adds no step of its own to the decode path).  For a request
 * whose pf_count[b] exceeds min(cap[b], cap_max), tokens claimed beyond the first
 * cap qualifiers by t give their staging rows to the qualifiers that were left out
 * (maps, pf_list and stage_kv rows rewritten); then pf_count[b] = min(count, cap).
 * The threshold used is theta[b] as it was before this call's EMA update.
 *   top-k arguments as echo_topk; cap, cap_max, host_base, layer, pf_list, pf_count,
 *   stage_kv as passed to echo_index_prefetch (all required).
 */
echo_status_t echo_topk_prefetch(const float *scores, const int32_t *seq_len, int32_t B,
                                 int32_t Lmax, int32_t k, int32_t *out_idx, float *kth,
                                 float *theta, float alpha, const int32_t *cap, int32_t cap_max,
                                 const int32_t *host_base, const echo_cache_layer_t *layer,
                                 int32_t *pf_list, int32_t *pf_count, void *stage_kv,
                                 echo_stream_t stream);

/*
 * A7 -- eviction with protection ([REV] "In-graph per-layer cache management":
 * release protects the current selection, then frees low-priority slots and
 * updates the maps; no data is written back).  Frees
 * m = max(0, *n_needed - n_free) slots: the resident tokens with the smallest
 * (priority, host index) among those with priority < current step (everything
 * touched in this step -- write-back, selection, prefetch bind -- is protected).
 *   n_needed: device int32 scalar.  Device errors: POOL_EXHAUSTED if fewer than m
 *   tokens are evictable (all of those are evicted).
 */
echo_status_t echo_cache_evict(const echo_cache_layer_t *layer, const int32_t *n_needed,
                               echo_stream_t stream);

/*
 * A8 -- allocation by a parallel scan of the free bitmap with one atomic count per
 * warp ([REV] "In-graph per-layer cache management").  Binds host_idx[0..*n) to
 * free slots (any slots): maps set, priority = current step, out_slot[i] = slot
 * (-1 if none was free).  host_idx [n_max], n device scalar (<= n_max), out_slot [n_max].
 * Device errors: POOL_EXHAUSTED if fewer than *n slots are free; HOST_INDEX.
 */
echo_status_t echo_cache_alloc(const echo_cache_layer_t *layer, const int32_t *host_idx,
                               const int32_t *n, int32_t n_max, int32_t *out_slot,
                               echo_stream_t stream);

/*
 * A6 + A7 + A8 + A9 + A10 -- recall after the exact top-k ([REV] "In-graph per-layer
 * cache management": find the missing entries from the map, allocate slots, and a GPU
 * kernel reads host memory directly to copy the KV; "Decode: ... recall exactly":
 * every selected token that is not resident is fetched before attention).
 * In order: (1) every selected resident token gets priority = step (protection);
 * (2) misses = selected tokens neither resident nor staged, listed in
 * miss_list[b, 0..n_miss[b]) (any order); (3) evict so that every staged row and
 * every miss has a slot (echo_cache_evict rule); (4) bind staged rows (pf_list) and
 * misses to free slots (echo_cache_alloc rule); (5) copy staged rows from stage_kv
 * and missed rows from host_kv (zero-copy 16-byte reads of pinned host memory);
 * (6) slot_idx[b,j] = slot of sel[b,j] (-1 where sel is -1).
 *   sel [B,k], host_base [B]; pf_list/pf_count/stage_kv as produced by
 *   echo_index_prefetch (pf_count may be NULL: nothing staged); miss_list [B,k],
 *   n_miss [B], slot_idx [B,k] out.
 */
echo_status_t echo_cache_recall(const echo_cache_layer_t *layer, const int32_t *sel,
                                const int32_t *host_base, int32_t B, int32_t k,
                                const int32_t *pf_list, const int32_t *pf_count, int32_t cap_max,
                                const void *stage_kv, int32_t *miss_list, int32_t *n_miss,
                                int32_t *slot_idx, echo_stream_t stream);

/*
 * A11 -- sparse MLA decode attention over the selected rows ([REV] "Problem and
 * motivation": MLA over the top-2048 tokens; latents are 576 wide, values are the
 * first 512 dims).  For each b and head h:
 *   logit_j = scale * q[b,h,:] . kv[slot_idx[b,j], :]   (all 576 dims; -1 skipped)
 *   out[b,h,:] = softmax_j(logit) . kv[slot_idx[b,j], 0:512];  lse[b,h] = log sum_j exp(logit_j)
 *   q [B,Hq,576] dtype; kv [kv_rows,576] dtype (a layer's gpu_kv, or any dense
 *   buffer); out [B,Hq,512] dtype; lse [B,Hq] float32.
 *   dtype ECHO_BF16 (Hq = 128, tensor cores) or ECHO_F32 (any Hq <= 128).
 *   workspace: echo_sparse_mla_workspace_bytes(B, Hq, k) bytes of device memory.
 * A row with no valid entry gives out = 0 and lse = -inf.  The result depends only on
 * the rows and their order in slot_idx, so attention over the cache equals attention
 * over any other buffer holding the same rows in the same order (lossless check).
 */
size_t echo_sparse_mla_workspace_bytes(int32_t B, int32_t Hq, int32_t k);
echo_status_t echo_sparse_mla_decode(const void *q, const void *kv, int32_t kv_rows, int32_t dtype,
                                     const int32_t *slot_idx, int32_t B, int32_t Hq, int32_t k,
                                     float scale, void *out, float *lse, void *workspace,
                                     size_t workspace_bytes, echo_stream_t stream);

/*
 * N4 -- sparse attention of a GQA layer with several KV heads ([REV] critique: a
 * KV-head dimension; reading R26).  A group n is one (request, KV head) pair; its G
 * query heads attend over the rows selected for it:
 *   logit_j = scale * q[n,g,:] . kv[slot_idx[n,j], 0:d]          (-1 entries skipped)
 *   out[n,g,:] = softmax_j(logit) . kv[slot_idx[n,j], d:2d];  lse[n,g] = log sum_j exp(logit_j)
 *   q [NG,G,d] dtype (a request's [Hq,d] queries with query head i = h*G + g belong to
 *   KV head h); kv [kv_rows, 2d] dtype (key then value per row, a layer's gpu_kv with
 *   row_elems = 2d); slot_idx [NG,k]; out [NG,G,d] dtype; lse [NG,G] float32.
 *   d = 64 or 128; 1 <= G <= 16; dtype ECHO_BF16 (tensor cores) or ECHO_F32.
 *   workspace: echo_sparse_gqa_workspace_bytes(NG, G, d, k) bytes of device memory
 *   (0 when the call needs none).
 * A group with no valid entry gives out = 0 and lse = -inf.
 */
size_t echo_sparse_gqa_workspace_bytes(int32_t NG, int32_t G, int32_t d, int32_t k);
echo_status_t echo_sparse_gqa_decode(const void *q, const void *kv, int32_t kv_rows, int32_t dtype,
                                     const int32_t *slot_idx, int32_t NG, int32_t G, int32_t d, int32_t k,
                                     float scale, void *out, float *lse, void *workspace,
                                     size_t workspace_bytes, echo_stream_t stream);

/*
 * Sparse MLA decode for callers that cannot allocate device memory.  The paper has
 * no counterpart: this is a packaging variant of echo_sparse_mla_decode for code
 * that may not call cudaMalloc (or any allocating runtime or framework routine) at
 * run time -- for example a plug-in running inside another engine's memory pool, a
 * process whose allocator is owned by someone else, or a step being recorded where
 * allocation is not allowed.  It computes exactly what echo_sparse_mla_decode
 * computes, with the same arguments minus the workspace: the split partials live in
 * a scratch array built into the library (ECHO_MLA_NOALLOC_SCRATCH_BYTES, 32 MiB,
 * held on every GPU that loads the library until the process exits).
 *   - Sizes: the call needs echo_sparse_mla_workspace_bytes(B, Hq, k) <= 32 MiB
 *     (for Hq = 128 and k = 2048 that is up to 15 requests); larger calls return
 *     ECHO_ERR_SCRATCH_LIMIT and launch nothing.
 *   - Set-up: the first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  A failed look-up returns ECHO_ERR_CUDA.
 *   - Sharing: every call on a device uses the same scratch array, which keeps the
 *     last call's contents.  Nothing in it has to start at zero (each call writes
 *     every partial before reading it), but two calls that overlap on the GPU (on
 *     different streams, or from different threads) race and corrupt each other's
 *     results: serialise them.
 */
#define ECHO_MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
echo_status_t echo_sparse_mla_decode_noalloc(const void *q, const void *kv, int32_t kv_rows, int32_t dtype,
                                             const int32_t *slot_idx, int32_t B, int32_t Hq, int32_t k,
                                             float scale, void *out, float *lse, echo_stream_t stream);

/*
 * One layer's whole decode step, A1..A11, enqueued on one stream in the pages'
 * order ([REV] "Decode: predict the transfer, then recall exactly"): write-back,
 * reserve, score + prefetch, top-k + EMA, recall, sparse MLA.  With prefetch = 0 the
 * indexer runs without the fused prefetch (the unfused index -> top-k -> recall
 * sequence).  Every argument keeps the meaning it has in the single calls.
 */
typedef struct {
  int32_t B;
  const int32_t *host_base; /* [B]                                  */
  int32_t *seq_len;         /* [B] in/out                           */
  /* indexer */
  int32_t H, D, Lmax, idx_dtype;
  const void *q_idx;        /* [B,H,D]                              */
  const float *w_idx;       /* [B,H]                                */
  void *idx_k;              /* [B,Lmax,D]                           */
  const void *new_ik;       /* [B,D]                                */
  const void *new_kv;       /* [B,576]                              */
  float *theta;             /* [B] in/out                           */
  float alpha;
  int32_t k;
  int32_t prefetch;         /* 1 = fused prefetch, 0 = none         */
  int32_t cap_max, cap_div;
  int32_t *cap;             /* [B]                                  */
  float *scores;            /* [B,Lmax]                             */
  int32_t *pf_list;         /* [B,cap_max]                          */
  int32_t *pf_count;        /* [B]                                  */
  void *stage_kv;           /* [B*cap_max,576]                      */
  int32_t *sel;             /* [B,k]                                */
  float *kth;               /* [B]                                  */
  int32_t *miss_list;       /* [B,k]                                */
  int32_t *n_miss;          /* [B]                                  */
  int32_t *slot_idx;        /* [B,k]                                */
  /* attention */
  int32_t Hq;
  const void *q_mla;        /* [B,Hq,576]                           */
  float scale;
  void *out;                /* [B,Hq,512]                           */
  float *lse;               /* [B,Hq]                               */
  void *mla_workspace;
  size_t mla_workspace_bytes;
  /* optional profiling hook: two cudaEvent_t recorded around the indexer launch
   * (as external event nodes when the step is captured in a graph); NULL: none */
  void *index_events[2];
} echo_step_args_t;

echo_status_t echo_decode_layer_step(const echo_cache_layer_t *layer, const echo_step_args_t *a,
                                     echo_stream_t stream);

/* Synchronises the stream's device and copies counters[ECHO_CTR_STATUS] to
 * *host_status.  Returns ECHO_ERR_CUDA if the device reported an error. */
echo_status_t echo_cache_status(const echo_cache_layer_t *layer, int32_t *host_status);

/* Synchronising copy of the whole counters block to host_counters[ECHO_NUM_COUNTERS]. */
echo_status_t echo_cache_read_counters(const echo_cache_layer_t *layer, int32_t *host_counters);

/*
 * P1 -- prefill chunk indexing ([REV] "Prefill: overlap recall across query blocks":
 * the chunk is scored in query blocks; a 256-bucket coarse histogram picks the
 * buckets certainly above the selection boundary and leaves the threshold bucket
 * for later, after the predicted k-th score is subtracted; the KV of block i's
 * candidates moves while block i+1 is scored; exact top-k and recall follow).
 *
 * echo_prefill_index: scores of one query block of one request.  Query j sits at
 * position pos0 + j and scores the tokens t <= pos0 + j (causal, its own key
 * included): scores[j, t] = sum_h w[j,h] * ReLU(q[j,h,:] . idx_k[t,:]).  Also the
 * per-query histogram hist[j, b] = #{t : bucket(scores[j,t] - kth_pred[j]) == b},
 * bucket(d) = top 8 bits of the order-preserving 32-bit key of d (non-negative d:
 * sign bit set; negative d: every bit inverted; -0 counts as +0), d in float32.
 *   q [Q,64,128] e4m3 (16-byte aligned), w [Q,64] f32, idx_k [Lmax,128] e4m3 (this
 *   request's indexer keys, 16-byte aligned), pos0 + Q <= Lmax, kth_pred [Q] f32;
 *   scores [Q,Lmax] f32 out (entries past each query's causal range untouched);
 *   hist [Q,256] u32 out (zeroed by the call); status: optional device int32 that
 *   receives ECHO_ERR_TIMEOUT if a bounded wait gave up.
 *   H must be 64 and D 128 (ECHO_ERR_UNSUPPORTED otherwise).
 */
echo_status_t echo_prefill_index(const void *q, const float *w, const void *idx_k, int32_t Q, int32_t H,
                                 int32_t D, int32_t Lmax, int32_t pos0, const float *kth_pred,
                                 float *scores, uint32_t *hist, int32_t *status, echo_stream_t stream);

/*
 * P1 -- candidates of a scored block.  For query j with L_j = pos0 + j + 1 tokens:
 * thr[j] = the bucket holding the k-th largest d (counted from bucket 255 down), or
 * -1 when L_j <= k; candidates = tokens whose bucket is strictly above thr[j] (each
 * is in the exact top-k).  Candidate tokens are OR-ed into bitmap (bit t of word
 * t/32; the union over the block's queries); cand_count[j] = their number.
 *   scores/hist as produced by echo_prefill_index; thr, cand_count [Q] (may be
 *   NULL); bitmap [ceil(Lmax/32)] u32, in/out.
 */
echo_status_t echo_prefill_candidates(const float *scores, const uint32_t *hist, int32_t Q, int32_t Lmax,
                                      int32_t pos0, int32_t k, const float *kth_pred, int32_t *thr,
                                      int32_t *cand_count, uint32_t *bitmap, echo_stream_t stream);

/* P1 -- OR the tokens of rows x row_len token lists (entries < 0 or >= nbits are
 * skipped) into bitmap [ceil(nbits/32)]: the union of a block's exact selections. */
echo_status_t echo_mark_tokens(const int32_t *tok, int32_t rows, int32_t row_len, uint32_t *bitmap,
                               int32_t nbits, echo_stream_t stream);

/* P1 -- bitmap -> list: list[0..count) = the set tokens in ascending order, the rest
 * of list[0..cap) = -1; *count (device int32) = number of set tokens (only the first
 * cap are written).  The bitmap is left all-zero.  The list is the selection row of
 * a one-request echo_cache_recall (the block's union, recalled once). */
echo_status_t echo_token_list(uint32_t *bitmap, int32_t nbits, int32_t *list, int32_t cap, int32_t *count,
                              echo_stream_t stream);

/*
 * Prefill sparse attention, slot translation ([REV] "Prefill: overlap recall across
 * query blocks": once a block's union is resident, each of its queries attends over
 * its own exact selection; [REV] "Problem and motivation": MLA over the selected
 * tokens).  For every entry of rows x k token lists:
 *   out_slot[r, j] = host2gpu[base_r + tok[r, j]]  (tok >= 0), else -1,
 * with base_r = host_base[r] when per_row_base != 0, host_base[0] otherwise.  The
 * result is the slot_idx of echo_sparse_mla_decode with one "request" per query row.
 * A listed token that is not resident gives -1 and sets the layer's sticky status to
 * ECHO_ERR_NOT_RESIDENT; a host index outside [0, n_host) gives -1 and sets
 * ECHO_ERR_HOST_INDEX.  Reads the maps only.
 *   tok, out_slot [rows, k] i32 (device); host_base [rows] or [1] i32 (device).
 */
echo_status_t echo_translate_slots(const echo_cache_layer_t *layer, const int32_t *tok, int32_t rows, int32_t k,
                                   const int32_t *host_base, int32_t per_row_base, int32_t *out_slot,
                                   echo_stream_t stream);

/*
 * N1 -- model-wide host pool ([REV] "In-graph per-layer cache management": each
 * layer's GPU cache is managed inside the graph, the host pool for the whole model).
 * One pinned buffer (caller-owned, echo_host_pool_bytes long) holds every layer's
 * host rows: layer l's rows are [l * rows_per_layer, (l + 1) * rows_per_layer) of
 * ECHO_KV_WIDTH-wide latents.  A request's context takes the same row range in every
 * layer, so one allocation serves all layers and the request's host_base is shared
 * by them.  Row ranges are handed out first fit from a sorted, coalesced free list
 * kept inside the struct (at most ECHO_HOST_POOL_MAX_RANGES free ranges).
 * Host-side code: no CUDA call except echo_host_pool_layer.  Not thread-safe: one
 * caller at a time per pool.
 */
#define ECHO_HOST_POOL_MAX_RANGES 1024

typedef struct {
  void *base;                  /* pinned host buffer                            */
  int32_t n_layers;
  int32_t kv_dtype;            /* ECHO_F32 or ECHO_BF16                         */
  int64_t rows_per_layer;
  int64_t rows_in_use;
  int32_t n_free;              /* free ranges: ascending, disjoint, coalesced   */
  int64_t free_first[ECHO_HOST_POOL_MAX_RANGES];
  int64_t free_rows[ECHO_HOST_POOL_MAX_RANGES];
} echo_host_pool_t;

/* Bytes of the pinned buffer: n_layers * rows_per_layer rows of 576 elements (0 on bad sizes). */
size_t echo_host_pool_bytes(int32_t n_layers, int64_t rows_per_layer, int32_t kv_dtype);

/* Describe base as a pool of n_layers x rows_per_layer rows, all free. */
echo_status_t echo_host_pool_init(echo_host_pool_t *pool, void *base, int32_t n_layers, int64_t rows_per_layer,
                                  int32_t kv_dtype);

/* Take `rows` consecutive rows (the lowest free range that holds them) in every layer:
 * *first_row = their first row (a request's host_base).  ECHO_ERR_POOL_EXHAUSTED when
 * no free range is long enough (nothing changes). */
echo_status_t echo_host_pool_alloc(echo_host_pool_t *pool, int64_t rows, int64_t *first_row);

/* Give a range back; it is merged with free neighbours.  ECHO_ERR_INVALID_ARG if it is
 * out of range or overlaps a free range (a double free); ECHO_ERR_UNSUPPORTED if the free
 * list would need more than ECHO_HOST_POOL_MAX_RANGES entries (nothing changes). */
echo_status_t echo_host_pool_free(echo_host_pool_t *pool, int64_t first_row, int64_t rows);

/* Layer l's rows: host pointer and device-visible pointer (cudaHostGetDevicePointer of the
 * pinned buffer), for echo_cache_layer_t.host_kv with n_host = rows_per_layer. */
echo_status_t echo_host_pool_layer(const echo_host_pool_t *pool, int32_t layer, void **host_rows,
                                   void **host_rows_dev);

/*
 * N4 -- block-sparse selection ([REV] critique: block-sparse / GQA adaptation; reading
 * R25).  echo_block_scores: for each request b and block j < ceil(seq_len[b] / T),
 * bscores[b, j] = the largest of scores[b, j*T .. min(seq_len[b], j*T + T)); seq_len_blk[b]
 * = ceil(seq_len[b] / T).  Then echo_topk over (bscores, seq_len_blk, k/T) selects the
 * blocks exactly (ties to the lower block) and keeps theta as the EMA of the k/T-th
 * block score.
 *   scores [B, Lmax] f32; seq_len [B]; bscores [B, ceil(Lmax / T)] f32 out; seq_len_blk [B] out.
 */
echo_status_t echo_block_scores(const float *scores, const int32_t *seq_len, int32_t B, int32_t Lmax, int32_t T,
                                float *bscores, int32_t *seq_len_blk, echo_stream_t stream);

/*
 * N4 -- token slots of the selected blocks, for echo_sparse_mla_decode over the GPU
 * pool read as [n_gpu * T, 576]: out[b, j*T + i] = block_slot[b, j] * T + i when
 * sel_blk[b, j] >= 0, block_slot[b, j] >= 0 and sel_blk[b, j]*T + i < seq_len[b];
 * else -1.
 *   sel_blk, block_slot [B, kb] i32 (the block top-k and the recall's slot_idx);
 *   seq_len [B]; out [B, kb*T] i32.
 */
echo_status_t echo_expand_block_slots(const int32_t *sel_blk, const int32_t *block_slot, const int32_t *seq_len,
                                      int32_t B, int32_t kb, int32_t T, int32_t *out, echo_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* ECHO_H */
