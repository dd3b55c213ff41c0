/*
 * echo_oracle.cpp -- plain CPU oracle of the ECHO per-layer decode hot path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke() and
 * bench.py's CPU-baseline / reference legs load this library (through
 * oracle/cpp_oracle.py).  The CUDA library never includes, links or calls it, and
 * the two share no code: no kernels, headers, helpers, tables or pre/post
 * processing.  Inputs reach both sides only through the seeded generators, which
 * hold none of the method's arithmetic.
 *
 * Plain, slow C++17: every floating-point step in double (the EMA in float, as the
 * method keeps it), loops in the order the pages state the computation, library
 * primitives (std::sort, exp, log) as single steps.  Compiled with
 * -ffp-contract=off, so no multiply-add is fused.  OpenMP only spreads independent
 * token scores over cores; each score is one thread's loop in a fixed order.
 *
 * Sources (cited below by tag and section):
 *   [REV]   "ECHO: Efficient KV Cache Offloading with Lossless Prefetching for
 *           Serving Native Sparse Attention LLMs (OSDI 2026)" review page
 *           (awesome-system-papers).  Sections "Problem and motivation",
 *           "Key observations" (Obs. 2), "In-graph per-layer cache management",
 *           "Decode: predict the transfer, then recall exactly",
 *           "Prefill: overlap recall across query blocks".
 *   [DSA]   DeepSeek-V3.2-Exp report, listed among the show notes' sources: the
 *           lightning indexer score sum_h w_h * ReLU(q_h . k_t).
 *
 * Parity unpinned: the prefill bucket mapping (reading R19 below).  The pages fix a
 * 256-bucket coarse histogram of the score minus the predicted k-th score, but print
 * no example of the mapping; its properties (monotone in d, finer near d = 0) are
 * pinned, the exact mapping is not.
 *
 * Readings taken where the pages are silent:
 *   R1  indexer score: no extra scale; every t < L_b is scored, the token written
 *       back in this step included.
 *   R2  top-k with L < k selects all L tokens; kth is the smallest selected score;
 *       L = 0 selects nothing and kth = -inf.
 *   R3  equal scores: the lower token index wins.
 *   R4  EMA: theta <- alpha*kth + (1-alpha)*theta in float, each operation rounded;
 *       theta = +inf before the first observation, which sets theta = kth.
 *   R5  "above the threshold" is strict: score > theta.
 *   R6  the prefetch counter is per (request, layer, step); under the cap the
 *       lowest token indices win.
 *   R7  cap_b = min(cap_max, ceil(L_b / cap_div)) when cap_div > 0, else cap_max.
 *   R8  eviction priority = step of the last touch (write-back, prefetch bind,
 *       selection); victims are the smallest (priority, host index) among resident
 *       tokens with priority < s, so everything touched in step s is protected.
 *   R9  prefetched rows are staged during scoring and bound to GPU slots in the
 *       recall of the same step, after the selection is protected; every staged
 *       row is bound.
 *   R10 the new token of each step enters both the host pool and the GPU cache.
 *   R15 host index of token t of request b is host_base[b] + t.
 *   R16 the write-back begins a step: s <- s + 1.
 *   R17 a recall that cannot free enough slots evicts every eligible token, binds
 *       what it can (staged rows first, then misses, in (b, t) order) and reports
 *       pool exhaustion.
 *   R18 prefill: query j of a block that starts at pos0 scores t <= pos0 + j.
 *   R19 prefill bucket: d = score - kth_pred in float (one rounding); bucket = top 8
 *       bits of the order-preserving 32-bit key of d (non-negative: sign bit set;
 *       negative: every bit inverted; -0 counts as +0).
 *   R20 prefill threshold bucket = the bucket of the query's k-th largest d, counted
 *       down from bucket 255; candidates = tokens in strictly higher buckets.  A
 *       query with at most k tokens has every token as a candidate.
 *   R21 a block's recall list is the union of its queries' tokens, ascending.
 *   R23 adaptive cap (optional): with u_b = the tokens of request b's selection in
 *       the previous step that were not resident when that step began (its
 *       prefetched hits plus its misses) and e_b = that step's relative prediction
 *       error |theta - kth| / |kth| (float; 0 when either is not finite or kth = 0),
 *       cap_b = min(R7's cap, ceil((1 + e_b) * u_b) + slack); before any
 *       observation (u_b < 0) R7's cap alone.
 *   R25 block granularity (optional): T consecutive tokens of a request form a block
 *       (the request's host base a multiple of T), the unit of residency.  A block's
 *       score is the largest score of its tokens; the selection is the exact top-k/T
 *       blocks (ties to the lower block), theta the EMA of the k/T-th block score.  The
 *       write-back writes every new token to the host pool.  First each token that
 *       starts a block takes a slot for it (evicting the LRU-smallest block not touched
 *       in this step if none is free), in request order; then the block that receives
 *       each token, if resident, is touched in this step (so the binds of one step do
 *       not depend on the order of the requests' rows).  A token in the middle of a
 *       block that is not resident takes no slot (a later recall copies the whole block
 *       from the host, the new token included).  Attention runs over every token of the
 *       selected blocks below the context length.  Metadata is the per-token formula
 *       over blocks: 4 * N_H / T + 13 * N_G / T bytes.  No fused prefetch.
 *   R26 several KV heads (optional): a GQA layer with n_kv KV heads of dimension d and
 *       G query heads per KV head adds a KV-head dimension to the cache: each (request,
 *       KV head) pair is a unit of its own (own host rows of 2d values per token: key
 *       then value, own indexer scores and top-k, own residency), so the metadata grows
 *       by n_kv and its per-unit rules (R1-R25) are unchanged.  Query head i of a
 *       request attends with KV head i / G over that head's selected tokens, logits
 *       scaled by 1/sqrt(d).
 */

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

constexpr int64_t kNotResident = -1;
constexpr int32_t kOk = 0;
constexpr int32_t kPoolExhausted = 5;
constexpr int32_t kHostIndex = 6;

const double kInf = std::numeric_limits<double>::infinity();

inline double key_value(const void *keys, int key_dtype, int64_t i) {
  return key_dtype == 1 ? (double)static_cast<const float *>(keys)[i] : static_cast<const double *>(keys)[i];
}

}  // namespace

extern "C" {

/* One layer's GPU cache state ([REV] "In-graph per-layer cache management": a free
 * bitmap, eviction priorities and a bidirectional host<->GPU map).  The arrays
 * belong to the caller; the oracle's functions read and write them in place. */
typedef struct {
  int64_t n_gpu, n_host;
  int64_t *host2gpu;   /* [n_host] slot of each host token, -1 = not resident */
  int64_t *gpu2host;   /* [n_gpu]  host token in each slot, -1 = free          */
  int64_t *priority;   /* [n_gpu]  step of the slot's last touch               */
  uint8_t *free_map;   /* [n_gpu]  1 = free                                    */
  int64_t step;        /* current decode step s                                */
  int32_t status;      /* first error seen (0 = none)                          */
} orc_cache_t;

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* [REV] "In-graph per-layer cache management": 4 bytes per host token (the
 * host->GPU entry) and per GPU slot 4 (GPU->host) + 4 (priority) + 4 (index
 * buffer) + 1 (free byte) = 13 bytes. */
int64_t orc_metadata_bytes(int64_t n_host, int64_t n_gpu) { return 4 * n_host + 13 * n_gpu; }

/* Lightning indexer ([REV] "Problem and motivation"; [DSA]):
 *   score(t) = sum_h w[h] * max(0, q[h] . key[t])      (double)
 * q [H, D], w [H], keys [L, D] (key_dtype 0 = double, 1 = float) -> out [L]. */
void orc_indexer_scores(const double *q, const double *w, int64_t H, int64_t D, const void *keys, int key_dtype,
                        int64_t L, double *out) {
#pragma omp parallel for schedule(static) if (L * H * D > (int64_t)1 << 20)
  for (int64_t t = 0; t < L; ++t) {
    double score = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d) dot += q[h * D + d] * key_value(keys, key_dtype, t * D + d);
      const double relu = dot > 0.0 ? dot : 0.0;
      score += w[h] * relu;
    }
    out[t] = score;
  }
}

/* Store double scores as float, refusing any that float cannot hold exactly (on the
 * synthetic FP8 grid every score is exact).  Returns -1, or the first bad index. */
int64_t orc_to_f32_exact(const double *x, int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) {
    const float f = (float)x[i];
    if ((double)f != x[i]) return i;
    out[i] = f;
  }
  return -1;
}

/* Exact top-k ([REV] "Problem and motivation": top 2048; "Decode: ... recall
 * exactly"): the k highest scores, equal scores going to the lower token index
 * (R2, R3).  sel gets min(k, L) token indices, best first; kth the last one's score
 * (-inf when L == 0).  Returns the number selected. */
int64_t orc_topk_select(const double *s, int64_t L, int64_t k, int64_t *sel, double *kth) {
  std::vector<int64_t> order(L);
  std::iota(order.begin(), order.end(), (int64_t)0);
  std::sort(order.begin(), order.end(), [s](int64_t a, int64_t b) {
    if (s[a] != s[b]) return s[a] > s[b];
    return a < b;
  });
  const int64_t n = std::min(k, L);
  for (int64_t i = 0; i < n; ++i) sel[i] = order[i];
  *kth = n > 0 ? s[order[n - 1]] : -kInf;
  return n;
}

/* EMA of the k-th score ([REV] "Key observations" Obs. 2: smoothing 0.5), R4:
 * float, one rounding per operation. */
float orc_ema_update(float theta, float kth, float alpha) {
  if (std::isinf(kth) && kth < 0.0f) return theta;     /* nothing selected: unchanged */
  if (std::isinf(theta) && theta > 0.0f) return kth;   /* first observation */
  const float a = alpha;
  const float b = 1.0f - a;
  const float x = a * kth;
  const float y = b * theta;
  return x + y;
}

/* R7: the cap grows with the context ([REV] "Decode: ...": the limit grows with the
 * context length). */
int64_t orc_prefetch_cap(int64_t L, int64_t cap_max, int64_t cap_div) {
  if (cap_max <= 0) return 0;
  if (cap_div > 0) {
    const int64_t c = L >= 0 ? (L + cap_div - 1) / cap_div : -((-L) / cap_div);
    return std::min(cap_max, c);
  }
  return cap_max;
}

/* R23: relative prediction error of one step, in float: |theta - kth| / |kth| ([REV]
 * "Decode: predict the transfer ...": theta predicts this step's k-th score). */
float orc_prediction_error(float theta, float kth) {
  if (!std::isfinite(theta) || !std::isfinite(kth) || kth == 0.0f) return 0.0f;
  const float d = std::fabs(theta - kth);
  return d / std::fabs(kth);
}

/* R23: the adaptive cap -- last step's transfer, grown by the predictor's relative
 * error, plus a slack; never above the context rule R7.  new_rows < 0: no
 * observation yet. */
int64_t orc_adaptive_cap(int64_t L, int64_t cap_max, int64_t cap_div, int64_t new_rows, float pred_err,
                         int64_t slack) {
  const int64_t base = orc_prefetch_cap(L, cap_max, cap_div);
  if (new_rows < 0 || base <= 0) return base;
  const float grow = 1.0f + pred_err;
  const float want = std::min(grow * (float)new_rows, 1.0e9f);   /* a huge error: no limit but R7's */
  const int64_t c = (int64_t)std::ceil(want) + slack;
  return std::min(base, std::max<int64_t>(c, 0));
}

/* Tokens prefetched while scoring ([REV] "Decode: predict the transfer ..."): score
 * strictly above the EMA threshold (R5), not resident, and among the first cap such
 * tokens by ascending index (R6).  theta = +inf or NaN marks none.  resident [L]
 * is 0/1.  Returns the count written to out. */
int64_t orc_prefetch_marks(const double *scores, int64_t L, float theta, const uint8_t *resident, int64_t cap,
                           int64_t *out) {
  if (cap <= 0 || !std::isfinite(theta)) return 0;
  int64_t n = 0;
  for (int64_t t = 0; t < L && n < cap; ++t)
    if (scores[t] > (double)theta && !resident[t]) out[n++] = t;
  return n;
}

/* Sparse MLA decode ([REV] "Problem and motivation": MLA attention over the
 * selected tokens).  q [Hq, D], latents [n, D] (n >= 1), in double:
 *   logit_j = scale * sum_d q[d] c_j[d]        (all D dims)
 *   p_j     = exp(logit_j - m) / sum_i exp(logit_i - m),  m = max_j logit_j
 *   out     = sum_j p_j c_j[0 : v_width],      lse = m + log(sum_j exp(logit_j - m))
 * out [Hq, v_width], lse [Hq]. */
void orc_sparse_mla_decode(const double *q, int64_t Hq, const double *c, int64_t n, int64_t D, double scale,
                           int64_t v_width, double *out, double *lse) {
  std::vector<double> logit(n), e(n);
  for (int64_t h = 0; h < Hq; ++h) {
    double m = -kInf;
    for (int64_t j = 0; j < n; ++j) {
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d) dot += q[h * D + d] * c[j * D + d];
      logit[j] = scale * dot;
      if (logit[j] > m) m = logit[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      e[j] = std::exp(logit[j] - m);
      l += e[j];
    }
    for (int64_t v = 0; v < v_width; ++v) out[h * v_width + v] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      const double p = e[j] / l;
      for (int64_t v = 0; v < v_width; ++v) out[h * v_width + v] += p * c[j * D + v];
    }
    lse[h] = m + std::log(l);
  }
}

/* Sparse attention of one KV head with several query heads (N4, reading R26: a GQA
 * layer's KV head is its own unit of selection; its G query heads attend over the
 * tokens selected for it).  q [G, d]; rows [n, 2d] hold each selected token's key
 * (dims 0..d-1) and value (dims d..2d-1), n >= 1; in double:
 *   logit_j = scale * sum_e q[e] key_j[e]
 *   out     = sum_j softmax(logit)_j value_j,   lse = m + log(sum_j exp(logit_j - m))
 * out [G, d], lse [G]. */
void orc_sparse_gqa_decode(const double *q, int64_t G, const double *rows, int64_t n, int64_t d, double scale,
                           double *out, double *lse) {
  const int64_t w = 2 * d;
  std::vector<double> logit(n);
  for (int64_t g = 0; g < G; ++g) {
    double m = -kInf;
    for (int64_t j = 0; j < n; ++j) {
      double dot = 0.0;
      for (int64_t e = 0; e < d; ++e) dot += q[g * d + e] * rows[j * w + e];
      logit[j] = scale * dot;
      m = std::max(m, logit[j]);
    }
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) z += std::exp(logit[j] - m);
    for (int64_t e = 0; e < d; ++e) out[g * d + e] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      const double p = std::exp(logit[j] - m) / z;
      for (int64_t e = 0; e < d; ++e) out[g * d + e] += p * rows[j * w + d + e];
    }
    lse[g] = m + std::log(z);
  }
}

/* Textbook dense attention over a whole cache with a mask (a second, independent
 * formulation used to check orc_sparse_mla_decode): masked logits are -inf. */
void orc_dense_masked_attention(const double *q, int64_t Hq, const double *cache, int64_t N, int64_t D,
                                const uint8_t *mask, double scale, int64_t v_width, double *out) {
  std::vector<double> logit(N);
  for (int64_t h = 0; h < Hq; ++h) {
    double m = -kInf;
    for (int64_t j = 0; j < N; ++j) {
      if (!mask[j]) {
        logit[j] = -kInf;
        continue;
      }
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d) dot += q[h * D + d] * cache[j * D + d];
      logit[j] = scale * dot;
      m = std::max(m, logit[j]);
    }
    double z = 0.0;
    for (int64_t j = 0; j < N; ++j) z += mask[j] ? std::exp(logit[j] - m) : 0.0;
    for (int64_t v = 0; v < v_width; ++v) {
      double acc = 0.0;
      for (int64_t j = 0; j < N; ++j)
        if (mask[j]) acc += std::exp(logit[j] - m) / z * cache[j * D + v];
      out[h * v_width + v] = acc;
    }
  }
}

/* ------------------------------------------------------------------ cache --
 * [REV] "In-graph per-layer cache management".  Slot numbers chosen here (the lowest
 * free slot first) are one valid choice; residency, priorities and the maps'
 * consistency are what a comparison uses. */

static void flag(orc_cache_t *c, int32_t code) {
  if (c->status == kOk) c->status = code;
}

void orc_cache_reset(orc_cache_t *c) {
  for (int64_t h = 0; h < c->n_host; ++h) c->host2gpu[h] = kNotResident;
  for (int64_t g = 0; g < c->n_gpu; ++g) {
    c->gpu2host[g] = kNotResident;
    c->priority[g] = 0;
    c->free_map[g] = 1;
  }
  c->step = 0;
  c->status = kOk;
}

int64_t orc_cache_n_free(const orc_cache_t *c) {
  int64_t n = 0;
  for (int64_t g = 0; g < c->n_gpu; ++g) n += c->free_map[g] ? 1 : 0;
  return n;
}

/* R8: the m resident slots with the smallest (priority, host index) among those
 * with priority < current step; fewer if not enough are eligible.  Returns the
 * count written to out (slots, in that order). */
int64_t orc_cache_lru_victims(const orc_cache_t *c, int64_t m, int64_t *out) {
  if (m <= 0) return 0;
  std::vector<int64_t> elig;
  for (int64_t g = 0; g < c->n_gpu; ++g)
    if (c->gpu2host[g] >= 0 && c->priority[g] < c->step) elig.push_back(g);
  std::sort(elig.begin(), elig.end(), [c](int64_t a, int64_t b) {
    if (c->priority[a] != c->priority[b]) return c->priority[a] < c->priority[b];
    return c->gpu2host[a] < c->gpu2host[b];
  });
  const int64_t n = std::min<int64_t>(m, (int64_t)elig.size());
  for (int64_t i = 0; i < n; ++i) out[i] = elig[i];
  return n;
}

/* Free slots; no data moves back, the host already holds every row ([REV] "In-graph
 * ...": no write-back on eviction).  hosts_out (may be NULL) gets the evicted host
 * indices in slot order. */
void orc_cache_evict(orc_cache_t *c, const int64_t *slots, int64_t n, int64_t *hosts_out) {
  for (int64_t i = 0; i < n; ++i) {
    const int64_t g = slots[i];
    const int64_t h = c->gpu2host[g];
    if (hosts_out) hosts_out[i] = h;
    if (h >= 0) c->host2gpu[h] = kNotResident;
    c->gpu2host[g] = kNotResident;
    c->free_map[g] = 1;
  }
}

/* Give host token h the lowest free slot at or after `from`, stamped with the
 * current step.  Returns the slot, or -1 when none is free. */
static int64_t bind_from(orc_cache_t *c, int64_t h, int64_t from) {
  for (int64_t g = from; g < c->n_gpu; ++g) {
    if (!c->free_map[g]) continue;
    c->free_map[g] = 0;
    c->gpu2host[g] = h;
    c->host2gpu[h] = g;
    c->priority[g] = c->step;
    return g;
  }
  return kNotResident;
}

int64_t orc_cache_bind(orc_cache_t *c, int64_t h) { return bind_from(c, h, 0); }

/* A1, write-back ([REV] "In-graph per-layer cache management": every token's KV is
 * backed up to the host when generated; R10, R16).  Begins step s; for each request
 * in order, its new token (host index host_base[b] + seq_len[b]) takes a free slot if
 * there is one, else evicts the LRU-smallest token with priority < s.  seq_len is
 * incremented in place; new_h gets the new host indices. */
void orc_cache_writeback(orc_cache_t *c, const int64_t *host_base, int64_t *seq_len, int64_t B, int64_t *new_h) {
  c->step += 1;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t h = host_base[b] + seq_len[b];
    new_h[b] = h;
    seq_len[b] += 1;
    if (h < 0 || h >= c->n_host) {
      flag(c, kHostIndex);
      continue;
    }
    const int64_t g = c->host2gpu[h];
    if (g >= 0) {                          /* already resident: refresh its stamp */
      c->priority[g] = c->step;
      continue;
    }
    if (orc_cache_n_free(c) == 0) {
      int64_t v;
      if (orc_cache_lru_victims(c, 1, &v) == 0) {
        flag(c, kPoolExhausted);
        continue;
      }
      orc_cache_evict(c, &v, 1, nullptr);
    }
    bind_from(c, h, 0);
  }
}

/* A6..A10, recall after the exact top-k ([REV] "Decode: ... recall exactly"; "In-graph
 * per-layer cache management": find the selected tokens missing from the map,
 * protect the selection, evict low-priority tokens, allocate, copy from the host).
 *   sel     [sel_off[B]]  selected token indices, request b at [sel_off[b], sel_off[b+1])
 *   staged  [st_off[B]]   tokens prefetched for each request in this step (R9)
 * Order: (1) stamp every resident selected token with the current step (protection,
 * R8); (2) tokens to bind = every staged token, then the misses, each in (b, t)
 * order; (3) evict the LRU-smallest eligible tokens so that enough slots are free;
 * (4) bind (R17 when the pool runs out); (5) report, per selected entry, its host
 * index if resident.
 * Outputs per selected entry: cat (0 hit, 1 prefetched hit, 2 miss) and slot_host
 * (host index, or -1 if it could not be bound).  evicted gets the evicted host
 * indices ascending, n_evicted their count.  Returns the recall's status. */
int32_t orc_cache_recall(orc_cache_t *c, int64_t B, const int64_t *host_base, const int64_t *sel,
                         const int64_t *sel_off, const int64_t *staged, const int64_t *st_off, int8_t *cat,
                         int64_t *slot_host, int64_t *evicted, int64_t *n_evicted) {
  std::vector<std::vector<int64_t>> staged_sorted(B), misses(B);
  for (int64_t b = 0; b < B; ++b) {
    staged_sorted[b].assign(staged + st_off[b], staged + st_off[b + 1]);
    std::sort(staged_sorted[b].begin(), staged_sorted[b].end());
    staged_sorted[b].erase(std::unique(staged_sorted[b].begin(), staged_sorted[b].end()), staged_sorted[b].end());
  }
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t j = sel_off[b]; j < sel_off[b + 1]; ++j) {
      const int64_t t = sel[j];
      const int64_t g = c->host2gpu[host_base[b] + t];
      if (g >= 0) {
        c->priority[g] = c->step;            /* protect: touched in this step */
        cat[j] = 0;
      } else if (std::binary_search(staged_sorted[b].begin(), staged_sorted[b].end(), t)) {
        cat[j] = 1;
      } else {
        cat[j] = 2;
        misses[b].push_back(t);
      }
    }
    std::sort(misses[b].begin(), misses[b].end());
  }
  std::vector<int64_t> to_bind;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t : staged_sorted[b]) to_bind.push_back(host_base[b] + t);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t : misses[b]) to_bind.push_back(host_base[b] + t);
  const int64_t need = (int64_t)to_bind.size() - orc_cache_n_free(c);
  std::vector<int64_t> victims(std::max<int64_t>(need, 0));
  const int64_t nv = orc_cache_lru_victims(c, need, victims.data());
  std::vector<int64_t> hosts(nv);
  orc_cache_evict(c, victims.data(), nv, hosts.data());
  std::sort(hosts.begin(), hosts.end());
  for (int64_t i = 0; i < nv; ++i) evicted[i] = hosts[i];
  *n_evicted = nv;
  int32_t status = kOk;
  if (need > nv) {
    status = kPoolExhausted;
    flag(c, kPoolExhausted);
  }
  /* no slot is freed while binding, so the lowest free slot only moves forward */
  int64_t cursor = 0;
  for (int64_t h : to_bind) {
    const int64_t g = bind_from(c, h, cursor);
    if (g == kNotResident) break;
    cursor = g + 1;
  }
  for (int64_t b = 0; b < B; ++b)
    for (int64_t j = sel_off[b]; j < sel_off[b + 1]; ++j) {
      const int64_t h = host_base[b] + sel[j];
      slot_host[j] = c->host2gpu[h] >= 0 ? h : kNotResident;
    }
  return status;
}

/* Map invariants of [REV] "In-graph per-layer cache management".  Returns 0 when
 * all hold, else the number of the first that fails:
 *   1 host2gpu[gpu2host[g]] == g for every used slot g
 *   2 gpu2host[host2gpu[h]] == h for every resident token h
 *   3 free_map[g] <=> gpu2host[g] == -1
 *   4 resident count == used count <= n_gpu */
int32_t orc_cache_check_invariants(const orc_cache_t *c) {
  int64_t used = 0, res = 0;
  for (int64_t g = 0; g < c->n_gpu; ++g) {
    const int64_t h = c->gpu2host[g];
    if (h >= 0) {
      ++used;
      if (h >= c->n_host || c->host2gpu[h] != g) return 1;
    }
    if ((c->free_map[g] != 0) != (h < 0)) return 3;
  }
  for (int64_t h = 0; h < c->n_host; ++h) {
    const int64_t g = c->host2gpu[h];
    if (g >= 0) {
      ++res;
      if (g >= c->n_gpu || c->gpu2host[g] != h) return 2;
    }
  }
  if (res != used || used > c->n_gpu) return 4;
  return 0;
}

/* One decode step of one layer, A1..A10 in the pages' order ([REV] "Decode: predict
 * the transfer, then recall exactly"): write-back, score every past token, mark
 * above-threshold non-resident tokens for prefetch, exact top-k + EMA, recall.
 * (Attention, A11, is orc_sparse_mla_decode over the selected rows.)
 *   keys[b]     [seq_len[b] + 1, D] indexer keys of request b, this step's new key
 *               included (key_dtype 0 = double, 1 = float)
 *   q_idx [B, H, D], w_idx [B, H], theta_in [B] (the EMA before this step)
 * Outputs: new_h [B]; scores [B, s_stride] float; caps [B]; staged [B, st_stride]
 * with counts staged_n [B]; sel [B, k] with counts sel_n [B]; kth [B]; theta_out [B];
 * per selected entry (row b at b * k) cat and slot_host; evicted [n_gpu] with count
 * n_evicted.  seq_len is incremented in place.  adaptive != 0 takes the caps from
 * R23 with ad_new_rows / ad_pred_err [B] (the previous step's, in) and leaves this
 * step's in them (out).
 * Returns the recall's status, or -1 when a score is not exact in float
 * (bad_req, bad_tok say where; nothing after the scoring has run). */
int32_t orc_decode_layer_step(orc_cache_t *c, int64_t B, const int64_t *host_base, int64_t *seq_len,
                              const void *const *keys, int key_dtype, int64_t H, int64_t D, const double *q_idx,
                              const double *w_idx, const float *theta_in, float *theta_out, int64_t k,
                              int64_t cap_max, int64_t cap_div, float alpha, int prefetch, int64_t *new_h,
                              float *scores, int64_t s_stride, int64_t *caps, int64_t *staged, int64_t *staged_n,
                              int64_t st_stride, int64_t *sel, int64_t *sel_n, float *kth, int8_t *cat,
                              int64_t *slot_host, int64_t *evicted, int64_t *n_evicted, int64_t *bad_req,
                              int64_t *bad_tok, int adaptive, int64_t slack, int64_t *ad_new_rows,
                              float *ad_pred_err) {
  /* A1 */
  orc_cache_writeback(c, host_base, seq_len, B, new_h);
  /* A3 + A4: scores, then the prefetch marks against the threshold before this step */
  std::vector<double> sd;
  std::vector<uint8_t> resident;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t L = seq_len[b];
    sd.assign(L, 0.0);
    orc_indexer_scores(q_idx + b * H * D, w_idx + b * H, H, D, keys[b], key_dtype, L, sd.data());
    float *sb = scores + b * s_stride;
    const int64_t bad = orc_to_f32_exact(sd.data(), L, sb);
    if (bad >= 0) {
      *bad_req = b;
      *bad_tok = bad;
      return -1;
    }
    caps[b] = !prefetch ? 0
              : adaptive ? orc_adaptive_cap(L, cap_max, cap_div, ad_new_rows[b], ad_pred_err[b], slack)
                         : orc_prefetch_cap(L, cap_max, cap_div);
    resident.assign(L, 0);
    for (int64_t t = 0; t < L; ++t) {
      const int64_t h = host_base[b] + t;
      resident[t] = (h >= 0 && h < c->n_host && c->host2gpu[h] >= 0) ? 1 : 0;
    }
    staged_n[b] = orc_prefetch_marks(sd.data(), L, theta_in[b], resident.data(), std::min(caps[b], st_stride),
                                     staged + b * st_stride);
  }
  /* A5: exact top-k and the EMA */
  std::vector<int64_t> sel_off(B + 1, 0), st_off(B + 1, 0), sel_flat, st_flat;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t L = seq_len[b];
    sd.assign(L, 0.0);
    for (int64_t t = 0; t < L; ++t) sd[t] = (double)scores[b * s_stride + t];
    double kv;
    sel_n[b] = orc_topk_select(sd.data(), L, k, sel + b * k, &kv);
    kth[b] = (float)kv;
    theta_out[b] = orc_ema_update(theta_in[b], (float)kv, alpha);
    if (adaptive) ad_pred_err[b] = orc_prediction_error(theta_in[b], (float)kv);
    sel_off[b + 1] = sel_off[b] + sel_n[b];
    st_off[b + 1] = st_off[b] + staged_n[b];
    for (int64_t j = 0; j < sel_n[b]; ++j) sel_flat.push_back(sel[b * k + j]);
    for (int64_t j = 0; j < staged_n[b]; ++j) st_flat.push_back(staged[b * st_stride + j]);
  }
  /* A6..A10 */
  std::vector<int8_t> cat_flat(sel_flat.size());
  std::vector<int64_t> sh_flat(sel_flat.size());
  const int32_t st = orc_cache_recall(c, B, host_base, sel_flat.data(), sel_off.data(), st_flat.data(),
                                      st_off.data(), cat_flat.data(), sh_flat.data(), evicted, n_evicted);
  for (int64_t b = 0; b < B; ++b) {
    int64_t fresh = 0;
    for (int64_t j = 0; j < sel_n[b]; ++j) {
      cat[b * k + j] = cat_flat[sel_off[b] + j];
      slot_host[b * k + j] = sh_flat[sel_off[b] + j];
      fresh += cat[b * k + j] != 0 ? 1 : 0;       /* prefetched hit or miss */
    }
    if (adaptive) ad_new_rows[b] = fresh;
  }
  return st;
}

/* ------------------------------------------------------- block granularity --
 * [REV] critique (adapting the design to block-sparse / GQA models: metadata per
 * block of tokens instead of per token); reading R25. */

/* Block scores: out[j] = max of scores[j*T .. min(L, j*T+T)), j < ceil(L / T). */
int64_t orc_block_scores(const double *scores, int64_t L, int64_t T, double *out) {
  const int64_t nb = (L + T - 1) / T;
  for (int64_t j = 0; j < nb; ++j) {
    double m = -kInf;
    for (int64_t t = j * T; t < std::min(L, j * T + T); ++t) m = std::max(m, scores[t]);
    out[j] = m;
  }
  return nb;
}

/* Write-back in block mode (R25, R16): begins step s.  First every new token that
 * starts a block that is not resident takes a slot for that block, in request order
 * (LRU victims among the slots not touched in this step); then the block that
 * receives each new token (host row host_base[b] + seq_len[b], block that row / T),
 * if resident now, is touched in this step.  A token in the middle of a block that is
 * not resident takes no slot.  seq_len grows in place; new_blk gets the blocks. */
void orc_cache_writeback_blocks(orc_cache_t *c, const int64_t *host_base, int64_t *seq_len, int64_t B, int64_t T,
                                int64_t *new_blk) {
  c->step += 1;
  std::vector<char> ok(B, 0);
  for (int64_t b = 0; b < B; ++b) {
    const int64_t h = host_base[b] + seq_len[b];
    const int64_t hb = h / T;
    new_blk[b] = hb;
    seq_len[b] += 1;
    if (h < 0 || hb >= c->n_host) {
      flag(c, kHostIndex);
      continue;
    }
    ok[b] = 1;
    if (h % T != 0 || c->host2gpu[hb] >= 0) continue;  /* mid-block, or already resident */
    if (orc_cache_n_free(c) == 0) {
      int64_t v;
      if (orc_cache_lru_victims(c, 1, &v) == 0) {
        flag(c, kPoolExhausted);
        continue;
      }
      orc_cache_evict(c, &v, 1, nullptr);
    }
    bind_from(c, hb, 0);
  }
  for (int64_t b = 0; b < B; ++b)                       /* the receiving block is touched */
    if (ok[b] && c->host2gpu[new_blk[b]] >= 0) c->priority[c->host2gpu[new_blk[b]]] = c->step;
}

/* One decode step in block mode (R25): write-back, token scores, block scores, exact
 * top-k/T blocks and the EMA of the k/T-th block score, recall of the missing blocks.
 * Arguments as orc_decode_layer_step with host_base in tokens (a multiple of T per
 * request); outputs: scores [B, s_stride] (tokens), bscores [B, b_stride] and their
 * counts nblk [B], sel [B, kb] (block indices) with counts sel_n, kth (k/T-th block
 * score), theta_out, per selected block cat and slot_host (host block or -1), and the
 * evicted host blocks.  Returns the recall's status, -1 on an inexact score. */
int32_t orc_decode_layer_step_blocks(orc_cache_t *c, int64_t B, const int64_t *host_base, int64_t *seq_len, int64_t T,
                                     const void *const *keys, int key_dtype, int64_t H, int64_t D,
                                     const double *q_idx, const double *w_idx, const float *theta_in,
                                     float *theta_out, int64_t kb, float alpha, int64_t *new_blk, float *scores,
                                     int64_t s_stride, double *bscores, int64_t b_stride, int64_t *nblk,
                                     int64_t *sel, int64_t *sel_n, float *kth, int8_t *cat, int64_t *slot_host,
                                     int64_t *evicted, int64_t *n_evicted, int64_t *bad_req, int64_t *bad_tok) {
  orc_cache_writeback_blocks(c, host_base, seq_len, B, T, new_blk);
  std::vector<double> sd;
  std::vector<int64_t> sel_off(B + 1, 0), sel_flat, base_blk(B);
  for (int64_t b = 0; b < B; ++b) {
    const int64_t L = seq_len[b];
    sd.assign(L, 0.0);
    orc_indexer_scores(q_idx + b * H * D, w_idx + b * H, H, D, keys[b], key_dtype, L, sd.data());
    const int64_t bad = orc_to_f32_exact(sd.data(), L, scores + b * s_stride);
    if (bad >= 0) {
      *bad_req = b;
      *bad_tok = bad;
      return -1;
    }
    nblk[b] = orc_block_scores(sd.data(), L, T, bscores + b * b_stride);
    double kv;
    sel_n[b] = orc_topk_select(bscores + b * b_stride, nblk[b], kb, sel + b * kb, &kv);
    kth[b] = (float)kv;
    theta_out[b] = orc_ema_update(theta_in[b], (float)kv, alpha);
    sel_off[b + 1] = sel_off[b] + sel_n[b];
    for (int64_t j = 0; j < sel_n[b]; ++j) sel_flat.push_back(sel[b * kb + j]);
    base_blk[b] = host_base[b] / T;
  }
  std::vector<int64_t> st_off(B + 1, 0), st_flat(1, 0);
  std::vector<int8_t> cat_flat(sel_flat.size() + 1);
  std::vector<int64_t> sh_flat(sel_flat.size() + 1);
  const int32_t st = orc_cache_recall(c, B, base_blk.data(), sel_flat.data(), sel_off.data(), st_flat.data(),
                                      st_off.data(), cat_flat.data(), sh_flat.data(), evicted, n_evicted);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t j = 0; j < sel_n[b]; ++j) {
      cat[b * kb + j] = cat_flat[sel_off[b] + j];
      slot_host[b * kb + j] = sh_flat[sel_off[b] + j];
    }
  return st;
}

/* ---------------------------------------------------------------- prefill --
 * [REV] "Prefill: overlap recall across query blocks": a 256-bucket coarse histogram
 * picks the strictly-high buckets now and leaves the threshold bucket for later;
 * subtracting the predicted k-th score makes the buckets near the boundary finer.
 * The exact per-query top-k and the recall follow. */

/* Order-preserving 32-bit key of float values from the IEEE-754 bit pattern: larger
 * float, larger key; -0 and +0 share the key of +0. */
void orc_order_key_f32(const float *x, int64_t n, uint32_t *out) {
  for (int64_t i = 0; i < n; ++i) {
    float v = x[i];
    if (v == 0.0f) v = 0.0f;
    uint32_t u;
    std::memcpy(&u, &v, sizeof u);
    out[i] = (u >> 31) ? ~u : (u | 0x80000000u);
  }
}

/* R19: bucket 0..255 of each score, the top byte of the key of score - kth_pred, the
 * difference taken in float.  Parity unpinned (a reading of the pages). */
void orc_prefill_buckets(const float *s, int64_t n, float kth_pred, int32_t *out) {
  for (int64_t i = 0; i < n; ++i) {
    const float d = s[i] - kth_pred;
    uint32_t key;
    orc_order_key_f32(&d, 1, &key);
    out[i] = (int32_t)(key >> 24);
  }
}

void orc_prefill_histogram(const float *s, int64_t n, float kth_pred, int64_t *hist) {
  std::vector<int32_t> bk(n);
  orc_prefill_buckets(s, n, kth_pred, bk.data());
  for (int i = 0; i < 256; ++i) hist[i] = 0;
  for (int64_t i = 0; i < n; ++i) hist[bk[i]] += 1;
}

/* R20: threshold bucket and candidate tokens of one query.  thr = bucket of the k-th
 * largest d (-1 when the query has at most k tokens); cand = ascending token indices
 * in buckets above thr.  Returns the candidate count. */
int64_t orc_prefill_candidates(const float *s, int64_t L, float kth_pred, int64_t k, int64_t *cand,
                               int32_t *thr_out) {
  if (L <= k) {
    *thr_out = -1;
    for (int64_t t = 0; t < L; ++t) cand[t] = t;
    return L;
  }
  std::vector<int32_t> bk(L);
  orc_prefill_buckets(s, L, kth_pred, bk.data());
  int64_t hist[256];
  for (int i = 0; i < 256; ++i) hist[i] = 0;
  for (int64_t t = 0; t < L; ++t) hist[bk[t]] += 1;
  int32_t thr = 0;
  int64_t above = 0;
  for (int bkt = 255; bkt >= 0; --bkt) {        /* count down from the top bucket */
    if (above + hist[bkt] >= k) {
      thr = bkt;
      break;
    }
    above += hist[bkt];
  }
  *thr_out = thr;
  int64_t n = 0;
  for (int64_t t = 0; t < L; ++t)
    if (bk[t] > thr) cand[n++] = t;
  return n;
}

/* R21: union of token lists, ascending.  Returns the count written to out. */
int64_t orc_token_union(const int64_t *tok, int64_t n, int64_t *out) {
  std::vector<int64_t> v(tok, tok + n);
  std::sort(v.begin(), v.end());
  v.erase(std::unique(v.begin(), v.end()), v.end());
  for (size_t i = 0; i < v.size(); ++i) out[i] = v[i];
  return (int64_t)v.size();
}

/* One prefill query block (R18): query j (position pos0 + j) scores keys[0 .. pos0+j]
 * in double, stored as float (exact on the grid); then its histogram, threshold
 * bucket and candidates against kth_pred[j]; then its exact top-k.
 *   q [Q, H, D], w [Q, H], keys [>= pos0 + Q, D] (key_dtype as orc_indexer_scores)
 * Outputs: scores [Q, s_stride] (row j has pos0 + j + 1 valid entries), hist [Q, 256],
 * thr [Q], cand [Q, s_stride] with counts cand_n [Q], sel [Q, k] with counts sel_n [Q],
 * kth [Q].  Returns -1, or (query * 2^32 + token) of the first inexact score. */
int64_t orc_prefill_block(const double *q, const double *w, int64_t Q, int64_t H, int64_t D, const void *keys,
                          int key_dtype, int64_t pos0, const float *kth_pred, int64_t k, float *scores,
                          int64_t s_stride, int64_t *hist, int32_t *thr, int64_t *cand, int64_t *cand_n,
                          int64_t *sel, int64_t *sel_n, float *kth) {
  std::vector<double> sd;
  for (int64_t j = 0; j < Q; ++j) {
    const int64_t L = pos0 + j + 1;
    sd.assign(L, 0.0);
    orc_indexer_scores(q + j * H * D, w + j * H, H, D, keys, key_dtype, L, sd.data());
    float *sj = scores + j * s_stride;
    const int64_t bad = orc_to_f32_exact(sd.data(), L, sj);
    if (bad >= 0) return (j << 32) + bad;
    orc_prefill_histogram(sj, L, kth_pred[j], hist + j * 256);
    cand_n[j] = orc_prefill_candidates(sj, L, kth_pred[j], k, cand + j * s_stride, thr + j);
    double kv;
    sel_n[j] = orc_topk_select(sd.data(), L, k, sel + j * k, &kv);
    kth[j] = (float)kv;
  }
  return -1;
}

}  // extern "C"
