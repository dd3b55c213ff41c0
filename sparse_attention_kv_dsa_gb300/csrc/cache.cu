// Per-layer GPU cache manager of ECHO on sm_103a.
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// section "In-graph per-layer cache management": a preallocated free bitmap,
// eviction priorities, index buffers and a bidirectional host<->GPU map; allocation
// by a parallel scan plus atomic counts; release protects the current selection,
// then frees low-priority slots and updates the maps; no data moves back on
// eviction; recall finds the missing entries from the map, allocates, and a GPU
// kernel reads host memory directly to copy the KV.  Everything here runs on fixed
// grids with device-side counts so a whole step can be captured in one CUDA Graph.
//
// Kernels
//   reset_kernel    empty cache
//   reserve_kernel  per-request prefetch budget (A2)
//   mgr_kernel      one cooperative launch over the whole GPU (one CTA per SM) per
//                   call, in phases separated by bounded grid barriers:
//                   recall only: protect hits and list misses (A6);
//                   LRU victim selection: every CTA keeps the victim keys of its
//                   slice of slots in shared memory; an MSB-first radix select
//                   builds each digit's histogram from per-CTA shared histograms
//                   added into a global one, and every CTA derives the same digit
//                   from it (no broadcast step); only the bits below the largest
//                   key's top bit are visited;
//                   eviction and binding: victims ranked by one global atomic per
//                   warp and rebound at once to the tokens that need a slot; free
//                   slots found by a warp-ballot scan of the free bitmap with one
//                   atomic per warp (A7 + A8);
//                   then the data: write-back of the new token (A1), or the recall's
//                   zero-copy host reads and staged rows into slots plus the slot
//                   translation (A9 + A10).
//                   Modes: write-back, recall, alloc, evict.  A recall also ranks the
//                   next write-back's victims (the pending list).
//   wb_fast_kernel  one CTA: the write-back from the pending list, launched before the
//                   cooperative write-back, which then returns at once if it was done

#include <algorithm>

#include "common.cuh"

namespace echo {

// ------------------------------------------------------------------ reset --
__global__ void reset_kernel(echo_cache_layer_t L) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < L.n_host) L.host2gpu[i] = -1;
  if (i < L.n_gpu) {
    L.gpu2host[i] = -1;
    L.priority[i] = 0;
    L.index_buf[i] = 0;
    L.free_map[i] = 1;
  }
  if (i < ECHO_NUM_COUNTERS) L.counters[i] = (i == ECHO_CTR_N_FREE) ? L.n_gpu : 0;
}

// ---------------------------------------------------------------- reserve --
// Prefetch budget of request b for a step whose context length is len: the context
// rule min(cap_max, ceil(len / cap_div)), or cap_max when cap_div is 0; with the
// adaptive state, at most the last step's transfer grown by the prediction error
// plus the slack.  Clears the transfer count for this step's recall to fill; call it
// once per request and step.
__device__ __forceinline__ int budget_cap(const echo_cache_layer_t &L, int b, int32_t len, int cap_max,
                                          int cap_div) {
  int c = 0;
  if (cap_max > 0) c = max(cap_div > 0 ? min(cap_max, (len + cap_div - 1) / cap_div) : cap_max, 0);
  if (L.pf_new_rows) {
    const int32_t u = L.pf_new_rows[b];
    if (u >= 0 && c > 0) {
      const float grow = __fadd_rn(1.0f, L.pf_pred_err[b]);
      const float want = fminf(__fmul_rn(grow, (float)u), 1.0e9f);
      c = min(c, max((int)ceilf(want) + L.cap_slack, 0));
    }
    L.pf_new_rows[b] = 0;
  }
  return c;
}

__global__ void reserve_kernel(echo_cache_layer_t L, const int32_t *seq_len, int B, int cap_max, int cap_div,
                               int32_t *cap, int32_t *pf_count) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    cap[b] = budget_cap(L, b, seq_len[b], cap_max, cap_div);
    pf_count[b] = 0;
  }
}

// ---------------------------------------------------------------- manager --
enum { MODE_WRITEBACK = 0, MODE_RECALL = 1, MODE_ALLOC = 2, MODE_EVICT = 3 };

// Counter words 16..31 belong to the manager (zero between calls, except the barrier
// count, which only grows):
enum {
  MG_BAR = 16,         // words 16-17: grid barrier arrivals (uint64, a multiple of the grid between barriers)
  MG_ABORT = 18,       // a barrier wait gave up: every CTA leaves
  MG_FAST = 19,        // the write-back was done by wb_fast_kernel (set by it before every
                       // cooperative write-back it precedes)
  MG_PRE_N = 20,       // entries in the pending victim list (0 = none)
  MG_PRE_STEP = 21,    // step of the recall that wrote the list
  MG_VCUR = 22,        // victim rank cursor
  MG_SCUR = 23,        // free-slot scan cursor
  MG_SMALL_HIST = 24,  // words 24..29: the histograms of pools with fewer than 6 slots
  MG_PCUR = 30,        // pending-list cursor
};

// Pending victims.  A write-back evicts the B least recently used slots, and between a
// recall and the next step's write-back no slot changes: so the recall's LRU selection
// can also rank the next B victims (a second target rank in the same radix passes)
// and leave them, with their keys, at the end of index_buf.  The write-back then binds
// them in one CTA (wb_fast_kernel) after checking that every entry still holds its key,
// and its cooperative launch returns at once; any other case takes the full path.
// Pools of at least PRE_POOL slots keep this layout of index_buf in every mode:
//   [0, 12288)               two sets of three 2048-bin histograms (6 x 2048 words)
//   [12288, +MAXB)           the recall's miss counters
//   [n_gpu - 3 PRE_MAX, n_gpu)  pending list: slot, key low word, key high word
constexpr int PRE_MAX = 256;    // requests per recall that leave a list

struct ManageParams {
  echo_cache_layer_t L;
  int mode;
  int dbits;              // radix digit width
  uint32_t *hist;         // 3 global histograms of 2^dbits words: index_buf, or counter words 24..29
                          // for pools too small to hold them
  int32_t *miss_cnt;      // per-request miss counters (zero between calls) after the histograms in
                          // index_buf, or null: n_miss is zeroed and a grid barrier follows
  int cached;             // victim keys fit in shared memory
  // write-back
  const void *new_kv;
  const void *new_ik;
  void *idx_k;
  int D, Lmax, ik_dtype;
  const int32_t *host_base;
  int32_t *seq_len;
  int B;
  // recall
  const int32_t *sel;
  int k;
  const int32_t *pf_list;
  const int32_t *pf_count;
  int cap_max;
  const void *stage_kv;
  int32_t *miss_list;
  int32_t *n_miss;
  int32_t *slot_idx;
  // alloc
  const int32_t *host_idx;
  const int32_t *n_ptr;
  int n_max;
  int32_t *out_slot;
  // evict
  const int32_t *n_needed;
  // write-back followed by the prefetch budget of the step (echo_cache_reserve's rule)
  int32_t *rs_cap;
  int32_t *rs_pf_count;
  int rs_cap_max, rs_cap_div;
  // pending victims (pools of at least PRE_POOL slots)
  uint32_t *hist2;        // second histogram set (recall), or null
  int32_t *pend;          // pending list: slot[PRE_MAX], key low[PRE_MAX], key high[PRE_MAX]
  int pre_n;              // recall: extra victims to rank for the next write-back (0 = none)
  int fast_checked;       // write-back: wb_fast_kernel ran first; return if it did the work
};

constexpr int MG_THREADS = 512;
constexpr int MG_WARPS = MG_THREADS / 32;
constexpr int MG_MAXBITS = 11;                  // 2048-bin digits at most
constexpr int MG_BPT = (1 << MG_MAXBITS) / MG_THREADS;   // bins per thread in the digit search
constexpr int MAXB = 1024;                      // requests per call handled by the manager
constexpr size_t MG_KEY_SMEM = 192 * 1024;      // victim keys cached per CTA (bytes)
constexpr int PRE_POOL = 6 * (1 << MG_MAXBITS) + MAXB + 3 * PRE_MAX;
static_assert(PRE_POOL == ECHO_PENDING_LIST_MIN_SLOTS, "index_buf layout and the header agree");

struct MgShared {
  uint32_t hist[1 << MG_MAXBITS];
  int32_t pre_a[MAXB + 1];             // prefixes of the token lists
  int32_t pre_b[MAXB + 1];
  uint32_t warp_sums[32];
  uint64_t warp_sums2[32];             // two packed counts per warp (digit searches)
  uint32_t wcnt[MG_WARPS];             // per-warp counts (block reductions, victim ranks)
  uint32_t wcnt1[MG_WARPS];            // per-warp pending-list counts
  int64_t tok0[MAXB];                  // per request: host index of token 0 (write-back: of the new token)
  uint32_t hist1[1 << MG_MAXBITS];     // second target's histogram, once its prefix differs
  uint32_t res[2];                     // [0] chosen digit, [1] count above it
  uint32_t res1[2];                    // the same for the second target
  uint32_t base;                       // this CTA's first rank from a global cursor
  uint32_t base1;                      // its first pending-list position
};

__device__ __forceinline__ int bitlen_u64(uint64_t x) { return x ? 64 - __clzll((long long)x) : 0; }

// Reads of words that other CTAs of the same launch write go around L1.
__device__ __forceinline__ int32_t ldcg(const int32_t *p) { return __ldcg(p); }

// Grid-wide barrier of a cooperative launch with a bounded wait.  Arrivals count up
// a 64-bit word by one per CTA; a barrier is complete when it reaches the next
// multiple of the grid size.  A CTA that has waited ~1 s sets TIMEOUT and the abort
// word; every CTA then leaves the kernel.  All CTAs must call it the same number of
// times.  Returns false on abort.
__device__ __noinline__ bool grid_sync(int32_t *ctr) {
  __shared__ int32_t gs_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long *cnt = reinterpret_cast<unsigned long long *>(ctr + MG_BAR);
    unsigned long long old, cur;
    asm volatile("fence.acq_rel.gpu;\n\tatom.relaxed.gpu.global.add.u64 %0, [%1], 1;" : "=l"(old) : "l"(cnt) : "memory");
    const unsigned long long target = (old / gridDim.x + 1) * gridDim.x;
    int ok = 1, spins = 0;
    uint64_t t0 = 0;
    while (true) {
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(cur) : "l"(cnt) : "memory");
      if (cur >= target) break;
      if (++spins == 256) {
        spins = 0;
        if (*reinterpret_cast<volatile int32_t *>(ctr + MG_ABORT)) { ok = 0; break; }
        if (!t0) {
          t0 = global_ns();
        } else if (global_ns() - t0 > kWaitLimitNs) {
          set_status(ctr, ECHO_ERR_TIMEOUT);
          atomicExch(ctr + MG_ABORT, 1);
          ok = 0;
          break;
        }
      }
    }
    gs_ok = ok;
  }
  __syncthreads();
  return gs_ok != 0;
}

// Inclusive scan over the CTA of two counts packed in 64 bits (the low count's block
// total stays below 2^32, so nothing carries into the high half).
__device__ __forceinline__ uint64_t block_incl_scan2(uint64_t v, uint64_t *warp_sums, uint64_t *total) {
  const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= (uint32_t)o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    uint64_t w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= (uint32_t)o) w += n;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  if (wid > 0) v += warp_sums[wid - 1];
  *total = warp_sums[nw - 1];
  __syncthreads();
  return v;
}

// Sum over the CTA (every thread gets it); ends with a barrier.
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t *wcnt) {
  v = __reduce_add_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) wcnt[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int w = 0; w < MG_WARPS; ++w) t += wcnt[w];
  __syncthreads();
  return t;
}

// Victim key of a slot: larger key = smaller (priority, host index) = evicted first;
// 0 = not evictable (free, or touched in the current step).
__device__ __forceinline__ uint64_t victim_key(int32_t h, int32_t p, int32_t step, int hbits, uint64_t hmax) {
  if (h < 0 || p >= step || p < 0) return 0;
  return (((uint64_t)(int64_t)(step - 1 - p) << hbits) | (hmax - (uint64_t)h)) + 1;
}

__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t *warp_sums, uint32_t *total) {
  const uint32_t lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= (uint32_t)o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= (uint32_t)o) w += n;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  if (wid > 0) v += warp_sums[wid - 1];
  *total = warp_sums[nw - 1];
  __syncthreads();
  return v;
}

// Tokens per host index / slot: 1, or T on a layer with block granularity.
__device__ __forceinline__ int blk_tokens(const echo_cache_layer_t &L) {
  return L.block_tokens > 1 ? L.block_tokens : 1;
}

// Does the new token at host row h need a slot of its own?  Per token: when it is not
// resident; in blocks: when it starts its block and the block is not resident.
__device__ __forceinline__ bool wb_needs_slot(const echo_cache_layer_t &L, int64_t h) {
  const int T = blk_tokens(L);
  return (h % T) == 0 && ldcg(L.host2gpu + h / T) < 0;
}

// Write-back of request b's new token by one warp (A1): its host pool row, its GPU slot
// row if it has a slot (its binding is visible), its indexer key; the prefetch budget
// of the step when the call carries one; the request's length grows by one.  In block
// mode the GPU row is the token's row in its block's slot.
__device__ __forceinline__ void writeback_row(const ManageParams &P, int b, int lane, int32_t step) {
  const echo_cache_layer_t &L = P.L;
  int32_t *ctr = L.counters;
  const int esz = L.kv_dtype == ECHO_F32 ? 4 : 2;
  const int64_t rb = (int64_t)kv_row_elems(L) * esz;   // bytes of one token row
  const int chunks = (int)(rb / 16);                    // 72 (bf16 latent) or 144 (f32)
  const int32_t l = P.seq_len[b];
  const int T = blk_tokens(L);
  const int64_t h = (int64_t)P.host_base[b] + l;
  const bool bad_h = h < 0 || h >= (int64_t)L.n_host * T, bad_l = l >= P.Lmax;
  if (P.rs_cap && lane == 0) {                           // budget from the length after this write-back
    const int32_t len = (bad_h || bad_l) ? l : l + 1;
    P.rs_cap[b] = budget_cap(L, b, len, P.rs_cap_max, P.rs_cap_div);
    P.rs_pf_count[b] = 0;
  }
  if (bad_h) { if (lane == 0) set_status(ctr, ECHO_ERR_HOST_INDEX); return; }
  if (bad_l) { if (lane == 0) set_status(ctr, ECHO_ERR_INVALID_ARG); return; }
  const int32_t g = __ldcg(L.host2gpu + h / T);
  const uint4 *src = reinterpret_cast<const uint4 *>((const char *)P.new_kv + (int64_t)b * rb);
  uint4 *hdst = reinterpret_cast<uint4 *>((char *)L.host_kv + h * rb);
  uint4 *gdst = g >= 0 ? reinterpret_cast<uint4 *>((char *)L.gpu_kv + ((int64_t)g * T + h % T) * rb) : nullptr;
  for (int c = lane; c < chunks; c += 32) {
    const uint4 v = src[c];
    hdst[c] = v;
    if (gdst) gdst[c] = v;
  }
  if (g >= 0 && lane == 0) L.priority[g] = step;         // refresh an already resident token
  if (g < 0 && (h % T) == 0 && lane == 0) set_status(ctr, ECHO_ERR_POOL_EXHAUSTED);
  const int kesz = P.ik_dtype == ECHO_F32 ? 4 : 1;
  const char *ks = (const char *)P.new_ik + (int64_t)b * P.D * kesz;
  char *kd = (char *)P.idx_k + ((int64_t)b * P.Lmax + l) * P.D * kesz;
  for (int c = lane; c < P.D * kesz / 4; c += 32)
    reinterpret_cast<uint32_t *>(kd)[c] = reinterpret_cast<const uint32_t *>(ks)[c];
  __syncwarp();
  if (lane == 0) P.seq_len[b] = l + 1;
}

__global__ void __launch_bounds__(MG_THREADS, 1) mgr_kernel(const __grid_constant__ ManageParams P) {
  extern __shared__ __align__(16) unsigned char dsm[];
  MgShared &S = *reinterpret_cast<MgShared *>(dsm);
  uint64_t *keys = reinterpret_cast<uint64_t *>(dsm + ((sizeof(MgShared) + 15) & ~size_t(15)));
  const echo_cache_layer_t &L = P.L;
  int32_t *ctr = L.counters;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t gtid = blockIdx.x * (int64_t)MG_THREADS + tid;
  const int64_t gthreads = (int64_t)gridDim.x * MG_THREADS;
  const int64_t gwarp = gtid >> 5, gwarps = gthreads >> 5;
  // a write-back that wb_fast_kernel completed (the word is set before this launch)
  if (P.mode == MODE_WRITEBACK && P.fast_checked && ldcg(ctr + MG_FAST) != 0) return;

  const int32_t step0 = ldcg(ctr + ECHO_CTR_STEP);
  const int32_t step = P.mode == MODE_WRITEBACK ? step0 + 1 : step0;
  const int32_t n_free0 = ldcg(ctr + ECHO_CTR_N_FREE);

  // ---- recall: protect every selected resident token, list the misses (A6) ----
  // Miss positions come from per-request counters that are zero on entry (the
  // manager's scratch), or from n_miss zeroed behind a grid barrier.
  int32_t *mcnt = P.miss_cnt ? P.miss_cnt : P.n_miss;
  if (P.mode == MODE_RECALL) {
    if (!P.miss_cnt) {
      if (blockIdx.x == 0)
        for (int b = tid; b < P.B; b += MG_THREADS) P.n_miss[b] = 0;
      if (!grid_sync(ctr)) return;
    }
    uint32_t hit = 0, staged = 0, miss = 0;
    const int64_t nsel = (int64_t)P.B * P.k;
    for (int64_t i = gtid; i < nsel; i += gthreads) {
      const int b = (int)(i / P.k);
      const int32_t t = P.sel[i];
      if (t < 0) continue;
      const int64_t h = (int64_t)P.host_base[b] + t;
      if (h >= L.n_host) {
        set_status(ctr, ECHO_ERR_HOST_INDEX);
        continue;
      }
      const int32_t g = ldcg(L.host2gpu + h);
      if (g >= 0) {
        L.priority[g] = step;                            // protect the selection
        ++hit;
      } else if (g <= -2) {
        ++staged;
        if (L.pf_new_rows) atomicAdd(L.pf_new_rows + b, 1);   // this step's transfer (adaptive cap)
      } else {
        const int32_t pos = atomicAdd(mcnt + b, 1);
        P.miss_list[(int64_t)b * P.k + pos] = t;
        ++miss;
        if (L.pf_new_rows) atomicAdd(L.pf_new_rows + b, 1);
      }
    }
    hit = block_sum(hit, S.wcnt);
    staged = block_sum(staged, S.wcnt);
    miss = block_sum(miss, S.wcnt);
    if (tid == 0) {
      if (hit) atomicAdd(ctr + ECHO_CTR_HITS, (int)hit);
      if (staged) atomicAdd(ctr + ECHO_CTR_STAGED_HITS, (int)staged);
      if (miss) atomicAdd(ctr + ECHO_CTR_MISSES, (int)miss);
    }
    if (!grid_sync(ctr)) return;
    if (P.miss_cnt && blockIdx.x == 0)
      for (int b = tid; b < P.B; b += MG_THREADS) P.n_miss[b] = ldcg(P.miss_cnt + b);
  }

  // ---- this CTA's slice of slots; its first key vectors are loaded now, so the
  // loads overlap the list prefixes below (used only if victims are needed) ----
  const int per = ((L.n_gpu + (int)gridDim.x - 1) / (int)gridDim.x + 3) & ~3;   // 16-byte aligned starts
  const int g0 = min(L.n_gpu, (int)blockIdx.x * per), g1 = min(L.n_gpu, g0 + per);
  const int nloc = g1 - g0;
  const bool cached = P.cached != 0;
  const int n4 = nloc >> 2;
  const int4 *g2h4 = reinterpret_cast<const int4 *>(L.gpu2host + g0);
  const int4 *pr4 = reinterpret_cast<const int4 *>(L.priority + g0);
  int4 hv0 = make_int4(-1, -1, -1, -1), pv0 = make_int4(0, 0, 0, 0);
  if (cached && P.mode != MODE_ALLOC && tid < n4) {
    hv0 = __ldcg(g2h4 + tid);
    pv0 = __ldcg(pr4 + tid);
  }

  // ---- the tokens that need a slot: list A (+ list B), same in every CTA ----
  // write-back: A = new tokens not yet resident; recall: A = staged rows,
  // B = misses; alloc: A = host_idx[0..n).
  if (P.mode == MODE_WRITEBACK) {
    block_prefix(P.B, [&](int b) {
      const int32_t l = P.seq_len[b];
      const int64_t h = (int64_t)P.host_base[b] + l;
      const bool ok = h >= 0 && h < (int64_t)L.n_host * blk_tokens(L) && l < P.Lmax;
      return (ok && wb_needs_slot(L, h)) ? 1 : 0;
    }, S.pre_a);
  } else if (P.mode == MODE_RECALL) {
    const int32_t *pfc = P.pf_count;
    const int cm = P.cap_max;
    block_prefix(P.B, [&](int b) { return pfc ? min(max(pfc[b], 0), cm) : 0; }, S.pre_a);
    block_prefix(P.B, [&](int b) { return (int)ldcg(mcnt + b); }, S.pre_b);
  }
  if (P.mode == MODE_WRITEBACK || P.mode == MODE_RECALL)
    for (int b = tid; b < P.B; b += MG_THREADS)   // write-back: host index of the new token's slot owner
      S.tok0[b] = P.mode == MODE_WRITEBACK ? ((int64_t)P.host_base[b] + P.seq_len[b]) / blk_tokens(L)
                                           : (int64_t)P.host_base[b];
  __syncthreads();
  int nA = 0, nB = 0;
  if (P.mode == MODE_WRITEBACK) nA = S.pre_a[P.B];
  if (P.mode == MODE_RECALL) { nA = S.pre_a[P.B]; nB = S.pre_b[P.B]; }
  if (P.mode == MODE_ALLOC) nA = min(max(*P.n_ptr, 0), P.n_max);
  const int n_bind = (P.mode == MODE_EVICT) ? 0 : nA + nB;
  int m_req = 0;                                         // victims wanted
  if (P.mode == MODE_WRITEBACK || P.mode == MODE_RECALL) m_req = max(0, n_bind - n_free0);
  if (P.mode == MODE_EVICT) m_req = max(0, *P.n_needed - n_free0);
  // tokens of ranks [0, n_scan) go to slots that were already free (bitmap scan);
  // tokens of ranks [n_scan, n_bind) go straight to this call's victims
  const int n_scan = min(max((int)n_free0, 0), n_bind);
  // the write-back's list reads host2gpu, which bindings change: no CTA may bind
  // before every CTA has its list (with eviction the barrier after the keys does it)
  if (P.mode == MODE_WRITEBACK && m_req == 0)
    if (!grid_sync(ctr)) return;

  // host index of the token of rank r (and its request)
  auto token_of = [&](uint32_t r, int *req) -> int64_t {
    if (P.mode == MODE_WRITEBACK) {
      int b = 0;                                   // rank r -> request (B is small)
      while (b + 1 < P.B && S.pre_a[b + 1] <= (int)r) ++b;
      *req = b;
      return S.tok0[b];
    } else if (P.mode == MODE_RECALL) {
      const int32_t *pre = (int)r < nA ? S.pre_a : S.pre_b;
      const int rr = (int)r < nA ? (int)r : (int)r - nA;
      int lo = 0, hi = P.B - 1;                    // last b with pre[b] <= rr
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= rr) lo = mid; else hi = mid - 1;
      }
      const int b = lo, ii = rr - pre[b];
      const int32_t t = (int)r < nA ? P.pf_list[(int64_t)b * P.cap_max + ii] : ldcg(P.miss_list + (int64_t)b * P.k + ii);
      *req = b;
      return S.tok0[b] + t;
    }
    *req = 0;
    return P.host_idx[r];
  };
  // bind the token of rank r to slot g (a victim, or a slot taken from the bitmap)
  auto bind = [&](int g, uint32_t r) {
    int b = 0;
    const int64_t h = token_of(r, &b);
    if (h >= 0 && h < L.n_host) {
      L.free_map[g] = 0;
      L.gpu2host[g] = (int32_t)h;
      L.host2gpu[h] = g;
      L.priority[g] = step;
      if (P.mode == MODE_ALLOC && P.out_slot) P.out_slot[r] = g;
    } else {
      L.gpu2host[g] = -1;
      L.free_map[g] = 1;
      set_status(ctr, ECHO_ERR_HOST_INDEX);
      if (P.mode == MODE_ALLOC && P.out_slot) P.out_slot[r] = -1;
    }
  };

  const int hbits = bitlen_u64((uint64_t)max(L.n_host - 1, 1));
  const uint64_t hmax = (1ull << hbits) - 1;
  auto key_at = [&](int i) -> uint64_t {        // i: index within the slice
    return cached ? keys[i] : victim_key(ldcg(L.gpu2host + g0 + i), ldcg(L.priority + g0 + i), step, hbits, hmax);
  };

  uint32_t m_eff = 0;
  bool two = false;                                       // a pending list is ranked (uniform)
  uint64_t prefix1 = 0;                                   // its last key
  if (m_req > 0) {                                        // uniform across the grid
    // keys of the slice (4 slots per thread and iteration)
    if (cached) {
      for (int j = tid; j < n4; j += MG_THREADS) {
        const int4 hv = j == tid ? hv0 : __ldcg(g2h4 + j), pv = j == tid ? pv0 : __ldcg(pr4 + j);
        keys[4 * j] = victim_key(hv.x, pv.x, step, hbits, hmax);
        keys[4 * j + 1] = victim_key(hv.y, pv.y, step, hbits, hmax);
        keys[4 * j + 2] = victim_key(hv.z, pv.z, step, hbits, hmax);
        keys[4 * j + 3] = victim_key(hv.w, pv.w, step, hbits, hmax);
      }
      for (int i = 4 * n4 + tid; i < nloc; i += MG_THREADS)
        keys[i] = victim_key(ldcg(L.gpu2host + g0 + i), ldcg(L.priority + g0 + i), step, hbits, hmax);
      __syncthreads();
    }
    // MSB-first radix select of the m_eff-th largest key (keys are unique) over the
    // bitlen(step) + hbits + 1 bits a key can have.  The first digit's histogram
    // also counts the evictable slots, which bounds m_eff.  A recall that leaves a
    // pending list selects a second rank, m_eff + pre_n, in the same passes: while
    // the two prefixes agree one histogram serves both, after that each has its own.
    uint64_t prefix = 0;
    uint32_t above = 0, above1 = 0, tgt1 = 0;
    int left = bitlen_u64((uint64_t)max(step, 0)) + hbits + 1, pass = 0;
    const int nb_all = 1 << P.dbits;
    while (left > 0) {
      const int w = min(P.dbits, left), shift = left - w, nbins = 1 << w;
      const bool split = two && prefix1 != prefix;       // the second target needs its own counts
      uint32_t *gh = P.hist + (pass % 3) * nb_all;
      uint32_t *gh1 = split ? P.hist2 + (pass % 3) * nb_all : gh;
      for (int i = tid; i < nbins; i += MG_THREADS) {
        S.hist[i] = 0;
        if (split) S.hist1[i] = 0;
      }
      __syncthreads();
      const uint64_t hi_mask = (shift + w >= 64) ? 0ull : (~0ull << (shift + w));
      for (int base = 0; base < nloc; base += MG_THREADS) {   // uniform trip count per warp
        const int i = base + tid;
        const uint64_t kk = i < nloc ? key_at(i) : 0;
        const uint32_t dg = (uint32_t)((kk >> shift) & (uint64_t)(nbins - 1));
        hist_add_warp(S.hist, kk != 0 && (kk & hi_mask) == (prefix & hi_mask), dg);
        if (split) hist_add_warp(S.hist1, kk != 0 && (kk & hi_mask) == (prefix1 & hi_mask), dg);
      }
      __syncthreads();
      for (int i = tid; i < nbins; i += MG_THREADS) {
        if (S.hist[i]) atomicAdd(gh + i, S.hist[i]);
        if (split && S.hist1[i]) atomicAdd(gh1 + i, S.hist1[i]);
      }
      if (!grid_sync(ctr)) return;
      // the histograms of two passes ago were read by every CTA before this barrier:
      // clear them for the pass after next
      for (int64_t i = gtid; i < nb_all; i += gthreads) {
        P.hist[((pass + 2) % 3) * nb_all + i] = 0;
        if (P.hist2) P.hist2[((pass + 2) % 3) * nb_all + i] = 0;
      }
      // the digits from the global counts: this thread's MG_BPT consecutive bins of
      // each histogram (both loaded before either is used), one block scan of both,
      // and the bin where the count from the top reaches the target
      uint32_t cb[MG_BPT], cb1[MG_BPT], mine = 0, mine1 = 0;
#pragma unroll
      for (int j = 0; j < MG_BPT; ++j) {
        const int d = MG_BPT * tid + j;
        cb[j] = d < nbins ? (uint32_t)__ldcg(reinterpret_cast<const int32_t *>(gh + d)) : 0u;
        cb1[j] = (split && d < nbins) ? (uint32_t)__ldcg(reinterpret_cast<const int32_t *>(gh1 + d)) : 0u;
      }
#pragma unroll
      for (int j = 0; j < MG_BPT; ++j) {
        mine += cb[j];
        mine1 += cb1[j];
      }
      uint64_t tot2;
      const uint64_t incl2 = block_incl_scan2(((uint64_t)mine1 << 32) | mine, S.warp_sums2, &tot2);
      const uint32_t tot = (uint32_t)tot2, incl = (uint32_t)incl2;
      if (pass == 0) {                                   // tot = evictable slots
        m_eff = min((uint32_t)m_req, tot);
        if (blockIdx.x == 0 && tid == 0 && m_eff < (uint32_t)m_req) set_status(ctr, ECHO_ERR_POOL_EXHAUSTED);
        if (m_eff == 0) break;                           // uniform: every CTA read the same counts
        two = P.pre_n > 0 && m_eff == (uint32_t)m_req && m_eff + (uint32_t)P.pre_n <= tot;
        tgt1 = m_eff + (uint32_t)P.pre_n;
      }
      auto search = [&](const uint32_t (&c)[MG_BPT], uint32_t inc, uint32_t tt, uint32_t need, uint32_t *res) {
        uint32_t sfx = tt - inc;                         // keys in bins above mine
#pragma unroll
        for (int j = MG_BPT - 1; j >= 0; --j) {          // my bins, from the top
          if (sfx < need && need <= sfx + c[j]) { res[0] = MG_BPT * tid + j; res[1] = sfx; }
          sfx += c[j];
        }
      };
      search(cb, incl, tot, m_eff - above, S.res);
      if (two) {
        if (split) search(cb1, (uint32_t)(incl2 >> 32), (uint32_t)(tot2 >> 32), tgt1 - above1, S.res1);
        else search(cb, incl, tot, tgt1 - above1, S.res1);
      }
      __syncthreads();
      prefix |= (uint64_t)S.res[0] << shift;
      above += S.res[1];
      if (two) {
        prefix1 |= (uint64_t)S.res1[0] << shift;
        above1 += S.res1[1];
      }
      left = shift;
      ++pass;
      __syncthreads();
    }
    if (m_eff > 0) {
      const uint64_t kstar = prefix;
      // evict every key >= kstar (exactly m_eff tokens).  The CTA counts its victims,
      // takes a block of ranks with one atomic, and victim v is rebound at once to
      // the token of rank n_scan + v, or freed if none is left (evict mode).  With a
      // pending list, keys in [prefix1, kstar) (exactly pre_n of them) are listed the
      // same way.  Each slot's key is read before its own lane changes the slot.
      uint32_t nv = 0, np = 0;
      for (int base = 0; base < nloc; base += MG_THREADS) {
        const int i = base + tid;
        const uint64_t kk = i < nloc ? key_at(i) : 0;
        nv += __popc(__ballot_sync(0xffffffffu, kk != 0 && kk >= kstar));
        np += __popc(__ballot_sync(0xffffffffu, two && kk != 0 && kk >= prefix1 && kk < kstar));
      }
      if (lane == 0) {                                   // per-warp counts
        S.wcnt[tid >> 5] = nv;
        S.wcnt1[tid >> 5] = np;
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t t = 0, t1 = 0;
        for (int w = 0; w < MG_WARPS; ++w) {
          const uint32_t x = S.wcnt[w], x1 = S.wcnt1[w];
          S.wcnt[w] = t;
          S.wcnt1[w] = t1;
          t += x;
          t1 += x1;
        }
        S.base = t ? atomicAdd(reinterpret_cast<unsigned int *>(ctr + MG_VCUR), t) : 0u;
        S.base1 = t1 ? atomicAdd(reinterpret_cast<unsigned int *>(ctr + MG_PCUR), t1) : 0u;
      }
      __syncthreads();
      uint32_t rank = S.base + S.wcnt[tid >> 5], pos = S.base1 + S.wcnt1[tid >> 5];
      for (int base = 0; base < nloc; base += MG_THREADS) {
        const int i = base + tid;
        const uint64_t kk = i < nloc ? key_at(i) : 0;
        const bool isv = kk != 0 && kk >= kstar;
        const bool isp = two && kk != 0 && kk >= prefix1 && kk < kstar;
        const uint32_t bal = __ballot_sync(0xffffffffu, isv);
        const uint32_t balp = __ballot_sync(0xffffffffu, isp);
        if (isv) {
          const int g = g0 + i;
          const int64_t h_old = cached ? (int64_t)(hmax - ((kk - 1) & hmax)) : (int64_t)ldcg(L.gpu2host + g);
          L.host2gpu[h_old] = -1;
          const uint32_t r = (uint32_t)n_scan + rank + __popc(bal & lanemask_lt());
          if (r < (uint32_t)n_bind) {
            bind(g, r);
          } else {
            L.gpu2host[g] = -1;
            L.free_map[g] = 1;
          }
        }
        if (isp) {
          const uint32_t q = pos + __popc(balp & lanemask_lt());
          if (q < (uint32_t)P.pre_n) {
            P.pend[q] = g0 + i;
            P.pend[PRE_MAX + q] = (int32_t)(uint32_t)kk;
            P.pend[2 * PRE_MAX + q] = (int32_t)(uint32_t)(kk >> 32);
          }
        }
        rank += __popc(bal);
        pos += __popc(balp);
      }
      __syncthreads();
    }
  }

  // ---- slots that were already free: warp-ballot scan of this CTA's slice of the
  // bitmap; the CTA takes a block of ranks with one atomic; ranks [0, n_scan) bind ----
  if (n_scan > 0) {
    uint32_t nf = 0;
    for (int base = 0; base < nloc; base += MG_THREADS) {
      const int i = base + tid;
      nf += __popc(__ballot_sync(0xffffffffu, i < nloc && __ldcg(L.free_map + g0 + i) != 0));
    }
    if (lane == 0) S.wcnt[tid >> 5] = nf;
    __syncthreads();
    if (tid == 0) {
      uint32_t t = 0;
      for (int w = 0; w < MG_WARPS; ++w) { const uint32_t x = S.wcnt[w]; S.wcnt[w] = t; t += x; }
      S.base = t ? atomicAdd(reinterpret_cast<unsigned int *>(ctr + MG_SCUR), t) : 0u;
    }
    __syncthreads();
    uint32_t rank = S.base + S.wcnt[tid >> 5];
    for (int base = 0; base < nloc && rank < (uint32_t)n_scan; base += MG_THREADS) {   // warp-uniform
      const int i = base + tid;
      const bool fr = i < nloc && __ldcg(L.free_map + g0 + i) != 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, fr);
      if (fr) {
        const uint32_t r = rank + __popc(bal & lanemask_lt());
        if (r < (uint32_t)n_scan) bind(g0 + i, r);
      }
      rank += __popc(bal);
    }
  }
  if (!grid_sync(ctr)) return;                           // every binding visible

  // ---- data ---------------------------------------------------------------------
  const int esz = L.kv_dtype == ECHO_F32 ? 4 : 2;
  const int64_t row_bytes = (int64_t)blk_tokens(L) * kv_row_elems(L) * esz;   // one host index / slot
  const int chunks = (int)(row_bytes / 16);             // 72 (bf16) or 144 (f32) per latent token
  if (P.mode == MODE_WRITEBACK) {
    // host pool row, GPU slot row and indexer key of each new token; one warp per request
    for (int64_t b = gwarp; b < P.B; b += gwarps) writeback_row(P, (int)b, lane, step);
  } else if (P.mode == MODE_RECALL) {
    // rows: rank r < nA from staging, else from the host pool (zero-copy reads).
    const int n = nA + nB;
    auto resolve = [&](int64_t r, const uint4 **src, uint4 **dst) {
      *src = nullptr;
      *dst = nullptr;
      int b = 0;
      const int64_t h = token_of((uint32_t)r, &b);
      if (h < 0 || h >= L.n_host) return;
      const int32_t g = ldcg(L.host2gpu + h);
      if (g < 0) return;                                  // not bound: pool exhausted
      if (r < nA) {
        const int ii = (int)r - S.pre_a[b];
        *src = reinterpret_cast<const uint4 *>((const char *)P.stage_kv + ((int64_t)b * P.cap_max + ii) * KV_W * esz);
      } else {
        *src = reinterpret_cast<const uint4 *>((const char *)L.host_kv + h * row_bytes);
      }
      *dst = reinterpret_cast<uint4 *>((char *)L.gpu_kv + (int64_t)g * row_bytes);
    };
    if (chunks <= 144) {
      // token rows: lane j < 4 resolves row r0 + j (list entry, host index, slot) so
      // the four lookups run in parallel; then the warp moves the four rows together
      for (int64_t r0 = gwarp * 4; r0 < n; r0 += gwarps * 4) {
        const uint4 *my_src = nullptr;
        uint4 *my_dst = nullptr;
        if (lane < 4 && r0 + lane < n) resolve(r0 + lane, &my_src, &my_dst);
        const uint4 *src[4];
        uint4 *dst[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          src[j] = reinterpret_cast<const uint4 *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_src), j));
          dst[j] = reinterpret_cast<uint4 *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_dst), j));
        }
        warp_copy_rows4(src, dst, chunks);
      }
    } else {
      // rows of several KB (blocks of tokens, wide rows): one warp per 6 KB segment of
      // a row, so that a few large rows still spread over the whole grid
      constexpr int SEG = 384;
      const int segs = (chunks + SEG - 1) / SEG;
      for (int64_t u = gwarp; u < (int64_t)n * segs; u += gwarps) {
        const int64_t r = u / segs;
        const int c0 = (int)(u % segs) * SEG, c1 = min(chunks, c0 + SEG);
        const uint4 *my_src = nullptr;
        uint4 *my_dst = nullptr;
        if (lane == 0) resolve(r, &my_src, &my_dst);
        const uint4 *src = reinterpret_cast<const uint4 *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_src), 0));
        uint4 *dst = reinterpret_cast<uint4 *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_dst), 0));
        if (src) warp_copy_span(src, dst, c0, c1);
      }
    }
    // slot translation for every selected entry (A10)
    for (int64_t i = gtid; i < (int64_t)P.B * P.k; i += gthreads) {
      const int32_t t = P.sel[i];
      int32_t g = -1;
      if (t >= 0) {
        const int64_t h = (int64_t)P.host_base[i / P.k] + t;
        if (h >= 0 && h < L.n_host) g = ldcg(L.host2gpu + h);
        if (g < 0) g = -1;
      }
      P.slot_idx[i] = g;
    }
  }

  // ---- counters and the manager's scratch words ---------------------------------
  if (m_req > 0) {                                      // clear the global histograms
    for (int64_t i = gtid; i < (int64_t)3 << P.dbits; i += gthreads) {
      P.hist[i] = 0;
      if (P.hist2) P.hist2[i] = 0;
    }
  }
  if (P.mode == MODE_RECALL && P.miss_cnt)               // and the miss counters
    for (int64_t b = gtid; b < P.B; b += gthreads) P.miss_cnt[b] = 0;
  if (blockIdx.x == 0 && tid == 0) {
    const uint32_t scur = (uint32_t)ldcg(ctr + MG_SCUR);
    const uint32_t bound_scan = min(scur, (uint32_t)n_scan);
    const uint32_t bound_victims = min(m_eff, (uint32_t)(n_bind - n_scan));
    const uint32_t bound = bound_scan + bound_victims;
    if (n_bind > 0 && bound < (uint32_t)n_bind) set_status(ctr, ECHO_ERR_POOL_EXHAUSTED);
    ctr[ECHO_CTR_N_FREE] = n_free0 + (int32_t)m_eff - (int32_t)bound;
    ctr[ECHO_CTR_EVICT_M] = (int32_t)m_eff;
    if (P.mode == MODE_WRITEBACK) {           // a write-back begins a step: clear its stats
      ctr[ECHO_CTR_STEP] = step;
      for (int i = ECHO_CTR_HITS; i <= ECHO_CTR_QUALIFIED; ++i) ctr[i] = 0;
      ctr[ECHO_CTR_WB_EVICTED] = (int32_t)m_eff;
    }
    if (P.mode == MODE_RECALL) {
      ctr[ECHO_CTR_NEED] = n_bind;
      ctr[ECHO_CTR_EVICTED] = (int32_t)m_eff;
      ctr[ECHO_CTR_BOUND] = (int32_t)bound;
    }
    ctr[MG_VCUR] = 0;
    ctr[MG_SCUR] = 0;
    ctr[MG_PCUR] = 0;
    ctr[MG_PRE_N] = two ? P.pre_n : 0;                 // every other call drops the list
    ctr[MG_PRE_STEP] = step;
  }
}

// ------------------------------------------------------ write-back, fast --
// The write-back from the pending list, in one CTA: the new tokens that need a slot
// (the full path's rule), then, when every condition of the list holds, its m_req
// largest keys are evicted and bound to them in rank order, the rows are written and
// the counters updated exactly as the full path would; MG_FAST tells the cooperative
// launch that follows whether anything is left to do.  Conditions: the list was left
// by a recall of the current step, no free slot would be used (the full path binds
// those first), it holds at least m_req entries, and every entry's slot still holds
// the key recorded for it.  Victims beyond the list's first B ranks cannot be needed:
// m_req <= B <= pre_n.
constexpr int WF_THREADS = 512;

__global__ void __launch_bounds__(WF_THREADS, 1) wb_fast_kernel(const __grid_constant__ ManageParams P) {
  __shared__ int32_t pre_a[MAXB + 1];
  __shared__ uint64_t pkey[PRE_MAX];
  __shared__ int fast_s;
  const echo_cache_layer_t &L = P.L;
  int32_t *ctr = L.counters;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t step0 = ldcg(ctr + ECHO_CTR_STEP), n_free0 = ldcg(ctr + ECHO_CTR_N_FREE);
  const int32_t pre_n = ldcg(ctr + MG_PRE_N), pre_step = ldcg(ctr + MG_PRE_STEP);
  const int32_t step = step0 + 1;
  // thread i < PRE_MAX reads list entry i and its slot's state now, so these loads
  // overlap the token list below (entries past pre_n are not used)
  static_assert(PRE_MAX <= WF_THREADS, "one list entry per thread");
  int32_t g_i = -1, gh_i = -1, gp_i = 0;
  uint64_t k_i = 0;
  if (tid < PRE_MAX) {
    g_i = ldcg(P.pend + tid);
    k_i = ((uint64_t)(uint32_t)ldcg(P.pend + 2 * PRE_MAX + tid) << 32) | (uint32_t)ldcg(P.pend + PRE_MAX + tid);
    if (g_i >= 0 && g_i < L.n_gpu) {
      gh_i = ldcg(L.gpu2host + g_i);
      gp_i = ldcg(L.priority + g_i);
    }
  }
  block_prefix(P.B, [&](int b) {
    const int32_t l = P.seq_len[b];
    const int64_t h = (int64_t)P.host_base[b] + l;
    const bool ok = h >= 0 && h < (int64_t)L.n_host * blk_tokens(L) && l < P.Lmax;
    return (ok && wb_needs_slot(L, h)) ? 1 : 0;
  }, pre_a);
  const int n_bind = pre_a[P.B];
  const int m_req = max(0, n_bind - n_free0);
  const int n_scan = min(max((int)n_free0, 0), n_bind);
  bool fast = pre_n > 0 && pre_n <= PRE_MAX && pre_step == step0 && n_scan == 0 && m_req <= pre_n;
  if (fast) {
    const int hbits = bitlen_u64((uint64_t)max(L.n_host - 1, 1));
    const uint64_t hmax = (1ull << hbits) - 1;
    if (tid == 0) fast_s = 1;
    __syncthreads();
    if (tid < pre_n) {
      const bool ok = g_i >= 0 && g_i < L.n_gpu && k_i != 0 && victim_key(gh_i, gp_i, step0, hbits, hmax) == k_i;
      if (!ok) fast_s = 0;
      pkey[tid] = k_i;
    }
    __syncthreads();
    fast = fast_s != 0;
  }
  if (!fast) {                                           // uniform: one CTA
    if (tid == 0) ctr[MG_FAST] = 0;
    return;
  }
  // entry i of rank r (largest key first) is a victim if r < m_req and takes the
  // token of rank r; keys are unique
  if (tid < pre_n) {
    int r = 0;
    for (int j = 0; j < pre_n; ++j) r += pkey[j] > k_i;
    if (r < m_req) {
      int lo = 0, hi = P.B - 1;                          // last b with pre_a[b] <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre_a[mid] <= r) lo = mid; else hi = mid - 1;
      }
      const int32_t g = g_i;
      const int64_t h = ((int64_t)P.host_base[lo] + P.seq_len[lo]) / blk_tokens(L);
      L.host2gpu[gh_i] = -1;
      L.free_map[g] = 0;
      L.gpu2host[g] = (int32_t)h;
      L.host2gpu[h] = g;
      L.priority[g] = step;
    }
  }
  __syncthreads();                                       // bindings visible to the block
  for (int b = warp; b < P.B; b += WF_THREADS / 32) writeback_row(P, b, lane, step);
  __syncthreads();
  if (tid == 0) {
    ctr[ECHO_CTR_EVICT_M] = m_req;                       // n_free unchanged: every victim is bound
    ctr[ECHO_CTR_STEP] = step;
    for (int i = ECHO_CTR_HITS; i <= ECHO_CTR_QUALIFIED; ++i) ctr[i] = 0;
    ctr[ECHO_CTR_WB_EVICTED] = m_req;
    ctr[MG_PRE_N] = 0;
    ctr[MG_FAST] = 1;
  }
}

// ------------------------------------------------------------- host side --
int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

static int digit_bits(int n_gpu, int reserve) {   // 3 histograms of 2^bits words (+ reserve) in index_buf
  int b = 1;
  while (b < MG_MAXBITS && (3 << (b + 1)) + reserve <= n_gpu) ++b;
  return b;
}

static cudaError_t run_manage(ManageParams P, cudaStream_t st) {
  const int grid = sm_count();                  // one CTA per SM, all co-resident
  const int per = ((P.L.n_gpu + grid - 1) / grid + 3) & ~3;
  P.cached = (size_t)per * 8 <= MG_KEY_SMEM;
  // the recall's miss counters follow the histograms when the pool leaves room for them
  const int nmc = P.mode == MODE_RECALL ? P.B : 0;
  if (P.L.n_gpu >= PRE_POOL) {
    // the fixed layout with a pending victim list (see PRE_POOL)
    constexpr int nb = 1 << MG_MAXBITS;
    P.dbits = MG_MAXBITS;
    P.hist = reinterpret_cast<uint32_t *>(P.L.index_buf);
    P.miss_cnt = nmc > 0 ? P.L.index_buf + 6 * nb : nullptr;
    P.pend = P.L.index_buf + P.L.n_gpu - 3 * PRE_MAX;
    if (P.mode == MODE_RECALL && P.B <= PRE_MAX) {
      P.hist2 = reinterpret_cast<uint32_t *>(P.L.index_buf + 3 * nb);
      P.pre_n = P.B;
    }
  } else {
    P.dbits = digit_bits(P.L.n_gpu, nmc);
    if ((3 << P.dbits) + nmc > P.L.n_gpu) P.dbits = digit_bits(P.L.n_gpu, 0);
    const bool in_buf = (3 << P.dbits) <= P.L.n_gpu;
    P.hist = in_buf ? reinterpret_cast<uint32_t *>(P.L.index_buf)
                    : reinterpret_cast<uint32_t *>(P.L.counters + MG_SMALL_HIST);
    P.miss_cnt = (nmc > 0 && (3 << P.dbits) + nmc <= P.L.n_gpu) ? P.L.index_buf + (3 << P.dbits) : nullptr;
  }
  if (P.mode == MODE_WRITEBACK && P.L.n_gpu >= PRE_POOL) {
    // the write-back from a pending list, when there is one; the cooperative launch
    // below returns at once if it was done
    wb_fast_kernel<<<1, WF_THREADS, 0, st>>>(P);
    const cudaError_t fe = cudaGetLastError();
    if (fe != cudaSuccess) return fe;
    P.fast_checked = 1;
  }
  const size_t smem = ((sizeof(MgShared) + 15) & ~size_t(15)) + (P.cached ? (size_t)per * 8 : 0);
  cudaError_t e = cudaFuncSetAttribute(mgr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(MG_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mgr_kernel, P);
}

static bool layer_ok(const echo_cache_layer_t *L) {
  if (!L || L->row_elems < 0 || L->row_elems > (1 << 16) || L->block_tokens < 0 || L->block_tokens > 4096)
    return false;
  const int esz = L->kv_dtype == ECHO_F32 ? 4 : 2;
  return L->n_gpu > 0 && L->n_host > 0 && L->host2gpu && L->gpu2host && L->priority && L->index_buf &&
         L->free_map && L->counters && L->gpu_kv && L->host_kv && (kv_row_elems(*L) * esz) % 16 == 0 &&
         (L->kv_dtype == ECHO_F32 || L->kv_dtype == ECHO_BF16) &&
         ((reinterpret_cast<uintptr_t>(L->gpu2host) | reinterpret_cast<uintptr_t>(L->priority) |
           reinterpret_cast<uintptr_t>(L->counters)) & 15) == 0;
}

}  // namespace echo

using namespace echo;

extern "C" {

size_t echo_cache_metadata_bytes(int64_t n_host, int64_t n_gpu) {
  return (size_t)(4 * n_host + 13 * n_gpu);
}

void echo_abi_struct_sizes(size_t out[3]) {
  out[0] = sizeof(echo_cache_layer_t);
  out[1] = sizeof(echo_step_args_t);
  out[2] = sizeof(echo_host_pool_t);
}

echo_status_t echo_host_device_pointer(void *host_ptr, void **dev_ptr) {
  if (!host_ptr || !dev_ptr) return ECHO_ERR_INVALID_ARG;
  ECHO_CUDA_OK(cudaHostGetDevicePointer(dev_ptr, host_ptr, 0));
  return ECHO_OK;
}

int32_t echo_device_sm_count(void) { return sm_count(); }

echo_status_t echo_cache_reset(const echo_cache_layer_t *layer, echo_stream_t stream) {
  if (!layer_ok(layer)) return ECHO_ERR_INVALID_ARG;
  const int64_t n = std::max<int64_t>(std::max(layer->n_host, layer->n_gpu), ECHO_NUM_COUNTERS);
  reset_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(*layer);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

echo_status_t echo_cache_writeback(const echo_cache_layer_t *layer, const void *new_kv, const void *new_ik,
                                   void *idx_k, int32_t D, int32_t Lmax, int32_t ik_dtype,
                                   const int32_t *host_base, int32_t *seq_len, int32_t B, echo_stream_t stream) {
  return echo::cache_writeback_reserve(layer, new_kv, new_ik, idx_k, D, Lmax, ik_dtype, host_base, seq_len, B, 0, 0,
                                       nullptr, nullptr, stream);
}

}  // extern "C"

namespace echo {

// echo_cache_writeback, optionally followed in the same launch by echo_cache_reserve
// (cap != NULL); used by the step executor.
echo_status_t cache_writeback_reserve(const echo_cache_layer_t *layer, const void *new_kv, const void *new_ik,
                                      void *idx_k, int32_t D, int32_t Lmax, int32_t ik_dtype,
                                      const int32_t *host_base, int32_t *seq_len, int32_t B, int32_t cap_max,
                                      int32_t cap_div, int32_t *cap, int32_t *pf_count, echo_stream_t stream) {
  if (!layer_ok(layer) || !new_kv || !new_ik || !idx_k || !host_base || !seq_len) return ECHO_ERR_INVALID_ARG;
  if (cap && (!pf_count || cap_max < 0 || cap_div < 0)) return ECHO_ERR_INVALID_ARG;
  if (B <= 0 || B > MAXB || D <= 0 || Lmax <= 0 || (ik_dtype != ECHO_E4M3 && ik_dtype != ECHO_F32))
    return ECHO_ERR_INVALID_ARG;
  if ((D * (ik_dtype == ECHO_F32 ? 4 : 1)) % 4 != 0 || layer->n_gpu < B) return ECHO_ERR_UNSUPPORTED;
  ManageParams P = {};
  P.L = *layer;
  P.mode = MODE_WRITEBACK;
  P.new_kv = new_kv;
  P.new_ik = new_ik;
  P.idx_k = idx_k;
  P.D = D;
  P.Lmax = Lmax;
  P.ik_dtype = ik_dtype;
  P.host_base = host_base;
  P.seq_len = seq_len;
  P.B = B;
  P.rs_cap = cap;
  P.rs_pf_count = pf_count;
  P.rs_cap_max = cap_max;
  P.rs_cap_div = cap_div;
  ECHO_CUDA_OK(run_manage(P, (cudaStream_t)stream));
  return ECHO_OK;
}

}  // namespace echo

extern "C" {

echo_status_t echo_cache_reserve(const echo_cache_layer_t *layer, const int32_t *seq_len, int32_t B,
                                 int32_t cap_max, int32_t cap_div, int32_t *cap, int32_t *pf_count,
                                 echo_stream_t stream) {
  if (!layer_ok(layer) || !seq_len || !cap || !pf_count || B <= 0 || cap_max < 0 || cap_div < 0)
    return ECHO_ERR_INVALID_ARG;
  reserve_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(*layer, seq_len, B, cap_max, cap_div, cap, pf_count);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

echo_status_t echo_cache_evict(const echo_cache_layer_t *layer, const int32_t *n_needed, echo_stream_t stream) {
  if (!layer_ok(layer) || !n_needed) return ECHO_ERR_INVALID_ARG;
  ManageParams P = {};
  P.L = *layer;
  P.mode = MODE_EVICT;
  P.n_needed = n_needed;
  ECHO_CUDA_OK(run_manage(P, (cudaStream_t)stream));
  return ECHO_OK;
}

echo_status_t echo_cache_alloc(const echo_cache_layer_t *layer, const int32_t *host_idx, const int32_t *n,
                               int32_t n_max, int32_t *out_slot, echo_stream_t stream) {
  if (!layer_ok(layer) || !host_idx || !n || n_max < 0) return ECHO_ERR_INVALID_ARG;
  ManageParams P = {};
  P.L = *layer;
  P.mode = MODE_ALLOC;
  P.host_idx = host_idx;
  P.n_ptr = n;
  P.n_max = n_max;
  P.out_slot = out_slot;
  ECHO_CUDA_OK(run_manage(P, (cudaStream_t)stream));
  return ECHO_OK;
}

echo_status_t echo_cache_recall(const echo_cache_layer_t *layer, const int32_t *sel, const int32_t *host_base,
                                int32_t B, int32_t k, const int32_t *pf_list, const int32_t *pf_count,
                                int32_t cap_max, const void *stage_kv, int32_t *miss_list, int32_t *n_miss,
                                int32_t *slot_idx, echo_stream_t stream) {
  if (!layer_ok(layer) || !sel || !host_base || !miss_list || !n_miss || !slot_idx) return ECHO_ERR_INVALID_ARG;
  if (B <= 0 || B > MAXB || k <= 0) return ECHO_ERR_INVALID_ARG;
  if (pf_count && (!pf_list || !stage_kv || cap_max <= 0)) return ECHO_ERR_INVALID_ARG;
  if (pf_count && !layer_takes_prefetch(layer)) return ECHO_ERR_UNSUPPORTED;
  ManageParams P = {};
  P.L = *layer;
  P.mode = MODE_RECALL;
  P.host_base = host_base;
  P.B = B;
  P.sel = sel;
  P.k = k;
  P.pf_list = pf_list;
  P.pf_count = pf_count;
  P.cap_max = pf_count ? cap_max : 0;
  P.stage_kv = stage_kv;
  P.miss_list = miss_list;
  P.n_miss = n_miss;
  P.slot_idx = slot_idx;
  ECHO_CUDA_OK(run_manage(P, (cudaStream_t)stream));
  return ECHO_OK;
}

echo_status_t echo_cache_status(const echo_cache_layer_t *layer, int32_t *host_status) {
  if (!layer || !layer->counters || !host_status) return ECHO_ERR_INVALID_ARG;
  ECHO_CUDA_OK(cudaDeviceSynchronize());
  ECHO_CUDA_OK(cudaMemcpy(host_status, layer->counters + ECHO_CTR_STATUS, sizeof(int32_t), cudaMemcpyDeviceToHost));
  return ECHO_OK;
}

echo_status_t echo_cache_read_counters(const echo_cache_layer_t *layer, int32_t *host_counters) {
  if (!layer || !layer->counters || !host_counters) return ECHO_ERR_INVALID_ARG;
  ECHO_CUDA_OK(cudaDeviceSynchronize());
  ECHO_CUDA_OK(cudaMemcpy(host_counters, layer->counters, sizeof(int32_t) * ECHO_NUM_COUNTERS,
                          cudaMemcpyDeviceToHost));
  return ECHO_OK;
}

}  // extern "C"
