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
//   reset_kernel          empty cache
//   reserve_kernel        per-request prefetch budget (A2)
//   manage_kernel<CL>     one thread-block cluster: LRU victim selection by radix
//                         select over keys held in shared memory, eviction, and
//                         allocation by warp-ballot scan of the free bitmap with one
//                         atomic per warp; modes write-back (A1), recall bind (A7+A8),
//                         alloc (A8), evict (A7)
//   miss_kernel           protect hits, list misses (A6)
//   copy_translate_kernel zero-copy host reads + staged rows into slots, slot ids (A9, A10)

#include <algorithm>
#include <cooperative_groups.h>

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
__global__ void reserve_kernel(echo_cache_layer_t L, const int32_t *seq_len, int B, int cap_max, int cap_div,
                               int32_t *cap, int32_t *pf_count) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int c = 0;
    if (cap_max > 0) {
      const int l = seq_len[b];
      c = cap_div > 0 ? min(cap_max, (l + cap_div - 1) / cap_div) : cap_max;
      c = max(c, 0);
    }
    cap[b] = c;
    pf_count[b] = 0;
  }
}

// ------------------------------------------------------ cluster management --
enum { MODE_WRITEBACK = 0, MODE_RECALL = 1, MODE_ALLOC = 2, MODE_EVICT = 3 };

struct ManageParams {
  echo_cache_layer_t L;
  int mode;
  // write-back
  const void *new_kv;
  const void *new_ik;
  void *idx_k;
  int D, Lmax, ik_dtype;
  const int32_t *host_base;
  int32_t *seq_len;
  int B;
  // recall
  const int32_t *pf_list;
  const int32_t *pf_count;
  int cap_max;
  const int32_t *miss_list;
  const int32_t *n_miss;
  int k;
  // alloc
  const int32_t *host_idx;
  const int32_t *n_ptr;
  int n_max;
  int32_t *out_slot;
  // evict
  const int32_t *n_needed;
};

constexpr int MG_THREADS = 1024;
constexpr int NBINS = 2048;          // 11-bit radix digits
constexpr int KEYCAP = 24 * 1024;    // 64-bit keys cached per CTA (192 KB)
constexpr int MAXB = 1024;           // requests per call handled by the manager

struct MgShared {
  uint32_t hist[2][NBINS];
  uint32_t warp_sums[32];
  uint32_t res[4];                   // [0] chosen digit, [1] count above it
  uint32_t cursor;                   // allocation cursor (CTA 0's copy is used)
  uint32_t cnt;                      // eligible count of this CTA
  uint32_t vcnt, vcur;               // victims of this CTA, victim-rank cursor
  int32_t pre_a[MAXB + 1];           // prefixes of the token lists
  int32_t pre_b[MAXB + 1];
};

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

__device__ __forceinline__ int bitlen_u64(uint64_t x) { return x ? 64 - __clzll((long long)x) : 0; }

// Victim key of slot g: larger key = smaller (priority, host index) = evicted first.
// 0 = not evictable (free, or touched in the current step).
__device__ __forceinline__ uint64_t victim_key(const echo_cache_layer_t &L, int g, int32_t step, int hbits,
                                               uint64_t hmax) {
  const int32_t h = L.gpu2host[g];
  if (h < 0) return 0;
  const int32_t p = L.priority[g];
  if (p >= step || p < 0) return 0;
  const uint64_t age = (uint64_t)(int64_t)(step - 1 - p);
  return ((age << hbits) | (hmax - (uint64_t)h)) + 1;
}

template <int CL>
__global__ void __launch_bounds__(MG_THREADS, 1) manage_kernel(ManageParams P) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char dsm[];
  MgShared &S = *reinterpret_cast<MgShared *>(dsm);
  uint64_t *keys = reinterpret_cast<uint64_t *>(dsm + ((sizeof(MgShared) + 15) & ~size_t(15)));
  const echo_cache_layer_t &L = P.L;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  int32_t *ctr = L.counters;

  const int32_t step0 = ctr[ECHO_CTR_STEP];
  const int32_t step = P.mode == MODE_WRITEBACK ? step0 + 1 : step0;
  const int32_t n_free0 = ctr[ECHO_CTR_N_FREE];

  // ---- the tokens that need a slot: list A (+ list B) ------------------
  // write-back: A = new tokens not yet resident; recall: A = staged rows,
  // B = misses; alloc: A = host_idx[0..n).
  int nA = 0, nB = 0;
  if (P.mode == MODE_WRITEBACK) {
    block_prefix(P.B, [&](int b) {
      const int32_t l = P.seq_len[b];
      const int64_t h = (int64_t)P.host_base[b] + l;
      const bool ok = h >= 0 && h < L.n_host && l < P.Lmax;
      return (ok && L.host2gpu[h] < 0) ? 1 : 0;
    }, S.pre_a);
  } else if (P.mode == MODE_RECALL) {
    const int32_t *pfc = P.pf_count;
    const int cm = P.cap_max;
    block_prefix(P.B, [&](int b) { return pfc ? min(max(pfc[b], 0), cm) : 0; }, S.pre_a);
    block_prefix(P.B, [&](int b) { return (int)P.n_miss[b]; }, S.pre_b);
  }
  if (tid == 0) { S.cursor = 0; S.cnt = 0; S.vcnt = 0; S.vcur = 0; }
  __syncthreads();
  if (P.mode == MODE_WRITEBACK) nA = S.pre_a[P.B];
  if (P.mode == MODE_RECALL) { nA = S.pre_a[P.B]; nB = S.pre_b[P.B]; }
  if (P.mode == MODE_ALLOC) nA = min(max(*P.n_ptr, 0), P.n_max);
  const int n_bind = (P.mode == MODE_EVICT) ? 0 : nA + nB;

  int m_req = 0;                           // victims wanted
  if (P.mode == MODE_WRITEBACK || P.mode == MODE_RECALL) m_req = max(0, n_bind - n_free0);
  if (P.mode == MODE_EVICT) m_req = max(0, *P.n_needed - n_free0);

  // ---- this CTA's slot range ----------------------------------------------
  const int per = ((L.n_gpu + CL - 1) / CL + 3) & ~3;     // slices start 16-byte aligned
  const int g0 = min(L.n_gpu, (int)rank * per), g1 = min(L.n_gpu, g0 + per);
  const int nloc = g1 - g0;
  const bool cached = per <= KEYCAP;
  int hbits = bitlen_u64((uint64_t)max(L.n_host - 1, 1));
  const uint64_t hmax = (1ull << hbits) - 1;
  const int nb = bitlen_u64((uint64_t)max(step, 1)) + hbits + 1;

  // tokens of ranks [0, n_scan) go to slots that were already free (bitmap scan);
  // tokens of ranks [n_scan, n_bind) go straight to this call's victims
  const int n_scan = min(max((int)n_free0, 0), n_bind);
  // host index of the token of rank r
  auto token_of = [&](uint32_t r, int *req) -> int64_t {
    if (P.mode == MODE_WRITEBACK) {
      int b = 0;                                   // rank r -> request (B is small)
      while (b + 1 < P.B && S.pre_a[b + 1] <= (int)r) ++b;
      *req = b;
      return (int64_t)P.host_base[b] + P.seq_len[b];
    } else if (P.mode == MODE_RECALL) {
      const int32_t *pre = (int)r < nA ? S.pre_a : S.pre_b;
      const int rr = (int)r < nA ? (int)r : (int)r - nA;
      int lo = 0, hi = P.B - 1;                    // last b with pre[b] <= rr
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= rr) lo = mid; else hi = mid - 1;
      }
      const int b = lo, ii = rr - pre[b];
      const int32_t t = (int)r < nA ? P.pf_list[(int64_t)b * P.cap_max + ii] : P.miss_list[(int64_t)b * P.k + ii];
      *req = b;
      return (int64_t)P.host_base[b] + t;
    }
    *req = 0;
    return P.host_idx[r];
  };
  // bind the token of rank r to slot g (slot already removed from the free bitmap)
  auto bind = [&](int g, uint32_t r) {
    int b = 0;
    const int64_t h = token_of(r, &b);
    if (h >= 0 && h < L.n_host) {
      L.free_map[g] = 0;
      L.gpu2host[g] = (int32_t)h;
      L.host2gpu[h] = g;
      L.priority[g] = step;
      if (P.mode == MODE_WRITEBACK) L.index_buf[b] = g;
      if (P.mode == MODE_ALLOC && P.out_slot) P.out_slot[r] = g;
    } else {
      L.gpu2host[g] = -1;
      L.free_map[g] = 1;
      set_status(ctr, ECHO_ERR_HOST_INDEX);
      if (P.mode == MODE_ALLOC && P.out_slot) P.out_slot[r] = -1;
    }
  };

  uint32_t m_eff = 0;
  uint64_t kstar = ~0ull;
  if (m_req > 0) {                                         // uniform across the cluster
    // load keys (4 slots per thread and iteration, both arrays as int4), count evictable
    uint32_t c = 0;
    const int n4 = nloc >> 2;
    const int4 *g2h4 = reinterpret_cast<const int4 *>(L.gpu2host + g0);
    const int4 *pr4 = reinterpret_cast<const int4 *>(L.priority + g0);
    auto key_of = [&](int32_t hh, int32_t pp) -> uint64_t {
      if (hh < 0 || pp >= step || pp < 0) return 0;
      return (((uint64_t)(int64_t)(step - 1 - pp) << hbits) | (hmax - (uint64_t)hh)) + 1;
    };
    for (int j = tid; j < n4; j += MG_THREADS) {
      const int4 hv = g2h4[j], pv = pr4[j];
      const uint64_t k0 = key_of(hv.x, pv.x), k1 = key_of(hv.y, pv.y), k2 = key_of(hv.z, pv.z),
                     k3 = key_of(hv.w, pv.w);
      if (cached) {
        keys[4 * j] = k0; keys[4 * j + 1] = k1; keys[4 * j + 2] = k2; keys[4 * j + 3] = k3;
      }
      c += (k0 != 0) + (k1 != 0) + (k2 != 0) + (k3 != 0);
    }
    for (int i = 4 * n4 + tid; i < nloc; i += MG_THREADS) {
      const uint64_t kk = victim_key(L, g0 + i, step, hbits, hmax);
      if (cached) keys[i] = kk;
      c += kk != 0;
    }
    c = __reduce_add_sync(0xffffffffu, c);
    if ((tid & 31) == 0) atomicAdd(&S.cnt, c);
    __syncthreads();
    cluster_sync();
    uint32_t total = 0;
    for (uint32_t r = 0; r < CL; ++r) total += *cluster.map_shared_rank(&S.cnt, r);
    m_eff = min((uint32_t)m_req, total);
    if (rank == 0 && tid == 0 && m_eff < (uint32_t)m_req) set_status(ctr, ECHO_ERR_POOL_EXHAUSTED);

    if (m_eff > 0) {
      // MSB-first radix select of the m_eff-th largest key (keys are unique).
      uint64_t prefix = 0;
      uint32_t above = 0;
      int left = nb, buf = 0;
      while (left > 0) {
        const int w = min(11, left), shift = left - w;
        uint32_t *h = S.hist[buf];
        for (int i = tid; i < NBINS; i += MG_THREADS) h[i] = 0;
        __syncthreads();
        const uint64_t hi_mask = (shift + w >= 64) ? 0ull : (~0ull << (shift + w));
        for (int base = 0; base < nloc; base += MG_THREADS) {   // uniform trip count per warp
          const int i = base + tid;
          uint64_t kk = 0;
          if (i < nloc) kk = cached ? keys[i] : victim_key(L, g0 + i, step, hbits, hmax);
          hist_add_warp(h, kk != 0 && (kk & hi_mask) == (prefix & hi_mask),
                        (uint32_t)((kk >> shift) & ((1u << w) - 1)));
        }
        __syncthreads();
        cluster_sync();
        // global counts of my two bins; find the digit (descending)
        const int d1 = 2 * tid + 1, d0 = 2 * tid;
        uint32_t c1 = 0, c0 = 0;
#pragma unroll
        for (uint32_t r = 0; r < CL; ++r) {             // plain loads, issued together
          const uint2 v = *reinterpret_cast<const uint2 *>(cluster.map_shared_rank(&h[d0], r));
          c0 += v.x;
          c1 += v.y;
        }
        uint32_t tot;
        const uint32_t incl = block_incl_scan(c0 + c1, S.warp_sums, &tot);
        const uint32_t sfx = tot - incl;                     // keys in bins above mine
        const uint32_t need = m_eff - above;
        if (sfx < need && need <= sfx + c1) { S.res[0] = d1; S.res[1] = sfx; }
        else if (sfx + c1 < need && need <= sfx + c1 + c0) { S.res[0] = d0; S.res[1] = sfx + c1; }
        __syncthreads();
        prefix |= (uint64_t)S.res[0] << shift;
        above += S.res[1];
        left = shift;
        buf ^= 1;
        __syncthreads();
      }
      kstar = prefix;
      // evict every key >= kstar (exactly m_eff tokens).  Victims are ranked across
      // the cluster (prefix of per-CTA counts; any order inside a CTA) and victim v
      // is rebound at once to the token of rank n_scan + v, or freed if none is left.
      uint32_t nv = 0;
      for (int base = 0; base < nloc; base += MG_THREADS) {
        const int i = base + tid;
        uint64_t kk = 0;
        if (i < nloc) kk = cached ? keys[i] : victim_key(L, g0 + i, step, hbits, hmax);
        nv += __popc(__ballot_sync(0xffffffffu, kk != 0 && kk >= kstar));
      }
      if ((tid & 31) == 0) atomicAdd(&S.vcnt, nv);
      __syncthreads();
      cluster_sync();
      uint32_t vbase = 0;
      for (uint32_t r = 0; r < rank; ++r) vbase += *cluster.map_shared_rank(&S.vcnt, r);
      for (int base = 0; base < nloc; base += MG_THREADS) {
        const int i = base + tid;
        uint64_t kk = 0;
        if (i < nloc) kk = cached ? keys[i] : victim_key(L, g0 + i, step, hbits, hmax);
        const bool isv = kk != 0 && kk >= kstar;
        const uint32_t bal = __ballot_sync(0xffffffffu, isv);
        uint32_t wb = 0;
        if ((tid & 31) == 0 && bal) wb = atomicAdd(&S.vcur, (uint32_t)__popc(bal));
        wb = __shfl_sync(0xffffffffu, wb, 0);
        if (isv) {
          const int g = g0 + i;
          L.host2gpu[L.gpu2host[g]] = -1;
          const uint32_t r = (uint32_t)n_scan + vbase + wb + __popc(bal & lanemask_lt());
          if (r < (uint32_t)n_bind) {
            bind(g, r);
          } else {
            L.gpu2host[g] = -1;
            L.free_map[g] = 1;
          }
        }
      }
    }
  }
  cluster_sync();                                      // evictions visible cluster-wide

  // ---- allocation of already-free slots: warp-ballot scan of the free bitmap
  // with one atomic count per warp (ranks [0, n_scan)) ----------------------
  const uint32_t cursor_addr = map_dsmem(&S.cursor, 0);
  if (n_scan > 0) {
    const int lane = tid & 31;
    for (int base = 0; base < nloc; base += MG_THREADS) {
      // stop early once every token has a slot (one read per warp, uniform)
      uint32_t cur = 0;
      if (lane == 0) cur = ld_dsmem_u32(cursor_addr);
      if (__shfl_sync(0xffffffffu, cur, 0) >= (uint32_t)n_scan) break;
      const int i = base + tid;
      const bool fr = i < nloc && L.free_map[g0 + i] != 0;
      const uint32_t bal = __ballot_sync(0xffffffffu, fr);
      uint32_t wbase = 0;
      if (lane == 0 && bal) {
        uint32_t old;
        asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(cursor_addr), "r"((uint32_t)__popc(bal)) : "memory");
        wbase = old;
      }
      wbase = __shfl_sync(0xffffffffu, wbase, 0);
      if (fr) {
        const uint32_t r = wbase + __popc(bal & lanemask_lt());
        if (r < (uint32_t)n_scan) bind(g0 + i, r);
      }
    }
  }
  cluster_sync();                                      // bindings visible cluster-wide

  // ---- write-back data: host pool row, GPU slot row, indexer key ----------
  if (P.mode == MODE_WRITEBACK) {
    const int warps = MG_THREADS / 32, wid = tid >> 5, lane = tid & 31;
    const int esz = L.kv_dtype == ECHO_F32 ? 4 : 2;
    const int row_chunks = KV_W * esz / 16;
    for (int b = rank * warps + wid; b < P.B; b += CL * warps) {
      const int32_t l = P.seq_len[b];
      const int64_t h = (int64_t)P.host_base[b] + l;
      if (h < 0 || h >= L.n_host) { if (lane == 0) set_status(ctr, ECHO_ERR_HOST_INDEX); continue; }
      if (l >= P.Lmax) { if (lane == 0) set_status(ctr, ECHO_ERR_INVALID_ARG); continue; }
      const int32_t g = L.host2gpu[h];
      const uint4 *src = reinterpret_cast<const uint4 *>((const char *)P.new_kv + (int64_t)b * KV_W * esz);
      uint4 *hdst = reinterpret_cast<uint4 *>((char *)L.host_kv + h * KV_W * esz);
      uint4 *gdst = g >= 0 ? reinterpret_cast<uint4 *>((char *)L.gpu_kv + (int64_t)g * KV_W * esz) : nullptr;
      for (int c = lane; c < row_chunks; c += 32) {
        const uint4 v = src[c];
        hdst[c] = v;
        if (gdst) gdst[c] = v;
      }
      if (g >= 0 && lane == 0) L.priority[g] = step;     // refresh an already resident token
      if (g < 0 && lane == 0) set_status(ctr, ECHO_ERR_POOL_EXHAUSTED);
      const int kesz = P.ik_dtype == ECHO_F32 ? 4 : 1;
      const char *ks = (const char *)P.new_ik + (int64_t)b * P.D * kesz;
      char *kd = (char *)P.idx_k + ((int64_t)b * P.Lmax + l) * P.D * kesz;
      for (int c = lane; c < P.D * kesz / 4; c += 32)
        reinterpret_cast<uint32_t *>(kd)[c] = reinterpret_cast<const uint32_t *>(ks)[c];
      __syncwarp();
      if (lane == 0) P.seq_len[b] = l + 1;
    }
  }

  // ---- counters (CTA 0, after everything) ---------------------------------
  cluster_sync();
  if (rank == 0 && tid == 0) {
    const uint32_t bound_scan = min(S.cursor, (uint32_t)n_scan);
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
  }
}

// --------------------------------------------------------- miss detection --
__global__ void miss_kernel(echo_cache_layer_t L, const int32_t *sel, const int32_t *host_base, int B, int k,
                            int32_t *miss_list, int32_t *n_miss, int32_t *slot_idx) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int32_t step = L.counters[ECHO_CTR_STEP];
  uint32_t hit = 0, staged = 0, miss = 0;
  if (i < (int64_t)B * k) {
    const int b = (int)(i / k);
    const int32_t t = sel[i];
    int32_t out = -1;
    if (t >= 0) {
      const int64_t h = (int64_t)host_base[b] + t;
      if (h >= L.n_host) {
        set_status(L.counters, ECHO_ERR_HOST_INDEX);
      } else {
        const int32_t g = L.host2gpu[h];
        if (g >= 0) {
          L.priority[g] = step;                      // protect the selection
          out = g;
          hit = 1;
        } else if (g <= -2) {
          staged = 1;
        } else {
          const int32_t pos = atomicAdd(&n_miss[b], 1);
          miss_list[(int64_t)b * k + pos] = t;
          miss = 1;
        }
      }
    }
    slot_idx[i] = out;
  }
  hit = __reduce_add_sync(0xffffffffu, hit);
  staged = __reduce_add_sync(0xffffffffu, staged);
  miss = __reduce_add_sync(0xffffffffu, miss);
  if ((threadIdx.x & 31) == 0) {
    if (hit) atomicAdd(&L.counters[ECHO_CTR_HITS], (int)hit);
    if (staged) atomicAdd(&L.counters[ECHO_CTR_STAGED_HITS], (int)staged);
    if (miss) atomicAdd(&L.counters[ECHO_CTR_MISSES], (int)miss);
  }
}

// --------------------------------------------------- copy + slot translate --
constexpr int CT_THREADS = 256;
constexpr int CT_ROWS = 4;           // rows in flight per warp

__global__ void __launch_bounds__(CT_THREADS) copy_translate_kernel(
    echo_cache_layer_t L, const int32_t *sel, const int32_t *host_base, int B, int k, const int32_t *pf_list,
    const int32_t *pf_count, int cap_max, const void *stage_kv, const int32_t *miss_list, const int32_t *n_miss,
    int32_t *slot_idx) {
  __shared__ int32_t pre_a[MAXB + 1], pre_b[MAXB + 1];
  block_prefix(B, [&](int b) { return pf_count ? min(max(pf_count[b], 0), cap_max) : 0; }, pre_a);
  block_prefix(B, [&](int b) { return (int)n_miss[b]; }, pre_b);
  const int nA = pre_a[B], n = nA + pre_b[B];
  const int esz = L.kv_dtype == ECHO_F32 ? 4 : 2;
  const int chunks = KV_W * esz / 16;                 // 72 (bf16) or 144 (f32)
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)CT_THREADS + threadIdx.x) >> 5;
  const int64_t nw = (gridDim.x * (int64_t)CT_THREADS) >> 5;

  // rows: r < nA from staging, else from the host pool.  Lane j < CT_ROWS resolves
  // row r0 + j (list entry, host index, slot) so the 4 lookups run in parallel.
  for (int64_t r0 = gw * CT_ROWS; r0 < n; r0 += nw * CT_ROWS) {
    const uint4 *my_src = nullptr;
    uint4 *my_dst = nullptr;
    const int64_t r = r0 + lane;
    if (lane < CT_ROWS && r < n) {
      const bool staged = r < nA;
      const int32_t *pre = staged ? pre_a : pre_b;
      const int rr = staged ? (int)r : (int)(r - nA);
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= rr) lo = mid; else hi = mid - 1;
      }
      const int b = lo, ii = rr - pre[b];
      const int32_t t = staged ? pf_list[(int64_t)b * cap_max + ii] : miss_list[(int64_t)b * k + ii];
      const int64_t h = (int64_t)host_base[b] + t;
      if (h >= 0 && h < L.n_host) {
        const int32_t g = L.host2gpu[h];
        if (g >= 0) {                                       // not bound: pool exhausted
          my_src = staged ? reinterpret_cast<const uint4 *>((const char *)stage_kv +
                                                            ((int64_t)b * cap_max + ii) * KV_W * esz)
                          : reinterpret_cast<const uint4 *>((const char *)L.host_kv + h * KV_W * esz);
          my_dst = reinterpret_cast<uint4 *>((char *)L.gpu_kv + (int64_t)g * KV_W * esz);
        }
      }
    }
    const uint4 *src[CT_ROWS];
    uint4 *dst[CT_ROWS];
#pragma unroll
    for (int j = 0; j < CT_ROWS; ++j) {
      src[j] = reinterpret_cast<const uint4 *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_src), j));
      dst[j] = reinterpret_cast<uint4 *>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(my_dst), j));
    }
    warp_copy_rows4(src, dst, chunks);
  }

  // slot translation for every selected entry (A10)
  const int64_t tid = blockIdx.x * (int64_t)CT_THREADS + threadIdx.x;
  const int64_t nt = gridDim.x * (int64_t)CT_THREADS;
  for (int64_t i = tid; i < (int64_t)B * k; i += nt) {
    const int32_t t = sel[i];
    int32_t g = -1;
    if (t >= 0) {
      const int64_t h = (int64_t)host_base[i / k] + t;
      if (h >= 0 && h < L.n_host) g = L.host2gpu[h];
      if (g < 0) g = -1;
    }
    slot_idx[i] = g;
  }
}

// ------------------------------------------------------------- host side --
static int g_cluster = 0;  // chosen cluster size for manage_kernel (16 if allowed, else 8)

static size_t manage_smem(int CL, int n_gpu) {
  const int per = ((n_gpu + CL - 1) / CL + 3) & ~3;
  size_t s = (sizeof(MgShared) + 15) & ~size_t(15);
  if (per <= KEYCAP) s += (size_t)per * 8;
  return s;
}

template <int CL>
static cudaError_t launch_manage(const ManageParams &P, cudaStream_t st) {
  const size_t smem = manage_smem(CL, P.L.n_gpu);
  cudaError_t e = cudaFuncSetAttribute(manage_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (CL > 8) {
    e = cudaFuncSetAttribute(manage_kernel<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL, 1, 1);
  cfg.blockDim = dim3(MG_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, manage_kernel<CL>, P);
}

static int pick_cluster(int n_gpu) {
  if (g_cluster) return g_cluster;
  int cl = 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(16, 1, 1);
  cfg.blockDim = dim3(MG_THREADS, 1, 1);
  cfg.dynamicSmemBytes = manage_smem(16, std::max(n_gpu, 1));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 16;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(manage_kernel<16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
      cudaFuncSetAttribute(manage_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)cfg.dynamicSmemBytes) == cudaSuccess) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, manage_kernel<16>, &cfg) == cudaSuccess && n > 0) cl = 16;
  }
  cudaGetLastError();
  g_cluster = cl;
  return cl;
}

static cudaError_t run_manage(const ManageParams &P, cudaStream_t st) {
  const int cl = pick_cluster(P.L.n_gpu);
  return cl == 16 ? launch_manage<16>(P, st) : launch_manage<8>(P, st);
}

static bool layer_ok(const echo_cache_layer_t *L) {
  return L && L->n_gpu > 0 && L->n_host > 0 && L->host2gpu && L->gpu2host && L->priority && L->index_buf &&
         L->free_map && L->counters && L->gpu_kv && L->host_kv &&
         (L->kv_dtype == ECHO_F32 || L->kv_dtype == ECHO_BF16) &&
         ((reinterpret_cast<uintptr_t>(L->gpu2host) | reinterpret_cast<uintptr_t>(L->priority)) & 15) == 0;
}

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

}  // namespace echo

using namespace echo;

extern "C" {

size_t echo_cache_metadata_bytes(int64_t n_host, int64_t n_gpu) {
  return (size_t)(4 * n_host + 13 * n_gpu);
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
  if (!layer_ok(layer) || !new_kv || !new_ik || !idx_k || !host_base || !seq_len) return ECHO_ERR_INVALID_ARG;
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
  ECHO_CUDA_OK(run_manage(P, (cudaStream_t)stream));
  return ECHO_OK;
}

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
  cudaStream_t st = (cudaStream_t)stream;
  ECHO_CUDA_OK(cudaMemsetAsync(n_miss, 0, sizeof(int32_t) * B, st));
  const int64_t nsel = (int64_t)B * k;
  miss_kernel<<<(unsigned)((nsel + 255) / 256), 256, 0, st>>>(*layer, sel, host_base, B, k, miss_list, n_miss,
                                                                slot_idx);
  ECHO_LAUNCH_OK();
  ManageParams P = {};
  P.L = *layer;
  P.mode = MODE_RECALL;
  P.host_base = host_base;
  P.B = B;
  P.pf_list = pf_list;
  P.pf_count = pf_count;
  P.cap_max = pf_count ? cap_max : 0;
  P.miss_list = miss_list;
  P.n_miss = n_miss;
  P.k = k;
  ECHO_CUDA_OK(run_manage(P, st));
  const int grid = sm_count() * 4;
  copy_translate_kernel<<<grid, CT_THREADS, 0, st>>>(*layer, sel, host_base, B, k, pf_list, pf_count,
                                                     pf_count ? cap_max : 0, stage_kv, miss_list, n_miss, slot_idx);
  ECHO_LAUNCH_OK();
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
