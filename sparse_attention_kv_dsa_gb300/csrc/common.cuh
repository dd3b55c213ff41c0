// Shared device helpers of the ECHO library (sm_103a): status words, bounded waits,
// order-preserving keys, and inline-PTX wrappers for mbarrier, TMA, cp.async and
// tcgen05 (5th-generation tensor cores with TMEM accumulators).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "echo.h"

#define ECHO_CUDA_OK(expr)                                 \
  do {                                                     \
    cudaError_t e__ = (expr);                              \
    if (e__ != cudaSuccess) return ECHO_ERR_CUDA;          \
  } while (0)

#define ECHO_LAUNCH_OK()                                   \
  do {                                                     \
    cudaError_t e__ = cudaGetLastError();                  \
    if (e__ != cudaSuccess) return ECHO_ERR_CUDA;          \
  } while (0)

namespace echo {

constexpr int KV_W = ECHO_KV_WIDTH;   // 576
constexpr int V_W = ECHO_V_WIDTH;     // 512

// Values per token row of a layer's pools: 576 unless the layer sets row_elems.
__host__ __device__ __forceinline__ int kv_row_elems(const echo_cache_layer_t &L) {
  return L.row_elems > 0 ? L.row_elems : KV_W;
}

// The fused prefetch stages 576-wide token rows: layers with block granularity or
// another row width take none.
inline bool layer_takes_prefetch(const echo_cache_layer_t *L) {
  return L->block_tokens <= 1 && kv_row_elems(*L) == KV_W;
}

// ---------------------------------------------------------------- status --
__device__ __forceinline__ void set_status(int32_t *counters, int32_t code) {
  if (counters) atomicCAS(counters + ECHO_CTR_STATUS, 0, code);
}

// 1-second bound on every spin in this library (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ float keys --
// Order-preserving map float -> uint32 (larger float -> larger key); -0 == +0.
__device__ __forceinline__ uint32_t f32_key(float x) {
  uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_f32(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// ---------------------------------------------------------------- smem ----
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// -------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity; false after ~1 s.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// The same load with an L2 eviction-priority policy (from l2_evict_first_policy).
__device__ __forceinline__ void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                                 int32_t c0, int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
// Policy for data read once: evicted from L2 first, so it does not push out data that
// the next kernels read again (scores, cache metadata).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// -------------------------------------------------------------- cp.async --
// 16-byte global -> shared copy; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Every cp.async of this thread so far, committed to a group or not, has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, FP8 e4m3 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem], bf16/f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// mbarrier arrives once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive 32-bit TMEM columns of this thread's lane (32x32b shape, x32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (64-bit): start address,
// leading / stride byte offsets (>> 4), version 1, layout (swizzle) type.
enum : uint32_t { LAYOUT_NONE = 0, LAYOUT_SW128 = 2 };
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 0x7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 / kind::f8f6f4: f32 accumulator,
// a/b formats, K-major (0) or MN-major (1) operands, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t a_fmt, uint32_t b_fmt, uint32_t a_mn_major,
                                                  uint32_t b_mn_major, uint32_t M, uint32_t N) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (a_mn_major << 15) | (b_mn_major << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t FMT_E4M3 = 0;  // kind::f8f6f4
constexpr uint32_t FMT_BF16 = 1;  // kind::f16

// --------------------------------------------------------- cluster / DSMEM --
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_dsmem(const void *p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_dsmem_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void atom_add_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ------------------------------------------------------------ host utils --
int sm_count();
cudaError_t check_launch();
// 2-D byte tensor [rows, 128] with a [box_rows, 128] box and 128-byte swizzle (TMA).
bool make_map_128B(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows);
echo_status_t cache_writeback_reserve(const echo_cache_layer_t *layer, const void *new_kv, const void *new_ik,
                                      void *idx_k, int32_t D, int32_t Lmax, int32_t ik_dtype,
                                      const int32_t *host_base, int32_t *seq_len, int32_t B, int32_t cap_max,
                                      int32_t cap_div, int32_t *cap, int32_t *pf_count, echo_stream_t stream);

}  // namespace echo

namespace echo {
// Warp-cooperative copy of up to 4 rows of `chunks` 16-byte chunks each (src may be
// host-mapped memory).  All loads of a batch are issued before any store so that
// several rows are in flight on the host link.  Rows with a null src are skipped.
// Chunks [c0, c1) of one row by a warp, four 16-byte loads per lane in flight.
__device__ __forceinline__ void warp_copy_span(const uint4 *src, uint4 *dst, int c0, int c1) {
  const int lane = threadIdx.x & 31;
  for (int base = c0; base < c1; base += 128) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = base + lane + 32 * u;
      if (c < c1) v[u] = __ldg(src + c);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = base + lane + 32 * u;
      if (c < c1) dst[c] = v[u];
    }
  }
}

__device__ __forceinline__ void warp_copy_rows4(const uint4 *const (&src)[4], uint4 *const (&dst)[4],
                                                int chunks) {
  const int lane = threadIdx.x & 31;
  for (int c0 = 0; c0 < chunks; c0 += 96) {
    uint4 v[4][3];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        const int c = c0 + lane + 32 * u;
        if (src[j] && c < chunks) v[j][u] = __ldg(src[j] + c);
      }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        const int c = c0 + lane + 32 * u;
        if (src[j] && c < chunks) dst[j][c] = v[j][u];
      }
  }
}
}  // namespace echo

namespace echo {
// Histogram increment aggregated over the warp: lanes with the same bin add once
// (keys of scores and of LRU ages cluster in few bins).  All 32 lanes must call it.
__device__ __forceinline__ void hist_add_warp(uint32_t *h, bool in, uint32_t bin) {
  const uint32_t key = in ? bin : 0xFFFFFFFFu;
  const uint32_t m = __match_any_sync(0xFFFFFFFFu, key);
  if (in && (int)(threadIdx.x & 31) == __ffs(m) - 1) atomicAdd(&h[bin], (uint32_t)__popc(m));
}
}  // namespace echo

namespace echo {
// Exclusive prefix of f(0..n-1) into pre[0..n] (pre[n] = total), computed by the
// whole block in parallel (every thread loads its own value; no serial loop over
// global loads).  Every thread of the block must call it; it ends with a barrier.
template <typename F>
__device__ __forceinline__ void block_prefix(int n, F f, int32_t *pre) {
  __shared__ int32_t bp_warp[32];
  __shared__ int32_t bp_carry;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  if (n <= 32) {                                   // a batch of requests: one warp, one barrier
    if (wid == 0) {
      const int v = lane < n ? f(lane) : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane < n) pre[lane] = x - v;
      if (lane == 31) pre[n] = x;
    }
    __syncthreads();
    return;
  }
  if (threadIdx.x == 0) bp_carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int v = i < n ? f(i) : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) bp_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int w = lane < nw ? bp_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      bp_warp[lane] = w;
    }
    __syncthreads();
    const int incl = x + (wid > 0 ? bp_warp[wid - 1] : 0);
    const int carry = bp_carry;
    if (i < n) pre[i] = carry + incl - v;
    __syncthreads();
    if (threadIdx.x == 0) bp_carry = carry + bp_warp[nw - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) pre[n] = bp_carry;
  __syncthreads();
}
}  // namespace echo
