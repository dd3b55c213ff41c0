// Sparse MLA decode attention over the selected cache slots (sm_103a).
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// "Problem and motivation": after the indexer selects the top-2048 tokens, MLA
// attention runs over their cached latent vectors (576 wide; the first 512 dims are
// the values).  Per request b and head h:
//   logit_j = scale * q[b,h,:] . c_j ;  out = softmax(logit) . c[:, :512] ;  lse.
//
// Split over the selected list: each CTA takes 256 consecutive entries of one
// request and 16 heads, streams the gathered rows through shared memory 32 at a
// time with an online softmax, and writes (o, m, l) partials; a combine kernel
// merges the splits in a fixed order.  The result depends only on the rows and
// their order in slot_idx, so attention over the cache is bitwise identical to
// attention over any buffer holding the same rows in the same order.

#include <algorithm>
#include <atomic>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace echo {

constexpr int MS_SPLIT = 256;   // selected entries per CTA
constexpr int MS_CHUNK = 32;    // rows per shared-memory chunk
constexpr int MS_HEADS = 16;    // heads per CTA
constexpr int MS_THREADS = 256;

struct MlaPart {
  float *o;   // [B, S, Hq, 512]
  float *ml;  // [B, S, Hq, 2]
};

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void __launch_bounds__(MS_THREADS)
    mla_split_kernel(const T *q, const T *kv, int kv_rows, const int32_t *slot_idx, int Hq, int k, float scale,
                     MlaPart part) {
  extern __shared__ float smf[];
  float *qs = smf;                                   // [16][576]
  float *cs = qs + MS_HEADS * KV_W;                  // [32][576]
  float *os = cs + MS_CHUNK * KV_W;                  // [16][512]
  float *lg = os + MS_HEADS * V_W;                   // [16][32]
  float *mrun = lg + MS_HEADS * MS_CHUNK;            // [16]
  float *lrun = mrun + MS_HEADS;                     // [16]
  float *corr = lrun + MS_HEADS;                     // [16]
  __shared__ int32_t slots[MS_CHUNK];

  const int s = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int S = gridDim.x;
  const int h0 = hg * MS_HEADS;
  const int nh = min(MS_HEADS, Hq - h0);
  const int tid = threadIdx.x;
  const int j0 = s * MS_SPLIT, j1 = min(k, j0 + MS_SPLIT);

  for (int i = tid; i < MS_HEADS * KV_W; i += MS_THREADS) {
    const int h = i / KV_W, d = i % KV_W;
    qs[i] = h < nh ? to_f(q[((int64_t)b * Hq + h0 + h) * KV_W + d]) : 0.f;
  }
  for (int i = tid; i < MS_HEADS * V_W; i += MS_THREADS) os[i] = 0.f;
  if (tid < MS_HEADS) { mrun[tid] = -INFINITY; lrun[tid] = 0.f; }

  for (int c0 = j0; c0 < j1; c0 += MS_CHUNK) {
    __syncthreads();
    if (tid < MS_CHUNK) {
      const int j = c0 + tid;
      int32_t g = j < j1 ? slot_idx[(int64_t)b * k + j] : -1;
      if (g >= kv_rows) g = -1;
      slots[tid] = g;
    }
    __syncthreads();
    for (int i = tid; i < MS_CHUNK * KV_W; i += MS_THREADS) {
      const int r = i / KV_W, d = i % KV_W;
      const int32_t g = slots[r];
      cs[i] = g >= 0 ? to_f(kv[(int64_t)g * KV_W + d]) : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < MS_HEADS * MS_CHUNK; i += MS_THREADS) {
      const int h = i / MS_CHUNK, r = i % MS_CHUNK;
      float acc = 0.f;
      const float *qh = qs + h * KV_W, *cr = cs + r * KV_W;
      for (int d = 0; d < KV_W; ++d) acc = fmaf(qh[d], cr[d], acc);
      lg[i] = (slots[r] >= 0 && h < nh) ? acc * scale : -INFINITY;
    }
    __syncthreads();
    if (tid < MS_HEADS) {
      float mx = mrun[tid];
      for (int r = 0; r < MS_CHUNK; ++r) mx = fmaxf(mx, lg[tid * MS_CHUNK + r]);
      float sum = 0.f;
      for (int r = 0; r < MS_CHUNK; ++r) {
        const float x = lg[tid * MS_CHUNK + r];
        const float p = (x == -INFINITY) ? 0.f : expf(x - mx);
        lg[tid * MS_CHUNK + r] = p;
        sum += p;
      }
      const float c = (mrun[tid] == -INFINITY) ? 0.f : expf(mrun[tid] - mx);
      corr[tid] = c;
      lrun[tid] = lrun[tid] * c + sum;
      mrun[tid] = mx;
    }
    __syncthreads();
    for (int i = tid; i < MS_HEADS * V_W; i += MS_THREADS) {
      const int h = i / V_W, d = i % V_W;
      float acc = os[i] * corr[h];
      const float *p = lg + h * MS_CHUNK;
      for (int r = 0; r < MS_CHUNK; ++r) acc = fmaf(p[r], cs[r * KV_W + d], acc);
      os[i] = acc;
    }
  }
  __syncthreads();
  for (int i = tid; i < nh * V_W; i += MS_THREADS) {
    const int h = i / V_W, d = i % V_W;
    part.o[(((int64_t)b * S + s) * Hq + h0 + h) * V_W + d] = os[i];
  }
  if (tid < nh) {
    part.ml[(((int64_t)b * S + s) * Hq + h0 + tid) * 2 + 0] = mrun[tid];
    part.ml[(((int64_t)b * S + s) * Hq + h0 + tid) * 2 + 1] = lrun[tid];
  }
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Merge the splits of one (request, head) in split order.
template <typename T>
__global__ void mla_combine_kernel(MlaPart part, int S, int Hq, T *out, float *lse) {
  const int h = blockIdx.x, b = blockIdx.y;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, part.ml[(((int64_t)b * S + s) * Hq + h) * 2]);
  float Lsum = 0.f;
  for (int s = 0; s < S; ++s) {
    const float m = part.ml[(((int64_t)b * S + s) * Hq + h) * 2];
    if (m != -INFINITY) Lsum += expf(m - M) * part.ml[(((int64_t)b * S + s) * Hq + h) * 2 + 1];
  }
  for (int d = threadIdx.x; d < V_W; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) {
      const float m = part.ml[(((int64_t)b * S + s) * Hq + h) * 2];
      if (m != -INFINITY) acc += expf(m - M) * part.o[(((int64_t)b * S + s) * Hq + h) * V_W + d];
    }
    out[((int64_t)b * Hq + h) * V_W + d] = from_f<T>(Lsum > 0.f ? acc / Lsum : 0.f);
  }
  if (threadIdx.x == 0) lse[(int64_t)b * Hq + h] = Lsum > 0.f ? M + logf(Lsum) : -INFINITY;
}

static int mla_splits(int k) { return (k + MS_SPLIT - 1) / MS_SPLIT; }

// ===================================================== bf16 tensor-core path ==
// CTA = (request b, split s of 256 selected entries), all 128 heads.
//   phase 1  S[128 x 256] = Q . C^T over nine 64-dim chunks: Q chunk by TMA,
//            gathered C chunk by cp.async into the 128-byte-swizzled K-major
//            layout; tcgen05.mma kind::f16 M=128 N=256 K=16, f32 in TMEM.
//   softmax  one thread per head row and half of the columns reads its logits
//            from TMEM and writes the bf16 probabilities P back into TMEM over
//            the logits it has read (tokens 0-127 -> columns 0-63, 128-255 ->
//            columns 128-191; two per 32-bit column).
//   phase 2  O = P . V in eight blocks of 64 value dims: the MMA takes P from
//            TMEM and a 64-token x 64-dim V stage (MN-major) from shared memory,
//            accumulating into one of two 64-column TMEM buffers (columns 64-127
//            and 192-255), so block j's epilogue overlaps block j+1's MMAs; the
//            whole phase-1 region is a 12-stage V ring (96 KB in flight).
//            The epilogue writes O / l as bf16 partials, plus (m, l) per head.
// Warps 0-3 load (cp.async), run half of the softmax and the epilogues; warps 5-8
// the other half of the softmax; warp 4 issues the MMAs from one thread.  256 TMEM
// columns and ~100 KB shared memory per CTA: two CTAs per SM overlap each other's
// phases.
constexpr int TC_T = 256;                 // selected entries per CTA
constexpr int TC_THREADS = 288;         // warps 0-3 loads/softmax/epilogue, 4 MMA, 5-8 softmax
constexpr int TC_QCH = 128 * 128;         // Q chunk bytes (128 heads x 64 dims)
constexpr int TC_KCH = TC_T * 128;        // C chunk bytes (256 rows x 64 dims)
constexpr int TC_STAGE = TC_QCH + TC_KCH; // 48 KB
constexpr int TC_VROWS = 64;              // tokens per V stage (four K-steps)
constexpr int TC_VCH = TC_VROWS * 128;    // V stage bytes (64 tokens x 64 dims)
constexpr int TC_VST = 12;                // V ring stages
constexpr int TC_SPB = TC_T / TC_VROWS;   // stages per 64-dim output block (4)
constexpr int TC_NV = 8 * TC_SPB;         // V stages per CTA (eight blocks)
constexpr int TC_REGION = 2 * TC_STAGE;   // 96 KB, phase 1 ring / V ring
static_assert(TC_VST * TC_VCH <= TC_REGION, "the V ring reuses the phase-1 region");
static_assert(TC_VST - 2 <= 10, "cp_async_wait_upto covers the ring");

struct TcShared {
  uint64_t full[2], empty[2], qfull[2];
  uint64_t s_full, p_full, o_full[2], o_empty[2];
  uint64_t vfull[TC_VST], vempty[TC_VST];
  uint32_t tmem_base;
  int fail;                                // set when a bounded wait gave up
  int32_t slots[TC_T];
  uint32_t vmask[TC_T / 32];
  float mpart[2][128], lpart[2][128];      // per head: max and sum of each half of the columns
};
constexpr size_t TC_SMEM = 1024 + TC_REGION + sizeof(TcShared);

struct TcPart {
  __nv_bfloat16 *o;   // [B, S, 128, 512] normalised partial outputs
  float *ml;          // [B, S, 128, 2]
};

// TMEM column of the bf16 pair holding tokens t, t+1 of P (t even)
__device__ __forceinline__ uint32_t p_col(int t) { return (uint32_t)((t >> 1) + (t >= TC_T / 2 ? TC_T / 4 : 0)); }

// 16 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// tcgen05.mma kind::f16 with A (M x 16) read from TMEM at a_tmem
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Wait until at most n (0..10) of this thread's cp.async groups are pending.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    case 7: cp_async_wait<7>(); break;
    case 8: cp_async_wait<8>(); break;
    case 9: cp_async_wait<9>(); break;
    default: cp_async_wait<10>(); break;
  }
}

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk16) {
  // byte offset of 16-byte chunk `chunk16` of row `row` in a 128B-swizzled
  // K-major tile whose rows are 128 bytes apart
  return (row >> 3) * 1024 + (row & 7) * 128 + ((chunk16 ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(TC_THREADS, 2)
    mla_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __nv_bfloat16 *kv, int kv_rows,
                  const int32_t *slot_idx, int k, float scale, TcPart part) {
  extern __shared__ unsigned char tc_raw[];
  unsigned char *R = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
  TcShared &S = *reinterpret_cast<TcShared *>(R + TC_REGION);
  unsigned char *V = R;                       // phase 2: V ring (12 x 8 KB)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, b = blockIdx.y, nsplit = gridDim.x;
  const int j0 = s * TC_T;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.full[i], 128);
      mbar_init(&S.empty[i], 1);
      mbar_init(&S.qfull[i], 1);
    }
    for (int i = 0; i < TC_VST; ++i) {
      mbar_init(&S.vfull[i], 128);
      mbar_init(&S.vempty[i], 1);
    }
    S.fail = 0;
    mbar_init(&S.s_full, 1);
    mbar_init(&S.p_full, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.o_full[i], 1);
      mbar_init(&S.o_empty[i], 128);
    }
    fence_mbar_init();
  }
  for (int i = tid; i < TC_T; i += TC_THREADS) {
    const int j = j0 + i;
    int32_t g = j < k ? slot_idx[(int64_t)b * k + j] : -1;
    g = (g >= 0 && g < kv_rows) ? g : -1;
    S.slots[i] = g;
    const uint32_t bal = __ballot_sync(0xffffffffu, g >= 0);   // whole warps: 160 and 256 are multiples of 32
    if (lane == 0) S.vmask[i >> 5] = bal;
  }
  if (warp == 4) {
    tmem_alloc(&S.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool ok = true;

  // Softmax of one half of the 256 columns (half 0: warps 0-3, half 1: warps 5-8) for
  // head row (warp & 3) * 32 + lane: row max and sum exchanged between the halves
  // through shared memory (named barriers 1 and 2 of the 256 softmax threads); writes
  // bf16 P for its columns and arrives on p_full.  Returns the row's max and sum.
  auto softmax_half = [&](int half, float &m_out, float &l_out) {
    const int hr = (warp & 3) * 32 + lane;
    const uint32_t tr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t *vmask = S.vmask;             // validity of the 256 entries (set before the first barrier)
    const int cb = half * (TC_T / 2), ce = cb + TC_T / 2;
    float m = -INFINITY;
    for (int c0 = cb; c0 < ce; c0 += 64) {       // two TMEM loads per wait
      uint32_t r[32], r2[32];
      tmem_ld32(tr + c0, r);
      tmem_ld32(tr + c0 + 32, r2);
      tmem_wait_ld();
      const uint32_t vm = vmask[c0 >> 5], vm2 = vmask[(c0 >> 5) + 1];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if ((vm >> j) & 1u) m = fmaxf(m, __uint_as_float(r[j]));
        if ((vm2 >> j) & 1u) m = fmaxf(m, __uint_as_float(r2[j]));
      }
    }
    S.mpart[half][hr] = m;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    m = fmaxf(S.mpart[0][hr], S.mpart[1][hr]);
    const float c2 = scale * 1.4426950408889634f;      // scale * log2(e)
    const float mc = m * c2;
    float l = 0.f;
    // 32 probabilities -> 16 bf16 pairs -> 16 TMEM columns of this row, over logits
    // this thread has already read (p_col(c0) < c0 within its half)
    auto write_p = [&](int c0, const uint32_t (&r)[32], uint32_t vm) {
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = ((vm >> j) & 1u) ? exp2f(fmaf(__uint_as_float(r[j]), c2, -mc)) : 0.f;
        const float p1 = ((vm >> (j + 1)) & 1u) ? exp2f(fmaf(__uint_as_float(r[j + 1]), c2, -mc)) : 0.f;
        l += p0 + p1;
        __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
        pk[j >> 1] = *reinterpret_cast<uint32_t *>(&v2);
      }
      tmem_st16(tr + p_col(c0), pk);
    };
    for (int c0 = cb; c0 < ce; c0 += 64) {       // two TMEM loads per wait
      uint32_t r[32], r2[32];
      tmem_ld32(tr + c0, r);
      tmem_ld32(tr + c0 + 32, r2);
      tmem_wait_ld();
      write_p(c0, r, vmask[c0 >> 5]);
      write_p(c0 + 32, r2, vmask[(c0 >> 5) + 1]);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&S.p_full);
    S.lpart[half][hr] = l;
    asm volatile("bar.sync 2, 256;" ::: "memory");
    m_out = m;
    l_out = S.lpart[0][hr] + S.lpart[1][hr];
  };

  if (warp < 4) {
    // ------------------------------------------------ phase 1 loads --
    const int row_base = tid;                          // 128 threads
    for (int dc = 0; dc < 9; ++dc) {
      const int st = dc & 1;
      if (!mbar_wait(&S.empty[st], ((dc >> 1) & 1) ^ 1)) { ok = false; break; }
      unsigned char *qb = R + st * TC_STAGE, *kb = qb + TC_QCH;
      if (tid == 0) {
        mbar_arrive_expect_tx(&S.qfull[st], TC_QCH);
        tma_load_2d(qb, &qmap, &S.qfull[st], dc * 64, b * 128);
      }
      // 256 rows x 8 chunks: thread handles chunk (tid & 7) of rows (tid >> 3) + 16 i
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int r = (row_base >> 3) + 16 * i, c = row_base & 7;
        const int32_t g = S.slots[r];
        const __nv_bfloat16 *src = kv + (int64_t)(g >= 0 ? g : 0) * KV_W + dc * 64 + c * 8;
        cp_async_16(kb + sw128(r, c), src, g >= 0 ? 16u : 0u);
      }
      cp_async_commit();
      if (dc > 0) {
        cp_async_wait<1>();
        fence_proxy_async_smem();
        mbar_arrive(&S.full[(dc - 1) & 1]);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    mbar_arrive(&S.full[8 & 1]);

    // ------------------------------------------------------ softmax --
    if (!mbar_wait(&S.s_full, 0)) ok = false;
    tc_fence_after();
    // V loads of the first stages can start: phase 1 no longer reads smem
    auto load_v = [&](int vc) {                        // block vc / TC_SPB, tokens (vc % TC_SPB) * 64
      const int st = vc % TC_VST, j = vc / TC_SPB, r0 = (vc % TC_SPB) * TC_VROWS;
      unsigned char *vb = V + st * TC_VCH;
#pragma unroll
      for (int i = 0; i < TC_VROWS * 8 / 128; ++i) {
        const int idx = tid + 128 * i;                 // rows x 8 chunks of 16 B (64 dims)
        const int r = idx >> 3, c = idx & 7;
        const int32_t g = S.slots[r0 + r];
        const __nv_bfloat16 *src = kv + (int64_t)(g >= 0 ? g : 0) * KV_W + j * 64 + c * 8;
        cp_async_16(vb + r * 128 + ((c ^ (r & 7)) << 4), src, g >= 0 ? 16u : 0u);
      }
      cp_async_commit();
    };
    for (int vc = 0; vc < TC_VST; ++vc) load_v(vc);
    const int h = tid;                                  // head row = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    float m = 0.f, l = 0.f;
    softmax_half(0, m, l);

    // ------------------------------------------- phase 2 loads + epilogue --
    // epilogue of 64-dim block j: O / l from its TMEM buffer to bf16 partials, stored
    // in groups of 8 dims with heads innermost ([b][s][dim/8][head][8]), so the 32
    // heads of a warp write one contiguous 512-byte run per store
    auto epilogue = [&](int j) {
      if (!mbar_wait(&S.o_full[j & 1], (j >> 1) & 1)) ok = false;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16 *dst = part.o + (((int64_t)b * nsplit + s) * 64 + j * 8) * 128 * 8 + (int64_t)h * 8;
      uint32_t r[32], r2[32];
      const uint32_t ob = trow + ((j & 1) ? 192u : 64u);
      tmem_ld32(ob, r);
      tmem_ld32(ob + 32, r2);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&S.o_empty[j & 1]);                  // the values are in registers
      auto store_o = [&](int c0, const uint32_t (&v)[32]) {
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 32; q += 2) {
          __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(v[q]) * inv, __uint_as_float(v[q + 1]) * inv);
          pk[q >> 1] = *reinterpret_cast<uint32_t *>(&v2);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)                    // dims 64 j + c0 + 8q .. + 7
          *reinterpret_cast<uint4 *>(dst + (int64_t)((c0 >> 3) + q) * 128 * 8) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      };
      store_o(0, r);
      store_o(32, r2);
    };
    for (int vc = 0; vc < TC_NV; ++vc) {
      // stage vc was issued earlier; wait for it (later groups may stay in flight):
      // groups issued after stage vc so far: vc+1 .. vc+TC_VST-2 (refills lag one iteration)
      cp_async_wait_upto(max(0, min(TC_VST - 2, TC_NV - 1 - vc)));
      fence_proxy_async_smem();
      mbar_arrive(&S.vfull[vc % TC_VST]);
      // refill the buffer of the stage delivered one iteration ago (likely consumed
      // by now), not the one just delivered: the other stages stay in flight
      if (vc >= 1 && vc - 1 + TC_VST < TC_NV) {
        const int pv = vc - 1;
        if (!mbar_wait(&S.vempty[pv % TC_VST], (pv / TC_VST) & 1)) { ok = false; }
        load_v(pv + TC_VST);
      }
      // block j = vc / TC_SPB is delivered: write out the block before it
      if (vc % TC_SPB == TC_SPB - 1 && vc >= TC_SPB) epilogue(vc / TC_SPB - 1);
    }
    epilogue(TC_NV / TC_SPB - 1);
    part.ml[(((int64_t)b * nsplit + s) * 128 + h) * 2 + 0] = m == -INFINITY ? -INFINITY : m * scale;
    part.ml[(((int64_t)b * nsplit + s) * 128 + h) * 2 + 1] = l;
  } else if (warp > 4) {
    // ------------------------------------------- second half of the softmax --
    if (!mbar_wait(&S.s_full, 0)) ok = false;
    tc_fence_after();
    float m = 0.f, l = 0.f;
    softmax_half(1, m, l);
  } else if (lane == 0) {
    // ------------------------------------------------------------- MMA --
    constexpr uint32_t id1 = instr_desc(FMT_BF16, FMT_BF16, 0, 0, 128, TC_T);
    for (int dc = 0; dc < 9 && ok; ++dc) {
      const int st = dc & 1;
      if (!mbar_wait(&S.qfull[st], (dc >> 1) & 1) || !mbar_wait(&S.full[st], (dc >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const uint64_t ad = smem_desc(smem_u32(R + st * TC_STAGE), 16, 1024, LAYOUT_SW128);
      const uint64_t bd = smem_desc(smem_u32(R + st * TC_STAGE + TC_QCH), 16, 1024, LAYOUT_SW128);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, id1, (dc | kk) ? 1u : 0u);
      mma_commit(&S.empty[st]);
    }
    mma_commit(&S.s_full);
    if (ok && !mbar_wait(&S.p_full, 0)) ok = false;
    tc_fence_after();
    // block j: O_j[128 x 64] = P[128 x 256] . V[256 x 64 dims of block j]; P from TMEM
    constexpr uint32_t id2 = instr_desc(FMT_BF16, FMT_BF16, 0, 1, 128, 64);
    for (int j = 0; j < TC_NV / TC_SPB && ok; ++j) {
      if (j >= 2) {                                    // this buffer's previous block is written out
        if (!mbar_wait(&S.o_empty[j & 1], ((j >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
      }
      const uint32_t d = tmem + ((j & 1) ? 192u : 64u);
      for (int s4 = 0; s4 < TC_SPB && ok; ++s4) {
        const int vc = j * TC_SPB + s4, st = vc % TC_VST;
        if (!mbar_wait(&S.vfull[st], (vc / TC_VST) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < TC_VROWS / 16; ++kk) {
          const int t0 = s4 * TC_VROWS + kk * 16;      // tokens of this K-step
          const uint64_t bd = smem_desc(smem_u32(V + st * TC_VCH + kk * 16 * 128), TC_VCH, 1024, LAYOUT_SW128);
          mma_f16_ts(d, tmem + p_col(t0), bd, id2, (s4 | kk) ? 1u : 0u);
        }
        mma_commit(&S.vempty[st]);
      }
      mma_commit(&S.o_full[j & 1]);
    }
  }
  if (!ok) S.fail = 1;                                // a bounded wait gave up
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 256);
  if (S.fail && tid < 128) {
    // this split's partial is not valid: the combine skips a split whose max is -inf
    part.ml[(((int64_t)b * nsplit + s) * 128 + tid) * 2 + 0] = -INFINITY;
    part.ml[(((int64_t)b * nsplit + s) * 128 + tid) * 2 + 1] = 0.f;
  }
}

// Merge the bf16 partials of one (request, head) in split order.  A block of 256
// threads covers 4 heads; each thread produces 8 consecutive output dims.
template <int NSMAX>
__global__ void __launch_bounds__(256) mla_tc_combine_kernel(TcPart part, int nsplit, __nv_bfloat16 *out,
                                                             float *lse, int drop) {
  // block: two groups of 8 dims (j) x 128 heads; warp w: heads 32 (w & 3) + lane of group
  // j = 2 blockIdx.x + (w >> 2), so every load of a partial is a contiguous 512-byte run
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = 32 * (warp & 3) + lane;
  const int j = 2 * blockIdx.x + (warp >> 2);
  const float *ml = part.ml + ((int64_t)b * nsplit * 128 + h) * 2;                  // split s at ml[s * 256]
  const __nv_bfloat16 *po = part.o + (((int64_t)b * nsplit * 64 + j) * 128 + h) * 8;  // split s at po[s * 65536]
  float M = -INFINITY;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float Lsum = 0.f;
  auto add = [&](float m, float l, const uint4 &v) {
    const float w = (m == -INFINITY || l <= 0.f) ? 0.f : expf(m - M) * l;
    Lsum += w;
    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[2 * q] = fmaf(w, __bfloat162float(p2[q].x), acc[2 * q]);
      acc[2 * q + 1] = fmaf(w, __bfloat162float(p2[q].y), acc[2 * q + 1]);
    }
  };
  if (nsplit <= NSMAX) {
    // every split's (m, l) and partial issued together, then merged in split order
    float m[NSMAX], l[NSMAX];
    uint4 v[NSMAX];
#pragma unroll
    for (int s = 0; s < NSMAX; ++s) {
      if (s < nsplit) {
        m[s] = __ldg(ml + (int64_t)s * 256);
        l[s] = __ldg(ml + (int64_t)s * 256 + 1);
        v[s] = __ldg(reinterpret_cast<const uint4 *>(po + (int64_t)s * 64 * 128 * 8));
      }
    }
#pragma unroll
    for (int s = 0; s < NSMAX; ++s)
      if (s < nsplit) M = fmaxf(M, m[s]);
#pragma unroll
    for (int s = 0; s < NSMAX; ++s)
      if (s < nsplit) add(m[s], l[s], v[s]);
  } else {
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldg(ml + (int64_t)s * 256));
    for (int s = 0; s < nsplit; ++s)
      add(__ldg(ml + (int64_t)s * 256), __ldg(ml + (int64_t)s * 256 + 1),
          __ldg(reinterpret_cast<const uint4 *>(po + (int64_t)s * 64 * 128 * 8)));
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  uint4 o;
  __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) o2[q] = __floats2bfloat162_rn(acc[2 * q] * inv, acc[2 * q + 1] * inv);
  *reinterpret_cast<uint4 *>(out + ((int64_t)b * 128 + h) * V_W + 8 * j) = o;
  // the per-split logits are scaled, so M and lse are in logit units
  if (j == 0) lse[(int64_t)b * 128 + h] = Lsum > 0.f ? M + logf(Lsum) : -INFINITY;
  if (drop) {
    // The partials are dead once merged: their L2 lines are dropped without being
    // written back, so the next kernels' streams do not pay for evicting them.  Each
    // split's chunks of this warp are 512 contiguous bytes (4 lines), read only here;
    // lane i drops line i & 3 of splits (i >> 2), (i >> 2) + 8, ...
    __syncwarp();
    const __nv_bfloat16 *p0 = po - lane * 8;
    for (int s = lane >> 2; s < nsplit; s += 8) {
      const __nv_bfloat16 *line = p0 + (int64_t)s * 64 * 128 * 8 + (lane & 3) * 64;
      asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
    }
  }
}

// Q as a 2-D bf16 tensor [rows, 576] with a [128 rows x 64 dims] box, 128-byte swizzle.
static bool make_q_map(CUtensorMap *m, const void *base, uint64_t rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  const cuuint64_t dims[2] = {KV_W, rows};
  const cuuint64_t strides[1] = {KV_W * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace echo

using namespace echo;

extern "C" size_t echo_sparse_mla_workspace_bytes(int32_t B, int32_t Hq, int32_t k) {
  if (B <= 0 || Hq <= 0 || k <= 0) return 0;
  const size_t S = (size_t)mla_splits(k);
  return (size_t)B * S * Hq * (V_W + 2) * sizeof(float);
}

extern "C" echo_status_t echo_sparse_mla_decode(const void *q, const void *kv, int32_t kv_rows, int32_t dtype,
                                                const int32_t *slot_idx, int32_t B, int32_t Hq, int32_t k,
                                                float scale, void *out, float *lse, void *workspace,
                                                size_t workspace_bytes, echo_stream_t stream) {
  if (!q || !kv || !slot_idx || !out || !lse || !workspace || B <= 0 || Hq <= 0 || k <= 0 || kv_rows <= 0)
    return ECHO_ERR_INVALID_ARG;
  if (Hq > 128) return ECHO_ERR_UNSUPPORTED;
  if (workspace_bytes < echo_sparse_mla_workspace_bytes(B, Hq, k)) return ECHO_ERR_INVALID_ARG;
  const int S = mla_splits(k);
  MlaPart part;
  part.o = reinterpret_cast<float *>(workspace);
  part.ml = part.o + (size_t)B * S * Hq * V_W;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t smem = sizeof(float) * (MS_HEADS * KV_W + MS_CHUNK * KV_W + MS_HEADS * V_W + MS_HEADS * MS_CHUNK +
                                       3 * MS_HEADS);
  dim3 grid(S, (Hq + MS_HEADS - 1) / MS_HEADS, B);
  if (dtype == ECHO_F32) {
    ECHO_CUDA_OK(cudaFuncSetAttribute(mla_split_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    mla_split_kernel<float><<<grid, MS_THREADS, smem, st>>>((const float *)q, (const float *)kv, kv_rows, slot_idx,
                                                            Hq, k, scale, part);
    ECHO_LAUNCH_OK();
    mla_combine_kernel<float><<<dim3(Hq, B), 128, 0, st>>>(part, S, Hq, (float *)out, lse);
  } else if (dtype == ECHO_BF16) {
    if (Hq != 128) return ECHO_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) return ECHO_ERR_INVALID_ARG;
    const int ns = (k + TC_T - 1) / TC_T;
    if (ns > 64) return ECHO_ERR_UNSUPPORTED;
    TcPart tp;
    tp.o = reinterpret_cast<__nv_bfloat16 *>(workspace);
    tp.ml = reinterpret_cast<float *>(tp.o + (size_t)B * ns * 128 * 512);
    CUtensorMap qmap;
    if (!make_q_map(&qmap, q, (uint64_t)B * 128)) return ECHO_ERR_CUDA;
    ECHO_CUDA_OK(cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM));
    mla_tc_kernel<<<dim3(ns, B), TC_THREADS, TC_SMEM, st>>>(qmap, (const __nv_bfloat16 *)kv, kv_rows, slot_idx, k,
                                                            scale, tp);
    ECHO_LAUNCH_OK();
    // the partials' lines are dropped after the merge when they are whole lines
    const int drop = (reinterpret_cast<uintptr_t>(workspace) & 127) == 0;
    mla_tc_combine_kernel<8><<<dim3(32, B), 256, 0, st>>>(tp, ns, (__nv_bfloat16 *)out, lse, drop);
  } else {
    return ECHO_ERR_UNSUPPORTED;
  }
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

// ----------------------------------------------- variant without allocation --
// For callers that may not allocate device memory: the split partials go to a
// scratch array compiled into the library instead of a caller workspace.  Every
// GPU that loads the library holds the array until the process exits.
namespace {
static __device__ __align__(256) unsigned char g_mla_noalloc_scratch[ECHO_MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// device address of the array, per device; host threads that make their first call
// on a device at the same time may both look it up, and both store the same value
std::atomic<void *> g_scratch_addr[kMaxDevices];
}  // namespace

extern "C" echo_status_t echo_sparse_mla_decode_noalloc(const void *q, const void *kv, int32_t kv_rows,
                                                        int32_t dtype, const int32_t *slot_idx, int32_t B,
                                                        int32_t Hq, int32_t k, float scale, void *out, float *lse,
                                                        echo_stream_t stream) {
  if (!q || !kv || !slot_idx || !out || !lse || B <= 0 || Hq <= 0 || k <= 0 || kv_rows <= 0)
    return ECHO_ERR_INVALID_ARG;
  const size_t need = echo_sparse_mla_workspace_bytes(B, Hq, k);
  if (need == 0) return ECHO_ERR_INVALID_ARG;
  if (need > (size_t)ECHO_MLA_NOALLOC_SCRATCH_BYTES) return ECHO_ERR_SCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ECHO_ERR_CUDA;
  void *scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!scratch) {
    // host code cannot use the array's name as a device address: look it up once
    // per device, with that device current
    if (cudaGetSymbolAddress(&scratch, g_mla_noalloc_scratch) != cudaSuccess || !scratch) return ECHO_ERR_CUDA;
    g_scratch_addr[dev].store(scratch, std::memory_order_release);
  }
  return echo_sparse_mla_decode(q, kv, kv_rows, dtype, slot_idx, B, Hq, k, scale, out, lse, scratch,
                                (size_t)ECHO_MLA_NOALLOC_SCRATCH_BYTES, stream);
}
