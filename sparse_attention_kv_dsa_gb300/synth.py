"""Seeded synthetic inputs for the decode hot path.

This module only draws numbers.  It holds none of the method's arithmetic (no
scoring, selection, cache policy or attention), so that the tests can hand the
very same tensors to the CUDA library and to the CPU oracle.

Workloads stand in for the pages' long-context traces (InfiniteBench 80K-100K
inputs, ShareGPT requests): no dataset or trained weights are used.

Value recipes
  * indexer keys / queries: integers on [-G, G] times 2^-3 (G = 8 for the FP8
    workloads, 4 for the float32 one).  Every value is exact in FP8 e4m3, every
    product is exact in float32, and the 64-head weighted sum stays below 2^24
    units of 2^-10, so float32 scores are exact in any summation order.
  * head weights: {1..16} * 2^-4 (FP8 workloads) or {0.25, 0.5} (float32 one).
  * query drift between steps: q <- clip(round(rho*q + sqrt(1-rho^2)*sigma*eps)),
    eps ~ N(0, 1), sigma = standard deviation of the uniform grid.
  * MLA latents and MLA queries: N(0, 1), rounded to bf16 (float32 for the tiny one).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

MASK64 = (1 << 64) - 1


def mix_seed(*parts: int) -> int:
    """splitmix64 over the parts: independent substreams per (config, layer,
    request, step, purpose)."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x + (int(p) & MASK64) + 0x9E3779B97F4A7C15) & MASK64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        x = z ^ (z >> 31)
    return x & 0x7FFFFFFFFFFFFFFF


def gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


@dataclass
class Workload:
    """One synthetic workload (sizes of the pages' decode/prefill settings)."""
    name: str
    cfg_id: int
    layers: int
    batch: int
    ctx: list                    # per-request context length at the first step
    h_idx: int                   # indexer heads
    d_idx: int                   # indexer head dim
    grid: int                    # indexer values are integers in [-grid, grid] * 2^-3
    w_values: list               # head weights are drawn from this list
    topk: int
    h_q: int                     # MLA query heads
    kv_fp32: bool                # latents in float32 (else bf16)
    n_gpu: int                   # GPU slots per layer
    n_host: int                  # host pool rows per layer
    steps: int
    rho: float                   # query drift
    cap_max: int
    cap_div: int
    alpha: float = 0.5
    cap_sweep: list = field(default_factory=list)
    prefill_chunk: int = 0
    prefill_blocks: list = field(default_factory=list)
    kv_width: int = 576          # values per cached token row (576: MLA latent; 2d: a KV head's key, value)
    kv_heads: int = 0            # 0: MLA; n: GQA, every request split into n (request, KV head) groups

    @property
    def seed(self) -> int:
        return 0xEC40 + self.cfg_id

    @property
    def max_ctx(self) -> int:
        return max(self.ctx) + self.steps + 8

    @property
    def host_base(self) -> list:
        """Each request owns a contiguous host range, in request order."""
        base, out = 0, []
        for b in range(self.batch):
            out.append(base)
            base += self.ctx[b] + self.steps + 8
        return out

    @property
    def q_width(self) -> int:
        """Values per attention query head: 576 (MLA) or the KV head's dimension d."""
        return self.kv_width // 2 if self.kv_heads else self.kv_width

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(float(self.q_width))


def _ctx_uniform(seed: int, n: int, lo: int, hi: int) -> list:
    g = gen(mix_seed(seed, 0xC7C))
    return [int(v) for v in torch.randint(lo, hi + 1, (n,), generator=g).tolist()]


def workloads() -> dict:
    """The synthetic workloads, keyed by name."""
    w16 = [i / 16.0 for i in range(1, 17)]
    out = {}
    out["tiny-fp32-b1-ctx4k"] = Workload(
        name="tiny-fp32-b1-ctx4k", cfg_id=1, layers=1, batch=1, ctx=[4096], h_idx=4, d_idx=64,
        grid=4, w_values=[0.25, 0.5], topk=256, h_q=16, kv_fp32=True, n_gpu=1024, n_host=8192,
        steps=8, rho=0.9, cap_max=512, cap_div=0)
    out["decode-b8-ctx64k"] = Workload(
        name="decode-b8-ctx64k", cfg_id=2, layers=1, batch=8, ctx=[65536] * 8, h_idx=64, d_idx=128,
        grid=8, w_values=w16, topk=2048, h_q=128, kv_fp32=False, n_gpu=200_000, n_host=2_000_000,
        steps=64, rho=0.97, cap_max=4096, cap_div=32)
    ctx3 = _ctx_uniform(0xEC40 + 3, 32, 80_000, 100_000)
    out["saturated-b32-ctx80k-100k-4layer"] = Workload(
        name="saturated-b32-ctx80k-100k-4layer", cfg_id=3, layers=4, batch=32, ctx=ctx3, h_idx=64,
        d_idx=128, grid=8, w_values=w16, topk=2048, h_q=128, kv_fp32=False, n_gpu=200_000,
        n_host=3_300_000, steps=256, rho=0.995, cap_max=4096, cap_div=32)
    out["lowlocality-b16-ctx100k"] = Workload(
        name="lowlocality-b16-ctx100k", cfg_id=4, layers=1, batch=16, ctx=[100_000] * 16, h_idx=64,
        d_idx=128, grid=8, w_values=w16, topk=2048, h_q=128, kv_fp32=False, n_gpu=110_000,
        n_host=2_000_000, steps=16, rho=math.sqrt(0.5), cap_max=4096, cap_div=0,
        cap_sweep=[0, 1024, 4096, 16384])
    # a model-sized stack: 61 layers (the pages' per-model metadata over per-layer size),
    # 8 requests of ShareGPT-like length, a GPU pool smaller than the context so every
    # layer evicts at the steady state
    ctx6 = _ctx_uniform(0xEC40 + 6, 8, 16_000, 24_000)
    out["model-61layer-b8-ctx20k"] = Workload(
        name="model-61layer-b8-ctx20k", cfg_id=6, layers=61, batch=8, ctx=ctx6, h_idx=64, d_idx=128, grid=8,
        w_values=w16, topk=2048, h_q=128, kv_fp32=False, n_gpu=65_536, n_host=sum(c + 128 + 8 for c in ctx6),
        steps=128, rho=0.97, cap_max=4096, cap_div=32)
    # a GQA layer with several KV heads: 16 requests x 8 KV heads (128 groups of 8 query
    # heads, d = 128), each group selecting its own top-2048 tokens
    ctx7 = _ctx_uniform(0xEC40 + 7, 16, 32_000, 48_000)
    g7 = gqa_workload("gqa-b16x8kv-ctx32k-48k-2layer", ctx=ctx7, kv_heads=8, group=8, head_dim=128, h_idx=64,
                      topk=2048, steps=64, rho=0.97, cfg_id=7)
    g7.layers, g7.n_gpu = 2, 128 * 2048 * 3
    out[g7.name] = g7
    out["prefill-chunk2048-ctx100k"] = Workload(
        name="prefill-chunk2048-ctx100k", cfg_id=5, layers=1, batch=1, ctx=[100_000], h_idx=64,
        d_idx=128, grid=8, w_values=w16, topk=2048, h_q=128, kv_fp32=False, n_gpu=200_000,
        n_host=2_000_000, steps=0, rho=0.9, cap_max=0, cap_div=32, prefill_chunk=2048,
        prefill_blocks=[256, 512])
    return out


def small_workload(name="small-b3", *, batch=None, ctx=(700, 1500, 333), h_idx=64, d_idx=128, grid=8,
                   topk=256, h_q=128, kv_fp32=False, n_gpu=2048, steps=4, rho=0.9, cap_max=64,
                   cap_div=0, w_values=None) -> Workload:
    """A small workload that the oracle finishes in seconds but that still spans
    several tiles and a ragged tail."""
    batch = len(ctx) if batch is None else batch
    assert batch == len(ctx)
    n_host = sum(c + steps + 8 for c in ctx) + 64
    return Workload(name=name, cfg_id=100, layers=1, batch=batch, ctx=list(ctx), h_idx=h_idx,
                    d_idx=d_idx, grid=grid, w_values=w_values or [i / 16.0 for i in range(1, 17)],
                    topk=topk, h_q=h_q, kv_fp32=kv_fp32, n_gpu=n_gpu, n_host=n_host, steps=steps,
                    rho=rho, cap_max=cap_max, cap_div=cap_div)


def gqa_workload(name="gqa-small", *, ctx=(700, 1500, 333), kv_heads=4, group=8, head_dim=128, h_idx=64,
                 d_idx=128, grid=8, topk=256, kv_fp32=False, n_gpu=4096, steps=4, rho=0.9, cfg_id=101) -> Workload:
    """A GQA layer with several KV heads: each request of context ctx[r] becomes kv_heads
    groups (request r, KV head h) = row r * kv_heads + h of every per-group tensor, each
    with its own indexer queries and keys, host rows of 2 * head_dim values and top-k;
    group's queries are the request's query heads h * group .. h * group + group - 1."""
    gctx = [c for c in ctx for _ in range(kv_heads)]
    n_host = sum(c + steps + 8 for c in gctx) + 64
    return Workload(name=name, cfg_id=cfg_id, layers=1, batch=len(gctx), ctx=gctx, h_idx=h_idx, d_idx=d_idx,
                    grid=grid, w_values=[i / 16.0 for i in range(1, 17)], topk=topk, h_q=group, kv_fp32=kv_fp32,
                    n_gpu=n_gpu, n_host=n_host, steps=steps, rho=rho, cap_max=0, cap_div=0,
                    kv_width=2 * head_dim, kv_heads=kv_heads)


# ---------------------------------------------------------------- draws ----
def grid_ints(seed: int, shape, grid: int, device="cpu") -> torch.Tensor:
    """Integers uniform on [-grid, grid] (int8)."""
    g = gen(seed, device)
    return torch.randint(-grid, grid + 1, tuple(shape), generator=g, device=device, dtype=torch.int8)


def grid_drift(seed: int, q_int: torch.Tensor, grid: int, rho: float) -> torch.Tensor:
    """AR(1) drift of grid integers, re-quantised onto the grid."""
    g = gen(seed, q_int.device)
    sigma = math.sqrt(((2 * grid + 1) ** 2 - 1) / 12.0)
    eps = torch.randn(q_int.shape, generator=g, device=q_int.device, dtype=torch.float64)
    x = rho * q_int.to(torch.float64) + math.sqrt(max(0.0, 1.0 - rho * rho)) * sigma * eps
    return torch.clamp(torch.round(x), -grid, grid).to(torch.int8)


def choice(seed: int, shape, values, device="cpu") -> torch.Tensor:
    g = gen(seed, device)
    idx = torch.randint(0, len(values), tuple(shape), generator=g, device=device)
    return torch.tensor(values, dtype=torch.float32, device=device)[idx]


def normal(seed: int, shape, dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    g = gen(seed, device)
    return torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32).to(dtype)


def grid_to_float(x_int: torch.Tensor) -> torch.Tensor:
    """Grid integers -> their real values (x * 2^-3), float32."""
    return x_int.to(torch.float32) * 0.125


def grid_to_fp8(x_int: torch.Tensor) -> torch.Tensor:
    """Grid integers -> FP8 e4m3 (exact on the grid)."""
    return grid_to_float(x_int).to(torch.float8_e4m3fn)


# ---------------------------------------------------- per-purpose streams ----
P_KEYS, P_QIDX, P_W, P_DRIFT, P_LAT, P_QMLA, P_NEWKV, P_NEWIK, P_PFQ, P_PFW, P_PFQMLA = range(1, 12)


def keys_for(wl: Workload, layer: int, b: int, L: int, device="cpu") -> torch.Tensor:
    return grid_ints(mix_seed(wl.seed, P_KEYS, layer, b), (L, wl.d_idx), wl.grid, device)


def qidx_initial(wl: Workload, layer: int, device="cpu") -> torch.Tensor:
    return grid_ints(mix_seed(wl.seed, P_QIDX, layer), (wl.batch, wl.h_idx, wl.d_idx), wl.grid, device)


def qidx_next(wl: Workload, layer: int, step: int, q_int: torch.Tensor) -> torch.Tensor:
    return grid_drift(mix_seed(wl.seed, P_DRIFT, layer, step), q_int, wl.grid, wl.rho)


def weights_for(wl: Workload, layer: int, device="cpu") -> torch.Tensor:
    return choice(mix_seed(wl.seed, P_W, layer), (wl.batch, wl.h_idx), wl.w_values, device)


def latents_for(wl: Workload, layer: int, rows: int, row0: int = 0, device="cpu") -> torch.Tensor:
    dt = torch.float32 if wl.kv_fp32 else torch.bfloat16
    return normal(mix_seed(wl.seed, P_LAT, layer, row0), (rows, wl.kv_width), dt, device)


def qmla_for(wl: Workload, layer: int, step: int, device="cpu") -> torch.Tensor:
    dt = torch.float32 if wl.kv_fp32 else torch.bfloat16
    return normal(mix_seed(wl.seed, P_QMLA, layer, step), (wl.batch, wl.h_q, wl.q_width), dt, device)


def new_kv_for(wl: Workload, layer: int, step: int, device="cpu") -> torch.Tensor:
    dt = torch.float32 if wl.kv_fp32 else torch.bfloat16
    return normal(mix_seed(wl.seed, P_NEWKV, layer, step), (wl.batch, wl.kv_width), dt, device)


def new_ik_for(wl: Workload, layer: int, step: int, device="cpu") -> torch.Tensor:
    return grid_ints(mix_seed(wl.seed, P_NEWIK, layer, step), (wl.batch, wl.d_idx), wl.grid, device)


def prefill_queries(wl: Workload, layer: int, n: int, device="cpu") -> torch.Tensor:
    """Indexer queries of n consecutive prefill positions [n, H, D] (grid integers):
    an AR(1) chain with correlation wl.rho from one position to the next."""
    q = grid_ints(mix_seed(wl.seed, P_PFQ, layer), (wl.h_idx, wl.d_idx), wl.grid, "cpu")
    out = torch.empty((n, wl.h_idx, wl.d_idx), dtype=torch.int8)
    for j in range(n):
        out[j] = q
        q = grid_drift(mix_seed(wl.seed, P_PFQ, layer, j + 1), q, wl.grid, wl.rho)
    return out.to(device)


def prefill_weights(wl: Workload, layer: int, n: int, device="cpu") -> torch.Tensor:
    """Indexer head weights of n prefill positions [n, H]."""
    return choice(mix_seed(wl.seed, P_PFW, layer), (n, wl.h_idx), wl.w_values, device)


def prefill_qmla(wl: Workload, layer: int, n: int, row0: int = 0, device="cpu") -> torch.Tensor:
    """MLA queries of n prefill positions starting at chunk row row0 [n, Hq, 576]."""
    dt = torch.float32 if wl.kv_fp32 else torch.bfloat16
    return normal(mix_seed(wl.seed, P_PFQMLA, layer, row0), (n, wl.h_q, 576), dt, device)
