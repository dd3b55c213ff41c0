"""Buffers of one layer's decode step and the step-argument struct.

Plumbing only: allocates the device tensors (and the pinned host pool), loads the
seeded synthetic context into them, and fills echo_step_args_t so that one call of
echo_decode_layer_step runs the whole step in the library's kernels.  The argument
pointers never change, so a step can be captured in a CUDA Graph and replayed;
per-step inputs are copied into the fixed input buffers before each replay.
"""

from __future__ import annotations

import math

import torch

from . import echo as E
from . import synth as S


class SharedScratch:
    """Buffers used by one layer at a time (shared by the layers of a step)."""

    def __init__(self, wl: S.Workload, device, cap_max: int):
        B = wl.batch
        kvdt = torch.float32 if wl.kv_fp32 else torch.bfloat16
        self.cap_max = max(int(cap_max), 1)
        self.scores = torch.empty(B, wl.max_ctx, dtype=torch.float32, device=device)
        self.stage_kv = torch.empty(B * self.cap_max, E.KV_WIDTH, dtype=kvdt, device=device)
        ws = E.mla_workspace_bytes(B, wl.h_q, wl.topk)
        self.mla_ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)


class DecodeLayer:
    """State and buffers of one layer for a workload."""

    def __init__(self, wl: S.Workload, layer: int, device="cuda", *, prefetch=True, cap_max=None,
                 scratch: SharedScratch | None = None, fill=True, gen_device=None):
        dev = torch.device(device)
        self.wl, self.layer, self.device = wl, layer, dev
        B, Lmax = wl.batch, wl.max_ctx
        kvdt = torch.float32 if wl.kv_fp32 else torch.bfloat16
        ikdt = torch.float32 if wl.kv_fp32 else torch.float8_e4m3fn
        self.kvdt, self.ikdt = kvdt, ikdt
        self.cap_max = int(wl.cap_max if cap_max is None else cap_max)
        self.prefetch = bool(prefetch) and self.cap_max > 0
        self.scratch = scratch or SharedScratch(wl, dev, max(self.cap_max, 1))
        assert self.scratch.cap_max >= self.cap_max
        self.cache = E.LayerCache(wl.n_gpu, wl.n_host, kvdt, dev)
        self.idx_k = torch.zeros(B, Lmax, wl.d_idx, dtype=ikdt, device=dev)
        self.host_base = torch.tensor(wl.host_base, dtype=torch.int32, device=dev)
        self.seq_len = torch.tensor(wl.ctx, dtype=torch.int32, device=dev)
        self.theta = torch.full((B,), math.inf, dtype=torch.float32, device=dev)
        self.cap = torch.zeros(B, dtype=torch.int32, device=dev)
        self.pf_count = torch.zeros(B, dtype=torch.int32, device=dev)
        self.pf_list = torch.full((B, max(self.cap_max, 1)), -1, dtype=torch.int32, device=dev)
        self.sel = torch.empty(B, wl.topk, dtype=torch.int32, device=dev)
        self.kth = torch.empty(B, dtype=torch.float32, device=dev)
        self.miss_list = torch.empty(B, wl.topk, dtype=torch.int32, device=dev)
        self.n_miss = torch.zeros(B, dtype=torch.int32, device=dev)
        self.slot_idx = torch.empty(B, wl.topk, dtype=torch.int32, device=dev)
        self.out = torch.empty(B, wl.h_q, E.V_WIDTH, dtype=kvdt, device=dev)
        self.lse = torch.empty(B, wl.h_q, dtype=torch.float32, device=dev)
        # per-step inputs (fixed buffers)
        self.q_idx = torch.zeros(B, wl.h_idx, wl.d_idx, dtype=ikdt, device=dev)
        self.w_idx = S.weights_for(wl, layer, "cpu").to(dev)
        self.new_ik = torch.zeros(B, wl.d_idx, dtype=ikdt, device=dev)
        self.new_kv = torch.zeros(B, E.KV_WIDTH, dtype=kvdt, device=dev)
        self.q_mla = torch.zeros(B, wl.h_q, E.KV_WIDTH, dtype=kvdt, device=dev)
        self.cache.reset()
        if fill:
            self.fill_context(gen_device=gen_device)
        self.args = self.make_args()

    # ------------------------------------------------------------------ data --
    def fill_context(self, chunk_rows: int = 1 << 20, gen_device=None):
        """Seeded context: indexer keys of every past token (GPU resident) and every
        past latent in the pinned host pool.  gen_device picks the generator (values
        depend on it): "cpu" for cases the oracle recomputes, the GPU for speed."""
        wl, dev = self.wl, self.device
        gen_dev = gen_device or (dev if dev.type == "cuda" else "cpu")
        for b in range(wl.batch):
            kint = S.keys_for(wl, self.layer, b, wl.ctx[b], gen_dev)
            self.idx_k[b, :wl.ctx[b]] = self.to_ik(kint)
        n = self.cache.n_host
        for r0 in range(0, n, chunk_rows):
            r1 = min(n, r0 + chunk_rows)
            self.cache.host_kv[r0:r1].copy_(S.latents_for(wl, self.layer, r1 - r0, r0, gen_dev).cpu())
        torch.cuda.synchronize(dev) if dev.type == "cuda" else None

    def to_ik(self, x_int: torch.Tensor) -> torch.Tensor:
        if self.ikdt == torch.float32:
            return S.grid_to_float(x_int).to(self.device)
        return S.grid_to_fp8(x_int.to(self.device))

    def set_step_inputs(self, q_int, new_ik_int, new_kv, q_mla):
        self.q_idx.copy_(self.to_ik(q_int))
        self.new_ik.copy_(self.to_ik(new_ik_int))
        self.new_kv.copy_(new_kv)
        self.q_mla.copy_(q_mla)

    def load_step_inputs(self, q_ik, new_ik, new_kv, q_mla, non_blocking=False):
        """Copy one step's inputs, already in the kernels' dtypes, into the fixed buffers."""
        self.q_idx.copy_(q_ik, non_blocking=non_blocking)
        self.new_ik.copy_(new_ik, non_blocking=non_blocking)
        self.new_kv.copy_(new_kv, non_blocking=non_blocking)
        self.q_mla.copy_(q_mla, non_blocking=non_blocking)

    # ------------------------------------------------------------------ args --
    def make_args(self, prefetch: bool | None = None) -> E.StepArgsT:
        wl, sc = self.wl, self.scratch
        pf = self.prefetch if prefetch is None else (bool(prefetch) and self.cap_max > 0)
        p = E.ptr
        a = E.StepArgsT()
        a.B = wl.batch
        a.host_base, a.seq_len = p(self.host_base), p(self.seq_len)
        a.H, a.D, a.Lmax, a.idx_dtype = wl.h_idx, wl.d_idx, wl.max_ctx, E.dtype_code(self.ikdt)
        a.q_idx, a.w_idx, a.idx_k = p(self.q_idx), p(self.w_idx), p(self.idx_k)
        a.new_ik, a.new_kv = p(self.new_ik), p(self.new_kv)
        a.theta, a.alpha, a.k = p(self.theta), wl.alpha, wl.topk
        a.prefetch, a.cap_max, a.cap_div, a.cap = int(pf), max(self.cap_max, 1), wl.cap_div, p(self.cap)
        a.scores, a.pf_list, a.pf_count, a.stage_kv = p(sc.scores), p(self.pf_list), p(self.pf_count), p(sc.stage_kv)
        a.sel, a.kth, a.miss_list, a.n_miss, a.slot_idx = (p(self.sel), p(self.kth), p(self.miss_list),
                                                           p(self.n_miss), p(self.slot_idx))
        a.Hq, a.q_mla, a.scale = wl.h_q, p(self.q_mla), wl.scale
        a.out, a.lse = p(self.out), p(self.lse)
        a.mla_workspace, a.mla_workspace_bytes = p(sc.mla_ws), sc.mla_ws.numel()
        self._args_pf = pf
        return a

    def step(self, stream=None, args: E.StepArgsT | None = None):
        E.decode_layer_step(self.cache, args or self.args, stream)

    def step_ops(self, stream=None, *, defer_cap: bool = True):
        """The same step issued as its separate entry points.  defer_cap=False keeps
        the exact prefetch cap inside the indexer call (its own small launch) and uses
        the plain top-k; True defers it into the top-k launch, as the fused step does."""
        wl, sc, c = self.wl, self.scratch, self.cache
        pf = self.prefetch
        E.cache_writeback(c, self.new_kv, self.new_ik, self.idx_k, self.host_base, self.seq_len, stream)
        if pf:
            E.cache_reserve(c, self.seq_len, self.cap_max, wl.cap_div, self.cap, self.pf_count, stream)
        E.index_prefetch(self.q_idx, self.w_idx, self.idx_k, self.seq_len, self.theta, sc.scores, layer=c,
                         cap=self.cap if pf else None, cap_max=self.cap_max, host_base=self.host_base,
                         pf_list=self.pf_list, pf_count=self.pf_count, stage_kv=sc.stage_kv,
                         defer_cap=pf and defer_cap, stream=stream)
        if pf and defer_cap:
            E.topk_prefetch(sc.scores, self.seq_len, wl.topk, self.sel, self.kth, self.theta, wl.alpha, layer=c,
                            cap=self.cap, cap_max=self.cap_max, host_base=self.host_base, pf_list=self.pf_list,
                            pf_count=self.pf_count, stage_kv=sc.stage_kv, stream=stream)
        else:
            E.topk(sc.scores, self.seq_len, wl.topk, self.sel, self.kth, self.theta, wl.alpha, stream)
        E.cache_recall(c, self.sel, self.host_base, self.miss_list, self.n_miss, self.slot_idx,
                       pf_list=self.pf_list if pf else None, pf_count=self.pf_count if pf else None,
                       cap_max=self.cap_max, stage_kv=sc.stage_kv, stream=stream)
        E.sparse_mla_decode(self.q_mla, c.gpu_kv, self.slot_idx, wl.scale, self.out, self.lse, sc.mla_ws, stream)

    # ------------------------------------------------------------- snapshot --
    def snapshot(self) -> dict:
        """Host copy of the cache state (for hand-off to the oracle)."""
        c = self.cache
        return {"host2gpu": c.host2gpu.cpu().numpy().copy(), "gpu2host": c.gpu2host.cpu().numpy().copy(),
                "priority": c.priority.cpu().numpy().copy(), "free_map": c.free_map.cpu().numpy().copy(),
                "counters": c.counters.cpu().numpy().copy(), "seq_len": self.seq_len.cpu().numpy().copy(),
                "theta": self.theta.cpu().numpy().copy()}


class StepInputs:
    """Seeded per-step inputs of every layer, generated up front (resident in HBM)."""

    def __init__(self, wl: S.Workload, layers: int, steps: int, device="cuda", gen_device=None):
        gd = gen_device or device
        self.q_int, self.new_ik, self.new_kv, self.q_mla = [], [], [], []
        for l in range(layers):
            q = S.qidx_initial(wl, l, "cpu")
            ql, ikl, kvl, qml = [], [], [], []
            for s in range(steps):
                ql.append(q.to(device))
                ikl.append(S.new_ik_for(wl, l, s, "cpu").to(device))
                kvl.append(S.new_kv_for(wl, l, s, gd).to(device))
                qml.append(S.qmla_for(wl, l, s, gd).to(device))
                q = S.qidx_next(wl, l, s, q)
            self.q_int.append(ql)
            self.new_ik.append(ikl)
            self.new_kv.append(kvl)
            self.q_mla.append(qml)
        # the same indexer inputs in the kernels' dtype (FP8 e4m3 or float32)
        cast = (lambda x: S.grid_to_float(x)) if wl.kv_fp32 else (lambda x: S.grid_to_fp8(x))
        self.q_ik = [[cast(x) for x in ql] for ql in self.q_int]
        self.new_ik_ik = [[cast(x) for x in il] for il in self.new_ik]
