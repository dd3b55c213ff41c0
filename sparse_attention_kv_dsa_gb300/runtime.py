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
                 scratch: SharedScratch | None = None, fill=True, gen_device=None, adaptive_slack=None,
                 host_kv=None, host_base=None):
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
        # host_kv: this layer's rows of a model-wide pool (E.HostPool.layer_rows), with the
        # requests' host_base from its allocator; default: a pinned buffer of its own
        self.cache = E.LayerCache(wl.n_gpu, wl.n_host, kvdt, dev, host_kv=host_kv)
        self.idx_k = torch.zeros(B, Lmax, wl.d_idx, dtype=ikdt, device=dev)
        self.host_base = torch.tensor(wl.host_base if host_base is None else host_base, dtype=torch.int32,
                                      device=dev)
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
        if adaptive_slack is not None:                    # the adaptive prefetch cap
            self.cache.enable_adaptive_cap(B, adaptive_slack)
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

    def make_io_set(self) -> "StepIO":
        """A second set of this layer's per-step input and output buffers, with step
        arguments that point at them (every other pointer is shared with self.args).
        The returned object owns the tensors: keep it alive as long as any CUDA Graph
        captured on its arguments may replay."""
        return StepIO(self)

    def step(self, stream=None, args: E.StepArgsT | None = None):
        E.decode_layer_step(self.cache, args or self.args, stream)

    def step_ops(self, stream=None, *, defer_cap: bool = True):
        """The same step issued as its separate entry points.  defer_cap=False keeps
        the exact prefetch cap inside the indexer call (its own small launch) and uses
        the plain top-k; True defers it into the top-k launch, as the fused step does."""
        wl, sc, c = self.wl, self.scratch, self.cache
        pf = self.prefetch
        if pf and not defer_cap and c.struct.pf_new_rows:
            raise ValueError("the adaptive cap needs echo_topk_prefetch (defer_cap=True): the plain top-k does "
                             "not record the prediction error")
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


class BlockDecodeLayer:
    """One layer's decode step with block granularity: T consecutive tokens of a
    request form one host index and one GPU slot (T rows of the pools).  The step is
    the library's entry points in order: write-back of the new token, indexer scores,
    block scores (largest token score of each block), exact top-kb blocks with the EMA
    of the kb-th block score, recall of the missing blocks, the selected blocks' token
    slots, sparse attention over those tokens.  No fused prefetch in this mode.

    With a GQA workload (wl.kv_heads > 0) every "request" of this layer is one
    (request, KV head) group with rows of that head's key and value, and attention is
    each group's query heads over its own selection; otherwise sparse MLA."""

    def __init__(self, wl: S.Workload, layer: int, T: int, kb: int, device="cuda", *, n_gpu_blocks=None,
                 fill=True, gen_device=None):
        dev = torch.device(device)
        assert T >= 1 and kb >= 1
        self.wl, self.layer, self.device, self.T, self.kb = wl, layer, dev, int(T), int(kb)
        B, Lmax = wl.batch, wl.max_ctx
        kvdt = torch.float32 if wl.kv_fp32 else torch.bfloat16
        ikdt = torch.float32 if wl.kv_fp32 else torch.float8_e4m3fn
        self.kvdt, self.ikdt = kvdt, ikdt
        bases, off = [], 0                                 # block-aligned host rows per request
        for c in wl.ctx:
            bases.append(off)
            off += -(-(c + wl.steps + 8) // T) * T
        self.n_host_blocks = off // T
        self.n_gpu_blocks = int(n_gpu_blocks if n_gpu_blocks is not None else max(wl.n_gpu // T, 1))
        self.cache = E.LayerCache(self.n_gpu_blocks, self.n_host_blocks, kvdt, dev, block_tokens=T,
                                  row_elems=wl.kv_width)
        i32 = torch.int32
        self.host_base = torch.tensor(bases, dtype=i32, device=dev)              # tokens
        self.host_base_blk = torch.tensor([x // T for x in bases], dtype=i32, device=dev)
        self.seq_len = torch.tensor(wl.ctx, dtype=i32, device=dev)
        self.seq_len_blk = torch.zeros(B, dtype=i32, device=dev)
        self.theta = torch.full((B,), math.inf, dtype=torch.float32, device=dev)
        self.idx_k = torch.zeros(B, Lmax, wl.d_idx, dtype=ikdt, device=dev)
        self.scores = torch.empty(B, Lmax, dtype=torch.float32, device=dev)
        self.nbmax = -(-Lmax // T)
        self.bscores = torch.empty(B, self.nbmax, dtype=torch.float32, device=dev)
        self.sel = torch.empty(B, kb, dtype=i32, device=dev)                      # selected blocks
        self.kth = torch.empty(B, dtype=torch.float32, device=dev)
        self.miss_list = torch.empty(B, kb, dtype=i32, device=dev)
        self.n_miss = torch.zeros(B, dtype=i32, device=dev)
        self.slot_blk = torch.empty(B, kb, dtype=i32, device=dev)
        self.slot_idx = torch.empty(B, kb * T, dtype=i32, device=dev)              # token rows of gpu_kv
        # attention: sparse MLA, or (several KV heads) each group's query heads over its rows
        self.gqa = wl.kv_heads > 0
        vw = wl.q_width if self.gqa else E.V_WIDTH
        self.out = torch.empty(B, wl.h_q, vw, dtype=kvdt, device=dev)
        self.lse = torch.empty(B, wl.h_q, dtype=torch.float32, device=dev)
        ws = (E.gqa_workspace_bytes(B, wl.h_q, wl.q_width, kb * T) if self.gqa
              else E.mla_workspace_bytes(B, wl.h_q, kb * T))
        self.mla_ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.q_idx = torch.zeros(B, wl.h_idx, wl.d_idx, dtype=ikdt, device=dev)
        self.w_idx = S.weights_for(wl, layer, "cpu").to(dev)
        self.new_ik = torch.zeros(B, wl.d_idx, dtype=ikdt, device=dev)
        self.new_kv = torch.zeros(B, wl.kv_width, dtype=kvdt, device=dev)
        self.q_mla = torch.zeros(B, wl.h_q, wl.q_width, dtype=kvdt, device=dev)
        self.cache.reset()
        if fill:
            self.fill_context(gen_device=gen_device)

    def fill_context(self, chunk_rows: int = 1 << 20, gen_device=None):
        """Seeded context: every past token's indexer key (GPU) and every host row's
        latent (row r of the pool gets the r-th latent of the stream)."""
        wl, dev = self.wl, self.device
        gen_dev = gen_device or (dev if dev.type == "cuda" else "cpu")
        for b in range(wl.batch):
            self.idx_k[b, :wl.ctx[b]] = self.to_ik(S.keys_for(wl, self.layer, b, wl.ctx[b], gen_dev))
        n = self.cache.host_kv.shape[0]
        for r0 in range(0, n, chunk_rows):
            r1 = min(n, r0 + chunk_rows)
            self.cache.host_kv[r0:r1].copy_(S.latents_for(wl, self.layer, r1 - r0, r0, gen_dev).cpu())
        torch.cuda.synchronize(dev) if dev.type == "cuda" else None

    to_ik = DecodeLayer.to_ik
    set_step_inputs = DecodeLayer.set_step_inputs
    load_step_inputs = DecodeLayer.load_step_inputs

    STAGES = ("writeback", "index", "block_topk", "recall", "mla")

    def step(self, stream=None, mark=None):
        """Enqueue one step; mark(i), if given, is called after stage i of STAGES."""
        wl, c, T = self.wl, self.cache, self.T
        mark = mark or (lambda i: None)
        E.cache_writeback(c, self.new_kv, self.new_ik, self.idx_k, self.host_base, self.seq_len, stream)
        mark(0)
        E.index_prefetch(self.q_idx, self.w_idx, self.idx_k, self.seq_len, self.theta, self.scores, stream=stream)
        mark(1)
        E.block_scores(self.scores, self.seq_len, T, self.bscores, self.seq_len_blk, stream)
        E.topk(self.bscores, self.seq_len_blk, self.kb, self.sel, self.kth, self.theta, wl.alpha, stream)
        mark(2)
        E.cache_recall(c, self.sel, self.host_base_blk, self.miss_list, self.n_miss, self.slot_blk, stream=stream)
        mark(3)
        E.expand_block_slots(self.sel, self.slot_blk, self.seq_len, T, self.slot_idx, stream)
        if self.gqa:
            E.sparse_gqa_decode(self.q_mla, c.gpu_kv, self.slot_idx, wl.scale, self.out, self.lse, self.mla_ws,
                                stream)
        else:
            E.sparse_mla_decode(self.q_mla, c.gpu_kv, self.slot_idx, wl.scale, self.out, self.lse, self.mla_ws,
                                stream)
        mark(4)


class StepIO:
    """Per-step input and output buffers of one layer beside the layer's own set
    (double buffering: a copy stream fills one set while a step computes on the
    other).  Holds the tensors for as long as the object lives."""

    def __init__(self, dl: DecodeLayer):
        self.q_idx = torch.empty_like(dl.q_idx)
        self.new_ik = torch.empty_like(dl.new_ik)
        self.new_kv = torch.empty_like(dl.new_kv)
        self.q_mla = torch.empty_like(dl.q_mla)
        self.out = torch.empty_like(dl.out)
        self.lse = torch.empty_like(dl.lse)
        a = dl.make_args()
        p = E.ptr
        a.q_idx, a.new_ik, a.new_kv, a.q_mla = p(self.q_idx), p(self.new_ik), p(self.new_kv), p(self.q_mla)
        a.out, a.lse = p(self.out), p(self.lse)
        self.args = a

    @property
    def inputs(self):
        return (self.q_idx, self.new_ik, self.new_kv, self.q_mla)


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


class PrefillChunk:
    """One request's prefill chunk through the library's prefill entry points.

    The chunk's queries are scored in blocks of `block` queries.  A block is ready
    when every token selected by its exact per-query top-k is resident.  Modes:
      "serial"  one stream: score block i, top-k, recall the union, then block i+1;
      "overlap" scoring and top-k on s1; block i's recall on s2 overlaps block i+1;
      "echo"    as "overlap", and block i's histogram candidates are recalled on s2
                as soon as it is scored, before its top-k finishes; the exact recall
                afterwards only fetches what the candidates missed.
    The exact k-th scores of block i are block i+1's predictions (query j for query
    j); the first block predicts +inf, i.e. it has no candidates.  With attend=True
    each block's queries then run sparse MLA over their own selections (after the
    block's union is resident), so a block is done when its attention is."""

    def __init__(self, wl: S.Workload, block: int, device="cuda", layer: int = 0, gen_device=None,
                 record: bool = False, attend: bool = False):
        dev = torch.device(device)
        self.wl, self.block, self.device = wl, int(block), dev
        gd = gen_device or (dev if dev.type == "cuda" else "cpu")
        self.ctx, self.chunk = int(wl.ctx[0]), int(wl.prefill_chunk)
        assert self.chunk % self.block == 0
        self.nblocks = self.chunk // self.block
        self.k = wl.topk
        self.Lmax = self.ctx + self.chunk
        L = self.Lmax
        self.cache = E.LayerCache(wl.n_gpu, wl.n_host, torch.bfloat16, dev)
        self.cache.reset()
        # host pool rows of this request (context and chunk), keys, chunk queries
        for r0 in range(0, L, 1 << 20):
            r1 = min(L, r0 + (1 << 20))
            self.cache.host_kv[r0:r1].copy_(S.latents_for(wl, layer, r1 - r0, r0, gd).cpu())
        self.idx_k = S.grid_to_fp8(S.keys_for(wl, layer, 0, L, gd).to(dev)).contiguous()
        self.q_all = S.grid_to_fp8(S.prefill_queries(wl, layer, L, "cpu")[self.ctx:].to(dev)).contiguous()
        self.w_all = S.prefill_weights(wl, layer, L, "cpu")[self.ctx:].to(dev).contiguous()
        Q, nw = self.block, (L + 31) // 32
        i32 = torch.int32
        self.scores = [torch.empty(Q, L, device=dev) for _ in range(2)]
        self.hist = [torch.empty(Q, 256, dtype=i32, device=dev) for _ in range(2)]
        self.kth = [torch.empty(Q, device=dev) for _ in range(2)]
        self.theta = [torch.empty(Q, device=dev) for _ in range(2)]
        self.sel = [torch.empty(Q, self.k, dtype=i32, device=dev) for _ in range(2)]
        self.thr = [torch.empty(Q, dtype=i32, device=dev) for _ in range(2)]
        self.cand = [torch.empty(Q, dtype=i32, device=dev) for _ in range(2)]
        self.bitmap = [torch.zeros(nw, dtype=i32, device=dev) for _ in range(2)]
        self.lst = [torch.empty(1, L, dtype=i32, device=dev) for _ in range(2)]
        self.count = [torch.empty(1, dtype=i32, device=dev) for _ in range(2)]
        self.miss = [torch.empty(1, L, dtype=i32, device=dev) for _ in range(2)]
        self.nmiss = [torch.zeros(1, dtype=i32, device=dev) for _ in range(2)]
        self.nmiss_c = [torch.zeros(1, dtype=i32, device=dev) for _ in range(2)]
        self.slot = [torch.empty(1, L, dtype=i32, device=dev) for _ in range(2)]
        self.seq = [torch.arange(self.ctx + i * Q + 1, self.ctx + (i + 1) * Q + 1, dtype=i32, device=dev)
                    for i in range(self.nblocks)]
        self.kpred = [torch.empty(Q, device=dev) for _ in range(2)]   # the block's predictions
        self.hb = torch.zeros(1, dtype=i32, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.s1 = torch.cuda.Stream(dev)
        self.s2 = torch.cuda.Stream(dev)
        # attend=True: after a block's exact recall, its queries' sparse MLA over their
        # own selections (slots translated from the selections), written to out / lse
        self.attend = bool(attend)
        if attend:
            self.q_mla = S.prefill_qmla(wl, layer, self.chunk, 0, gd).to(dev).contiguous()
            self.slot_q = torch.empty(Q, self.k, dtype=i32, device=dev)
            self.out = torch.empty(self.chunk, wl.h_q, E.V_WIDTH, dtype=torch.bfloat16, device=dev)
            self.lse = torch.empty(self.chunk, wl.h_q, device=dev)
            self.mla_ws = torch.empty(E.mla_workspace_bytes(Q, wl.h_q, self.k), dtype=torch.uint8, device=dev)
        # record=True keeps every block's outputs (copied on the stream that made them,
        # after the fact) for checks; the two rotating buffers above hold only the last two
        self.rec = None
        if record:
            nb = self.nblocks
            self.rec = {"kpred": torch.empty(nb, Q, device=dev), "kth": torch.empty(nb, Q, device=dev),
                        "sel": torch.empty(nb, Q, self.k, dtype=i32, device=dev),
                        "cand": torch.zeros(nb, Q, dtype=i32, device=dev),
                        "thr": torch.zeros(nb, Q, dtype=i32, device=dev),
                        "n_union": torch.zeros(nb, dtype=i32, device=dev),
                        "n_miss": torch.zeros(nb, dtype=i32, device=dev),
                        "n_miss_cand": torch.zeros(nb, dtype=i32, device=dev)}

    def reset(self):
        self.cache.reset()
        for b in self.bitmap:
            b.zero_()

    def run(self, mode: str = "echo"):
        """Enqueue the whole chunk; returns (start, end) events on s1."""
        assert mode in ("serial", "overlap", "echo")
        Q, k, L = self.block, self.k, self.Lmax
        s1 = self.s1
        s2 = self.s1 if mode == "serial" else self.s2
        ev_topk = [torch.cuda.Event() for _ in range(self.nblocks)]
        ev_done = [torch.cuda.Event() for _ in range(self.nblocks)]
        ev_scored = [torch.cuda.Event() for _ in range(self.nblocks)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(s1)
        s2.wait_stream(s1)
        for i in range(self.nblocks):
            p = i % 2
            pos0 = self.ctx + i * Q
            kp = self.kpred[p]
            with torch.cuda.stream(s1):
                if i >= 2:
                    s1.wait_event(ev_done[i - 2])                # buffers of parity p are free
                if i == 0:
                    kp.fill_(float("inf"))
                else:
                    kp.copy_(self.kth[(i - 1) % 2])
                E.prefill_index(self.q_all[i * Q:(i + 1) * Q], self.w_all[i * Q:(i + 1) * Q], self.idx_k, pos0,
                                kp, self.scores[p], self.hist[p], self.status, s1)
                ev_scored[i].record(s1)
            if mode == "echo":
                with torch.cuda.stream(s2):                      # candidates move while s1 goes on
                    s2.wait_event(ev_scored[i])
                    E.prefill_candidates(self.scores[p], self.hist[p], pos0, k, kp, self.bitmap[p], self.thr[p],
                                         self.cand[p], s2)
                    E.token_list(self.bitmap[p], L, self.lst[p], self.count[p], s2)
                    E.cache_recall(self.cache, self.lst[p], self.hb, self.miss[p], self.nmiss_c[p], self.slot[p],
                                   stream=s2)
            with torch.cuda.stream(s1):
                self.theta[p].copy_(kp)
                E.topk(self.scores[p], self.seq[i], k, self.sel[p], self.kth[p], self.theta[p], 0.5, s1)
                if self.rec is not None:
                    self.rec["kpred"][i].copy_(kp)
                    self.rec["sel"][i].copy_(self.sel[p])
                    self.rec["kth"][i].copy_(self.kth[p])
                ev_topk[i].record(s1)
            with torch.cuda.stream(s2):
                s2.wait_event(ev_topk[i])
                if self.rec is not None and mode == "echo":
                    self.rec["cand"][i].copy_(self.cand[p])
                    self.rec["thr"][i].copy_(self.thr[p])
                    self.rec["n_miss_cand"][i].copy_(self.nmiss_c[p][0])
                E.mark_tokens(self.sel[p], self.bitmap[p], L, s2)
                E.token_list(self.bitmap[p], L, self.lst[p], self.count[p], s2)
                E.cache_recall(self.cache, self.lst[p], self.hb, self.miss[p], self.nmiss[p], self.slot[p],
                               stream=s2)
                if self.rec is not None:
                    self.rec["n_union"][i].copy_(self.count[p][0])
                    self.rec["n_miss"][i].copy_(self.nmiss[p][0])
                if self.attend:
                    E.translate_slots(self.cache, self.sel[p], self.hb, self.slot_q, s2)
                    E.sparse_mla_decode(self.q_mla[i * Q:(i + 1) * Q], self.cache.gpu_kv, self.slot_q,
                                        self.wl.scale, self.out[i * Q:(i + 1) * Q], self.lse[i * Q:(i + 1) * Q],
                                        self.mla_ws, s2)
                ev_done[i].record(s2)
        s1.wait_stream(s2)
        end.record(s1)
        return start, end
