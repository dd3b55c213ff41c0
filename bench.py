"""Decode throughput of the ECHO hot path (index + recall + sparse MLA) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl echo|reference]
                    [--workload NAME] [--no-prefetch]

A step is one pass of the whole hot path over one batch: for every layer, the
write-back of each request's new token, the prefetch budget, lightning-indexer
scoring with fused threshold prefetch, exact top-k with the EMA update, recall of
every missing selected token, and sparse MLA decode.  The whole step is one CUDA
Graph replay.  Inputs are seeded synthetic tensors already resident in HBM when
the timed region starts (value); the e2e figure repeats the measurement with the
step inputs copied from pinned host memory and the attention output copied back
inside the timed region.  Default workload: 4 independent layers, batch 32,
contexts uniform in [80K, 100K], top-2048, 200K GPU slots per layer.

Multi-GPU: one process per GPU (torchrun); each rank runs an independent replica
(requests shard with no exchange), the timed region is bracketed by barriers and
the slowest rank's time is used; value = all ranks' tokens / that time.

--impl reference times the CPU oracle (the only reference there is) on a bounded
sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s (index+recall+sparse MLA) at 100K ctx; indexer & recall GB/s"
DEFAULT_WL = "saturated-b32-ctx80k-100k-4layer"


# ------------------------------------------------------------ distributed ----
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    """Largest value over ranks (the slowest rank's time)."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int) -> float:
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks ----
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu = ids[gpu_index] if gpu_index < len(ids) else gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # let the sampler start before the timed region: spawning it must not
            # delay the first launches after the start event
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers ----
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def kernel_traffic(kernel_src, workload: str):
    """DRAM bytes per launch of the indexer from the committed ncu summary, if it was
    taken on the current source of the kernel (its file and the shared device header;
    else None)."""
    p = os.path.join(ROOT, "profiles", "indexer_traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f)
    srcs = [kernel_src] if isinstance(kernel_src, str) else list(kernel_src)
    h = hashlib.sha256(b"".join(open(f, "rb").read() for f in srcs)).hexdigest()[:16]
    if d.get("source_sha") != h:
        return None, "kernel changed since the ncu capture"
    per = d.get("per_workload", {}).get(workload)
    return (per.get("dram_bytes_per_launch") if per else None), d.get("note")


# ---------------------------------------------------------- CPU baseline ----
def oracle_sample(wl, n_req: int, seed_layer: int = 0, threads: int = 0):
    """Time the CPU oracle on a bounded sample: one layer's decode step for the
    first n_req requests of the workload (cold cache), with `threads` OpenMP threads
    (0 = every core).  Returns (seconds, tokens)."""
    import numpy as np
    import torch
    import oracle as O
    from sparse_attention_kv_dsa_gb300 import synth as S
    ctx = wl.ctx[:n_req]
    sub = S.Workload(name=wl.name, cfg_id=wl.cfg_id, layers=1, batch=n_req, ctx=list(ctx), h_idx=wl.h_idx,
                     d_idx=wl.d_idx, grid=wl.grid, w_values=wl.w_values, topk=wl.topk, h_q=wl.h_q,
                     kv_fp32=wl.kv_fp32, n_gpu=wl.n_gpu, n_host=sum(c + 16 for c in ctx) + 16, steps=8,
                     rho=wl.rho, cap_max=wl.cap_max, cap_div=wl.cap_div)
    new_ik = S.grid_to_float(S.new_ik_for(sub, seed_layer, 0)).numpy()
    keys = [np.concatenate([S.grid_to_float(S.keys_for(sub, seed_layer, b, ctx[b])).numpy(), new_ik[b:b + 1]])
            for b in range(n_req)]
    lat = S.latents_for(sub, seed_layer, sub.n_host, 0)                 # bf16 host pool rows
    q = S.grid_to_float(S.qidx_initial(sub, seed_layer)).numpy()
    w = S.weights_for(sub, seed_layer).numpy()
    qm = S.qmla_for(sub, seed_layer, 0).float().numpy()
    cache = O.LayerCache(sub.n_gpu, sub.n_host)
    seq = np.array(ctx, dtype=np.int64)
    hb = sub.host_base
    theta = np.full(n_req, np.inf, dtype=np.float32)
    O.set_threads(threads or cpu_cores())
    t0 = time.perf_counter()
    O.decode_layer_step(cache, host_base=hb, seq_len=seq, keys_of=lambda b, L: keys[b][:L], q_idx=q, w_idx=w,
                        theta=theta, k=sub.topk, cap_max=sub.cap_max, cap_div=sub.cap_div, q_mla=qm,
                        latent_of=lambda h: lat[torch.from_numpy(np.asarray(h))].double().numpy(),
                        scale=sub.scale)
    return time.perf_counter() - t0, n_req


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, budget_s: float = 15.0) -> dict:
    """Oracle tokens/s on this host's cores: one layer-step of a few requests with
    OpenMP on every core (the baseline), and of one request on one thread; per-request
    layer-step cost x layers."""
    cores = cpu_cores()
    t1, _ = oracle_sample(wl, 1, threads=1)                 # single thread, one request
    n_req = max(1, min(wl.batch, int(budget_s / 3 / max(t1 / cores, 1e-3))))
    n_req = min(n_req, 8)
    tn, _ = oracle_sample(wl, n_req, threads=cores)
    tok_s = n_req / (tn * wl.layers)
    return {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"one decode step of one layer for the first {n_req} requests (ctx {min(wl.ctx[:n_req])}-"
                      f"{max(wl.ctx[:n_req])}), cold cache, C++ oracle with OpenMP on {cores} threads; "
                      f"scaled by {wl.layers} layers",
            "single_thread": {"value": 1.0 / (t1 * wl.layers), "unit": "tokens/s", "cores": 1,
                              "sample": f"one layer-step of 1 request (ctx {wl.ctx[0]}), one thread, "
                                        f"x{wl.layers} layers"}}


# ----------------------------------------------------------- reference arm ----
def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    from sparse_attention_kv_dsa_gb300 import synth as S
    wl = S.workloads()[args.workload]
    cores = cpu_cores()
    n_req = 2                                               # requests per sampled step
    oracle_sample(wl, 1, threads=cores)                     # import / page-in warm-up
    for _ in range(args.warmup):
        oracle_sample(wl, n_req, threads=cores)
    t_total, toks = 0.0, 0
    for _ in range(args.steps):
        t, n = oracle_sample(wl, n_req, threads=cores)
        t_total += t * wl.layers                            # the sampled requests through every layer
        toks += n
    value = toks / t_total
    sample = (f"one layer-step of the first {n_req} requests (ctx {min(wl.ctx[:n_req])}-{max(wl.ctx[:n_req])}) "
              f"per step, C++ oracle with OpenMP on {cores} threads, x{wl.layers} layers")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "sample": f"{n_req} requests per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- echo arm ----
def run_echo(args, ws, rank, local):
    import ctypes
    import torch
    import sparse_attention_kv_dsa_gb300.echo as E
    from sparse_attention_kv_dsa_gb300 import synth as S
    from sparse_attention_kv_dsa_gb300.runtime import DecodeLayer, SharedScratch, StepInputs

    lib = E.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = S.workloads()[args.workload]
    if args.layers:
        wl.layers = int(args.layers)
    layers = wl.layers
    # step inputs: pool fill + warm-up + timed + e2e + stage leg, within the workload's steps
    n_warm = max(args.warmup - 1, 2)                       # after the first (eager) step
    base_steps = 1 + n_warm + args.steps + args.steps + PROBE_STEPS
    if base_steps > wl.steps + 8:
        raise SystemExit(f"--steps/--warmup need {base_steps} decode steps; {wl.name} has {wl.steps}")
    fill_max = max(0, min(args.fill_max, wl.steps + 8 - base_steps))
    total_steps = base_steps + fill_max
    prefetch = not args.no_prefetch
    scratch = SharedScratch(wl, dev, wl.cap_max)
    # the model-wide host pool: one pinned buffer with every layer's rows; each request's
    # context takes one row range, shared by all layers
    pool = E.HostPool(layers, wl.n_host, torch.float32 if wl.kv_fp32 else torch.bfloat16)
    host_base = [pool.alloc(c + wl.steps + 8) for c in wl.ctx]
    assert host_base == wl.host_base
    L = [DecodeLayer(wl, l, dev, prefetch=prefetch, scratch=scratch, gen_device=dev, host_kv=pool.layer_rows(l),
                     host_base=host_base) for l in range(layers)]
    inp = StepInputs(wl, layers, total_steps, dev, gen_device=dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()

    h_in = {}                      # pinned host copies of the e2e leg's step inputs (made later)
    h_out = [torch.empty(L[l].out.shape, dtype=L[l].out.dtype, pin_memory=True) for l in range(layers)]

    def timing_event(external=False):
        return torch.cuda.Event(enable_timing=True, external=True) if external else \
            torch.cuda.Event(enable_timing=True)

    # events recorded inside the captured graphs (around each layer's indexer launch,
    # and between the stages of the probe graph) need external events
    try:
        timing_event(external=True)
        ext_ok = True
    except TypeError:
        ext_ok = False

    # Buffer sets: set 0 is each layer's own step-input/output buffers, sets 1.. are
    # StepIO objects that own theirs.  Each set has its own captured graph of the whole
    # step and its own indexer events, so a replay's events stay readable until the
    # same set replays again, NSETS steps later.
    io = [None] + [[dl.make_io_set() for dl in L] for _ in range(NSETS - 1)]

    def set_args(p, l):
        return L[l].args if p == 0 else io[p][l].args

    def set_inputs(p, l):
        dl = L[l]
        return (dl.q_idx, dl.new_ik, dl.new_kv, dl.q_mla) if p == 0 else io[p][l].inputs

    def set_out(p, l):
        return L[l].out if p == 0 else io[p][l].out

    def layer_step(l, st):
        # the step's kernels issued through the separate entry points (the prefetch
        # budget as its own launch), with events between the stages
        dl = L[l]
        a = dl.args
        h = st.cuda_stream
        mark = lambda i: st_ev[l][i].record(st)
        mark(0)
        E.check(lib.echo_cache_writeback(dl.cache.ref, a.new_kv, a.new_ik, a.idx_k, a.D, a.Lmax, a.idx_dtype,
                                         a.host_base, a.seq_len, a.B, h))
        mark(1)
        if a.prefetch:
            E.check(lib.echo_cache_reserve(dl.cache.ref, a.seq_len, a.B, a.cap_max, a.cap_div, a.cap,
                                           a.pf_count, h))
        mark(2)
        enqueue_index_topk(lib, dl, h, between=lambda: mark(3))
        mark(4)
        E.check(lib.echo_cache_recall(dl.cache.ref, a.sel, a.host_base, a.B, a.k,
                                      a.pf_list if a.prefetch else None, a.pf_count if a.prefetch else None,
                                      a.cap_max, a.stage_kv, a.miss_list, a.n_miss, a.slot_idx, h))
        mark(5)
        E.check(lib.echo_sparse_mla_decode(a.q_mla, dl.cache.struct.gpu_kv, dl.cache.n_gpu,
                                           dl.cache.struct.kv_dtype, a.slot_idx, a.B, a.Hq, a.k,
                                           ctypes.c_float(a.scale), a.out, a.lse, a.mla_workspace,
                                           a.mla_workspace_bytes, h))
        mark(6)

    def load_inputs(s, st):
        with torch.cuda.stream(st):
            for l in range(layers):
                L[l].load_step_inputs(inp.q_ik[l][s], inp.new_ik_ik[l][s], inp.new_kv[l][s], inp.q_mla[l][s])

    # first step eagerly (cold cache), then capture one whole step per buffer set
    s_idx = 0
    load_inputs(s_idx, stream)
    with torch.cuda.stream(stream):
        for l in range(layers):
            L[l].step(stream=stream)
    s_idx += 1
    stream.synchronize()
    ix_ev = [[(timing_event(True), timing_event(True)) for _ in range(layers)] for _ in range(NSETS)] \
        if ext_ok else None
    if ext_ok:
        # the timed graphs are the library's own step (echo_decode_layer_step) with its
        # profiling hook recording events around each layer's indexer launch
        for p in range(NSETS):
            for l in range(layers):
                for j in range(2):
                    ix_ev[p][l][j].record(stream)            # creates the events
                    set_args(p, l).index_events[j] = ix_ev[p][l][j].cuda_event
        stream.synchronize()
    graphs = []
    for p in range(NSETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(layers):
                L[l].step(stream=stream, args=set_args(p, l))
        graphs.append(g)
    probe, st_ev = None, None                             # the same step with events between stages
    if ext_ok:
        st_ev = [[timing_event(True) for _ in range(7)] for _ in range(layers)]
        probe = torch.cuda.CUDAGraph()
        with torch.cuda.graph(probe, stream=stream):
            for l in range(layers):
                layer_step(l, stream)
    torch.cuda.synchronize()

    # Step i of a run uses buffer set i % NSETS.  A copy stream stages step i+1's inputs
    # while step i computes and, in the end-to-end leg, reads step i's attention output
    # back to pinned host memory once it is done.
    cs = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(NSETS)]
    ev_done = [torch.cuda.Event() for _ in range(NSETS)]

    def stage_inputs(i, s, from_host):
        p = i % NSETS
        with torch.cuda.stream(cs):
            if i >= NSETS:
                cs.wait_event(ev_done[p])                    # set p: step i-NSETS has computed
            for l in range(layers):
                src = h_in[(l, s)] if from_host else \
                    (inp.q_ik[l][s], inp.new_ik_ik[l][s], inp.new_kv[l][s], inp.q_mla[l][s])
                for dst, x in zip(set_inputs(p, l), src):
                    dst.copy_(x, non_blocking=True)
            ev_in[p].record(cs)

    def run_pipelined(s0, n, from_host, sample_ix=False):
        """Steps s0 .. s0+n-1 back to back.  Returns the (start, end) events of every
        replay and, with sample_ix, every replay's per-layer indexer time (ms): the
        host reads replay i's in-graph events while replays i+1 .. i+NSETS-1 are
        queued, before replay i+NSETS records them again."""
        cs.wait_stream(stream)
        stage_inputs(0, s0, from_host)
        evs = [(timing_event(), timing_event()) for _ in range(n)]
        ix = []

        def read_ix(j):
            q = j % NSETS
            evs[j][1].synchronize()
            ix.append([ix_ev[q][l][0].elapsed_time(ix_ev[q][l][1]) for l in range(layers)])

        for i in range(n):
            p = i % NSETS
            if i + 1 < n:
                stage_inputs(i + 1, s0 + i + 1, from_host)
            stream.wait_event(ev_in[p])
            evs[i][0].record(stream)
            with torch.cuda.stream(stream):
                graphs[p].replay()
            evs[i][1].record(stream)
            ev_done[p].record(stream)
            if from_host:
                with torch.cuda.stream(cs):
                    cs.wait_event(ev_done[p])
                    for l in range(layers):
                        h_out[l].copy_(set_out(p, l), non_blocking=True)
            if sample_ix and i >= NSETS - 1:
                read_ix(i - (NSETS - 1))
        if sample_ix:
            for j in range(max(0, n - (NSETS - 1)), n):
                read_ix(j)
        return evs, ix

    # steady state of the pool: untimed steps until every layer has fewer free slots
    # than its last step bound, so that every timed step evicts (or fill_max steps)
    fill = 0
    while fill < fill_max:
        load_inputs(s_idx, stream)
        with torch.cuda.stream(stream):
            graphs[0].replay()
        s_idx += 1
        fill += 1
        stream.synchronize()
        ctr = [dl.cache.read_counters() for dl in L]
        if all(c[E.CTR_N_FREE] < max(c[E.CTR_BOUND], 1) for c in ctr):
            break
    n_free_at_start = [int(dl.cache.read_counters()[E.CTR_N_FREE]) for dl in L]

    # pinned host copies of the e2e leg's inputs, made before the warm-up: pinning new
    # host memory right before the timed region slowed its first steps
    e2e_first = s_idx + n_warm + args.steps
    for l in range(layers):
        for s in range(e2e_first, e2e_first + args.steps):
            h_in[(l, s)] = (inp.q_ik[l][s].cpu().pin_memory(), inp.new_ik_ik[l][s].cpu().pin_memory(),
                            inp.new_kv[l][s].cpu().pin_memory(), inp.q_mla[l][s].cpu().pin_memory())

    run_pipelined(s_idx, n_warm, from_host=False)         # every graph, as timed
    s_idx += n_warm
    stream.synchronize()
    for dl in L:
        assert dl.cache.status() == 0, f"device status {dl.cache.status()} after warm-up"

    # ---------------- timed region: inputs resident in HBM ----------------
    seq0 = [dl.seq_len.cpu().double() for dl in L]        # context lengths before the first timed step
    ev0, ev1 = timing_event(), timing_event()
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # the stream first spins for a few ms so that the host has queued the first
        # replays before ev0: the events time the device's work, not the host's issue
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(2e6) * NSETS)
        ev0.record(stream)
        step_ev, ix_samples = run_pipelined(s_idx, args.steps, from_host=False, sample_ix=ext_ok)
        stream.wait_stream(cs)
        ev1.record(stream)
        stream.synchronize()
    s_idx += args.steps
    torch.cuda.synchronize()
    barrier(ws)
    t_ms = ev0.elapsed_time(ev1)
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    step_gap_ms = [step_ev[i][1].elapsed_time(step_ev[i + 1][0]) for i in range(len(step_ev) - 1)]
    statuses = [dl.cache.status() for dl in L]
    t_ms_max = max_over_ranks(t_ms, ws)
    tokens = sum_over_ranks(wl.batch * args.steps, ws)
    value = tokens / (t_ms_max / 1e3)

    # ---------------- e2e: inputs from pinned host, outputs back ----------------
    assert s_idx == e2e_first
    h2d_bytes = sum(sum(x.numel() * x.element_size() for x in h_in[(l, e2e_first)]) for l in range(layers))
    d2h_bytes = sum(h_out[l].numel() * h_out[l].element_size() for l in range(layers))
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = timing_event(), timing_event()
    e0.record(stream)
    e2e_ev, _ = run_pipelined(s_idx, args.steps, from_host=True)
    s_idx += args.steps
    stream.wait_stream(cs)
    e1.record(stream)
    stream.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    e2e_value = tokens / (e2e_ms / 1e3)
    e2e_step_ms = [a.elapsed_time(b) for a, b in e2e_ev]

    # ------- per-stage times and counters inside the graph (probe replays, untimed) -------
    stages, telemetry, per_step = {}, None, []
    row_bytes = 576 * (4 if wl.kv_fp32 else 2)
    recall_gbs_samples = []
    ctr_tot = {"hits": 0, "staged_hits": 0, "misses": 0}
    if not args.skip_stages and probe is not None:
        names = ["writeback", "reserve", "index_prefetch", "topk", "recall", "mla"]
        per = {n: [] for n in names}
        tele = {"qualified": [], "staged": [], "useful": [], "final_recall": [], "theta_rel_err": []}
        for _ in range(PROBE_STEPS):
            load_inputs(s_idx, stream)
            theta_before = [dl.theta.clone() for dl in L]       # the prediction this step scores against
            with torch.cuda.stream(stream):
                probe.replay()
            s_idx += 1
            stream.synchronize()
            us = {n: [st_ev[l][i].elapsed_time(st_ev[l][i + 1]) * 1e3 for l in range(layers)]
                  for i, n in enumerate(names)}
            for n in names:
                per[n].append(sum(us[n]) / layers)
            rec = {"step": None, "hits": [], "staged_hits": [], "misses": [], "qualified": [], "staged": []}
            for l, dl in enumerate(L):
                c = dl.cache.read_counters()
                rec["step"] = c[E.CTR_STEP]
                for key, idx in (("hits", E.CTR_HITS), ("staged_hits", E.CTR_STAGED_HITS),
                                 ("misses", E.CTR_MISSES), ("qualified", E.CTR_QUALIFIED),
                                 ("staged", E.CTR_STAGED)):
                    rec[key].append(int(c[idx]))
                ctr_tot["hits"] += c[E.CTR_HITS]
                ctr_tot["staged_hits"] += c[E.CTR_STAGED_HITS]
                ctr_tot["misses"] += c[E.CTR_MISSES]
                tele["qualified"].append(c[E.CTR_QUALIFIED])
                tele["staged"].append(c[E.CTR_STAGED])
                tele["useful"].append(c[E.CTR_STAGED_HITS])
                tele["final_recall"].append(c[E.CTR_MISSES])
                # this layer's host-link rows over this layer's recall time, same step
                if c[E.CTR_MISSES] > 0 and us["recall"][l] > 0:
                    recall_gbs_samples.append(c[E.CTR_MISSES] * row_bytes / (us["recall"][l] * 1e-6) / 1e9)
                th, kth = theta_before[l].cpu(), dl.kth.cpu()
                ok = torch.isfinite(th) & torch.isfinite(kth) & (kth != 0)
                if bool(ok.any()):
                    tele["theta_rel_err"].append(float(((th[ok] - kth[ok]).abs() / kth[ok].abs()).median()))
            rec["recall_us"] = [round(x, 2) for x in us["recall"]]
            per_step.append(rec)
        stages = {n + "_us": round(statistics.median(v), 2) for n, v in per.items()}
        # every layer's cache management of a step: write-back and recall ([REV] "Experiments
        # and results": all-layer management time; the budget is part of the step's write-back
        # launch, the probe's separate reserve launch is left out)
        mgmt = [sum(per[n][i] for n in ("writeback", "recall")) * layers for i in range(PROBE_STEPS)]
        stages["all_layer_management_us"] = round(statistics.median(mgmt), 1)
        stages["how"] = "CUDA events between the stages inside a graph of the step issued through the separate " \
                        "entry points (reserve as its own launch), median of %d steps, mean over layers" % PROBE_STEPS
        mean = lambda v: (sum(v) / len(v)) if v else None
        telemetry = {
            "qualified_rows": mean(tele["qualified"]),
            "prefetched_rows": mean(tele["staged"]),
            "prefetched_rows_selected": mean(tele["useful"]),
            "useless_prefetch_bytes": (mean(tele["staged"]) - mean(tele["useful"])) * row_bytes if tele["staged"] else None,
            "final_recall_rows": mean(tele["final_recall"]),
            "final_recall_bytes": mean(tele["final_recall"]) * row_bytes if tele["final_recall"] else None,
            "theta_rel_err_median": statistics.median(tele["theta_rel_err"]) if tele["theta_rel_err"] else None,
            "how": "per layer and step, mean over %d probe steps x %d layers: rows above the threshold and not "
                   "resident (before the cap), rows prefetched during scoring, "
                   "those the exact top-k then selected, the bytes of the rest, rows recalled after the top-k; "
                   "median over requests of |theta - kth| / |kth| (EMA prediction vs this step's k-th score)"
                   % (PROBE_STEPS, layers)}

    # ---------------- roofline of the dominant kernel (indexer) ----------------
    peaks = measured_peaks()
    # a step's write-back appends one token before scoring: the timed steps score
    # seq0 + 1 .. seq0 + steps tokens per request
    mean_ctx = sum(float(x.mean()) for x in seq0) / layers + (args.steps + 1) / 2.0
    ix_bytes = wl.batch * mean_ctx * (wl.d_idx + 4)               # keys read + scores written
    ix_flat = [x for row in ix_samples for x in row]
    ix_avg_ms = statistics.median(ix_flat) if ix_flat else stages.get("index_prefetch_us", 0.0) / 1e3
    achieved = ix_bytes / (ix_avg_ms / 1e3) / 1e9 if ix_avg_ms else None
    csrc = os.path.join(ROOT, "sparse_attention_kv_dsa_gb300", "csrc")
    traffic, tnote = kernel_traffic([os.path.join(csrc, "indexer.cu"), os.path.join(csrc, "common.cuh")], wl.name)
    sel_total = ctr_tot["hits"] + ctr_tot["staged_hits"] + ctr_tot["misses"]
    clocks = clk.summary()
    link = None if args.skip_host_link else host_link(dev)
    alloc = None if args.skip_host_link else allocator_bench(dev)
    if rank != 0:
        return 0
    step_roof = step_roofline(wl, mean_ctx, ix_bytes, telemetry, link, peaks, layers, t_ms_max / args.steps)
    recall_gbs = statistics.median(recall_gbs_samples) if recall_gbs_samples else None
    if recall_gbs is not None and link is not None:
        assert recall_gbs <= 1.05 * link["peak_gbs"], \
            f"recall GB/s {recall_gbs:.1f} above the measured host link {link['peak_gbs']:.1f}: a counting error"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+bf16 (f32 accumulate)", "data": "synthetic",
        "config": {"workload": wl.name, "layers": layers, "batch": wl.batch,
                   "ctx": f"{min(wl.ctx)}-{max(wl.ctx)}", "topk": wl.topk, "gpu_slots": wl.n_gpu,
                   "host_slots": wl.n_host, "prefetch": prefetch, "cuda_graph": True,
                   "parallelism": f"replicas x{ws}",
                   "pool_fill_steps": fill, "gpu_free_slots_at_warmup": n_free_at_start,
                   "host_pool": f"model-wide: {layers} layers x {wl.n_host} rows in one pinned buffer",
                   "l2": "inputs larger than L2 (indexer keys %.0f MB per layer)" % (wl.batch * mean_ctx * 128 / 1e6)},
        "step_roofline": step_roof,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": (achieved / peaks["hbm_gbs"]) if achieved else None, "traffic": traffic,
                     "kernel": "indexer_fp8_kernel",
                     "algorithmic_bytes_per_launch": ix_bytes,
                     "avg_launch_ms": ix_avg_ms,
                     "launch_samples": len(ix_flat),
                     "timing": ("median over every timed replay and layer of CUDA events recorded around the "
                                "indexer launch inside the timed graphs") if ix_flat else "eager stage leg",
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic_note": tnote},
        "cpu_baseline": cpu_baseline(wl) if not args.skip_cpu else None,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "step_ms": [round(x, 3) for x in e2e_step_ms],
                "how": "library step replayed as a CUDA Graph; each step's inputs copied from pinned host memory "
                       "and its attention output read back inside the timed region, on a copy stream that "
                       "overlaps the next step's inputs with the current step (%d buffer sets)" % NSETS},
        "step_ms": [round(x, 3) for x in step_ms],
        "step_gap_ms_max": round(max(step_gap_ms), 3) if step_gap_ms else None,
        "gpu_launches": launches_per_step(prefetch, wl.n_gpu) * layers * args.steps,
        "clocks": clocks,
        "stages_us": stages,
        "probe_steps": per_step,
        "prefetch_telemetry": telemetry,
        "indexer_gbs": achieved,
        "recall_gbs": recall_gbs,
        "recall_gbs_how": "per layer and probe step: rows recalled from the host after the top-k x row bytes / "
                          "that layer's recall time in the same step; median",
        "host_link": link,
        "recall_kernel_frac_of_host_link": (link["zero_copy_recall_gbs"] / link["memcpy_h2d_gbs"]) if link else None,
        "allocator": alloc,
        "hit_rate": (ctr_tot["hits"] / sel_total) if sel_total else None,
        "hit_rate_after_prefetch": ((ctr_tot["hits"] + ctr_tot["staged_hits"]) / sel_total) if sel_total else None,
        "device_status": statuses,
    }
    print(json.dumps(line), flush=True)
    return 0


NSETS = 3
PROBE_STEPS = 6


def step_roofline(wl, mean_ctx, ix_bytes, telemetry, link, peaks, layers, ms_per_step):
    """The step's ceiling: for one layer, every stage's algorithmic bytes at the measured
    HBM copy rate (host bytes at the measured host link), sparse MLA at the larger of
    its bytes and its flops at the bf16 GEMM rate; summed over the layers and set
    against the measured step time."""
    hbm = peaks["hbm_gbs"] * 1e9
    bf16 = peaks["bf16_tflops"] * 1e12 if peaks.get("bf16_tflops") else None
    link_bps = link["peak_gbs"] * 1e9 if link else None
    B, k, row = wl.batch, wl.topk, 576 * (4 if wl.kv_fp32 else 2)
    us = {}
    us["writeback"] = (B * (row + wl.d_idx)) / hbm * 1e6 + ((B * row) / link_bps * 1e6 if link_bps else 0.0)
    us["indexer"] = ix_bytes / hbm * 1e6
    us["topk"] = (4.0 * B * mean_ctx + 8.0 * B * k) / hbm * 1e6
    staged = telemetry["prefetched_rows"] if telemetry else 0.0
    final = telemetry["final_recall_rows"] if telemetry else 0.0
    us["recall"] = (13.0 * wl.n_gpu + 2.0 * staged * row) / hbm * 1e6 + \
        ((final + staged) * row / link_bps * 1e6 if link_bps else 0.0)
    mla_bytes = B * k * row + B * wl.h_q * 576 * 2 + B * wl.h_q * 512 * 2
    mla_flops = B * wl.h_q * k * 2.0 * (576 + 512)
    us["sparse_mla"] = max(mla_bytes / hbm, mla_flops / bf16 if bf16 else 0.0) * 1e6
    ceil_ms = sum(us.values()) * layers / 1e3
    return {"ceiling_us_per_layer": {n: round(v, 2) for n, v in us.items()},
            "ceiling_ms_per_step": round(ceil_ms, 4), "measured_ms_per_step": round(ms_per_step, 4),
            "frac": round(ceil_ms / ms_per_step, 3) if ms_per_step else None,
            "ceiling_tokens_per_s": round(B / (ceil_ms / 1e3)) if ceil_ms else None,
            "how": "per layer: write-back rows and keys, indexer keys + scores, top-k scores + selection, "
                   "recall metadata (13 B per GPU slot) + staged rows twice in HBM + prefetched and missed rows "
                   "over the measured host link (both omitted without it), sparse MLA max(bytes at HBM, "
                   "flops at the bf16 GEMM rate); HBM and bf16 peaks from MEASURED_PEAKS.json"}


def launches_per_step(prefetch: bool, n_gpu: int) -> int:
    """Kernels of one layer step (echo_decode_layer_step): write-back with the step's
    prefetch budget (the single-CTA write-back from the pending victim list on pools of
    at least ECHO_PENDING_LIST_MIN_SLOTS slots, then the cooperative manager), indexer 1,
    top-k 1 (with the deferred exact prefetch cap when prefetching), recall 1
    (cooperative manager: protect, miss list, evict+bind, copy, translate), MLA 2
    (split + combine)."""
    import sparse_attention_kv_dsa_gb300.echo as E
    return (2 if n_gpu >= E.PENDING_LIST_MIN_SLOTS else 1) + 1 + 1 + 1 + 2


def enqueue_index_topk(lib, dl, h, between=None):
    """The indexer and the top-k of one layer step as echo_decode_layer_step issues
    them (cap fix-up deferred into the top-k launch); between() runs after the indexer
    call, to record an event."""
    import ctypes
    import sparse_attention_kv_dsa_gb300.echo as E
    a = dl.args
    pf = bool(a.prefetch)
    E.check(lib.echo_index_prefetch(a.q_idx, a.w_idx, a.idx_k, a.seq_len, a.B, a.H, a.D, a.Lmax, a.idx_dtype,
                                    a.theta, a.cap if pf else None, a.cap_max, a.host_base, dl.cache.ref, a.scores,
                                    a.pf_list, a.pf_count, a.stage_kv, E.PF_DEFER_CAP if pf else 0, h))
    if between is not None:
        between()
    if pf:
        E.check(lib.echo_topk_prefetch(a.scores, a.seq_len, a.B, a.Lmax, a.k, a.sel, a.kth, a.theta,
                                       ctypes.c_float(a.alpha), a.cap, a.cap_max, a.host_base, dl.cache.ref,
                                       a.pf_list, a.pf_count, a.stage_kv, h))
    else:
        E.check(lib.echo_topk(a.scores, a.seq_len, a.B, a.Lmax, a.k, a.sel, a.kth, a.theta, ctypes.c_float(a.alpha),
                              h))


def stage_timing(L, inp, s_idx, stream, layers, loaded=False) -> dict:
    """Average per-layer time of each stage of one step, eager, events on the stream.
    With loaded=True the step inputs are already in the layers' input buffers."""
    import ctypes
    import torch
    import sparse_attention_kv_dsa_gb300.echo as E
    lib = E.lib()
    names = ["writeback", "reserve", "index_prefetch", "topk", "recall", "mla"]
    acc = {n: 0.0 for n in names}
    for l in range(layers):
        dl = L[l]
        a = dl.args
        if not loaded:
            dl.load_step_inputs(inp.q_ik[l][s_idx], inp.new_ik_ik[l][s_idx], inp.new_kv[l][s_idx],
                                inp.q_mla[l][s_idx])
        torch.cuda.synchronize()
        h = stream.cuda_stream
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        ev[0].record(stream)
        E.check(lib.echo_cache_writeback(dl.cache.ref, a.new_kv, a.new_ik, a.idx_k, a.D, a.Lmax, a.idx_dtype,
                                         a.host_base, a.seq_len, a.B, h))
        ev[1].record(stream)
        if a.prefetch:
            E.check(lib.echo_cache_reserve(dl.cache.ref, a.seq_len, a.B, a.cap_max, a.cap_div, a.cap, a.pf_count, h))
        ev[2].record(stream)
        enqueue_index_topk(lib, dl, h, between=lambda: ev[3].record(stream))
        ev[4].record(stream)
        E.check(lib.echo_cache_recall(dl.cache.ref, a.sel, a.host_base, a.B, a.k, a.pf_list if a.prefetch else None,
                                      a.pf_count if a.prefetch else None, a.cap_max, a.stage_kv, a.miss_list,
                                      a.n_miss, a.slot_idx, h))
        ev[5].record(stream)
        E.check(lib.echo_sparse_mla_decode(a.q_mla, dl.cache.struct.gpu_kv, dl.cache.n_gpu, dl.cache.struct.kv_dtype,
                                           a.slot_idx, a.B, a.Hq, a.k, ctypes.c_float(a.scale), a.out, a.lse,
                                           a.mla_workspace, a.mla_workspace_bytes, h))
        ev[6].record(stream)
        stream.synchronize()
        for i, n in enumerate(names):
            acc[n] += ev[i].elapsed_time(ev[i + 1]) * 1e3 / layers
    return {n + "_us": round(v, 2) for n, v in acc.items()}


def host_link(dev) -> dict:
    """Host-to-GPU bandwidth on this machine: a large pinned cudaMemcpyAsync, and a large
    all-miss zero-copy recall through the library's own recall kernels (16-byte
    loads of pinned host memory).  The roof for recall is the larger of the two."""
    import torch
    import sparse_attention_kv_dsa_gb300.echo as E
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 0.0
    for _ in range(3):
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, src.numel() / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del src, dst
    B, k = 32, 2048
    n = B * k
    host = torch.zeros(n, 576, dtype=torch.bfloat16, pin_memory=True)
    layer = E.LayerCache(n, n, torch.bfloat16, dev, host_kv=host)
    sel = torch.arange(k, dtype=torch.int32, device=dev).repeat(B, 1).contiguous()
    base = (torch.arange(B, dtype=torch.int32, device=dev) * k).contiguous()
    miss = torch.empty(B, k, dtype=torch.int32, device=dev)
    nmiss = torch.empty(B, dtype=torch.int32, device=dev)
    slot = torch.empty(B, k, dtype=torch.int32, device=dev)
    sweep = []
    for kk in (8, 32, 128, 512, 2048):                      # 256 .. 65536 missed rows
        s_ = sel[:, :kk].contiguous()
        m_, sl_ = miss[:, :kk].contiguous(), slot[:, :kk].contiguous()
        t_best = None
        for _ in range(3):
            layer.reset()
            torch.cuda.synchronize()
            e0.record()
            E.cache_recall(layer, s_, base, m_, nmiss, sl_)
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) * 1e3
            t_best = t if t_best is None else min(t_best, t)
        sweep.append({"rows": B * kk, "us": round(t_best, 1), "gbs": round(B * kk * 1152 / (t_best * 1e-6) / 1e9, 1)})
    zc = sweep[-1]["gbs"]
    return {"memcpy_h2d_gbs": best, "zero_copy_recall_gbs": zc, "peak_gbs": max(best, zc), "recall_miss_sweep": sweep,
            "how": "1 GiB pinned cudaMemcpyAsync; echo_cache_recall of 256 .. 65536 missed 1152-B rows into an "
                   "empty pool (best of 3 each); the largest gives zero_copy_recall_gbs"}


def allocator_bench(dev) -> dict:
    """The cache's allocator alone, the analog of the pages' alloc + free microbenchmark:
    on a full pool of 200,000 slots whose tokens were all last touched in an earlier step,
    echo_cache_evict frees the n least recently used slots and echo_cache_alloc binds n host
    indices to the freed slots (the ones just evicted, so the pool stays full and every pair
    evicts the next n in LRU order).  K pairs are captured in one CUDA Graph, as the decode
    step runs them, and timed per pair over one replay; evict and alloc are also timed apart
    with events recorded inside the graph.  Best of 3 replays per n."""
    import torch
    import sparse_attention_kv_dsa_gb300.echo as E
    i32 = torch.int32
    n_gpu, n_host, K = 200_000, 200_000, 16
    layer = E.LayerCache(n_gpu, n_host, torch.bfloat16, dev)
    out = torch.empty(n_gpu, dtype=i32, device=dev)
    all_hosts = torch.arange(n_gpu, dtype=i32, device=dev)
    n_all = torch.tensor([n_gpu], dtype=i32, device=dev)
    st = torch.cuda.Stream(dev)
    rows = []
    for n in (32, 512, 2048, 8192):
        need = torch.tensor([n], dtype=i32, device=dev)
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * K + 1)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            with torch.cuda.graph(g, stream=st):
                ev[0].record(st)
                for j in range(K):
                    E.cache_evict(layer, need, stream=st)
                    ev[2 * j + 1].record(st)
                    E.cache_alloc(layer, all_hosts[j * n:(j + 1) * n], need, out, stream=st)
                    ev[2 * j + 2].record(st)
        best = None
        for _ in range(3):
            # refill: every host index resident, touched in step 0, now step 1
            layer.reset()
            E.cache_alloc(layer, all_hosts, n_all, out)
            torch.cuda.synchronize()
            layer.counters[E.CTR_STEP] = 1
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            ev_us = [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(2 * K)]
            t = (sum(ev_us[0::2]) / K, sum(ev_us[1::2]) / K)
            best = t if best is None or sum(t) < sum(best) else best
        rows.append({"n": n, "evict_us": round(best[0], 1), "alloc_us": round(best[1], 1),
                     "evict_alloc_us": round(sum(best), 1)})
        del g
    status = layer.status()
    del layer
    torch.cuda.empty_cache()
    return {"pool_slots": n_gpu, "sweep": rows, "status": status,
            "how": "full pool of 200,000 slots; echo_cache_evict of the n least recently used, then echo_cache_alloc "
                   "of the n host indices just evicted; 16 pairs in one CUDA Graph, events inside the graph, mean "
                   "per pair, best of 3 replays (the pages: alloc + free 6-8 us on H20, context only)"}


def run_compare_prefetch(args, local) -> int:
    """Index + top-k + recall latency per layer-step, fused prefetch against the
    unfused index -> top-k -> recall sequence, on identical inputs.  Each mode's
    whole layer step is captured in one CUDA Graph (as it runs in production) and
    the segment from the indexer to the end of the recall is timed with events
    recorded inside the graph; eager per-stage times are reported beside it."""
    import ctypes
    import torch
    import sparse_attention_kv_dsa_gb300.echo as E
    from sparse_attention_kv_dsa_gb300 import synth as S
    from sparse_attention_kv_dsa_gb300.runtime import DecodeLayer, SharedScratch, StepInputs
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = S.workloads()[args.workload]
    wl.layers = 1
    steps = args.warmup + args.steps
    inp = StepInputs(wl, 1, steps + 1, dev, gen_device=dev)
    lib = E.lib()
    res = {}
    for mode in ("fused", "unfused"):
        sc = SharedScratch(wl, dev, wl.cap_max)
        dl = DecodeLayer(wl, 0, dev, prefetch=(mode == "fused"), scratch=sc, gen_device=dev)
        a = dl.args
        st = torch.cuda.Stream(dev)
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]

        def seg(stream):
            h = stream.cuda_stream
            E.check(lib.echo_cache_writeback(dl.cache.ref, a.new_kv, a.new_ik, a.idx_k, a.D, a.Lmax, a.idx_dtype,
                                             a.host_base, a.seq_len, a.B, h))
            if a.prefetch:
                E.check(lib.echo_cache_reserve(dl.cache.ref, a.seq_len, a.B, a.cap_max, a.cap_div, a.cap,
                                               a.pf_count, h))
            ev[0].record(stream)
            enqueue_index_topk(lib, dl, h, between=lambda: ev[1].record(stream))
            ev[2].record(stream)
            E.check(lib.echo_cache_recall(dl.cache.ref, a.sel, a.host_base, a.B, a.k,
                                          a.pf_list if a.prefetch else None, a.pf_count if a.prefetch else None,
                                          a.cap_max, a.stage_kv, a.miss_list, a.n_miss, a.slot_idx, h))
            ev[3].record(stream)
            E.check(lib.echo_sparse_mla_decode(a.q_mla, dl.cache.struct.gpu_kv, dl.cache.n_gpu,
                                               dl.cache.struct.kv_dtype, a.slot_idx, a.B, a.Hq, a.k,
                                               ctypes.c_float(a.scale), a.out, a.lse, a.mla_workspace,
                                               a.mla_workspace_bytes, h))

        dl.load_step_inputs(inp.q_ik[0][0], inp.new_ik_ik[0][0], inp.new_kv[0][0], inp.q_mla[0][0])
        with torch.cuda.stream(st):
            seg(st)                                     # first step eagerly (cold cache)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            seg(st)
        t_graph, t_ix, t_tk, t_rc, hits, staged, misses, rows, qual = [], [], [], [], 0, 0, 0, 0, 0
        for s in range(1, steps):
            dl.load_step_inputs(inp.q_ik[0][s], inp.new_ik_ik[0][s], inp.new_kv[0][s], inp.q_mla[0][s])
            with torch.cuda.stream(st):
                g.replay()
            st.synchronize()
            if s >= args.warmup:
                t_graph.append(ev[0].elapsed_time(ev[3]) * 1e3)
                t_ix.append(ev[0].elapsed_time(ev[1]) * 1e3)
                t_tk.append(ev[1].elapsed_time(ev[2]) * 1e3)
                t_rc.append(ev[2].elapsed_time(ev[3]) * 1e3)
                c = dl.cache.read_counters()
                hits += c[8]; staged += c[9]; misses += c[10]; rows += c[12]; qual += c[15]
        sel_n = hits + staged + misses
        res[mode] = {"index_topk_recall_us_in_graph": statistics.median(t_graph),
                     "stages_us_in_graph": {"index_prefetch_us": statistics.median(t_ix),
                                            "topk_us": statistics.median(t_tk),
                                            "recall_us": statistics.median(t_rc)},
                     "hit_rate": hits / sel_n, "hit_rate_after_prefetch": (hits + staged) / sel_n,
                     "misses_per_step": misses / args.steps,
                     "staged_rows_per_step": rows / args.steps, "qualifying_per_step": qual / args.steps,
                     "prefetch_precision": (staged / rows) if rows else None}
        del g, dl, sc
        torch.cuda.empty_cache()
    line = {"mode": "compare-prefetch", "workload": wl.name, "steps": args.steps, "warmup": args.warmup, **res,
            "speedup_fused": res["unfused"]["index_topk_recall_us_in_graph"] /
                             res["fused"]["index_topk_recall_us_in_graph"]}
    print(json.dumps(line), flush=True)
    return 0


def run_prefill(args, local) -> int:
    """Prefill chunk indexing of one request (a 2048-token chunk at positions 100K...):
    the time until every block's exact selection is resident (and, *_attn_us, until
    every block's queries have attended over their selections), for the serial
    pipeline, the overlapped one, and the overlapped one with the histogram
    candidates recalled early; plus the scoring kernel against the FP8 tensor roof
    (FP8 peak = 2 x the measured bf16 GEMM peak, the nominal dense ratio)."""
    import torch
    import sparse_attention_kv_dsa_gb300.echo as E
    from sparse_attention_kv_dsa_gb300 import synth as S
    from sparse_attention_kv_dsa_gb300.runtime import PrefillChunk
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = S.workloads()[args.workload]
    peaks = measured_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    out = {"mode": "prefill", "workload": wl.name, "ctx": wl.ctx[0], "chunk": wl.prefill_chunk, "topk": wl.topk,
           "reps": args.steps, "blocks": {}}
    for block in wl.prefill_blocks:
        pc = PrefillChunk(wl, block, dev, attend=True)
        res = {}
        for attend in (False, True):
            pc.attend = attend                              # with each block's sparse attention
            for mode in ("serial", "overlap", "echo"):
                ts = []
                for rep in range(args.warmup + args.steps):
                    pc.reset()
                    torch.cuda.synchronize()
                    t0, t1 = pc.run(mode)
                    torch.cuda.synchronize()
                    if rep >= args.warmup:
                        ts.append(t0.elapsed_time(t1) * 1e3)
                assert int(pc.status.item()) == 0 and pc.cache.status() == 0
                res[mode + ("_attn" if attend else "") + "_us"] = round(statistics.median(ts), 1)
        pc.attend = False
        # candidate recall vs exact recall of the last block (echo mode state)
        res["last_block_candidates"] = int(pc.cand[(pc.nblocks - 1) % 2].sum().item())
        res["last_block_misses_after_candidates"] = int(pc.nmiss[(pc.nblocks - 1) % 2].item())
        res["last_block_candidate_recall_misses"] = int(pc.nmiss_c[(pc.nblocks - 1) % 2].item())
        res["speedup_echo_vs_serial"] = round(res["serial_us"] / res["echo_us"], 3)
        res["speedup_echo_vs_overlap"] = round(res["overlap_us"] / res["echo_us"], 3)
        res["speedup_echo_vs_serial_with_attention"] = round(res["serial_attn_us"] / res["echo_attn_us"], 3)
        # the scoring kernel alone: middle block, CUDA events after a device-side delay
        i = pc.nblocks // 2
        pos0 = pc.ctx + i * block
        kp = torch.full((block,), 40.0, device=dev)
        ks = []
        for rep in range(5):
            torch.cuda._sleep(400000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            E.prefill_index(pc.q_all[i * block:(i + 1) * block], pc.w_all[i * block:(i + 1) * block], pc.idx_k,
                            pos0, kp, pc.scores[0], pc.hist[0], pc.status)
            e1.record()
            torch.cuda.synchronize()
            ks.append(e0.elapsed_time(e1) * 1e3)
        us = statistics.median(ks)
        flops = 2.0 * 64 * 128 * sum(pos0 + j + 1 for j in range(block))
        res["prefill_index_us"] = round(us, 1)
        res["prefill_index_roofline"] = {"bound": "tensor", "achieved": flops / (us * 1e-6) / 1e12,
                                         "peak": fp8_peak, "unit": "TFLOP/s",
                                         "frac": flops / (us * 1e-6) / 1e12 / fp8_peak,
                                         "peak_source": peaks["source"] + " bf16 GEMM x 2 (FP8 nominal ratio)"}
        out["blocks"][str(block)] = res
        del pc
        torch.cuda.empty_cache()
    print(json.dumps(out), flush=True)
    return 0


def run_cap_sweep(args, local) -> int:
    """Low-locality workload: miss-list size and recall time against the prefetch cap,
    for the fixed caps of the sweep and the adaptive cap (last step's transfer grown by
    the prediction error, plus a slack, at most the sweep's largest cap)."""
    import torch
    from sparse_attention_kv_dsa_gb300 import synth as S
    from sparse_attention_kv_dsa_gb300.runtime import DecodeLayer, SharedScratch, StepInputs
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = S.workloads()[args.workload]
    wl.layers = 1
    steps = args.warmup + args.steps
    inp = StepInputs(wl, 1, steps, dev, gen_device=dev)
    row_bytes = 576 * (4 if wl.kv_fp32 else 2)
    caps = [(c, None) for c in (wl.cap_sweep or [0, wl.cap_max])]
    caps.append((max(c for c, _ in caps), ADAPTIVE_SLACK))
    rows = []
    for cap, slack in caps:
        sc = SharedScratch(wl, dev, max(cap, 1))
        dl = DecodeLayer(wl, 0, dev, prefetch=cap > 0, cap_max=cap, scratch=sc, gen_device=dev,
                         adaptive_slack=slack)
        acc = {"index_prefetch_us": [], "topk_us": [], "recall_us": [], "misses": [], "staged": [], "staged_hits": [],
               "qualified": [], "cap_mean": [], "pred_err_median": []}
        for s in range(steps):
            dl.load_step_inputs(inp.q_ik[0][s], inp.new_ik_ik[0][s], inp.new_kv[0][s], inp.q_mla[0][s])
            st = stage_timing([dl], None, None, torch.cuda.current_stream(), 1, loaded=True)
            if s >= args.warmup:
                c = dl.cache.read_counters()
                for n in ("index_prefetch_us", "topk_us", "recall_us"):
                    acc[n].append(st[n])
                acc["misses"].append(c[10]); acc["staged"].append(c[12]); acc["staged_hits"].append(c[9])
                acc["qualified"].append(c[15])
                acc["cap_mean"].append(float(dl.cap.float().mean()))
                if slack is not None:
                    acc["pred_err_median"].append(float(dl.cache.pf_pred_err.median()))
        row = {"cap": cap if slack is None else f"adaptive (slack {slack}, at most {cap})",
               **{n: statistics.median(v) for n, v in acc.items() if v}}
        row["useless_prefetch_bytes"] = (row["staged"] - row["staged_hits"]) * row_bytes
        row["final_recall_bytes"] = row["misses"] * row_bytes
        rows.append(row)
        del dl, sc
        torch.cuda.empty_cache()
    print(json.dumps({"mode": "cap-sweep", "workload": wl.name, "steps": args.steps, "warmup": args.warmup,
                      "per_cap": rows,
                      "how": "per step medians of one layer: rows qualified / staged during scoring / staged and "
                             "selected, rows recalled after the top-k (misses), the mean per-request cap, and stage "
                             "times from events between the separate entry points"}), flush=True)
    return 0


ADAPTIVE_SLACK = 256


def run_blocks(args, local) -> int:
    """Decode with block granularity (T tokens per host index and GPU slot, the top-k/T
    blocks selected): every layer's step (write-back, indexer, block scores and block
    top-k, recall of whole blocks, sparse MLA over the selected blocks' tokens)
    captured in one CUDA Graph per step; per-replay CUDA events; per-stage times from
    a second graph with events between the stages."""
    import torch
    from sparse_attention_kv_dsa_gb300 import synth as S
    from sparse_attention_kv_dsa_gb300.runtime import BlockDecodeLayer, StepInputs
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = S.workloads()[args.workload]
    if args.layers:
        wl.layers = args.layers
    T = args.blocks
    kb = wl.topk // T
    steps = args.warmup + args.steps + 2
    inp = StepInputs(wl, wl.layers, steps, dev, gen_device=dev)
    L = [BlockDecodeLayer(wl, l, T, kb, dev, gen_device=dev) for l in range(wl.layers)]
    st = torch.cuda.Stream(dev)
    names = BlockDecodeLayer.STAGES
    sev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(names) + 1)]
           for _ in range(wl.layers)]

    def whole(stream, probe=False):
        with torch.cuda.stream(stream):
            for l, dl in enumerate(L):
                if probe:
                    sev[l][0].record(stream)
                dl.step(stream, mark=(lambda i, l=l: sev[l][i + 1].record(stream)) if probe else None)

    def load(s):
        for l, dl in enumerate(L):
            dl.load_step_inputs(inp.q_ik[l][s], inp.new_ik_ik[l][s], inp.new_kv[l][s], inp.q_mla[l][s])

    load(0)
    whole(st)                                            # first step eagerly (cold cache)
    st.synchronize()
    g, gp = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        whole(st)
    with torch.cuda.graph(gp, stream=st):
        whole(st, probe=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_step, misses, hits, stage = [], [], [], {n: [] for n in names}
    for s in range(1, steps):
        load(s)
        with torch.cuda.stream(st):
            probe = s == steps - 1 or s >= args.warmup + args.steps
            e0.record(st)
            (gp if probe else g).replay()
            e1.record(st)
        st.synchronize()
        if s < args.warmup:
            continue
        ctr = [dl.cache.read_counters() for dl in L]
        if probe:
            for l in range(wl.layers):
                for i, n in enumerate(names):
                    stage[n].append(sev[l][i].elapsed_time(sev[l][i + 1]) * 1e3)
        else:
            t_step.append(e0.elapsed_time(e1))
            misses.append(sum(c[10] for c in ctr))
            hits.append(sum(c[8] for c in ctr))
    status = [dl.cache.status() for dl in L]
    ms = statistics.median(t_step)
    row_bytes = T * wl.kv_width * (4 if wl.kv_fp32 else 2)
    n_req = wl.batch // max(wl.kv_heads, 1)
    print(json.dumps({
        "mode": "blocks", "workload": wl.name, "layers": wl.layers, "batch": n_req,
        "kv_heads": wl.kv_heads or None, "attention": "gqa" if wl.kv_heads else "mla",
        "block_tokens": T, "blocks_selected": kb, "gpu_blocks": L[0].n_gpu_blocks, "host_blocks": L[0].n_host_blocks,
        "steps": len(t_step), "warmup": args.warmup, "ms_per_step": ms, "step_ms": [round(x, 3) for x in t_step],
        "tokens_per_s": n_req / (ms * 1e-3),
        "stages_us_per_layer": {n + "_us": round(statistics.median(v), 2) for n, v in stage.items() if v},
        "block_hit_rate": sum(hits) / max(sum(hits) + sum(misses), 1),
        "recalled_blocks_per_step": statistics.median(misses),
        "recall_bytes_per_step": statistics.median(misses) * row_bytes,
        "device_status": status,
        "how": "one CUDA Graph per step over every layer, CUDA events around each replay (inputs loaded "
               "before the start event); stage times from a graph with events between the stages"}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="echo", choices=["echo", "reference"])
    ap.add_argument("--workload", default=None, help=f"default {DEFAULT_WL}")
    ap.add_argument("--no-prefetch", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-stages", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling)")
    ap.add_argument("--compare-prefetch", action="store_true",
                    help="fused vs unfused index+top-k+recall latency (default workload: decode-b8-ctx64k)")
    ap.add_argument("--cap-sweep", action="store_true",
                    help="prefetch-cap sweep (default workload: lowlocality-b16-ctx100k)")
    ap.add_argument("--skip-host-link", action="store_true")
    ap.add_argument("--prefill", action="store_true",
                    help="prefill chunk indexing: serial / overlapped / candidate-prefetch pipelines "
                         "(default workload: prefill-chunk2048-ctx100k)")
    ap.add_argument("--blocks", type=int, default=0,
                    help="decode with block granularity: T tokens per host index and GPU slot")
    ap.add_argument("--fill-max", type=int, default=96,
                    help="untimed steps, at most, that bring the GPU pool to its steady (full) state")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    ws, rank, local = dist_setup()
    if args.compare_prefetch:
        args.workload = args.workload or "decode-b8-ctx64k"
        return run_compare_prefetch(args, local)
    if args.cap_sweep:
        args.workload = args.workload or "lowlocality-b16-ctx100k"
        return run_cap_sweep(args, local)
    if args.prefill:
        args.workload = args.workload or "prefill-chunk2048-ctx100k"
        return run_prefill(args, local)
    if args.blocks:
        args.workload = args.workload or DEFAULT_WL
        return run_blocks(args, local)
    args.workload = args.workload or DEFAULT_WL
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_echo(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
