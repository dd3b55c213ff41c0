"""Single C-ABI calls on the GPU against the oracle and the golden hand-worked
examples: indexer, top-k + EMA, cache manager (LRU golden sequence, evict, alloc),
recall copies, sparse MLA, and the device status word."""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import sparse_attention_kv_dsa_gb300.echo as E
from sparse_attention_kv_dsa_gb300 import synth as S

pytestmark = pytest.mark.gpu
dev = "cuda"


def golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ indexer --
def test_indexer_hand_example_f32(golden_dir):
    g = golden(golden_dir, "indexer_8tok.json")
    q = torch.zeros(1, 2, 4, device=dev)
    q[0, :, :2] = torch.tensor(g["q"], dtype=torch.float32)
    keys = torch.zeros(1, 8, 4, device=dev)
    keys[0, :, :2] = torch.tensor(g["keys"], dtype=torch.float32)
    w = torch.tensor([g["w"]], dtype=torch.float32, device=dev)
    scores = torch.full((1, 8), -7.0, device=dev)
    E.index_prefetch(q, w, keys, torch.tensor([8], dtype=torch.int32, device=dev),
                     torch.tensor([math.inf], device=dev), scores)
    torch.cuda.synchronize()
    assert scores[0].cpu().tolist() == g["scores"]


@pytest.mark.parametrize("ctx", [(1, 128, 129), (700, 1500, 333, 4096, 5)])
def test_indexer_fp8_bit_exact(ctx):
    wl = S.small_workload("ix", ctx=ctx)
    B, Lmax = wl.batch, wl.max_ctx
    keys = torch.zeros(B, Lmax, 128, dtype=torch.int8)
    for b in range(B):
        keys[b, :ctx[b]] = S.keys_for(wl, 0, b, ctx[b])
    q = S.qidx_initial(wl, 0)
    w = S.weights_for(wl, 0)
    scores = torch.full((B, Lmax), -1.0, device=dev)
    E.index_prefetch(S.grid_to_fp8(q.to(dev)), w.to(dev), S.grid_to_fp8(keys.to(dev)),
                     torch.tensor(ctx, dtype=torch.int32, device=dev), torch.full((B,), math.inf, device=dev), scores)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    for b in range(B):
        ref = O.to_f32_exact(O.indexer_scores(S.grid_to_float(q[b]).numpy(), w[b].numpy(),
                                              S.grid_to_float(keys[b, :ctx[b]]).numpy()))
        assert np.array_equal(sc[b, :ctx[b]], ref), f"request {b}"
        assert np.all(sc[b, ctx[b]:] == -1.0), "wrote past the context"


def test_indexer_fp8_extreme_grid_values():
    # every product at +1 (the largest sums) and mixed signs: still exact
    B, L = 2, 300
    q = torch.full((B, 64, 128), 8, dtype=torch.int8)
    q[1, ::2] = -8
    keys = torch.full((B, L, 128), 8, dtype=torch.int8)
    keys[:, 1::3] = -8
    w = torch.ones(B, 64)
    scores = torch.zeros(B, L, device=dev)
    E.index_prefetch(S.grid_to_fp8(q.to(dev)), w.to(dev), S.grid_to_fp8(keys.to(dev)),
                     torch.tensor([L, L], dtype=torch.int32, device=dev), torch.full((B,), math.inf, device=dev),
                     scores)
    torch.cuda.synchronize()
    for b in range(B):
        ref = O.to_f32_exact(O.indexer_scores(S.grid_to_float(q[b]).numpy(), w[b].numpy(),
                                              S.grid_to_float(keys[b]).numpy()))
        assert np.array_equal(scores[b].cpu().numpy(), ref)
    assert scores[0, 0].item() == 8192.0


# -------------------------------------------------------------------- top-k --
def run_topk(scores_list, k, theta0, alpha=0.5, kth0=None):
    B = len(scores_list)
    Lmax = max(max(len(s) for s in scores_list), 1)
    sc = torch.full((B, Lmax), -123.0)
    for b, s in enumerate(scores_list):
        sc[b, :len(s)] = torch.tensor(s, dtype=torch.float32)
    sc = sc.to(dev)
    seq = torch.tensor([len(s) for s in scores_list], dtype=torch.int32, device=dev)
    out = torch.full((B, k), -5, dtype=torch.int32, device=dev)
    kth = torch.empty(B, device=dev) if kth0 is None else torch.tensor(kth0, dtype=torch.float32, device=dev)
    theta = torch.tensor(theta0, dtype=torch.float32, device=dev)
    E.topk(sc, seq, k, out, kth, theta, alpha)
    torch.cuda.synchronize()
    return out.cpu().numpy(), kth.cpu().numpy(), theta.cpu().numpy()


def check_topk(scores_list, k, theta0, alpha=0.5, kth0=None):
    out, kth, theta = run_topk(scores_list, k, theta0, alpha, kth0)
    for b, s in enumerate(scores_list):
        s = np.asarray(s, dtype=np.float32)
        sel, kv = O.topk_select(s, k)
        n = len(sel)
        assert set(out[b, :n].tolist()) == set(sel.tolist()), f"request {b}"
        assert np.all(out[b, n:] == -1)
        assert kth[b] == np.float32(kv)
        assert theta[b] == O.ema_update(theta0[b], kv, alpha)


def test_topk_hand_example(golden_dir):
    g = golden(golden_dir, "indexer_8tok.json")
    out, kth, theta = run_topk([g["scores"], g["scores"]], 3, [math.inf, 1.0])
    assert sorted(out[0].tolist()) == g["top3"] and kth[0] == g["top3_kth"]
    assert theta[0] == np.float32(0.75) and theta[1] == np.float32(g["ema"]["out"])


def test_topk_random_with_ties_and_edges():
    rng = np.random.default_rng(0)
    k = 256
    lists = [rng.integers(0, 40, L).astype(np.float32) / 8 for L in (0, 1, 255, 256, 257, 3000, 70_001)]
    lists.append(np.full(5000, 2.5, dtype=np.float32))           # all equal: lowest indices
    lists.append(rng.standard_normal(9000).astype(np.float32))   # negative scores too
    check_topk(lists, k, [math.inf, 1.0, 2.0, math.inf, 3.0, 4.0, 5.0, math.inf, 0.5])


def test_topk_all_equal_takes_lowest_indices():
    out, kth, _ = run_topk([np.full(10_000, 7.0)], 2048, [math.inf])
    assert sorted(out[0].tolist()) == list(range(2048)) and kth[0] == 7.0


def test_topk_many_rows():
    # more rows than two per SM (prefill blocks run one row per query): ragged lengths,
    # ties, rows shorter than k, predictions inside and outside the window
    rng = np.random.default_rng(4)
    n_rows = 2 * E.lib().echo_device_sm_count() + 5
    k = 256
    lists, thetas = [], []
    for r in range(n_rows):
        L = int(rng.integers(0, 4000)) if r % 7 else int(rng.integers(0, 300))
        lists.append((rng.integers(0, 200, L) / 16.0).astype(np.float32))
        thetas.append([math.inf, 3.0, 11.5, 0.25][r % 4])
    check_topk(lists, k, thetas)


def test_topk_many_long_rows_take_smaller_clusters():
    # more rows than clusters of eight fit in one wave, each too long for one CTA's
    # shared memory: clusters of two; predictions inside, above and below the window
    rng = np.random.default_rng(8)
    n_rows = E.lib().echo_device_sm_count() // 4 + 3
    lists = [(rng.integers(0, 2 ** 14, int(rng.integers(30_000, 46_000))) / 1024.0).astype(np.float32)
             for _ in range(n_rows)]
    check_topk(lists, 2048, [[math.inf, 15.6, 60.0, 1.0][r % 4] for r in range(n_rows)])
    lists = [(rng.integers(0, 2 ** 14, int(rng.integers(70_000, 90_000))) / 1024.0).astype(np.float32)
             for _ in range(n_rows)]                                    # clusters of four
    check_topk(lists, 2048, [[15.6, math.inf][r % 2] for r in range(n_rows)])


def test_topk_candidate_lists_and_their_fallbacks():
    # a prediction near the k-th score: the last pass and the output read the per-warp
    # candidate lists; ties at the k-th key spread over every warp and CTA; a window
    # that holds nearly every key overflows the lists and falls back to full passes
    rng = np.random.default_rng(6)
    L = 100_000
    a = (rng.integers(0, 2 ** 14, L) / 1024.0).astype(np.float32)          # k-th near 15.7
    b = rng.choice(np.array([0.0, 1.0, 2.0], np.float32), L, p=[0.6, 0.35, 0.05])   # ~5000 twos
    c = (2.5 + rng.integers(-8, 8, L) / 4096.0).astype(np.float32)         # all in the window
    # windows above and below the k-th key: full passes
    check_topk([a, b, c, a, a], 2048, [15.6, 2.0, 2.5, 60.0, 1.0])


def test_topk_window_width_from_the_previous_kth():
    # the k-th score left in kth by the previous call sizes the window around theta:
    # no hint (NaN, -inf), a hint at theta (the narrowest window, 2^17 keys each side;
    # the k-th key just inside it), a hint at theta whose window misses the k-th key (full
    # passes), and a far hint (the widest window) all give the exact selection
    rng = np.random.default_rng(9)
    a = (rng.integers(0, 2 ** 14, 100_000) / 1024.0).astype(np.float32)  # k-th near 15.7
    rows = [a] * 6
    check_topk(rows, 2048, [15.6, 15.6, 15.6, 15.0, 15.6, 16.2],
               kth0=[math.nan, -math.inf, 15.6, 15.0, 1.0, 16.2])


def test_topk_large_context_k2048():
    rng = np.random.default_rng(1)
    lists = [(rng.integers(0, 2 ** 14, 100_000) / 1024.0).astype(np.float32) for _ in range(3)]
    check_topk(lists, 2048, [math.inf, 10.0, 5.5])


# ----------------------------------------------------- cache: golden LRU ----
class TinyLayer:
    """A layer cache driven by direct API calls (no indexer)."""

    def __init__(self, n_gpu, n_host, B=1, kv32=True):
        self.dt = torch.float32 if kv32 else torch.bfloat16
        host = S.normal(5, (n_host, 576), self.dt).pin_memory()
        self.c = E.LayerCache(n_gpu, n_host, self.dt, dev, host_kv=host)
        self.c.reset()
        self.idx_k = torch.zeros(B, 64, 4, device=dev)
        torch.cuda.synchronize()

    def writeback(self, host_base, seq_len, new_kv=None):
        B = seq_len.shape[0]
        new_kv = new_kv if new_kv is not None else torch.zeros(B, 576, dtype=self.dt, device=dev)
        E.cache_writeback(self.c, new_kv, torch.zeros(B, 4, device=dev), self.idx_k, host_base, seq_len)

    def recall(self, sel, host_base, staged=None, cap_max=8):
        B, k = sel.shape
        miss = torch.empty(B, k, dtype=torch.int32, device=dev)
        n_miss = torch.empty(B, dtype=torch.int32, device=dev)
        slot = torch.empty(B, k, dtype=torch.int32, device=dev)
        kw = {}
        if staged is not None:
            pf_list = torch.full((B, cap_max), -1, dtype=torch.int32, device=dev)
            pf_count = torch.zeros(B, dtype=torch.int32, device=dev)
            stage = torch.zeros(B * cap_max, 576, dtype=self.dt, device=dev)
            for b, toks in enumerate(staged):
                for i, t in enumerate(toks):
                    row = b * cap_max + i
                    pf_list[b, i] = t
                    h = int(host_base[b]) + t
                    self.c.host2gpu[h] = -2 - row                 # state hand-off: staged mark
                    stage[row] = self.c.host_kv[h].to(dev)
                pf_count[b] = len(toks)
            kw = dict(pf_list=pf_list, pf_count=pf_count, cap_max=cap_max, stage_kv=stage)
        E.cache_recall(self.c, sel, host_base, miss, n_miss, slot, **kw)
        torch.cuda.synchronize()
        return miss.cpu().numpy(), n_miss.cpu().numpy(), slot.cpu().numpy()


def test_lru_golden_sequence_on_gpu(golden_dir):
    from harness import gpu_residency, check_gpu_maps
    g = golden(golden_dir, "lru_ng4.json")
    t = TinyLayer(g["n_gpu"], g["n_host"])
    hb = torch.tensor(g["host_base"], dtype=torch.int32, device=dev)
    seq = torch.tensor([g["seq_len0"]], dtype=torch.int32, device=dev)
    for st in g["steps"]:
        t.writeback(hb, seq)
        torch.cuda.synchronize()
        assert gpu_residency(t.c) == {int(k): v for k, v in st["after_wb"].items()}
        t.c.counters[2] = 0                                   # clear the sticky status between steps
        sel = torch.tensor([st["sel"]], dtype=torch.int32, device=dev)
        miss, n_miss, slot = t.recall(sel, hb, staged=[st["staged"]] if st["staged"] else None)
        assert sorted(miss[0, :n_miss[0]].tolist()) == st["misses"]
        assert gpu_residency(t.c) == {int(k): v for k, v in st["resident"].items()}
        g2h = t.c.gpu2host.cpu().numpy()
        got = [int(g2h[s]) if s >= 0 else -1 for s in slot[0]]
        assert got == st["slot_host"]
        assert t.c.status() == st["status"]
        t.c.counters[2] = 0
        check_gpu_maps(t.c)
        # recalled rows hold the host data
        kv = t.c.gpu_kv.cpu()
        for s, h in zip(slot[0], got):
            if s >= 0:
                assert torch.equal(kv[s], t.c.host_kv[h])


def test_evict_and_alloc_match_oracle_victims():
    from harness import gpu_residency, check_gpu_maps
    rng = np.random.default_rng(3)
    for trial in range(6):
        n_gpu, n_host = int(rng.integers(50, 3000)), 10_000
        t = TinyLayer(n_gpu, n_host)
        oc = O.LayerCache(n_gpu, n_host)
        # random resident state with priorities < step, handed to both sides
        used = rng.choice(n_gpu, int(rng.integers(0, n_gpu + 1)), replace=False)
        hosts = rng.choice(n_host, used.size, replace=False)
        prio = rng.integers(0, 9, used.size)
        step = 9
        for g_, h_, p_ in zip(used, hosts, prio):
            oc.free[g_] = False
            oc.gpu2host[g_] = h_
            oc.host2gpu[h_] = g_
            oc.priority[g_] = p_
        oc.step = step
        t.c.gpu2host.copy_(torch.tensor(oc.gpu2host, dtype=torch.int32))
        t.c.host2gpu.copy_(torch.tensor(oc.host2gpu, dtype=torch.int32))
        t.c.priority.copy_(torch.tensor(oc.priority, dtype=torch.int32))
        t.c.free_map.copy_(torch.tensor(oc.free.astype(np.uint8)))
        t.c.counters[0] = step
        t.c.counters[1] = int(oc.free.sum())
        need = int(rng.integers(0, n_gpu + 5))
        E.cache_evict(t.c, torch.tensor([need], dtype=torch.int32, device=dev))
        torch.cuda.synchronize()
        v = oc.lru_victims(max(0, need - oc.n_free()))
        oc.evict(v)
        assert gpu_residency(t.c) == oc.resident_priority()
        check_gpu_maps(t.c)
        expect_status = 0 if need - (n_gpu - used.size) <= used.size else 5
        assert t.c.status() == expect_status
        t.c.counters[2] = 0
        # allocate some new tokens (any free slots), stamped with the step
        free_hosts = np.setdiff1d(np.arange(n_host), oc.gpu2host[oc.gpu2host >= 0])
        n = int(min(oc.n_free(), rng.integers(0, 200)))
        toks = rng.choice(free_hosts, n, replace=False).astype(np.int32)
        out = torch.full((max(n, 1),), -7, dtype=torch.int32, device=dev)
        hi = torch.tensor(toks if n else np.zeros(1, np.int32), device=dev)
        E.cache_alloc(t.c, hi, torch.tensor([n], dtype=torch.int32, device=dev), out)
        torch.cuda.synchronize()
        for h_ in toks:
            oc.bind(int(h_))
        assert gpu_residency(t.c) == oc.resident_priority()
        check_gpu_maps(t.c)
        o = out.cpu().numpy()[:n]
        assert np.all(t.c.gpu2host.cpu().numpy()[o] == toks)


def test_pending_victim_writeback_matches_oracle():
    # Pools of at least 14080 slots: each recall also ranks the next write-back's B
    # victims, and the write-back binds them in one CTA.  Residency must equal the
    # oracle's LRU after every call; manager word 19 tells which path the write-back
    # took.  The iterations cover: free slots left (full path), a new token made resident by
    # the recall (fewer victims than listed), a write-back of a subset of the requests,
    # an eviction between recall and write-back (list dropped), two recalls in a step.
    from harness import gpu_residency, check_gpu_maps
    n_gpu, n_host, B, k = 14336, 60000, 6, 1536
    t = TinyLayer(n_gpu, n_host, B=B, kv32=False)
    t.idx_k = torch.zeros(B, 9600, 4, device=dev)
    oc = O.LayerCache(n_gpu, n_host)
    hb_np = np.arange(B, dtype=np.int64) * 9700
    hb = torch.tensor(hb_np, dtype=torch.int32, device=dev)
    seq_np = np.full(B, 9000, dtype=np.int64)
    rng = np.random.default_rng(11)
    path = []

    def writeback(reqs):
        seq_t = torch.tensor(seq_np[reqs], dtype=torch.int32, device=dev)
        t.writeback(hb[reqs].contiguous(), seq_t)
        torch.cuda.synchronize()
        s_sub = seq_np[reqs].copy()
        oc.writeback(hb_np[reqs], s_sub)
        seq_np[reqs] = s_sub
        assert np.array_equal(seq_t.cpu().numpy(), s_sub)
        path.append(int(t.c.counters[19].item()))
        assert gpu_residency(t.c) == oc.resident_priority(), "residency after the write-back"
        check_gpu_maps(t.c)
        assert t.c.status() == 0

    def recall(extra=None, sel_np=None):
        if sel_np is None:
            sel_np = np.stack([rng.choice(int(seq_np[b]), k, replace=False) for b in range(B)]).astype(np.int32)
        if extra is not None:                                  # request 0's next new token
            sel_np[0, 0] = extra
        miss, n_miss, slot = t.recall(torch.tensor(sel_np, device=dev), hb)
        rec = oc.recall([sel_np[b] for b in range(B)], hb_np, [np.zeros(0, dtype=np.int64)] * B)
        assert rec.status == 0 and t.c.status() == 0
        for b in range(B):
            assert set(miss[b, :n_miss[b]].tolist()) == set(rec.misses[b])
        assert gpu_residency(t.c) == oc.resident_priority(), "residency after the recall"
        check_gpu_maps(t.c)
        return sel_np

    for it in range(11):
        writeback(np.arange(B))
        sel = recall(extra=int(seq_np[0]) if it == 5 else None)
        if it == 7:
            # a second recall in the same step: the same selection with 60 tokens per
            # request replaced (the first one's tokens are protected now)
            for b in range(B):
                fresh = np.setdiff1d(np.arange(int(seq_np[b])), sel[b])
                sel[b, :60] = rng.choice(fresh, 60, replace=False)
            recall(sel_np=sel)
        if it == 8:
            n = torch.tensor([40], dtype=torch.int32, device=dev)
            E.cache_evict(t.c, n)
            torch.cuda.synchronize()
            oc.evict(oc.lru_victims(40 - oc.n_free()))
            assert gpu_residency(t.c) == oc.resident_priority()
        if it == 9:
            writeback(np.array([1, 3, 4]))                     # a subset of the requests
            recall()
    # iteration 0 is cold, iteration 1 has free slots: full path; once the pool is full
    # the write-back takes the list, except after the eviction of iteration 8
    assert path[0] == 0 and path[1] == 0
    assert all(p == 1 for p in path[2:9]), path
    assert path[9] == 0, "the eviction must drop the list"
    assert path[10] == 1 and path[11] == 1, path
    # the oracle's victims of a write-back are the list's: the last write-back evicted B
    assert int(t.c.counters[13].item()) == B


# ---------------------------------------------------------- status words ----
def test_status_host_index_out_of_range():
    t = TinyLayer(8, 16)
    hb = torch.tensor([14], dtype=torch.int32, device=dev)
    seq = torch.tensor([5], dtype=torch.int32, device=dev)    # h = 19 >= n_host
    t.writeback(hb, seq)
    assert t.c.status() == E.ERR_HOST_INDEX


def test_invalid_arguments_are_rejected():
    t = TinyLayer(8, 16)
    with pytest.raises(E.EchoError) as ei:
        E.topk(torch.zeros(1, 4, device=dev), torch.tensor([4], dtype=torch.int32, device=dev), 0,
               torch.zeros(1, 1, dtype=torch.int32, device=dev), torch.zeros(1, device=dev),
               torch.zeros(1, device=dev))
    assert ei.value.code == E.ERR_INVALID_ARG
    with pytest.raises(E.EchoError) as ei:
        q = torch.zeros(1, 32, 128, dtype=torch.float8_e4m3fn, device=dev)   # FP8 path needs 64 heads
        E.index_prefetch(q, torch.zeros(1, 32, device=dev), torch.zeros(1, 128, 128, dtype=torch.float8_e4m3fn,
                                                                         device=dev),
                         torch.tensor([4], dtype=torch.int32, device=dev), torch.zeros(1, device=dev),
                         torch.zeros(1, 128, device=dev))
    assert ei.value.code == E.ERR_UNSUPPORTED
    del t


# ---------------------------------------------------------------- attention --
def mla(q, kv, idx, scale):
    B, Hq, _ = q.shape
    k = idx.shape[1]
    out = torch.empty(B, Hq, 512, dtype=q.dtype, device=dev)
    lse = torch.empty(B, Hq, device=dev)
    ws = torch.empty(E.mla_workspace_bytes(B, Hq, k), dtype=torch.uint8, device=dev)
    E.sparse_mla_decode(q, kv, idx, scale, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse


# bf16 k = 2048 / 300 / 600 / 1300 / 2600 / 4096 / 4700: 4 / 1 / 2 / 3 / 6 / 8 / 10 splits
# of 512 entries (the combine takes its register path up to 8 splits and its loop beyond)
@pytest.mark.parametrize("dtype,Hq,k", [(torch.bfloat16, 128, 2048), (torch.bfloat16, 128, 300),
                                        (torch.bfloat16, 128, 600), (torch.bfloat16, 128, 1300),
                                        (torch.bfloat16, 128, 2600), (torch.bfloat16, 128, 4096),
                                        (torch.bfloat16, 128, 4700),
                                        (torch.float32, 16, 256), (torch.float32, 16, 77)])
def test_mla_vs_oracle(dtype, Hq, k):
    B, N = 3, 5000
    kv = S.normal(11, (N, 576), dtype)
    q = S.normal(12, (B, Hq, 576), dtype)
    g = torch.Generator().manual_seed(13)
    idx = torch.stack([torch.randperm(N, generator=g)[:k] for _ in range(B)]).to(torch.int32)
    idx[1, k // 2:] = -1                       # a request with padding
    scale = 1 / math.sqrt(576)
    out, lse = mla(q.to(dev), kv.to(dev), idx.to(dev), scale)
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-5
    for b in range(B):
        sel = idx[b][idx[b] >= 0].long()
        o, l = O.sparse_mla_decode(q[b].double().numpy(), kv[sel].double().numpy(), scale)
        assert np.abs(out[b].float().cpu().numpy() - o).max() <= tol
        assert np.abs(lse[b].cpu().numpy() - l).max() <= (2e-2 if dtype == torch.bfloat16 else 1e-4)


def test_mla_closed_forms(golden_dir):
    g = golden(golden_dir, "mla_closed_form.json")
    for dtype in (torch.float32, torch.bfloat16):
        Hq = 16 if dtype == torch.float32 else 128
        kv = S.normal(21, (6, 576), dtype).to(dev)
        kv[0, 0], kv[1, 0] = 0.0, 1.0
        q = torch.zeros(1, Hq, 576, dtype=dtype, device=dev)
        q[..., 0] = math.log(3.0)
        out, lse = mla(q, kv, torch.tensor([[0, 1]], dtype=torch.int32, device=dev), 1.0)
        p = g["two_token"]["p"]
        exp = (p[0] * kv[0, :512].double() + p[1] * kv[1, :512].double()).cpu().numpy()
        tol = 1e-5 if dtype == torch.float32 else 2e-2
        assert np.abs(out[0].float().cpu().numpy() - exp[None]).max() <= tol
        # bf16 rounds q = ln 3 to 1.1015625, so the closed form holds to bf16 precision there
        assert np.abs(lse.cpu().numpy() - g["two_token"]["lse"]).max() <= (1e-5 if dtype == torch.float32 else 5e-3)
        out, _ = mla(q, kv, torch.tensor([[3]], dtype=torch.int32, device=dev), 1.0)    # single token: a copy
        assert torch.equal(out[0], kv[3, :512].expand(Hq, 512))
        n = g["equal_logits"]["n"]
        out, lse = mla(torch.zeros_like(q), kv, torch.arange(n, dtype=torch.int32, device=dev)[None], 1.0)
        assert np.abs(out[0].float().cpu().numpy() - kv[:n, :512].double().mean(0).cpu().numpy()[None]).max() <= tol
        assert abs(lse[0, 0].item() - math.log(n)) < 1e-5


def test_mla_no_valid_entry():
    q = torch.ones(1, 16, 576, device=dev)
    out, lse = mla(q, torch.ones(4, 576, device=dev), torch.full((1, 8), -1, dtype=torch.int32, device=dev), 1.0)
    assert torch.all(out == 0) and torch.all(torch.isinf(lse)) and torch.all(lse < 0)
