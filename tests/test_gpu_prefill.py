"""Prefill chunk indexing on the GPU against the oracle: block scores (bit-exact on
the FP8 grid), the 256-bucket histograms, threshold buckets and candidate sets, the
bitmap unions and token lists, the exact per-query top-k of the block, and the
recall of a block's union through the one-request recall.  Small blocks span
several key tiles, a ragged tile tail and a query count that is not a multiple of
four; the full-size block (512 queries at positions 100K...) is checked on samples
and by invariants."""

import numpy as np
import pytest
import torch

import oracle as O
import sparse_attention_kv_dsa_gb300.echo as E
from sparse_attention_kv_dsa_gb300 import synth as S

pytestmark = pytest.mark.gpu
dev = "cuda"


def block_inputs(wl, pos0, Q, seed_layer=0):
    L = pos0 + Q
    k_int = S.keys_for(wl, seed_layer, 0, L + 5)           # a few spare rows past the block
    q_int = S.prefill_queries(wl, seed_layer, pos0 + Q)[pos0:pos0 + Q]
    w = S.prefill_weights(wl, seed_layer, pos0 + Q)[pos0:pos0 + Q]
    return k_int, q_int, w


def run_block(k_int, q_int, w, pos0, kth_pred, k):
    Q = q_int.shape[0]
    Lmax = k_int.shape[0]
    keys = S.grid_to_fp8(k_int.to(dev))
    q = S.grid_to_fp8(q_int.to(dev)).contiguous()
    scores = torch.full((Q, Lmax), float("nan"), device=dev)
    hist = torch.empty(Q, 256, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kp = torch.tensor(kth_pred, dtype=torch.float32, device=dev)
    E.prefill_index(q, w.to(dev), keys, pos0, kp, scores, hist, status)
    nw = (Lmax + 31) // 32
    bitmap = torch.zeros(nw, dtype=torch.int32, device=dev)
    thr = torch.empty(Q, dtype=torch.int32, device=dev)
    cnt = torch.empty(Q, dtype=torch.int32, device=dev)
    E.prefill_candidates(scores, hist, pos0, k, kp, bitmap, thr, cnt)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return scores, hist, bitmap, thr, cnt


@pytest.mark.parametrize("pos0,Q,k", [(2500, 37, 256), (300, 8, 64), (1000, 4, 2048)])
def test_prefill_block_matches_oracle(pos0, Q, k):
    wl = S.workloads()["prefill-chunk2048-ctx100k"]
    k_int, q_int, w = block_inputs(wl, pos0, Q)
    keys_f = S.grid_to_float(k_int).numpy().astype(np.float64)
    qf = S.grid_to_float(q_int).numpy().astype(np.float64)
    wf = w.numpy().astype(np.float64)
    rng = np.random.default_rng(pos0)
    kth_pred = (rng.integers(0, 40, Q) * 0.25).astype(np.float32)   # any prediction; both sides use it
    kth_pred[0] = np.inf                                             # first block: nothing predicted
    scores, hist, bitmap, thr, cnt = run_block(k_int, q_int, w, pos0, kth_pred, k)
    ref = O.prefill_block(qf, wf, keys_f, pos0, kth_pred, k)
    sc = scores.cpu().numpy()
    hi = hist.cpu().numpy().astype(np.int64)
    th = thr.cpu().numpy()
    cn = cnt.cpu().numpy()
    for j in range(Q):
        L = pos0 + j + 1
        assert np.array_equal(sc[j, :L], ref["scores"][j]), f"scores, query {j}"
        assert np.isnan(sc[j, L:]).all(), "entries past the causal range are untouched"
        assert np.array_equal(hi[j], ref["hist"][j]), f"histogram, query {j}"
        assert th[j] == ref["thr"][j], f"threshold bucket, query {j}"
        assert cn[j] == len(ref["cand"][j]), f"candidate count, query {j}"
    # union of the candidates, as a bitmap and as a token list
    words = bitmap.cpu().numpy().view(np.uint32)
    got = [t for t in range(words.size * 32) if (words[t >> 5] >> (t & 31)) & 1]
    assert got == ref["cand_union"].tolist()
    lst = torch.empty(k_int.shape[0], dtype=torch.int32, device=dev)
    count = torch.empty(1, dtype=torch.int32, device=dev)
    E.token_list(bitmap, k_int.shape[0], lst, count)
    torch.cuda.synchronize()
    n = int(count.item())
    assert n == len(ref["cand_union"])
    assert lst[:n].cpu().tolist() == ref["cand_union"].tolist() and bool((lst[n:] == -1).all())
    assert int(bitmap.abs().sum().item()) == 0, "token_list leaves the bitmap clear"
    # exact per-query top-k of the block through the decode top-k (one row per query)
    seq = torch.arange(pos0 + 1, pos0 + Q + 1, dtype=torch.int32, device=dev)
    sel = torch.empty(Q, k, dtype=torch.int32, device=dev)
    kth = torch.empty(Q, device=dev)
    theta = torch.tensor(kth_pred, device=dev)
    E.topk(scores.nan_to_num(nan=-1.0), seq, k, sel, kth, theta)
    torch.cuda.synchronize()
    s_np = sel.cpu().numpy()
    for j in range(Q):
        n_j = min(k, pos0 + j + 1)
        assert set(s_np[j, :n_j].tolist()) == set(ref["sel"][j].tolist()), f"top-k, query {j}"
        assert set(ref["cand"][j].tolist()) <= set(s_np[j, :n_j].tolist())
    assert np.array_equal(kth.cpu().numpy(), ref["kth"])
    # union of the selections
    E.mark_tokens(sel, bitmap, k_int.shape[0])
    E.token_list(bitmap, k_int.shape[0], lst, count)
    torch.cuda.synchronize()
    n = int(count.item())
    assert lst[:n].cpu().tolist() == ref["sel_union"].tolist()


def test_prefill_union_recall_matches_oracle():
    # the block's union recalled as one request: residency as in the oracle's recall
    from harness import check_gpu_maps, gpu_residency
    wl = S.small_workload("prefill-recall", ctx=(3000,), topk=128, n_gpu=1500, steps=1)
    base = 7
    n_host = 3100 + base
    cache = E.LayerCache(wl.n_gpu, n_host, torch.bfloat16, dev)
    cache.reset()
    cache.host_kv.copy_(S.latents_for(wl, 0, n_host))
    oc = O.LayerCache(wl.n_gpu, n_host)
    rng = np.random.default_rng(2)
    lat = cache.host_kv.float().numpy()
    for rnd in range(3):                                   # later rounds evict earlier ones
        toks = np.unique(rng.integers(0, 3000, 700 + 300 * rnd))
        bitmap = torch.zeros(3100 // 32 + 1, dtype=torch.int32, device=dev)
        E.mark_tokens(torch.tensor(toks, dtype=torch.int32, device=dev).view(1, -1), bitmap, 3100)
        lst = torch.empty(1, 3100, dtype=torch.int32, device=dev)
        count = torch.empty(1, dtype=torch.int32, device=dev)
        E.token_list(bitmap, 3100, lst, count)
        miss = torch.empty(1, 3100, dtype=torch.int32, device=dev)
        nmiss = torch.zeros(1, dtype=torch.int32, device=dev)
        slot = torch.empty(1, 3100, dtype=torch.int32, device=dev)
        hb = torch.tensor([base], dtype=torch.int32, device=dev)
        cache.counters[0] += 1                               # a new step for the priorities
        E.cache_recall(cache, lst, hb, miss, nmiss, slot)
        torch.cuda.synchronize()
        assert cache.status() == 0
        oc.step += 1
        rec = oc.recall([toks], [base], [np.zeros(0, dtype=np.int64)])
        assert rec.status == 0
        assert set(miss[0, :int(nmiss.item())].cpu().tolist()) == set(rec.misses[0])
        assert gpu_residency(cache) == oc.resident_priority()
        check_gpu_maps(cache)
        s_np = slot[0].cpu().numpy()
        n = int(count.item())
        kv = cache.gpu_kv.float().cpu().numpy()
        assert np.array_equal(kv[s_np[:n]], lat[base + toks])


@pytest.mark.slow
def test_prefill_full_block_512_at_100k_sampled():
    wl = S.workloads()["prefill-chunk2048-ctx100k"]
    pos0, Q, k = 100_000, 512, 2048
    k_int, q_int, w = block_inputs(wl, pos0, Q)
    kth_pred = np.full(Q, 40.0, dtype=np.float32)
    scores, hist, bitmap, thr, cnt = run_block(k_int, q_int, w, pos0, kth_pred, k)
    keys_f = S.grid_to_float(k_int).numpy().astype(np.float64)
    qf = S.grid_to_float(q_int).numpy().astype(np.float64)
    wf = w.numpy().astype(np.float64)
    hi = hist.cpu().numpy().astype(np.int64)
    assert np.array_equal(hi.sum(1), pos0 + 1 + np.arange(Q)), "every causal token counted once"
    rng = np.random.default_rng(9)
    for j in rng.choice(Q, 3, replace=False):
        L = pos0 + j + 1
        row = scores[j, :L].cpu().numpy()
        ts = rng.choice(L, 64, replace=False)
        ref = O.to_f32_exact(O.indexer_scores(qf[j], wf[j], keys_f[ts]))
        assert np.array_equal(row[ts], ref), f"sampled scores, query {j}"
        # the bucket rule recomputed by the oracle on the GPU's own row
        assert np.array_equal(hi[j], O.prefill_histogram(row, kth_pred[j]))
        t_j, c_j = O.prefill_candidates(row, kth_pred[j], k)
        assert int(thr[j].item()) == t_j and int(cnt[j].item()) == len(c_j)
    # one query scored in full by the oracle: exact candidates and top-k
    j = int(rng.integers(Q))
    L = pos0 + j + 1
    full = O.to_f32_exact(O.indexer_scores(qf[j], wf[j], keys_f[:L]))
    assert np.array_equal(scores[j, :L].cpu().numpy(), full)
    seq = torch.arange(pos0 + 1, pos0 + Q + 1, dtype=torch.int32, device=dev)
    sel = torch.empty(Q, k, dtype=torch.int32, device=dev)
    kth = torch.empty(Q, device=dev)
    E.topk(scores.nan_to_num(nan=-1.0), seq, k, sel, kth, torch.tensor(kth_pred, device=dev))
    torch.cuda.synchronize()
    osel, okth = O.topk_select(full, k)
    assert set(sel[j].cpu().tolist()) == set(osel.tolist()) and float(kth[j]) == np.float32(okth)
