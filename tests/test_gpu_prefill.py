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


# ------------------------------------------------- chunk pipeline (PrefillChunk) --
def _small_chunk_workload():
    """A 256-token chunk at positions 3000.. (several blocks of 64 or 128 queries),
    top-256, a GPU pool larger than the whole context (the chunk never evicts)."""
    w16 = [i / 16.0 for i in range(1, 17)]
    return S.Workload(name="prefill-chunk256-ctx3000", cfg_id=105, layers=1, batch=1, ctx=[3000], h_idx=64,
                      d_idx=128, grid=8, w_values=w16, topk=256, h_q=128, kv_fp32=False, n_gpu=4096,
                      n_host=3300, steps=0, rho=0.9, cap_max=0, cap_div=32, prefill_chunk=256,
                      prefill_blocks=[64, 128])


_ORACLE_CHUNKS = {}


def oracle_chunk(wl, block, mode):
    """The chunk's blocks in order through the oracle: each block predicts with the
    previous block's exact k-th scores (+inf for the first), then (echo mode) its
    histogram candidates are recalled, then the union of its exact selections, each
    as one request of host base 0."""
    ctx, chunk, k = wl.ctx[0], wl.prefill_chunk, wl.topk
    L = ctx + chunk
    key = (wl.name, block)
    if key not in _ORACLE_CHUNKS:
        keys = S.grid_to_float(S.keys_for(wl, 0, 0, L)).numpy()
        q = S.grid_to_float(S.prefill_queries(wl, 0, L)[ctx:]).numpy().astype(np.float64)
        w = S.prefill_weights(wl, 0, L)[ctx:].numpy().astype(np.float64)
        kpred = np.full(block, np.inf, dtype=np.float32)
        blocks = []
        for i in range(chunk // block):
            pos0 = ctx + i * block
            r = O.prefill_block(q[i * block:(i + 1) * block], w[i * block:(i + 1) * block], keys, pos0, kpred, k)
            blocks.append(dict(r, kpred=kpred.copy()))
            kpred = r["kth"].copy()
        _ORACLE_CHUNKS[key] = blocks
    blocks = _ORACLE_CHUNKS[key]
    oc = O.LayerCache(wl.n_gpu, wl.n_host)
    recs = []
    for b in blocks:
        rc = oc.recall([b["cand_union"]], [0], [np.zeros(0, dtype=np.int64)]) if mode == "echo" else None
        rs = oc.recall([b["sel_union"]], [0], [np.zeros(0, dtype=np.int64)])
        recs.append((rc, rs))
    return blocks, recs, oc


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("mode", ["serial", "overlap", "echo"])
def test_prefill_chunk_pipeline_matches_oracle(block, mode):
    """runtime.PrefillChunk.run, the overlapped chunk pipeline, against the oracle:
    every block's predictions (the previous block's k-th scores), exact selections,
    k-th scores, candidates and threshold buckets (echo mode), union sizes and miss
    counts of its recalls, and the residency at the end of the chunk."""
    from harness import check_gpu_maps, gpu_residency
    from sparse_attention_kv_dsa_gb300.runtime import PrefillChunk
    wl = _small_chunk_workload()
    pc = PrefillChunk(wl, block, dev, gen_device="cpu", record=True)
    pc.reset()
    pc.run(mode)
    torch.cuda.synchronize()
    assert int(pc.status.item()) == 0 and pc.cache.status() == 0
    blocks, recs, oc = oracle_chunk(wl, block, mode)
    rec = {n: v.cpu().numpy() for n, v in pc.rec.items()}
    for i, (ob, (rc, rs)) in enumerate(zip(blocks, recs)):
        assert np.array_equal(rec["kpred"][i], ob["kpred"]), f"block {i}: predictions (previous block's k-th)"
        assert np.array_equal(rec["kth"][i], ob["kth"]), f"block {i}: k-th scores"
        for j in range(block):
            assert set(rec["sel"][i][j].tolist()) == set(ob["sel"][j].tolist()), f"block {i} query {j}: top-k"
        assert rec["n_union"][i] == len(ob["sel_union"]), f"block {i}: selection union"
        assert rec["n_miss"][i] == len(rs.misses[0]), f"block {i}: misses of the exact recall"
        if mode == "echo":
            assert np.array_equal(rec["thr"][i], ob["thr"]), f"block {i}: threshold buckets"
            assert rec["cand"][i].tolist() == [len(c) for c in ob["cand"]], f"block {i}: candidate counts"
            assert rec["n_miss_cand"][i] == len(rc.misses[0]), f"block {i}: misses of the candidate recall"
    assert gpu_residency(pc.cache) == oc.resident_priority(), "residency at the end of the chunk"
    check_gpu_maps(pc.cache)
    # every resident slot holds its host row
    g2h = pc.cache.gpu2host.cpu().numpy()
    used = np.nonzero(g2h >= 0)[0]
    kv = pc.cache.gpu_kv[torch.from_numpy(used).cuda()].float().cpu().numpy()
    assert np.array_equal(kv, pc.cache.host_kv[torch.from_numpy(g2h[used]).long()].float().numpy())


@pytest.mark.slow
def test_prefill_chunk_full_size_echo_sampled():
    """The full chunk (2048 queries at positions 100,000..) in echo mode, blocks of 512:
    the prediction chain across blocks, selections of every query (valid, distinct,
    causal), residency = union of every block's selections, and two sampled queries
    scored in full by the oracle (exact top-k, k-th, candidates)."""
    from harness import check_gpu_maps, gpu_residency
    from sparse_attention_kv_dsa_gb300.runtime import PrefillChunk
    wl = S.workloads()["prefill-chunk2048-ctx100k"]
    block, k, ctx = 512, wl.topk, wl.ctx[0]
    pc = PrefillChunk(wl, block, dev, gen_device="cpu", record=True)
    pc.reset()
    pc.run("echo")
    torch.cuda.synchronize()
    assert int(pc.status.item()) == 0 and pc.cache.status() == 0
    rec = {n: v.cpu().numpy() for n, v in pc.rec.items()}
    nb = pc.nblocks
    assert np.all(np.isinf(rec["kpred"][0]))
    for i in range(1, nb):
        assert np.array_equal(rec["kpred"][i], rec["kth"][i - 1]), f"block {i}: prediction chain"
    union = set()
    for i in range(nb):
        pos0 = ctx + i * block
        for j in range(block):
            s_ij = rec["sel"][i][j]
            assert len(set(s_ij.tolist())) == k and s_ij.min() >= 0 and s_ij.max() <= pos0 + j
            union.update(s_ij.tolist())
    assert gpu_residency(pc.cache) == {t: 0 for t in union}, "residency = union of the selections"
    check_gpu_maps(pc.cache)
    L = ctx + wl.prefill_chunk
    keys = S.grid_to_float(S.keys_for(wl, 0, 0, L)).numpy()
    q = S.grid_to_float(S.prefill_queries(wl, 0, L)[ctx:]).numpy().astype(np.float64)
    w = S.prefill_weights(wl, 0, L)[ctx:].numpy().astype(np.float64)
    rng = np.random.default_rng(12)
    for i, j in ((int(rng.integers(1, nb)), int(rng.integers(block))), (0, int(rng.integers(block)))):
        pos0 = ctx + i * block
        sc = O.to_f32_exact(O.indexer_scores(q[i * block + j], w[i * block + j], keys[:pos0 + j + 1]))
        osel, okth = O.topk_select(sc, k)
        assert set(rec["sel"][i][j].tolist()) == set(osel.tolist()), f"block {i} query {j}: top-k"
        assert rec["kth"][i][j] == np.float32(okth)
        thr, cand = O.prefill_candidates(sc, rec["kpred"][i][j], k)
        assert rec["thr"][i][j] == thr and rec["cand"][i][j] == len(cand), f"block {i} query {j}: candidates"


@pytest.mark.parametrize("mode", ["overlap", "echo"])
def test_prefill_block_attention_matches_oracle(mode):
    """Prefill sparse attention: once a block's union is resident, each query attends
    over its own exact selection.  Against the oracle's attention over the host rows
    of the oracle's selection (every head of one query per block, 8 heads of two
    more), and bitwise against the same kernel over a dense copy of the host pool
    with the same token lists (lossless)."""
    from sparse_attention_kv_dsa_gb300.runtime import PrefillChunk
    wl = _small_chunk_workload()
    block = 64
    pc = PrefillChunk(wl, block, dev, gen_device="cpu", record=True, attend=True)
    pc.reset()
    pc.run(mode)
    torch.cuda.synchronize()
    assert int(pc.status.item()) == 0 and pc.cache.status() == 0
    blocks, _, _ = oracle_chunk(wl, block, mode)
    L = wl.ctx[0] + wl.prefill_chunk
    lat = S.latents_for(wl, 0, L, 0).float().numpy()
    qm = S.prefill_qmla(wl, 0, wl.prefill_chunk).float().numpy()
    out = pc.out.float().cpu().numpy()
    lse = pc.lse.cpu().numpy()
    rng = np.random.default_rng(4)
    for i, ob in enumerate(blocks):
        for n, j in enumerate(rng.choice(block, 3, replace=False)):
            row = i * block + int(j)
            heads = np.arange(wl.h_q) if n == 0 else rng.choice(wl.h_q, 8, replace=False)
            o, l_ = O.sparse_mla_decode(qm[row, heads], lat[ob["sel"][j]], wl.scale)
            assert np.abs(out[row, heads] - o).max() <= 2e-2, f"block {i} query {j}: attention"
            assert np.abs(lse[row, heads] - l_).max() <= 2e-2, f"block {i} query {j}: lse"
    # lossless: the same kernel over a dense buffer holding the host rows, token lists
    # in the same order as the GPU's selections
    dense = pc.cache.host_kv.to(dev)
    sel = pc.rec["sel"]
    for i in range(pc.nblocks):
        o2 = torch.empty(block, wl.h_q, 512, dtype=torch.bfloat16, device=dev)
        l2 = torch.empty(block, wl.h_q, device=dev)
        E.sparse_mla_decode(pc.q_mla[i * block:(i + 1) * block], dense, sel[i].contiguous(), wl.scale, o2, l2,
                            pc.mla_ws)
        torch.cuda.synchronize()
        assert torch.equal(o2, pc.out[i * block:(i + 1) * block]), f"block {i}: lossless"
        assert torch.equal(l2, pc.lse[i * block:(i + 1) * block])


def test_translate_slots_flags_tokens_without_a_slot():
    wl = S.small_workload("translate", ctx=(300,), topk=16, n_gpu=64, steps=1)
    cache = E.LayerCache(wl.n_gpu, wl.n_host, torch.bfloat16, dev)
    cache.reset()
    tok = torch.tensor([[5, 7, -1, 9]], dtype=torch.int32, device=dev)
    lst = torch.tensor([[5, 7, -1]], dtype=torch.int32, device=dev)
    hb = torch.tensor([3], dtype=torch.int32, device=dev)
    miss = torch.empty(1, 3, dtype=torch.int32, device=dev)
    nmiss = torch.zeros(1, dtype=torch.int32, device=dev)
    slot = torch.empty(1, 3, dtype=torch.int32, device=dev)
    E.cache_recall(cache, lst, hb, miss, nmiss, slot)           # tokens 5 and 7 become resident
    out = torch.empty_like(tok)
    E.translate_slots(cache, tok, hb, out)
    torch.cuda.synchronize()
    h2g = cache.host2gpu.cpu().numpy()
    got = out.cpu().numpy()[0]
    assert got[0] == h2g[8] >= 0 and got[1] == h2g[10] >= 0 and got[2] == -1
    assert got[3] == -1 and cache.status() == E.ERR_NOT_RESIDENT
