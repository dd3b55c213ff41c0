"""Pins of the CPU oracle against things other than itself: hand-worked examples
from the pages' definitions (tests/golden), closed forms, brute force on tiny
inputs, invariants and special cases.  No GPU needed."""

import json
import math
import os
import random

import numpy as np
import pytest

import oracle as O


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ------------------------------------------------------------- indexer ----
def test_indexer_hand_example(golden_dir):
    g = load(golden_dir, "indexer_8tok.json")
    s = O.indexer_scores(np.array(g["q"]), np.array(g["w"]), np.array(g["keys"]))
    assert s.tolist() == g["scores"]


def test_indexer_bruteforce_loops():
    rng = np.random.default_rng(1)
    for _ in range(20):
        H, D, L = rng.integers(1, 6), rng.integers(1, 9), rng.integers(0, 12)
        q = rng.integers(-4, 5, (H, D)) / 8.0
        k = rng.integers(-4, 5, (L, D)) / 8.0
        w = rng.choice([0.25, 0.5, 1.0], H)
        ref = []
        for t in range(L):
            tot = 0.0
            for h in range(H):
                d = math.fsum(q[h, i] * k[t, i] for i in range(D))
                tot += w[h] * max(0.0, d)
            ref.append(tot)
        assert np.array_equal(O.indexer_scores(q, w, k), np.array(ref, dtype=np.float64).reshape(-1))


def test_indexer_negative_heads_do_not_count():
    # a head whose dot product is negative contributes nothing (ReLU), however large w is
    q = np.array([[1.0, 0.0], [-1.0, 0.0]])
    k = np.array([[2.0, 5.0]])
    assert O.indexer_scores(q, np.array([1.0, 100.0]), k).tolist() == [2.0]


def test_indexer_fp8_grid_is_exact_in_f32():
    # full-size heads on the FP8 grid: float64 scores are exact in float32, and a
    # float32 accumulation in a scrambled order gives the identical value
    rng = np.random.default_rng(7)
    q = rng.integers(-8, 9, (64, 128)) / 8.0
    k = rng.integers(-8, 9, (300, 128)) / 8.0
    w = rng.integers(1, 17, 64) / 16.0
    k[0] = 1.0
    q[:] = np.where(rng.random(q.shape) < 0.02, 1.0, q)
    s = O.indexer_scores(q, w, k)
    s32 = O.to_f32_exact(s)                       # raises if not exact
    perm_h = rng.permutation(64)
    perm_d = rng.permutation(128)
    for t in range(0, 300, 37):
        acc = np.float32(0)
        for h in perm_h:
            d = np.float32(0)
            for i in perm_d:
                d = np.float32(d + np.float32(q[h, i] * k[t, i]))
            acc = np.float32(acc + np.float32(np.float32(w[h]) * max(np.float32(0), d)))
        assert acc == s32[t]
    # worst case of the bound: every product +1, every weight 1 -> 64 * 128 = 2^13
    big = O.indexer_scores(np.ones((64, 128)), np.ones(64), np.ones((1, 128)))
    assert big[0] == 8192.0 and O.to_f32_exact(big)[0] == np.float32(8192.0)


def test_to_f32_exact_rejects_inexact():
    with pytest.raises(ValueError):
        O.to_f32_exact(np.array([1.0 + 2.0 ** -30]))


# ---------------------------------------------------------------- top-k ----
def test_topk_hand_example(golden_dir):
    g = load(golden_dir, "indexer_8tok.json")
    s = np.array(g["scores"], dtype=np.float32)
    sel, kth = O.topk_select(s, 3)
    assert sorted(sel.tolist()) == g["top3"] and kth == g["top3_kth"]
    sel, kth = O.topk_select(s, 4)
    assert sorted(sel.tolist()) == g["top4"] and kth == g["top4_kth"]


def brute_topk(s, k):
    order = sorted(range(len(s)), key=lambda t: (-float(s[t]), t))
    return order[:k]


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(3)
    for _ in range(200):
        L = int(rng.integers(0, 40))
        k = int(rng.integers(1, 45))
        s = rng.integers(0, 6, L).astype(np.float32) / 4
        sel, kth = O.topk_select(s, k)
        ref = brute_topk(s, k)
        assert sel.tolist() == ref
        if ref:
            assert kth == float(s[ref[-1]])
        else:
            assert kth == -math.inf


def test_topk_all_equal_takes_lowest_indices():
    s = np.full(1000, 3.5, dtype=np.float32)
    sel, kth = O.topk_select(s, 256)
    assert sorted(sel.tolist()) == list(range(256)) and kth == 3.5


def test_topk_short_context_takes_all():
    s = np.array([5.0, 1.0, 3.0], dtype=np.float32)
    sel, kth = O.topk_select(s, 8)
    assert sorted(sel.tolist()) == [0, 1, 2] and kth == 1.0


def test_topk_selection_invariants():
    rng = np.random.default_rng(5)
    s = rng.integers(0, 50, 5000).astype(np.float32)
    k = 700
    sel, kth = O.topk_select(s, k)
    mask = np.zeros(s.size, bool)
    mask[sel] = True
    assert np.all(s[~mask] <= kth) and np.all(s[mask] >= kth)
    eq_sel = np.nonzero(mask & (s == kth))[0]
    eq_uns = np.nonzero(~mask & (s == kth))[0]
    assert eq_uns.size == 0 or eq_uns.min() > eq_sel.max()


# ------------------------------------------------------------------ EMA ----
def test_ema_examples(golden_dir):
    g = load(golden_dir, "indexer_8tok.json")["ema"]
    assert O.ema_update(g["theta"], g["kth"], g["alpha"]) == np.float32(g["out"])
    assert O.ema_update(math.inf, 0.75) == np.float32(0.75)          # first observation
    th = np.float32(math.inf)
    for _ in range(5):
        th = O.ema_update(th, 4.25)                                   # constant kth: fixed point
    assert th == np.float32(4.25)
    assert O.ema_update(2.0, -math.inf) == np.float32(2.0)            # empty selection: unchanged


def test_ema_direction_textbook_cases():
    # textbook EMA S <- alpha*x + (1-alpha)*S: alpha = 1 keeps only the new
    # observation, alpha = 0 keeps the old estimate
    assert O.ema_update(3.0, 7.5, alpha=1.0) == np.float32(7.5)
    assert O.ema_update(3.0, 7.5, alpha=0.0) == np.float32(3.0)
    assert O.ema_update(3.0, 7.0, alpha=0.75) == np.float32(6.0)


def test_ema_rounds_in_float32():
    # 0.5*1 + 0.5*2^-24 = 0.5 + 2^-25 is a tie between 0.5 and its float32
    # successor; the update returns a float32 rounded to nearest even (0.5), not
    # the float64 value 0.50000003
    assert O.ema_update(1.0, 2.0 ** -24) == np.float32(0.5)
    assert float(O.ema_update(1.0, 2.0 ** -24)) != 0.5 + 2.0 ** -25


# ------------------------------------------------------------- prefetch ----
def test_prefetch_hand_example(golden_dir):
    g = load(golden_dir, "indexer_8tok.json")
    s = np.array(g["scores"], dtype=np.float32)
    p = g["prefetch"]
    res = np.zeros(8, bool)
    res[p["resident"]] = True
    assert O.prefetch_marks(s, p["theta"], res, 2).tolist() == p["cap2"]
    assert O.prefetch_marks(s, p["theta"], res, 3).tolist() == p["cap3"]
    assert O.prefetch_marks(s, p["theta"], res, 8).tolist() == p["cap8"]
    assert O.prefetch_marks(s, math.inf, res, 8).tolist() == []
    # strict '>': a threshold equal to a score does not mark it
    assert O.prefetch_marks(s, 0.75, res, 8).tolist() == []
    sel, _ = O.topk_select(s, 3)
    staged = set(p["cap3"])
    miss_pf = sorted(t for t in sel if not res[t] and t not in staged)
    miss_nopf = sorted(t for t in sel if not res[t])
    assert miss_pf == p["top3_misses_with_prefetch"] and miss_nopf == p["top3_misses_without_prefetch"]


def test_prefetch_cap_rule():
    assert O.prefetch_cap(65536, 4096, 32) == 2048
    assert O.prefetch_cap(100_000, 4096, 32) == 3125
    assert O.prefetch_cap(100_001, 4096, 32) == 3126
    assert O.prefetch_cap(1, 4096, 32) == 1
    assert O.prefetch_cap(4096, 512, 0) == 512
    assert O.prefetch_cap(4096, 0, 32) == 0


def test_prefetch_under_cap_is_order_free():
    # when no more than cap tokens qualify, the lowest-index rule and any other
    # order give the same set
    rng = np.random.default_rng(11)
    s = rng.integers(0, 100, 3000).astype(np.float32)
    res = rng.random(3000) < 0.5
    q = np.nonzero((s > 90) & ~res)[0]
    assert set(O.prefetch_marks(s, 90.0, res, q.size + 5).tolist()) == set(q.tolist())
    assert O.prefetch_marks(s, 90.0, res, 7).tolist() == q[:7].tolist()


# --------------------------------------------------------- cache / LRU ----
def test_metadata_closed_form():
    assert O.metadata_bytes(2_000_000, 200_000) == 10_600_000      # "about 10 MB per layer"
    assert O.metadata_bytes(8192, 1024) == 46_080
    # 61 layers -> about 610 MB per model (617 MiB)
    assert abs(61 * O.metadata_bytes(2_000_000, 200_000) / 2 ** 20 - 616.7) < 0.1


def test_lru_golden_sequence(golden_dir):
    g = load(golden_dir, "lru_ng4.json")
    c = O.LayerCache(g["n_gpu"], g["n_host"])
    seq = np.array([g["seq_len0"]], dtype=np.int64)
    for st in g["steps"]:
        new = c.writeback(g["host_base"], seq)
        assert new.tolist() == [st["new"]]
        assert c.resident_priority() == {int(k): v for k, v in st["after_wb"].items()}
        c.check_invariants()
        r = c.recall([np.array(st["sel"])], g["host_base"], [np.array(st["staged"], dtype=np.int64)])
        assert r.hits[0] == st["hits"]
        assert r.staged_hits[0] == st["staged_hits"]
        assert r.misses[0] == st["misses"]
        assert r.evicted.tolist() == st["evicted"]
        assert r.status == st["status"]
        assert r.slot_host[0] == st["slot_host"]
        assert c.resident_priority() == {int(k): v for k, v in st["resident"].items()}
        c.check_invariants()


def brute_victims(c, m):
    cands = [(int(c.priority[g]), int(c.gpu2host[g]), g) for g in range(c.n_gpu)
             if c.gpu2host[g] >= 0 and c.priority[g] < c.step]
    cands.sort()
    return sorted(x[2] for x in cands[:m])


def test_cache_random_sequences_against_bruteforce():
    rng = random.Random(2)
    for trial in range(30):
        ng = rng.randint(1, 12)
        nh = 64
        c = O.LayerCache(ng, nh)
        B = rng.randint(1, 3)
        base = [0, 20, 40][:B]
        seq = np.array([rng.randint(1, 10) for _ in range(B)], dtype=np.int64)
        for step in range(8):
            before = c.resident_priority()
            c.writeback(base, seq)
            c.check_invariants()
            sel = [np.array(rng.sample(range(int(seq[b])), min(int(seq[b]), rng.randint(0, 6))))
                   for b in range(B)]
            staged = []
            for b in range(B):
                cand = [t for t in range(int(seq[b])) if c.host2gpu[base[b] + t] < 0]
                staged.append(np.array(sorted(rng.sample(cand, min(len(cand), rng.randint(0, 2)))),
                                       dtype=np.int64))
            # expected victims computed independently before the recall mutates
            protect = {base[b] + int(t) for b in range(B) for t in sel[b]}
            need = sum(len(s) for s in staged) + sum(
                1 for b in range(B) for t in sel[b]
                if c.host2gpu[base[b] + int(t)] < 0 and int(t) not in set(staged[b].tolist()))
            r = c.recall(sel, base, staged)
            c.check_invariants()
            # no selected token is ever evicted by the recall
            assert not (set(r.evicted.tolist()) & protect)
            # every selected token is resident afterwards unless the pool ran out
            if r.status == O.ST_OK:
                for b in range(B):
                    for t in sel[b]:
                        assert c.host2gpu[base[b] + int(t)] >= 0
            assert len(r.evicted) <= max(0, need)
            del before


def test_lru_victims_match_bruteforce():
    rng = np.random.default_rng(4)
    for _ in range(50):
        c = O.LayerCache(20, 200)
        c.step = 10
        used = rng.choice(20, rng.integers(0, 21), replace=False)
        hosts = rng.choice(200, used.size, replace=False)
        for g, h in zip(used, hosts):
            c.free[g] = False
            c.gpu2host[g] = h
            c.host2gpu[h] = g
            c.priority[g] = rng.integers(0, 12)
        m = int(rng.integers(0, 22))
        assert sorted(c.lru_victims(m).tolist()) == brute_victims(c, m)


# ------------------------------------------------------------ attention ----
def test_mla_two_token_closed_form(golden_dir):
    g = load(golden_dir, "mla_closed_form.json")["two_token"]
    rng = np.random.default_rng(0)
    c = rng.standard_normal((2, 576))
    c[:, 0] = [0.0, 1.0]
    q = np.zeros((3, 576))
    q[:, 0] = math.log(3.0)
    out, lse = O.sparse_mla_decode(q, c, 1.0)
    exp = g["p"][0] * c[0, :512] + g["p"][1] * c[1, :512]
    assert np.allclose(out, exp[None, :], rtol=0, atol=1e-14)
    assert np.allclose(lse, g["lse"], rtol=0, atol=1e-14)


def test_mla_single_token_is_exact_copy():
    rng = np.random.default_rng(1)
    c = rng.standard_normal((1, 576))
    q = rng.standard_normal((4, 576))
    out, lse = O.sparse_mla_decode(q, c, 0.05)
    assert np.array_equal(out, np.repeat(c[:, :512], 4, axis=0))
    assert np.allclose(lse, 0.05 * (q @ c[0]), rtol=0, atol=1e-12)


def test_mla_equal_logits_is_mean(golden_dir):
    n = load(golden_dir, "mla_closed_form.json")["equal_logits"]["n"]
    rng = np.random.default_rng(2)
    c = rng.standard_normal((n, 576))
    out, lse = O.sparse_mla_decode(np.zeros((2, 576)), c, 1.0)
    assert np.allclose(out, c[:, :512].mean(0)[None], rtol=0, atol=1e-14)
    assert np.allclose(lse, math.log(n), rtol=0, atol=1e-14)


def test_mla_matches_dense_masked_and_bruteforce():
    rng = np.random.default_rng(3)
    N, n = 40, 9
    cache = rng.standard_normal((N, 576))
    idx = rng.choice(N, n, replace=False)
    q = rng.standard_normal((3, 576))
    out, lse = O.sparse_mla_decode(q, cache[idx], 0.04)
    mask = np.zeros(N, bool)
    mask[idx] = True
    dense = O.dense_masked_attention(q, cache, mask, 0.04)
    assert np.allclose(out, dense, rtol=0, atol=1e-12)
    # brute force with exactly summed logits and normaliser
    for h in range(3):
        lg = [0.04 * math.fsum(q[h, d] * cache[j, d] for d in range(576)) for j in idx]
        mx = max(lg)
        z = math.fsum(math.exp(x - mx) for x in lg)
        assert abs(lse[h] - (mx + math.log(z))) < 1e-12
        for d in (0, 17, 511):
            o = math.fsum(math.exp(x - mx) / z * cache[j, d] for x, j in zip(lg, idx))
            assert abs(out[h, d] - o) < 1e-12
    # permuting the selection does not change the result
    perm = rng.permutation(n)
    out2, lse2 = O.sparse_mla_decode(q, cache[idx[perm]], 0.04)
    assert np.allclose(out2, out, rtol=0, atol=1e-12) and np.allclose(lse2, lse, rtol=0, atol=1e-12)


# ------------------------------------------------------- one decode step ----
def test_decode_step_small_properties():
    from sparse_attention_kv_dsa_gb300 import synth as S
    wl = S.small_workload(ctx=(300, 520, 129), topk=64, n_gpu=400, cap_max=40, steps=3)
    B = wl.batch
    keys = [S.grid_to_float(S.keys_for(wl, 0, b, wl.max_ctx)).numpy() for b in range(B)]
    lat = S.latents_for(wl, 0, wl.n_host).float().numpy()
    c = O.LayerCache(wl.n_gpu, wl.n_host)
    seq = np.array(wl.ctx, dtype=np.int64)
    theta = np.full(B, np.inf, dtype=np.float32)
    qi = S.qidx_initial(wl, 0)
    w = S.weights_for(wl, 0).numpy()
    for s in range(wl.steps):
        q = S.grid_to_float(qi).numpy()
        qm = S.qmla_for(wl, 0, s).float().numpy()
        r = O.decode_layer_step(c, host_base=wl.host_base, seq_len=seq, keys_of=lambda b, L: keys[b][:L],
                                q_idx=q, w_idx=w, theta=theta, k=wl.topk, cap_max=wl.cap_max,
                                cap_div=wl.cap_div, q_mla=qm, latent_of=lambda h: lat[h], scale=wl.scale)
        c.check_invariants()
        for b in range(B):
            assert r.scores[b].shape[0] == seq[b]
            assert len(r.sel[b]) == min(wl.topk, int(seq[b]))
            if s == 0:
                assert r.staged[b].size == 0            # theta = +inf: nothing prefetched
            else:
                assert np.all(r.scores[b][r.staged[b]] > theta[b])
                assert r.staged[b].size <= r.cap[b]
            for t in r.sel[b]:                           # every selected token resident
                assert c.host2gpu[wl.host_base[b] + int(t)] >= 0
            # attention over the resident copy equals attention over the host rows
            hosts = wl.host_base[b] + np.asarray(r.sel[b])
            o, _ = O.sparse_mla_decode(qm[b], lat[hosts], wl.scale)
            assert np.array_equal(o, r.out[b])
        theta = r.theta
        qi = S.qidx_next(wl, 0, s, qi)


# ------------------------------------------------------------------ prefill --
def test_order_key_sorts_like_the_floats():
    # order-preserving key: sorting by key sorts the values; -0 and +0 share a key
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(500) * 10.0 ** rng.integers(-30, 30, 500),
                        [0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45]]).astype(np.float32)
    key = O.order_key_f32(x)
    xs = np.sort(x.astype(np.float64))
    ks = np.sort(key)
    assert np.array_equal(O.order_key_f32(xs.astype(np.float32)), ks)
    for i in range(len(x)):                              # pairwise order on a sample
        for j in range(0, len(x), 37):
            assert (x[i] < x[j]) == (key[i] < key[j]) or x[i] == x[j]
    assert O.order_key_f32(np.float32(-0.0)) == O.order_key_f32(np.float32(0.0)) == 0x80000000


def test_prefill_bucket_hand_values():
    # bucket = top byte of the key of d = score - kth_pred (IEEE-754 worked by hand):
    #   d = 1.0  -> bits 0x3F800000 -> key 0xBF800000 -> 191;  d = 0.5 -> 0xBF000000 -> 191
    #   d = 2.0  -> 0x40000000 -> key 0xC0000000 -> 192;       d = 0 -> 0x80000000 -> 128
    #   d = -1.0 -> bits 0xBF800000 -> key ~bits = 0x407FFFFF -> 64
    #   d = 1e-38 (subnormal-adjacent) -> key 0x806CE3EE -> 128
    kth = 10.0
    scores = np.array([11.0, 10.5, 12.0, 10.0, 9.0, 10.0 + 1e-6], dtype=np.float32)
    got = O.prefill_buckets(scores, kth)
    d = scores - np.float32(kth)
    assert got.tolist()[:5] == [191, 191, 192, 128, 64]
    # 1e-6 above 10 is not representable exactly: the float32 difference decides
    assert got[5] == (O.order_key_f32(d[5:6])[0] >> 24)
    assert O.prefill_buckets(np.array([1e-38], np.float32), 0.0)[0] == 128


def test_prefill_candidates_brute_force():
    # threshold bucket holds the k-th largest d; candidates are exactly the tokens in
    # strictly higher buckets; they all rank above the k-th, so they are in the top-k
    rng = np.random.default_rng(11)
    for trial in range(60):
        L = int(rng.integers(1, 90))
        k = int(rng.integers(1, 40))
        s = (rng.integers(-40, 41, L) * 0.125).astype(np.float32)
        kth_pred = float(rng.integers(-20, 21) * 0.25)
        thr, cand = O.prefill_candidates(s, kth_pred, k)
        d = s - np.float32(kth_pred)
        bk = [(int(O.order_key_f32(d[t:t + 1])[0]) >> 24) for t in range(L)]   # per element
        if L <= k:
            assert thr == -1 and cand.tolist() == list(range(L))
            continue
        kth_d = sorted(d.tolist(), reverse=True)[k - 1]
        assert thr == int(O.order_key_f32(np.float32(kth_d))) >> 24
        assert cand.tolist() == [t for t in range(L) if bk[t] > thr]
        top, _ = O.topk_select(s, k)
        assert set(cand.tolist()) <= set(top.tolist())
        assert len(cand) <= k - 1


def test_prefill_scores_causal_brute_force():
    # explicit loops over heads and dims for one token of each query
    rng = np.random.default_rng(3)
    Q, H, D, pos0 = 3, 4, 8, 5
    q = rng.integers(-8, 9, (Q, H, D)) * 0.125
    w = rng.integers(1, 17, (Q, H)) / 16.0
    keys = rng.integers(-8, 9, (pos0 + Q, D)) * 0.125
    sc = O.prefill_scores(q, w, keys, pos0)
    assert [len(x) for x in sc] == [pos0 + 1, pos0 + 2, pos0 + 3]
    for j in range(Q):
        for t in (0, pos0 + j):
            tot = 0.0
            for h in range(H):
                dot = 0.0
                for c in range(D):
                    dot += q[j, h, c] * keys[t, c]
                tot += w[j, h] * max(dot, 0.0)
            assert sc[j][t] == tot


def test_token_union_and_block_properties():
    assert O.token_union([[5, 1, 3], [3, 9], []]).tolist() == [1, 3, 5, 9]
    rng = np.random.default_rng(5)
    Q, H, D, pos0, k = 4, 4, 8, 40, 6
    q = rng.integers(-8, 9, (Q, H, D)) * 0.125
    w = rng.integers(1, 17, (Q, H)) / 16.0
    keys = rng.integers(-8, 9, (pos0 + Q, D)) * 0.125
    kth_pred = np.full(Q, 1.5, dtype=np.float32)
    r = O.prefill_block(q, w, keys, pos0, kth_pred, k)
    assert set(r["cand_union"].tolist()) <= set(r["sel_union"].tolist())
    for j in range(Q):
        assert r["hist"][j].sum() == pos0 + j + 1
        assert r["kth"][j] == np.float32(np.sort(r["scores"][j])[::-1][k - 1])


def test_writeback_victims_continue_the_recall_lru_order():
    # After the recall of step s has protected the selection and evicted its m victims
    # (the m smallest (priority, host) among slots untouched in step s), the write-back
    # of step s+1 evicts the next B of that same order, as long as enough of them are
    # left: the GPU manager ranks them during the recall and binds them at the write-back.
    rng = np.random.default_rng(21)
    checked = 0
    for trial in range(25):
        B = int(rng.integers(1, 7))
        span, n_gpu = 600, 300
        oc = O.LayerCache(n_gpu, span * B)
        host_base = np.arange(B, dtype=np.int64) * span
        s = 12
        hosts = rng.choice(np.concatenate([host_base[b] + np.arange(550) for b in range(B)]), n_gpu, replace=False)
        for g, h in enumerate(hosts):
            oc.free[g] = False
            oc.gpu2host[g] = h
            oc.host2gpu[h] = g
            oc.priority[g] = int(rng.integers(0, s))
        oc.step = s
        sel = [rng.choice(550, int(rng.integers(5, 200 // B + 6)), replace=False) for _ in range(B)]
        # the order the recall evicts in: protection first, then (priority, host)
        prio = oc.priority.copy()
        for b in range(B):
            for t in sel[b]:
                g = oc.host2gpu[host_base[b] + t]
                if g >= 0:
                    prio[g] = s
        used = np.nonzero(oc.gpu2host >= 0)[0]
        elig = used[prio[used] < s]
        order = oc.gpu2host[elig[np.lexsort((oc.gpu2host[elig], prio[elig]))]]
        rec = oc.recall(sel, host_base, [np.zeros(0, dtype=np.int64)] * B)
        assert rec.status == 0
        m = rec.evicted.size
        assert set(rec.evicted.tolist()) == set(order[:m].tolist())
        if m == 0 or order.size < m + B or oc.n_free() != 0:
            continue
        before = set(oc.resident_hosts().tolist())
        seq = np.full(B, 580, dtype=np.int64)                 # new tokens, not resident
        oc.writeback(host_base, seq)
        gone = before - set(oc.resident_hosts().tolist())
        assert gone == set(order[m:m + B].tolist()), f"trial {trial}"
        checked += 1
    assert checked >= 10, "too few trials reached the write-back"


# ------------------------------------------------------- adaptive cap (R23) --
def test_prediction_error_hand_values():
    # |theta - kth| / |kth| in float32: 0.25 / 0.75 rounds to the float nearest 1/3
    assert O.prediction_error(1.0, 0.75) == np.float32(1.0 / 3.0)
    assert O.prediction_error(0.5, 1.0) == np.float32(0.5)
    assert O.prediction_error(-2.0, -4.0) == np.float32(0.5)      # relative to |kth|, not to theta
    assert O.prediction_error(np.inf, 3.0) == 0.0                  # before the first observation
    assert O.prediction_error(3.0, 0.0) == 0.0 and O.prediction_error(3.0, -np.inf) == 0.0


def test_adaptive_cap_hand_values():
    # R7 at 64K with cap_div 32 is 2048
    assert O.adaptive_cap(65536, 4096, 32, -1, 0.0, 256) == 2048     # no observation: R7
    assert O.adaptive_cap(65536, 4096, 32, 100, 0.5, 256) == 150 + 256
    assert O.adaptive_cap(65536, 4096, 32, 100, 0.0, 256) == 356
    assert O.adaptive_cap(65536, 4096, 32, 101, 0.5, 0) == 152      # ceil(151.5)
    assert O.adaptive_cap(65536, 4096, 32, 5000, 0.0, 256) == 2048   # never above R7
    assert O.adaptive_cap(65536, 0, 32, 100, 0.0, 256) == 0          # prefetch off
    assert O.adaptive_cap(1000, 512, 0, 10, 0.0, 3) == 13            # constant cap rule below


def test_adaptive_cap_properties():
    rng = np.random.default_rng(31)
    for _ in range(300):
        L, cm, cd = int(rng.integers(1, 200000)), int(rng.integers(0, 20000)), int(rng.choice([0, 16, 32]))
        u, e, sl = int(rng.integers(0, 5000)), np.float32(rng.random() * 2), int(rng.integers(0, 500))
        c = O.adaptive_cap(L, cm, cd, u, e, sl)
        base = O.prefetch_cap(L, cm, cd)
        assert 0 <= c <= base
        # exact predictor (e = 0) and no slack: the cap is last step's transfer
        assert O.adaptive_cap(L, cm, cd, u, 0.0, 0) == min(base, u)
        # a worse prediction or a larger transfer never lowers the cap
        assert O.adaptive_cap(L, cm, cd, u, e + np.float32(0.25), sl) >= c
        assert O.adaptive_cap(L, cm, cd, u + 7, e, sl) >= c


def test_adaptive_state_follows_the_steps():
    # the state after a step is its transfer (prefetched hits + misses) and its error
    from sparse_attention_kv_dsa_gb300 import synth as S
    wl = S.small_workload(ctx=(300, 520), topk=64, n_gpu=400, cap_max=40, cap_div=8, steps=3)
    B = wl.batch
    keys = [S.grid_to_float(S.keys_for(wl, 0, b, wl.max_ctx)).numpy() for b in range(B)]
    c = O.LayerCache(wl.n_gpu, wl.n_host)
    ad = O.AdaptiveCap(B, 5)
    seq = np.array(wl.ctx, dtype=np.int64)
    theta = np.full(B, np.inf, dtype=np.float32)
    qi = S.qidx_initial(wl, 0)
    w = S.weights_for(wl, 0).numpy()
    for s in range(wl.steps):
        prev_new, prev_err = ad.new_rows.copy(), ad.pred_err.copy()
        r = O.decode_layer_step(c, host_base=wl.host_base, seq_len=seq, keys_of=lambda b, L: keys[b][:L],
                                q_idx=S.grid_to_float(qi).numpy(), w_idx=w, theta=theta, k=wl.topk,
                                cap_max=wl.cap_max, cap_div=wl.cap_div, adaptive=ad)
        for b in range(B):
            assert r.cap[b] == O.adaptive_cap(int(seq[b]), wl.cap_max, wl.cap_div, int(prev_new[b]), prev_err[b], 5)
            assert ad.new_rows[b] == len(r.recall.staged_hits[b]) + len(r.recall.misses[b])
            assert ad.pred_err[b] == O.prediction_error(theta[b], r.kth[b])
        if s == 0:
            assert r.cap == [O.prefetch_cap(int(L), wl.cap_max, wl.cap_div) for L in seq]
        theta = r.theta
        qi = S.qidx_next(wl, 0, s, qi)


# -------------------------------------------------- block granularity (R25) --
def test_block_scores_are_block_maxima():
    assert O.block_scores([1.0, 5.0, 2.0, 7.0, 3.0], 2).tolist() == [5.0, 7.0, 3.0]   # short last block
    rng = np.random.default_rng(41)
    for _ in range(50):
        L, T = int(rng.integers(1, 300)), int(rng.choice([1, 4, 16, 64]))
        s = rng.integers(-50, 50, L) * 0.25
        assert O.block_scores(s, T).tolist() == [max(s[j:j + T]) for j in range(0, L, T)]


def test_block_writeback_hand_sequence():
    # T = 4, two GPU slots (blocks), one request whose host rows start at 0, 3 tokens so far:
    #   s1: token 3, middle of block 0, not resident      -> no slot
    #   s2: token 4 starts block 1                         -> free slot, priority 2
    #       recall selects blocks {0, 1}: 1 protected (2), 0 missing -> the other slot (2)
    #   s3..s5: tokens 5, 6, 7 in resident block 1        -> its priority 3, 4, 5
    #   s6: token 8 starts block 2, no free slot           -> evict block 0 (priority 2), bind 2 (6)
    c = O.LayerCache(2, 8)
    seq = np.array([3], dtype=np.int64)
    assert c.writeback_blocks([0], seq, 4).tolist() == [0] and c.resident_priority() == {}
    assert c.writeback_blocks([0], seq, 4).tolist() == [1] and c.resident_priority() == {1: 2}
    r = c.recall([np.array([0, 1])], [0], [np.zeros(0, dtype=np.int64)])
    assert r.misses == [[0]] and r.hits == [[1]] and c.resident_priority() == {0: 2, 1: 2}
    for s in (3, 4, 5):
        c.writeback_blocks([0], seq, 4)
        assert c.resident_priority() == {0: 2, 1: s}
    assert c.writeback_blocks([0], seq, 4).tolist() == [2]
    assert c.resident_priority() == {1: 5, 2: 6} and seq.tolist() == [9]
    c.check_invariants()


def test_block_writeback_binds_before_touching():
    # T = 2, one GPU slot, two requests (host rows from 0 and from 100):
    #   s1: request 0's row 0 starts block 0 -> the free slot; request 1's row 101 is mid-block 50
    #   s2: request 1's row 102 starts block 51 and evicts block 0 (stamp 1 < 2), although
    #       request 0's row 1 lands in block 0 in the same step: binds come before touches
    c = O.LayerCache(1, 64)
    seq = np.array([0, 1], dtype=np.int64)
    assert c.writeback_blocks([0, 100], seq, 2).tolist() == [0, 50] and c.resident_priority() == {0: 1}
    assert c.writeback_blocks([0, 100], seq, 2).tolist() == [0, 51] and c.resident_priority() == {51: 2}
    assert c.status == 0 and seq.tolist() == [2, 3]
    c.check_invariants()


def test_block_metadata_closed_form():
    # the per-token formula over blocks: 2M host rows and 200K GPU rows in blocks of 64
    assert O.metadata_bytes(2_000_000 // 64, 200_000 // 64) == 4 * 31250 + 13 * 3125


def test_block_decode_step_properties():
    from sparse_attention_kv_dsa_gb300 import synth as S
    T, kb = 16, 6
    wl = S.small_workload(ctx=(300, 520, 129), topk=kb * T, n_gpu=40, cap_max=0, steps=4)
    B = wl.batch
    base = [(hb + T - 1) // T * T for hb in wl.host_base]            # block-aligned host rows
    n_host_blk = (base[-1] + wl.ctx[-1] + wl.steps + 8 + T) // T + 1
    keys = [S.grid_to_float(S.keys_for(wl, 0, b, wl.max_ctx)).numpy() for b in range(B)]
    lat = S.latents_for(wl, 0, n_host_blk * T).float().numpy()
    c = O.LayerCache(wl.n_gpu, n_host_blk)
    seq = np.array(wl.ctx, dtype=np.int64)
    theta = np.full(B, np.inf, dtype=np.float32)
    qi = S.qidx_initial(wl, 0)
    w = S.weights_for(wl, 0).numpy()
    for s in range(wl.steps):
        q = S.grid_to_float(qi).numpy()
        qm = S.qmla_for(wl, 0, s).float().numpy()
        r = O.decode_layer_step_blocks(c, host_base=base, seq_len=seq, T=T, keys_of=lambda b, L: keys[b][:L],
                                       q_idx=q, w_idx=w, theta=theta, kb=kb, q_mla=qm,
                                       latent_of=lambda h: lat[h], scale=wl.scale)
        c.check_invariants()
        for b in range(B):
            L = int(seq[b])
            bs = np.array([r.scores[b][j:j + T].max() for j in range(0, L, T)], dtype=np.float64)
            assert np.array_equal(r.bscores[b], bs)
            order = sorted(range(bs.shape[0]), key=lambda j: (-bs[j], j))[:kb]
            assert r.sel[b].tolist() == order
            assert r.kth[b] == np.float32(bs[order[-1]])
            for j in r.sel[b]:                                 # every selected block resident
                assert c.host2gpu[base[b] // T + int(j)] >= 0
            toks = [j * T + i for j in order for i in range(T) if j * T + i < L]
            o, _ = O.sparse_mla_decode(qm[b], lat[base[b] + np.array(toks)], wl.scale)
            assert np.array_equal(o, r.out[b])
            assert r.theta[b] == O.ema_update(theta[b], r.kth[b], 0.5)
        theta = r.theta
        qi = S.qidx_next(wl, 0, s, qi)


# ------------------------------------------------ several KV heads (R26) --
def test_gqa_single_token_is_its_value():
    rng = np.random.default_rng(61)
    q, row = rng.standard_normal((4, 16)), rng.standard_normal((1, 32))
    out, lse = O.sparse_gqa_decode(q, row, 0.25)
    assert np.array_equal(out, np.repeat(row[:, 16:], 4, axis=0))
    assert np.allclose(lse, 0.25 * (q @ row[0, :16]), rtol=0, atol=1e-14)


def test_gqa_zero_keys_average_the_values():
    rng = np.random.default_rng(62)
    rows = rng.standard_normal((5, 16))
    rows[:, :8] = 0.0
    out, lse = O.sparse_gqa_decode(rng.standard_normal((3, 8)), rows, 0.5)
    assert np.allclose(out, np.repeat(rows[:, 8:].mean(axis=0, keepdims=True), 3, axis=0), rtol=0, atol=1e-15)
    assert np.allclose(lse, np.log(5.0), rtol=0, atol=1e-15)


def test_gqa_two_token_closed_form():
    # keys e1 and 0, one head q = 3 e1, scale 0.5: logits 1.5 and 0, weights 1/(1+e^-1.5) and the rest
    rows = np.zeros((2, 8))
    rows[0, 0] = 1.0
    rows[0, 4:] = [1.0, 2.0, 3.0, 4.0]
    rows[1, 4:] = [-1.0, 0.0, 5.0, 2.0]
    q = np.array([[3.0, 0.0, 0.0, 0.0]])
    out, lse = O.sparse_gqa_decode(q, rows, 0.5)
    p = 1.0 / (1.0 + math.exp(-1.5))
    assert np.allclose(out[0], p * rows[0, 4:] + (1 - p) * rows[1, 4:], rtol=0, atol=1e-15)
    assert abs(lse[0] - (1.5 + math.log(1.0 + math.exp(-1.5)))) < 1e-15


def test_gqa_is_mla_with_the_key_in_the_rope_dims():
    # an MLA row [value | zeros | key | zeros] with the query on the key's dims gives the
    # same logits and the same weighted values (d = 64 fits into dims 512..575)
    rng = np.random.default_rng(63)
    d, n, G = 64, 37, 6
    rows = rng.standard_normal((n, 2 * d))
    q = rng.standard_normal((G, d))
    lat = np.zeros((n, 576))
    lat[:, :d] = rows[:, d:]
    lat[:, 512:512 + d] = rows[:, :d]
    q576 = np.zeros((G, 576))
    q576[:, 512:512 + d] = q
    o1, l1 = O.sparse_gqa_decode(q, rows, 0.125)
    o2, l2 = O.sparse_mla_decode(q576, lat, 0.125)
    assert np.allclose(o1, o2[:, :d], rtol=0, atol=1e-13) and np.allclose(l1, l2, rtol=0, atol=1e-13)
