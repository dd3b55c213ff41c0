"""The C++ oracle against the independent numpy restatement of the same definitions
(oracle.numpy_oracle), on seeded random inputs: every integer, index, residency and
float32 output equal element by element; attention (exp/log in two libraries) within
1e-12.  Plus property pins of the prefill bucket mapping.  No GPU needed."""

import numpy as np
import pytest

import oracle as O
from oracle import numpy_oracle as N
from sparse_attention_kv_dsa_gb300 import synth as S


def test_indexer_scores_agree():
    rng = np.random.default_rng(21)
    for _ in range(30):
        H, D, L = int(rng.integers(1, 9)), int(rng.integers(1, 33)), int(rng.integers(0, 300))
        q = rng.integers(-8, 9, (H, D)) / 8.0
        k = rng.integers(-8, 9, (L, D)) / 8.0
        w = rng.integers(1, 17, H) / 16.0
        assert np.array_equal(O.indexer_scores(q, w, k), N.indexer_scores(q, w, k))
        assert np.array_equal(O.indexer_scores(q, w, k.astype(np.float32)), N.indexer_scores(q, w, k))


def test_topk_ema_marks_agree():
    rng = np.random.default_rng(22)
    for _ in range(200):
        L = int(rng.integers(0, 120))
        k = int(rng.integers(1, 60))
        s = (rng.integers(-6, 7, L) * 0.5).astype(np.float64)       # heavy ties
        sel_c, kth_c = O.topk_select(s, k)
        sel_n, kth_n = N.topk_select(s, k)
        assert sel_c.tolist() == sel_n.tolist() and kth_c == kth_n
        th = np.float32(rng.choice([np.inf, rng.normal() * 3]))
        alpha = float(rng.choice([0.5, 0.25, 0.0, 1.0, 0.3]))
        a, b = O.ema_update(th, kth_c, alpha), N.ema_update(th, kth_n, alpha)
        assert (np.isnan(a) and np.isnan(b)) or a == b
        res = rng.random(L) < 0.3
        cap = int(rng.integers(0, 40))
        assert O.prefetch_marks(s, th, res, cap).tolist() == N.prefetch_marks(s, th, res, cap).tolist()
        for Lc, cm, cd in ((L, cap, 0), (L * 97, cap, 32), (L, 0, 5), (0, 7, 3)):
            assert O.prefetch_cap(Lc, cm, cd) == N.prefetch_cap(Lc, cm, cd)
    assert O.metadata_bytes(2_000_000, 200_000) == N.metadata_bytes(2_000_000, 200_000)


def test_attention_agrees():
    rng = np.random.default_rng(23)
    for n in (1, 2, 17, 300):
        q = rng.standard_normal((8, 576))
        c = rng.standard_normal((n, 576))
        oc, lc = O.sparse_mla_decode(q, c, 1 / 24)
        on, ln = N.sparse_mla_decode(q, c, 1 / 24)
        assert np.abs(oc - on).max() <= 1e-12 and np.abs(lc - ln).max() <= 1e-12
        mask = rng.random(n) < 0.6
        mask[0] = True
        dc = O.dense_masked_attention(q, c, mask, 1 / 24)
        dn = N.dense_masked_attention(q, c, mask, 1 / 24)
        assert np.abs(dc - dn).max() <= 1e-12


def _same_cache(a, b):
    assert np.array_equal(a.host2gpu >= 0, b.host2gpu >= 0)
    assert a.resident_priority() == b.resident_priority()
    assert np.array_equal(a.gpu2host, b.gpu2host) and np.array_equal(a.free, b.free)
    assert a.step == b.step and a.status == b.status


def test_cache_sequences_agree():
    # write-backs and recalls (with staged rows) on small pools, with exhaustion
    rng = np.random.default_rng(24)
    for trial in range(25):
        ng, B, span = int(rng.integers(4, 60)), int(rng.integers(1, 5)), 50
        nh = B * span
        a, b = O.LayerCache(ng, nh), N.LayerCache(ng, nh)
        base = np.arange(B, dtype=np.int64) * span
        seq_a = rng.integers(5, 20, B).astype(np.int64)
        seq_b = seq_a.copy()
        for s in range(6):
            na, nb = a.writeback(base, seq_a), b.writeback(base, seq_b)
            assert np.array_equal(na, nb) and np.array_equal(seq_a, seq_b)
            _same_cache(a, b)
            sel, staged = [], []
            for r in range(B):
                L = int(seq_a[r])
                sel.append(rng.choice(L, size=int(rng.integers(0, min(L, 8) + 1)), replace=False))
                nonres = [t for t in range(L) if a.host2gpu[base[r] + t] < 0 and t not in set(sel[-1].tolist())]
                staged.append(np.array(sorted(rng.choice(nonres, size=min(len(nonres), int(rng.integers(0, 4))),
                                                         replace=False)), dtype=np.int64) if nonres else
                              np.zeros(0, dtype=np.int64))
            ra, rb = a.recall(sel, base, staged), b.recall(sel, base, staged)
            assert (ra.hits, ra.staged_hits, ra.misses, ra.slot_host, ra.status) == \
                   (rb.hits, rb.staged_hits, rb.misses, rb.slot_host, rb.status)
            assert np.array_equal(ra.evicted, rb.evicted)
            _same_cache(a, b)
            a.check_invariants()
            m = int(rng.integers(0, 6))
            assert np.array_equal(a.lru_victims(m), b.lru_victims(m))


def test_decode_steps_agree():
    # whole decode steps in lockstep, prefetch on, the cap binding sometimes
    wl = S.small_workload(ctx=(300, 520, 129), topk=64, n_gpu=400, cap_max=12, steps=4)
    B = wl.batch
    keys = [S.grid_to_float(S.keys_for(wl, 0, b, wl.max_ctx)).numpy() for b in range(B)]
    lat = S.latents_for(wl, 0, wl.n_host).float().numpy()
    a, b = O.LayerCache(wl.n_gpu, wl.n_host), N.LayerCache(wl.n_gpu, wl.n_host)
    seq_a, seq_b = np.array(wl.ctx, dtype=np.int64), np.array(wl.ctx, dtype=np.int64)
    th_a = th_b = np.full(B, np.inf, dtype=np.float32)
    qi = S.qidx_initial(wl, 0)
    w = S.weights_for(wl, 0).numpy()
    for s in range(wl.steps):
        q = S.grid_to_float(qi).numpy()
        qm = S.qmla_for(wl, 0, s).float().numpy()
        kw = dict(keys_of=lambda r, L: keys[r][:L], q_idx=q, w_idx=w, k=wl.topk, cap_max=wl.cap_max,
                  cap_div=wl.cap_div, q_mla=qm, latent_of=lambda h: lat[h], scale=wl.scale)
        ra = O.decode_layer_step(a, host_base=wl.host_base, seq_len=seq_a, theta=th_a, **kw)
        rb = N.decode_layer_step(b, host_base=wl.host_base, seq_len=seq_b, theta=th_b, **kw)
        assert np.array_equal(seq_a, seq_b) and np.array_equal(ra.new_host, rb.new_host)
        for r in range(B):
            assert np.array_equal(ra.scores[r], rb.scores[r])
            assert ra.sel[r].tolist() == rb.sel[r].tolist()
            assert ra.staged[r].tolist() == rb.staged[r].tolist()
        assert ra.cap == rb.cap
        assert np.array_equal(ra.kth, rb.kth) and np.array_equal(ra.theta, rb.theta)
        assert (ra.recall.hits, ra.recall.staged_hits, ra.recall.misses, ra.recall.slot_host) == \
               (rb.recall.hits, rb.recall.staged_hits, rb.recall.misses, rb.recall.slot_host)
        assert np.array_equal(ra.recall.evicted, rb.recall.evicted)
        assert np.abs(ra.out - rb.out).max() <= 1e-12 and np.abs(ra.lse - rb.lse).max() <= 1e-12
        _same_cache(a, b)
        th_a, th_b = ra.theta, rb.theta
        qi = S.qidx_next(wl, 0, s, qi)


def test_prefill_block_agrees():
    rng = np.random.default_rng(25)
    Q, H, D, pos0, k = 5, 4, 16, 70, 9
    q = rng.integers(-8, 9, (Q, H, D)) * 0.125
    w = rng.integers(1, 17, (Q, H)) / 16.0
    keys = rng.integers(-8, 9, (pos0 + Q, D)) * 0.125
    for kth_pred in (np.full(Q, np.inf, np.float32), (rng.integers(-8, 9, Q) * 0.5).astype(np.float32)):
        a = O.prefill_block(q, w, keys, pos0, kth_pred, k)
        b = N.prefill_block(q, w, keys, pos0, kth_pred, k)
        for key in ("hist", "thr", "kth", "cand_union", "sel_union"):
            assert np.array_equal(a[key], b[key]), key
        for j in range(Q):
            assert np.array_equal(a["scores"][j], b["scores"][j])
            assert a["cand"][j].tolist() == b["cand"][j].tolist()
            assert a["sel"][j].tolist() == b["sel"][j].tolist()


# ------------------------------------------------- prefill bucket properties --
# The pages fix a 256-bucket coarse histogram of d = score - predicted k-th score and
# say that subtracting the prediction makes the buckets near the boundary (d = 0)
# finer.  The mapping itself is a reading (parity unpinned); these pin what the
# pages do fix: the bucket order follows d, zero splits the range, and a bucket's
# width grows with |d| (relative, not absolute, resolution).
def _bk(d):
    return O.prefill_buckets(np.asarray(d, dtype=np.float32), 0.0)


def test_bucket_monotone_in_d():
    rng = np.random.default_rng(26)
    d = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-38, 38, 4000),
                        [0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3e38, -3e38]]).astype(np.float32)
    d = np.sort(d)
    b = _bk(d)
    assert np.all(np.diff(b) >= 0), "bucket index must not decrease as d grows"
    assert b.min() >= 0 and b.max() <= 255


def test_bucket_zero_splits_the_range():
    rng = np.random.default_rng(27)
    pos = np.abs(rng.standard_normal(2000)).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 2000)
    pos = pos[pos > 0].astype(np.float32)
    assert np.all(_bk(pos) >= 128) and np.all(_bk(-pos) <= 127)
    assert _bk([0.0])[0] == _bk([-0.0])[0] == 128


def test_bucket_width_grows_with_distance_from_zero():
    # two values in one bucket differ by less than a factor 4 (each bucket spans a
    # bounded ratio of |d|), so an absolute bucket width is proportional to |d|:
    # buckets are finest next to the predicted k-th score
    rng = np.random.default_rng(28)
    x = np.abs(rng.standard_normal(20000)).astype(np.float32) * np.float32(2.0) ** rng.integers(-60, 60, 20000)
    x = x[(x > 1e-30) & (x < 1e30)].astype(np.float32)
    for sgn in (1.0, -1.0):
        v = np.float32(sgn) * x
        b = _bk(v)
        for bucket in np.unique(b):
            m = np.abs(v[b == bucket].astype(np.float64))
            assert m.max() / m.min() < 4.0
    # equal numbers of buckets per factor of |d|: as many buckets cover [2^-20, 2^-10]
    # as cover [2^10, 2^20], so a fixed-width interval near 0 holds far more buckets
    lo = np.float32(2.0) ** np.arange(-20, -10, 0.25, dtype=np.float32)
    hi = np.float32(2.0) ** np.arange(10, 20, 0.25, dtype=np.float32)
    assert len(np.unique(_bk(lo))) == len(np.unique(_bk(hi))) >= 4
    near = np.linspace(-1.0, 1.0, 4001, dtype=np.float32)
    far = np.linspace(1000.0, 1002.0, 4001, dtype=np.float32)
    assert len(np.unique(_bk(near))) >= 10 * len(np.unique(_bk(far)))


@pytest.mark.parametrize("shift", [0.0, 37.5, -12.25])
def test_bucket_depends_on_score_minus_prediction(shift):
    # the bucket is a function of score - kth_pred only (where that difference is exact)
    rng = np.random.default_rng(29)
    d = (rng.integers(-4000, 4001, 500) * 0.125).astype(np.float32)
    s = (d + np.float32(shift)).astype(np.float32)
    assert np.array_equal(O.prefill_buckets(s, shift), _bk(d))


def test_adaptive_cap_steps_agree():
    wl = S.small_workload(ctx=(300, 520, 129), topk=64, n_gpu=400, cap_max=60, cap_div=6, steps=4)
    B = wl.batch
    keys = [S.grid_to_float(S.keys_for(wl, 0, b, wl.max_ctx)).numpy() for b in range(B)]
    a, b_ = O.LayerCache(wl.n_gpu, wl.n_host), N.LayerCache(wl.n_gpu, wl.n_host)
    ada, adb = O.AdaptiveCap(B, 7), N.AdaptiveCap(B, 7)
    seq_a, seq_b = np.array(wl.ctx, dtype=np.int64), np.array(wl.ctx, dtype=np.int64)
    th_a = th_b = np.full(B, np.inf, dtype=np.float32)
    qi = S.qidx_initial(wl, 0)
    w = S.weights_for(wl, 0).numpy()
    for s in range(wl.steps):
        kw = dict(keys_of=lambda r, L: keys[r][:L], q_idx=S.grid_to_float(qi).numpy(), w_idx=w, k=wl.topk,
                  cap_max=wl.cap_max, cap_div=wl.cap_div)
        ra = O.decode_layer_step(a, host_base=wl.host_base, seq_len=seq_a, theta=th_a, adaptive=ada, **kw)
        rb = N.decode_layer_step(b_, host_base=wl.host_base, seq_len=seq_b, theta=th_b, adaptive=adb, **kw)
        assert ra.cap == rb.cap
        assert np.array_equal(ada.new_rows, adb.new_rows) and np.array_equal(ada.pred_err, adb.pred_err)
        for r in range(B):
            assert ra.staged[r].tolist() == rb.staged[r].tolist()
        _same_cache(a, b_)
        th_a, th_b = ra.theta, rb.theta
        qi = S.qidx_next(wl, 0, s, qi)


def test_block_writeback_and_scores_agree():
    rng = np.random.default_rng(42)
    for trial in range(20):
        T = int(rng.choice([2, 4, 8]))
        ng, B = int(rng.integers(2, 12)), int(rng.integers(1, 4))
        span = 64
        a, b_ = O.LayerCache(ng, B * span // T), N.LayerCache(ng, B * span // T)
        base = np.arange(B, dtype=np.int64) * span
        seq_a = rng.integers(1, 20, B).astype(np.int64)
        seq_b = seq_a.copy()
        for s in range(12):
            assert np.array_equal(a.writeback_blocks(base, seq_a, T), N.writeback_blocks(b_, base, seq_b, T))
            _same_cache(a, b_)
            if rng.random() < 0.5:                              # a recall of some blocks
                sel = [rng.choice(int(seq_a[r] + T - 1) // T, size=1, replace=False) for r in range(B)]
                ra = a.recall(sel, base // T, [np.zeros(0, dtype=np.int64)] * B)
                rb = b_.recall(sel, base // T, [np.zeros(0, dtype=np.int64)] * B)
                assert (ra.hits, ra.misses, ra.status) == (rb.hits, rb.misses, rb.status)
                _same_cache(a, b_)
        s = rng.integers(-30, 30, 200) * 0.5
        assert np.array_equal(O.block_scores(s, T), N.block_scores(s, T))


def test_gqa_attention_cpp_vs_numpy():
    rng = np.random.default_rng(64)
    for G, d, n in ((1, 8, 1), (8, 128, 300), (16, 64, 77)):
        q, rows = rng.standard_normal((G, d)), rng.standard_normal((n, 2 * d))
        oc, lc = O.sparse_gqa_decode(q, rows, d ** -0.5)
        on, ln = N.sparse_gqa_decode(q, rows, d ** -0.5)
        assert np.allclose(oc, on, rtol=0, atol=1e-12) and np.allclose(lc, ln, rtol=0, atol=1e-12)
