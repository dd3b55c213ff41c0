"""Whole decode steps on the GPU against the oracle, element by element, at sizes
the oracle finishes in seconds (several tiles, ragged tails, eviction pressure,
the cap binding, cold start), plus CUDA Graph replay and the lossless check."""

import numpy as np
import pytest
import torch

from sparse_attention_kv_dsa_gb300 import synth as S

pytestmark = pytest.mark.gpu


def run(wl, steps=None, ops=None, **kw):
    from harness import Lockstep
    ls = Lockstep(wl, **kw)
    stats = []
    for _ in range(steps or wl.steps):
        r = ls.step(ops=ops)
        stats.append(ls.compare(r))
    return ls, stats


def test_fp8_steps_with_prefetch():
    wl = S.small_workload("fp8-b3", ctx=(700, 1500, 333), topk=256, n_gpu=2048, steps=5, cap_max=256, rho=0.9)
    ls, st = run(wl)
    assert sum(s["staged_hits"] for s in st[1:]) > 0, "prefetch never hit: test does not exercise it"


def test_fp8_steps_without_prefetch():
    wl = S.small_workload("fp8-b3-nopf", ctx=(700, 1500, 333), topk=256, n_gpu=2048, steps=3, cap_max=256)
    run(wl, prefetch=False)


def test_fp8_lru_pressure():
    # 3 x 128 selected + new tokens per step into 500 slots: the LRU evicts every step
    wl = S.small_workload("fp8-pressure", ctx=(1200, 900, 2100), topk=128, n_gpu=500, steps=5, cap_max=64, rho=0.7)
    ls, st = run(wl)
    assert ls.dl.cache.read_counters()[11] >= 0


def test_fp8_cap_binds_exact_first_tokens():
    # a tiny cap: qualifying tokens outnumber it, the exact "first cap by t" rule applies
    wl = S.small_workload("fp8-capbind", ctx=(1800, 2500), topk=256, n_gpu=4096, steps=4, cap_max=8, rho=0.5)
    ls, st = run(wl)
    ctr = ls.dl.cache.read_counters()
    assert ctr[15] > ctr[12], "qualifying tokens did not exceed the cap"


@pytest.mark.parametrize("defer_cap", [False, True])
def test_fp8_cap_binds_through_separate_entry_points(defer_cap):
    # the exact cap restored by the indexer's own fix-up launch, or deferred into the
    # top-k launch (echo_topk_prefetch): both must give the oracle's staged set
    wl = S.small_workload("fp8-capbind-ops", ctx=(1800, 2500, 400), topk=256, n_gpu=4096, steps=4, cap_max=8,
                          rho=0.5)
    ls, st = run(wl, ops={"defer_cap": defer_cap})
    ctr = ls.dl.cache.read_counters()
    assert ctr[15] > ctr[12], "qualifying tokens did not exceed the cap"


# a pool of at least ECHO_PENDING_LIST_MIN_SLOTS slots under eviction pressure: the recall's
# victim selection finishes on the candidate list of its first radix pass
@pytest.mark.parametrize("prefetch", [True, False])
def test_fp8_large_pool_evictions(prefetch):
    wl = S.small_workload("fp8-bigpool", ctx=(9000, 7000, 8100), topk=2048, n_gpu=14336, steps=7, cap_max=256,
                          rho=0.6)
    ls, st = run(wl, prefetch=prefetch)
    assert ls.dl.cache.read_counters()[11] > 0, "the recall never evicted"


@pytest.mark.parametrize("slack", [4, 300])
def test_fp8_adaptive_cap(slack):
    # the cap follows the last step's transfer and prediction error (small slack: it
    # binds and the exact "first cap by t" rule runs; large slack: the context rule)
    wl = S.small_workload("fp8-adaptive", ctx=(1800, 2500, 700), topk=256, n_gpu=4096, steps=5, cap_max=1024,
                          cap_div=4, rho=0.6)
    ls, st = run(wl, adaptive_slack=slack)
    assert ls.dl.cache.pf_new_rows.min().item() >= 0


def test_fp8_adaptive_cap_through_separate_entry_points():
    # echo_cache_writeback + echo_cache_reserve + echo_index_prefetch + echo_topk_prefetch
    # (which records the prediction error) + echo_cache_recall
    wl = S.small_workload("fp8-adaptive-ops", ctx=(1800, 2500), topk=256, n_gpu=4096, steps=4, cap_max=1024,
                          cap_div=4, rho=0.6)
    run(wl, ops={"defer_cap": True}, adaptive_slack=4)


def test_fp8_cap_grows_with_context():
    wl = S.small_workload("fp8-capdiv", ctx=(3000, 640), topk=128, n_gpu=2048, steps=3, cap_max=4096, cap_div=32,
                          rho=0.6)
    run(wl)


def test_single_tile_and_ragged_tails():
    wl = S.small_workload("fp8-ragged", ctx=(1, 127, 128, 129, 257), topk=64, n_gpu=1024, steps=3, cap_max=32)
    run(wl)


def test_tiny_fp32_workload_all_steps():
    wl = S.workloads()["tiny-fp32-b1-ctx4k"]
    run(wl)


def test_graph_replay_matches_eager():
    from harness import Lockstep
    wl = S.small_workload("graph", ctx=(900, 1400), topk=128, n_gpu=1024, steps=4, cap_max=64)
    ls = Lockstep(wl)
    r = ls.step()                       # eager first step (cold cache)
    ls.compare(r)
    dl = ls.dl
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    # capture one step; replay it for the next steps with fresh inputs copied in
    snap_inputs = (dl.q_idx.clone(), dl.new_ik.clone(), dl.new_kv.clone(), dl.q_mla.clone())
    # capture on a side stream: the captured work is not run during capture
    state = {k: v.clone() for k, v in [("h2g", dl.cache.host2gpu), ("g2h", dl.cache.gpu2host),
                                       ("pr", dl.cache.priority), ("fm", dl.cache.free_map),
                                       ("ctr", dl.cache.counters), ("seq", dl.seq_len), ("th", dl.theta),
                                       ("ik", dl.idx_k)]}
    with torch.cuda.graph(g, stream=s):
        dl.step(stream=s)
    # restore anything the capture might have touched (nothing runs during capture)
    for k, t in [("h2g", dl.cache.host2gpu), ("g2h", dl.cache.gpu2host), ("pr", dl.cache.priority),
                 ("fm", dl.cache.free_map), ("ctr", dl.cache.counters), ("seq", dl.seq_len), ("th", dl.theta),
                 ("ik", dl.idx_k)]:
        assert torch.equal(t, state[k])
    del snap_inputs
    for _ in range(3):
        l, s_ = ls.layer, ls.s
        dl.set_step_inputs(ls.inp.q_int[l][s_], ls.inp.new_ik[l][s_], ls.inp.new_kv[l][s_], ls.inp.q_mla[l][s_])
        g.replay()
        torch.cuda.synchronize()
        # advance the oracle with the same inputs (Lockstep.step without the GPU call)
        r = _oracle_only_step(ls)
        ls.compare(r)


def _oracle_only_step(ls):
    import oracle as O
    wl, l, s = ls.wl, ls.layer, ls.s
    new_ik = S.grid_to_float(ls.inp.new_ik[l][s].cpu()).numpy()
    new_kv = ls.inp.new_kv[l][s].float().cpu().numpy()
    for b in range(wl.batch):
        ls.keys[b] = np.concatenate([ls.keys[b], new_ik[b:b + 1]])
        ls.lat[wl.host_base[b] + ls.seq[b]] = new_kv[b]
    r = O.decode_layer_step(ls.oc, host_base=wl.host_base, seq_len=ls.seq, keys_of=lambda b, L: ls.keys[b][:L],
                            q_idx=S.grid_to_float(ls.inp.q_int[l][s].cpu()).numpy(), w_idx=ls.w, theta=ls.theta,
                            k=wl.topk, cap_max=ls.cap_max if ls.prefetch else 0, cap_div=wl.cap_div,
                            alpha=wl.alpha, q_mla=ls.inp.q_mla[l][s].float().cpu().numpy(),
                            latent_of=lambda h: ls.lat[h], scale=wl.scale)
    ls.theta = r.theta
    ls.s += 1
    return r


def test_lossless_attention_equals_dense_resident_buffer():
    """Attention over the cache slots is bitwise equal to the same kernel over a fully
    resident buffer (the host pool copied to the GPU) with the same tokens in the same
    list order."""
    from harness import Lockstep
    import sparse_attention_kv_dsa_gb300.echo as E
    for kv32 in (False, True):
        wl = S.small_workload("lossless", ctx=(1000, 600), topk=128, n_gpu=300, steps=3, cap_max=32,
                              kv_fp32=kv32, h_idx=4 if kv32 else 64, d_idx=64 if kv32 else 128, grid=4 if kv32 else 8,
                              w_values=[0.25, 0.5] if kv32 else None, h_q=16 if kv32 else 128)
        ls = Lockstep(wl)
        for _ in range(wl.steps):
            ls.compare(ls.step())
            dl = ls.dl
            dense = dl.cache.host_kv.to("cuda")
            sel = dl.sel
            dense_idx = torch.where(sel >= 0, sel + dl.host_base[:, None], torch.full_like(sel, -1))
            out2 = torch.empty_like(dl.out)
            lse2 = torch.empty_like(dl.lse)
            E.sparse_mla_decode(dl.q_mla, dense, dense_idx.contiguous(), wl.scale, out2, lse2, dl.scratch.mla_ws)
            torch.cuda.synchronize()
            assert torch.equal(out2, dl.out) and torch.equal(lse2, dl.lse)
