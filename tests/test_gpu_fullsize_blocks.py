"""Block granularity and several KV heads at the sizes the benchmark times, by state
hand-off: the oracle takes the GPU's cache state before a step (block residency,
priorities, EMA thresholds, context lengths) and recomputes the whole step
(decode_layer_step_blocks); the step's outputs are compared element by element.

* decode at 64K x 8 (the MLA latent), blocks of 16 tokens, a GPU pool of 1536 blocks so
  every step evicts: two steps, every attention head of one request per step and eight
  heads of two others.
* the GQA workload (16 requests x 8 KV heads = 128 groups of 8 query heads, contexts
  32K-48K), blocks of 16 tokens: one step, attention of eight groups; the same with one
  token per host index and slot, attention of six groups.
* the saturated workload (32 requests at 80K-100K) with blocks of 64 tokens and the
  bench's pool of 3125 blocks: one step, eight heads of three requests.
The rows attention reads are checked against rows built from the inputs alone (the host
pool as filled before any step, and the step inputs for the tokens written back since).
"""

import numpy as np
import pytest
import torch

import oracle as O
from sparse_attention_kv_dsa_gb300 import synth as S

from harness import check_gpu_maps, gpu_residency

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def build(wl, T, kb, n_gpu_blocks, steps_before, steps_total, latents_on_gpu=False):
    """latents_on_gpu: draw the host pool's latents with the GPU generator (fast at the
    largest sizes; the oracle reads them back from the pool), then overwrite the context
    keys with the CPU generator's, which the oracle regenerates."""
    from sparse_attention_kv_dsa_gb300.runtime import BlockDecodeLayer, StepInputs
    wl.layers = 1
    dev = torch.device("cuda")
    dl = BlockDecodeLayer(wl, 0, T, kb, dev, n_gpu_blocks=n_gpu_blocks,
                          gen_device="cuda" if latents_on_gpu else "cpu")
    if latents_on_gpu:
        for b in range(wl.batch):
            dl.idx_k[b, :wl.ctx[b]] = dl.to_ik(S.keys_for(wl, 0, b, wl.ctx[b], "cpu"))
        torch.cuda.synchronize()
    inp = StepInputs(wl, 1, steps_total, dev, gen_device="cpu")   # CPU streams: the oracle regenerates them
    for s in range(steps_before):
        dl.load_step_inputs(inp.q_ik[0][s], inp.new_ik_ik[0][s], inp.new_kv[0][s], inp.q_mla[0][s])
        dl.step()
    torch.cuda.synchronize()
    keys = [S.grid_to_float(S.keys_for(wl, 0, b, wl.ctx[b])).numpy() for b in range(wl.batch)]
    for s in range(steps_before):                          # the keys the steps already appended
        nik = S.grid_to_float(S.new_ik_for(wl, 0, s)).numpy()
        for b in range(wl.batch):
            keys[b] = np.concatenate([keys[b], nik[b:b + 1]])
    return dl, inp, keys


def expected_rows(wl, dl, inp, b, toks, base):
    """Latent rows of group b's tokens from the inputs alone: context tokens from the
    host pool as filled before any step, later tokens from the step input that wrote
    them back."""
    toks = np.asarray(toks, dtype=np.int64)
    ctx = wl.ctx[b]
    out = dl.cache.host_kv[torch.from_numpy(base + np.minimum(toks, ctx - 1))].float().numpy()
    for i, t in enumerate(toks):
        if t >= ctx:
            out[i] = inp.new_kv[0][int(t - ctx)][b].float().cpu().numpy()
    return out


def handoff_step(wl, dl, inp, s, keys, attn_groups, rng):
    T, kb = dl.T, dl.kb
    oc = O.LayerCache(dl.n_gpu_blocks, dl.n_host_blocks)
    oc.host2gpu[:] = dl.cache.host2gpu.cpu().numpy()
    oc.gpu2host[:] = dl.cache.gpu2host.cpu().numpy()
    oc.priority[:] = dl.cache.priority.cpu().numpy()
    oc.free[:] = dl.cache.free_map.cpu().numpy().astype(bool)
    oc.step = int(dl.cache.counters[0].item())
    oc.check_invariants()
    seq = dl.seq_len.cpu().numpy().astype(np.int64)
    theta = dl.theta.cpu().numpy()
    bases = dl.host_base.cpu().numpy().astype(np.int64)
    nik = S.grid_to_float(S.new_ik_for(wl, 0, s)).numpy()
    for b in range(wl.batch):
        keys[b] = np.concatenate([keys[b], nik[b:b + 1]])
    dl.load_step_inputs(inp.q_ik[0][s], inp.new_ik_ik[0][s], inp.new_kv[0][s], inp.q_mla[0][s])
    dl.step()
    torch.cuda.synchronize()
    assert dl.cache.status() == 0
    r = O.decode_layer_step_blocks(oc, host_base=bases, seq_len=seq, T=T, keys_of=lambda b, L: keys[b][:L],
                                   q_idx=S.grid_to_float(inp.q_int[0][s].cpu()).numpy(),
                                   w_idx=dl.w_idx.cpu().numpy(), theta=theta, kb=kb, alpha=wl.alpha)
    assert r.recall.status == 0
    scores = dl.scores.cpu().numpy()
    bsc = dl.bscores.cpu().numpy()
    sel = dl.sel.cpu().numpy()
    miss, n_miss = dl.miss_list.cpu().numpy(), dl.n_miss.cpu().numpy()
    for b in range(wl.batch):
        L = int(seq[b])
        assert np.array_equal(scores[b, :L], r.scores[b]), f"token scores, request {b}"
        assert np.array_equal(bsc[b, :r.bscores[b].shape[0]].astype(np.float64), r.bscores[b]), f"block scores {b}"
        assert set(sel[b].tolist()) - {-1} == set(r.sel[b].tolist()), f"selected blocks, request {b}"
        assert set(miss[b, :n_miss[b]].tolist()) == set(r.recall.misses[b]), f"missing blocks, request {b}"
    assert np.array_equal(dl.kth.cpu().numpy(), r.kth) and np.array_equal(dl.theta.cpu().numpy(), r.theta)
    assert gpu_residency(dl.cache) == oc.resident_priority(), "residency / priorities"
    check_gpu_maps(dl.cache)
    ctr = dl.cache.counters.cpu().numpy()
    hits = sum(len(x) for x in r.recall.hits)
    ms = sum(len(x) for x in r.recall.misses)
    assert (ctr[8], ctr[10]) == (hits, ms), "hit / miss counters"
    # attention (and the rows it read) against the oracle over the host rows of the
    # oracle's selection; the host pool holds every token written so far
    kv = dl.cache.gpu_kv
    slot = dl.slot_idx.cpu().numpy()
    qa = inp.q_mla[0][s].float().cpu().numpy()
    out = dl.out.float().cpu().numpy()
    lse = dl.lse.cpu().numpy()
    for b, heads in attn_groups:
        L = int(seq[b])
        toks = O.block_tokens(r.sel[b], T, L)
        rows = expected_rows(wl, dl, inp, b, toks, bases[b])
        valid = slot[b] >= 0
        got = kv[torch.from_numpy(slot[b][valid]).long().cuda()].float().cpu().numpy()
        assert valid.sum() == toks.size
        gpu_toks = np.array([int(sel[b, j // T]) * T + j % T for j in np.nonzero(valid)[0]])
        assert np.array_equal(got, expected_rows(wl, dl, inp, b, gpu_toks, bases[b])), "rows read"
        if wl.kv_heads:
            o, l_ = O.sparse_gqa_decode(qa[b, heads], rows, wl.scale)
        else:
            o, l_ = O.sparse_mla_decode(qa[b, heads], rows, wl.scale)
        assert np.abs(out[b, heads] - o).max() <= 2e-2, f"attention, request {b}"
        assert np.abs(lse[b, heads] - l_).max() <= 2e-2, f"lse, request {b}"
    return ms


def test_blocks_of_16_at_64k_by_state_handoff():
    wl = S.workloads()["decode-b8-ctx64k"]
    dl, inp, keys = build(wl, 16, 128, 1536, steps_before=2, steps_total=4)
    rng = np.random.default_rng(16)
    misses = 0
    for s in (2, 3):
        others = [int(x) for x in rng.choice([b for b in range(wl.batch) if b != s], 2, replace=False)]
        groups = [(s, np.arange(wl.h_q))] + [(b, rng.choice(wl.h_q, 8, replace=False)) for b in others]
        misses += handoff_step(wl, dl, inp, s, keys, groups, rng)
    assert misses > 0


def test_gqa_groups_at_full_size_by_state_handoff():
    wl = S.workloads()["gqa-b16x8kv-ctx32k-48k-2layer"]
    dl, inp, keys = build(wl, 16, 128, wl.n_gpu // 16, steps_before=2, steps_total=3)
    rng = np.random.default_rng(17)
    groups = [(int(n), np.arange(wl.h_q)) for n in rng.choice(wl.batch, 8, replace=False)]
    assert handoff_step(wl, dl, inp, 2, keys, groups, rng) > 0


def test_blocks_of_64_at_the_saturated_size():
    # the launch configuration of bench.py --blocks 64: 32 requests at 80K-100K, 32 blocks
    # of 64 tokens selected, a pool of 3125 blocks
    wl = S.workloads()["saturated-b32-ctx80k-100k-4layer"]
    dl, inp, keys = build(wl, 64, 32, wl.n_gpu // 64, steps_before=2, steps_total=3, latents_on_gpu=True)
    rng = np.random.default_rng(64)
    groups = [(int(b), rng.choice(wl.h_q, 8, replace=False)) for b in rng.choice(wl.batch, 3, replace=False)]
    handoff_step(wl, dl, inp, 2, keys, groups, rng)


def test_gqa_token_granular_at_full_size():
    # the GQA workload with one token per host index and slot (bench.py --blocks 1)
    wl = S.workloads()["gqa-b16x8kv-ctx32k-48k-2layer"]
    dl, inp, keys = build(wl, 1, wl.topk, wl.n_gpu, steps_before=2, steps_total=3, latents_on_gpu=True)
    rng = np.random.default_rng(65)
    groups = [(int(n), np.arange(wl.h_q)) for n in rng.choice(wl.batch, 6, replace=False)]
    assert handoff_step(wl, dl, inp, 2, keys, groups, rng) > 0
