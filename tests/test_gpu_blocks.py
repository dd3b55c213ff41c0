"""Block granularity on the GPU against the oracle, step by step (R25).

BlockDecodeLayer runs the library's entry points with T tokens per host index and
GPU slot; the oracle runs decode_layer_step_blocks on the same seeded inputs.
Compared exactly: token scores, block scores and counts, the selected block sets,
the k/T-th block score and theta, the miss sets, residency with priorities, the
hit/miss counters, every resident block's rows below the context length (lossless),
the token slots handed to attention; the attention output within the bf16 / fp32
tolerances of the token-granular tests."""

import numpy as np
import pytest
import torch

import oracle as O
from sparse_attention_kv_dsa_gb300 import synth as S

from harness import ATOL_BF16, ATOL_F32, check_gpu_maps, gpu_residency

pytestmark = pytest.mark.gpu


def _run(wl, T, kb, n_gpu_blocks, steps):
    from sparse_attention_kv_dsa_gb300.runtime import BlockDecodeLayer, StepInputs
    dl = BlockDecodeLayer(wl, 0, T, kb, "cuda", n_gpu_blocks=n_gpu_blocks, gen_device="cpu")
    inp = StepInputs(wl, 1, steps, "cuda", gen_device="cpu")
    B = wl.batch
    bases = dl.host_base.cpu().numpy().astype(np.int64)
    oc = O.LayerCache(dl.n_gpu_blocks, dl.n_host_blocks)
    keys = [S.grid_to_float(S.keys_for(wl, 0, b, wl.ctx[b])).numpy().astype(np.float64) for b in range(B)]
    lat = dl.cache.host_kv.float().numpy().astype(np.float64)
    seq = np.array(wl.ctx, dtype=np.int64)
    theta = np.full(B, np.inf, dtype=np.float32)
    w = dl.w_idx.cpu().numpy()
    tot_miss = 0
    for s in range(steps):
        dl.set_step_inputs(inp.q_int[0][s], inp.new_ik[0][s], inp.new_kv[0][s], inp.q_mla[0][s])
        dl.step()
        torch.cuda.synchronize()
        new_ik = S.grid_to_float(inp.new_ik[0][s].cpu()).numpy()
        new_kv = inp.new_kv[0][s].float().cpu().numpy()
        for b in range(B):
            keys[b] = np.concatenate([keys[b], new_ik[b:b + 1]])
            lat[bases[b] + seq[b]] = new_kv[b]
        q_att = inp.q_mla[0][s].float().cpu().numpy()
        gqa = wl.kv_heads > 0
        r = O.decode_layer_step_blocks(oc, host_base=bases, seq_len=seq, T=T, keys_of=lambda b, L: keys[b][:L],
                                       q_idx=S.grid_to_float(inp.q_int[0][s].cpu()).numpy(), w_idx=w,
                                       theta=theta, kb=kb, alpha=wl.alpha, q_mla=None if gqa else q_att,
                                       latent_of=lambda rows: lat[rows], scale=wl.scale)
        if gqa:                                   # each group's query heads over its own selection
            r.out = np.zeros((B, wl.h_q, wl.q_width))
            r.lse = np.zeros((B, wl.h_q))
            for b in range(B):
                toks = O.block_tokens(r.sel[b], T, int(seq[b]))
                r.out[b], r.lse[b] = O.sparse_gqa_decode(q_att[b], lat[bases[b] + toks], wl.scale)
        theta = r.theta
        assert dl.cache.status() == r.recall.status == 0
        assert np.array_equal(dl.seq_len.cpu().numpy(), seq)
        scores = dl.scores.cpu().numpy()
        bsc = dl.bscores.cpu().numpy()
        nblk = dl.seq_len_blk.cpu().numpy()
        sel = dl.sel.cpu().numpy()
        miss = dl.miss_list.cpu().numpy()
        n_miss = dl.n_miss.cpu().numpy()
        slot_blk = dl.slot_blk.cpu().numpy()
        slot = dl.slot_idx.cpu().numpy()
        g2h = dl.cache.gpu2host.cpu().numpy()
        for b in range(B):
            L = int(seq[b])
            assert np.array_equal(scores[b, :L], r.scores[b]), f"token scores, request {b}"
            assert nblk[b] == r.bscores[b].shape[0] == -(-L // T)
            assert np.array_equal(bsc[b, :nblk[b]].astype(np.float64), r.bscores[b]), f"block scores, request {b}"
            n = min(kb, int(nblk[b]))
            assert set(sel[b, :n].tolist()) == set(r.sel[b].tolist()), f"selected blocks, request {b}"
            assert np.all(sel[b, n:] == -1)
            assert set(miss[b, :n_miss[b]].tolist()) == set(r.recall.misses[b]), f"missing blocks, request {b}"
            for j in range(kb):                   # the token slots handed to attention
                for i in range(T):
                    want = -1
                    if j < n and sel[b, j] * T + i < L:
                        assert g2h[slot_blk[b, j]] == bases[b] // T + sel[b, j]
                        want = int(slot_blk[b, j]) * T + i
                    assert slot[b, j * T + i] == want, f"slot of request {b}, block entry {j}, token {i}"
        assert np.array_equal(dl.kth.cpu().numpy(), r.kth), "k/T-th block score"
        assert np.array_equal(dl.theta.cpu().numpy(), r.theta), "EMA threshold"
        assert gpu_residency(dl.cache) == oc.resident_priority(), "residency / priorities"
        check_gpu_maps(dl.cache)
        ctr = dl.cache.counters.cpu().numpy()
        hits = sum(len(x) for x in r.recall.hits)
        ms = sum(len(x) for x in r.recall.misses)
        assert (ctr[8], ctr[10]) == (hits, ms), "hit / miss counters"
        tot_miss += ms
        # lossless: every resident block holds its host rows below the context length
        kv = dl.cache.gpu_kv.float().cpu().numpy()
        for g in np.nonzero(g2h >= 0)[0]:
            row0 = int(g2h[g]) * T
            b = int(np.searchsorted(bases, row0, side="right")) - 1
            n_valid = min(T, int(bases[b] + seq[b]) - row0)
            assert np.array_equal(kv[g * T:g * T + n_valid], lat[row0:row0 + n_valid].astype(np.float32)), \
                f"rows of resident block {g2h[g]}"
        out = dl.out.float().cpu().numpy()
        tol = ATOL_F32 if wl.kv_fp32 else ATOL_BF16
        assert float(np.abs(out - r.out).max()) <= tol, "attention output"
        assert float(np.abs(dl.lse.cpu().numpy() - r.lse).max()) <= (1e-4 if wl.kv_fp32 else 2e-2)
    return tot_miss


def test_blocks_of_16_with_evictions():
    wl = S.small_workload(ctx=(300, 520, 129), topk=96, n_gpu=640, cap_max=0, steps=8)
    assert _run(wl, 16, 6, 24, wl.steps) > 0


def test_blocks_of_64_several_tiles_bf16():
    wl = S.small_workload(ctx=(3000, 5200, 1290), topk=256, n_gpu=4096, cap_max=0, steps=6)
    _run(wl, 64, 4, 20, wl.steps)


def test_blocks_fp32_short_requests_and_padding():
    # one request shorter than kb blocks (padding), T that does not divide the lengths
    wl = S.small_workload(ctx=(40, 700, 333), kv_fp32=True, topk=120, n_gpu=512, cap_max=0, steps=5)
    _run(wl, 12, 10, 40, wl.steps)


def test_single_token_blocks_match_the_token_step():
    # T = 1 is the token-granular cache without prefetch
    wl = S.small_workload(ctx=(700, 1500, 333), topk=256, n_gpu=1024, cap_max=0, steps=4)
    _run(wl, 1, 256, 1024, wl.steps)


# ------------------------------------------------ several KV heads (R26) --
def test_gqa_groups_in_blocks_of_16_bf16():
    # 3 requests x 4 KV heads = 12 groups, 8 query heads each, d = 128
    wl = S.gqa_workload(ctx=(300, 520, 129), kv_heads=4, group=8, head_dim=128, topk=96, steps=6)
    assert _run(wl, 16, 6, 90, wl.steps) > 0


def test_gqa_token_granular_fp32_d64():
    wl = S.gqa_workload(ctx=(700, 333), kv_heads=2, group=16, head_dim=64, topk=300, kv_fp32=True, steps=4)
    _run(wl, 1, 300, 2048, wl.steps)
