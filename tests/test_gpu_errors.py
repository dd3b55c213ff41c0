"""Error paths on the GPU: a recall that cannot free enough slots (the sticky status and
consistent maps), and the calls that block layers, wide rows and unsupported GQA shapes
reject before launching anything."""

import numpy as np
import pytest
import torch

import sparse_attention_kv_dsa_gb300.echo as E

from harness import check_gpu_maps

pytestmark = pytest.mark.gpu
dev = torch.device("cuda")


def test_recall_beyond_the_pool_sets_pool_exhausted_and_keeps_the_maps():
    # 8 GPU slots, one request selecting 16 tokens of which none is resident: the recall
    # binds 8 of them (nothing else is resident, so nothing can be evicted) and flags it
    c = E.LayerCache(8, 64, torch.bfloat16, dev)
    c.reset()
    sel = torch.arange(16, dtype=torch.int32, device=dev).view(1, 16)
    base = torch.zeros(1, dtype=torch.int32, device=dev)
    miss = torch.empty(1, 16, dtype=torch.int32, device=dev)
    n_miss = torch.empty(1, dtype=torch.int32, device=dev)
    slot = torch.empty(1, 16, dtype=torch.int32, device=dev)
    E.cache_recall(c, sel, base, miss, n_miss, slot)
    torch.cuda.synchronize()
    assert c.status() == E.ERR_POOL_EXHAUSTED
    check_gpu_maps(c)
    g2h = c.gpu2host.cpu().numpy()
    assert np.all(g2h >= 0) and set(g2h.tolist()) <= set(range(16))      # every slot holds a selected token
    s = slot.cpu().numpy()[0]
    assert (s >= 0).sum() == 8 and n_miss.item() == 16
    for j, g in enumerate(s):                                                # bound entries point at their token
        if g >= 0:
            assert g2h[g] == j


def _block_layer():
    c = E.LayerCache(16, 64, torch.bfloat16, dev, block_tokens=4)
    c.reset()
    return c


def test_block_layers_reject_the_fused_prefetch_and_the_whole_step_call():
    c = _block_layer()
    B, k = 1, 4
    sel = torch.zeros(B, k, dtype=torch.int32, device=dev)
    base = torch.zeros(B, dtype=torch.int32, device=dev)
    pf_list = torch.zeros(B, 8, dtype=torch.int32, device=dev)
    pf_count = torch.zeros(B, dtype=torch.int32, device=dev)
    stage = torch.zeros(B * 8, 576, dtype=torch.bfloat16, device=dev)
    out = [torch.empty(B, k, dtype=torch.int32, device=dev) for _ in range(2)]
    n_miss = torch.empty(B, dtype=torch.int32, device=dev)
    with pytest.raises(E.EchoError) as ei:
        E.cache_recall(c, sel, base, out[0], n_miss, out[1], pf_list=pf_list, pf_count=pf_count, cap_max=8,
                       stage_kv=stage)
    assert ei.value.code == E.ERR_UNSUPPORTED
    q = torch.zeros(B, 64, 128, dtype=torch.float8_e4m3fn, device=dev)
    with pytest.raises(E.EchoError) as ei:
        E.index_prefetch(q, torch.zeros(B, 64, device=dev), torch.zeros(B, 128, 128, dtype=torch.float8_e4m3fn,
                                                                       device=dev),
                         torch.tensor([16], dtype=torch.int32, device=dev), torch.zeros(B, device=dev),
                         torch.zeros(B, 128, device=dev), layer=c, cap=torch.full((B,), 8, dtype=torch.int32,
                                                                                  device=dev),
                         cap_max=8, host_base=base, pf_list=pf_list, pf_count=pf_count, stage_kv=stage)
    assert ei.value.code == E.ERR_UNSUPPORTED
    a = E.StepArgsT()
    with pytest.raises(E.EchoError) as ei:
        E.decode_layer_step(c, a)
    assert ei.value.code == E.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert c.status() == E.OK                                                # nothing was launched


def test_wide_rows_reject_the_whole_step_call():
    c = E.LayerCache(16, 64, torch.bfloat16, dev, row_elems=256)
    c.reset()
    with pytest.raises(E.EchoError) as ei:
        E.decode_layer_step(c, E.StepArgsT())
    assert ei.value.code == E.ERR_UNSUPPORTED


@pytest.mark.parametrize("G,d", [(17, 128), (8, 96), (8, 256)])
def test_gqa_rejects_unsupported_shapes(G, d):
    q = torch.zeros(2, G, d, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(64, 2 * d, dtype=torch.bfloat16, device=dev)
    slot = torch.zeros(2, 8, dtype=torch.int32, device=dev)
    out = torch.empty(2, G, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(2, G, device=dev)
    with pytest.raises(E.EchoError) as ei:
        E.sparse_gqa_decode(q, kv, slot, d ** -0.5, out, lse)
    assert ei.value.code == E.ERR_UNSUPPORTED


def test_gqa_needs_its_workspace_for_several_splits():
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(64, 256, dtype=torch.bfloat16, device=dev)
    slot = torch.zeros(2, 600, dtype=torch.int32, device=dev)                # three splits
    out = torch.empty(2, 8, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(2, 8, device=dev)
    with pytest.raises(E.EchoError) as ei:
        E.sparse_gqa_decode(q, kv, slot, 128 ** -0.5, out, lse)              # no workspace
    assert ei.value.code == E.ERR_INVALID_ARG
