"""The GQA attention call (several KV heads) against the oracle on single calls:
random queries and rows, selections with -1 padding and ragged lengths, one to
several splits, G = 1, 8, 16, d = 64 and 128, bf16 and float32."""

import numpy as np
import pytest
import torch

import oracle as O

from harness import ATOL_BF16, ATOL_F32

pytestmark = pytest.mark.gpu


def _case(NG, G, d, k, rows, dtype, seed, pad_frac=0.1, empty_groups=()):
    import sparse_attention_kv_dsa_gb300.echo as E
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(NG, G, d, generator=g).to(dtype)
    kv = torch.randn(rows, 2 * d, generator=g).to(dtype)
    slot = torch.randint(0, rows, (NG, k), generator=g, dtype=torch.int32)
    slot[torch.rand(NG, k, generator=g) < pad_frac] = -1
    for n in empty_groups:
        slot[n] = -1
    out = torch.empty(NG, G, d, dtype=dtype, device="cuda")
    lse = torch.empty(NG, G, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(E.gqa_workspace_bytes(NG, G, d, k), 16), dtype=torch.uint8, device="cuda")
    scale = d ** -0.5
    E.sparse_gqa_decode(q.cuda(), kv.cuda(), slot.cuda(), scale, out, lse, ws)
    torch.cuda.synchronize()
    qn, kvn, sn = q.double().numpy(), kv.double().numpy(), slot.numpy()
    on, ln = out.double().cpu().numpy(), lse.double().cpu().numpy()
    tol = ATOL_BF16 if dtype == torch.bfloat16 else ATOL_F32
    for n in range(NG):
        sel = sn[n][sn[n] >= 0]
        if sel.size == 0:
            assert np.all(on[n] == 0) and np.all(np.isneginf(ln[n])), f"empty group {n}"
            continue
        ref, lref = O.sparse_gqa_decode(qn[n], kvn[sel], scale)
        assert np.abs(on[n] - ref).max() <= tol, f"group {n}: out err {np.abs(on[n] - ref).max()}"
        assert np.abs(ln[n] - lref).max() <= (2e-2 if dtype == torch.bfloat16 else 1e-4), f"group {n}: lse"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("G,d", [(8, 128), (16, 64), (1, 128), (5, 64)])
def test_one_split_and_ragged_tiles(dtype, G, d):
    _case(6, G, d, 200, 3000, dtype, seed=G * 100 + d, empty_groups=(3,))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_several_splits_with_a_ragged_last_one(dtype):
    _case(10, 8, 128, 2048 + 77, 50000, dtype, seed=7, empty_groups=(0,))


def test_single_row_selection_and_heavy_padding():
    _case(4, 16, 128, 1, 10, torch.bfloat16, seed=3, pad_frac=0.0)
    _case(4, 8, 128, 700, 5000, torch.bfloat16, seed=4, pad_frac=0.9)
