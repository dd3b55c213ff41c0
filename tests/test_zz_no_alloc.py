"""The sparse MLA decode variant for callers that may not allocate device memory
(for example code running inside another engine's memory pool, or a process whose
allocator belongs to someone else).  It keeps its split partials in scratch built
into the library instead of a caller workspace; its results must match the regular
entry point's.  Kept in a file collected last so that a failure here does not stop
a run before every other test has run."""

import math

import numpy as np
import pytest
import torch

import sparse_attention_kv_dsa_gb300.echo as E
from sparse_attention_kv_dsa_gb300 import synth as S

dev = "cuda"


def _inputs(seed, dtype, B, Hq, k, N=3000):
    kv = S.normal(seed, (N, 576), dtype).to(dev)
    q = S.normal(seed + 1, (B, Hq, 576), dtype).to(dev)
    g = torch.Generator().manual_seed(seed + 2)
    idx = torch.stack([torch.randperm(N, generator=g)[:k] for _ in range(B)]).to(torch.int32)
    idx[0, k // 3:] = -1                                   # a request with padding
    return q, kv, idx.to(dev)


def _regular(q, kv, idx, scale):
    B, Hq, _ = q.shape
    out = torch.empty(B, Hq, 512, dtype=q.dtype, device=dev)
    lse = torch.empty(B, Hq, device=dev)
    ws = torch.empty(E.mla_workspace_bytes(B, Hq, idx.shape[1]), dtype=torch.uint8, device=dev)
    E.sparse_mla_decode(q, kv, idx, scale, out, lse, ws)
    return out, lse


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,Hq,k,B", [(torch.bfloat16, 128, 2048, 3), (torch.float32, 16, 300, 2)])
def test_noalloc_matches_regular_entry_point_twice(dtype, Hq, k, B):
    scale = 1 / math.sqrt(576)
    for call, seed in enumerate((101, 202)):               # two calls in a row; the scratch keeps the
        q, kv, idx = _inputs(seed, dtype, B, Hq, k)        # first call's contents when the second starts
        ref_out, ref_lse = _regular(q, kv, idx, scale)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        E.sparse_mla_decode_noalloc(q, kv, idx, scale, out, lse)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all(), f"call {call}: non-finite output"
        # the same kernels on the same inputs, and the split merge runs in a fixed
        # order: any difference would be a stale or overlapping partial in the scratch
        assert torch.equal(out, ref_out), f"call {call}: output differs from the regular entry point"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from the regular entry point"


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_scratch():
    B, Hq, k = 64, 128, 2048                                # needs more than 32 MiB of partials
    assert E.mla_workspace_bytes(B, Hq, k) > E.MLA_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, Hq, 576, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(16, 576, dtype=torch.bfloat16, device=dev)
    idx = torch.zeros(B, k, dtype=torch.int32, device=dev)
    out = torch.empty(B, Hq, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hq, device=dev)
    with pytest.raises(E.EchoError) as ei:
        E.sparse_mla_decode_noalloc(q, kv, idx, 1.0, out, lse)
    assert ei.value.code == E.ERR_SCRATCH_LIMIT
