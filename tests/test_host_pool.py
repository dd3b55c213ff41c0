"""The model-wide host pool's row allocator (echo_host_pool_*, host code) against a
brute-force model of the row space: first fit, coalescing, exhaustion, double frees,
fragmentation limits, and the layer layout.  No GPU needed (unpinned buffers)."""

import ctypes
import random

import pytest
import torch

import sparse_attention_kv_dsa_gb300.echo as E


def test_bytes_and_layer_layout():
    assert E.lib().echo_host_pool_bytes(61, 1000, E.BF16) == 61 * 1000 * 576 * 2
    assert E.lib().echo_host_pool_bytes(3, 7, E.F32) == 3 * 7 * 576 * 4
    assert E.lib().echo_host_pool_bytes(0, 7, E.F32) == 0
    p = E.HostPool(4, 50, torch.bfloat16, pinned=False)
    for l in range(4):
        v = p.layer_rows(l)                     # the view's address is the library's layer offset
        assert v.shape == (50, 576) and v.data_ptr() == p.buf.data_ptr() + l * 50 * 1152


def test_first_fit_and_coalescing_against_bruteforce():
    rng = random.Random(5)
    n = 3000
    p = E.HostPool(2, n, torch.bfloat16, pinned=False)
    used = [False] * n
    live = []

    def first_fit(rows):
        run = 0
        for i in range(n):
            run = run + 1 if not used[i] else 0
            if run == rows:
                return i - rows + 1
        return None

    for it in range(3000):
        if live and (rng.random() < 0.45 or len(live) > 60):
            first, rows = live.pop(rng.randrange(len(live)))
            p.free(first, rows)
            for i in range(first, first + rows):
                used[i] = False
        else:
            rows = rng.choice([1, 2, 7, 40, 133, 500])
            want = first_fit(rows)
            if want is None:
                with pytest.raises(E.EchoError) as ei:
                    p.alloc(rows)
                assert ei.value.code == E.ERR_POOL_EXHAUSTED
                continue
            got = p.alloc(rows)
            assert got == want, f"step {it}: first fit"
            for i in range(got, got + rows):
                assert not used[i]
                used[i] = True
            live.append((got, rows))
        # the free list is exactly the maximal free runs, ascending
        runs, i = [], 0
        while i < n:
            if not used[i]:
                j = i
                while j < n and not used[j]:
                    j += 1
                runs.append((i, j - i))
                i = j
            else:
                i += 1
        assert p.free_ranges() == runs
        assert p.rows_in_use == sum(used)


def test_double_free_and_out_of_range_are_rejected():
    p = E.HostPool(1, 100, torch.bfloat16, pinned=False)
    a = p.alloc(10)
    b = p.alloc(10)
    p.free(a, 10)
    for first, rows in ((a, 10), (a + 5, 10), (b + 5, 10), (95, 10), (-1, 2), (0, 0)):
        with pytest.raises(E.EchoError) as ei:
            p.free(first, rows)
        assert ei.value.code == E.ERR_INVALID_ARG
    assert p.free_ranges() == [(0, 10), (20, 80)]
    p.free(b, 10)
    assert p.free_ranges() == [(0, 100)] and p.rows_in_use == 0


def test_fragmentation_limit_leaves_the_pool_unchanged():
    n = 2 * E.HOST_POOL_MAX_RANGES + 4
    p = E.HostPool(1, n, torch.bfloat16, pinned=False)
    firsts = [p.alloc(1) for _ in range(n)]
    for f in firsts[0::2][:E.HOST_POOL_MAX_RANGES]:   # every other row: as many free ranges as allowed
        p.free(f, 1)
    before = p.free_ranges()
    with pytest.raises(E.EchoError) as ei:
        p.free(firsts[2 * E.HOST_POOL_MAX_RANGES + 2], 1)   # one more isolated range
    assert ei.value.code == E.ERR_UNSUPPORTED
    assert p.free_ranges() == before
    p.free(firsts[1], 1)                                # joins two ranges: always possible
    assert len(p.free_ranges()) == E.HOST_POOL_MAX_RANGES - 1
