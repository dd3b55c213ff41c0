"""Python face of the C++ oracle (oracle/echo_oracle.cpp).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import or run anything in
this package.  The CUDA library never imports it and the two share no code.

Every step of the method runs in the C++ library; this module only converts
arrays (numpy in, numpy out) and keeps the same interface as the numpy oracle in
``oracle/numpy_oracle.py``, which stays as an independent cross-check.  The cache
state lives in numpy arrays that the C++ functions update in place, so tests can
read it, or set it for a state hand-off, element by element.

Sources: see the header of echo_oracle.cpp ([REV] the ECHO review page, [DSA] the
DeepSeek-V3.2-Exp report) and the readings R1..R21 listed there.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

KV_WIDTH = 576          # MLA latent width                    [REV] "Problem and motivation"
V_WIDTH = 512           # value part of the latent (reading R13)
NOT_RESIDENT = -1

# status codes (same meaning as the library's, defined independently)
ST_OK = 0
ST_POOL_EXHAUSTED = 5
ST_HOST_INDEX = 6

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_F = ctypes.c_float
_D = ctypes.c_double


class _CacheT(ctypes.Structure):
    _fields_ = [("n_gpu", _I64), ("n_host", _I64), ("host2gpu", _P), ("gpu2host", _P), ("priority", _P),
                ("free_map", _P), ("step", _I64), ("status", _I32)]


_SIG = {
    "orc_set_threads": (None, [ctypes.c_int]),
    "orc_max_threads": (ctypes.c_int, []),
    "orc_metadata_bytes": (_I64, [_I64, _I64]),
    "orc_indexer_scores": (None, [_P, _P, _I64, _I64, _P, ctypes.c_int, _I64, _P]),
    "orc_to_f32_exact": (_I64, [_P, _I64, _P]),
    "orc_topk_select": (_I64, [_P, _I64, _I64, _P, ctypes.POINTER(_D)]),
    "orc_ema_update": (_F, [_F, _F, _F]),
    "orc_prefetch_cap": (_I64, [_I64, _I64, _I64]),
    "orc_prefetch_marks": (_I64, [_P, _I64, _F, _P, _I64, _P]),
    "orc_prediction_error": (_F, [_F, _F]),
    "orc_adaptive_cap": (_I64, [_I64, _I64, _I64, _I64, _F, _I64]),
    "orc_sparse_mla_decode": (None, [_P, _I64, _P, _I64, _I64, _D, _I64, _P, _P]),
    "orc_sparse_gqa_decode": (None, [_P, _I64, _P, _I64, _I64, _D, _P, _P]),
    "orc_dense_masked_attention": (None, [_P, _I64, _P, _I64, _I64, _P, _D, _I64, _P]),
    "orc_cache_reset": (None, [_P]),
    "orc_cache_n_free": (_I64, [_P]),
    "orc_cache_lru_victims": (_I64, [_P, _I64, _P]),
    "orc_cache_evict": (None, [_P, _P, _I64, _P]),
    "orc_cache_bind": (_I64, [_P, _I64]),
    "orc_cache_writeback": (None, [_P, _P, _P, _I64, _P]),
    "orc_cache_recall": (_I32, [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "orc_cache_check_invariants": (_I32, [_P]),
    "orc_decode_layer_step": (_I32, [_P, _I64, _P, _P, _P, ctypes.c_int, _I64, _I64, _P, _P, _P, _P, _I64, _I64,
                                     _I64, _F, ctypes.c_int, _P, _P, _I64, _P, _P, _P, _I64, _P, _P, _P, _P, _P,
                                     _P, _P, _P, _P, ctypes.c_int, _I64, _P, _P]),
    "orc_block_scores": (_I64, [_P, _I64, _I64, _P]),
    "orc_cache_writeback_blocks": (None, [_P, _P, _P, _I64, _I64, _P]),
    "orc_decode_layer_step_blocks": (_I32, [_P, _I64, _P, _P, _I64, _P, ctypes.c_int, _I64, _I64, _P, _P, _P, _P,
                                            _I64, _F, _P, _P, _I64, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                            _P]),
    "orc_order_key_f32": (None, [_P, _I64, _P]),
    "orc_prefill_buckets": (None, [_P, _I64, _F, _P]),
    "orc_prefill_histogram": (None, [_P, _I64, _F, _P]),
    "orc_prefill_candidates": (_I64, [_P, _I64, _F, _I64, _P, _P]),
    "orc_token_union": (_I64, [_P, _I64, _P]),
    "orc_prefill_block": (_I64, [_P, _P, _I64, _I64, _I64, _P, ctypes.c_int, _I64, _P, _I64, _P, _I64, _P, _P, _P,
                                 _P, _P, _P, _P]),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """Load the oracle library, building it first if it is missing or stale.
    ECHO_ORACLE_LIB names another build of the same source to load instead (the
    mutation tests load deliberately broken copies of the oracle this way)."""
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(os.environ.get("ECHO_ORACLE_LIB") or _build.build())
        for name, (res, args) in _SIG.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _c(x, dtype) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=dtype)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


# --------------------------------------------------------------------------
# metadata size -- [REV] "In-graph per-layer cache management"
# --------------------------------------------------------------------------
def metadata_bytes(n_host: int, n_gpu: int) -> int:
    return int(lib().orc_metadata_bytes(int(n_host), int(n_gpu)))


# --------------------------------------------------------------------------
# lightning indexer -- [REV] "Problem and motivation"; [DSA]
# --------------------------------------------------------------------------
def _keys_arg(keys):
    keys = np.asarray(keys)
    if keys.dtype == np.float32:
        return np.ascontiguousarray(keys), 1
    return _c(keys, np.float64), 0


def indexer_scores(q, w, keys) -> np.ndarray:
    """score(t) = sum_h w[h] * max(0, q[h] . keys[t]); q [H, D], w [H], keys [L, D] -> [L] float64."""
    q = _c(q, np.float64)
    w = _c(w, np.float64).reshape(-1)
    H, D = q.shape
    k, kd = _keys_arg(keys)
    L = int(k.shape[0]) if k.ndim else 0
    out = np.zeros(L, dtype=np.float64)
    if L:
        assert k.shape[1] == D
        lib().orc_indexer_scores(_p(q), _p(w), H, D, _p(k), kd, L, _p(out))
    return out


def to_f32_exact(x) -> np.ndarray:
    x = _c(x, np.float64).reshape(-1)
    out = np.zeros(x.shape[0], dtype=np.float32)
    bad = int(lib().orc_to_f32_exact(_p(x), x.shape[0], _p(out)))
    if bad >= 0:
        raise ValueError(f"score not exact in float32 at t={bad}")
    return out


# --------------------------------------------------------------------------
# exact top-k + EMA -- [REV] "Problem and motivation", "Decode: ...", "Key observations"
# --------------------------------------------------------------------------
def topk_select(scores, k: int):
    s = _c(scores, np.float64).reshape(-1)
    L = s.shape[0]
    sel = np.zeros(max(min(int(k), L), 1), dtype=np.int64)
    kth = _D()
    n = int(lib().orc_topk_select(_p(s), L, int(k), _p(sel), ctypes.byref(kth)))
    return sel[:n].copy(), float(kth.value)


def ema_update(theta, kth, alpha: float = 0.5) -> np.float32:
    return np.float32(lib().orc_ema_update(float(np.float32(theta)), float(kth), float(np.float32(alpha))))


def prefetch_cap(L: int, cap_max: int, cap_div: int) -> int:
    return int(lib().orc_prefetch_cap(int(L), int(cap_max), int(cap_div)))


def prediction_error(theta, kth) -> np.float32:
    """R23: |theta - kth| / |kth| in float32 (0 when either is not finite or kth = 0)."""
    return np.float32(lib().orc_prediction_error(float(np.float32(theta)), float(np.float32(kth))))


def adaptive_cap(L: int, cap_max: int, cap_div: int, new_rows: int, pred_err, slack: int) -> int:
    """R23: min(R7's cap, ceil((1 + pred_err) * new_rows) + slack); R7 alone when new_rows < 0."""
    return int(lib().orc_adaptive_cap(int(L), int(cap_max), int(cap_div), int(new_rows),
                                      float(np.float32(pred_err)), int(slack)))


class AdaptiveCap:
    """State of the adaptive cap (R23) of one layer: per request the previous step's
    transfer (new_rows, -1 before any step) and prediction error."""

    def __init__(self, B: int, slack: int):
        self.new_rows = np.full(B, -1, dtype=np.int64)
        self.pred_err = np.zeros(B, dtype=np.float32)
        self.slack = int(slack)


def prefetch_marks(scores, theta, resident, cap: int) -> np.ndarray:
    s = _c(scores, np.float64).reshape(-1)
    r = _c(np.asarray(resident, dtype=bool), np.uint8).reshape(-1)
    L = s.shape[0]
    out = np.zeros(max(min(int(cap), L), 1), dtype=np.int64)
    n = int(lib().orc_prefetch_marks(_p(s), L, float(np.float32(theta)), _p(r), int(cap), _p(out)))
    return out[:n].copy()


# --------------------------------------------------------------------------
# sparse MLA decode -- [REV] "Problem and motivation"
# --------------------------------------------------------------------------
def sparse_mla_decode(q, latents, scale: float, v_width: int = V_WIDTH):
    q = _c(q, np.float64)
    c = _c(latents, np.float64)
    Hq, D = q.shape
    n = c.shape[0]
    out = np.zeros((Hq, v_width), dtype=np.float64)
    lse = np.zeros(Hq, dtype=np.float64)
    lib().orc_sparse_mla_decode(_p(q), Hq, _p(c), n, D, float(scale), int(v_width), _p(out), _p(lse))
    return out, lse


def sparse_gqa_decode(q, rows, scale: float):
    """Attention of one KV head's G query heads over its selected tokens (R26):
    q [G, d], rows [n, 2d] (key then value).  Returns out [G, d], lse [G]."""
    q = _c(q, np.float64)
    c = _c(rows, np.float64)
    G, d = q.shape
    assert c.ndim == 2 and c.shape[1] == 2 * d and c.shape[0] >= 1
    out = np.zeros((G, d), dtype=np.float64)
    lse = np.zeros(G, dtype=np.float64)
    lib().orc_sparse_gqa_decode(_p(q), G, _p(c), c.shape[0], d, float(scale), _p(out), _p(lse))
    return out, lse


def dense_masked_attention(q, cache, mask, scale: float, v_width: int = V_WIDTH):
    q = _c(q, np.float64)
    c = _c(cache, np.float64)
    m = _c(np.asarray(mask, dtype=bool), np.uint8)
    Hq, D = q.shape
    out = np.zeros((Hq, v_width), dtype=np.float64)
    lib().orc_dense_masked_attention(_p(q), Hq, _p(c), c.shape[0], D, _p(m), float(scale), int(v_width), _p(out))
    return out


# --------------------------------------------------------------------------
# per-layer GPU cache manager -- [REV] "In-graph per-layer cache management"
# --------------------------------------------------------------------------
@dataclass
class RecallResult:
    hits: list            # per request: selected tokens resident at recall time
    staged_hits: list     # per request: selected tokens that were prefetched this step
    misses: list          # per request: selected tokens copied from the host now
    evicted: np.ndarray   # host indices evicted by this recall
    slot_host: list       # per request: host index of the slot behind each selected entry
    status: int = ST_OK


class LayerCache:
    """One layer's GPU cache state in numpy arrays (host2gpu, gpu2host, priority as
    int64, free as bool) that the C++ functions update in place."""

    def __init__(self, n_gpu: int, n_host: int):
        self.n_gpu, self.n_host = int(n_gpu), int(n_host)
        self.host2gpu = np.full(self.n_host, NOT_RESIDENT, dtype=np.int64)
        self.gpu2host = np.full(self.n_gpu, NOT_RESIDENT, dtype=np.int64)
        self.priority = np.zeros(self.n_gpu, dtype=np.int64)
        self.free = np.ones(self.n_gpu, dtype=bool)
        self._s = _CacheT(self.n_gpu, self.n_host, _p(self.host2gpu), _p(self.gpu2host), _p(self.priority),
                          _p(self.free), 0, ST_OK)

    def __setattr__(self, name, value):
        # the arrays are shared with the C++ side: assigning a whole array copies into them
        if name in ("host2gpu", "gpu2host", "priority", "free") and name in self.__dict__:
            self.__dict__[name][...] = value
            return
        object.__setattr__(self, name, value)

    @property
    def ref(self):
        return ctypes.byref(self._s)

    @property
    def step(self) -> int:
        return int(self._s.step)

    @step.setter
    def step(self, v: int) -> None:
        self._s.step = int(v)

    @property
    def status(self) -> int:
        return int(self._s.status)

    @status.setter
    def status(self, v: int) -> None:
        self._s.status = int(v)

    # -- views -------------------------------------------------------------
    def resident_hosts(self) -> np.ndarray:
        return np.sort(self.gpu2host[self.gpu2host >= 0])

    def resident_priority(self) -> dict:
        used = np.nonzero(self.gpu2host >= 0)[0]
        return {int(self.gpu2host[g]): int(self.priority[g]) for g in used}

    def n_free(self) -> int:
        return int(lib().orc_cache_n_free(self.ref))

    # -- primitives ----------------------------------------------------------
    def reset(self) -> None:
        lib().orc_cache_reset(self.ref)

    def lru_victims(self, m: int) -> np.ndarray:
        m = int(m)
        if m <= 0:
            return np.zeros(0, dtype=np.int64)
        out = np.zeros(m, dtype=np.int64)
        n = int(lib().orc_cache_lru_victims(self.ref, m, _p(out)))
        return out[:n].copy()

    def evict(self, slots) -> np.ndarray:
        s = _c(slots, np.int64).reshape(-1)
        hosts = np.zeros(max(s.shape[0], 1), dtype=np.int64)
        lib().orc_cache_evict(self.ref, _p(s), s.shape[0], _p(hosts))
        return hosts[:s.shape[0]].copy()

    def bind(self, h: int) -> int:
        return int(lib().orc_cache_bind(self.ref, int(h)))

    # -- A1 ------------------------------------------------------------------
    def writeback(self, host_base, seq_len) -> np.ndarray:
        """Begin a step and write each request's new token (R10, R16); seq_len is
        incremented in place.  Returns the new host indices."""
        hb = _c(host_base, np.int64).reshape(-1)
        own = isinstance(seq_len, np.ndarray) and seq_len.dtype == np.int64 and seq_len.flags.c_contiguous
        seq = seq_len if own else np.array(seq_len, dtype=np.int64)
        B = seq.shape[0]
        new_h = np.zeros(max(B, 1), dtype=np.int64)
        lib().orc_cache_writeback(self.ref, _p(hb), _p(seq), B, _p(new_h))
        if not own:
            seq_len[:] = seq
        return new_h[:B].copy()

    # -- A6..A10 ---------------------------------------------------------------
    def recall(self, sel, host_base, staged) -> RecallResult:
        B = len(sel)
        hb = _c(host_base, np.int64).reshape(-1)
        sel = [_c(x, np.int64).reshape(-1) for x in sel]
        staged = [_c(x, np.int64).reshape(-1) for x in staged]
        sel_off = np.zeros(B + 1, dtype=np.int64)
        st_off = np.zeros(B + 1, dtype=np.int64)
        sel_off[1:] = np.cumsum([x.shape[0] for x in sel]) if B else []
        st_off[1:] = np.cumsum([x.shape[0] for x in staged]) if B else []
        sel_flat = np.concatenate(sel + [np.zeros(1, dtype=np.int64)])
        st_flat = np.concatenate(staged + [np.zeros(1, dtype=np.int64)])
        n_sel = int(sel_off[-1])
        cat = np.zeros(max(n_sel, 1), dtype=np.int8)
        sh = np.zeros(max(n_sel, 1), dtype=np.int64)
        ev = np.zeros(max(self.n_gpu, 1), dtype=np.int64)
        nev = _I64()
        st = int(lib().orc_cache_recall(self.ref, B, _p(hb), _p(sel_flat), _p(sel_off), _p(st_flat), _p(st_off),
                                        _p(cat), _p(sh), _p(ev), ctypes.byref(nev)))
        return _recall_result(sel, sel_off, cat, sh, ev[:nev.value].copy(), st)

    def writeback_blocks(self, host_base, seq_len, T: int) -> np.ndarray:
        """Block-mode write-back (R25); seq_len grows in place.  Returns each request's
        block of its new token."""
        hb = _c(host_base, np.int64).reshape(-1)
        own = isinstance(seq_len, np.ndarray) and seq_len.dtype == np.int64 and seq_len.flags.c_contiguous
        seq = seq_len if own else np.array(seq_len, dtype=np.int64)
        B = seq.shape[0]
        out = np.zeros(max(B, 1), dtype=np.int64)
        lib().orc_cache_writeback_blocks(self.ref, _p(hb), _p(seq), B, int(T), _p(out))
        if not own:
            seq_len[:] = seq
        return out[:B].copy()

    def check_invariants(self) -> None:
        code = int(lib().orc_cache_check_invariants(self.ref))
        assert code == 0, {1: "host2gpu[gpu2host[g]] != g", 2: "gpu2host[host2gpu[h]] != h",
                           3: "free bitmap disagrees with gpu2host", 4: "resident / used counts"}.get(code, code)


def _recall_result(sel, sel_off, cat, sh, evicted, status) -> RecallResult:
    hits, staged_hits, misses, slot_host = [], [], [], []
    for b, s_b in enumerate(sel):
        c_b = cat[sel_off[b]:sel_off[b + 1]]
        hits.append(sorted(int(t) for t in s_b[c_b == 0]))
        staged_hits.append(sorted(int(t) for t in s_b[c_b == 1]))
        misses.append(sorted(int(t) for t in s_b[c_b == 2]))
        slot_host.append([int(h) for h in sh[sel_off[b]:sel_off[b + 1]]])
    return RecallResult(hits, staged_hits, misses, np.sort(evicted), slot_host, int(status))


# --------------------------------------------------------------------------
# one decode step of one layer: A1..A11 in the pages' order
# --------------------------------------------------------------------------
@dataclass
class StepResult:
    new_host: np.ndarray
    scores: list          # per request float32 [L_b]
    cap: list
    staged: list          # per request: prefetched token indices (ascending)
    sel: list             # per request: selected token indices (selection order)
    kth: np.ndarray       # float32 [B]
    theta: np.ndarray     # float32 [B] after the EMA
    recall: RecallResult
    out: np.ndarray | None
    lse: np.ndarray | None


def decode_layer_step(cache: LayerCache, *, host_base, seq_len, keys_of, q_idx, w_idx, theta,
                      k: int, cap_max: int, cap_div: int, alpha: float = 0.5,
                      q_mla=None, latent_of=None, scale: float | None = None,
                      prefetch: bool = True, adaptive: AdaptiveCap | None = None) -> StepResult:
    """One layer's decode step ([REV] "Decode: predict the transfer, then recall
    exactly"): A1..A10 in orc_decode_layer_step, then A11 (orc_sparse_mla_decode)
    over the rows latent_of(host indices) of each request's selection.  With
    `adaptive` the caps follow R23 and its state moves on to this step's values.

    keys_of(b, L) -> [L, D] indexer keys of request b, this step's new key included
    (L = seq_len[b] + 1); seq_len is incremented in place; theta: float32 [B]."""
    hb = _c(host_base, np.int64).reshape(-1)
    own = isinstance(seq_len, np.ndarray) and seq_len.dtype == np.int64 and seq_len.flags.c_contiguous
    seq = seq_len if own else np.array(seq_len, dtype=np.int64)
    B = seq.shape[0]
    Ls = [int(x) + 1 for x in seq]
    keys = [np.asarray(keys_of(b, Ls[b])) for b in range(B)]
    if all(x.dtype == np.float32 for x in keys):
        keys, kd = [np.ascontiguousarray(x) for x in keys], 1
    else:
        keys, kd = [_c(x, np.float64) for x in keys], 0
    q = _c(q_idx, np.float64)
    H, D = q.shape[1], q.shape[2]
    w = _c(w_idx, np.float64).reshape(B, H)
    th_in = _c(theta, np.float32).reshape(-1)
    kptr = (ctypes.c_void_p * max(B, 1))(*[_p(x) for x in keys])
    Lmax = max(Ls) if B else 1
    caps = [prefetch_cap(L, cap_max, cap_div) if prefetch else 0 for L in Ls]   # R23 never exceeds these
    st_stride = max(caps + [1])
    ad_new = adaptive.new_rows if adaptive is not None else np.zeros(max(B, 1), dtype=np.int64)
    ad_err = adaptive.pred_err if adaptive is not None else np.zeros(max(B, 1), dtype=np.float32)
    new_h = np.zeros(max(B, 1), dtype=np.int64)
    scores = np.zeros((max(B, 1), Lmax), dtype=np.float32)
    cap_out = np.zeros(max(B, 1), dtype=np.int64)
    staged = np.zeros((max(B, 1), st_stride), dtype=np.int64)
    staged_n = np.zeros(max(B, 1), dtype=np.int64)
    sel = np.zeros((max(B, 1), max(int(k), 1)), dtype=np.int64)
    sel_n = np.zeros(max(B, 1), dtype=np.int64)
    kth = np.zeros(max(B, 1), dtype=np.float32)
    th_out = np.zeros(max(B, 1), dtype=np.float32)
    cat = np.zeros((max(B, 1), max(int(k), 1)), dtype=np.int8)
    sh = np.zeros((max(B, 1), max(int(k), 1)), dtype=np.int64)
    ev = np.zeros(max(cache.n_gpu, 1), dtype=np.int64)
    nev, bad_b, bad_t = _I64(), _I64(), _I64()
    st = int(lib().orc_decode_layer_step(
        cache.ref, B, _p(hb), _p(seq), kptr, kd, H, D, _p(q), _p(w), _p(th_in), _p(th_out), int(k), int(cap_max),
        int(cap_div), float(np.float32(alpha)), int(bool(prefetch)), _p(new_h), _p(scores), Lmax, _p(cap_out),
        _p(staged), _p(staged_n), st_stride, _p(sel), _p(sel_n), _p(kth), _p(cat), _p(sh), _p(ev),
        ctypes.byref(nev), ctypes.byref(bad_b), ctypes.byref(bad_t), int(adaptive is not None),
        int(adaptive.slack if adaptive is not None else 0), _p(ad_new), _p(ad_err)))
    if not own:
        seq_len[:] = seq
    if st == -1:
        raise ValueError(f"score not exact in float32 at request {bad_b.value}, t={bad_t.value}")
    sels = [sel[b, :sel_n[b]].copy() for b in range(B)]
    sel_off = np.zeros(B + 1, dtype=np.int64)
    sel_off[1:] = np.cumsum(sel_n[:B])
    cat_flat = np.concatenate([cat[b, :sel_n[b]] for b in range(B)] + [np.zeros(0, dtype=np.int8)])
    sh_flat = np.concatenate([sh[b, :sel_n[b]] for b in range(B)] + [np.zeros(0, dtype=np.int64)])
    rec = _recall_result(sels, sel_off, cat_flat, sh_flat, ev[:nev.value].copy(), st)
    out = lse = None
    if q_mla is not None:
        Hq = q_mla.shape[1]
        out = np.zeros((B, Hq, V_WIDTH))
        lse = np.zeros((B, Hq))
        for b in range(B):
            hosts = int(hb[b]) + sels[b]
            if hosts.size == 0:
                continue
            o, l_ = sparse_mla_decode(q_mla[b], latent_of(hosts), float(scale))
            out[b], lse[b] = o, l_
    return StepResult(new_h[:B].copy(), [scores[b, :Ls[b]].copy() for b in range(B)],
                      [int(x) for x in cap_out[:B]], [staged[b, :staged_n[b]].copy() for b in range(B)], sels,
                      kth[:B].copy(), th_out[:B].copy(), rec, out, lse)


# --------------------------------------------------------------------------
# prefill chunk indexing -- [REV] "Prefill: overlap recall across query blocks"
# --------------------------------------------------------------------------
def prefill_scores(q_blk, w_blk, keys, pos0: int) -> list:
    """Scores of every query of a block over its causal range (R18): query j has
    pos0 + j + 1 entries (float64)."""
    return [indexer_scores(q_blk[j], w_blk[j], np.asarray(keys)[:pos0 + j + 1]) for j in range(q_blk.shape[0])]


def order_key_f32(x) -> np.ndarray:
    """Order-preserving key of float32 values (same shape as x)."""
    shape = np.shape(x)
    x = _c(x, np.float32).reshape(-1)
    out = np.zeros(max(x.shape[0], 1), dtype=np.uint32)
    lib().orc_order_key_f32(_p(x), x.shape[0], _p(out))
    return out[:x.shape[0]].astype(np.uint64).reshape(shape)


def prefill_buckets(scores_f32, kth_pred) -> np.ndarray:
    """R19 (parity unpinned: a reading of the pages); same shape as scores_f32."""
    shape = np.shape(scores_f32)
    s = _c(scores_f32, np.float32).reshape(-1)
    out = np.zeros(max(s.shape[0], 1), dtype=np.int32)
    lib().orc_prefill_buckets(_p(s), s.shape[0], float(np.float32(kth_pred)), _p(out))
    return out[:s.shape[0]].astype(np.int64).reshape(shape)


def prefill_histogram(scores_f32, kth_pred) -> np.ndarray:
    s = _c(scores_f32, np.float32).reshape(-1)
    hist = np.zeros(256, dtype=np.int64)
    lib().orc_prefill_histogram(_p(s), s.shape[0], float(np.float32(kth_pred)), _p(hist))
    return hist


def prefill_candidates(scores_f32, kth_pred, k: int):
    """R20: (thr, cand) of one query; thr = -1 when it has at most k tokens."""
    s = _c(scores_f32, np.float32).reshape(-1)
    cand = np.zeros(max(s.shape[0], 1), dtype=np.int64)
    thr = _I32()
    n = int(lib().orc_prefill_candidates(_p(s), s.shape[0], float(np.float32(kth_pred)), int(k), _p(cand),
                                         ctypes.byref(thr)))
    return int(thr.value), cand[:n].copy()


def token_union(lists) -> np.ndarray:
    """R21: union of token index lists, ascending."""
    flat = np.concatenate([_c(x, np.int64).reshape(-1) for x in lists] + [np.zeros(0, dtype=np.int64)])
    out = np.zeros(max(flat.shape[0], 1), dtype=np.int64)
    n = int(lib().orc_token_union(_p(flat), flat.shape[0], _p(out)))
    return out[:n].copy()


def prefill_block(q_blk, w_blk, keys, pos0: int, kth_pred, k: int):
    """One query block: scores, histograms, candidates and their union, then the
    exact per-query top-k and the union of the selections (keys [>= pos0 + Q, D])."""
    q = _c(q_blk, np.float64)
    Q, H, D = q.shape
    w = _c(w_blk, np.float64).reshape(Q, H)
    kk, kd = _keys_arg(np.asarray(keys)[:pos0 + Q])
    kp = _c(kth_pred, np.float32).reshape(-1)
    S = pos0 + Q
    scores = np.zeros((Q, S), dtype=np.float32)
    hist = np.zeros((Q, 256), dtype=np.int64)
    thr = np.zeros(Q, dtype=np.int32)
    cand = np.zeros((Q, S), dtype=np.int64)
    cand_n = np.zeros(Q, dtype=np.int64)
    sel = np.zeros((Q, max(int(k), 1)), dtype=np.int64)
    sel_n = np.zeros(Q, dtype=np.int64)
    kth = np.zeros(Q, dtype=np.float32)
    bad = int(lib().orc_prefill_block(_p(q), _p(w), Q, H, D, _p(kk), kd, int(pos0), _p(kp), int(k), _p(scores), S,
                                      _p(hist), _p(thr), _p(cand), _p(cand_n), _p(sel), _p(sel_n), _p(kth)))
    if bad >= 0:
        raise ValueError(f"score not exact in float32 at query {bad >> 32}, t={bad & 0xFFFFFFFF}")
    sc = [scores[j, :pos0 + j + 1].copy() for j in range(Q)]
    cands = [cand[j, :cand_n[j]].copy() for j in range(Q)]
    sels = [sel[j, :sel_n[j]].copy() for j in range(Q)]
    return {"scores": sc, "hist": hist, "thr": thr.astype(np.int64), "cand": cands,
            "cand_union": token_union(cands), "sel": sels, "kth": kth, "sel_union": token_union(sels)}


# --------------------------------------------------------------------------
# block granularity -- [REV] critique (block-sparse / GQA adaptation); reading R25
# --------------------------------------------------------------------------
def block_scores(scores, T: int) -> np.ndarray:
    """Largest score of each block of T tokens (the last block may be short)."""
    s = _c(scores, np.float64).reshape(-1)
    L = s.shape[0]
    out = np.zeros(max((L + T - 1) // T, 1), dtype=np.float64)
    n = int(lib().orc_block_scores(_p(s), L, int(T), _p(out)))
    return out[:n].copy()


def block_tokens(sel_blocks, T: int, L: int) -> np.ndarray:
    """Tokens of the selected blocks, in selection order, below the context length L."""
    toks = [int(j) * T + i for j in np.asarray(sel_blocks).reshape(-1) for i in range(T) if int(j) * T + i < L]
    return np.array(toks, dtype=np.int64)


@dataclass
class BlockStepResult:
    new_block: np.ndarray
    scores: list          # per request float32 [L_b] (tokens)
    bscores: list         # per request float64 [ceil(L_b / T)]
    sel: list             # per request: selected block indices (selection order)
    kth: np.ndarray       # float32 [B]: the k/T-th block score
    theta: np.ndarray     # float32 [B]
    recall: RecallResult  # over blocks
    out: np.ndarray | None
    lse: np.ndarray | None


def decode_layer_step_blocks(cache: LayerCache, *, host_base, seq_len, T: int, keys_of, q_idx, w_idx, theta,
                             kb: int, alpha: float = 0.5, q_mla=None, latent_of=None,
                             scale: float | None = None) -> BlockStepResult:
    """One decode step in block mode (R25): orc_decode_layer_step_blocks, then attention
    over every token of the selected blocks below the context length (host rows
    latent_of(host token rows)).  host_base in tokens, a multiple of T per request."""
    hb = _c(host_base, np.int64).reshape(-1)
    assert np.all(hb % T == 0), "each request's host rows must start a block"
    own = isinstance(seq_len, np.ndarray) and seq_len.dtype == np.int64 and seq_len.flags.c_contiguous
    seq = seq_len if own else np.array(seq_len, dtype=np.int64)
    B = seq.shape[0]
    Ls = [int(x) + 1 for x in seq]
    keys = [np.asarray(keys_of(b, Ls[b])) for b in range(B)]
    if all(x.dtype == np.float32 for x in keys):
        keys, kd = [np.ascontiguousarray(x) for x in keys], 1
    else:
        keys, kd = [_c(x, np.float64) for x in keys], 0
    q = _c(q_idx, np.float64)
    H, D = q.shape[1], q.shape[2]
    w = _c(w_idx, np.float64).reshape(B, H)
    th_in = _c(theta, np.float32).reshape(-1)
    kptr = (ctypes.c_void_p * max(B, 1))(*[_p(x) for x in keys])
    Lmax = max(Ls) if B else 1
    bstride = (Lmax + T - 1) // T
    new_b = np.zeros(max(B, 1), dtype=np.int64)
    scores = np.zeros((max(B, 1), Lmax), dtype=np.float32)
    bsc = np.zeros((max(B, 1), bstride), dtype=np.float64)
    nblk = np.zeros(max(B, 1), dtype=np.int64)
    sel = np.zeros((max(B, 1), max(int(kb), 1)), dtype=np.int64)
    sel_n = np.zeros(max(B, 1), dtype=np.int64)
    kth = np.zeros(max(B, 1), dtype=np.float32)
    th_out = np.zeros(max(B, 1), dtype=np.float32)
    cat = np.zeros((max(B, 1), max(int(kb), 1)), dtype=np.int8)
    sh = np.zeros((max(B, 1), max(int(kb), 1)), dtype=np.int64)
    ev = np.zeros(max(cache.n_gpu, 1), dtype=np.int64)
    nev, bad_b, bad_t = _I64(), _I64(), _I64()
    st = int(lib().orc_decode_layer_step_blocks(
        cache.ref, B, _p(hb), _p(seq), int(T), kptr, kd, H, D, _p(q), _p(w), _p(th_in), _p(th_out), int(kb),
        float(np.float32(alpha)), _p(new_b), _p(scores), Lmax, _p(bsc), bstride, _p(nblk), _p(sel), _p(sel_n),
        _p(kth), _p(cat), _p(sh), _p(ev), ctypes.byref(nev), ctypes.byref(bad_b), ctypes.byref(bad_t)))
    if not own:
        seq_len[:] = seq
    if st == -1:
        raise ValueError(f"score not exact in float32 at request {bad_b.value}, t={bad_t.value}")
    sels = [sel[b, :sel_n[b]].copy() for b in range(B)]
    sel_off = np.zeros(B + 1, dtype=np.int64)
    sel_off[1:] = np.cumsum(sel_n[:B])
    cat_flat = np.concatenate([cat[b, :sel_n[b]] for b in range(B)] + [np.zeros(0, dtype=np.int8)])
    sh_flat = np.concatenate([sh[b, :sel_n[b]] for b in range(B)] + [np.zeros(0, dtype=np.int64)])
    rec = _recall_result(sels, sel_off, cat_flat, sh_flat, ev[:nev.value].copy(), st)
    out = lse = None
    if q_mla is not None:
        Hq = q_mla.shape[1]
        out = np.zeros((B, Hq, V_WIDTH))
        lse = np.zeros((B, Hq))
        for b in range(B):
            toks = block_tokens(sels[b], T, Ls[b])
            if toks.size == 0:
                continue
            o, l_ = sparse_mla_decode(q_mla[b], latent_of(int(hb[b]) + toks), float(scale))
            out[b], lse[b] = o, l_
    return BlockStepResult(new_b[:B].copy(), [scores[b, :Ls[b]].copy() for b in range(B)],
                           [bsc[b, :nblk[b]].copy() for b in range(B)], sels, kth[:B].copy(), th_out[:B].copy(), rec,
                           out, lse)
