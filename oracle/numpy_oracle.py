"""Numpy restatement of the CPU oracle for the ECHO per-layer decode hot path.

The oracle proper is the plain C++ library (oracle/echo_oracle.cpp); this module
states the same definitions again in numpy, independently, and the tests require
the two to agree.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of ``bench.py``
may import or run anything in this package.  The CUDA library
(``sparse_attention_kv_dsa_gb300``) never imports it, and the two share no code:
no kernels, headers, helpers, tables or pre/post-processing.  Inputs reach both
sides only through the seeded generators in ``sparse_attention_kv_dsa_gb300.synth``,
which hold none of the method's arithmetic.

Plain numpy, float64 for every floating-point step, written so that each
function can be checked against the pages by eye.  Library primitives used as
single steps: matmul, lexsort, exp/log.

Sources (cited below by tag and section):
  [REV]   "ECHO: Efficient KV Cache Offloading with Lossless Prefetching for
          Serving Native Sparse Attention LLMs (OSDI 2026)" review page,
          awesome-system-papers wiki.  Sections:
            "Problem and motivation"                 (DSA indexer -> top-2048 -> MLA)
            "Key observations", Obs. 2 (Fig 7-8)     (EMA of the k-th score, smoothing 0.5)
            "In-graph per-layer cache management"    (free bitmap, eviction priority,
                                                      index buffers, bidirectional map,
                                                      scan+atomic allocation, protect-then-evict,
                                                      no write-back on evict, recall,
                                                      metadata 4*N_H + 13*N_G bytes)
            "Decode: predict the transfer, then recall exactly"  (EMA threshold prefetch,
                                                      global capped counter, exact top-k,
                                                      recall of every missing token)
            "Prefill: overlap recall across query blocks"  (256-bucket coarse histogram)
  [NOTES] "ECHO: Lossless KV Cache Offloading for Sparse Attention LLMs" podcast show
          notes (fixed-size integer tensors on the GPU; guess when, not which).
  [DSA]   DeepSeek-V3.2-Exp report, listed among the show notes' sources: the
          lightning indexer score sum_h w_h * ReLU(q_h . k_t).

Parity unpinned: prefill_buckets.  The pages fix a 256-bucket coarse histogram of the
score minus the predicted k-th score, but no printed example fixes the bucket mapping
(R19); the candidate rule built on it is pinned by brute force on that mapping only.

Readings taken where the pages are silent:
  R1  indexer score: no extra scale; every t < L_b is scored, the token written
      back in this step included.
  R2  top-k with L < k selects all L tokens; the rest of the row is -1; kth is the
      smallest selected score.  L = 0 selects nothing and kth = -inf.
  R3  equal scores: the lower token index wins.
  R4  EMA: theta <- alpha*kth + (1-alpha)*theta, alpha = 0.5, float32 with every
      operation rounded (no fused multiply-add); theta = +inf before the first
      observation and the first observation sets theta = kth.
  R5  "above the threshold" is strict: score > theta.
  R6  the prefetch counter is per (request, layer, step); under the cap the lowest
      token indices win (first cap_b qualifying tokens by ascending t).
  R7  cap_b = min(cap_max, ceil(L_b / cap_div)) when cap_div > 0, else cap_max.
  R8  eviction priority = step of last touch (write-back, prefetch bind, selection);
      victims are the smallest (priority, host index) among resident tokens with
      priority < s, so everything touched in step s is protected.
  R9  prefetched rows are copied during scoring into a per-request staging area;
      they are bound to GPU slots in the recall of the same step, after the
      selected resident tokens have been protected; every staged row is bound.
  R10 the new token of each step enters both the host pool and the GPU cache.
  R11 the GPU cache starts empty; the host pool holds every context token.
  R15 host index of token t of request b is host_base[b] + t.
  R16 the write-back begins a step: s <- s + 1.
  R18 prefill: query j of a block that starts at position pos0 scores the tokens
      t <= pos0 + j (causal; its own key included).
  R19 prefill bucket of a token: d = score - kth_pred in float32 (one rounding);
      bucket = top 8 bits of the order-preserving 32-bit key of d (non-negative:
      sign bit set; negative: every bit inverted; -0 counts as +0).
  R20 prefill threshold bucket = the bucket holding the query's k-th largest d
      (histogram counted down from bucket 255); candidates = tokens in buckets
      strictly above it, so every candidate is in the exact top-k.  A query with
      at most k tokens has every token as a candidate.
  R21 the block's recall list is the union of its queries' tokens, ascending.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

KV_WIDTH = 576          # MLA latent width                    [REV] "Problem and motivation"
V_WIDTH = 512           # value part of the latent (reading R13: the first 512 latent dims)
NOT_RESIDENT = -1

# status codes (same meaning as the library's, defined independently)
ST_OK = 0
ST_POOL_EXHAUSTED = 5
ST_HOST_INDEX = 6


# --------------------------------------------------------------------------
# metadata size -- [REV] "In-graph per-layer cache management"
# --------------------------------------------------------------------------
def metadata_bytes(n_host: int, n_gpu: int) -> int:
    """Per-layer manager metadata: a 4-byte host->GPU entry per host token, and per
    GPU slot 4 (GPU->host) + 4 (priority) + 4 (index buffer) + 1 (free byte)."""
    return 4 * int(n_host) + 13 * int(n_gpu)


# --------------------------------------------------------------------------
# lightning indexer -- [REV] "Problem and motivation"; [DSA]
# --------------------------------------------------------------------------
def indexer_scores(q: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """score(t) = sum_h w[h] * max(0, q[h] . keys[t])   (float64).

    q [H, D], w [H], keys [L, D]  ->  [L] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros(0, dtype=np.float64)
    dots = keys @ q.T                         # [L, H]
    return np.maximum(dots, 0.0) @ w          # [L]


def to_f32_exact(x: np.ndarray) -> np.ndarray:
    """Store float64 scores as float32, refusing any that float32 cannot hold
    exactly (on the synthetic grid every score is exact)."""
    x = np.asarray(x, dtype=np.float64)
    y = x.astype(np.float32)
    if not np.array_equal(y.astype(np.float64), x):
        bad = np.nonzero(y.astype(np.float64) != x)[0][:4]
        raise ValueError(f"score not exact in float32 at t={bad.tolist()}")
    return y


# --------------------------------------------------------------------------
# exact top-k -- [REV] "Problem and motivation" (top 2048),
#                      "Decode: ... recall exactly" (exact selection)
# --------------------------------------------------------------------------
def topk_select(scores: np.ndarray, k: int):
    """The k highest scores, equal scores going to the lower token index (R2, R3).

    Returns (sel, kth): sel = token indices in selection order (best first),
    len min(k, L); kth = score of the last selected token (-inf when L == 0).
    """
    s = np.asarray(scores, dtype=np.float64)
    L = s.shape[0]
    t = np.arange(L)
    order = np.lexsort((t, -s))               # primary: score descending; then t ascending
    n = min(int(k), L)
    sel = order[:n].astype(np.int64)
    kth = float(s[sel[-1]]) if n > 0 else -math.inf
    return sel, kth


def ema_update(theta: float, kth: float, alpha: float = 0.5) -> np.float32:
    """EMA of the k-th score in float32, one rounding per operation (R4).
    [REV] "Key observations" Obs. 2: EMA with smoothing coefficient 0.5."""
    th = np.float32(theta)
    kv = np.float32(kth)
    if math.isinf(float(kv)) and float(kv) < 0:      # nothing selected: unchanged
        return th
    if math.isinf(float(th)) and float(th) > 0:      # first observation
        return kv
    a = np.float32(alpha)
    b = np.float32(np.float32(1.0) - a)
    return np.float32(np.float32(a * kv) + np.float32(b * th))


def prefetch_cap(L: int, cap_max: int, cap_div: int) -> int:
    """R7: the cap grows with the context ([REV] "Decode: ..." -- the limit grows
    with the context length)."""
    if cap_max <= 0:
        return 0
    if cap_div > 0:
        return min(int(cap_max), -(-int(L) // int(cap_div)))
    return int(cap_max)


def prediction_error(theta, kth) -> np.float32:
    """R23: relative error of the threshold as a prediction of the k-th score, float32."""
    th, kv = np.float32(theta), np.float32(kth)
    if not (math.isfinite(float(th)) and math.isfinite(float(kv))) or float(kv) == 0.0:
        return np.float32(0.0)
    return np.float32(np.float32(abs(np.float32(th - kv))) / np.float32(abs(kv)))


def adaptive_cap(L: int, cap_max: int, cap_div: int, new_rows: int, pred_err, slack: int) -> int:
    """R23: last step's transfer grown by the prediction error, plus slack, at most R7's cap."""
    base = prefetch_cap(L, cap_max, cap_div)
    if new_rows < 0 or base <= 0:
        return base
    want = np.float32(np.float32(np.float32(1.0) + np.float32(pred_err)) * np.float32(new_rows))
    want = min(want, np.float32(1.0e9))
    return min(base, max(int(math.ceil(float(want))) + int(slack), 0))


@dataclass
class AdaptiveCap:
    """Per request: the previous step's transfer (-1 before any step) and prediction error."""
    B: int
    slack: int

    def __post_init__(self):
        self.new_rows = np.full(self.B, -1, dtype=np.int64)
        self.pred_err = np.zeros(self.B, dtype=np.float32)


def prefetch_marks(scores: np.ndarray, theta: float, resident: np.ndarray, cap: int) -> np.ndarray:
    """Tokens prefetched while scoring ([REV] "Decode: predict the transfer ..."):
    score above the EMA threshold (strictly, R5), not resident, and among the
    first `cap` such tokens by ascending token index (R6).  theta = +inf marks none.

    scores [L] (float32 values), resident [L] bool.
    """
    s = np.asarray(scores, dtype=np.float64)
    if cap <= 0 or not math.isfinite(float(theta)):
        return np.zeros(0, dtype=np.int64)
    q = np.nonzero((s > float(np.float32(theta))) & ~np.asarray(resident, dtype=bool))[0]
    return q[:cap].astype(np.int64)


# --------------------------------------------------------------------------
# sparse MLA decode -- [REV] "Problem and motivation" (MLA over the selected tokens)
# --------------------------------------------------------------------------
def sparse_mla_decode(q: np.ndarray, latents: np.ndarray, scale: float, v_width: int = V_WIDTH):
    """Attention of every query head over the gathered latents (float64).

    q [Hq, 576], latents [n, 576] (the selected tokens, n >= 1).
    logits = scale * q . c_j over all 576 dims; p = softmax over j;
    out = sum_j p_j c_j[:v_width]; lse = log sum_j exp(logits_j).
    Returns (out [Hq, v_width], lse [Hq]).
    """
    q = np.asarray(q, dtype=np.float64)
    c = np.asarray(latents, dtype=np.float64)
    logits = float(scale) * (q @ c.T)                  # [Hq, n]
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e / l) @ c[:, :v_width]
    lse = m[:, 0] + np.log(l[:, 0])
    return out, lse


def sparse_gqa_decode(q: np.ndarray, rows: np.ndarray, scale: float):
    """One KV head's G query heads over its selected tokens (R26), float64.
    q [G, d]; rows [n, 2d]: key in the first d values, value in the last d."""
    q = np.asarray(q, dtype=np.float64)
    c = np.asarray(rows, dtype=np.float64)
    d = q.shape[1]
    logits = float(scale) * (q @ c[:, :d].T)           # [G, n]
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    z = e.sum(axis=1, keepdims=True)
    return (e / z) @ c[:, d:], m[:, 0] + np.log(z[:, 0])


def dense_masked_attention(q: np.ndarray, cache: np.ndarray, mask: np.ndarray, scale: float,
                           v_width: int = V_WIDTH):
    """Textbook dense attention over a whole cache with a boolean mask: a second,
    independent formulation used to check sparse_mla_decode."""
    q = np.asarray(q, dtype=np.float64)
    c = np.asarray(cache, dtype=np.float64)
    logits = float(scale) * (q @ c.T)
    logits = np.where(np.asarray(mask, dtype=bool)[None, :], logits, -np.inf)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    out = p @ c[:, :v_width]
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


@dataclass
class LayerCache:
    """State of one layer's GPU cache: host->GPU map, GPU->host map, priorities,
    free bitmap.  Slot numbers chosen here (lowest free slot first) are one valid
    choice; only residency, priorities and the maps' consistency are compared."""
    n_gpu: int
    n_host: int
    host2gpu: np.ndarray = field(init=False)
    gpu2host: np.ndarray = field(init=False)
    priority: np.ndarray = field(init=False)
    free: np.ndarray = field(init=False)
    step: int = 0
    status: int = ST_OK

    def __post_init__(self):
        self.host2gpu = np.full(self.n_host, NOT_RESIDENT, dtype=np.int64)
        self.gpu2host = np.full(self.n_gpu, NOT_RESIDENT, dtype=np.int64)
        self.priority = np.zeros(self.n_gpu, dtype=np.int64)
        self.free = np.ones(self.n_gpu, dtype=bool)

    # -- views -------------------------------------------------------------
    def resident_hosts(self) -> np.ndarray:
        return np.sort(self.gpu2host[self.gpu2host >= 0])

    def resident_priority(self) -> dict:
        used = np.nonzero(self.gpu2host >= 0)[0]
        return {int(self.gpu2host[g]): int(self.priority[g]) for g in used}

    def n_free(self) -> int:
        return int(self.free.sum())

    def _flag(self, code: int):
        if self.status == ST_OK:
            self.status = code

    # -- primitives ----------------------------------------------------------
    def lru_victims(self, m: int) -> np.ndarray:
        """The m resident slots with the smallest (priority, host index) among those
        with priority < current step (R8).  Fewer if not enough are eligible."""
        if m <= 0:
            return np.zeros(0, dtype=np.int64)
        used = np.nonzero(self.gpu2host >= 0)[0]
        elig = used[self.priority[used] < self.step]
        order = np.lexsort((self.gpu2host[elig], self.priority[elig]))
        return elig[order[:m]]

    def evict(self, slots: np.ndarray) -> np.ndarray:
        """Free slots; no data moves back (the host already holds every row)."""
        hosts = self.gpu2host[slots].copy()
        self.host2gpu[hosts] = NOT_RESIDENT
        self.gpu2host[slots] = NOT_RESIDENT
        self.free[slots] = True
        return hosts

    def bind(self, h: int) -> int:
        """Give host token h the lowest free slot, stamped with the current step."""
        free = np.nonzero(self.free)[0]
        if free.size == 0:
            return NOT_RESIDENT
        g = int(free[0])
        self.free[g] = False
        self.gpu2host[g] = h
        self.host2gpu[h] = g
        self.priority[g] = self.step
        return g

    # -- A1: write-back of each request's new token ------------------------
    def writeback(self, host_base, seq_len) -> np.ndarray:
        """Begin step s (R16); for each request in order write its new token
        (host index host_base[b] + seq_len[b]) to the host pool and a GPU slot:
        a free slot if there is one, else evict the LRU-smallest token with
        priority < s.  [REV] "In-graph per-layer cache management": every token's
        KV is backed up to the host when generated.  Returns the new host indices
        and increments seq_len in place."""
        self.step += 1
        new_h = np.zeros(len(seq_len), dtype=np.int64)
        for b in range(len(seq_len)):
            h = int(host_base[b]) + int(seq_len[b])
            new_h[b] = h
            seq_len[b] += 1
            if h < 0 or h >= self.n_host:
                self._flag(ST_HOST_INDEX)
                continue
            g = int(self.host2gpu[h])
            if g >= 0:                       # already resident: refresh its stamp
                self.priority[g] = self.step
                continue
            if self.n_free() == 0:
                v = self.lru_victims(1)
                if v.size == 0:
                    self._flag(ST_POOL_EXHAUSTED)
                    continue
                self.evict(v)
            self.bind(h)
        return new_h

    # -- A6..A10: recall after the exact top-k -------------------------------
    def recall(self, sel, host_base, staged) -> RecallResult:
        """[REV] "Decode: ... recall exactly" and "In-graph per-layer cache
        management": find the selected tokens missing from the map, protect the
        selection, evict low-priority tokens, allocate, copy from the host.

        sel[b]    selected token indices of request b (any order)
        staged[b] token indices prefetched (staged) for request b in this step
        Order: (1) stamp every resident selected token with the current step
        (protection, R8); (2) tokens to bind = all staged tokens, then the misses,
        each in (b, t) order; (3) evict the LRU-smallest eligible tokens so that
        enough slots are free; (4) bind; (5) report each selected entry's host index.
        """
        B = len(sel)
        hits, staged_hits, misses = [], [], []
        staged_sets = [set(int(t) for t in staged[b]) for b in range(B)]
        for b in range(B):
            hb, sb, mb = [], [], []
            for t in sel[b]:
                t = int(t)
                h = int(host_base[b]) + t
                g = int(self.host2gpu[h])
                if g >= 0:
                    self.priority[g] = self.step
                    hb.append(t)
                elif t in staged_sets[b]:
                    sb.append(t)
                else:
                    mb.append(t)
            hits.append(sorted(hb))
            staged_hits.append(sorted(sb))
            misses.append(sorted(mb))
        to_bind = []
        for b in range(B):
            to_bind += [int(host_base[b]) + int(t) for t in sorted(staged_sets[b])]
        for b in range(B):
            to_bind += [int(host_base[b]) + t for t in misses[b]]
        need = len(to_bind) - self.n_free()
        victims = self.lru_victims(need)
        evicted = self.evict(victims) if victims.size else np.zeros(0, dtype=np.int64)
        status = ST_OK
        if need > victims.size:
            status = ST_POOL_EXHAUSTED
            self._flag(ST_POOL_EXHAUSTED)
        for h in to_bind:
            if self.bind(h) == NOT_RESIDENT:
                break
        slot_host = []
        for b in range(B):
            row = []
            for t in sel[b]:
                h = int(host_base[b]) + int(t)
                row.append(h if self.host2gpu[h] >= 0 else NOT_RESIDENT)
            slot_host.append(row)
        return RecallResult(hits, staged_hits, misses, np.sort(evicted), slot_host, status)

    def check_invariants(self) -> None:
        """Map invariants of [REV] "In-graph per-layer cache management"."""
        used = np.nonzero(self.gpu2host >= 0)[0]
        assert np.all(self.host2gpu[self.gpu2host[used]] == used)
        res = np.nonzero(self.host2gpu >= 0)[0]
        assert np.all(self.gpu2host[self.host2gpu[res]] == res)
        assert np.array_equal(self.free, self.gpu2host < 0)
        assert used.size + int(self.free.sum()) == self.n_gpu
        assert res.size == used.size <= self.n_gpu


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
    """Run one layer's decode step in the pages' order ([REV] "Decode: predict the
    transfer, then recall exactly"): write-back, score every past token, mark
    above-threshold non-resident tokens for prefetch, exact top-k + EMA, recall,
    sparse MLA.

    keys_of(b, L) -> [L, D] indexer keys of request b (after this step's append)
    latent_of(hosts) -> [n, 576] latents of host indices (host pool rows)
    theta: float32 [B], updated copy returned.
    """
    B = len(seq_len)
    new_h = cache.writeback(host_base, seq_len)
    scores, caps, staged, sels = [], [], [], []
    kth = np.full(B, -np.inf, dtype=np.float32)
    theta_new = np.array(theta, dtype=np.float32).copy()
    for b in range(B):
        L = int(seq_len[b])
        s = to_f32_exact(indexer_scores(q_idx[b], w_idx[b], keys_of(b, L)))
        scores.append(s)
        if not prefetch:
            cap = 0
        elif adaptive is not None:
            cap = adaptive_cap(L, cap_max, cap_div, int(adaptive.new_rows[b]), adaptive.pred_err[b], adaptive.slack)
        else:
            cap = prefetch_cap(L, cap_max, cap_div)
        caps.append(cap)
        hosts = int(host_base[b]) + np.arange(L)
        resident = cache.host2gpu[hosts] >= 0
        staged.append(prefetch_marks(s, theta_new[b], resident, cap))
    for b in range(B):
        sel, kv = topk_select(scores[b], k)
        sels.append(sel)
        kth[b] = np.float32(kv)
        if adaptive is not None:
            adaptive.pred_err[b] = prediction_error(theta_new[b], kv)
        theta_new[b] = ema_update(theta_new[b], kv, alpha)
    rec = cache.recall(sels, host_base, staged)
    if adaptive is not None:
        for b in range(B):
            adaptive.new_rows[b] = len(rec.staged_hits[b]) + len(rec.misses[b])
    out = lse = None
    if q_mla is not None:
        Hq = q_mla.shape[1]
        out = np.zeros((B, Hq, V_WIDTH))
        lse = np.zeros((B, Hq))
        for b in range(B):
            hosts = int(host_base[b]) + np.asarray(sels[b], dtype=np.int64)
            if hosts.size == 0:
                continue
            o, l = sparse_mla_decode(q_mla[b], latent_of(hosts), scale)
            out[b], lse[b] = o, l
    return StepResult(new_h, scores, caps, staged, sels, kth, theta_new, rec, out, lse)


# --------------------------------------------------------------------------
# prefill chunk indexing -- [REV] "Prefill: overlap recall across query blocks"
# (a 256-bucket coarse histogram picks the strictly-high buckets now and leaves
# the threshold bucket for later; subtracting the predicted k-th score makes the
# buckets near the boundary finer); the exact top-k and recall follow.
# --------------------------------------------------------------------------
def prefill_scores(q_blk: np.ndarray, w_blk: np.ndarray, keys: np.ndarray, pos0: int) -> list:
    """Scores of every query of a block over its causal range (R18).

    q_blk [Q, H, D], w_blk [Q, H], keys [>= pos0 + Q, D]  ->  list of Q float64
    arrays, query j of length pos0 + j + 1."""
    return [indexer_scores(q_blk[j], w_blk[j], keys[:pos0 + j + 1]) for j in range(q_blk.shape[0])]


def order_key_f32(x) -> np.ndarray:
    """Order-preserving uint32 key of float32 values, from the IEEE-754 bit
    pattern: larger float -> larger key; -0 and +0 share the key of +0."""
    x = np.asarray(x, dtype=np.float32).copy()
    x[x == 0] = 0.0                                  # -0 -> +0
    u = x.view(np.uint32).astype(np.uint64)
    neg = (u >> 31) == 1
    key = np.where(neg, (~u) & 0xFFFFFFFF, u | 0x80000000)
    return key.astype(np.uint64)


def prefill_buckets(scores_f32: np.ndarray, kth_pred: float) -> np.ndarray:
    """Bucket 0..255 of each score (R19): top byte of the key of score - kth_pred,
    the difference taken in float32.  Parity unpinned: a reading of the pages, which
    print no example of the mapping."""
    d = np.asarray(scores_f32, dtype=np.float32) - np.float32(kth_pred)   # float32 op
    return (order_key_f32(d) >> 24).astype(np.int64)


def prefill_histogram(scores_f32: np.ndarray, kth_pred: float) -> np.ndarray:
    """The 256-bucket histogram of one query's scores."""
    return np.bincount(prefill_buckets(scores_f32, kth_pred), minlength=256).astype(np.int64)


def prefill_candidates(scores_f32: np.ndarray, kth_pred: float, k: int):
    """Threshold bucket and candidate tokens of one query (R20).

    Returns (thr, cand): thr = bucket of the k-th largest d (-1 when the query has
    at most k tokens); cand = ascending token indices with bucket > thr."""
    s = np.asarray(scores_f32, dtype=np.float32)
    L = s.shape[0]
    bk = prefill_buckets(s, kth_pred)
    if L <= k:
        return -1, np.arange(L, dtype=np.int64)
    hist = np.bincount(bk, minlength=256)
    above = 0
    thr = 0
    for bkt in range(255, -1, -1):                   # count down from the top bucket
        if above + hist[bkt] >= k:
            thr = bkt
            break
        above += hist[bkt]
    return thr, np.nonzero(bk > thr)[0].astype(np.int64)


def token_union(lists) -> np.ndarray:
    """Union of token index lists, ascending (R21)."""
    lists = [np.asarray(x, dtype=np.int64) for x in lists]
    if not lists:
        return np.zeros(0, dtype=np.int64)
    return np.unique(np.concatenate(lists))


def prefill_block(q_blk, w_blk, keys, pos0: int, kth_pred, k: int):
    """One query block: scores, histograms, candidates and their union, then the
    exact per-query top-k and the union of the selections.

    Returns a dict with 'scores' (float32 per query), 'hist' [Q, 256], 'thr' [Q],
    'cand' (per query), 'cand_union', 'sel' (per query, selection order), 'kth' [Q]
    and 'sel_union'."""
    Q = q_blk.shape[0]
    scores = [to_f32_exact(s) for s in prefill_scores(q_blk, w_blk, keys, pos0)]
    hist = np.stack([prefill_histogram(scores[j], kth_pred[j]) for j in range(Q)])
    thr, cand, sel, kth = [], [], [], np.zeros(Q, dtype=np.float32)
    for j in range(Q):
        t_j, c_j = prefill_candidates(scores[j], kth_pred[j], k)
        thr.append(t_j)
        cand.append(c_j)
        s_j, kv = topk_select(scores[j], k)
        sel.append(s_j)
        kth[j] = np.float32(kv)
    return {"scores": scores, "hist": hist, "thr": np.array(thr), "cand": cand,
            "cand_union": token_union(cand), "sel": sel, "kth": kth, "sel_union": token_union(sel)}



# --------------------------------------------------------------------------
# block granularity -- [REV] critique (block-sparse / GQA adaptation); reading R25
# --------------------------------------------------------------------------
def block_scores(scores, T: int) -> np.ndarray:
    """Largest score of each block of T tokens."""
    s = np.asarray(scores, dtype=np.float64)
    return np.array([s[j:j + T].max() for j in range(0, s.shape[0], T)], dtype=np.float64)


def writeback_blocks(cache: LayerCache, host_base, seq_len, T: int) -> np.ndarray:
    """Block-mode write-back (R25) on a numpy LayerCache; seq_len grows in place.
    New blocks take their slots first, then the receiving blocks are touched."""
    cache.step += 1
    out = np.zeros(len(seq_len), dtype=np.int64)
    ok = np.zeros(len(seq_len), dtype=bool)
    for b in range(len(seq_len)):
        h = int(host_base[b]) + int(seq_len[b])
        hb = h // T
        out[b] = hb
        seq_len[b] += 1
        if h < 0 or hb >= cache.n_host:
            cache._flag(ST_HOST_INDEX)
            continue
        ok[b] = True
        if h % T or cache.host2gpu[hb] >= 0:
            continue
        if cache.n_free() == 0:
            v = cache.lru_victims(1)
            if v.size == 0:
                cache._flag(ST_POOL_EXHAUSTED)
                continue
            cache.evict(v)
        cache.bind(hb)
    for b in np.nonzero(ok)[0]:
        g = int(cache.host2gpu[out[b]])
        if g >= 0:
            cache.priority[g] = cache.step
    return out
