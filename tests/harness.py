"""Lockstep runs of the CUDA decode step and the CPU oracle on the same seeded
inputs, with element-by-element comparisons.  Inputs come from the seeded
generators only (CPU streams, so both sides see identical values)."""

from __future__ import annotations

import numpy as np
import torch

import oracle as O
from sparse_attention_kv_dsa_gb300 import synth as S

ATOL_BF16 = 2e-2    # attention output, bf16 inputs
ATOL_F32 = 1e-5     # attention output, float32 inputs


def gpu_residency(cache) -> dict:
    g2h = cache.gpu2host.cpu().numpy()
    pr = cache.priority.cpu().numpy()
    used = g2h >= 0
    return {int(h): int(p) for h, p in zip(g2h[used], pr[used])}


def check_gpu_maps(cache) -> None:
    """Map invariants on the device arrays: mutual inverse, free bitmap, counts."""
    h2g = cache.host2gpu.cpu().numpy().astype(np.int64)
    g2h = cache.gpu2host.cpu().numpy().astype(np.int64)
    fm = cache.free_map.cpu().numpy()
    used = np.nonzero(g2h >= 0)[0]
    assert np.all(h2g[g2h[used]] == used), "host2gpu[gpu2host[g]] != g"
    res = np.nonzero(h2g >= 0)[0]
    assert np.all(g2h[h2g[res]] == res), "gpu2host[host2gpu[h]] != h"
    assert np.array_equal(fm.astype(bool), g2h < 0), "free bitmap disagrees with gpu2host"
    ctr = cache.counters.cpu().numpy()
    assert ctr[1] == int((g2h < 0).sum()), "n_free counter"
    assert res.size == used.size <= cache.n_gpu
    assert not np.any(h2g <= -2), "staged marks left after the recall"


class Lockstep:
    """One layer of a workload run on the GPU (DecodeLayer) and in the oracle."""

    def __init__(self, wl: S.Workload, *, prefetch=True, cap_max=None, layer=0, adaptive_slack=None):
        from sparse_attention_kv_dsa_gb300.runtime import DecodeLayer, StepInputs
        self.wl = wl
        self.dl = DecodeLayer(wl, layer, "cuda", prefetch=prefetch, cap_max=cap_max, gen_device="cpu",
                              adaptive_slack=adaptive_slack)
        self.adaptive = O.AdaptiveCap(wl.batch, adaptive_slack) if adaptive_slack is not None else None
        self.inp = StepInputs(wl, layer + 1, wl.steps, "cuda", gen_device="cpu")
        self.layer = layer
        self.oc = O.LayerCache(wl.n_gpu, wl.n_host)
        self.keys = [S.grid_to_float(S.keys_for(wl, layer, b, wl.ctx[b])).numpy().astype(np.float64)
                     for b in range(wl.batch)]
        self.lat = self.dl.cache.host_kv.float().numpy().astype(np.float64)
        self.seq = np.array(wl.ctx, dtype=np.int64)
        self.theta = np.full(wl.batch, np.inf, dtype=np.float32)
        self.w = self.dl.w_idx.cpu().numpy()
        self.cap_max = self.dl.cap_max
        self.prefetch = self.dl.prefetch
        self.s = 0

    def step(self, args=None, ops=None):
        """One step on both sides; ops (a dict of DecodeLayer.step_ops arguments)
        issues the GPU step as separate entry-point calls instead of the fused one."""
        wl, l, s = self.wl, self.layer, self.s
        dl = self.dl
        dl.set_step_inputs(self.inp.q_int[l][s], self.inp.new_ik[l][s], self.inp.new_kv[l][s], self.inp.q_mla[l][s])
        if ops is not None:
            dl.step_ops(**ops)
        else:
            dl.step(args=args)
        torch.cuda.synchronize()
        new_ik = S.grid_to_float(self.inp.new_ik[l][s].cpu()).numpy()
        new_kv = self.inp.new_kv[l][s].float().cpu().numpy()
        for b in range(wl.batch):
            self.keys[b] = np.concatenate([self.keys[b], new_ik[b:b + 1]])
            self.lat[wl.host_base[b] + self.seq[b]] = new_kv[b]
        r = O.decode_layer_step(self.oc, host_base=wl.host_base, seq_len=self.seq,
                                keys_of=lambda b, L: self.keys[b][:L],
                                q_idx=S.grid_to_float(self.inp.q_int[l][s].cpu()).numpy(), w_idx=self.w,
                                theta=self.theta, k=wl.topk, cap_max=self.cap_max if self.prefetch else 0,
                                cap_div=wl.cap_div, alpha=wl.alpha,
                                q_mla=self.inp.q_mla[l][s].float().cpu().numpy(),
                                latent_of=lambda h: self.lat[h], scale=wl.scale, adaptive=self.adaptive)
        self.theta = r.theta
        self.s += 1
        return r

    def compare(self, r, *, attention=True) -> dict:
        """Element-by-element comparison of the step just run; returns stats."""
        wl, dl = self.wl, self.dl
        B = wl.batch
        status = dl.cache.status()
        assert status == r.recall.status == 0 or status == r.recall.status, f"device status {status}"
        assert np.array_equal(dl.seq_len.cpu().numpy(), self.seq), "context lengths"
        scores = dl.scratch.scores.cpu().numpy()
        sel = dl.sel.cpu().numpy()
        pf_list = dl.pf_list.cpu().numpy()
        pf_count = dl.pf_count.cpu().numpy()
        miss = dl.miss_list.cpu().numpy()
        n_miss = dl.n_miss.cpu().numpy()
        slot = dl.slot_idx.cpu().numpy()
        g2h = dl.cache.gpu2host.cpu().numpy()
        for b in range(B):
            L = int(self.seq[b])
            assert np.array_equal(scores[b, :L], r.scores[b]), f"scores differ, request {b}"
            n = min(wl.topk, L)
            assert set(sel[b, :n].tolist()) == set(r.sel[b].tolist()), f"top-k set differs, request {b}"
            assert np.all(sel[b, n:] == -1), "padding"
            if self.prefetch:
                got = set(pf_list[b, :pf_count[b]].tolist())
                assert pf_count[b] == len(r.staged[b]), f"prefetch count, request {b}"
                assert got == set(r.staged[b].tolist()), f"prefetch set differs, request {b}"
            assert set(miss[b, :n_miss[b]].tolist()) == set(r.recall.misses[b]), f"miss set, request {b}"
            # slot translation: every selected entry points at its token
            hb = wl.host_base[b]
            for j in range(n):
                assert g2h[slot[b, j]] == hb + sel[b, j], "slot_idx"
        if self.prefetch:
            assert dl.cap.cpu().tolist() == r.cap, "per-request prefetch caps"
        if self.adaptive is not None:
            assert dl.cache.pf_new_rows.cpu().tolist() == self.adaptive.new_rows.tolist(), "adaptive: transfer"
            assert np.array_equal(dl.cache.pf_pred_err.cpu().numpy(), self.adaptive.pred_err), "adaptive: error"
        assert np.array_equal(dl.kth.cpu().numpy(), r.kth), "kth"
        assert np.array_equal(dl.theta.cpu().numpy(), r.theta), "EMA threshold"
        assert gpu_residency(dl.cache) == self.oc.resident_priority(), "residency / priorities"
        check_gpu_maps(dl.cache)
        ctr = dl.cache.counters.cpu().numpy()
        hits = sum(len(x) for x in r.recall.hits)
        sh = sum(len(x) for x in r.recall.staged_hits)
        ms = sum(len(x) for x in r.recall.misses)
        assert (ctr[8], ctr[9], ctr[10]) == (hits, sh, ms), "hit / prefetch-hit / miss counters"
        # recalled data: every selected slot holds its host row
        kv = dl.cache.gpu_kv.float().cpu().numpy()
        for b in range(B):
            n = min(wl.topk, int(self.seq[b]))
            hosts = wl.host_base[b] + sel[b, :n]
            assert np.array_equal(kv[slot[b, :n]], self.lat[hosts].astype(np.float32)), "recalled rows"
        err = None
        if attention:
            out = dl.out.float().cpu().numpy()
            err = float(np.abs(out - r.out).max())
            tol = ATOL_F32 if wl.kv_fp32 else ATOL_BF16
            assert err <= tol, f"attention max abs err {err} > {tol}"
            lse = dl.lse.cpu().numpy()
            assert float(np.abs(lse - r.lse).max()) <= (1e-4 if wl.kv_fp32 else 2e-2)
        return {"hits": hits, "staged_hits": sh, "misses": ms, "attn_err": err}
