"""Host logic of bench.py that needs no GPU: the launch count it claims per step, and
the DRAM-traffic record of the indexer, which is used only while the kernel's source
is the one the ncu capture was taken on."""

import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
IX = [os.path.join(ROOT, "sparse_attention_kv_dsa_gb300", "csrc", f) for f in ("indexer.cu", "common.cuh")]


def test_launches_per_step_follow_the_step_executor():
    import sparse_attention_kv_dsa_gb300.echo as E
    big, small = E.PENDING_LIST_MIN_SLOTS, E.PENDING_LIST_MIN_SLOTS - 1
    # write-back (+ the single-CTA launch on big pools), indexer, top-k, recall, MLA + combine
    assert bench.launches_per_step(True, big) == 7
    assert bench.launches_per_step(True, small) == 6
    assert bench.launches_per_step(False, big) == 7


def test_indexer_traffic_record_matches_the_current_source(monkeypatch):
    traffic, note = bench.kernel_traffic(IX, "saturated-b32-ctx80k-100k-4layer")
    assert traffic is not None and 380e6 < traffic < 400e6, "record taken on another source"
    assert "ncu" in note
    # a source with another digest (any edit of the kernel) invalidates the record
    real = bench.hashlib.sha256

    class Other:
        def __init__(self, data):
            self.h = real(data + b"// edited")

        def hexdigest(self):
            return self.h.hexdigest()

    monkeypatch.setattr(bench.hashlib, "sha256", Other)
    traffic2, note2 = bench.kernel_traffic(IX, "saturated-b32-ctx80k-100k-4layer")
    assert traffic2 is None and "changed" in note2


def test_step_roofline_sums_the_stage_ceilings():
    from sparse_attention_kv_dsa_gb300 import synth as S
    wl = S.workloads()["saturated-b32-ctx80k-100k-4layer"]
    peaks = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "source": "test"}
    r = bench.step_roofline(wl, 90_000.0, 32 * 90_000.0 * 132, {"prefetched_rows": 0.0, "final_recall_rows": 0.0},
                            None, peaks, 4, 1.0)
    us = r["ceiling_us_per_layer"]
    assert abs(us["indexer"] - 32 * 90_000 * 132 / 8e12 * 1e6) < 0.01          # 47.5 us
    assert abs(us["topk"] - (4 * 32 * 90_000 + 8 * 32 * 2048) / 8e12 * 1e6) < 0.01
    # sparse MLA: 18.3 GFLOP at 2 PFLOP/s (9.1 us) is below its 80 MB at 8 TB/s (10.0 us)
    assert abs(us["sparse_mla"] - (32 * 2048 * 1152 + 32 * 128 * (576 + 512) * 2) / 8e12 * 1e6) < 0.01
    assert abs(r["ceiling_ms_per_step"] - sum(us.values()) * 4 / 1e3) < 1e-3
    assert r["frac"] == round(r["ceiling_ms_per_step"] / 1.0, 3)
