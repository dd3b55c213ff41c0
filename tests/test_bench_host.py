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
