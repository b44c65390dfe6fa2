"""The bench's roofline `traffic` figure comes from the committed ncu record only
while the kernel source it was captured on is unchanged (host logic, no GPU)."""
import hashlib
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _record(kernel):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)[kernel]


def test_committed_records_are_used_only_for_their_source_and_show_no_rereads():
    for kernel in ("score", "decode"):
        rec = _record(kernel)
        src = os.path.join(ROOT, "sparse_decode_attention_quest_gb300", "csrc", rec["source"])
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if digest != rec["source_sha256_16"]:
            # the source changed since the capture: the bench reports no traffic figure
            assert bench._profile_traffic(kernel) is None
            continue
        assert bench._profile_traffic(kernel) == rec["bytes_per_launch_full_size"]
        # captured DRAM bytes within 2% of the algorithmic bytes: no re-reads
        ratio = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) / rec["algorithmic_bytes_captured"]
        assert 0.98 <= ratio <= 1.02, (kernel, ratio)
        assert rec["bytes_per_launch_full_size"] == round(
            (rec["dram_read_bytes"] + rec["dram_write_bytes"]) * rec["scale_to_full_size"])


def test_a_changed_source_drops_the_figure(tmp_path, monkeypatch):
    # a copy of the tree whose kernel source differs from the one the record names
    prof = tmp_path / "profiles"
    csrc = tmp_path / "sparse_decode_attention_quest_gb300" / "csrc"
    prof.mkdir()
    csrc.mkdir(parents=True)
    rec = _record("score")
    (prof / "traffic.json").write_text(json.dumps({"score": rec}))
    (csrc / rec["source"]).write_text("// another kernel\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._profile_traffic("score") is None
    assert bench._profile_traffic("decode") is None  # no record at all
