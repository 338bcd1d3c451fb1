"""The roofline's DRAM traffic comes from a committed ncu record and is valid
only for the kernel source it was captured from: the benchmark reports it while
the source hash matches and null (None) as soon as the kernel changes."""
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEY = "expert_mlp_kernel@decode_t4"


def test_recorded_traffic_matches_the_committed_kernel():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)[KEY]
    assert bench._traffic("expert_mlp_kernel", "decode_t4") == rec["dram_bytes_per_launch"]


def test_traffic_is_dropped_when_the_kernel_source_changes(tmp_path, monkeypatch):
    # a copy of the tree's record and kernel source, then one byte of the source changed
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(ROOT, "profiles", "dram_traffic.json"), tmp_path / "profiles")
    src_dir = tmp_path / "mxfp4_mixture_experts_gemv_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    src = os.path.join(ROOT, "mxfp4_mixture_experts_gemv_gb300", "csrc", "expert_gemm.cu")
    shutil.copy(src, src_dir)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("expert_mlp_kernel", "decode_t4") is not None
    with open(src_dir / "expert_gemm.cu", "a") as f:
        f.write("\n")
    assert bench._traffic("expert_mlp_kernel", "decode_t4") is None
    # an unknown kernel or workload has no record
    assert bench._traffic("expert_mlp_kernel", "prefill_t2048") is None
