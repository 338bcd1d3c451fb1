"""The roofline's DRAM traffic comes from a committed ncu record and is valid
only for the kernel source it was captured from: the benchmark reports it while
the source hash matches and null (None) as soon as the kernel changes."""
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEY = "expert_mlp_kernel@decode_t4"


def test_recorded_traffic_is_reported_only_for_its_kernel_source():
    import hashlib
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)[KEY]
    src = os.path.join(ROOT, "mxfp4_mixture_experts_gemv_gb300", "csrc", rec["source"])
    with open(src, "rb") as f:
        same = hashlib.sha256(f.read()).hexdigest()[:16] == rec["source_sha256_16"]
    want = rec["dram_bytes_per_launch"] if same else None
    assert bench._traffic("expert_mlp_kernel", "decode_t4") == want


def test_traffic_is_dropped_when_the_kernel_source_changes(tmp_path, monkeypatch):
    # a copy of the tree's record and kernel source, then one byte of the source changed
    # (the record names the copied source's hash, as a fresh capture would)
    import hashlib
    (tmp_path / "profiles").mkdir()
    src_dir = tmp_path / "mxfp4_mixture_experts_gemv_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    src = os.path.join(ROOT, "mxfp4_mixture_experts_gemv_gb300", "csrc", "expert_gemm.cu")
    shutil.copy(src, src_dir)
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    with open(src, "rb") as f:
        rec[KEY]["source_sha256_16"] = hashlib.sha256(f.read()).hexdigest()[:16]
    with open(tmp_path / "profiles" / "dram_traffic.json", "w") as f:
        json.dump(rec, f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("expert_mlp_kernel", "decode_t4") is not None
    with open(src_dir / "expert_gemm.cu", "a") as f:
        f.write("\n")
    assert bench._traffic("expert_mlp_kernel", "decode_t4") is None
    # an unknown kernel or workload has no record
    assert bench._traffic("expert_mlp_kernel", "prefill_t2048") is None
