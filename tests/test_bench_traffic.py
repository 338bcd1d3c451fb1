"""The roofline's DRAM traffic comes from a committed ncu record and is valid
only for the kernel sources it was captured from (the kernel file and the
headers it includes): the benchmark reports it while their hash matches and
null (None) as soon as any of them changes."""
import hashlib
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mxfp4_mixture_experts_gemv_gb300", "csrc")
KEY = "expert_mlp_kernel@decode_t4"


def _hash(root_csrc, names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(root_csrc, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def test_recorded_traffic_is_reported_only_for_its_kernel_sources():
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)[KEY]
    assert "expert_gemm.cu" in rec["sources"] and "expert_common.cuh" in rec["sources"]
    same = _hash(CSRC, rec["sources"]) == rec["sources_sha256_16"]
    want = rec["dram_bytes_per_launch"] if same else None
    assert bench._traffic("expert_mlp_kernel", "decode_t4") == want


def test_traffic_is_dropped_when_a_kernel_source_changes(tmp_path, monkeypatch):
    # a copy of the tree's record and kernel sources, then one byte of one header
    # changed (the record names the copied sources' hash, as a fresh capture would)
    (tmp_path / "profiles").mkdir()
    src_dir = tmp_path / "mxfp4_mixture_experts_gemv_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    for n in rec[KEY]["sources"]:
        shutil.copy(os.path.join(CSRC, n), src_dir)
    rec[KEY]["sources_sha256_16"] = _hash(str(src_dir), rec[KEY]["sources"])
    with open(tmp_path / "profiles" / "dram_traffic.json", "w") as f:
        json.dump(rec, f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("expert_mlp_kernel", "decode_t4") == rec[KEY]["dram_bytes_per_launch"]
    with open(src_dir / "expert_common.cuh", "a") as f:
        f.write("\n")
    assert bench._traffic("expert_mlp_kernel", "decode_t4") is None
    # an unknown kernel or workload has no record
    assert bench._traffic("expert_mlp_kernel", "prefill_t2048") is None
