"""Host-side helpers of bench.py (CPU only): the kernel source hash that keys the committed ncu
traffic figure, and the lookup of that figure."""
import os
import shutil

import pytest

import bench


def test_source_hash_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "kv_cache_decode_kvc_gb300", "csrc")
    root = tmp_path / "repo"
    dst = root / "kv_cache_decode_kvc_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    f = dst / "kvc_internal.cuh"
    text = f.read_text(encoding="utf-8")
    # comments and layout only: same hash
    f.write_text("// a new line comment\n/* and a\n block one */\n" + text.replace("\n", "\n\n", 3), encoding="utf-8")
    assert bench.kernel_source_hash() == h0
    # any change to the code: another hash
    f.write_text(text.replace("constexpr int MAX_B = 1024;", "constexpr int MAX_B = 1023;"), encoding="utf-8")
    assert bench.kernel_source_hash() != h0


def test_traffic_is_reported_only_for_the_profiled_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "decode_kernel_gqa8b_b24.md").write_text(
        "# summary\n\n- kernel_source_sha256: `abcdef0123456789`\n- dram_bytes_per_launch: `485959936`\n",
        encoding="utf-8")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profiles("abcdef0123456789") == pytest.approx(485959936.0)
    assert bench.traffic_from_profiles("0000000000000000") is None
    assert bench.traffic_from_profiles("abcdef0123456789", paged=16) is None  # no such summary

