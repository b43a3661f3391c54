"""Host-side pieces of bench.py that need no GPU."""
import hashlib
import os

import bench


def _profile(tmp_path, digest):
    p = tmp_path / "prof.md"
    p.write_text("# summary\n\n- gemm_tc.cu sha256[:16]: %s\n"
                 "- dram bytes per launch (verify-row call, M=61): 1054075904\n" % digest)
    return str(p)


def test_profile_traffic_reads_bytes_only_for_the_current_source(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "eagle_speculative_decoding_gb300", "csrc", "gemm_tc.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    monkeypatch.setattr(bench, "PROFILE", _profile(tmp_path, digest))
    assert bench.profile_traffic() == 1054075904.0
    monkeypatch.setattr(bench, "PROFILE", _profile(tmp_path, "0" * 16))
    assert bench.profile_traffic() is None
