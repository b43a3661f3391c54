"""Host-side pieces of bench.py that need no GPU."""
import hashlib
import os
import types

import torch

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


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.samples = lines
    return s


def test_clock_summary_uses_the_window_and_falls_back_to_loaded_samples():
    busy = "2070, 2070, 100, Not Active, Not Active, Not Active, Active"
    idle = "345, 2070, 0, Not Active, Not Active, Not Active, Not Active"
    s = _sampler([(1.0, idle), (2.0, busy), (3.0, busy), (9.0, idle)])
    w = s.summary(1.5, 3.5)
    assert w["window"] == "timed region" and w["sm_mhz"] == 2070 and w["samples"] == 2
    assert w["reasons"] == ["sw_power_cap"]
    # a timed region shorter than the sampling period: the loaded samples of the run
    f = s.summary(5.0, 5.01)
    assert f["samples"] == 2 and f["sm_mhz"] == 2070 and f["window"].startswith("whole GPU run")
    assert _sampler([]).summary(0, 1) is None
    assert _sampler([(1.0, "garbage")]).summary(0, 2) is None


def test_both_arms_print_the_same_config():
    for name in ("llama8b", "serve64"):
        a = bench.workload_config(name, 1)
        assert a == bench.workload_config(name, 1)
        assert a["workload"] == name and a["parallelism"] == "replicas x1"
    assert "7 times" in bench.workload_config("llama8b", 1)["l2"]


def test_cpu_samples_are_bounded_subsets_of_the_batch():
    assert bench.sample_requests("llama8b", False) == 1
    assert bench.sample_requests("serve64", False) == 8
    assert bench.sample_requests("serve64", True) == 4
    for name, c in bench.synth.CONFIGS.items():
        for one in (False, True):
            assert 1 <= bench.sample_requests(name, one) <= c["B"]


def test_call_work_is_the_algorithmic_bytes_and_flops():
    """Per-call work the rows divide by: llama8b's fused projection moves
    W_proj (3 d x d) plus h_low/mid/high and g (4 M d), 102.7 MB; its tree
    attention the prefix and tree K/V of 8 kv heads plus Q and O, 9.6 MB,
    with 4 R Hq D (ctx + R) flops; the statistics LM head W_U plus the rows."""
    wl = types.SimpleNamespace(B=1, R=61, d=4096, Hq=32, Hkv=8, D=128, V=128256,
                               w_lm=torch.empty(1, dtype=torch.bfloat16), ctx_lens=torch.tensor([2048]))
    byts, flops = bench.call_work(wl, "fuse_proj")
    assert byts == 3 * 4096 * 4096 * 2 + 4 * 61 * 4096 * 2 == 102_662_144
    assert flops == 2 * 61 * 12288 * 4096
    byts, flops = bench.call_work(wl, "tree_attn")
    assert byts == (2048 + 61) * 8 * 128 * 2 * 2 + 2 * 61 * 32 * 128 * 2 == 9_637_888
    assert flops == 4 * 61 * 32 * 128 * (2048 + 61)
    byts, flops = bench.call_work(wl, "lmhead_verify_stats")
    assert byts == 128256 * 4096 * 2 + 61 * 4096 * 2 and flops == 2 * 61 * 4096 * 128256
    assert bench.call_work(wl, "tree_verify") is None
