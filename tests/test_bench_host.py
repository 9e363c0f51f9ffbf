"""Host logic of the benchmark on CPU: the algorithmic byte models, the lookup
of recorded DRAM traffic by source digest, and the clock-sample summary."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

SERVING = synth.WORKLOADS["mamba2_serving_b256"]


def test_m2_conventional_bytes_are_two_state_passes_plus_token_io():
    w = SERVING
    B, H, P, N, G = w.batch, w.heads, w.head_dim, w.state_dim, w.groups
    tok_in = P * 2 + 2 + 2 * N * 2 / (H / G)
    want = B * H * (2 * P * N * 4 + tok_in + P * 2)
    assert bench.m2_step_bytes(w, 0, False, "conventional", "none", 2) == pytest.approx(want)


def test_m2_replay_bytes_structure():
    """A non-flush step reads the checkpoint once and appends one record; the
    flush writes the checkpoint; each buffered record adds its bytes; a read
    copy replaces the checkpoint read; low-precision checkpoints shrink it."""
    w = SERVING
    P, N, tiles = w.head_dim, w.state_dim, w.batch * w.heads
    nf0 = bench.m2_step_bytes(w, 0, False, "replay", "none", 2)
    nf5 = bench.m2_step_bytes(w, 5, False, "replay", "none", 2)
    record = P * 2 + 2 + N * 2 / (w.heads / w.groups)
    assert nf5 - nf0 == pytest.approx(5 * tiles * record)
    fl = bench.m2_step_bytes(w, 15, True, "replay", "none", 2)
    nf15 = bench.m2_step_bytes(w, 15, False, "replay", "none", 2)
    assert fl - nf15 == pytest.approx(tiles * (P * N * 4 - record))
    fp8 = bench.m2_step_bytes(w, 0, False, "replay", "fp8", 2)
    assert nf0 - fp8 == pytest.approx(tiles * (P * N * 4 - (P * N + 4)))
    f16 = bench.m2_step_bytes(w, 0, False, "replay", "none", 2, "f16")
    assert nf0 - f16 == pytest.approx(tiles * P * N * 2)
    # per 16-token window: replay moves about 17/32 of the conventional state bytes
    win = sum(bench.m2_step_bytes(w, c, c == 15, "replay", "none", 2) for c in range(16))
    conv = 16 * bench.m2_step_bytes(w, 0, False, "conventional", "none", 2)
    assert 0.53 < win / conv < 0.56


def test_gdn_bytes_with_a_read_copy():
    w = synth.WORKLOADS["gdn_serving_b256"]
    tiles, DV, DK = w.batch * w.heads, w.d_v, w.d_k
    plain = bench.gdn_step_bytes(w, 3, False, "replay", 2)
    copy = bench.gdn_step_bytes(w, 3, False, "replay", 2, "fp8")
    # the copy replaces the FP32 read; records carry v and beta as well (3 read + 1 appended)
    want = plain - tiles * (DV * DK * 4 - (DV * DK + DV / 16)) + tiles * 4 * (DV * 2 + 4)
    assert copy == pytest.approx(want)


def test_profiled_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "hybrid_ssm_decode_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "m2_replay_tma.cu").write_text("kernel v1")
    (csrc / "m2_pipeline.cuh").write_text("header")
    (tmp_path / "profiles").mkdir()
    digest = bench.source_digest("m2_replay_nf_kernel")
    (tmp_path / "profiles" / "x.md").write_text(
        "`traffic: kernel=m2_replay_nf_kernel workload=mamba2_serving_b256 batch=256 k=16 "
        f"bytes_per_launch=123 sources={digest}`\n")
    assert bench.profiled_traffic("m2_replay_nf_kernel", SERVING) == 123.0
    assert bench.profiled_traffic("m2_replay_nf_kernel", SERVING.replace(batch=64)) is None
    (csrc / "m2_replay_tma.cu").write_text("kernel v2")
    assert bench.profiled_traffic("m2_replay_nf_kernel", SERVING) is None


def test_draft_kernels_have_their_own_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "hybrid_ssm_decode_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("gdn_replay_tma.cu", "gdn_draft_tma.cu", "gdn_pipeline.cuh", "m2_replay_tma.cu",
                 "m2_draft_tma.cu", "m2_pipeline.cuh"):
        (csrc / name).write_text(name)
    d = {k: bench.source_digest(k) for k in ("gdn_replay_nf_kernel", "gdn_replay_draft_kernel",
                                             "m2_replay_nf_kernel", "m2_replay_draft_tma_kernel")}
    assert len(set(d.values())) == 4
    (csrc / "gdn_draft_tma.cu").write_text("changed")
    assert bench.source_digest("gdn_replay_draft_kernel") != d["gdn_replay_draft_kernel"]
    assert bench.source_digest("gdn_replay_nf_kernel") == d["gdn_replay_nf_kernel"]


def test_clock_summary_reads_samples_and_reasons(tmp_path):
    clk = bench.ClockSampler("0")
    clk.path = str(tmp_path / "clocks.csv")
    clk.proc = object()          # stands for a sampler that ran
    (tmp_path / "clocks.csv").write_text(
        "2070, 2070, 900.1, Not Active, Not Active, Not Active, Active\n"
        "2055, 2070, 1000.0, Not Active, Not Active, Not Active, Not Active\n"
        "[N/A], 2070, 0, Not Active, Not Active, Not Active, Not Active\n"
        "1980, 2070, 1100.0, Not Active, Active, Not Active, Not Active\n")
    s = clk.summary()
    assert s == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "samples": 3,
                 "reasons": ["hw_thermal_slowdown", "sw_power_cap"]}
    assert not os.path.exists(clk.path)


class _Props:
    L2_cache_size = 132 * 2**20


class _FakeTorch:
    class cuda:
        @staticmethod
        def get_device_properties(dev):
            return _Props


def test_small_states_rotate_over_layers_that_exceed_twice_l2():
    for batch in (1, 8, 16, 32, 64, 128, 256):
        state = batch * 128 * 64 * 128 * 4
        n = bench.rotation_layers(_FakeTorch, 0, state)
        assert n * state >= 2 * _Props.L2_cache_size
        assert (n - 1) * state < 2 * _Props.L2_cache_size
    assert bench.rotation_layers(_FakeTorch, 0, 256 * 128 * 64 * 128 * 4) == 1


def test_flush_split_follows_each_layers_own_step_count():
    # 3 layers round-robin, k = 4: launch j is its layer's (j // 3)-th step,
    # so the flush launches are j = 9, 10, 11 (and 21, 22, 23 ...)
    w = synth.WORKLOADS["mamba2_serving_b256"]
    w = synth.Mamba2Workload(**{**w.__dict__, "k": 4})
    warm, K = 2, 24
    per = [0.001] * K
    byts = [1e6] * K
    flush_j = {j for j in range(warm, warm + K) if (j // 3) % 4 == 3}
    for i in range(K):
        if warm + i in flush_j:
            per[i], byts[i] = 0.002, 3e6
    res = {"w": w, "per": per, "bytes": byts, "nf_kernel": "nf", "kernel": "fl", "layers": 3}
    out = bench.roofline_of(res, "replay", warm, 6000.0, "measured")
    assert out["split"]["flush"]["launches"] == len(flush_j) == 6
    assert out["split"]["flush"]["mean_us"] == pytest.approx(2.0)
    assert out["split"]["non_flush"]["mean_us"] == pytest.approx(1.0)
