"""The seeded input generators: deterministic, subset-consistent, and with
the stated distributions."""
import numpy as np

import synth


def test_deterministic_and_keyed():
    w = synth.WORKLOADS["mamba2_fp32_b4"]
    a, b = synth.mamba2_step(w, 3), synth.mamba2_step(w, 3)
    for key in a:
        np.testing.assert_array_equal(a[key].raw, b[key].raw)
    c = synth.mamba2_step(w, 4)
    assert not np.array_equal(a["x"].raw, c["x"].raw)
    assert not np.array_equal(a["B"].raw, a["C"].raw)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3], np.float32)
    bits = synth.bf16_round(x)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back[0] == 1.0
    assert back[1] == 1.0                 # tie -> even mantissa
    assert back[2] == 1.0 + 2 ** -6       # tie -> even (rounds up)
    assert back[3] == -2.5
    assert abs(back[4] - 3.0e-3) <= 3.0e-3 * 2 ** -8


def test_bf16_values_match_raw():
    w = synth.WORKLOADS["mamba2_serving_b256"].replace(batch=2, heads=16)
    s = synth.mamba2_step(w, 0)
    raw = (s["x"].raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(raw, s["x"].values)


def test_distributions():
    w = synth.WORKLOADS["mamba2_serving_b256"].replace(batch=16)
    s = synth.mamba2_step(w, 0)
    A, D = synth.mamba2_params(w)
    assert np.all(A <= -1.0) and np.all(A >= -16.0)
    assert abs(s["x"].values.std() - 1.0) < 0.02
    assert abs(s["B"].values.std() * np.sqrt(w.state_dim) - 1.0) < 0.05
    assert np.all(s["dt"].values > 0)
    g = synth.gdn_step(synth.WORKLOADS["gdn_serving_b256"].replace(batch=4), 0)
    nk = np.linalg.norm(g["k"].values, axis=-1)
    assert np.all(np.abs(nk - 1.0) < 1e-2)      # L2-normalised, then bf16-rounded
    assert np.all((g["alpha"].values > 0) & (g["alpha"].values < 1))
    assert np.all((g["beta"].values > 0) & (g["beta"].values < 1))


def test_acceptance_truncated_geometric():
    a = synth.acceptance(batch=512, rounds=64, draft=4, p=0.7)
    assert a.min() >= 0 and a.max() <= 4
    expected_mean = sum(0.7 ** j for j in range(1, 5))   # E[a] = p + p^2 + p^3 + p^4
    assert abs(a.mean() - expected_mean) < 0.03
    assert abs(np.mean(a == 4) - 0.7 ** 4) < 0.02
    assert abs(np.mean(a == 0) - 0.3) < 0.02


def test_slow_decay_workload_scales_only_dt():
    base = synth.WORKLOADS["mamba2_serving_b256"].replace(batch=2, dtype="f32")
    slow = synth.WORKLOADS["mamba2_slowdecay_b256"].replace(batch=2, dtype="f32")
    a, b = synth.mamba2_step(base, 5), synth.mamba2_step(slow, 5)
    for key in ("x", "B", "C"):
        np.testing.assert_array_equal(a[key].raw, b[key].raw)
    np.testing.assert_allclose(b["dt"].values, 0.05 * a["dt"].values, rtol=1e-6)
    np.testing.assert_array_equal(synth.mamba2_state0(base), synth.mamba2_state0(slow))


def test_checkpoint_and_copy_workloads_share_the_inputs():
    """The precision variants of the serving layer differ only in storage, so
    their inputs and start states are the serving layer's."""
    base = synth.WORKLOADS["mamba2_serving_b256"].replace(batch=2)
    for name in ("mamba2_fp8_b256", "mamba2_nvfp4_b256", "mamba2_f16ckpt_b256", "mamba2_fp8ckpt_b256",
                 "mamba2_fp8ckpt_nvfp4_b256", "mamba2_nvfp4ckpt_b256", "mamba2_f16ckpt_nvfp4_b256"):
        w = synth.WORKLOADS[name].replace(batch=2)
        a, b = synth.mamba2_step(base, 3), synth.mamba2_step(w, 3)
        for key in a:
            np.testing.assert_array_equal(a[key].raw, b[key].raw)
        np.testing.assert_array_equal(synth.mamba2_state0(base), synth.mamba2_state0(w))
