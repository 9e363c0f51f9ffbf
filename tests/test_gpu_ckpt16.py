"""FP16 checkpoint (Mamba-2 replay, bf16 inputs) on the GPU against the
oracle's FP16-checkpoint decode.

Tolerance: the kernels fold in FP32 and round to FP16, the oracle folds in
float64 and rounds; where the two folds fall on either side of an FP16
rounding midpoint the checkpoints differ by one FP16 ulp (2^-10 of the
value). One such element moves an output by at most 2^-10 |h_pn C_n|, well
under 2e-3 of the output vector's max-norm; the same bound holds per state
tile. Before the first flush both sides read the same FP16 values, so those
outputs are held to the FP32 tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import TOL_F32, TOL_LOW, gdn_layer, gdn_run_steps, host, m2_layer, m2_run_steps, tile_err, vec_err

pytestmark = pytest.mark.gpu

TOL_CK16 = 2e-3
SERVING = synth.WORKLOADS["mamba2_serving_b256"].replace(ckpt="f16")


def _ref(w, A, D, steps, fmt=None, windows=None, sub=slice(None)):
    ins = synth.mamba2_steps(w, 0, steps)
    args = [ins[k].values[:, sub] for k in ("x", "B", "C", "dt")]
    return oracle.m2_ckpt16(synth.mamba2_state0(w)[sub], A, D, *args, w.k, fmt=fmt, windows=windows)


def test_create_rounds_the_start_state_to_f16(cuda_lib):
    w = SERVING.replace(batch=2, heads=8, groups=1)
    layer, _, _ = m2_layer(w)
    ck = layer.ckpt()
    assert ck.dtype == torch.float16
    want = synth.mamba2_state0(w).astype(np.float16)
    np.testing.assert_array_equal(ck.cpu().numpy().view(np.uint16), want.view(np.uint16))


@pytest.mark.parametrize("fmt", [None, "fp8", "nvfp4"])
def test_ckpt16_decode_matches_oracle(cuda_lib, fmt):
    w = SERVING.replace(batch=3, heads=16, groups=2, k=8, steps=30, read_fmt=fmt or "none")
    layer, A, D = m2_layer(w, out_dtype="f32")
    y = m2_run_steps(layer, w, 0, w.steps, out_dtype="f32")
    y_ref, ck_ref = _ref(w, A, D, w.steps, fmt)
    if fmt is None:
        assert vec_err(y[: w.k - 1], y_ref[: w.k - 1]) < TOL_F32
        assert vec_err(y, y_ref) < TOL_CK16
    else:
        assert vec_err(y, y_ref) < TOL_LOW
    # flush-token outputs read the FP16 checkpoint itself
    flush = [t for t in range(w.steps) if (t + 1) % w.k == 0]
    y_plain, _ = _ref(w, A, D, w.steps)
    assert vec_err(y[flush], y_plain[flush]) < TOL_CK16
    assert tile_err(host(layer.ckpt()), ck_ref) < TOL_CK16
    assert layer.get_error()[0] == 0


def test_ckpt16_read_copy_leaves_the_checkpoint_alone(cuda_lib):
    """The FP16 checkpoint is bit-identical with and without a read copy."""
    w = SERVING.replace(batch=2, heads=8, groups=1, k=4, steps=9)
    a, _, _ = m2_layer(w, read_fmt="nvfp4")
    b, _, _ = m2_layer(w)
    m2_run_steps(a, w, 0, w.steps)
    m2_run_steps(b, w, 0, w.steps)
    assert torch.equal(a.ckpt(), b.ckpt())


def test_ckpt16_forced_flush_mid_window(cuda_lib):
    w = SERVING.replace(batch=2, heads=16, groups=2, k=8)
    layer, A, D = m2_layer(w, out_dtype="f32")
    y1 = m2_run_steps(layer, w, 0, 5, out_dtype="f32")
    layer.flush()
    assert not layer.counts().any().item()
    y2 = m2_run_steps(layer, w, 5, 19, out_dtype="f32")
    y_ref, _ = _ref(w, A, D, 24, windows=[5, 8, 8])
    assert vec_err(np.concatenate([y1, y2]), y_ref) < TOL_CK16
    layer.flush()
    _, ck_ref = _ref(w, A, D, 24, windows=[5, 8, 8, 3])
    assert tile_err(host(layer.ckpt()), ck_ref) < TOL_CK16


def test_ckpt16_serving_shape_sampled(cuda_lib):
    """Full serving batch over 48 steps (3 windows); sequences are
    independent, so a sampled subset is checked against the oracle."""
    w = SERVING
    steps = 48
    layer, A, D = m2_layer(w, out_dtype="f32")
    y = m2_run_steps(layer, w, 0, steps, out_dtype="f32")
    sub = np.array([0, 131, 255])
    y_ref, ck_ref = _ref(w, A, D, steps, sub=sub)
    assert vec_err(y[:, sub], y_ref) < TOL_CK16
    assert tile_err(host(layer.ckpt()[torch.from_numpy(sub).cuda()]), ck_ref) < TOL_CK16


# ----------------------------------------------------------------------------
# Gated DeltaNet with an FP16 checkpoint
# ----------------------------------------------------------------------------
GDN = synth.WORKLOADS["gdn_serving_b256"]


def _gdn_inputs(w, start, count, sub=slice(None)):
    ins = synth.gdn_steps(w, start, count)
    return [ins[k].values[:, sub] for k in ("q", "k", "v", "alpha", "beta")]


def _gdn_ck(layer, w, sub=slice(None)):
    return host(layer.ckpt()[sub]).reshape(-1, w.heads, w.d_v, w.d_k)


def test_gdn_create_rounds_the_start_state_to_f16(cuda_lib):
    w = GDN.replace(batch=2, heads=4)
    layer = gdn_layer(w, ckpt="f16")
    ck = layer.ckpt()
    assert ck.dtype == torch.float16
    want = synth.gdn_state0(w).astype(np.float16)
    np.testing.assert_array_equal(ck.cpu().numpy().reshape(want.shape).view(np.uint16), want.view(np.uint16))


def _gdn_check_windows(layer, w, windows, sub=slice(None), explicit=False):
    """Window by window, from the FP16 checkpoint the GPU stored: every output
    of the window is the recurrence continued from it (FP32 tolerance; the
    flush token's too), and the checkpoint the flush stores is the window's
    end state rounded to FP16 (TOL_CK16: a value whose FP32 and float64 folds
    fall on either side of an FP16 midpoint rounds one ulp apart)."""
    start, outs = 0, []
    for n in windows:
        ck = _gdn_ck(layer, w, sub)
        o = gdn_run_steps(layer, w, start, n, out_dtype="f32")
        args = _gdn_inputs(w, start, n, sub)
        o_ref, S_end = oracle.gdn_recurrence(ck, *args, scale=w.scale)
        assert vec_err(o[:, sub], o_ref) < TOL_F32
        if n < w.k and explicit:
            layer.flush()
        if n == w.k or explicit:
            assert tile_err(_gdn_ck(layer, w, sub), oracle.round_f16(S_end)) < TOL_CK16
        outs.append(o)
        start += n
    return np.concatenate(outs)


@pytest.mark.parametrize("dv,dk", [(128, 128), (64, 64), (128, 64)])
def test_gdn_ckpt16_window_by_window(cuda_lib, dv, dk):
    w = GDN.replace(batch=3, heads=4, d_v=dv, d_k=dk, k=8, scale=0.5)
    layer = gdn_layer(w, out_dtype="f32", ckpt="f16")
    o = _gdn_check_windows(layer, w, [8, 8, 8, 6])
    # the whole run against the oracle's FP16-checkpoint decode
    o_ref, ck_ref = oracle.gdn_ckpt16(synth.gdn_state0(w), *_gdn_inputs(w, 0, 30), w.k, scale=w.scale)
    assert vec_err(o[: w.k], o_ref[: w.k]) < TOL_F32
    assert vec_err(o, o_ref) < TOL_CK16
    layer.flush()
    _, ck_all = oracle.gdn_ckpt16(synth.gdn_state0(w), *_gdn_inputs(w, 0, 30), w.k, scale=w.scale,
                                  windows=[8, 8, 8, 6])
    assert tile_err(_gdn_ck(layer, w), ck_all) < TOL_CK16
    assert layer.get_error()[0] == 0


def test_gdn_ckpt16_forced_flush_mid_window(cuda_lib):
    w = GDN.replace(batch=2, heads=4, k=8)
    layer = gdn_layer(w, out_dtype="f32", ckpt="f16")
    _gdn_check_windows(layer, w, [5, 8, 7], explicit=True)
    assert not layer.counts().any().item()
    assert layer.get_error()[0] == 0


def test_gdn_ckpt16_serving_shape_sampled(cuda_lib):
    """The serving shape (B256, H32, 128 x 128) over 40 steps, sampled
    sequences window by window."""
    w = GDN
    layer = gdn_layer(w, out_dtype="f32", ckpt="f16")
    _gdn_check_windows(layer, w, [16, 16, 8], sub=np.array([0, 77, 255]))
    assert layer.get_error()[0] == 0
