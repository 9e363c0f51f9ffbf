"""Mamba-2 replay with the checkpoint in a read-copy tile format (FP8, or
NVFP4; an FP8 checkpoint may also be read through an NVFP4 copy) on the GPU,
against the oracle's low-precision-checkpoint decode.

Tolerance. The start state is quantised by the same rules on both sides, so
its codes match bit for bit and the first window's outputs are held to the
FP32 tolerance. Later windows fold in FP32 on the GPU and in float64 in the
oracle; where the two folds fall on either side of a code midpoint, a stored
element moves by one code step (up to 1/8 of it for FP8), which is rare (a
float32 rounding against a 2^-3 step) and stays within the low-precision
output tolerance; the stored codes must agree almost everywhere.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import TOL_F32, TOL_LOW, host, m2_layer, m2_run_steps, vec_err

pytestmark = pytest.mark.gpu

SERVING = synth.WORKLOADS["mamba2_serving_b256"]


def _ref(w, A, D, steps, fmt=None, windows=None, sub=slice(None)):
    ins = synth.mamba2_steps(w, 0, steps)
    args = [ins[k].values[:, sub] for k in ("x", "B", "C", "dt")]
    return oracle.m2_ckpt_lowp(synth.mamba2_state0(w)[sub], A, D, *args, w.k, w.ckpt, fmt=fmt, windows=windows)


def _stored(layer, w):
    """The GPU checkpoint decoded: (codes, block scales, tile scales) -> values."""
    codes = layer.ckpt().cpu().numpy().reshape(w.batch * w.heads, w.head_dim, -1)
    lay = layer.layout
    ts = layer.workspace[lay.ckpt_tscale:lay.ckpt_tscale + lay.ckpt_tscale_bytes].view(torch.float32).cpu().numpy()
    if w.ckpt == "fp8":
        vals = oracle.dequant_fp8(codes, ts)
    else:
        bsc = layer.workspace[lay.ckpt_bscale:lay.ckpt_bscale + lay.ckpt_bscale_bytes].cpu().numpy()
        vals = oracle.dequant_nvfp4(codes, bsc.reshape(w.batch * w.heads, w.head_dim, -1), ts)
    return codes, vals.reshape(w.batch, w.heads, w.head_dim, w.state_dim)


@pytest.mark.parametrize("store", ["fp8", "nvfp4"])
def test_create_stores_the_quantised_start_state(cuda_lib, store):
    w = SERVING.replace(batch=2, heads=8, groups=1, ckpt=store)
    layer, _, _ = m2_layer(w)
    codes, vals = _stored(layer, w)
    tiles = synth.mamba2_state0(w).reshape(-1, w.head_dim, w.state_dim).astype(np.float32)
    ref = oracle.quant_fp8(tiles) if store == "fp8" else oracle.quant_nvfp4(tiles)
    np.testing.assert_array_equal(codes, ref[0])
    np.testing.assert_array_equal(vals, oracle.store_tiles(synth.mamba2_state0(w), store))


@pytest.mark.parametrize("store,fmt", [("fp8", None), ("nvfp4", None)])
def test_tile_checkpoint_decode_matches_oracle(cuda_lib, store, fmt):
    w = SERVING.replace(batch=3, heads=16, groups=2, k=8, steps=30, ckpt=store, read_fmt=fmt or "none")
    layer, A, D = m2_layer(w, out_dtype="f32")
    y = m2_run_steps(layer, w, 0, w.steps, out_dtype="f32")
    y_ref, ck_ref = _ref(w, A, D, w.steps, fmt)
    if fmt is None:
        assert vec_err(y[: w.k - 1], y_ref[: w.k - 1]) < TOL_F32
    assert vec_err(y, y_ref) < TOL_LOW
    _, vals = _stored(layer, w)
    tmax = np.max(np.abs(ck_ref), axis=(2, 3), keepdims=True)
    assert np.mean(np.abs(vals - ck_ref) > 1e-5 * tmax) < 1e-3
    assert layer.get_error()[0] == 0


def _rc_copy(layer, w):
    lay = layer.layout
    ws = layer.workspace
    codes = ws[lay.rc_codes:lay.rc_codes + lay.rc_codes_bytes].cpu().numpy().reshape(w.batch * w.heads, w.head_dim, -1)
    bsc = ws[lay.rc_bscale:lay.rc_bscale + lay.rc_bscale_bytes].cpu().numpy().reshape(w.batch * w.heads, w.head_dim, -1)
    ts = ws[lay.rc_tscale:lay.rc_tscale + lay.rc_tscale_bytes].view(torch.float32).cpu().numpy()
    return codes, bsc, ts


@pytest.mark.parametrize("windows", [[8, 8, 8], [5, 8, 8]])
def test_fp8_checkpoint_with_nvfp4_copy_window_by_window(cuda_lib, windows):
    """An NVFP4 copy of an FP8 checkpoint quantises values on the FP8 grid,
    many of which sit exactly on NVFP4 rounding midpoints; a one-ulp change of
    the FP8 tile scale (the FP32 and float64 folds can pick neighbouring
    scales) then moves those codes. So each window is checked against the
    oracle started from the checkpoint the GPU stored: the copy is the NVFP4
    quantisation of its decoded values bit for bit, the outputs are the read-
    copy decode from it (FP32 tolerance), and the next stored checkpoint is
    the oracle's store of the fold almost everywhere. A window shorter than k
    ends in an explicit flush."""
    w = SERVING.replace(batch=2, heads=16, groups=2, k=8, ckpt="fp8", read_fmt="nvfp4")
    layer, A, D = m2_layer(w, out_dtype="f32")
    start = 0
    for n in windows:
        _, ck = _stored(layer, w)
        codes, bsc, ts = _rc_copy(layer, w)
        ref = oracle.quant_nvfp4(ck.reshape(-1, w.head_dim, w.state_dim).astype(np.float32))
        np.testing.assert_array_equal(codes, ref[0])
        np.testing.assert_array_equal(bsc, ref[1])
        np.testing.assert_array_equal(ts, ref[2])
        y, ins = m2_run_steps(layer, w, start, n, out_dtype="f32", return_inputs=True)
        if n < w.k:
            layer.flush()
        args = [ins[k].values for k in ("x", "B", "C", "dt")]
        y_ref = oracle.m2_readcopy(ck, A, D, *args, w.k, "nvfp4")
        assert vec_err(y, y_ref) < TOL_F32
        _, h_end = oracle.m2_recurrence(ck, A, D, *args)
        _, ck_new = _stored(layer, w)
        want = oracle.store_tiles(h_end, "fp8")
        tmax = np.max(np.abs(want), axis=(2, 3), keepdims=True)
        assert np.mean(np.abs(ck_new - want) > 1e-5 * tmax) < 1e-3
        start += n
    assert not layer.counts().any().item()
    assert layer.get_error()[0] == 0


def test_tile_checkpoint_forced_flush_mid_window(cuda_lib):
    w = SERVING.replace(batch=2, heads=16, groups=2, k=8, ckpt="nvfp4")
    layer, A, D = m2_layer(w, out_dtype="f32")
    y1 = m2_run_steps(layer, w, 0, 5, out_dtype="f32")
    layer.flush()
    assert not layer.counts().any().item()
    y2 = m2_run_steps(layer, w, 5, 19, out_dtype="f32")
    y_ref, _ = _ref(w, A, D, 24, windows=[5, 8, 8])
    assert vec_err(np.concatenate([y1, y2]), y_ref) < TOL_LOW
    layer.flush()
    _, ck_ref = _ref(w, A, D, 24, windows=[5, 8, 8, 3])
    _, vals = _stored(layer, w)
    tmax = np.max(np.abs(ck_ref), axis=(2, 3), keepdims=True)
    assert np.mean(np.abs(vals - ck_ref) > 1e-5 * tmax) < 1e-3


def test_fp8_checkpoint_serving_shape_sampled(cuda_lib):
    w = SERVING.replace(ckpt="fp8")
    steps = 48
    layer, A, D = m2_layer(w, out_dtype="f32")
    y = m2_run_steps(layer, w, 0, steps, out_dtype="f32")
    sub = np.array([0, 131, 255])
    y_ref, _ = _ref(w, A, D, steps, sub=sub)
    assert vec_err(y[:, sub], y_ref) < TOL_LOW
    assert layer.get_error()[0] == 0
