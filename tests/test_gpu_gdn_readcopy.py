"""Gated DeltaNet read copies (FP8 E4M3, NVFP4; one copy tile per 64-row
half) on the GPU against the oracle's read-copy decode: non-flush outputs
read the copy, flush outputs and the checkpoint follow the FP32 recurrence
(the flush replays the window's records), and the copy the flush writes is
bit-identical to the standalone quantiser's copy of the new checkpoint."""
import numpy as np
import pytest
import torch

import hybrid_ssm_decode_gb300 as rssm
import oracle
import synth
from _gpu import TOL_F32, gdn_layer, gdn_run_steps, host, tile_err, vec_err

pytestmark = pytest.mark.gpu

GDN = synth.WORKLOADS["gdn_serving_b256"]


def _inputs(w, start, count, sub=slice(None)):
    ins = synth.gdn_steps(w, start, count)
    return [ins[k].values[:, sub] for k in ("q", "k", "v", "alpha", "beta")]


def _copy_matches_quantiser(layer, w, fmt):
    """The copy region equals rssm_quantize of the FP32 checkpoint's halves."""
    lay = layer.layout
    halves = w.batch * w.heads * (w.d_v // 64)
    src = layer.ckpt().contiguous()
    ws = layer.workspace
    f = rssm.READ_FMT[fmt]
    codes = torch.zeros(lay.rc_codes_bytes, dtype=torch.uint8, device="cuda")
    bsc = torch.zeros(max(lay.rc_bscale_bytes, 1), dtype=torch.uint8, device="cuda")
    ts = torch.zeros(halves, dtype=torch.float32, device="cuda")
    rssm.rssm_quantize(f, halves, 64, w.d_k, src, codes, bsc if fmt == "nvfp4" else None, ts)
    assert torch.equal(ws[lay.rc_codes:lay.rc_codes + lay.rc_codes_bytes], codes)
    assert torch.equal(ws[lay.rc_tscale:lay.rc_tscale + lay.rc_tscale_bytes].view(torch.float32), ts)
    if fmt == "nvfp4":
        assert torch.equal(ws[lay.rc_bscale:lay.rc_bscale + lay.rc_bscale_bytes], bsc)


def _ckpt(layer, w):
    return host(layer.ckpt()).reshape(w.batch, w.heads, w.d_v, w.d_k)


def _check_windows(layer, w, fmt, windows, sub=slice(None), explicit=False):
    """Window by window, from the FP32 checkpoint the GPU stored: every
    64-row half's copy is the oracle quantiser's copy of that half bit for
    bit, the window's outputs are the oracle's read-copy decode started from
    that checkpoint (FP32 tolerance; the k-th token is the flush token and
    reads the checkpoint itself), and the checkpoint the flush stores is the
    recurrence of the window. explicit: a window shorter than k ends in an
    explicit flush. Returns the outputs of all windows."""
    lay, ws = layer.layout, layer.workspace
    dv, dk = w.d_v, w.d_k
    start, outs = 0, []
    for n in windows:
        ck = host(layer.ckpt()[sub])
        halves = ck.reshape(-1, 64, dk).astype(np.float32)
        codes = ws[lay.rc_codes:lay.rc_codes + lay.rc_codes_bytes].view(w.batch, w.heads, dv, -1)[sub]
        ts = ws[lay.rc_tscale:lay.rc_tscale + lay.rc_tscale_bytes].view(torch.float32).view(w.batch, -1)[sub]
        ref = (oracle.quant_fp8 if fmt == "fp8" else oracle.quant_nvfp4)(halves)
        np.testing.assert_array_equal(codes.cpu().numpy().reshape(halves.shape[0], 64, -1), ref[0])
        np.testing.assert_array_equal(ts.cpu().numpy().reshape(-1), ref[-1])
        if fmt == "nvfp4":
            bsc = ws[lay.rc_bscale:lay.rc_bscale + lay.rc_bscale_bytes].view(w.batch, w.heads, dv, dk // 16)[sub]
            np.testing.assert_array_equal(bsc.cpu().numpy().reshape(halves.shape[0], 64, -1), ref[1])
        o = gdn_run_steps(layer, w, start, n, out_dtype="f32")
        args = _inputs(w, start, n, sub)
        commit = n == w.k or explicit
        o_ref, _ = oracle.gdn_readcopy(ck, *args, w.k, fmt, scale=w.scale, windows=[n] if commit else [])
        assert vec_err(o[:, sub], o_ref) < TOL_F32
        if n < w.k and explicit:
            layer.flush()
            assert not layer.counts().any().item()
        if commit:
            _, S_end = oracle.gdn_recurrence(ck, *args, scale=w.scale)
            assert tile_err(_ckpt(layer, w)[sub], S_end) < TOL_F32
        outs.append(o)
        start += n
    return np.concatenate(outs)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_readcopy_matches_oracle(cuda_lib, fmt):
    w = GDN.replace(batch=3, heads=4, k=8, steps=30, read_fmt=fmt, scale=0.5)
    layer = gdn_layer(w, out_dtype="f32")
    o = _check_windows(layer, w, fmt, [8, 8, 8, 6])
    args = _inputs(w, 0, w.steps)
    o_ex, S_ex = oracle.gdn_recurrence(synth.gdn_state0(w), *args, scale=w.scale)
    # flush outputs are the exact recurrence's (the others carry the copy's
    # quantisation error)
    flush = [t for t in range(w.steps) if (t + 1) % w.k == 0]
    assert vec_err(o[flush], o_ex[flush]) < TOL_F32
    _copy_matches_quantiser(layer, w, fmt)
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("dv,dk", [(64, 64), (128, 64), (64, 128)])
def test_gdn_readcopy_tile_shapes(cuda_lib, dv, dk):
    w = GDN.replace(batch=2, heads=4, d_v=dv, d_k=dk, k=4, steps=10, read_fmt="fp8")
    layer = gdn_layer(w, out_dtype="f32")
    _check_windows(layer, w, "fp8", [4, 4, 2])
    _copy_matches_quantiser(layer, w, "fp8")


def test_gdn_readcopy_forced_flush_mid_window(cuda_lib):
    """An explicit flush after 5 tokens replays them too; the copy is then
    refreshed for every half, and after the last explicit flush the
    checkpoint is the exact recurrence of all 20 tokens."""
    w = GDN.replace(batch=2, heads=4, k=8, read_fmt="nvfp4")
    layer = gdn_layer(w, out_dtype="f32")
    _check_windows(layer, w, "nvfp4", [5, 8, 7], explicit=True)
    _copy_matches_quantiser(layer, w, "nvfp4")
    args = _inputs(w, 0, 20)
    _, S20 = oracle.gdn_recurrence(synth.gdn_state0(w), *args, scale=w.scale)
    assert tile_err(_ckpt(layer, w), S20) < TOL_F32
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_readcopy_serving_shape_sampled(cuda_lib, fmt):
    """Full serving batch over 40 steps (2 windows and a part); sequences are
    independent, so sampled ones are checked window by window."""
    w = GDN.replace(read_fmt=fmt)
    layer = gdn_layer(w, out_dtype="f32")
    _check_windows(layer, w, fmt, [16, 16, 8], sub=np.array([0, 77, 255]))
    assert layer.get_error()[0] == 0
