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
from _gpu import TOL_F32, TOL_LOW, gdn_layer, gdn_run_steps, host, tile_err, vec_err

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


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_readcopy_matches_oracle(cuda_lib, fmt):
    w = GDN.replace(batch=3, heads=4, k=8, steps=30, read_fmt=fmt, scale=0.5)
    layer = gdn_layer(w, out_dtype="f32")
    o = gdn_run_steps(layer, w, 0, w.steps, out_dtype="f32")
    args = _inputs(w, 0, w.steps)
    o_rc, S_rc = oracle.gdn_readcopy(synth.gdn_state0(w), *args, w.k, fmt, scale=w.scale)
    assert vec_err(o, o_rc) < TOL_LOW
    o_ex, _ = oracle.gdn_recurrence(synth.gdn_state0(w), *args, scale=w.scale)
    flush = [t for t in range(w.steps) if (t + 1) % w.k == 0]
    assert vec_err(o[flush], o_ex[flush]) < TOL_F32
    # 24 tokens committed (3 windows): the checkpoint is the FP32 recurrence
    assert tile_err(_ckpt(layer, w), S_rc) < TOL_F32
    _copy_matches_quantiser(layer, w, fmt)
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("dv,dk", [(64, 64), (128, 64), (64, 128)])
def test_gdn_readcopy_tile_shapes(cuda_lib, dv, dk):
    w = GDN.replace(batch=2, heads=4, d_v=dv, d_k=dk, k=4, steps=10, read_fmt="fp8")
    layer = gdn_layer(w, out_dtype="f32")
    o = gdn_run_steps(layer, w, 0, w.steps, out_dtype="f32")
    args = _inputs(w, 0, w.steps)
    o_rc, S_rc = oracle.gdn_readcopy(synth.gdn_state0(w), *args, w.k, "fp8", scale=w.scale)
    assert vec_err(o, o_rc) < TOL_LOW
    assert tile_err(_ckpt(layer, w), S_rc) < TOL_F32
    _copy_matches_quantiser(layer, w, "fp8")


def test_gdn_readcopy_forced_flush_mid_window(cuda_lib):
    """An explicit flush after 5 tokens replays them too; the copy is then
    refreshed for every half."""
    w = GDN.replace(batch=2, heads=4, k=8, read_fmt="nvfp4")
    layer = gdn_layer(w, out_dtype="f32")
    o1 = gdn_run_steps(layer, w, 0, 5, out_dtype="f32")
    layer.flush()
    assert not layer.counts().any().item()
    _copy_matches_quantiser(layer, w, "nvfp4")
    o2 = gdn_run_steps(layer, w, 5, 15, out_dtype="f32")
    args = _inputs(w, 0, 20)
    o_rc, _ = oracle.gdn_readcopy(synth.gdn_state0(w), *args, w.k, "nvfp4", scale=w.scale, windows=[5, 8])
    assert vec_err(np.concatenate([o1, o2]), o_rc) < TOL_LOW
    layer.flush()
    _, S20 = oracle.gdn_recurrence(synth.gdn_state0(w), *args, scale=w.scale)
    assert tile_err(_ckpt(layer, w), S20) < TOL_F32
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_readcopy_serving_shape_sampled(cuda_lib, fmt):
    """Full serving batch over 40 steps (2 windows and a part); sequences are
    independent, so sampled ones are checked against the oracle."""
    w = GDN.replace(read_fmt=fmt)
    steps = 40
    layer = gdn_layer(w, out_dtype="f32")
    o = gdn_run_steps(layer, w, 0, steps, out_dtype="f32")
    sub = np.array([0, 77, 255])
    args = _inputs(w, 0, steps, sub)
    o_rc, S_rc = oracle.gdn_readcopy(synth.gdn_state0(w)[sub], *args, w.k, fmt, scale=w.scale)
    assert vec_err(o[:, sub], o_rc) < TOL_LOW
    assert tile_err(_ckpt(layer, w)[sub], S_rc) < TOL_F32
    assert layer.get_error()[0] == 0
