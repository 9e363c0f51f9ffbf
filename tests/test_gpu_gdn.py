"""Gated DeltaNet replay decode (WY/UT window form) and the conventional
baseline on the GPU, against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import TOL_F32, TOL_LOW, gdn_layer, gdn_run_steps, host, tile_err, vec_err

pytestmark = pytest.mark.gpu

GDN = synth.WORKLOADS["gdn_serving_b256"]


def _oracle(w, start, count, subset=slice(None)):
    ins = synth.gdn_steps(w, start, count)
    a = [ins[k].values[:, subset] for k in ("q", "k", "v", "alpha", "beta")]
    return oracle.gdn_recurrence(synth.gdn_state0(w)[subset], *a, scale=w.scale)


@pytest.mark.parametrize("dv,dk", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_replay_matches_oracle(cuda_lib, dv, dk):
    w = GDN.replace(batch=3, heads=4, d_v=dv, d_k=dk, k=16, steps=40, dtype="f32")
    layer = gdn_layer(w)
    o = gdn_run_steps(layer, w, 0, w.steps)
    o_ref, S_ref = _oracle(w, 0, w.steps)
    assert vec_err(o, o_ref) < TOL_F32
    assert layer.counts()[0, 0].item() == w.steps % w.k
    layer.flush()
    assert tile_err(host(layer.ckpt()), S_ref) < TOL_F32


def test_conventional_matches_oracle(cuda_lib):
    w = GDN.replace(batch=3, heads=4, steps=12, dtype="f32")
    layer = gdn_layer(w, mode="conventional")
    o = gdn_run_steps(layer, w, 0, w.steps)
    o_ref, S_ref = _oracle(w, 0, w.steps)
    assert vec_err(o, o_ref) < TOL_F32
    assert tile_err(host(layer.ckpt()), S_ref) < TOL_F32


def test_k1_is_the_conventional_step(cuda_lib):
    w = GDN.replace(batch=2, heads=4, steps=8, dtype="f32", k=1)
    rep = gdn_layer(w)
    conv = gdn_layer(w, mode="conventional")
    assert vec_err(gdn_run_steps(rep, w, 0, 8), gdn_run_steps(conv, w, 0, 8)) < 1e-5
    assert tile_err(host(rep.ckpt()), host(conv.ckpt())) < 1e-5


@pytest.mark.parametrize("k", [4, 16, 32])
def test_bf16_inputs_k_sweep(cuda_lib, k):
    w = GDN.replace(batch=2, heads=8, k=k, steps=k + 5, scale=0.5)
    for out, tol in (("f32", TOL_F32), ("bf16", TOL_LOW)):
        layer = gdn_layer(w, out_dtype=out)
        o = gdn_run_steps(layer, w, 0, w.steps, out_dtype=out)
        o_ref, S_ref = _oracle(w, 0, w.steps)
        assert vec_err(o, o_ref) < tol


def test_flush_window_state(cuda_lib):
    """After exactly k tokens the checkpoint equals the state after k
    conventional steps; non-flush steps leave it untouched."""
    w = GDN.replace(batch=2, heads=4, steps=16, dtype="f32", k=16)
    layer = gdn_layer(w)
    s0 = layer.ckpt().clone()
    gdn_run_steps(layer, w, 0, 15)
    assert torch.equal(layer.ckpt(), s0)
    gdn_run_steps(layer, w, 15, 1)
    _, S_ref = _oracle(w, 0, 16)
    assert tile_err(host(layer.ckpt()), S_ref) < TOL_F32
    assert not layer.counts().any().item()


def test_serving_shape_sampled(cuda_lib):
    """B=256, H=32, d_k=d_v=128, bf16 q/k/v, across a flush; sampled sequences."""
    w = GDN
    steps = 20
    layer = gdn_layer(w, out_dtype="f32")
    o = gdn_run_steps(layer, w, 0, steps, out_dtype="f32")
    sub = np.array([0, 130, 255])
    o_ref, S_ref = _oracle(w, 0, steps, subset=sub)
    assert vec_err(o[:, sub], o_ref) < TOL_F32
    layer.flush()
    assert tile_err(host(layer.ckpt()[torch.from_numpy(sub).cuda()]), S_ref) < TOL_F32
