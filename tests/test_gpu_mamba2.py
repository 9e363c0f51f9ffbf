"""Mamba-2 replay decode and the conventional baseline on the GPU, against
the float64 oracle (the per-token recurrence)."""
import numpy as np
import pytest
import torch

import hybrid_ssm_decode_gb300 as rssm
import oracle
import synth
from _gpu import (TOL_F32, TOL_LOW, dev, gdn_layer, host, m2_layer, m2_out, m2_run_steps,
                  tile_err, vec_err)

pytestmark = pytest.mark.gpu

SMALL = synth.WORKLOADS["mamba2_fp32_b4"]                 # B4 H8 P64 N64 G1, FP32
SERVING = synth.WORKLOADS["mamba2_serving_b256"]          # B256 H128 P64 N128 G8, bf16


def _oracle(w, start_state, start, count, subset=None):
    A, D = synth.mamba2_params(w)
    ins = synth.mamba2_steps(w, start, count)
    sl = slice(None) if subset is None else subset
    x, Bm, C, dt = (ins[k].values[:, sl] for k in ("x", "B", "C", "dt"))
    return oracle.m2_recurrence(start_state[sl], A, D, x, Bm, C, dt)


def test_small_fp32_replay_matches_oracle(cuda_lib):
    w = SMALL
    layer, A, D = m2_layer(w)
    y = m2_run_steps(layer, w, 0, w.steps)
    y_ref, h_ref = _oracle(w, synth.mamba2_state0(w), 0, w.steps)
    assert vec_err(y, y_ref) < TOL_F32
    # 64 steps = 4 windows of k=16: the checkpoint is the full state, counts 0
    assert tile_err(host(layer.ckpt()), h_ref) < TOL_F32
    assert not layer.counts().any().item()
    assert layer.get_error()[0] == 0


def test_small_fp32_conventional_matches_oracle(cuda_lib):
    w = SMALL
    layer, A, D = m2_layer(w, mode="conventional")
    y = m2_run_steps(layer, w, 0, 24)
    y_ref, h_ref = _oracle(w, synth.mamba2_state0(w), 0, 24)
    assert vec_err(y, y_ref) < TOL_F32
    assert tile_err(host(layer.ckpt()), h_ref) < TOL_F32


def test_counts_and_checkpoint_every_step(cuda_lib):
    """Non-flush steps store no state; the flush step writes the state after k
    tokens. Counts follow (t+1) mod k exactly."""
    w = SMALL.replace(k=5, steps=13)
    layer, A, D = m2_layer(w)
    h0 = synth.mamba2_state0(w)
    ckpt_prev = layer.ckpt().clone()
    for t in range(w.steps):
        m2_run_steps(layer, w, t, 1)
        counts = layer.counts().cpu().numpy()
        assert np.all(counts == (t + 1) % w.k)
        if (t + 1) % w.k:
            assert torch.equal(layer.ckpt(), ckpt_prev)       # no state store
        else:
            _, h_ref = _oracle(w, h0, 0, t + 1)
            assert tile_err(host(layer.ckpt()), h_ref) < TOL_F32
            ckpt_prev = layer.ckpt().clone()


def test_k1_is_the_conventional_step(cuda_lib):
    w = SMALL.replace(k=1, steps=10)
    rep, _, _ = m2_layer(w)
    conv, _, _ = m2_layer(w, mode="conventional")
    y_rep = m2_run_steps(rep, w, 0, 10)
    y_conv = m2_run_steps(conv, w, 0, 10)
    assert vec_err(y_rep, y_conv) < 1e-5
    assert tile_err(host(rep.ckpt()), host(conv.ckpt())) < 1e-5


@pytest.mark.parametrize("k", [4, 8, 16, 32])
def test_k_sweep_bf16_inputs(cuda_lib, k):
    """Serving-shaped heads at a small batch; FP32 outputs isolate the
    kernel's arithmetic (1e-4), bf16 outputs add output rounding (2e-2)."""
    w = SERVING.replace(batch=2, heads=16, groups=2, k=k, steps=k + 7)
    for out, tol in (("f32", TOL_F32), ("bf16", TOL_LOW)):
        layer, A, D = m2_layer(w, out_dtype=out)
        y = m2_run_steps(layer, w, 0, w.steps, out_dtype=out)
        y_ref, h_ref = _oracle(w, synth.mamba2_state0(w), 0, w.steps)
        assert vec_err(y, y_ref) < tol
    layer.flush()
    assert tile_err(host(layer.ckpt()), h_ref) < TOL_F32


@pytest.mark.parametrize("P,N", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_tile_shapes(cuda_lib, P, N):
    w = SERVING.replace(batch=3, heads=4, groups=2, head_dim=P, state_dim=N, k=6, steps=14,
                        dtype="f32")
    layer, A, D = m2_layer(w)
    y = m2_run_steps(layer, w, 0, w.steps)
    y_ref, h_ref = _oracle(w, synth.mamba2_state0(w), 0, w.steps)
    assert vec_err(y, y_ref) < TOL_F32
    conv, _, _ = m2_layer(w, mode="conventional")
    assert vec_err(m2_run_steps(conv, w, 0, w.steps), y_ref) < TOL_F32


def test_forced_flush_mid_window_then_continue(cuda_lib):
    w = SMALL.replace(steps=30)
    layer, A, D = m2_layer(w)
    m2_run_steps(layer, w, 0, 5)
    layer.flush()
    assert not layer.counts().any().item()
    h0 = synth.mamba2_state0(w)
    _, h5 = _oracle(w, h0, 0, 5)
    assert tile_err(host(layer.ckpt()), h5) < TOL_F32
    y = m2_run_steps(layer, w, 5, 25)
    y_ref, _ = _oracle(w, h0, 0, 30)
    assert vec_err(y, y_ref[5:]) < TOL_F32


def test_deterministic(cuda_lib):
    w = SMALL.replace(steps=20)
    runs = []
    for _ in range(2):
        layer, _, _ = m2_layer(w)
        runs.append((m2_run_steps(layer, w, 0, 20), layer.ckpt().clone()))
    np.testing.assert_array_equal(runs[0][0], runs[1][0])
    assert torch.equal(runs[0][1], runs[1][1])


def test_tiny_and_zero_state(cuda_lib):
    w = SMALL.replace(batch=1, heads=1, groups=1, steps=7, k=3)
    layer, A, D = m2_layer(w, state0=False)
    y = m2_run_steps(layer, w, 0, 7)
    y_ref, _ = _oracle(w, np.zeros((1, 1, 64, 64), np.float32), 0, 7)
    assert vec_err(y, y_ref) < TOL_F32


def test_serving_shape_sampled_parity(cuda_lib):
    """The full serving layer (B=256, H=128, P=64, N=128, G=8, bf16, ~1 GiB
    checkpoint) in the launch configuration the benchmark times, across a
    flush; sequences are independent, so a sampled subset is checked exactly
    against the oracle."""
    w = SERVING
    steps = 20
    layer, A, D = m2_layer(w, out_dtype="f32")
    y = m2_run_steps(layer, w, 0, steps, out_dtype="f32")
    subset = np.array([0, 1, 97, 128, 255])
    y_ref, h_ref = _oracle(w, synth.mamba2_state0(w), 0, steps, subset=subset)
    assert vec_err(y[:, subset], y_ref) < TOL_F32
    layer.flush()
    assert tile_err(host(layer.ckpt()[torch.from_numpy(subset).cuda()]), h_ref) < TOL_F32
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("batch", [1, 8, 16])
def test_small_batch_serving_heads_across_a_flush(cuda_lib, batch):
    """The serving layer's heads at small batches, where the direct one-block-
    per-tile kernels run (one wave at batch 1, several at 8 and 16): the
    outputs of 20 steps, and the checkpoint that the 16th step's fold wrote,
    against the oracle on sampled sequences."""
    w = SERVING.replace(batch=batch)
    layer, A, D = m2_layer(w, out_dtype="f32")
    sub = np.array(sorted({0, batch // 2, batch - 1}))
    h0 = synth.mamba2_state0(w)
    y = m2_run_steps(layer, w, 0, w.k, out_dtype="f32")
    y_ref, h_ref = _oracle(w, h0, 0, w.k, subset=sub)
    assert vec_err(y[:, sub], y_ref) < TOL_F32
    assert not layer.counts().any().item()
    assert tile_err(host(layer.ckpt()[torch.from_numpy(sub).cuda()]), h_ref) < TOL_F32
    y2 = m2_run_steps(layer, w, w.k, 4, out_dtype="f32")
    y2_ref, _ = _oracle(w, h0, 0, w.k + 4, subset=sub)
    assert vec_err(y2[:, sub], y2_ref[w.k:]) < TOL_F32
    assert layer.get_error()[0] == 0


def test_lean_step_reports_a_tile_due_to_flush(cuda_lib):
    """While the handle knows every count is below k - 1, steps run the
    non-flush kernel. A tile whose count was set to k - 1 behind the handle's
    back is reported (RSSM_DEV_COUNT_RANGE) and left unchanged; every other
    tile steps as usual."""
    w = SMALL.replace(k=8)
    layer, A, D = m2_layer(w)
    m2_run_steps(layer, w, 0, 2)
    layer.counts()[0, 1] = w.k - 1
    ck = layer.ckpt().clone()
    st = synth.mamba2_steps(w, 2, 1)
    y = m2_out(w).fill_(float("nan"))
    layer.decode_step(y, 1, x=dev(st["x"][0]), Bm=dev(st["B"][0]), C=dev(st["C"][0]), dt=dev(st["dt"][0]))
    err = layer.get_error()
    assert err == (rssm.RSSM_DEV_COUNT_RANGE, 1, 1, w.k - 1)
    bad = torch.zeros(w.batch, w.heads, dtype=torch.bool, device="cuda")
    bad[0, 1] = True
    assert bool(torch.isnan(y[:, 0][bad]).all()) and not bool(torch.isnan(y[:, 0][~bad]).any())
    assert layer.counts()[0, 1].item() == w.k - 1
    assert bool((layer.counts()[~bad] == 3).all())
    assert torch.equal(layer.ckpt(), ck)
    y_ref, _ = _oracle(w, synth.mamba2_state0(w), 0, 3)
    assert vec_err(host(y[:, 0])[1:], y_ref[-1][1:]) < TOL_F32
