"""Low-precision read copies (FP8 E4M3, NVFP4): the writer is bit-exact with
the oracle's quantiser on the same FP32 tiles, the decode outputs match the
oracle's read-copy emulation, and the FP32 recurrence is untouched."""
import numpy as np
import pytest
import torch

import hybrid_ssm_decode_gb300 as rssm
import oracle
import synth
from _gpu import TOL_F32, TOL_LOW, dev, host, m2_layer, m2_run_steps, tile_err, vec_err

pytestmark = pytest.mark.gpu

SERVING = synth.WORKLOADS["mamba2_serving_b256"]


def _tiles(seed, n, rows, cols):
    rng = np.random.default_rng(seed)
    t = rng.standard_normal((n, rows, cols)) * 10.0 ** rng.integers(-6, 3, (n, 1, 1))
    t = t.astype(np.float32)
    t[0] = 0.0                                    # all-zero tile
    t[1, :, :16] = 0.0                            # zero blocks
    t[2] *= np.float32(1e-30)                     # block scales underflow
    return t


@pytest.mark.parametrize("rows,cols", [(64, 128), (64, 64), (128, 128)])
def test_quantize_bit_exact(cuda_lib, rows, cols):
    t = _tiles(rows + cols, 40, rows, cols)
    src = torch.from_numpy(t).cuda()
    n = t.shape[0]
    # FP8
    codes = torch.zeros((n, rows, cols), dtype=torch.uint8, device="cuda")
    ts = torch.zeros(n, dtype=torch.float32, device="cuda")
    rssm.rssm_quantize(rssm.RSSM_READ_FP8, n, rows, cols, src, codes, None, ts)
    c_ref, s_ref = oracle.quant_fp8(t)
    np.testing.assert_array_equal(ts.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)
    # NVFP4
    codes = torch.zeros((n, rows, cols // 2), dtype=torch.uint8, device="cuda")
    bsc = torch.zeros((n, rows, cols // 16), dtype=torch.uint8, device="cuda")
    rssm.rssm_quantize(rssm.RSSM_READ_NVFP4, n, rows, cols, src, codes, bsc, ts)
    c_ref, b_ref, s_ref = oracle.quant_nvfp4(t)
    np.testing.assert_array_equal(ts.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(bsc.cpu().numpy(), b_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_readcopy_decode_matches_oracle_emulation(cuda_lib, fmt):
    w = SERVING.replace(batch=3, heads=16, groups=2, k=8, steps=30, read_fmt=fmt)
    layer, A, D = m2_layer(w, out_dtype="f32")
    y = m2_run_steps(layer, w, 0, w.steps, out_dtype="f32")
    ins = synth.mamba2_steps(w, 0, w.steps)
    args = [ins[k].values for k in ("x", "B", "C", "dt")]
    y_rc = oracle.m2_readcopy(synth.mamba2_state0(w), A, D, *args, w.k, fmt)
    assert vec_err(y, y_rc) < TOL_LOW
    # flush-step outputs read the FP32 checkpoint
    flush = [t for t in range(w.steps) if (t + 1) % w.k == 0]
    y_ex, _ = oracle.m2_recurrence(synth.mamba2_state0(w), A, D, *args)
    assert vec_err(y[flush], y_ex[flush]) < TOL_F32


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_recurrence_unaffected_and_fused_writer_consistent(cuda_lib, fmt):
    """The FP32 checkpoint is bit-identical with and without a read copy, and
    the copy written by the fused flush equals the standalone writer's."""
    w = SERVING.replace(batch=2, heads=8, groups=1, k=4, steps=9, read_fmt=fmt)
    with_rc, _, _ = m2_layer(w)
    without, _, _ = m2_layer(w, read_fmt="none")
    m2_run_steps(with_rc, w, 0, w.steps)
    m2_run_steps(without, w, 0, w.steps)
    assert torch.equal(with_rc.ckpt(), without.ckpt())
    tiles = w.batch * w.heads
    P, N = w.head_dim, w.state_dim
    f = rssm.READ_FMT[fmt]
    codes = torch.zeros(with_rc.layout.rc_codes_bytes, dtype=torch.uint8, device="cuda")
    bsc = torch.zeros(max(with_rc.layout.rc_bscale_bytes, 1), dtype=torch.uint8, device="cuda")
    ts = torch.zeros(tiles, dtype=torch.float32, device="cuda")
    rssm.rssm_quantize(f, tiles, P, N, with_rc.ckpt(), codes, bsc, ts)
    lay = with_rc.layout
    ws = with_rc.workspace
    assert torch.equal(ws[lay.rc_codes:lay.rc_codes + lay.rc_codes_bytes], codes)
    assert torch.equal(ws[lay.rc_tscale:lay.rc_tscale + lay.rc_tscale_bytes].view(torch.float32), ts)
    if fmt == "nvfp4":
        assert torch.equal(ws[lay.rc_bscale:lay.rc_bscale + lay.rc_bscale_bytes], bsc)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_readcopy_serving_shape_sampled(cuda_lib, fmt):
    """Full serving batch with a read copy over 48 steps (3 windows),
    sampled sequences against the emulation."""
    w = SERVING.replace(read_fmt=fmt)
    steps = 48
    layer, A, D = m2_layer(w)
    y = m2_run_steps(layer, w, 0, steps)
    sub = np.array([0, 200])
    ins = synth.mamba2_steps(w, 0, steps)
    args = [ins[k].values[:, sub] for k in ("x", "B", "C", "dt")]
    y_rc = oracle.m2_readcopy(synth.mamba2_state0(w)[sub], A, D, *args, w.k, fmt)
    assert vec_err(y[:, sub], y_rc) < TOL_LOW


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_quantised_recurrence_baseline_matches_oracle(cuda_lib, fmt):
    """CONVENTIONAL mode with a read format: the state itself is stored in that
    format and re-quantised at every token. The oracle runs the same scheme in
    float64; code flips where the two round a value on either side of a grid
    midpoint are rare and stay within the low-precision tolerance."""
    w = synth.WORKLOADS["mamba2_fp32_b4"]
    S = 24
    layer, A, D = m2_layer(w, mode="conventional", read_fmt=fmt)
    y = m2_run_steps(layer, w, 0, S)
    ins = synth.mamba2_steps(w, 0, S)
    y_ref = oracle.m2_qrecurrence(synth.mamba2_state0(w), A, D,
                                  *(ins[k].values for k in ("x", "B", "C", "dt")), fmt)
    assert vec_err(y, y_ref) < TOL_LOW
    assert layer.get_error()[0] == 0
