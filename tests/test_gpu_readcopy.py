"""Low-precision read copies (FP8 E4M3, NVFP4): the writer is bit-exact with
the oracle's quantiser on the same FP32 tiles, the decode outputs match the
oracle's read-copy emulation, and the FP32 recurrence is untouched."""
import numpy as np
import pytest
import torch

import hybrid_ssm_decode_gb300 as rssm
import oracle
import synth
from _gpu import TOL_F32, TOL_LOW, dev, host, m2_copy_regions, m2_layer, m2_run_steps, tile_err, vec_err

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


def _check_windows(layer, w, A, D, fmt, windows, sub=slice(None)):
    """Window by window, from the checkpoint the GPU stored: the copy is the
    oracle quantiser's copy of that FP32 checkpoint bit for bit, and the
    window's outputs are the oracle's read-copy decode started from it, at the
    FP32 tolerance (the k-th token of a window is the flush token and reads
    the checkpoint itself). Returns the outputs of all windows."""
    P, N = w.head_dim, w.state_dim
    start, ys = 0, []
    for n in windows:
        ck = host(layer.ckpt()[sub])
        codes, bsc, ts = m2_copy_regions(layer, w, sub)
        ref = (oracle.quant_fp8 if fmt == "fp8" else oracle.quant_nvfp4)(ck.reshape(-1, P, N).astype(np.float32))
        np.testing.assert_array_equal(codes, ref[0])
        np.testing.assert_array_equal(ts, ref[-1])
        if fmt == "nvfp4":
            np.testing.assert_array_equal(bsc, ref[1])
        y, ins = m2_run_steps(layer, w, start, n, out_dtype="f32", return_inputs=True)
        args = [ins[k].values[:, sub] for k in ("x", "B", "C", "dt")]
        y_ref = oracle.m2_readcopy(ck, A, D, *args, w.k, fmt)
        assert vec_err(y[:, sub], y_ref) < TOL_F32
        if n == w.k:   # the flush stored the FP32 recurrence of the window
            _, h_end = oracle.m2_recurrence(ck, A, D, *args)
            assert tile_err(host(layer.ckpt()[sub]), h_end) < TOL_F32
        ys.append(y)
        start += n
    return np.concatenate(ys)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_readcopy_decode_matches_oracle_window_by_window(cuda_lib, fmt, dtype):
    w = SERVING.replace(batch=3, heads=16, groups=2, k=8, steps=30, read_fmt=fmt, dtype=dtype)
    layer, A, D = m2_layer(w, out_dtype="f32")
    y = _check_windows(layer, w, A, D, fmt, [8, 8, 8, 6])
    # flush-step outputs read the FP32 checkpoint: they are the exact
    # recurrence's (the other outputs carry the copy's quantisation error,
    # which the error-over-length measurement reports)
    ins = synth.mamba2_steps(w, 0, w.steps)
    args = [ins[k].values for k in ("x", "B", "C", "dt")]
    y_ex, _ = oracle.m2_recurrence(synth.mamba2_state0(w), A, D, *args)
    flush = [t for t in range(w.steps) if (t + 1) % w.k == 0]
    assert vec_err(y[flush], y_ex[flush]) < TOL_F32
    assert layer.get_error()[0] == 0


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
    """Full serving batch with a read copy over 48 steps (3 windows), sampled
    sequences checked window by window from the GPU's checkpoint."""
    w = SERVING.replace(read_fmt=fmt)
    layer, A, D = m2_layer(w, out_dtype="f32")
    _check_windows(layer, w, A, D, fmt, [16, 16, 16], sub=np.array([0, 200, 255]))
    assert layer.get_error()[0] == 0


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


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_quantised_recurrence_serving_shape_sampled(cuda_lib, fmt):
    """The quantised-recurrence baseline at the serving shape (B256, H128,
    P64, N128, G8, bf16 inputs) over 64 tokens, sampled sequences checked
    token by token from the state the GPU stored: the token's output is the
    recurrence step from the decoded state (FP32 tolerance), and the state it
    stores is the quantiser's encoding of that step's FP32 result, code for
    code almost everywhere (the kernel updates in FP32 and the oracle in
    float64, so a value near a code midpoint may round either way). Over the
    whole run such a flip persists in a quantised state, so the run as a whole
    is compared at the low-precision tolerance for FP8 only; NVFP4's coarser
    grid turns a flip into a larger change."""
    w = SERVING
    S = 64
    P, N = w.head_dim, w.state_dim
    layer, A, D = m2_layer(w, mode="conventional", read_fmt=fmt, out_dtype="f32")
    sub = np.array([0, 131])
    ins = synth.mamba2_steps(w, 0, S)
    args = [ins[k].values[:, sub] for k in ("x", "B", "C", "dt")]
    deq = oracle.dequant_fp8 if fmt == "fp8" else oracle.dequant_nvfp4
    quant = oracle.quant_fp8 if fmt == "fp8" else oracle.quant_nvfp4

    def stored():
        codes, bsc, ts = m2_copy_regions(layer, w, sub)
        q = (codes, ts) if fmt == "fp8" else (codes, bsc, ts)
        return codes, deq(*q).reshape(len(sub), w.heads, P, N)

    ys, flips, n_codes = [], 0, 0
    for s in range(S):
        _, h = stored()
        y = m2_run_steps(layer, w, s, 1, out_dtype="f32")
        y_ref, h_new = oracle.m2_recurrence(h, A, D, *(a[s:s + 1] for a in args))
        assert vec_err(y[:, sub], y_ref) < TOL_F32
        codes, _ = stored()
        want = quant(h_new.reshape(-1, P, N).astype(np.float32))[0]
        flips += int(np.count_nonzero(codes != want))
        n_codes += codes.size
        ys.append(y[0])
    assert flips <= 1e-3 * n_codes
    if fmt == "fp8":
        y_run = oracle.m2_qrecurrence(synth.mamba2_state0(w)[sub], A, D, *args, fmt)
        assert vec_err(np.stack(ys)[:, sub], y_run) < TOL_LOW
    assert layer.get_error()[0] == 0
