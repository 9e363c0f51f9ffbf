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
from _gpu import TOL_F32, dev, gdn_layer, gdn_run_steps, host, tile_err, vec_err

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


def _gdn_stored(layer, w, fmt, sub):
    """The quantised state the GPU stores for the sequences in the index
    array `sub`: codes [halves][64][...] and the decoded state
    [len(sub)][H][d_v][d_k]."""
    lay, ws = layer.layout, layer.workspace
    dv, dk = w.d_v, w.d_k
    codes = ws[lay.rc_codes:lay.rc_codes + lay.rc_codes_bytes].view(w.batch, w.heads, dv, -1)[sub]
    ts = ws[lay.rc_tscale:lay.rc_tscale + lay.rc_tscale_bytes].view(torch.float32).view(w.batch, -1)[sub]
    codes = codes.cpu().numpy().reshape(-1, 64, codes.shape[-1])
    ts = ts.cpu().numpy().reshape(-1)
    if fmt == "fp8":
        dec = oracle.dequant_fp8(codes, ts)
    else:
        bsc = ws[lay.rc_bscale:lay.rc_bscale + lay.rc_bscale_bytes].view(w.batch, w.heads, dv, dk // 16)[sub]
        dec = oracle.dequant_nvfp4(codes, bsc.cpu().numpy().reshape(-1, 64, dk // 16), ts)
    return codes, dec.reshape(len(sub), w.heads, dv, dk)


def _check_qrecurrence(layer, w, fmt, S, sub):
    """Token by token from the state the GPU stored: the token's output is
    the recurrence step from the decoded state (FP32 tolerance), and the
    state it stores is the quantiser's encoding of that step's result, code
    for code almost everywhere (the kernel updates in FP32 and the oracle in
    float64, so a value near a code midpoint may round either way; such a
    flip then persists in the quantised state, which is why whole runs are
    not compared). Returns the outputs [S][B][H][d_v]."""
    args = _inputs(w, 0, S, sub)
    quant = oracle.quant_fp8 if fmt == "fp8" else oracle.quant_nvfp4
    flips, n_codes, outs = 0, 0, []
    for s in range(S):
        _, st = _gdn_stored(layer, w, fmt, sub)
        o = gdn_run_steps(layer, w, s, 1, out_dtype="f32")
        o_ref, S_new = oracle.gdn_recurrence(st, *(a[s:s + 1] for a in args), scale=w.scale)
        assert vec_err(o[:, sub], o_ref) < TOL_F32, s
        codes, _ = _gdn_stored(layer, w, fmt, sub)
        want = quant(S_new.reshape(-1, 64, w.d_k).astype(np.float32))[0]
        flips += int(np.count_nonzero(codes != want))
        n_codes += codes.size
        outs.append(o[0])
    assert flips <= 1e-3 * n_codes
    return np.stack(outs)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gdn_quantised_recurrence_matches_oracle(cuda_lib, fmt, dtype):
    """CONVENTIONAL mode with a read format: the GDN state itself is kept in
    that format (one tile per 64-row half) and re-quantised at every token.
    Every sequence, 24 tokens; the first token also against the oracle's
    whole quantised recurrence (no flip can precede it)."""
    w = GDN.replace(batch=3, heads=4, dtype=dtype, read_fmt=fmt, scale=0.5)
    S = 24
    layer = gdn_layer(w, mode="conventional", out_dtype="f32")
    o = _check_qrecurrence(layer, w, fmt, S, np.arange(w.batch))
    o_ref = oracle.gdn_qrecurrence(synth.gdn_state0(w), *_inputs(w, 0, 1), fmt, scale=w.scale)
    assert vec_err(o[:1], o_ref) < TOL_F32
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_quantised_recurrence_serving_shape_sampled(cuda_lib, fmt):
    """The GDN quantised-recurrence baseline at the serving shape (B256, H32,
    128 x 128, bf16 inputs) over 64 tokens, sampled sequences checked token
    by token from the state the GPU stored."""
    w = GDN.replace(read_fmt=fmt)
    layer = gdn_layer(w, mode="conventional", out_dtype="f32")
    _check_qrecurrence(layer, w, fmt, 64, np.array([0, 131]))
    assert layer.get_error()[0] == 0


# ----------------------------------------------------------------------------
# speculative drafts that read the copy
# ----------------------------------------------------------------------------
def _round(w, r, T):
    """Round r's T draft tokens: device tensors [B][T][...] and oracle values [T][B][...]."""
    ins = synth.gdn_steps(w, r * T, T)
    keys = ("q", "k", "v", "alpha", "beta")
    devs = {n: dev(np.ascontiguousarray(np.swapaxes(ins[n].raw, 0, 1))) for n in keys}
    return devs, {n: ins[n].values for n in keys}


def _draft_layer(w, T):
    cfg = rssm.make_config(kind="gdn", mode="replay", batch=w.batch, heads=w.heads, head_dim=w.d_v,
                           state_dim=w.d_k, groups=1, k=w.k, max_draft=T, in_dtype=w.dtype, out_dtype="f32",
                           gdn_scale=w.scale, read_fmt=w.read_fmt)
    return rssm.Layer(cfg, None, None, dev(synth.gdn_state0(w)))


def _spec_check(layer, w, fmt, T, acc, sub):
    """Runs len(acc) rounds and checks every round of the sequences in `sub`
    from the FP32 checkpoint the GPU stored at that sequence's last fold: its
    copy is the oracle quantiser's bit for bit, and the round's draft outputs
    are the oracle's rounds since the fold (FP32 tolerance). Returns the
    committed counts."""
    keys = ("q", "k", "v", "alpha", "beta")
    R = acc.shape[0]
    per = [_round(w, r, T)[1] for r in range(R)]
    count = np.zeros(w.batch, np.int64)
    since = np.zeros(w.batch, np.int64)
    ck_fold = {int(b): _ckpt(layer, w)[b] for b in sub}
    lay, ws = layer.layout, layer.workspace
    for r in range(R):
        ck_now = np.stack([ck_fold[int(b)] for b in sub])
        halves = ck_now.reshape(-1, 64, w.d_k).astype(np.float32)
        ref = (oracle.quant_fp8 if fmt == "fp8" else oracle.quant_nvfp4)(halves)
        codes = ws[lay.rc_codes:lay.rc_codes + lay.rc_codes_bytes].view(w.batch, w.heads, w.d_v, -1)[sub]
        np.testing.assert_array_equal(codes.cpu().numpy().reshape(halves.shape[0], 64, -1), ref[0])
        d, _ = _round(w, r, T)
        o = torch.empty((w.batch, T, w.heads, w.d_v), dtype=torch.float32, device="cuda")
        layer.decode_step(o, T, **{n: d[n] for n in keys})
        layer.verify_rollback(torch.from_numpy(acc[r]).cuda())
        o = host(o).swapaxes(0, 1)                       # [T][B][H][DV]
        for b in sub:
            r0 = since[b]
            arr = [np.stack([per[q][n][:, b:b + 1] for q in range(r0, r + 1)]) for n in keys]
            o_ref, _, _ = oracle.gdn_speculative_readcopy(ck_fold[int(b)][None], *arr, acc[r0:r + 1, b:b + 1],
                                                          w.k, fmt, scale=w.scale)
            assert vec_err(o[:, b], o_ref[-1][:, 0]) < TOL_F32, (r, b)
        count += acc[r]
        folded = count >= w.k
        count[folded] = 0
        since[folded] = r + 1
        for b in sub:
            if folded[b]:
                ck_fold[int(b)] = _ckpt(layer, w)[b]
    return count


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("T,dv,dk", [(4, 128, 128), (2, 64, 64), (3, 128, 64)])
def test_gdn_spec_readcopy_rounds_match_oracle(cuda_lib, fmt, T, dv, dk):
    w = GDN.replace(batch=3, heads=4, d_v=dv, d_k=dk, k=8, scale=0.5, read_fmt=fmt)
    R = 10
    acc = synth.acceptance(w.batch, R, T, 0.7, seed=T + dv)
    acc[0, 0], acc[1, 1], acc[2, 2] = T, 0, T
    layer = _draft_layer(w, T)
    count = _spec_check(layer, w, fmt, T, acc, np.arange(w.batch))
    np.testing.assert_array_equal(layer.counts().cpu().numpy(), np.repeat(count[:, None], w.heads, 1))
    # the copy never reaches the recurrence: after a flush the checkpoint is
    # the exact committed state
    keys = ("q", "k", "v", "alpha", "beta")
    per = [_round(w, r, T)[1] for r in range(R)]
    arr = [np.stack([p[n] for p in per]) for n in keys]
    _, S_ref = oracle.gdn_speculative(synth.gdn_state0(w), *arr, acc, scale=w.scale)
    layer.flush()
    assert tile_err(_ckpt(layer, w), S_ref) < TOL_F32
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_spec_readcopy_then_plain_decode(cuda_lib, fmt):
    """Plain read-copy steps after drafting rounds continue from the same
    records: window by window against the oracle's read-copy decode from the
    checkpoint the GPU stored, after a flush that folds the drafted rounds."""
    w = GDN.replace(batch=2, heads=4, k=8, scale=0.5, read_fmt=fmt)
    T, R = 3, 4
    acc = synth.acceptance(w.batch, R, T, 0.7, seed=5)
    layer = _draft_layer(w, T)
    _spec_check(layer, w, fmt, T, acc, np.arange(w.batch))
    layer.flush()
    assert not layer.counts().any().item()
    _check_windows(layer, w, fmt, [8, 6])
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_gdn_spec_readcopy_serving_shape_sampled(cuda_lib, fmt):
    """The batch-512 speculative GDN shape (H32, 128 x 128), 4 drafts per
    round over 10 rounds (folds included); sampled sequences round by round."""
    w = synth.WORKLOADS["gdn_spec_b512"].replace(read_fmt=fmt)
    T, R = 4, 10
    acc = synth.acceptance(w.batch, R, T, w.accept_p)
    layer = _draft_layer(w, T)
    count = _spec_check(layer, w, fmt, T, acc, np.array([0, 300, 511]))
    np.testing.assert_array_equal(layer.counts().cpu().numpy()[:, 0], count)
    assert layer.get_error()[0] == 0
