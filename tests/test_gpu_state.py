"""State export / import and the host's knowledge of the record counts.

A sequence's state is its checkpoint, the inputs buffered since, and the
buffer pointer ("NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section
"ReplaySSM nasil calisir?", 2nd paragraph). The image that rssm_export_state
writes holds all three, so a fresh handle that imports it mid-window
continues with outputs, records and checkpoint bit-identical to an
uninterrupted run. After a speculative verify the counts differ per sequence
and live on the device; rssm_sync_counts brings them back to the host so that
plain steps run the non-flush kernel again.
"""
import numpy as np
import pytest
import torch

import hybrid_ssm_decode_gb300 as rssm
import oracle
import synth
from _gpu import TOL_F32, dev, gdn_layer, gdn_run_steps, host, m2_layer, m2_out, m2_run_steps, vec_err

pytestmark = pytest.mark.gpu

SERVING = synth.WORKLOADS["mamba2_serving_b256"]
GDN = synth.WORKLOADS["gdn_serving_b256"]
SPEC = synth.WORKLOADS["mamba2_spec_b512"]


def _same_state(a, b):
    """Every state region of two layers is bit-identical."""
    lay = a.layout
    for r in ("ckpt", "ckpt_bscale", "ckpt_tscale", "counts", "buf_x", "buf_b", "buf_dt", "buf_k", "buf_u",
              "buf_a", "buf_v", "buf_beta", "rc_codes", "rc_bscale", "rc_tscale"):
        off, n = getattr(lay, r), getattr(lay, r + "_bytes")
        if n:
            assert torch.equal(a.workspace[off:off + n], b.workspace[off:off + n]), r


@pytest.mark.parametrize("read_fmt,ckpt", [("none", "f32"), ("nvfp4", "f32"), ("fp8", "f32"), ("none", "f16")])
def test_mamba2_resume_mid_window_is_bit_identical(cuda_lib, read_fmt, ckpt):
    w = SERVING.replace(batch=4, heads=16, groups=2, k=16, read_fmt=read_fmt, ckpt=ckpt)
    a, A, D = m2_layer(w, out_dtype="f32")
    m2_run_steps(a, w, 0, 7, out_dtype="f32")                 # c = 7, mid-window
    image = a.export_state()
    assert image.numel() == rssm.rssm_state_bytes(a.handle)
    # a fresh handle on another workspace, started from a different state
    b, _, _ = m2_layer(w, out_dtype="f32", state0=False)
    b.import_state(image)
    assert b.count_summary() == (1, 7, 7)
    _same_state(a, b)
    ya = m2_run_steps(a, w, 7, 20, out_dtype="f32")           # crosses the flush at token 16
    yb = m2_run_steps(b, w, 7, 20, out_dtype="f32")
    np.testing.assert_array_equal(ya, yb)
    _same_state(a, b)
    assert a.get_error()[0] == 0 and b.get_error()[0] == 0
    if ckpt == "f32" and read_fmt == "none":
        # and the continued outputs are the recurrence's
        ins = synth.mamba2_steps(w, 0, 27)
        y_ref, _ = oracle.m2_recurrence(synth.mamba2_state0(w), A, D,
                                        *(ins[key].values for key in ("x", "B", "C", "dt")))
        assert vec_err(yb, y_ref[7:]) < TOL_F32


@pytest.mark.parametrize("read_fmt", ["none", "nvfp4"])
def test_gdn_resume_mid_window_is_bit_identical(cuda_lib, read_fmt):
    w = GDN.replace(batch=3, heads=4, k=16, read_fmt=read_fmt)
    a = gdn_layer(w, out_dtype="f32")
    gdn_run_steps(a, w, 0, 7, out_dtype="f32")
    image = a.export_state()
    cfg = a.cfg
    b = rssm.Layer(cfg, None, None, None)
    b.import_state(image)
    assert b.count_summary() == (1, 7, 7)
    _same_state(a, b)
    oa = gdn_run_steps(a, w, 7, 20, out_dtype="f32")
    ob = gdn_run_steps(b, w, 7, 20, out_dtype="f32")
    np.testing.assert_array_equal(oa, ob)
    _same_state(a, b)


def test_resume_with_speculative_records(cuda_lib):
    """An image taken after a verify (counts differ per sequence) resumes
    speculative rounds bit for bit."""
    w = SPEC.replace(batch=6, heads=8, groups=2, dtype="bf16", k=16)
    T = 4
    acc = synth.acceptance(w.batch, 6, T, w.accept_p, seed=5)
    layers = [m2_layer(w, max_draft=T, out_dtype="f32")[0] for _ in range(2)]

    def spec_round(layer, r):
        ins = synth.mamba2_steps(w, r * T, T)
        d = {k: dev(np.ascontiguousarray(np.swapaxes(ins[k].raw, 0, 1))) for k in ("x", "B", "C", "dt")}
        y = m2_out(w, T, "f32")
        layer.decode_step(y, T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
        layer.verify_rollback(torch.from_numpy(acc[r]).cuda())
        return host(y)

    for r in range(3):
        spec_round(layers[0], r)
    image = layers[0].export_state()
    layers[1].import_state(image)
    known, lo, hi = layers[1].count_summary()
    counts = layers[0].counts().cpu().numpy()
    assert known == 1 and lo == counts.min() and hi == counts.max()
    for r in range(3, 6):
        np.testing.assert_array_equal(spec_round(layers[0], r), spec_round(layers[1], r))
    _same_state(layers[0], layers[1])


def test_import_rejects_other_configurations(cuda_lib):
    w = SERVING.replace(batch=2, heads=8, groups=1, k=16)
    a, _, _ = m2_layer(w)
    image = a.export_state()
    other, _, _ = m2_layer(w, k=8)
    with pytest.raises(rssm.RssmError) as e:
        other.import_state(image)
    assert e.value.status == rssm.RSSM_ERR_INVALID_ARG
    bad = image.clone()
    bad[0] ^= 1                                               # not an image
    with pytest.raises(rssm.RssmError) as e:
        a.import_state(bad)
    assert e.value.status == rssm.RSSM_ERR_INVALID_ARG
    with pytest.raises(rssm.RssmError) as e:                  # too small
        rssm.rssm_import_state(a.handle, image, image.numel() - 256)
    assert e.value.status == rssm.RSSM_ERR_INVALID_ARG


def _kernel_names(fn):
    """Names of the CUDA kernels fn launches (CUPTI activity records)."""
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]


def test_counts_synced_after_rollback_bring_back_the_lean_kernel(cuda_lib):
    """After a verify the handle no longer knows the counts, so a plain step
    runs in two launches: the non-flush kernel over the tiles that do not
    complete their window and the step kernel over those that do.
    rssm_sync_counts reads the counts' summary from the device; the next
    steps then run the non-flush kernel alone wherever no tile flushes, and
    the outputs are bit-identical either way, through the flushes of the tiles
    that fill their window first."""
    w = SPEC.replace(batch=8, heads=8, groups=2, dtype="bf16", k=16)
    T = 4
    acc = synth.acceptance(w.batch, 3, T, w.accept_p, seed=11)
    acc[:, 0] = 4                                             # one sequence reaches 12 records
    synced, _, _ = m2_layer(w, max_draft=T, out_dtype="f32")
    unsynced, _, _ = m2_layer(w, max_draft=T, out_dtype="f32")
    for layer in (synced, unsynced):
        for r in range(3):
            ins = synth.mamba2_steps(w, r * T, T)
            d = {k: dev(np.ascontiguousarray(np.swapaxes(ins[k].raw, 0, 1))) for k in ("x", "B", "C", "dt")}
            layer.decode_step(m2_out(w, T, "f32"), T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
            layer.verify_rollback(torch.from_numpy(acc[r]).cuda())
        assert layer.count_summary() == (0, -1, -1)
    synced.sync_counts()
    counts = synced.counts()[:, 0].cpu().numpy()
    assert synced.count_summary() == (1, int(counts.min()), int(counts.max()))
    assert counts.max() == 12

    # the next step runs the non-flush kernel on the synced handle only
    ins = synth.mamba2_steps(w, 100, 1)
    args = {k: dev(ins[k][0]) for k in ("x", "B", "C", "dt")}
    names_s = _kernel_names(lambda: synced.decode_step(m2_out(w, 1, "f32"), 1, x=args["x"], Bm=args["B"],
                                                       C=args["C"], dt=args["dt"]))
    names_u = _kernel_names(lambda: unsynced.decode_step(m2_out(w, 1, "f32"), 1, x=args["x"], Bm=args["B"],
                                                         C=args["C"], dt=args["dt"]))
    if names_s and names_u:                                   # the profiler saw the launches
        # synced: the non-flush kernel alone; unsynced: the non-flush kernel
        # over the tiles that do not flush, then the step kernel over those that do
        assert any("m2_replay_nf_kernel" in n for n in names_s), names_s
        assert not any("m2_replay_step_tma_kernel" in n for n in names_s), names_s
        assert any("m2_replay_nf_kernel" in n for n in names_u), names_u
        assert any("m2_replay_step_tma_kernel" in n for n in names_u), names_u
    assert synced.count_summary() == (1, int(counts.min()) + 1, 13)
    # 10 more plain steps: the sequence at 13 flushes at its 16th record
    ys = m2_run_steps(synced, w, 101, 10, out_dtype="f32")
    yu = m2_run_steps(unsynced, w, 101, 10, out_dtype="f32")
    np.testing.assert_array_equal(ys, yu)
    assert torch.equal(synced.counts(), unsynced.counts())
    assert torch.equal(synced.ckpt(), unsynced.ckpt())
    counts_after = synced.counts()[:, 0].cpu().numpy()
    known, lo, hi = synced.count_summary()
    assert known == 1 and lo == counts_after.min() and hi == counts_after.max()
    assert synced.get_error()[0] == 0 and unsynced.get_error()[0] == 0


def test_device_error_forgets_the_counts(cuda_lib):
    """A tile whose count was changed behind the handle's back is left
    unchanged and reported; after that report the handle no longer trusts its
    own count tracking."""
    w = SERVING.replace(batch=2, heads=4, groups=1, k=8)
    layer, _, _ = m2_layer(w)
    m2_run_steps(layer, w, 0, 2)
    layer.counts()[1, 2] = 7                                  # due to flush in a lean step
    m2_run_steps(layer, w, 2, 1)
    assert layer.count_summary()[0] == 1
    code = layer.get_error()[0]
    assert code == rssm.RSSM_DEV_COUNT_RANGE
    assert layer.count_summary() == (0, -1, -1)


def _spec_rounds_then_plain(layer, w, T, acc, plain, step_in, out_T, run_plain):
    """Speculative rounds (drafts + verify), then `plain` one-token steps."""
    ys = []
    for r in range(acc.shape[0]):
        d = step_in(r * T, T)
        y = out_T(T)
        layer.decode_step(y, T, **d)
        layer.verify_rollback(torch.from_numpy(acc[r]).cuda())
        ys.append(host(y).swapaxes(0, 1))
    return np.stack(ys), run_plain(layer, w, 1000, plain)


def test_plain_steps_after_verify_match_the_oracle(cuda_lib):
    """Mixed counts after speculative rounds: every plain step flushes some
    tiles (in its second launch) and not others, for 20 steps; the outputs
    and the checkpoint follow the recurrence from the committed state."""
    w = SPEC.replace(batch=6, heads=8, groups=2, dtype="f32", k=8)
    T, R = 4, 5
    acc = synth.acceptance(w.batch, R, T, w.accept_p, seed=21)
    A, D = synth.mamba2_params(w)
    layer, _, _ = m2_layer(w, max_draft=T, out_dtype="f32")

    def step_in(start, n):
        ins = synth.mamba2_steps(w, start, n)
        return {kk: dev(np.ascontiguousarray(np.swapaxes(ins[k].raw, 0, 1)))
                for kk, k in (("x", "x"), ("Bm", "B"), ("C", "C"), ("dt", "dt"))}

    y_spec, y_plain = _spec_rounds_then_plain(
        layer, w, T, acc, 20, step_in, lambda t: m2_out(w, t, "f32"),
        lambda l, w_, s0, n: m2_run_steps(l, w_, s0, n, out_dtype="f32"))
    per = [synth.mamba2_steps(w, r * T, T) for r in range(R)]
    arr = {k: np.stack([p[k].values for p in per]) for k in ("x", "B", "C", "dt")}
    y_ref, h = oracle.m2_speculative(synth.mamba2_state0(w), A, D, arr["x"], arr["B"], arr["C"], arr["dt"], acc)
    assert vec_err(y_spec, y_ref) < TOL_F32
    ins = synth.mamba2_steps(w, 1000, 20)
    y_pref, h_end = oracle.m2_recurrence(h, A, D, *(ins[k].values for k in ("x", "B", "C", "dt")))
    assert vec_err(y_plain, y_pref) < TOL_F32
    layer.flush()
    from _gpu import tile_err
    assert tile_err(host(layer.ckpt()), h_end) < TOL_F32
    assert layer.get_error()[0] == 0


def test_gdn_plain_steps_after_verify_match_the_oracle(cuda_lib):
    w = GDN.replace(batch=4, heads=4, k=8, dtype="f32")
    T, R = 4, 5
    acc = synth.acceptance(w.batch, R, T, 0.7, seed=22)
    cfg = rssm.make_config(kind="gdn", batch=w.batch, heads=w.heads, head_dim=w.d_v, state_dim=w.d_k, k=w.k,
                           max_draft=T, in_dtype="f32", out_dtype="f32", gdn_scale=w.scale)
    layer = rssm.Layer(cfg, None, None, dev(synth.gdn_state0(w)))

    def step_in(start, n):
        ins = synth.gdn_steps(w, start, n)
        return {k: dev(np.ascontiguousarray(np.swapaxes(ins[k].raw, 0, 1)))
                for k in ("q", "k", "v", "alpha", "beta")}

    def out_T(t):
        return torch.empty((w.batch, t, w.heads, w.d_v), dtype=torch.float32, device="cuda")

    y_spec, y_plain = _spec_rounds_then_plain(layer, w, T, acc, 20, step_in, out_T,
                                              lambda l, w_, s0, n: gdn_run_steps(l, w_, s0, n, out_dtype="f32"))
    per = [synth.gdn_steps(w, r * T, T) for r in range(R)]
    arr = [np.stack([p[k].values for p in per]) for k in ("q", "k", "v", "alpha", "beta")]
    o_ref, S = oracle.gdn_speculative(synth.gdn_state0(w), *arr, acc, scale=w.scale)
    assert vec_err(y_spec, o_ref) < TOL_F32
    ins = synth.gdn_steps(w, 1000, 20)
    o_pref, S_end = oracle.gdn_recurrence(S, *(ins[k].values for k in ("q", "k", "v", "alpha", "beta")),
                                          scale=w.scale)
    assert vec_err(y_plain, o_pref) < TOL_F32
    layer.flush()
    from _gpu import tile_err
    assert tile_err(host(layer.ckpt()), S_end) < TOL_F32
    assert layer.get_error()[0] == 0
