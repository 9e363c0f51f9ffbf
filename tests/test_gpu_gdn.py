"""Gated DeltaNet replay decode (WY/UT window form) and the conventional
baseline on the GPU, against the float64 oracle."""
import numpy as np
import pytest
import torch

import hybrid_ssm_decode_gb300 as rssm
import oracle
import synth
from _gpu import TOL_F32, TOL_LOW, dev, gdn_layer, gdn_run_steps, host, tile_err, vec_err

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


@pytest.mark.parametrize("batch", [1, 16])
def test_small_batch_serving_heads_across_a_flush(cuda_lib, batch):
    """The serving layer's heads at small batches, where the direct kernels
    run (one wave at batch 1, several at 16): the outputs of 20 steps, and the
    checkpoint that the 16th step's fold wrote, against the oracle on sampled
    sequences."""
    w = GDN.replace(batch=batch)
    layer = gdn_layer(w, out_dtype="f32")
    sub = np.array(sorted({0, batch // 2, batch - 1}))
    o = gdn_run_steps(layer, w, 0, w.k, out_dtype="f32")
    o_ref, S_ref = _oracle(w, 0, w.k, subset=sub)
    assert vec_err(o[:, sub], o_ref) < TOL_F32
    assert not layer.counts().any().item()
    assert tile_err(host(layer.ckpt()[torch.from_numpy(sub).cuda()]), S_ref) < TOL_F32
    o2 = gdn_run_steps(layer, w, w.k, 4, out_dtype="f32")
    o2_ref, _ = _oracle(w, 0, w.k + 4, subset=sub)
    assert vec_err(o2[:, sub], o2_ref[w.k:]) < TOL_F32
    assert layer.get_error()[0] == 0


def _records(layer, w, slots):
    """The buffered records of slots [0, slots): k, u and alpha."""
    c = layer.cfg
    cap = layer.layout.capacity
    kdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    k = layer.region("buf_k", kdt, (c.batch, c.heads, cap, c.state_dim))[:, :, :slots]
    u = layer.region("buf_u", torch.float32, (c.batch, c.heads, c.head_dim // 64, cap, 64))[:, :, :, :slots]
    a = layer.region("buf_a", torch.float32, (c.batch, c.heads, cap))[:, :, :slots]
    return k, u, a


def test_pointer_moved_back_runs_the_fused_non_flush_branch(cuda_lib):
    """Move every window pointer back by one record just before a flush step.
    That step then flushes no tile, so the kernel that handles every tile runs
    its non-flush branch. Its outputs and records must equal, bit for bit, the
    lean non-flush kernel's on the same window (a layer that never saw the
    dropped token), and match the oracle on the token sequence without it."""
    w = GDN.replace(batch=3, heads=4, k=8, scale=0.5)      # bf16 inputs
    k = w.k
    ins = synth.gdn_steps(w, 0, k)

    def step(layer, s, fill=0.0):
        o = torch.full((w.batch, 1, w.heads, w.d_v), fill, dtype=torch.float32, device="cuda")
        layer.decode_step(o, 1, q=dev(ins["q"][s]), k=dev(ins["k"][s]), v=dev(ins["v"][s]),
                          alpha=dev(ins["alpha"][s]), beta=dev(ins["beta"][s]))
        return o

    a, b = gdn_layer(w, out_dtype="f32"), gdn_layer(w, out_dtype="f32")
    for s in range(k - 2):
        step(a, s)
    for s in range(k - 1):
        step(b, s)
    b.counts().sub_(1)                     # drop token k-2's record: a pointer move
    oa, ob = step(a, k - 1), step(b, k - 1)
    assert b.get_error()[0] == 0 and a.get_error()[0] == 0
    assert torch.equal(oa, ob)
    assert torch.equal(a.counts(), b.counts()) and bool((a.counts() == k - 1).all())
    assert torch.equal(a.ckpt(), b.ckpt())
    for ra, rb in zip(_records(a, w, k - 1), _records(b, w, k - 1)):
        assert torch.equal(ra, rb)

    seq = list(range(k - 2)) + [k - 1]
    vals = [ins[n].values[seq] for n in ("q", "k", "v", "alpha", "beta")]
    o_ref, S_ref = oracle.gdn_recurrence(synth.gdn_state0(w), *vals, scale=w.scale)
    assert vec_err(host(ob[:, 0]), o_ref[-1]) < TOL_F32

    # b's handle now takes the next step for a non-flush one, but every tile
    # is due to flush: the lean kernel reports them and leaves them alone
    ck = b.ckpt().clone()
    o = step(b, 0, fill=float("nan"))
    err = b.get_error()
    assert err[0] == rssm.RSSM_DEV_COUNT_RANGE and err[1] == w.batch * w.heads and err[3] == k - 1
    assert bool(torch.isnan(o).all()) and torch.equal(b.ckpt(), ck)
    assert bool((b.counts() == k - 1).all())
    b.flush()
    assert not b.counts().any().item()
    assert tile_err(host(b.ckpt()), S_ref) < TOL_F32


# ----------------------------------------------------------------------------
# speculative drafts (GDN): append unverified, roll back by the pointer
# ----------------------------------------------------------------------------
def _gdn_round(w, r, T):
    """Round r's T draft tokens: device tensors [B][T][...] and oracle values [T][B][...]."""
    ins = synth.gdn_steps(w, r * T, T)
    devs = {n: dev(np.ascontiguousarray(np.swapaxes(ins[n].raw, 0, 1))) for n in ("q", "k", "v", "alpha", "beta")}
    return devs, {n: ins[n].values for n in ("q", "k", "v", "alpha", "beta")}


def _gdn_draft_layer(w, T, out_dtype="f32", mode="replay"):
    cfg = rssm.make_config(kind="gdn", mode=mode, batch=w.batch, heads=w.heads, head_dim=w.d_v,
                           state_dim=w.d_k, groups=1, k=w.k, max_draft=T, in_dtype=w.dtype,
                           out_dtype=out_dtype, gdn_scale=w.scale)
    return rssm.Layer(cfg, None, None, dev(synth.gdn_state0(w)))


@pytest.mark.parametrize("T,dv,dk,dtype", [(4, 128, 128, "bf16"), (2, 64, 64, "f32"), (3, 128, 64, "f32")])
def test_gdn_spec_rounds_match_oracle(cuda_lib, T, dv, dk, dtype):
    w = GDN.replace(batch=3, heads=4, d_v=dv, d_k=dk, k=8, dtype=dtype, scale=0.5)
    R = 9
    acc = synth.acceptance(w.batch, R, T, 0.7, seed=T)
    acc[0, 0], acc[1, 1], acc[2, 2] = T, 0, T
    layer = _gdn_draft_layer(w, T)
    outs, per = [], []
    for r in range(R):
        d, vals = _gdn_round(w, r, T)
        o = torch.empty((w.batch, T, w.heads, w.d_v), dtype=torch.float32, device="cuda")
        layer.decode_step(o, T, q=d["q"], k=d["k"], v=d["v"], alpha=d["alpha"], beta=d["beta"])
        layer.verify_rollback(torch.from_numpy(acc[r]).cuda())
        outs.append(host(o).swapaxes(0, 1))          # [T][B][H][DV]
        per.append(vals)
    arr = {n: np.stack([p[n] for p in per]) for n in ("q", "k", "v", "alpha", "beta")}
    o_ref, S_ref = oracle.gdn_speculative(synth.gdn_state0(w), arr["q"], arr["k"], arr["v"], arr["alpha"],
                                          arr["beta"], acc, scale=w.scale)
    assert vec_err(np.stack(outs), o_ref) < TOL_F32
    assert layer.get_error()[0] == 0
    c = np.zeros(w.batch, np.int64)
    for a in acc:
        c = c + a
        c[c >= w.k] = 0
    np.testing.assert_array_equal(layer.counts().cpu().numpy(), np.repeat(c[:, None], w.heads, 1))
    layer.flush()
    assert tile_err(host(layer.ckpt()), S_ref) < TOL_F32


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gdn_snapshot_baseline_matches_oracle(cuda_lib, dtype):
    """The in-build snapshot save/restore baseline for GDN drafts
    (CONVENTIONAL mode, T > 1): T conventional steps writing a snapshot each,
    then the snapshot of the accepted prefix restored."""
    w = GDN.replace(batch=3, heads=4, k=8, dtype=dtype, scale=0.5)
    T, R = 4, 7
    acc = synth.acceptance(w.batch, R, T, 0.7, seed=9)
    acc[0, 0], acc[1, 1], acc[2, 2] = T, 0, T
    layer = _gdn_draft_layer(w, T, mode="conventional")
    outs, per = [], []
    for r in range(R):
        d, vals = _gdn_round(w, r, T)
        o = torch.empty((w.batch, T, w.heads, w.d_v), dtype=torch.float32, device="cuda")
        layer.decode_step(o, T, q=d["q"], k=d["k"], v=d["v"], alpha=d["alpha"], beta=d["beta"])
        layer.verify_rollback(torch.from_numpy(acc[r]).cuda())
        outs.append(host(o).swapaxes(0, 1))
        per.append(vals)
    arr = {n: np.stack([p[n] for p in per]) for n in ("q", "k", "v", "alpha", "beta")}
    o_ref, S_ref = oracle.gdn_speculative(synth.gdn_state0(w), arr["q"], arr["k"], arr["v"], arr["alpha"],
                                          arr["beta"], acc, scale=w.scale)
    assert vec_err(np.stack(outs), o_ref) < TOL_F32
    assert tile_err(host(layer.ckpt()), S_ref) < TOL_F32
    assert layer.get_error()[0] == 0


def test_gdn_rollback_of_all_drafts_is_a_noop(cuda_lib):
    """Draft T tokens and accept none: counts, state and every later output
    are bit-identical to a layer that never drafted."""
    w = GDN.replace(batch=2, heads=8, k=16, scale=0.5)
    T = 4
    a, b = _gdn_draft_layer(w, T), _gdn_draft_layer(w, T)
    gdn_run_steps(a, w, 0, 6, out_dtype="f32")
    gdn_run_steps(b, w, 0, 6, out_dtype="f32")
    d, _ = _gdn_round(w, 40, T)
    o = torch.empty((w.batch, T, w.heads, w.d_v), dtype=torch.float32, device="cuda")
    a.decode_step(o, T, q=d["q"], k=d["k"], v=d["v"], alpha=d["alpha"], beta=d["beta"])
    a.verify_rollback(torch.zeros(w.batch, dtype=torch.int32, device="cuda"))
    assert torch.equal(a.counts(), b.counts()) and torch.equal(a.ckpt(), b.ckpt())
    oa = gdn_run_steps(a, w, 6, 14, out_dtype="f32")
    ob = gdn_run_steps(b, w, 6, 14, out_dtype="f32")
    np.testing.assert_array_equal(oa, ob)
    assert torch.equal(a.ckpt(), b.ckpt())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gdn_first_draft_is_the_one_token_step(cuda_lib, dtype):
    """Draft 0 sees the window of a one-token step with the same inputs. With
    FP32 inputs the kernels share that arithmetic: bit-identical outputs and
    records. With bf16 inputs the draft kernel forms the key dots on the
    tensor cores, so they agree to the FP32 rounding of those sums."""
    w = GDN.replace(batch=2, heads=8, k=16, scale=0.5, dtype=dtype)
    T = 3
    a, b = _gdn_draft_layer(w, T), _gdn_draft_layer(w, T)
    gdn_run_steps(a, w, 0, 5, out_dtype="f32")
    gdn_run_steps(b, w, 0, 5, out_dtype="f32")
    d, _ = _gdn_round(w, 11, T)
    oa = torch.empty((w.batch, T, w.heads, w.d_v), dtype=torch.float32, device="cuda")
    a.decode_step(oa, T, q=d["q"], k=d["k"], v=d["v"], alpha=d["alpha"], beta=d["beta"])
    ob = torch.empty((w.batch, 1, w.heads, w.d_v), dtype=torch.float32, device="cuda")
    one = {n: t[:, :1].contiguous() for n, t in d.items()}
    b.decode_step(ob, 1, q=one["q"], k=one["k"], v=one["v"], alpha=one["alpha"], beta=one["beta"])
    a.verify_rollback(torch.ones(w.batch, dtype=torch.int32, device="cuda"))
    assert torch.equal(a.counts(), b.counts())
    if dtype == "f32":
        assert torch.equal(oa[:, 0], ob[:, 0])
        for ra, rb in zip(_records(a, w, 6), _records(b, w, 6)):
            assert torch.equal(ra, rb)
    else:
        assert vec_err(host(oa[:, 0]), host(ob[:, 0])) < 1e-5
        for ra, rb in zip(_records(a, w, 6), _records(b, w, 6)):
            assert vec_err(host(ra).reshape(ra.shape[0], -1), host(rb).reshape(rb.shape[0], -1)) < 1e-5
