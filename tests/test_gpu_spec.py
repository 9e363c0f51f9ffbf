"""Speculative drafts: replay (append unverified, roll back by moving the
buffer pointer) and the snapshot save/restore baseline, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import TOL_F32, dev, host, m2_layer, m2_out, m2_run_steps, tile_err, vec_err

pytestmark = pytest.mark.gpu

SPEC = synth.WORKLOADS["mamba2_spec_b512"]


def _round_inputs(w, r, T):
    """Inputs of round r as device tensors [B][T][...] and as oracle arrays [T][B][...]."""
    ins = synth.mamba2_steps(w, r * T, T)
    devs = {}
    for key in ("x", "B", "C", "dt"):
        raw = np.ascontiguousarray(np.swapaxes(ins[key].raw, 0, 1))
        devs[key] = dev(raw)
    return devs, {k: ins[k].values for k in ins}


def _run_spec(layer, w, rounds, T, accepted, out_dtype="f32"):
    ys = []
    for r in range(rounds):
        d, _ = _round_inputs(w, r, T)
        y = m2_out(w, T, out_dtype)
        layer.decode_step(y, T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
        layer.verify_rollback(torch.from_numpy(accepted[r]).cuda())
        ys.append(host(y).swapaxes(0, 1))           # [T][B][H][P]
    return np.stack(ys)


def _oracle_spec(w, rounds, T, accepted, subset=slice(None)):
    A, D = synth.mamba2_params(w)
    per = [_round_inputs(w, r, T)[1] for r in range(rounds)]
    arr = {k: np.stack([p[k][:, subset] for p in per]) for k in ("x", "B", "C", "dt")}
    return oracle.m2_speculative(synth.mamba2_state0(w)[subset], A, D, arr["x"], arr["B"],
                                 arr["C"], arr["dt"], accepted[:, subset])


def _expected_counts(accepted, k):
    c = np.zeros(accepted.shape[1], np.int64)
    for a in accepted:
        c = c + a
        c[c >= k] = 0
    return c


@pytest.mark.parametrize("mode", ["replay", "conventional"])
def test_spec_rounds_match_oracle(cuda_lib, mode):
    w = SPEC.replace(batch=6, heads=8, groups=2, dtype="f32", k=16)
    T, R = 4, 14
    acc = synth.acceptance(w.batch, R, T, w.accept_p, seed=3)
    acc[0, 0], acc[1, 1], acc[2, 2] = 0, 4, 0
    layer, A, D = m2_layer(w, mode=mode, max_draft=T)
    y = _run_spec(layer, w, R, T, acc)
    y_ref, h_ref = _oracle_spec(w, R, T, acc)
    assert vec_err(y, y_ref) < TOL_F32
    if mode == "replay":
        counts = layer.counts().cpu().numpy()
        np.testing.assert_array_equal(counts, np.repeat(_expected_counts(acc, w.k)[:, None], w.heads, 1))
        layer.flush()
    assert tile_err(host(layer.ckpt()), h_ref) < TOL_F32
    assert layer.get_error()[0] == 0


def test_rollback_of_all_drafts_is_a_noop(cuda_lib):
    """Append T drafts and accept none: counts, checkpoint and every later
    output are bit-identical to a run that never drafted."""
    w = SPEC.replace(batch=4, heads=8, groups=2, dtype="bf16", k=16)
    T = 4
    a, _, _ = m2_layer(w, max_draft=T)
    b, _, _ = m2_layer(w, max_draft=T)
    m2_run_steps(a, w, 0, 6)
    m2_run_steps(b, w, 0, 6)
    d, _ = _round_inputs(w, 50, T)
    y = m2_out(w, T)
    a.decode_step(y, T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
    a.verify_rollback(torch.zeros(w.batch, dtype=torch.int32, device="cuda"))
    assert torch.equal(a.counts(), b.counts())
    assert torch.equal(a.ckpt(), b.ckpt())
    ya = m2_run_steps(a, w, 6, 14)
    yb = m2_run_steps(b, w, 6, 14)
    np.testing.assert_array_equal(ya, yb)
    assert torch.equal(a.ckpt(), b.ckpt())


def test_out_of_range_acceptance_sets_error_and_keeps_sequence(cuda_lib):
    w = SPEC.replace(batch=3, heads=4, groups=1, dtype="f32", k=16)
    T = 4
    layer, _, _ = m2_layer(w, max_draft=T)
    d, _ = _round_inputs(w, 0, T)
    y = m2_out(w, T, "f32")
    layer.decode_step(y, T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
    layer.verify_rollback(torch.tensor([2, 7, -1], dtype=torch.int32, device="cuda"))
    code, count, where, value = layer.get_error()
    assert code == 1 and count == 2 and where in (1, 2) and value in (7, -1)
    counts = layer.counts().cpu().numpy()
    assert np.all(counts[0] == 2) and np.all(counts[1:] == 0)
    assert layer.get_error()[0] == 0      # reading clears the word


def test_host_state_errors(cuda_lib):
    import hybrid_ssm_decode_gb300 as rssm
    w = SPEC.replace(batch=2, heads=4, groups=1, dtype="f32")
    layer, _, _ = m2_layer(w, max_draft=4)
    d, _ = _round_inputs(w, 0, 4)
    y = m2_out(w, 4, "f32")
    with pytest.raises(rssm.RssmError) as e:
        layer.decode_step(y, 5, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
    assert e.value.status == rssm.RSSM_ERR_CAPACITY
    layer.decode_step(y, 4, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
    with pytest.raises(rssm.RssmError) as e:
        layer.decode_step(y, 4, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
    assert e.value.status == rssm.RSSM_ERR_STATE
    with pytest.raises(rssm.RssmError):
        layer.flush()
    layer.verify_rollback(torch.full((2,), 4, dtype=torch.int32, device="cuda"))
    layer.flush()


def test_spec_full_batch_sampled(cuda_lib):
    """The batch-512 serving shape (2 GiB checkpoint), 4 drafts per round,
    truncated-geometric acceptance; sampled sequences against the oracle."""
    w = SPEC
    T, R = 4, 6
    acc = synth.acceptance(w.batch, R, T, w.accept_p)
    layer, A, D = m2_layer(w, max_draft=T, out_dtype="f32")
    y = _run_spec(layer, w, R, T, acc)
    subset = np.array([0, 5, 300, 511])
    y_ref, h_ref = _oracle_spec(w, R, T, acc, subset=subset)
    assert vec_err(y[:, :, subset], y_ref) < TOL_F32
    np.testing.assert_array_equal(layer.counts().cpu().numpy()[:, 0], _expected_counts(acc, w.k))


@pytest.mark.parametrize("T,P,N,dtype", [(2, 64, 128, "f32"), (3, 128, 64, "bf16"), (8, 64, 64, "f32"),
                                         (5, 128, 128, "bf16")])
def test_draft_lengths_and_tile_shapes(cuda_lib, T, P, N, dtype):
    w = SPEC.replace(batch=3, heads=4, groups=2, head_dim=P, state_dim=N, dtype=dtype, k=8)
    R = 10
    acc = synth.acceptance(w.batch, R, T, w.accept_p, seed=T)
    acc[0, 0], acc[1, 1] = T, 0
    layer, A, D = m2_layer(w, max_draft=T, out_dtype="f32")
    y = _run_spec(layer, w, R, T, acc)
    y_ref, h_ref = _oracle_spec(w, R, T, acc)
    assert vec_err(y, y_ref) < TOL_F32
    np.testing.assert_array_equal(layer.counts().cpu().numpy()[:, 0], _expected_counts(acc, w.k))
    layer.flush()
    assert tile_err(host(layer.ckpt()), h_ref) < TOL_F32
    assert layer.get_error()[0] == 0


def test_first_draft_is_the_one_token_step(cuda_lib):
    """Draft 0 of a round sees the same window as a one-token step with the
    same inputs, and the kernels share that arithmetic: bit-identical outputs."""
    w = SPEC.replace(batch=4, heads=16, groups=4, dtype="bf16", k=16)
    T = 4
    a, _, _ = m2_layer(w, max_draft=T, out_dtype="f32")
    b, _, _ = m2_layer(w, max_draft=T, out_dtype="f32")
    m2_run_steps(a, w, 0, 5, out_dtype="f32")
    m2_run_steps(b, w, 0, 5, out_dtype="f32")
    d, _ = _round_inputs(w, 9, T)
    ya = m2_out(w, T, "f32")
    a.decode_step(ya, T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
    yb = m2_out(w, 1, "f32")
    b.decode_step(yb, 1, x=d["x"][:, :1].contiguous(), Bm=d["B"][:, :1].contiguous(),
                  C=d["C"][:, :1].contiguous(), dt=d["dt"][:, :1].contiguous())
    assert torch.equal(ya[:, 0], yb[:, 0])
    a.verify_rollback(torch.ones(w.batch, dtype=torch.int32, device="cuda"))
    assert torch.equal(a.counts(), b.counts())
