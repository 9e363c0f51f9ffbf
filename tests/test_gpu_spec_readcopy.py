"""Mamba-2 speculative drafts that read the low-precision read copy (FP8
E4M3, NVFP4) against the oracle's speculative read-copy rounds.

Round by round and sequence by sequence, from the FP32 checkpoint the GPU
stored at that sequence's last fold: the copy is the oracle quantiser's copy
of that checkpoint bit for bit, and the round's draft outputs are the oracle's
speculative read-copy outputs over the rounds since the fold (FP32
tolerance). The recurrence stays on the FP32 checkpoint: after a flush it is
the exact committed state."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import TOL_F32, dev, host, m2_copy_regions, m2_layer, m2_out, m2_run_steps, tile_err, vec_err

pytestmark = pytest.mark.gpu

SPEC = synth.WORKLOADS["mamba2_spec_b512"]


def _round_inputs(w, r, T):
    """Inputs of round r as device tensors [B][T][...] and as oracle arrays [T][B][...]."""
    ins = synth.mamba2_steps(w, r * T, T)
    devs = {key: dev(np.ascontiguousarray(np.swapaxes(ins[key].raw, 0, 1))) for key in ("x", "B", "C", "dt")}
    return devs, {k: ins[k].values for k in ins}


def _quant(fmt, ck, P, N):
    return (oracle.quant_fp8 if fmt == "fp8" else oracle.quant_nvfp4)(ck.reshape(-1, P, N).astype(np.float32))


def _run_and_check(layer, w, A, D, fmt, T, acc, sub):
    """Runs len(acc) rounds of T drafts with acceptances acc [R][B] and checks
    every round of the sequences in `sub` (see the module docstring).
    Returns the committed counts the host expects."""
    P, N = w.head_dim, w.state_dim
    R = acc.shape[0]
    per = [_round_inputs(w, r, T)[1] for r in range(R)]
    count = np.zeros(w.batch, np.int64)
    since_fold = np.zeros(w.batch, np.int64)          # first round after the sequence's last fold
    ck_fold = {int(b): host(layer.ckpt()[b]) for b in sub}
    for r in range(R):
        codes, bsc, ts = m2_copy_regions(layer, w, sub)
        ck_now = np.stack([ck_fold[int(b)] for b in sub])
        ref = _quant(fmt, ck_now, P, N)
        np.testing.assert_array_equal(codes, ref[0])
        np.testing.assert_array_equal(ts, ref[-1])
        if fmt == "nvfp4":
            np.testing.assert_array_equal(bsc, ref[1])
        d, _ = _round_inputs(w, r, T)
        y = m2_out(w, T, "f32")
        layer.decode_step(y, T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
        layer.verify_rollback(torch.from_numpy(acc[r]).cuda())
        y = host(y).swapaxes(0, 1)                      # [T][B][H][P]
        for b in sub:
            r0 = since_fold[b]
            arr = {k: np.stack([per[q][k][:, b:b + 1] for q in range(r0, r + 1)]) for k in ("x", "B", "C", "dt")}
            y_ref, _, _ = oracle.m2_speculative_readcopy(ck_fold[int(b)][None], A, D, arr["x"], arr["B"], arr["C"],
                                                         arr["dt"], acc[r0:r + 1, b:b + 1], w.k, fmt)
            assert vec_err(y[:, b], y_ref[-1][:, 0]) < TOL_F32, (r, b)
        count += acc[r]
        folded = count >= w.k
        count[folded] = 0
        since_fold[folded] = r + 1
        for b in sub:
            if folded[b]:
                ck_fold[int(b)] = host(layer.ckpt()[b])
    return count


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_spec_readcopy_rounds_match_oracle(cuda_lib, fmt, dtype):
    w = SPEC.replace(batch=5, heads=8, groups=2, dtype=dtype, k=8, read_fmt=fmt)
    T, R = 4, 14
    acc = synth.acceptance(w.batch, R, T, w.accept_p, seed=11)
    acc[0, 0], acc[1, 1], acc[2, 2], acc[3, 3] = 0, 4, 0, 4
    layer, A, D = m2_layer(w, max_draft=T, out_dtype="f32")
    count = _run_and_check(layer, w, A, D, fmt, T, acc, np.arange(w.batch))
    np.testing.assert_array_equal(layer.counts().cpu().numpy(), np.repeat(count[:, None], w.heads, 1))
    # the FP32 recurrence is untouched by the copy: after a flush the
    # checkpoint is the exact committed state
    per = [_round_inputs(w, r, T)[1] for r in range(R)]
    arr = {k: np.stack([p[k] for p in per]) for k in ("x", "B", "C", "dt")}
    _, h_ref = oracle.m2_speculative(synth.mamba2_state0(w), A, D, arr["x"], arr["B"], arr["C"], arr["dt"], acc)
    layer.flush()
    assert tile_err(host(layer.ckpt()), h_ref) < TOL_F32
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("T,P,N,fmt", [(2, 64, 64, "nvfp4"), (8, 128, 128, "fp8"), (5, 128, 64, "nvfp4")])
def test_spec_readcopy_draft_lengths_and_tile_shapes(cuda_lib, T, P, N, fmt):
    w = SPEC.replace(batch=3, heads=4, groups=2, head_dim=P, state_dim=N, dtype="bf16", k=8, read_fmt=fmt)
    R = 9
    acc = synth.acceptance(w.batch, R, T, w.accept_p, seed=T + P)
    acc[0, 0], acc[1, 1] = T, 0
    layer, A, D = m2_layer(w, max_draft=T, out_dtype="f32")
    _run_and_check(layer, w, A, D, fmt, T, acc, np.arange(w.batch))
    assert layer.get_error()[0] == 0


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_first_draft_is_the_one_token_readcopy_step(cuda_lib, fmt, dtype):
    """Draft 0 sees the one-token step's window and reads the same copy with
    the same arithmetic: bit-identical outputs."""
    w = SPEC.replace(batch=4, heads=16, groups=4, dtype=dtype, k=16, read_fmt=fmt)
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


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_spec_readcopy_serving_shape_sampled(cuda_lib, fmt):
    """The batch-512 serving shape, 4 drafts per round, truncated-geometric
    acceptance over 12 rounds (folds included); sampled sequences checked
    round by round."""
    w = SPEC.replace(read_fmt=fmt)
    T, R = 4, 12
    acc = synth.acceptance(w.batch, R, T, w.accept_p)
    layer, A, D = m2_layer(w, max_draft=T, out_dtype="f32")
    count = _run_and_check(layer, w, A, D, fmt, T, acc, np.array([0, 300, 511]))
    np.testing.assert_array_equal(layer.counts().cpu().numpy()[:, 0], count)
    assert layer.get_error()[0] == 0
