"""Failure detection on the device without a fault: a bounded wait that runs
out reports RSSM_DEV_TIMEOUT through the error word, the kernel returns, and
the context stays usable."""
import numpy as np
import pytest
import torch

import hybrid_ssm_decode_gb300 as rssm
import synth
from _gpu import TOL_F32, m2_layer, m2_run_steps, vec_err

import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ns", [1_000, 20_000_000])
def test_bounded_wait_runs_out_and_reports(cuda_lib, limit_ns):
    err = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    rssm.rssm_check_bounded_wait(limit_ns, err)
    torch.cuda.synchronize()
    code, count, tile, waited = err.cpu().tolist()
    assert (code, count, tile) == (rssm.RSSM_DEV_TIMEOUT, 1, -1)
    assert waited > limit_ns


def test_context_usable_after_a_timeout(cuda_lib):
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    rssm.rssm_check_bounded_wait(5_000_000, err)
    w = synth.WORKLOADS["mamba2_fp32_b4"]
    layer, A, D = m2_layer(w)
    y = m2_run_steps(layer, w, 0, 20)
    ins = synth.mamba2_steps(w, 0, 20)
    y_ref, _ = oracle.m2_recurrence(synth.mamba2_state0(w), A, D,
                                    *(ins[k].values for k in ("x", "B", "C", "dt")))
    assert vec_err(y, y_ref) < TOL_F32
    assert layer.get_error()[0] == 0
    assert err.cpu().tolist()[0] == rssm.RSSM_DEV_TIMEOUT
