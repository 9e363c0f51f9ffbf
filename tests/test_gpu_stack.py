"""The synthetic decode stack on the GPU against the oracle's float64 stack
with the same bf16 storage points. The stack's GEMMs round their outputs to
bf16 like the oracle; an element whose float32 and float64 values round to
neighbouring bf16 values moves a layer's delta by one bf16 ulp (2^-8 of the
element), which keeps the per-vector error of the deltas below 2e-2."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu import TOL_LOW, vec_err
from hybrid_ssm_decode_gb300.stack import M2Stack, StackShape

pytestmark = pytest.mark.gpu

SHAPE = StackShape(layers=2, batch=4, heads=8, head_dim=64, state_dim=64, groups=2, k=4)


def _host(t):
    return t.double().cpu().numpy()


def _run(stack, u_steps):
    outs = []
    for u in u_steps:
        outs.append(stack.step(u))
    torch.cuda.synchronize()
    return np.stack([_host(o) for o in outs])


@pytest.mark.parametrize("mode", ["replay", "conventional"])
def test_stack_matches_oracle(cuda_lib, mode):
    S = 6                                         # crosses a flush (k = 4)
    stack = M2Stack(SHAPE, mode=mode, seed=3)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    u_steps = [torch.randn((SHAPE.batch, SHAPE.d_model), generator=g, device="cuda").to(torch.bfloat16)
               for _ in range(S)]
    weights = [{k: _host(v) for k, v in w.items()} for w in stack.weights]
    params, states = [], []
    for li in range(SHAPE.layers):
        lw = synth.Mamba2Workload(f"stack_layer{li}", batch=SHAPE.batch, heads=SHAPE.heads,
                                  head_dim=SHAPE.head_dim, state_dim=SHAPE.state_dim, groups=SHAPE.groups,
                                  k=SHAPE.k, dtype="bf16", seed=3 * 1009 + li)
        params.append(synth.mamba2_params(lw))
        states.append(synth.mamba2_state0(lw))
    got = _run(stack, u_steps)
    u_in = np.stack([_host(u) for u in u_steps])
    ref, deltas, _ = oracle.m2_stack(u_in, weights, params, states)
    # the total change over both layers, per (step, sequence)
    assert vec_err(got - u_in, ref - u_in) < TOL_LOW
    for layer in stack.layers:
        assert layer.get_error()[0] == 0
    stack.close()


def test_replay_and_conventional_stacks_agree(cuda_lib):
    S = 9
    g = torch.Generator(device="cuda")
    g.manual_seed(8)
    u_steps = [torch.randn((SHAPE.batch, SHAPE.d_model), generator=g, device="cuda").to(torch.bfloat16)
               for _ in range(S)]
    a = M2Stack(SHAPE, mode="replay", seed=4)
    b = M2Stack(SHAPE, mode="conventional", seed=4)
    ya, yb = _run(a, u_steps), _run(b, u_steps)
    u_in = np.stack([_host(u) for u in u_steps])
    assert vec_err(ya - u_in, yb - u_in) < TOL_LOW
    a.close()
    b.close()
