"""A synthetic decode stack around the Mamba-2 SSM layer.

The pages set the SSM-kernel speedup beside a smaller speedup of the whole
decode step ("ReplaySSM beschleunigt das Decoding von Hybridmodellen ...",
section "Wichtige Details"; "NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu",
section "Durum trafiğini azaltma ve rollback'ın basitleştirilmesi"): the SSM
layer is one part of a step that also runs the layer's projections. This
module builds that step from random-weight parts, so the SSM layer's share
and the step-level speedup can be measured without a trained model.

One layer, for the hidden state u [B][d_model] (bf16), with d_inner = H * P
and d_model = d_inner / 2 (the Mamba-2 expansion factor of 2):

    n  = u / rms(u)                                  RMS normalisation
    x  = n W_x,  z = n W_z                           [B][d_inner] = [B][H][P]
    Bt = n W_B,  Ct = n W_C                          [B][G][N]
    dt = softplus(n W_dt + dt_bias)                  [B][H]
    y  = SSM decode step (x, Bt, Ct, dt)             librssm, this layer's state
    u  = u + (y * silu(z)) W_out                     residual

The projections are plain bf16 GEMMs (cuBLAS through torch.matmul) and the
element-wise steps are torch operations: they are the same in the replay and
conventional stacks, which differ only in the SSM layer's mode. Weights are
N(0, 1/fan_in), drawn from a seeded torch generator on the device.
"""
from __future__ import annotations

from dataclasses import dataclass

import synth

from . import Layer, make_config


@dataclass(frozen=True)
class StackShape:
    layers: int
    batch: int
    heads: int = 128
    head_dim: int = 64
    state_dim: int = 128
    groups: int = 8
    k: int = 16

    @property
    def d_inner(self) -> int:
        return self.heads * self.head_dim

    @property
    def d_model(self) -> int:
        return self.d_inner // 2


class M2Stack:
    """`shape.layers` Mamba-2 layers with random projections on one GPU.

    mode: "replay" or "conventional" (the SSM layer's mode); ckpt / read_fmt
    as in make_config. The weights depend on `seed` only, so two stacks with
    the same seed and different modes compute the same function.
    """

    def __init__(self, shape: StackShape, mode="replay", ckpt="f32", read_fmt="none", seed=0,
                 device="cuda"):
        import torch
        self.shape, self.mode = shape, mode
        s = shape
        gen = torch.Generator(device=device)
        gen.manual_seed(1000 + seed)

        def weight(rows, cols):
            w = torch.randn((rows, cols), generator=gen, device=device, dtype=torch.float32)
            return (w / rows ** 0.5).to(torch.bfloat16)

        self.weights = []
        self.layers = []
        for li in range(s.layers):
            w = {"x": weight(s.d_model, s.d_inner), "z": weight(s.d_model, s.d_inner),
                 "B": weight(s.d_model, s.groups * s.state_dim),
                 "C": weight(s.d_model, s.groups * s.state_dim),
                 "dt": weight(s.d_model, s.heads),
                 "out": weight(s.d_inner, s.d_model)}
            # dt_bias puts softplus(dt) near the synthetic workload's step sizes
            w["dt_bias"] = (torch.rand((s.heads,), generator=gen, device=device) * 2.0 - 4.0)
            self.weights.append(w)
            lw = synth.Mamba2Workload(f"stack_layer{li}", batch=s.batch, heads=s.heads,
                                      head_dim=s.head_dim, state_dim=s.state_dim, groups=s.groups,
                                      k=s.k, dtype="bf16", seed=seed * 1009 + li)
            A, D = synth.mamba2_params(lw)
            h0 = torch.from_numpy(synth.mamba2_state0(lw)).to(device)
            cfg = make_config(kind="mamba2", mode=mode, batch=s.batch, heads=s.heads,
                              head_dim=s.head_dim, state_dim=s.state_dim, groups=s.groups, k=s.k,
                              in_dtype="bf16", read_fmt=read_fmt, ckpt_dtype=ckpt)
            self.layers.append(Layer(cfg, torch.from_numpy(A).to(device), torch.from_numpy(D).to(device),
                                     h0))
        self.y = torch.empty((s.batch, 1, s.heads, s.head_dim), dtype=torch.bfloat16, device=device)

    def close(self):
        for layer in self.layers:
            layer.close()

    def step(self, u):
        """One decode step of every layer for the embeddings u [B][d_model]
        (bf16); returns the last layer's hidden state."""
        import torch
        import torch.nn.functional as F
        s = self.shape
        for w, layer in zip(self.weights, self.layers):
            uf = u.float()
            n = (uf * torch.rsqrt(uf.pow(2).mean(-1, keepdim=True) + 1e-6)).to(torch.bfloat16)
            x = n @ w["x"]
            z = n @ w["z"]
            Bt = n @ w["B"]
            Ct = n @ w["C"]
            dt = F.softplus((n @ w["dt"]).float() + w["dt_bias"]).to(torch.bfloat16)
            layer.decode_step(self.y, 1, x=x, Bm=Bt, C=Ct, dt=dt)
            g = self.y.view(s.batch, s.d_inner) * F.silu(z)
            u = u + g @ w["out"]
        return u

    def ssm_inputs(self, u):
        """The SSM layers' inputs (x, B, C, dt) for the embeddings u, per layer,
        with u passed through unchanged (to time the SSM layers alone)."""
        import torch
        import torch.nn.functional as F
        out = []
        for w in self.weights:
            uf = u.float()
            n = (uf * torch.rsqrt(uf.pow(2).mean(-1, keepdim=True) + 1e-6)).to(torch.bfloat16)
            dt = F.softplus((n @ w["dt"]).float() + w["dt_bias"]).to(torch.bfloat16)
            out.append((n @ w["x"], n @ w["B"], n @ w["C"], dt))
        return out
