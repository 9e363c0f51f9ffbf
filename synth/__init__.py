"""Seeded synthetic inputs for the ReplaySSM decode path.

This module is shared by the CUDA path's tests/benchmarks and by the float64
oracle. It holds shapes, value distributions and a seeded generator, and none
of the method's arithmetic: no decay, no state update, no output formula.

Every tensor is drawn from its own stream, keyed by (seed, tensor name, step),
with numpy's PCG64 seeded through SeedSequence. The full tensor is always
generated and then sliced, so a subset of sequences sees exactly the values it
would see inside the full batch (sequences are independent, so a subset run
of the oracle is exact for those sequences).

Values are produced in float64, cast to float32, then (for bf16 workloads)
rounded to bf16 with round-to-nearest-even. Both the GPU path and the oracle
consume the *rounded* values: `Tensor.values` (float64 holding the rounded
numbers) for the oracle, `Tensor.raw` (float32 array or uint16 bf16 bit
patterns) for upload.

Distributions follow the workload descriptions (Mamba-2 and Gated DeltaNet
decode layers):
  Mamba-2: h0~N(0, 0.1^2), x~N(0,1), B,C~N(0,1)/sqrt(N), dt=softplus(N(0,1)-2)
           (times dt_scale),
           A_h=-exp(U(log 1, log 16)), D_h~N(0,1).
  GDN:     S0~N(0, 0.1^2), q,k~N(0,1) then L2-normalised in float32,
           v~N(0,1), beta=sigmoid(N(0,1)), alpha=exp(-softplus(N(0,1)-3)).
"""
from __future__ import annotations

import dataclasses
import zlib
from dataclasses import dataclass

import numpy as np

__all__ = [
    "Mamba2Workload", "GDNWorkload", "Tensor", "WORKLOADS",
    "mamba2_params", "mamba2_state0", "mamba2_step", "mamba2_steps",
    "gdn_state0", "gdn_step", "gdn_steps", "acceptance", "bf16_round",
]


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Mamba2Workload:
    name: str
    batch: int
    heads: int
    head_dim: int       # P
    state_dim: int      # N
    groups: int         # G (B/C groups)
    k: int = 16         # flush threshold (buffer records per window)
    steps: int = 64
    dtype: str = "f32"  # input/output dtype: "f32" | "bf16"
    seed: int = 0
    draft: int = 1      # T drafts per speculative round (1 = plain decode)
    accept_p: float = 0.7
    read_fmt: str = "none"  # "none" | "fp8" | "nvfp4"
    ckpt: str = "f32"       # checkpoint storage: "f32" | "f16" | "fp8" | "nvfp4"
    dt_scale: float = 1.0   # step sizes times this (small: slow decay, long memory)

    def replace(self, **kw) -> "Mamba2Workload":
        return dataclasses.replace(self, **kw)

    @property
    def state_bytes(self) -> int:
        return self.batch * self.heads * self.head_dim * self.state_dim * 4


@dataclass(frozen=True)
class GDNWorkload:
    name: str
    batch: int
    heads: int
    d_k: int
    d_v: int
    k: int = 16
    steps: int = 64
    dtype: str = "bf16"
    seed: int = 0
    scale: float = 1.0
    draft: int = 1      # T drafts per speculative round (1 = plain decode)
    accept_p: float = 0.7
    read_fmt: str = "none"  # "none" | "fp8" | "nvfp4"
    ckpt: str = "f32"       # checkpoint storage: "f32" | "f16"

    def replace(self, **kw) -> "GDNWorkload":
        return dataclasses.replace(self, **kw)

    @property
    def state_bytes(self) -> int:
        return self.batch * self.heads * self.d_v * self.d_k * 4


WORKLOADS = {
    # Mamba-2 single layer, FP32 throughout (the small parity case).
    "mamba2_fp32_b4": Mamba2Workload("mamba2_fp32_b4", batch=4, heads=8, head_dim=64,
                                     state_dim=64, groups=1, k=16, steps=64, dtype="f32"),
    # Mamba-2 serving layer: ~1 GiB FP32 checkpoint, bf16 inputs.
    "mamba2_serving_b256": Mamba2Workload("mamba2_serving_b256", batch=256, heads=128,
                                          head_dim=64, state_dim=128, groups=8, k=16,
                                          steps=256, dtype="bf16"),
    # Gated DeltaNet decode layer, 128x128 FP32 state per head.
    "gdn_serving_b256": GDNWorkload("gdn_serving_b256", batch=256, heads=32, d_k=128,
                                    d_v=128, k=16, steps=256, dtype="bf16"),
    # Speculative decode on the serving shape at batch 512, 4 drafts per round.
    "mamba2_spec_b512": Mamba2Workload("mamba2_spec_b512", batch=512, heads=128, head_dim=64,
                                       state_dim=128, groups=8, k=16, steps=128, dtype="bf16",
                                       draft=4, accept_p=0.7),
    # The same with an NVFP4 read copy that the drafts read.
    "mamba2_spec_nvfp4_b512": Mamba2Workload("mamba2_spec_nvfp4_b512", batch=512, heads=128, head_dim=64,
                                             state_dim=128, groups=8, k=16, steps=128, dtype="bf16",
                                             draft=4, accept_p=0.7, read_fmt="nvfp4"),
    # Speculative decode on the GDN serving shape at batch 512, 4 drafts per round.
    "gdn_spec_b512": GDNWorkload("gdn_spec_b512", batch=512, heads=32, d_k=128, d_v=128, k=16,
                                 steps=128, dtype="bf16", draft=4, accept_p=0.7),
    # The same with an NVFP4 read copy that the drafts read.
    "gdn_spec_nvfp4_b512": GDNWorkload("gdn_spec_nvfp4_b512", batch=512, heads=32, d_k=128, d_v=128, k=16,
                                       steps=128, dtype="bf16", draft=4, accept_p=0.7, read_fmt="nvfp4"),
    # Low-precision read copies on the serving shape.
    "mamba2_nvfp4_b256": Mamba2Workload("mamba2_nvfp4_b256", batch=256, heads=128,
                                        head_dim=64, state_dim=128, groups=8, k=16,
                                        steps=4096, dtype="bf16", read_fmt="nvfp4"),
    "mamba2_fp8_b256": Mamba2Workload("mamba2_fp8_b256", batch=256, heads=128,
                                      head_dim=64, state_dim=128, groups=8, k=16,
                                      steps=4096, dtype="bf16", read_fmt="fp8"),
    # Gated DeltaNet with a low-precision read copy (one per 64-row half).
    "gdn_fp8_b256": GDNWorkload("gdn_fp8_b256", batch=256, heads=32, d_k=128, d_v=128, k=16,
                                steps=4096, dtype="bf16", read_fmt="fp8"),
    "gdn_nvfp4_b256": GDNWorkload("gdn_nvfp4_b256", batch=256, heads=32, d_k=128, d_v=128, k=16,
                                  steps=4096, dtype="bf16", read_fmt="nvfp4"),
    # Gated DeltaNet with an FP16 checkpoint (half the checkpoint bytes).
    "gdn_f16ckpt_b256": GDNWorkload("gdn_f16ckpt_b256", batch=256, heads=32, d_k=128, d_v=128, k=16,
                                    steps=4096, dtype="bf16", ckpt="f16"),
    # FP16 checkpoint on the serving shape (half the checkpoint bytes).
    "mamba2_f16ckpt_b256": Mamba2Workload("mamba2_f16ckpt_b256", batch=256, heads=128,
                                          head_dim=64, state_dim=128, groups=8, k=16,
                                          steps=4096, dtype="bf16", ckpt="f16"),
    # The checkpoint itself in a read-copy tile format: FP8 (alone, or read
    # through an NVFP4 copy) and NVFP4.
    "mamba2_fp8ckpt_b256": Mamba2Workload("mamba2_fp8ckpt_b256", batch=256, heads=128, head_dim=64,
                                          state_dim=128, groups=8, k=16, steps=4096, dtype="bf16",
                                          ckpt="fp8"),
    "mamba2_fp8ckpt_nvfp4_b256": Mamba2Workload("mamba2_fp8ckpt_nvfp4_b256", batch=256, heads=128,
                                                head_dim=64, state_dim=128, groups=8, k=16, steps=4096,
                                                dtype="bf16", ckpt="fp8", read_fmt="nvfp4"),
    "mamba2_nvfp4ckpt_b256": Mamba2Workload("mamba2_nvfp4ckpt_b256", batch=256, heads=128, head_dim=64,
                                            state_dim=128, groups=8, k=16, steps=4096, dtype="bf16",
                                            ckpt="nvfp4"),
    # The serving shape with step sizes scaled by 0.05: the state keeps a window's
    # rounding for many windows (for the error-over-length diagnostic).
    "mamba2_slowdecay_b256": Mamba2Workload("mamba2_slowdecay_b256", batch=256, heads=128,
                                            head_dim=64, state_dim=128, groups=8, k=16, steps=4096,
                                            dtype="bf16", dt_scale=0.05),
    # FP16 checkpoint with an NVFP4 read copy.
    "mamba2_f16ckpt_nvfp4_b256": Mamba2Workload("mamba2_f16ckpt_nvfp4_b256", batch=256,
                                                heads=128, head_dim=64, state_dim=128, groups=8,
                                                k=16, steps=4096, dtype="bf16", ckpt="f16",
                                                read_fmt="nvfp4"),
}


# --------------------------------------------------------------------------
# generator
# --------------------------------------------------------------------------
def _tensor_id(name: str) -> int:
    return zlib.crc32(name.encode("ascii")) & 0x7FFFFFFF


def _rng(seed: int, name: str, step: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, _tensor_id(name), int(step) + 1])
    return np.random.Generator(np.random.PCG64(ss))


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); returns the
    uint16 bit patterns. Inputs are finite."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return rounded.astype(np.uint16)


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclass
class Tensor:
    """A generated tensor: `raw` is what the GPU receives (float32 array, or
    uint16 bf16 bit patterns), `values` the same numbers as float64."""
    raw: np.ndarray
    values: np.ndarray
    dtype: str

    def __getitem__(self, idx) -> "Tensor":
        return Tensor(self.raw[idx], self.values[idx], self.dtype)


def _finish(v64: np.ndarray, dtype: str) -> Tensor:
    f32 = v64.astype(np.float32)
    if dtype == "f32":
        return Tensor(f32, f32.astype(np.float64), "f32")
    if dtype == "bf16":
        bits = bf16_round(f32)
        return Tensor(bits, _bf16_to_f64(bits), "bf16")
    raise ValueError(dtype)


def _softplus(z: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, z)


# --------------------------------------------------------------------------
# Mamba-2
# --------------------------------------------------------------------------
def mamba2_params(w: Mamba2Workload):
    """Per-head A_h (<0) and D_h, float32 (layer parameters)."""
    u = _rng(w.seed, "A", 0).uniform(np.log(1.0), np.log(16.0), size=w.heads)
    A = (-np.exp(u)).astype(np.float32)
    D = _rng(w.seed, "D", 0).standard_normal(w.heads).astype(np.float32)
    return A, D


def mamba2_state0(w: Mamba2Workload) -> np.ndarray:
    """Initial FP32 state h0 [B][H][P][N] ~ N(0, 0.1^2)."""
    shape = (w.batch, w.heads, w.head_dim, w.state_dim)
    return (0.1 * _rng(w.seed, "h0", 0).standard_normal(shape)).astype(np.float32)


def mamba2_step(w: Mamba2Workload, step: int) -> dict:
    """Inputs of one token position for every sequence:
    x [B][H][P], B [B][G][N], C [B][G][N], dt [B][H] (all in w.dtype)."""
    B, H, P, N, G = w.batch, w.heads, w.head_dim, w.state_dim, w.groups
    x = _rng(w.seed, "x", step).standard_normal((B, H, P))
    bm = _rng(w.seed, "B", step).standard_normal((B, G, N)) / np.sqrt(N)
    c = _rng(w.seed, "C", step).standard_normal((B, G, N)) / np.sqrt(N)
    dt = _softplus(_rng(w.seed, "dt", step).standard_normal((B, H)) - 2.0)
    if w.dt_scale != 1.0:
        dt = dt * w.dt_scale
    return {"x": _finish(x, w.dtype), "B": _finish(bm, w.dtype),
            "C": _finish(c, w.dtype), "dt": _finish(dt, w.dtype)}


def _stack(parts: list, dtype: str) -> Tensor:
    return Tensor(np.stack([p.raw for p in parts]), np.stack([p.values for p in parts]), dtype)


def mamba2_steps(w: Mamba2Workload, start: int, count: int) -> dict:
    """Steps [start, start+count) stacked on a leading axis: x [S][B][H][P] ..."""
    per = [mamba2_step(w, s) for s in range(start, start + count)]
    return {key: _stack([p[key] for p in per], w.dtype) for key in ("x", "B", "C", "dt")}


def acceptance(batch: int, rounds: int, draft: int, p: float, seed: int = 0) -> np.ndarray:
    """Accepted draft counts a[round][b] in 0..draft: consecutive Bernoulli(p)
    acceptances stopped at the first rejection (truncated geometric),
    P(a=j) = p^j (1-p) for j<draft, P(a=draft) = p^draft. int32."""
    u = _rng(seed, "accept", 0).uniform(size=(rounds, batch, draft))
    ok = u < p
    # a = index of the first rejection, or `draft` when all are accepted
    first_reject = np.where(ok.all(axis=2), draft, np.argmin(ok, axis=2))
    return first_reject.astype(np.int32)


# --------------------------------------------------------------------------
# Gated DeltaNet
# --------------------------------------------------------------------------
def gdn_state0(w: GDNWorkload) -> np.ndarray:
    """Initial FP32 state S0 [B][H][d_v][d_k] ~ N(0, 0.1^2)."""
    shape = (w.batch, w.heads, w.d_v, w.d_k)
    return (0.1 * _rng(w.seed, "S0", 0).standard_normal(shape)).astype(np.float32)


def _l2norm_f32(a: np.ndarray) -> np.ndarray:
    a = a.astype(np.float32)
    n = np.sqrt(np.sum(a * a, axis=-1, keepdims=True, dtype=np.float32))
    return (a / n).astype(np.float32)


def gdn_step(w: GDNWorkload, step: int) -> dict:
    """q,k [B][H][d_k], v [B][H][d_v] in w.dtype; alpha, beta [B][H] float32."""
    B, H = w.batch, w.heads
    q = _l2norm_f32(_rng(w.seed, "q", step).standard_normal((B, H, w.d_k)))
    k = _l2norm_f32(_rng(w.seed, "k", step).standard_normal((B, H, w.d_k)))
    v = _rng(w.seed, "v", step).standard_normal((B, H, w.d_v))
    beta = 1.0 / (1.0 + np.exp(-_rng(w.seed, "beta", step).standard_normal((B, H))))
    alpha = np.exp(-_softplus(_rng(w.seed, "alpha", step).standard_normal((B, H)) - 3.0))
    return {"q": _finish(q, w.dtype), "k": _finish(k, w.dtype), "v": _finish(v, w.dtype),
            "alpha": _finish(alpha, "f32"), "beta": _finish(beta, "f32")}


def gdn_steps(w: GDNWorkload, start: int, count: int) -> dict:
    per = [gdn_step(w, s) for s in range(start, start + count)]
    out = {}
    for key in ("q", "k", "v", "alpha", "beta"):
        out[key] = _stack([p[key] for p in per], per[0][key].dtype)
    return out
