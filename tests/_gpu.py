"""Shared helpers for the GPU parity tests: upload synthetic inputs, run the
library through its C ABI, and compare with the oracle.

Error metric: for each output vector (one (step, sequence, head)), the
max-norm of the difference divided by the max-norm of the oracle's vector;
the reported error is the maximum over all vectors. States are compared the
same way per (sequence, head) tile.
"""
import numpy as np
import torch

import hybrid_ssm_decode_gb300 as rssm
import synth

TOL_F32 = 1e-4      # FP32 arithmetic paths
TOL_LOW = 2e-2      # bf16 outputs, FP8/NVFP4 read copies


def dev(t):
    """synth.Tensor (or numpy array) -> torch CUDA tensor with the raw bits."""
    raw = t.raw if isinstance(t, synth.Tensor) else t
    raw = np.ascontiguousarray(raw)
    if raw.dtype == np.uint16:
        return torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(raw).cuda()


def vec_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over vectors (last axis) of |got-ref|_inf / |ref|_inf."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.max(np.abs(got - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)
    return float(np.max(num / den))


def tile_err(got: np.ndarray, ref: np.ndarray) -> float:
    """Per (sequence, head) tile of a [B][H][R][C] state."""
    s = got.shape
    return vec_err(np.reshape(got, s[:2] + (-1,)), np.reshape(ref, s[:2] + (-1,)))


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def m2_layer(w: synth.Mamba2Workload, mode="replay", out_dtype=None, k=None, max_draft=None,
             read_fmt=None, state0=True, ckpt=None):
    A, D = synth.mamba2_params(w)
    cfg = rssm.make_config(kind="mamba2", mode=mode, batch=w.batch, heads=w.heads,
                           head_dim=w.head_dim, state_dim=w.state_dim, groups=w.groups,
                           k=w.k if k is None else k,
                           max_draft=w.draft if max_draft is None else max_draft,
                           in_dtype=w.dtype, out_dtype=out_dtype,
                           read_fmt=w.read_fmt if read_fmt is None else read_fmt,
                           ckpt_dtype=w.ckpt if ckpt is None else ckpt)
    dA, dD = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    h0 = dev(synth.mamba2_state0(w)) if state0 else None
    layer = rssm.Layer(cfg, dA, dD, h0)
    return layer, A, D


def m2_out(w, T=1, out_dtype=None):
    dt = torch.float32 if (out_dtype or w.dtype) == "f32" else torch.bfloat16
    return torch.empty((w.batch, T, w.heads, w.head_dim), dtype=dt, device="cuda")


def m2_run_steps(layer, w, start, count, out_dtype=None, return_inputs=False):
    """Plain decode of steps [start, start+count); returns y [S][B][H][P] (float64)."""
    ys = []
    ins = synth.mamba2_steps(w, start, count)
    for s in range(count):
        y = m2_out(w, 1, out_dtype)
        layer.decode_step(y, 1, x=dev(ins["x"][s]), Bm=dev(ins["B"][s]), C=dev(ins["C"][s]),
                          dt=dev(ins["dt"][s]))
        ys.append(y[:, 0])
    out = np.stack([host(y) for y in ys])
    return (out, ins) if return_inputs else out


def gdn_layer(w: synth.GDNWorkload, mode="replay", out_dtype=None, k=None, read_fmt=None, ckpt="f32"):
    cfg = rssm.make_config(kind="gdn", mode=mode, batch=w.batch, heads=w.heads, head_dim=w.d_v,
                           state_dim=w.d_k, groups=1, k=w.k if k is None else k, max_draft=1,
                           in_dtype=w.dtype, out_dtype=out_dtype, gdn_scale=w.scale,
                           read_fmt=w.read_fmt if read_fmt is None else read_fmt, ckpt_dtype=ckpt)
    return rssm.Layer(cfg, None, None, dev(synth.gdn_state0(w)))


def gdn_run_steps(layer, w, start, count, out_dtype=None):
    dt = torch.float32 if (out_dtype or w.dtype) == "f32" else torch.bfloat16
    ins = synth.gdn_steps(w, start, count)
    ys = []
    for s in range(count):
        o = torch.empty((w.batch, 1, w.heads, w.d_v), dtype=dt, device="cuda")
        layer.decode_step(o, 1, q=dev(ins["q"][s]), k=dev(ins["k"][s]), v=dev(ins["v"][s]),
                          alpha=dev(ins["alpha"][s]), beta=dev(ins["beta"][s]))
        ys.append(o[:, 0])
    return np.stack([host(o) for o in ys])


def m2_copy_regions(layer, w, sub=slice(None)):
    """The Mamba-2 read copy in the workspace: codes, block scales (NVFP4,
    else None) and tile scales of the tiles of sequences `sub`, as numpy
    arrays [tiles][P][...], [tiles][P][N/16], [tiles]."""
    lay, ws = layer.layout, layer.workspace
    P, N = w.head_dim, w.state_dim
    codes = ws[lay.rc_codes:lay.rc_codes + lay.rc_codes_bytes].view(w.batch, w.heads, P, -1)[sub]
    ts = ws[lay.rc_tscale:lay.rc_tscale + lay.rc_tscale_bytes].view(torch.float32).view(w.batch, w.heads)[sub]
    bsc = None
    if lay.rc_bscale_bytes:
        bsc = ws[lay.rc_bscale:lay.rc_bscale + lay.rc_bscale_bytes].view(w.batch, w.heads, P, N // 16)[sub]
        bsc = bsc.cpu().numpy().reshape(-1, P, N // 16)
    return codes.cpu().numpy().reshape(-1, P, codes.shape[-1]), bsc, ts.cpu().numpy().reshape(-1)
