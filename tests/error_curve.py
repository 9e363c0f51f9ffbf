#!/usr/bin/env python3
"""Output error of the read-copy and low-precision-checkpoint paths over a long
decode, on the GPU, against the float64 oracle (test infrastructure: it runs
the oracle, so it lives with the tests and not in the benchmark).

    python tests/error_curve.py --steps 4096 [--workload mamba2_slowdecay_b256 | gdn_serving_b256]

Prints one JSON line.
"""
import argparse
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from bench import to_dev, workload  # noqa: E402


def error_curve(args):
    """Output error of the read-copy paths against the FP32 recurrence as the
    decode grows long: FP32 checkpoint alone, FP8 copy, NVFP4 copy, and the
    quantised-recurrence baseline (state kept in FP8 / NVFP4). The GPU
    runs all B sequences; 8 evenly spaced sequences are checked against the
    float64 oracle. Inputs cycle through a pool of 64 steps (a multiple of k,
    so every oracle chunk starts at a flush). Errors are the max over the
    checked (sequence, head) vectors at each marked step: of the whole output,
    and of the output minus its D x skip term. The marks are the last
    non-flush token of a window (15, 63, 255, ... tokens decoded), whose output
    reads a copy made 15 tokens earlier."""
    import torch
    import oracle
    import hybrid_ssm_decode_gb300 as rssm
    base = workload(args)
    S = args.steps
    # tokens decoded so far at each mark: the last non-flush token of a window
    # (the flush token's output reads the FP32 checkpoint, not the copy)
    marks = [m - 1 for m in (16, 64, 256, 1024, 4096, 16384) if m <= S]
    pool = 64
    B = base.batch
    sub = np.unique(np.linspace(0, B - 1, 8).astype(int))
    steps = synth.mamba2_steps(base, 0, pool)
    A, D = synth.mamba2_params(base)
    device = torch.device("cuda", 0)
    dA, dD = torch.from_numpy(A).to(device), torch.from_numpy(D).to(device)
    h0 = synth.mamba2_state0(base)
    dh0 = to_dev(torch, synth.Tensor(h0, None, "f32"), device)
    dins = {k: to_dev(torch, steps[k], device) for k in ("x", "B", "C", "dt")}
    sub_t = torch.from_numpy(sub).to(device)

    def gpu_run(read_fmt, mode="replay", ckpt="f32"):
        cfg = rssm.make_config(kind="mamba2", mode=mode, batch=B, heads=base.heads, head_dim=base.head_dim,
                               state_dim=base.state_dim, groups=base.groups, k=base.k, in_dtype=base.dtype,
                               out_dtype="f32", read_fmt=read_fmt, ckpt_dtype=ckpt)
        layer = rssm.Layer(cfg, dA, dD, dh0)
        y = torch.empty((B, 1, base.heads, base.head_dim), dtype=torch.float32, device=device)
        got = {}
        for s in range(S):
            j = s % pool
            layer.decode_step(y, 1, x=dins["x"][j], Bm=dins["B"][j], C=dins["C"][j], dt=dins["dt"][j])
            if s + 1 in marks:
                got[s + 1] = y[sub_t, 0].double().cpu().numpy()
        if layer.get_error()[0]:
            raise RuntimeError("device error word set")
        layer.close()
        return got

    runs = {fmt: gpu_run(fmt) for fmt in ("none", "fp8", "nvfp4")}
    # the quantised-recurrence baseline: the state itself kept in the format
    qruns = {fmt: gpu_run(fmt, "conventional") for fmt in ("fp8", "nvfp4")}
    # FP16 checkpoint, alone and under an NVFP4 read copy; FP8 checkpoint under
    # an NVFP4 copy; NVFP4 checkpoint (read itself)
    runs16 = {fmt: gpu_run(fmt, ckpt="f16") for fmt in ("none", "nvfp4")}
    run_fp8ck = gpu_run("nvfp4", ckpt="fp8")
    run_nvck = gpu_run("none", ckpt="nvfp4")
    # the oracle on the checked sequences, one pool-long chunk at a time
    vals = {k: steps[k].values[:, sub] for k in ("x", "B", "C", "dt")}
    truth, emul, emul16, emul8 = {}, {"fp8": {}, "nvfp4": {}}, {}, {}
    h = h0[sub].astype(np.float64)
    ck16 = h.copy()
    ck8 = h.copy()
    t0 = time.perf_counter()
    for c0 in range(0, S, pool):
        n = min(pool, S - c0)
        args_c = [vals[k][:n] for k in ("x", "B", "C", "dt")]
        want = [m for m in marks if c0 < m <= c0 + n]
        if want:
            for fmt in ("fp8", "nvfp4"):
                ye = oracle.m2_readcopy(h, A, D, *args_c, k=base.k, fmt=fmt)
                for m in want:
                    emul[fmt][m] = ye[m - c0 - 1]
        y, h = oracle.m2_recurrence(h, A, D, *args_c)
        for m in want:
            truth[m] = y[m - c0 - 1]
        # the chunk is a whole number of windows, so the FP16 checkpoint chains
        y16, ck16 = oracle.m2_ckpt16(ck16, A, D, *args_c, k=base.k)
        y8, ck8 = oracle.m2_ckpt_lowp(ck8, A, D, *args_c, base.k, "fp8", fmt="nvfp4", start_stored=c0 > 0)
        for m in want:
            emul16[m] = y16[m - c0 - 1]
            emul8[m] = y8[m - c0 - 1]
    # the quantised recurrence in float64 on two of the checked sequences, up
    # to the 1023rd token (numpy over the quantisers: slower than the C paths)
    qsub = 2
    qmarks = [m for m in marks if m <= 1023]
    qref = {"fp8": {}, "nvfp4": {}}
    if qmarks:
        n = max(qmarks)
        reps = (n + pool - 1) // pool
        qin = [np.concatenate([vals[k][:, :qsub]] * reps)[:n] for k in ("x", "B", "C", "dt")]
        for fmt in ("fp8", "nvfp4"):
            yq = oracle.m2_qrecurrence(h0[sub[:qsub]], A, D, *qin, fmt)
            for m in qmarks:
                qref[fmt][m] = yq[m - 1]
    oracle_s = time.perf_counter() - t0

    def err(got, ref, skip):
        num = np.max(np.abs(got - ref), axis=-1)
        return float(np.max(num / np.maximum(np.max(np.abs(ref), axis=-1), 1e-30))), \
            float(np.max(num / np.maximum(np.max(np.abs(ref - skip), axis=-1), 1e-30)))

    curve = []
    for m in marks:
        j = (m - 1) % pool
        skip = D[None, :, None] * steps["x"].values[j][sub]          # D_h x_t of the checked vectors
        row = {"step": m}
        for fmt in ("none", "fp8", "nvfp4"):
            e, es = err(runs[fmt][m], truth[m], skip)
            row[f"gpu_{fmt}"] = e
            row[f"gpu_{fmt}_state_term"] = es
        for fmt in ("fp8", "nvfp4"):
            e, es = err(emul[fmt][m], truth[m], skip)
            row[f"oracle_{fmt}_emulation"] = e
            row[f"oracle_{fmt}_emulation_state_term"] = es
            e, es = err(qruns[fmt][m], truth[m], skip)
            row[f"gpu_quantised_recurrence_{fmt}"] = e
            row[f"gpu_quantised_recurrence_{fmt}_state_term"] = es
            if m in qref[fmt]:
                e, _ = err(qruns[fmt][m][:qsub], qref[fmt][m], skip[:qsub])
                row[f"gpu_vs_oracle_quantised_recurrence_{fmt}"] = e
        for fmt in ("none", "nvfp4"):
            e, es = err(runs16[fmt][m], truth[m], skip)
            row[f"gpu_f16ckpt_{fmt}"] = e
            row[f"gpu_f16ckpt_{fmt}_state_term"] = es
        e, es = err(emul16[m], truth[m], skip)
        row["oracle_f16ckpt_emulation"] = e
        row["oracle_f16ckpt_emulation_state_term"] = es
        e, _ = err(runs16["none"][m], emul16[m], skip)
        row["gpu_vs_oracle_f16ckpt"] = e
        e, es = err(run_fp8ck[m], truth[m], skip)
        row["gpu_fp8ckpt_nvfp4"] = e
        row["gpu_fp8ckpt_nvfp4_state_term"] = es
        e, _ = err(run_fp8ck[m], emul8[m], skip)
        row["gpu_vs_oracle_fp8ckpt_nvfp4"] = e
        e, es = err(run_nvck[m], truth[m], skip)
        row["gpu_nvfp4ckpt"] = e
        row["gpu_nvfp4ckpt_state_term"] = es
        curve.append(row)
    print(json.dumps({"diagnostic": "read-copy error vs decode length", "workload": base.name, "batch": B,
                      "checked_sequences": sub.tolist(), "k": base.k, "input_pool_steps": pool,
                      "oracle_seconds": oracle_s, "curve": curve}), flush=True)


def gdn_error_curve(args):
    """The Gated DeltaNet form of error_curve: the FP32 checkpoint alone, the
    FP8 and NVFP4 read copies (one copy tile per 64-row half), the FP16
    checkpoint and the quantised-recurrence baseline (the state kept in the
    copy tiles), against
    the float64 recurrence on 8 checked sequences; the oracle's read-copy
    emulation, and on two sequences up to token 1023 the oracle's quantised
    recurrence, beside them."""
    import torch
    import oracle
    import hybrid_ssm_decode_gb300 as rssm
    base = workload(args)
    S = args.steps
    marks = [m - 1 for m in (16, 64, 256, 1024, 4096, 16384) if m <= S]
    pool = 64
    B = base.batch
    sub = np.unique(np.linspace(0, B - 1, 8).astype(int))
    keys = ("q", "k", "v", "alpha", "beta")
    steps = synth.gdn_steps(base, 0, pool)
    device = torch.device("cuda", 0)
    S0 = synth.gdn_state0(base)
    dS0 = to_dev(torch, synth.Tensor(S0, None, "f32"), device)
    dins = {k: to_dev(torch, steps[k], device) for k in keys}
    sub_t = torch.from_numpy(sub).to(device)

    def gpu_run(read_fmt, mode="replay", ckpt="f32"):
        cfg = rssm.make_config(kind="gdn", mode=mode, batch=B, heads=base.heads, head_dim=base.d_v,
                               state_dim=base.d_k, groups=1, k=base.k, in_dtype=base.dtype, out_dtype="f32",
                               gdn_scale=base.scale, read_fmt=read_fmt, ckpt_dtype=ckpt)
        layer = rssm.Layer(cfg, None, None, dS0)
        o = torch.empty((B, 1, base.heads, base.d_v), dtype=torch.float32, device=device)
        got = {}
        for s in range(S):
            j = s % pool
            layer.decode_step(o, 1, **{k: dins[k][j] for k in keys})
            if s + 1 in marks:
                got[s + 1] = o[sub_t, 0].double().cpu().numpy()
        if layer.get_error()[0]:
            raise RuntimeError("device error word set")
        layer.close()
        return got

    runs = {fmt: gpu_run(fmt) for fmt in ("none", "fp8", "nvfp4")}
    qruns = {fmt: gpu_run(fmt, "conventional") for fmt in ("fp8", "nvfp4")}
    run16 = gpu_run("none", ckpt="f16")
    vals = {k: steps[k].values[:, sub] for k in keys}
    truth, emul, emul16 = {}, {"fp8": {}, "nvfp4": {}}, {}
    St = S0[sub].astype(np.float64)
    ck16 = St.copy()
    t0 = time.perf_counter()
    for c0 in range(0, S, pool):
        n = min(pool, S - c0)
        args_c = [vals[k][:n] for k in keys]
        want = [m for m in marks if c0 < m <= c0 + n]
        if want:
            for fmt in ("fp8", "nvfp4"):
                oe, _ = oracle.gdn_readcopy(St, *args_c, base.k, fmt, scale=base.scale)
                for m in want:
                    emul[fmt][m] = oe[m - c0 - 1]
        o, St = oracle.gdn_recurrence(St, *args_c, scale=base.scale)
        for m in want:
            truth[m] = o[m - c0 - 1]
        # the chunk is a whole number of windows, so the FP16 checkpoint chains
        o16, ck16 = oracle.gdn_ckpt16(ck16, *args_c, base.k, scale=base.scale)
        for m in want:
            emul16[m] = o16[m - c0 - 1]
    qsub = 2
    qmarks = [m for m in marks if m <= 1023]
    qref = {"fp8": {}, "nvfp4": {}}
    if qmarks:
        n = max(qmarks)
        reps = (n + pool - 1) // pool
        qin = [np.concatenate([vals[k][:, :qsub]] * reps)[:n] for k in keys]
        for fmt in ("fp8", "nvfp4"):
            oq = oracle.gdn_qrecurrence(S0[sub[:qsub]], *qin, fmt, scale=base.scale)
            for m in qmarks:
                qref[fmt][m] = oq[m - 1]
    oracle_s = time.perf_counter() - t0

    def err(got, ref):
        num = np.max(np.abs(got - ref), axis=-1)
        return float(np.max(num / np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)))

    curve = []
    for m in marks:
        row = {"step": m}
        for fmt in ("none", "fp8", "nvfp4"):
            row[f"gpu_{fmt}"] = err(runs[fmt][m], truth[m])
        for fmt in ("fp8", "nvfp4"):
            row[f"oracle_{fmt}_emulation"] = err(emul[fmt][m], truth[m])
            row[f"gpu_quantised_recurrence_{fmt}"] = err(qruns[fmt][m], truth[m])
            if m in qref[fmt]:
                row[f"gpu_vs_oracle_quantised_recurrence_{fmt}"] = err(qruns[fmt][m][:qsub], qref[fmt][m])
        row["gpu_f16ckpt"] = err(run16[m], truth[m])
        row["oracle_f16ckpt_emulation"] = err(emul16[m], truth[m])
        row["gpu_vs_oracle_f16ckpt"] = err(run16[m], emul16[m])
        curve.append(row)
    print(json.dumps({"diagnostic": "GDN read-copy error vs decode length", "workload": base.name, "batch": B,
                      "checked_sequences": sub.tolist(), "k": base.k, "input_pool_steps": pool,
                      "oracle_seconds": oracle_s, "curve": curve}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--workload", default="mamba2_serving_b256",
                    choices=[k for k, w in synth.WORKLOADS.items() if "spec" not in k])
    ap.add_argument("--k", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0)
    args = ap.parse_args()
    if isinstance(synth.WORKLOADS[args.workload], synth.GDNWorkload):
        gdn_error_curve(args)
    else:
        error_curve(args)


if __name__ == "__main__":
    main()
