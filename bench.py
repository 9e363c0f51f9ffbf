#!/usr/bin/env python3
"""Benchmark of the ReplaySSM decode step (librssm) on GB300.

Default workload: the Mamba-2 serving layer, B=256, H=128, P=64, N=128, G=8,
bf16 inputs, FP32 checkpoint (1 GiB), k=16. One timed step = one decode step
of all 256 sequences (one kernel launch), inputs resident in HBM. The
checkpoint (1 GiB) is larger than L2 (129 MB) and is streamed every step, so
no extra L2 flush is needed between steps.

Prints one JSON line (rank 0):
  value        tokens/s over all ranks (B x K x N / max-over-ranks time)
  roofline     the replay step kernel: algorithmic bytes per launch / its mean
               CUDA-event duration, against the measured HBM copy bandwidth
  e2e          the same metric through the C ABI with host buffers: pinned
               host->device copies of each step's inputs and device->host copies
               of its outputs inside the timed region
  cpu_baseline the float64 oracle on the host cores, on a sample
  conventional the in-build conventional kernel on the same steps

--impl reference times the float64 oracle (the plain per-token recurrence) on
the host cores instead, on a bounded sample of the same workload per step.
Other workloads: --workload gdn_serving_b256 | mamba2_spec_b512 | mamba2_spec_nvfp4_b512 |
gdn_spec_b512 | gdn_spec_nvfp4_b512 | mamba2_nvfp4_b256 | mamba2_fp8_b256 | mamba2_f16ckpt_b256 |
mamba2_f16ckpt_nvfp4_b256 | mamba2_fp8ckpt_b256 | mamba2_fp8ckpt_nvfp4_b256 |
mamba2_nvfp4ckpt_b256 | gdn_fp8_b256 | gdn_nvfp4_b256 | gdn_f16ckpt_b256, --k for the k sweep, --batch for the batch sweep.
Diagnostic (one JSON line, not the contract line): --stack L times a synthetic
L-layer decode stack (random projections around the SSM layers), replay against
conventional.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "SSM-layer decode tokens/s at batch 256; achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic bytes per launch (what must cross HBM at least once)
# ---------------------------------------------------------------------------
def m2_step_bytes(w: synth.Mamba2Workload, c: int, flush: bool, mode: str, read_fmt: str,
                  out_size: int, ckpt: str = "f32") -> float:
    """Bytes of one plain decode launch over all B*H tiles, with c records
    already buffered per tile. B/C records and inputs are per group (shared
    by H/G heads) and counted once. ckpt: checkpoint storage ("f32"/"f16")."""
    B, H, P, N, G = w.batch, w.heads, w.head_dim, w.state_dim, w.groups
    s = 4 if w.dtype == "f32" else 2
    hpg = H / G
    state = {"f32": P * N * 4, "f16": P * N * 2, "fp8": P * N + 4, "nvfp4": P * N / 2 + P * N / 16 + 4}[ckpt]
    tok_in = P * s + s + 2 * N * s / hpg           # x_t, dt_t, B_t + C_t (group share)
    tok_out = P * out_size
    if mode == "conventional":
        return B * H * (2 * state + tok_in + tok_out)
    rc = {"none": 0, "fp8": P * N + 4, "nvfp4": P * N / 2 + P * N / 16 + 4}[read_fmt]
    read = state if (read_fmt == "none" or flush) else rc
    record = P * s + s + N * s / hpg
    per_tile = read + c * record + tok_in + tok_out + 8
    if flush:
        per_tile += state + rc
    else:
        per_tile += record
    return B * H * per_tile


def gdn_step_bytes(w: synth.GDNWorkload, c: int, flush: bool, mode: str, out_size: int,
                   read_fmt: str = "none", ckpt: str = "f32") -> float:
    """Bytes of one GDN decode launch over all B*H tiles, with c records
    buffered per tile. With a read copy the non-flush launch reads the copy
    (one scale per 64-row half) and the records also keep v and beta.
    ckpt: checkpoint storage ("f32"/"f16")."""
    B, H, DK, DV = w.batch, w.heads, w.d_k, w.d_v
    s = 4 if w.dtype == "f32" else 2
    state = DV * DK * (2 if ckpt == "f16" else 4)
    tok_in = 2 * DK * s + DV * s + 8                # q, k, v, alpha, beta
    tok_out = DV * out_size
    if mode == "conventional":
        return B * H * (2 * state + tok_in + tok_out)
    rc = {"none": 0, "fp8": DV * DK + DV / 16, "nvfp4": DV * DK / 2 + DV * DK / 16 + DV / 16}[read_fmt]
    record = DK * s + DV * 4 + 4                    # k_j, u_j, alpha_j
    if read_fmt != "none":
        record += DV * s + 4                        # v_j, beta_j
    read = state if (read_fmt == "none" or flush) else rc
    per_tile = read + c * record + tok_in + tok_out + 8
    per_tile += (state + rc) if flush else record
    return B * H * per_tile


def roofline_of(res, mode: str, warmup: int, peak: float, peak_kind: str) -> dict:
    """Roofline of the dominant kernel of an arm's result. Plain replay decode
    runs the lean non-flush kernel on k-1 of every k steps and the fused
    kernel on the flush step: the former is the dominant kernel, the latter is
    reported beside it ("split"), and so is the mean over all timed launches."""
    w = res["w"]
    per, byts = res["per"], res["bytes"]
    kernel_ms = sum(per)
    achieved = (sum(byts) / len(byts)) / (kernel_ms / len(per) / 1e3) / 1e9
    kernel = res.get("kernel", "replay step")
    dom_bytes, dom_ms, dom_n = sum(byts) / len(byts), kernel_ms / len(per), len(per)
    split = None
    if "flush_mask" not in res and mode == "replay":
        k, nl = w.k, res.get("layers", 1)   # launch j is its layer's (j // nl)-th step
        nf = [(p, b) for i, (p, b) in enumerate(zip(per, byts)) if ((warmup + i) // nl) % k != k - 1]
        fl = [(p, b) for i, (p, b) in enumerate(zip(per, byts)) if ((warmup + i) // nl) % k == k - 1]
        split = {}
        for name, lst in (("non_flush", nf), ("flush", fl)):
            if lst:
                ms = sum(p for p, _ in lst) / len(lst)
                gbs = sum(b for _, b in lst) / len(lst) / (ms / 1e3) / 1e9
                split[name] = {"launches": len(lst), "mean_us": ms * 1e3, "gbs": gbs, "frac": gbs / peak}
        if nf:
            dom_n = len(nf)
            dom_ms = sum(p for p, _ in nf) / dom_n
            dom_bytes = sum(b for _, b in nf) / dom_n
            kernel = res["nf_kernel"]
    dom_gbs = dom_bytes / (dom_ms / 1e3) / 1e9
    out = {"bound": "hbm", "achieved": dom_gbs, "peak": peak, "unit": "GB/s",
           "frac": dom_gbs / peak, "traffic": profiled_traffic(kernel, w),
           "kernel": kernel, "launches": dom_n, "mean_us": dom_ms * 1e3,
           "algorithmic_bytes_per_launch": dom_bytes, "peak_source": peak_kind,
           "all_launches": {"gbs": achieved, "frac": achieved / peak}}
    if split:
        out["split"] = split
    return out


# ---------------------------------------------------------------------------
# further workloads, measured briefly inside the default run
# ---------------------------------------------------------------------------
SUB_WORKLOADS = ("gdn_serving_b256", "mamba2_spec_b512", "mamba2_spec_nvfp4_b512", "gdn_spec_b512",
                 "gdn_spec_nvfp4_b512", "mamba2_fp8_b256", "mamba2_nvfp4_b256", "mamba2_f16ckpt_b256",
                 "gdn_f16ckpt_b256")


def sub_record(torch, rssm, args, name, device, peak, peak_kind, fp32_value, done=None):
    """One workload measured over a few windows (320 timed steps or 80
    speculative rounds after 16 / 8 of warm-up): its throughput, the roofline
    of its dominant kernel and its speed-up over the in-build baseline of the
    same run (the conventional kernel, the snapshot rollback, for the
    low-precision formats the FP32-checkpoint path of the main line, and for
    speculative rounds with a read copy the FP32 speculative record in
    `done`)."""
    import argparse as _ap
    a = _ap.Namespace(**vars(args))
    w = synth.WORKLOADS[name]
    spec = name.endswith("_b512") and "spec" in name
    a.workload, a.k, a.batch, a.mode, a.no_e2e = name, 0, 0, "replay", True
    a.steps, a.warmup = (80, 8) if spec else (320, 16)
    a.pool = 32
    lowp = getattr(w, "read_fmt", "none") != "none" or getattr(w, "ckpt", "f32") != "f32"
    a.no_compare = lowp
    if name.startswith("mamba2_spec"):
        res = spec_arm(torch, rssm, a, device, None)
    elif name.startswith("gdn_spec"):
        res = gdn_spec_arm(torch, rssm, a, device, None)
    elif isinstance(w, synth.GDNWorkload):
        res = gdn_arm(torch, rssm, a, device, None)
    else:
        res = m2_arm(torch, rssm, a, device, None)
    tokens = res.get("tokens", w.batch * a.steps)
    value = tokens / (res["total_ms"] / 1e3)
    rec = {"value": value, "unit": UNIT, "steps": a.steps, "warmup": a.warmup,
           "ms_per_step": res["total_ms"] / a.steps, "batch": w.batch, "k": w.k,
           "roofline": roofline_of(res, "replay", a.warmup, peak, peak_kind), "clocks": res["clocks"]}
    if "conv" in res:
        cv = res["conv"]
        cval = w.batch * a.steps / (cv["total_ms"] / 1e3)
        rec["baseline"] = {"name": "conventional kernel", "value": cval, "speedup": value / cval}
    if "spec" in res:
        sp = res["spec"]
        rec["spec"] = sp
        if "snapshot_baseline" in sp:
            rec["baseline"] = {"name": "snapshot save/restore", "value": sp["snapshot_baseline"]["committed_tokens_per_s"],
                               "speedup": sp["speedup_vs_snapshot"]}
    if lowp and spec:
        base_name = "gdn_spec_b512" if name.startswith("gdn") else "mamba2_spec_b512"
        base = (done or {}).get(base_name)
        if base:
            rec["baseline"] = {"name": f"FP32 checkpoint ({base_name})", "value": base["value"],
                               "speedup": value / base["value"]}
    elif lowp and isinstance(w, synth.GDNWorkload):
        base = (done or {}).get("gdn_serving_b256")
        if base:
            rec["baseline"] = {"name": "FP32 checkpoint (gdn_serving_b256)", "value": base["value"],
                               "speedup": value / base["value"]}
    elif lowp:
        rec["baseline"] = {"name": "FP32 checkpoint (main line)", "value": fp32_value, "speedup": value / fp32_value}
    return rec


def spec_then_plain(torch, rssm, device, rounds=6, plain=12):
    """Plain one-token steps after speculative verifies (batch-512 serving
    shape, T=4). Two identical layers run the same rounds; then one reads its
    record counts back from the device (rssm_sync_counts) and the other does
    not, and both run the same plain steps. After the verifies the counts
    differ between sequences, so most steps flush some tiles: the handle then
    runs the flush-only launch over those tiles and the lean kernel over the
    rest (with unknown counts too, that pair is its choice); only a step in
    which no tile flushes runs the lean kernel alone, which it chooses when
    the counts are known. An untimed pass first takes every launch's
    one-time setup. Reports the mean step time of each, timed with CUDA
    events on the launch stream."""
    w = synth.WORKLOADS["mamba2_spec_b512"]
    T = w.draft
    A, D = synth.mamba2_params(w)
    dA, dD = torch.from_numpy(A).to(device), torch.from_numpy(D).to(device)
    h0 = to_dev(torch, synth.Tensor(synth.mamba2_state0(w), None, "f32"), device)
    acc = synth.acceptance(w.batch, rounds, T, w.accept_p, seed=7)
    cfg = rssm.make_config(kind="mamba2", mode="replay", batch=w.batch, heads=w.heads, head_dim=w.head_dim,
                           state_dim=w.state_dim, groups=w.groups, k=w.k, max_draft=T, in_dtype=w.dtype)
    stream = torch.cuda.current_stream(device)
    keys = ("x", "B", "C", "dt")
    rin = []
    for r in range(rounds):
        ins = synth.mamba2_steps(w, r * T, T)
        rin.append({k: to_dev(torch, synth.Tensor(np.ascontiguousarray(np.swapaxes(ins[k].raw, 0, 1)), None,
                                                  ins[k].dtype), device) for k in keys})
    plain_in = synth.mamba2_steps(w, 10_000, plain)
    pin = {k: to_dev(torch, plain_in[k], device) for k in keys}
    ydt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    y1 = torch.empty((w.batch, 1, w.heads, w.head_dim), dtype=ydt, device=device)
    yT = torch.empty((w.batch, T, w.heads, w.head_dim), dtype=ydt, device=device)
    out = {}
    for synced in (None, False, True):   # None: the untimed pass
        layer = rssm.Layer(cfg, dA, dD, h0)
        for r in range(rounds):
            d = rin[r]
            layer.decode_step(yT, T, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"])
            layer.verify_rollback(torch.from_numpy(acc[r]).to(device))
        torch.cuda.synchronize()
        sync_ms = None
        if synced:
            t0 = time.perf_counter()
            layer.sync_counts()
            sync_ms = (time.perf_counter() - t0) * 1e3
        lean = [0]

        def launch(i):
            known, _, hi = layer.count_summary()
            lean[0] += int(known == 1 and hi + 1 < w.k)
            layer.decode_step(y1, 1, x=pin["x"][i], Bm=pin["B"][i], C=pin["C"][i], dt=pin["dt"][i], stream=stream)

        _, per = time_loop(torch, stream, plain, launch)
        if layer.get_error()[0]:
            raise RuntimeError("device error word set")
        layer.close()
        if synced is None:
            continue
        key = "synced" if synced else "unsynced"
        out[key] = {"mean_us": 1e3 * sum(per) / len(per), "lean_kernel_only_steps": lean[0]}
        if synced:
            out[key]["sync_counts_ms"] = sync_ms
    out["steps"] = plain
    out["rounds_before"] = rounds
    out["speedup"] = out["unsynced"]["mean_us"] / out["synced"]["mean_us"]
    return out


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
KERNEL_SOURCES = {
    "m2_replay": ("m2_replay_tma.cu", "m2_pipeline.cuh"),
    "m2_draft": ("m2_draft_tma.cu", "m2_pipeline.cuh"),
    "gdn": ("gdn_replay_tma.cu", "gdn_pipeline.cuh"),
    "gdn_draft": ("gdn_draft_tma.cu", "gdn_pipeline.cuh"),
}


def source_digest(kernel: str) -> str:
    """sha256 over the source files that define a replay kernel (its own .cu
    and its family's pipeline header; not the generic helpers)."""
    import hashlib
    family = "gdn" if kernel.startswith("gdn") else "m2_replay"
    if "draft" in kernel:
        family = "gdn_draft" if kernel.startswith("gdn") else "m2_draft"
    files = KERNEL_SOURCES[family]
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "hybrid_ssm_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(kernel: str, w) -> float | None:
    """DRAM bytes (read + write) per launch of `kernel` on this workload, as
    recorded from an ncu capture in profiles/*.md ("traffic:" lines), when the
    kernel's sources are unchanged since; else None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want = {"kernel": kernel, "workload": w.name, "batch": str(w.batch), "k": str(w.k)}
    digest = None
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                line = line.strip().strip("`")
                if not line.startswith("traffic:"):
                    continue
                kv = dict(p.split("=", 1) for p in line[len("traffic:"):].split() if "=" in p)
                if any(kv.get(key) != val for key, val in want.items()):
                    continue
                if digest is None:
                    digest = source_digest(kernel)
                if kv.get("sources") == digest:
                    return float(kv["bytes_per_launch"])
    return None
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"rssm_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        try:
            rows = [l.split(",") for l in open(self.path).read().strip().splitlines()]
            os.remove(self.path)
        except Exception:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 7:
                continue
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except ValueError:
                continue
            for n, v in zip(names, r[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_smi_id(torch, dev: int) -> str:
    """nvidia-smi id of a CUDA device: its PCI bus id when nvidia-smi knows it,
    else the index."""
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    if bus is not None:
        pci = f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:{getattr(props, 'pci_device_id', 0):02x}.0"
        try:
            r = subprocess.run(["nvidia-smi", "-i", pci, "--query-gpu=index", "--format=csv,noheader"],
                               capture_output=True, text=True, timeout=20)
            if r.returncode == 0 and r.stdout.strip():
                return pci
        except Exception:
            pass
    return str(dev)


# ---------------------------------------------------------------------------
# the librssm arm
# ---------------------------------------------------------------------------
def workload(args):
    w = synth.WORKLOADS[args.workload]
    if args.k:
        w = w.replace(k=args.k)
    if args.batch:
        w = w.replace(batch=args.batch)
    return w


def to_dev(torch, t, device):
    raw = np.ascontiguousarray(t.raw)
    if raw.dtype == np.uint16:
        return torch.from_numpy(raw.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(raw).to(device)


def to_pinned(torch, t):
    raw = np.ascontiguousarray(t.raw)
    if raw.dtype == np.uint16:
        return torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(raw).pin_memory()


def time_loop(torch, stream, K, launch, per_launch=True):
    """Run launch(i) for i < K on `stream`; returns (total_ms, per-launch ms list)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)] if per_launch else None
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        if per_launch:
            ev[i][0].record(stream)
        launch(i)
        if per_launch:
            ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev] if per_launch else []
    return t0.elapsed_time(t1), per


def rotation_layers(torch, device, state_bytes: int) -> int:
    """Independent layers stepped round-robin so that the states a timed run
    touches exceed twice L2: a single layer's state below that would stay in
    L2 from one step to the next, which no multi-layer decode sees (each layer
    is stepped once per token, the others' states in between). 1 at the
    serving sizes."""
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or 129 * 2**20
    return max(1, -(-2 * l2 // max(1, state_bytes)))


def l2_note(n_layers: int, state_bytes: int) -> str:
    if n_layers == 1:
        return "state streamed every step exceeds L2 (no extra flush)"
    return (f"{n_layers} independent layers stepped round-robin; their states "
            f"({n_layers * state_bytes / 1e6:.0f} MB) exceed twice L2 (no extra flush)")


def graph_window(torch, launch, done, k, K, device):
    """Steps replayed from a CUDA graph, so that host launch overhead is out
    of the timed region: plain steps until the record count returns to 0,
    then one window of k steps is captured and replayed K // k times (each
    replay starts and ends at count 0). With n layers stepped round-robin, k
    is the window times n. launch(i, stream) enqueues step i on `stream` and
    returns its status. Returns the mean step time in ms and the steps
    timed."""
    stream = torch.cuda.current_stream(device)
    while done % k:
        if launch(done, stream.cuda_stream):
            raise RuntimeError("decode step failed")
        done += 1
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream(device).cuda_stream
        for i in range(k):
            if launch(done + i, cap):
                raise RuntimeError("decode step failed during capture")
    g.replay()                                   # one more window of warm-up
    torch.cuda.synchronize()
    reps = max(1, K // k)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    del g
    return {"ms_per_step": t0.elapsed_time(t1) / (reps * k), "steps": reps * k}


def m2_arm(torch, rssm, args, device, dist):
    w = workload(args)
    mode = args.mode
    out_size = 4 if w.dtype == "f32" else 2
    K, W = args.steps, args.warmup
    pool = max(1, min(args.pool, K + W))
    steps = synth.mamba2_steps(w, 0, pool)
    A, D = synth.mamba2_params(w)
    dA, dD = torch.from_numpy(A).to(device), torch.from_numpy(D).to(device)
    h0 = to_dev(torch, synth.Tensor(synth.mamba2_state0(w), None, "f32"), device)
    keys = ("x", "B", "C", "dt")
    dins = {k: to_dev(torch, steps[k], device) for k in keys}        # [pool][B][...]
    ydt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    y = torch.empty((w.batch, 1, w.heads, w.head_dim), dtype=ydt, device=device)
    stream = torch.cuda.current_stream(device)
    state_bytes = w.batch * w.heads * w.head_dim * w.state_dim * 4
    n_layers = rotation_layers(torch, device, state_bytes)

    def run(mode_, read_fmt, ckpt):
        cfg = rssm.make_config(kind="mamba2", mode=mode_, batch=w.batch, heads=w.heads,
                               head_dim=w.head_dim, state_dim=w.state_dim, groups=w.groups, k=w.k,
                               max_draft=1, in_dtype=w.dtype, read_fmt=read_fmt, ckpt_dtype=ckpt)
        layers = [rssm.Layer(cfg, dA, dD, h0) for _ in range(n_layers)]
        inp = [rssm.Inputs(x=dins["x"][i].data_ptr(), Bm=dins["B"][i].data_ptr(),
                           C=dins["C"][i].data_ptr(), dt=dins["dt"][i].data_ptr())
               for i in range(pool)]
        lib, ya, st = rssm.load(), y.data_ptr(), stream.cuda_stream
        handles = [ly.handle for ly in layers]
        import ctypes
        inp_p = [ctypes.byref(x) for x in inp]

        def launch(i, off=0):
            j = i + off   # step j goes to layer j % n_layers, its (j // n_layers)-th step
            rc = lib.rssm_decode_step(handles[j % n_layers], 1, inp_p[j % pool], ya, st)
            if rc:
                raise rssm.RssmError("rssm_decode_step", rc)

        for i in range(W):
            launch(i)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        with ClockSampler(gpu_smi_id(torch, device.index or 0)) as clk:
            total, per = time_loop(torch, stream, K, lambda i: launch(i, W))
        if dist:
            dist.barrier()
        graph = None
        if args.graph:
            graph = graph_window(torch, lambda i, st_: lib.rssm_decode_step(handles[i % n_layers], 1,
                                                                            inp_p[i % pool], ya, st_),
                                 W + K, w.k * n_layers, K, device)
        for ly in layers:
            err = ly.get_error()
            if err[0]:
                raise RuntimeError(f"device error word {err}")
        # bytes per launch: step j (0-based from creation) is its layer's
        # (j // n_layers)-th, which holds c = that % k records before it
        byts = []
        for i in range(K):
            s = (W + i) // n_layers
            c = s % w.k if mode_ == "replay" else 0
            flush = mode_ == "replay" and c == w.k - 1
            byts.append(m2_step_bytes(w, c, flush, mode_, read_fmt, out_size, ckpt))
        for ly in layers:
            ly.close()
        return total, per, byts, clk.summary(), graph

    total, per, byts, clocks, graph = run(mode, w.read_fmt, w.ckpt)
    res = {"total_ms": total, "per": per, "bytes": byts, "clocks": clocks, "w": w,
           "kernel": "m2_replay_step_tma_kernel" if mode == "replay" else "m2_conv_step_kernel",
           "nf_kernel": "m2_replay_nf_kernel", "graph": graph, "layers": n_layers,
           "l2": l2_note(n_layers, state_bytes)}
    if not args.no_compare and mode == "replay":
        ctot, cper, cbytes, _, cgraph = run("conventional", "none", "f32")
        res["conv"] = {"total_ms": ctot, "per": cper, "bytes": cbytes, "graph": cgraph}
    if not args.no_e2e:
        res["e2e"] = m2_e2e(torch, rssm, w, steps, dA, dD, h0, mode, K, W, pool, device, dist)
    return res


def m2_e2e(torch, rssm, w, steps, dA, dD, h0, mode, K, W, pool, device, dist):
    """Through the public API with host buffers: every step copies its inputs
    from pinned host memory, decodes, and copies y back to pinned host
    memory. The copies run on a second stream, double-buffered, so step i+1's
    inputs travel while step i decodes; every copy is inside the timed
    region, which ends when the last output has reached the host."""
    keys = ("x", "B", "C", "dt")
    hins = {k: to_pinned(torch, steps[k]) for k in keys}
    dbuf = [{k: torch.empty(hins[k].shape[1:], dtype=hins[k].dtype, device=device) for k in keys}
            for _ in range(2)]
    ydt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    ys = [torch.empty((w.batch, 1, w.heads, w.head_dim), dtype=ydt, device=device) for _ in range(2)]
    yh = [torch.empty(ys[0].shape, dtype=ydt).pin_memory() for _ in range(2)]
    cfg = rssm.make_config(kind="mamba2", mode=mode, batch=w.batch, heads=w.heads,
                           head_dim=w.head_dim, state_dim=w.state_dim, groups=w.groups, k=w.k,
                           in_dtype=w.dtype, read_fmt=w.read_fmt, ckpt_dtype=w.ckpt)
    layer = rssm.Layer(cfg, dA, dD, h0)
    stream = torch.cuda.current_stream(device)
    cs = torch.cuda.Stream(device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        b = i % 2
        with torch.cuda.stream(cs):
            cs.wait_event(done[b])          # step i-2 has finished with these buffers
            for k in keys:
                dbuf[b][k].copy_(hins[k][i % pool], non_blocking=True)
            in_ready[b].record(cs)

    def step(i):
        b = i % 2
        stream.wait_event(in_ready[b])
        d = dbuf[b]
        layer.decode_step(ys[b], 1, x=d["x"], Bm=d["B"], C=d["C"], dt=d["dt"], stream=stream)
        done[b].record(stream)
        with torch.cuda.stream(cs):
            cs.wait_event(done[b])
            yh[b].copy_(ys[b], non_blocking=True)

    def run(n, first):
        copy_in(first)
        for i in range(first, first + n):
            if i + 1 < first + n:
                copy_in(i + 1)
            step(i)

    for b in range(2):
        done[b].record(stream)
    run(W, 0)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(cs)
    run(K, W)
    t1.record(cs)
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1)
    h2d = sum(dbuf[0][k].numel() * dbuf[0][k].element_size() for k in keys)
    d2h = ys[0].numel() * ys[0].element_size()
    layer.close()
    return {"total_ms": total, "h2d": h2d, "d2h": d2h}


def gdn_arm(torch, rssm, args, device, dist):
    w = workload(args)
    out_size = 4 if w.dtype == "f32" else 2
    K, W = args.steps, args.warmup
    pool = max(1, min(args.pool, K + W))
    steps = synth.gdn_steps(w, 0, pool)
    keys = ("q", "k", "v", "alpha", "beta")
    dins = {k: to_dev(torch, steps[k], device) for k in keys}
    S0 = to_dev(torch, synth.Tensor(synth.gdn_state0(w), None, "f32"), device)
    ydt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    o = torch.empty((w.batch, 1, w.heads, w.d_v), dtype=ydt, device=device)
    stream = torch.cuda.current_stream(device)
    state_bytes = w.batch * w.heads * w.d_v * w.d_k * 4
    n_layers = rotation_layers(torch, device, state_bytes)
    import ctypes

    def run(mode_):
        # the conventional comparison arm is plain; a conventional main arm
        # with a read format is the quantised-recurrence baseline
        rf = w.read_fmt if (mode_ == "replay" or args.mode == "conventional") else "none"
        ck = w.ckpt if mode_ == "replay" else "f32"
        cfg = rssm.make_config(kind="gdn", mode=mode_, batch=w.batch, heads=w.heads, head_dim=w.d_v,
                               state_dim=w.d_k, k=w.k, in_dtype=w.dtype, gdn_scale=w.scale, read_fmt=rf,
                               ckpt_dtype=ck)
        layers = [rssm.Layer(cfg, None, None, S0) for _ in range(n_layers)]
        inp = [rssm.Inputs(q=dins["q"][i].data_ptr(), k=dins["k"][i].data_ptr(),
                           v=dins["v"][i].data_ptr(), alpha=dins["alpha"][i].data_ptr(),
                           beta=dins["beta"][i].data_ptr()) for i in range(pool)]
        inp_p = [ctypes.byref(x) for x in inp]
        lib, oa, st = rssm.load(), o.data_ptr(), stream.cuda_stream
        handles = [ly.handle for ly in layers]

        def launch(i):
            rc = lib.rssm_decode_step(handles[i % n_layers], 1, inp_p[i % pool], oa, st)
            if rc:
                raise rssm.RssmError("rssm_decode_step", rc)

        for i in range(W):
            launch(i)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        with ClockSampler(gpu_smi_id(torch, device.index or 0)) as clk:
            total, per = time_loop(torch, stream, K, lambda i: launch(i + W))
        if dist:
            dist.barrier()
        graph = None
        if args.graph:
            graph = graph_window(torch, lambda i, st_: lib.rssm_decode_step(handles[i % n_layers], 1,
                                                                            inp_p[i % pool], oa, st_),
                                 W + K, w.k * n_layers, K, device)
        byts = []
        for i in range(K):
            s = (W + i) // n_layers
            c = s % w.k if mode_ == "replay" else 0
            byts.append(gdn_step_bytes(w, c, mode_ == "replay" and c == w.k - 1, mode_, out_size, rf, ck))
        for ly in layers:
            ly.close()
        return total, per, byts, clk.summary(), graph

    total, per, byts, clocks, graph = run(args.mode)
    res = {"total_ms": total, "per": per, "bytes": byts, "clocks": clocks, "w": w,
           "kernel": "gdn_replay_step_tma_kernel" if args.mode == "replay" else "gdn_conv_step_kernel",
           "nf_kernel": "gdn_replay_nf_kernel", "graph": graph, "layers": n_layers,
           "l2": l2_note(n_layers, state_bytes)}
    if not args.no_compare and args.mode == "replay":
        ctot, cper, cbytes, _, cgraph = run("conventional")
        res["conv"] = {"total_ms": ctot, "per": cper, "bytes": cbytes, "graph": cgraph}
    return res


def spec_arm(torch, rssm, args, device, dist):
    """Speculative rounds on the batch-512 serving shape: each round drafts T=4
    tokens per sequence (one decode_step) and resolves them with per-sequence
    acceptance counts (one verify_rollback). One timed step = one round.
    Replay rolls back by moving the buffer pointer; the baseline (conventional
    mode) writes a state snapshot per draft and restores one on verify."""
    import ctypes
    w = workload(args)
    T = w.draft
    K, W = args.steps, args.warmup
    pool = max(1, min(args.pool // 4, K + W))
    keys = ("x", "B", "C", "dt")
    per_round = [synth.mamba2_steps(w, r * T, T) for r in range(pool)]
    dins = {}
    for k in keys:
        raw = np.stack([np.swapaxes(pr[k].raw, 0, 1) for pr in per_round])  # [pool][B][T][...]
        dins[k] = to_dev(torch, synth.Tensor(np.ascontiguousarray(raw), None, per_round[0][k].dtype), device)
    acc = synth.acceptance(w.batch, pool, T, w.accept_p)
    dacc = torch.from_numpy(acc).to(device)
    A, D = synth.mamba2_params(w)
    dA, dD = torch.from_numpy(A).to(device), torch.from_numpy(D).to(device)
    h0 = to_dev(torch, synth.Tensor(synth.mamba2_state0(w), None, "f32"), device)
    ydt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    y = torch.empty((w.batch, T, w.heads, w.head_dim), dtype=ydt, device=device)
    stream = torch.cuda.current_stream(device)
    s = 4 if w.dtype == "f32" else 2
    B, H, P, N, G = w.batch, w.heads, w.head_dim, w.state_dim, w.groups
    state = P * N * 4
    rec = P * s + s + N * s * G / H
    # drafts read the read copy when there is one; a fold writes it too
    rc = {"none": 0, "fp8": P * N + 4, "nvfp4": P * N / 2 + P * N / 16 + 4}[w.read_fmt]

    def run(mode_):
        cfg = rssm.make_config(kind="mamba2", mode=mode_, batch=B, heads=H, head_dim=P, state_dim=N,
                               groups=G, k=w.k, max_draft=T, in_dtype=w.dtype,
                               read_fmt=w.read_fmt if mode_ == "replay" else "none")
        layer = rssm.Layer(cfg, dA, dD, h0)
        inp = [rssm.Inputs(x=dins["x"][i].data_ptr(), Bm=dins["B"][i].data_ptr(),
                           C=dins["C"][i].data_ptr(), dt=dins["dt"][i].data_ptr()) for i in range(pool)]
        inp_p = [ctypes.byref(x) for x in inp]
        lib, handle, ya, st = rssm.load(), layer.handle, y.data_ptr(), stream.cuda_stream
        ev = []

        def launch(i, timed):
            j = i % pool
            if timed:
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record(stream)
            rc = lib.rssm_decode_step(handle, T, inp_p[j], ya, st)
            if timed:
                e[1].record(stream)
            rc = rc or lib.rssm_verify_rollback(handle, dacc[j].data_ptr(), st)
            if timed:
                e[2].record(stream)
                ev.append(e)
            if rc:
                raise rssm.RssmError("speculative round", rc)

        for i in range(W):
            launch(i, False)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        with ClockSampler(gpu_smi_id(torch, device.index or 0)) as clk:
            total, _ = time_loop(torch, stream, K, lambda i: launch(i + W, True), per_launch=False)
        if dist:
            dist.barrier()
        if layer.get_error()[0]:
            raise RuntimeError("device error word set")
        draft_ms = [e[0].elapsed_time(e[1]) for e in ev]
        verify_ms = [e[1].elapsed_time(e[2]) for e in ev]
        # host model of the committed counts, for the byte model
        c = np.zeros(B, np.int64)
        for i in range(W):
            c = c + acc[i % pool]
            c[c >= w.k] = 0
        dbytes, vbytes, committed = [], [], 0
        for i in range(K):
            a = acc[(W + i) % pool]
            if mode_ == "replay":
                dbytes.append(B * H * ((rc or state) + np.mean(c) * rec + T * (rec + N * s * G / H + P * s) + 8))
                c2 = c + a
                fl = c2 >= w.k
                vbytes.append(H * (fl.sum() * (2 * state + rc) + np.sum(c2[fl]) * rec) + B * H * 8)
                c = np.where(fl, 0, c2)
            else:
                dbytes.append(B * H * (state + T * state + T * (rec + N * s * G / H + P * s)))
                vbytes.append(H * np.sum(a > 0) * 2 * state)
            committed += int(a.sum())
        layer.close()
        return total, draft_ms, verify_ms, dbytes, vbytes, committed, clk.summary()

    tot, dms, vms, db, vb, committed, clocks = run("replay")
    res = {"total_ms": tot, "per": dms, "bytes": db, "clocks": clocks, "w": w, "tokens": committed,
           "launches": 2 * K, "kernel": "m2_replay_draft_tma_kernel", "draft": T, "flush_mask": True}
    spec = {"rounds": K, "committed_tokens_per_s": committed / (tot / 1e3),
            "verified_positions_per_s": B * T * K / (tot / 1e3),
            "mean_accepted": committed / (B * K),
            "draft_kernel_us": 1e3 * sum(dms) / K, "verify_kernel_us": 1e3 * sum(vms) / K}
    if not args.no_compare:
        ctot, cdms, cvms, cdb, cvb, ccomm, _ = run("conventional")
        spec["snapshot_baseline"] = {
            "committed_tokens_per_s": ccomm / (ctot / 1e3), "ms_per_round": ctot / K,
            "draft_kernel_us": 1e3 * sum(cdms) / K, "restore_kernel_us": 1e3 * sum(cvms) / K,
            "draft_gbs": sum(cdb) / (sum(cdms) / 1e3) / 1e9}
        spec["speedup_vs_snapshot"] = ctot / tot
    spec["verify_gbs"] = (sum(vb) / (sum(vms) / 1e3) / 1e9) if sum(vms) > 0 else None
    res["spec"] = spec
    return res



def gdn_spec_arm(torch, rssm, args, device, dist):
    """Speculative rounds on the Gated DeltaNet serving shape at batch 512:
    each round drafts T=4 tokens per sequence (one decode_step) and resolves
    them with per-sequence acceptance counts (one verify_rollback). One timed
    step = one round. The baseline (conventional mode) writes a state
    snapshot per draft and restores the accepted one on verify."""
    import ctypes
    w = workload(args)
    T = w.draft
    K, W = args.steps, args.warmup
    pool = max(1, min(args.pool // 4, K + W))
    keys = ("q", "k", "v", "alpha", "beta")
    per_round = [synth.gdn_steps(w, r * T, T) for r in range(pool)]
    dins = {}
    for k in keys:
        raw = np.stack([np.swapaxes(pr[k].raw, 0, 1) for pr in per_round])   # [pool][B][T][...]
        dins[k] = to_dev(torch, synth.Tensor(np.ascontiguousarray(raw), None, per_round[0][k].dtype), device)
    acc = synth.acceptance(w.batch, pool, T, w.accept_p)
    dacc = torch.from_numpy(acc).to(device)
    S0 = to_dev(torch, synth.Tensor(synth.gdn_state0(w), None, "f32"), device)
    ydt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    o = torch.empty((w.batch, T, w.heads, w.d_v), dtype=ydt, device=device)
    stream = torch.cuda.current_stream(device)
    s = 4 if w.dtype == "f32" else 2
    B, H, DK, DV = w.batch, w.heads, w.d_k, w.d_v
    state = DV * DK * 4
    rec = DK * s + DV * 4 + 4
    tok_io = 2 * DK * s + DV * s + 8 + DV * s
    # drafts read the read copy when there is one; its records keep v and beta
    rc = {"none": 0, "fp8": DV * DK + DV / 16, "nvfp4": DV * DK / 2 + DV * DK / 16 + DV / 16}[w.read_fmt]
    if w.read_fmt != "none":
        rec += DV * s + 4

    def run(mode_):
        cfg = rssm.make_config(kind="gdn", mode=mode_, batch=B, heads=H, head_dim=DV, state_dim=DK, k=w.k,
                               max_draft=T, in_dtype=w.dtype, gdn_scale=w.scale,
                               read_fmt=w.read_fmt if mode_ == "replay" else "none")
        layer = rssm.Layer(cfg, None, None, S0)
        inp = [rssm.Inputs(q=dins["q"][i].data_ptr(), k=dins["k"][i].data_ptr(), v=dins["v"][i].data_ptr(),
                           alpha=dins["alpha"][i].data_ptr(), beta=dins["beta"][i].data_ptr())
               for i in range(pool)]
        inp_p = [ctypes.byref(x) for x in inp]
        lib, handle, oa, st = rssm.load(), layer.handle, o.data_ptr(), stream.cuda_stream
        ev = []

        def launch(i, timed):
            j = i % pool
            if timed:
                e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
                e[0].record(stream)
            rc = lib.rssm_decode_step(handle, T, inp_p[j], oa, st)
            if timed:
                e[1].record(stream)
            rc = rc or lib.rssm_verify_rollback(handle, dacc[j].data_ptr(), st)
            if timed:
                e[2].record(stream)
                ev.append(e)
            if rc:
                raise rssm.RssmError("speculative round", rc)

        for i in range(W):
            launch(i, False)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        with ClockSampler(gpu_smi_id(torch, device.index or 0)) as clk:
            total, _ = time_loop(torch, stream, K, lambda i: launch(i + W, True), per_launch=False)
        if dist:
            dist.barrier()
        if layer.get_error()[0]:
            raise RuntimeError("device error word set")
        dms = [e[0].elapsed_time(e[1]) for e in ev]
        vms = [e[1].elapsed_time(e[2]) for e in ev]
        c = np.zeros(B, np.int64)
        for i in range(W):
            c = c + acc[i % pool]
            c[c >= w.k] = 0
        dbytes, committed = [], 0
        for i in range(K):
            a = acc[(W + i) % pool]
            if mode_ == "replay":
                dbytes.append(B * H * ((rc or state) + np.mean(c) * rec + T * (rec + tok_io) + 8))
            else:
                dbytes.append(B * H * (state + T * state + T * tok_io))
            c = c + a
            c[c >= w.k] = 0
            committed += int(a.sum())
        layer.close()
        return total, dms, vms, dbytes, committed, clk.summary()

    total, dms, vms, dbytes, committed, clocks = run("replay")
    spec = {"rounds": K, "committed_tokens_per_s": committed / (total / 1e3),
            "verified_positions_per_s": B * T * K / (total / 1e3), "mean_accepted": committed / (B * K),
            "draft_kernel_us": 1e3 * sum(dms) / K, "verify_kernel_us": 1e3 * sum(vms) / K}
    if not args.no_compare:
        ctot, cdms, cvms, cdb, ccomm, _ = run("conventional")
        spec["snapshot_baseline"] = {
            "committed_tokens_per_s": ccomm / (ctot / 1e3), "ms_per_round": ctot / K,
            "draft_kernel_us": 1e3 * sum(cdms) / K, "restore_kernel_us": 1e3 * sum(cvms) / K,
            "draft_gbs": sum(cdb) / (sum(cdms) / 1e3) / 1e9}
        spec["speedup_vs_snapshot"] = ctot / total
    return {"total_ms": total, "per": dms, "bytes": dbytes, "clocks": clocks, "w": w, "tokens": committed,
            "launches": 2 * K, "kernel": "gdn_replay_draft_kernel", "draft": T, "flush_mask": True, "spec": spec}


def cpu_baseline(workload: str, seconds: float = 10.0):
    """The float64 oracle on the host cores, on a growing sample of the same
    workload until about `seconds` of CPU time has been spent."""
    import oracle
    w = synth.WORKLOADS[workload]
    cores = oracle.max_threads()
    if isinstance(w, synth.GDNWorkload):
        n_seq, n_steps = 4, 16
        ins = synth.gdn_steps(w, 0, n_steps)
        S0 = synth.gdn_state0(w)
        t0 = time.perf_counter()
        done = 0
        while time.perf_counter() - t0 < seconds:
            sl = slice(0, n_seq)
            oracle.gdn_recurrence(S0[sl], *(ins[k].values[:, sl] for k in ("q", "k", "v", "alpha", "beta")),
                                  scale=w.scale)
            done += n_seq * n_steps
        el = time.perf_counter() - t0
        return {"value": done / el, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{n_seq} sequences x {w.heads} heads x {n_steps} steps, repeated for {el:.1f} s "
                          "(float64 per-token recurrence, OpenMP over (sequence, head) tiles)"}
    n_seq, n_steps = 16, 16
    ins = synth.mamba2_steps(w, 0, n_steps)
    A, D = synth.mamba2_params(w)
    h0 = synth.mamba2_state0(w)[:n_seq]
    args = [ins[k].values[:, :n_seq] for k in ("x", "B", "C", "dt")]
    t0 = time.perf_counter()
    done = 0
    while time.perf_counter() - t0 < seconds:
        oracle.m2_recurrence(h0, A, D, *args)
        done += n_seq * n_steps
    el = time.perf_counter() - t0
    return {"value": done / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_seq} sequences x {w.heads} heads x {n_steps} steps of {workload}, repeated for "
                      f"{el:.1f} s (float64 per-token recurrence, OpenMP over (sequence, head) tiles)"}


# ---------------------------------------------------------------------------
# reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------
def reference_arm(args, rank, world):
    if rank != 0:
        return
    import oracle
    w = synth.WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    budget_s = 150.0
    cores = oracle.max_threads()
    if isinstance(w, synth.GDNWorkload):
        raise SystemExit("--impl reference covers the Mamba-2 workloads")
    A, D = synth.mamba2_params(w)
    pool = 16
    ins = synth.mamba2_steps(w, 0, pool)
    # one step = one decode token for n_seq sequences (all heads), state carried over
    n_seq = 1
    h = synth.mamba2_state0(w)[:n_seq].astype(np.float64)
    sub = {k: ins[k].values[:, :n_seq] for k in ("x", "B", "C", "dt")}

    def step(i, h):
        j = i % pool
        _, h = oracle.m2_recurrence(h, A, D, *(sub[k][j:j + 1] for k in ("x", "B", "C", "dt")))
        return h

    t0 = time.perf_counter()
    h = step(0, h)
    one = time.perf_counter() - t0
    # keep the whole run within the budget: time at most this many steps
    max_steps = max(3, int(budget_s / max(one, 1e-6)))
    k_eff = min(K, max_steps)
    w_eff = min(W, 3)
    for i in range(w_eff):
        h = step(i, h)
    t0 = time.perf_counter()
    for i in range(k_eff):
        h = step(i, h)
    el = time.perf_counter() - t0
    value = n_seq * k_eff / el
    sample = (f"{n_seq} sequence x {w.heads} heads per step, {k_eff} timed steps"
              + (f" of the requested {K}" if k_eff < K else "")
              + "; float64 per-token recurrence (OpenMP over heads)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": k_eff, "warmup": w_eff, "ms_per_step": el / k_eff * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "heads": w.heads, "head_dim": w.head_dim,
                       "state_dim": w.state_dim, "groups": w.groups, "k": w.k, "inputs": w.dtype},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# synthetic layer stack (diagnostic, not the contract line)
# ---------------------------------------------------------------------------
def stack_bench(args):
    """Decode-step time of a synthetic stack of Mamba-2 layers with random
    projections (hybrid_ssm_decode_gb300.stack), replay against conventional
    SSM layers; everything but the SSM layer's mode is the same. One window
    of k steps (each with a fresh embedding from a resident pool of k) is
    captured as a CUDA graph after warm-up, so host launch overhead is out of
    the timed region, and replayed K / k times. The SSM layers alone (the
    same decode steps on resident inputs) are captured and timed the same
    way, which gives their share of the step. Prints one diagnostic JSON
    line."""
    import torch
    import hybrid_ssm_decode_gb300 as rssm
    from hybrid_ssm_decode_gb300.stack import M2Stack, StackShape
    rssm.load()
    w = workload(args)
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    shape = StackShape(layers=args.stack, batch=w.batch, heads=w.heads, head_dim=w.head_dim,
                       state_dim=w.state_dim, groups=w.groups, k=w.k)
    k = w.k
    reps = max(1, args.steps // k)
    W = ((max(args.warmup, 3) + k - 1) // k) * k              # whole windows
    g = torch.Generator(device=device)
    g.manual_seed(11)
    pool = torch.randn((k, shape.batch, shape.d_model), generator=g, device=device).to(torch.bfloat16)

    def timed(fn, n):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(n):
            fn()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    res = {}
    for mode in ("replay", "conventional"):
        stack = M2Stack(shape, mode=mode, ckpt=w.ckpt if mode == "replay" else "f32",
                        read_fmt=w.read_fmt if mode == "replay" else "none")
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(side):
            for i in range(W):
                stack.step(pool[i % k])
        torch.cuda.current_stream(device).wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            for i in range(k):
                stack.step(pool[i])
        graph.replay()                                       # one more window of warm-up
        torch.cuda.synchronize()
        with ClockSampler(gpu_smi_id(torch, 0)) as clk:
            total = timed(graph.replay, reps)
        # the SSM layers alone on resident inputs, one window
        ins = stack.ssm_inputs(pool[0])
        sg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sg, capture_error_mode="thread_local"):
            for i in range(k):
                for layer, (x, Bt, Ct, dt) in zip(stack.layers, ins):
                    layer.decode_step(stack.y, 1, x=x, Bm=Bt, C=Ct, dt=dt)
        sg.replay()
        torch.cuda.synchronize()
        ssm = timed(sg.replay, reps)
        for layer in stack.layers:
            if layer.get_error()[0]:
                raise RuntimeError("device error word set")
        steps = reps * k
        res[mode] = {"ms_per_step": total / steps, "tokens_per_s": shape.batch * steps / (total / 1e3),
                     "ssm_layers_ms_per_step": ssm / steps, "ssm_share": ssm / total, "clocks": clk.summary()}
        del graph, sg
        stack.close()
        del stack
        torch.cuda.empty_cache()
    w_bytes = 2 * (shape.d_model * (2 * shape.d_inner + 2 * shape.groups * shape.state_dim + shape.heads)
                   + shape.d_inner * shape.d_model)
    print(json.dumps({"diagnostic": "synthetic decode stack", "workload": w.name, "layers": shape.layers,
                      "batch": shape.batch, "d_model": shape.d_model, "d_inner": shape.d_inner, "k": k,
                      "checkpoint": w.ckpt, "read_fmt": w.read_fmt, "steps": reps * k, "warmup": W + k,
                      "cuda_graph": f"one window of {k} steps", "weight_bytes_per_layer": w_bytes,
                      "replay": res["replay"], "conventional": res["conventional"],
                      "step_speedup": res["conventional"]["ms_per_step"] / res["replay"]["ms_per_step"]}),
          flush=True)


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6400)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="rssm", choices=["rssm", "reference"])
    ap.add_argument("--workload", default="mamba2_serving_b256",
                    choices=[k for k in synth.WORKLOADS if k != "mamba2_fp32_b4"])
    ap.add_argument("--mode", default="replay", choices=["replay", "conventional"])
    ap.add_argument("--k", type=int, default=0, help="flush threshold (default: the workload's 16)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling)")
    ap.add_argument("--pool", type=int, default=64, help="distinct input steps resident in HBM")
    ap.add_argument("--no-compare", action="store_true", help="skip the conventional-kernel run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--graph", action="store_true",
                    help="plain decode: also time one window replayed from a CUDA graph")
    ap.add_argument("--no-sub", action="store_true",
                    help="default workload only: skip the brief runs of the other workloads")
    ap.add_argument("--stack", type=int, default=0,
                    help="diagnostic: decode-step time of a synthetic stack of this many layers")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.stack:
        stack_bench(args)
        return
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import torch
    import hybrid_ssm_decode_gb300 as rssm
    rssm.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=device)
        dist = tdist

    w = synth.WORKLOADS[args.workload]
    if args.workload.startswith("mamba2_spec"):
        res = spec_arm(torch, rssm, args, device, dist)
    elif args.workload.startswith("gdn_spec"):
        res = gdn_spec_arm(torch, rssm, args, device, dist)
    elif isinstance(w, synth.GDNWorkload):
        res = gdn_arm(torch, rssm, args, device, dist)
    else:
        res = m2_arm(torch, rssm, args, device, dist)

    from hybrid_ssm_decode_gb300.replicas import aggregate
    w = res["w"]
    K = args.steps
    tokens, total_ms = aggregate(res.get("tokens", w.batch * K), res["total_ms"], dist, device)
    value = tokens / (total_ms / 1e3)

    peak, peak_kind = measured_peaks()

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "mode": args.mode, "batch": w.batch,
                       "inputs": w.dtype, "checkpoint": getattr(w, "ckpt", "f32"), "k": w.k,
                       "l2": res.get("l2", "state streamed every step exceeds L2 (no extra flush)"),
                       "parallelism": f"{world} independent replica(s), no collective"}}
    if isinstance(w, synth.Mamba2Workload):
        line["config"].update({"heads": w.heads, "head_dim": w.head_dim, "state_dim": w.state_dim,
                               "groups": w.groups, "read_fmt": w.read_fmt})
    else:
        line["config"].update({"heads": w.heads, "d_k": w.d_k, "d_v": w.d_v, "read_fmt": w.read_fmt})
    if "draft" in res:
        line["config"]["draft"] = res["draft"]
    if res.get("layers", 1) > 1:
        line["config"]["layers"] = res["layers"]
    line["roofline"] = roofline_of(res, args.mode, args.warmup, peak, peak_kind)
    line["gpu_launches"] = res.get("launches", K)
    line["clocks"] = res["clocks"]
    if "conv" in res:
        cv = res["conv"]
        cval = w.batch * K * world / (cv["total_ms"] / 1e3)
        cach = (sum(cv["bytes"]) / len(cv["bytes"])) / (sum(cv["per"]) / len(cv["per"]) / 1e3) / 1e9
        line["conventional"] = {"value": cval, "unit": UNIT, "ms_per_step": cv["total_ms"] / K,
                                "gbs": cach, "frac": cach / peak, "speedup": value / cval}
        # state bytes per window moved by each (algorithmic)
    if res.get("graph"):
        gr = res["graph"]
        line["graph"] = {"value": w.batch * world / (gr["ms_per_step"] / 1e3), "unit": UNIT,
                         "ms_per_step": gr["ms_per_step"], "steps": gr["steps"],
                         "note": "one window of k steps (of every layer) captured as a CUDA graph and replayed"}
        cg = res.get("conv", {}).get("graph")
        if cg:
            line["graph"]["conventional_value"] = w.batch * world / (cg["ms_per_step"] / 1e3)
            line["graph"]["speedup"] = cg["ms_per_step"] / gr["ms_per_step"]
    if "e2e" in res:
        e = res["e2e"]
        line["e2e"] = {"value": w.batch * K * world / (e["total_ms"] / 1e3), "unit": UNIT,
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]}
    for key in ("spec",):
        if key in res:
            line[key] = res[key]
    if world == 1 and not args.no_sub and args.workload == "mamba2_serving_b256" and not args.k \
            and not args.batch and args.mode == "replay":
        subs = {}
        for n in SUB_WORKLOADS:
            subs[n] = sub_record(torch, rssm, args, n, device, peak, peak_kind, value, subs)
        line["workloads"] = subs
        line["plain_after_verify"] = spec_then_plain(torch, rssm, device)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(args.workload if args.workload in
                                            ("mamba2_serving_b256", "gdn_serving_b256") else
                                            "mamba2_serving_b256")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
