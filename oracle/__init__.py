"""Float64 CPU oracle for the ReplaySSM decode path.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The CUDA path neither
imports it nor shares code with it.

The arithmetic lives in ``rssm_oracle.c`` (plain C, float64, OpenMP over
(sequence, head) tiles). This module builds that library with gcc and wraps
it with numpy arrays. The speculative-decode driver at the bottom is plain
Python over the same C recurrence.

Pinned by ``tests/test_oracle_pins.py`` (closed forms, brute-force matrix
products, special cases) and by ``tests/test_quant_spec.py`` (OCP FP8/FP4
value tables). Every function has at least one pin there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rssm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "librssm_oracle.so")
_lock = threading.Lock()
_lib = None

FMT = {"fp8": 1, "nvfp4": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, f64, p = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.orc_m2_recurrence.argtypes = [i64] * 6 + [p] * 9 + [i32]
            lib.orc_m2_recurrence.restype = i32
            lib.orc_m2_readcopy.argtypes = [i64] * 6 + [p] * 7 + [i64, i32, p, i32]
            lib.orc_m2_readcopy.restype = i32
            lib.orc_gdn_recurrence.argtypes = [i64] * 5 + [f64] + [p] * 8 + [i32]
            lib.orc_gdn_recurrence.restype = i32
            lib.orc_e4m3_encode_array.argtypes = [i64, p, p]
            lib.orc_e2m1_encode_array.argtypes = [i64, p, p]
            lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_decode.restype = f64
            lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_decode.restype = f64
            lib.orc_quant_fp8.argtypes = [i64, i64, p, p, p]
            lib.orc_quant_nvfp4.argtypes = [i64, i64, i64, p, p, p, p]
            lib.orc_quant_nvfp4.restype = i32
            lib.orc_dequant_fp8.argtypes = [i64, i64, p, p, p]
            lib.orc_dequant_nvfp4.argtypes = [i64, i64, i64, p, p, p, p]
            lib.orc_max_threads.restype = i32
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().orc_max_threads())


# --------------------------------------------------------------------------
# Mamba-2
# --------------------------------------------------------------------------
def m2_recurrence(h0, A, D, x, Bm, C, dt, nsteps=None, threads=0):
    """Per-token Mamba-2 recurrence in float64.

    h0 [B][H][P][N]; x [S][B][H][P]; Bm, C [S][B][G][N]; dt [S][B][H];
    A, D [H]. Returns (y [S][B][H][P], h [B][H][P][N]). With `nsteps` [B],
    sequence b runs only its first nsteps[b] tokens (later y rows are NaN).
    """
    h = np.array(h0, dtype=np.float64, order="C", copy=True)
    x, Bm, C, dt = (_c(a, np.float64) for a in (x, Bm, C, dt))
    A, D = _c(A, np.float64), _c(D, np.float64)
    S, B, H, P = x.shape
    N, G = h.shape[3], Bm.shape[2]
    y = np.full((S, B, H, P), np.nan)
    ns = None if nsteps is None else _c(nsteps, np.int32)
    rc = _load().orc_m2_recurrence(B, H, P, N, G, S, _ptr(A), _ptr(D), _ptr(h), _ptr(x),
                                   _ptr(Bm), _ptr(C), _ptr(dt), _ptr(ns), _ptr(y), threads)
    if rc:
        raise ValueError("orc_m2_recurrence: invalid arguments")
    return y, h


def m2_readcopy(h0, A, D, x, Bm, C, dt, k, fmt, threads=0):
    """Mamba-2 plain decode whose non-flush outputs read a low-precision copy
    of the checkpoint (fmt 'fp8' or 'nvfp4') made at start and at every flush
    (every k tokens). Returns y [S][B][H][P]."""
    h = np.array(h0, dtype=np.float64, order="C", copy=True)
    x, Bm, C, dt = (_c(a, np.float64) for a in (x, Bm, C, dt))
    A, D = _c(A, np.float64), _c(D, np.float64)
    S, B, H, P = x.shape
    N, G = h.shape[3], Bm.shape[2]
    y = np.empty((S, B, H, P))
    rc = _load().orc_m2_readcopy(B, H, P, N, G, S, _ptr(A), _ptr(D), _ptr(h), _ptr(x), _ptr(Bm),
                                 _ptr(C), _ptr(dt), k, FMT[fmt], _ptr(y), threads)
    if rc:
        raise ValueError("orc_m2_readcopy: invalid arguments")
    return y


def m2_qrecurrence(h0, A, D, x, Bm, C, dt, fmt):
    """The quantised-recurrence baseline ("NVIDIA ve Dao AI Lab, ... ReplaySSM'i
    sundu", section "Kuantizasyon hatasinin sinirlandirilmasi": a quantised
    SSM state recurs, so its rounding error accumulates with length). The
    Mamba-2 state lives in a low-precision tile format (fmt 'fp8' or 'nvfp4',
    the read-copy formats). It is quantised at the start; then every token
    dequantises it, applies the decode step in float64, emits
    y = h C + D x from the updated state, and quantises the updated state
    (rounded to float32, the quantisers' input type) for the next token.
    Returns y [S][B][H][P]. Plain numpy over the library quantisers above.
    """
    h = np.array(h0, dtype=np.float64)
    x, Bm, C, dt = (np.asarray(a, np.float64) for a in (x, Bm, C, dt))
    A, D = np.asarray(A, np.float64), np.asarray(D, np.float64)
    S, B, H, P = x.shape
    N, G = h.shape[3], Bm.shape[2]
    grp = np.arange(H) // (H // G)                     # head -> B/C group
    tiles = h.reshape(B * H, P, N)

    def quant(t):
        t32 = t.astype(np.float32)
        return quant_fp8(t32) if fmt == "fp8" else quant_nvfp4(t32)

    def dequant(q):
        return dequant_fp8(*q) if fmt == "fp8" else dequant_nvfp4(*q)

    q = quant(tiles)
    y = np.empty((S, B, H, P))
    for s in range(S):
        h = dequant(q).reshape(B, H, P, N)
        a = np.exp(dt[s] * A[None, :])                   # [B][H]
        Bs, Cs = Bm[s][:, grp], C[s][:, grp]             # [B][H][N]
        h = a[..., None, None] * h + (dt[s][..., None] * x[s])[..., None] * Bs[:, :, None, :]
        y[s] = np.einsum("bhpn,bhn->bhp", h, Cs) + D[None, :, None] * x[s]
        q = quant(h.reshape(B * H, P, N))
    return y


def round_f16(a) -> np.ndarray:
    """An FP32 value rounded to IEEE binary16 (round to nearest, ties to
    even), returned as float64. Inputs are first rounded to float32."""
    with np.errstate(over="ignore"):
        return np.asarray(a, np.float64).astype(np.float32).astype(np.float16).astype(np.float64)


def store_tiles(h, store) -> np.ndarray:
    """The checkpoint h [B][H][P][N] as stored (float64 values): rounded to
    FP16 ("f16"), or each (sequence, head) tile quantised to the FP8 or NVFP4
    tile format ("fp8", "nvfp4": the read-copy formats) and decoded."""
    h = np.asarray(h, np.float64)
    if store == "f16":
        return round_f16(h)
    tiles = h.reshape(-1, h.shape[-2], h.shape[-1]).astype(np.float32)
    if store == "fp8":
        d = dequant_fp8(*quant_fp8(tiles))
    elif store == "nvfp4":
        d = dequant_nvfp4(*quant_nvfp4(tiles))
    else:
        raise ValueError(store)
    return d.reshape(h.shape)


def m2_ckpt_lowp(h0, A, D, x, Bm, C, dt, k, store, fmt=None, windows=None, start_stored=False, threads=0):
    """Mamba-2 replay decode with a low-precision checkpoint ("NVIDIA ve Dao AI
    Lab, ... ReplaySSM'i sundu", section "Kuantizasyon hatasinin
    sinirlandirilmasi": the recurrence checkpoint kept in FP16 or FP8 with
    NVFP4 reads, against a full NVFP4 checkpoint). `store` is the checkpoint
    format (store_tiles). The checkpoint is h0 as stored. Each commit window
    continues the float64 recurrence from the stored checkpoint; its outputs
    are those of that recurrence (or, with fmt 'fp8'/'nvfp4', of the
    read-copy decode whose copy is made from the stored values, the window's
    k-th token being the flush token that reads the checkpoint itself). At
    the window's end the state after its tokens is stored as the new
    checkpoint.

    windows: lengths of the successive commit windows (each <= k; a window of
    length k ends in the automatic flush, a shorter one in an explicit
    flush). Default: windows of k, with any remainder left uncommitted.
    start_stored: h0 is already a stored checkpoint (continuing a decode).
    Returns (y [S][B][H][P], checkpoint after the last commit [B][H][P][N]).
    """
    S = np.shape(x)[0]
    if windows is None:
        windows = [k] * (S // k)
        tail = S - k * len(windows)
    else:
        windows = list(windows)
        tail = S - sum(windows)
        if tail < 0 or tail >= k or any(w < 1 or w > k for w in windows):
            raise ValueError("m2_ckpt_lowp: bad windows")
    ck = np.array(h0, np.float64) if start_stored else store_tiles(h0, store)
    ys = []
    start = 0
    for n, commit in [(w, True) for w in windows] + ([(tail, False)] if tail else []):
        sl = slice(start, start + n)
        args = (x[sl], Bm[sl], C[sl], dt[sl])
        y, h_end = m2_recurrence(ck, A, D, *args, threads=threads)
        if fmt is not None:
            y = m2_readcopy(ck, A, D, *args, k, fmt, threads=threads)
        ys.append(y)
        if commit:
            ck = store_tiles(h_end, store)
        start += n
    return np.concatenate(ys) if ys else np.empty((0,) + np.shape(x)[1:]), ck


def m2_ckpt16(h0, A, D, x, Bm, C, dt, k, fmt=None, windows=None, threads=0):
    """m2_ckpt_lowp with the checkpoint in FP16 (IEEE binary16, round to
    nearest even from the float32 value)."""
    return m2_ckpt_lowp(h0, A, D, x, Bm, C, dt, k, "f16", fmt=fmt, windows=windows, threads=threads)


def m2_speculative(h0, A, D, x, Bm, C, dt, accepted, threads=0):
    """Speculative rounds on the Mamba-2 recurrence.

    x [R][T][B][H][P] etc. are the T draft tokens of each of R rounds;
    accepted [R][B] in 0..T. In each round the draft outputs are the recurrence
    continued from the committed state (on a copy). Then the committed state
    advances by accepted[r][b] of those tokens. Rejected drafts never touch it.
    Returns (y [R][T][B][H][P], committed state after the last round).
    """
    h = np.array(h0, dtype=np.float64, copy=True)
    R, T = x.shape[0], x.shape[1]
    ys = []
    for r in range(R):
        y, _ = m2_recurrence(h, A, D, x[r], Bm[r], C[r], dt[r], threads=threads)
        ys.append(y)
        _, h = m2_recurrence(h, A, D, x[r], Bm[r], C[r], dt[r], nsteps=accepted[r],
                             threads=threads)
    return np.stack(ys), h


def m2_speculative_readcopy(h0, A, D, x, Bm, C, dt, accepted, k, fmt, threads=0):
    """Speculative rounds whose draft outputs read a low-precision copy of the
    checkpoint ("NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", sections "Durum
    trafigini azaltma ve rollback'in basitlestirilmesi" and "Kuantizasyon
    hatasinin sinirlandirilmasi": drafts are appended to the buffer, and reads
    may come from the low-precision copy while the recurrence stays on the
    high-precision checkpoint).

    Each sequence's state is its checkpoint (its state at its last fold; h0 at
    the start) plus the tokens committed since. A draft's output is the
    recurrence's output continued from the committed state, with the
    checkpoint's term read from the copy instead:
        y = y_exact + gamma (copy - ckpt) C,
    gamma = exp(A * sum of dt over the tokens since the checkpoint, up to and
    including the draft). The copy is the read-copy format's quantisation of
    the checkpoint (store_tiles). After each verify the committed state
    advances by accepted[r][b] drafts; a sequence whose tokens since its
    checkpoint reach k folds them: its checkpoint becomes its state and its
    copy is remade. Rejected drafts touch nothing.

    x [R][T][B][H][P] etc. as m2_speculative. Returns (y [R][T][B][H][P],
    committed state, checkpoint)."""
    h = np.array(h0, np.float64, copy=True)
    ck = h.copy()
    cp = store_tiles(ck, fmt)
    A = np.asarray(A, np.float64)
    R, T, B, H, P = np.shape(x)
    G = np.shape(Bm)[3]
    grp = np.arange(H) // (H // G)
    since = np.zeros((B, H))                    # sum of dt since the checkpoint
    count = np.zeros(B, np.int64)               # tokens since the checkpoint
    ys = []
    for r in range(R):
        y, _ = m2_recurrence(h, A, D, x[r], Bm[r], C[r], dt[r], threads=threads)
        dtr = np.asarray(dt[r], np.float64)
        gam = np.exp(A[None, None, :] * (since[None] + np.cumsum(dtr, axis=0)))     # [T][B][H]
        Ch = np.asarray(C[r], np.float64)[:, :, grp]                                # [T][B][H][N]
        corr = np.einsum("bhpn,tbhn->tbhp", cp - ck, Ch)
        ys.append(y + gam[..., None] * corr)
        acc = np.asarray(accepted[r], np.int64)
        _, h = m2_recurrence(h, A, D, x[r], Bm[r], C[r], dt[r], nsteps=acc, threads=threads)
        for b in range(B):
            since[b] += dtr[: acc[b], b].sum(axis=0)
        count = count + acc
        fold = count >= k
        if fold.any():
            ck[fold] = h[fold]
            cp[fold] = store_tiles(h[fold], fmt)
            since[fold] = 0.0
            count[fold] = 0
    return np.stack(ys), h, ck


# --------------------------------------------------------------------------
# Synthetic decode stack (context for the step-level speedup)
# --------------------------------------------------------------------------
def round_bf16(a) -> np.ndarray:
    """Values rounded to bfloat16 (via float32; round to nearest, ties to
    even), returned as float64. Inputs are finite."""
    bits = np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32)).view(np.uint32).astype(np.uint64)
    r = ((bits + np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)) << np.uint64(16)
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def m2_stack(u_steps, weights, params, states, threads=0):
    """The synthetic Mamba-2 decode stack in float64 with its bf16 storage
    points. Per layer and step, for the hidden state u [B][d_model]:
    n = bf16(u / sqrt(mean(u^2) + 1e-6)); x = bf16(n W_x); z = bf16(n W_z);
    B = bf16(n W_B); C = bf16(n W_C); dt = bf16(softplus(bf16(n W_dt) + dt_bias));
    y = bf16(Mamba-2 step of the layer's state); g = bf16(y * bf16(silu(z)));
    delta = bf16(g W_out); u = bf16(u + delta). Softplus(v) = log(1 + e^v),
    silu(v) = v / (1 + e^-v), RMS normalisation without a weight.

    u_steps [S][B][d_model]: the input embedding of each step. weights: per
    layer a dict of float64 arrays x, z, B, C, dt ([d_model][...]), out
    ([d_inner][d_model]) and dt_bias [H]. params: per layer (A, D). states:
    per layer h [B][H][P][N] (copied). Returns (u_out [S][B][d_model],
    deltas [S][layers][B][d_model], final states).
    """
    states = [np.array(h, np.float64, copy=True) for h in states]
    S = len(u_steps)
    L = len(weights)
    outs, deltas = [], []
    for t in range(S):
        u = np.asarray(u_steps[t], np.float64)
        dl = []
        for li in range(L):
            w, (A, D), h = weights[li], params[li], states[li]
            Bsz, H, P, N = h.shape
            G = w["B"].shape[1] // N
            n = round_bf16(u / np.sqrt(np.mean(u * u, axis=-1, keepdims=True) + 1e-6))
            x = round_bf16(n @ w["x"]).reshape(1, Bsz, H, P)
            z = round_bf16(n @ w["z"])
            Bt = round_bf16(n @ w["B"]).reshape(1, Bsz, G, N)
            Ct = round_bf16(n @ w["C"]).reshape(1, Bsz, G, N)
            v = round_bf16(n @ w["dt"]) + np.asarray(w["dt_bias"], np.float64)
            dt = round_bf16(np.logaddexp(0.0, v)).reshape(1, Bsz, H)
            y, states[li] = m2_recurrence(h, A, D, x, Bt, Ct, dt, threads=threads)
            y = round_bf16(y[0]).reshape(Bsz, H * P)
            g = round_bf16(y * round_bf16(z / (1.0 + np.exp(-z))))
            delta = round_bf16(g @ w["out"])
            u = round_bf16(u + delta)
            dl.append(delta)
        outs.append(u)
        deltas.append(np.stack(dl))
    return np.stack(outs), np.stack(deltas), states


# --------------------------------------------------------------------------
# Gated DeltaNet
# --------------------------------------------------------------------------
def gdn_recurrence(S0, q, k, v, alpha, beta, scale=1.0, nsteps=None, threads=0):
    """Per-token Gated DeltaNet recurrence in float64.

    S0 [B][H][DV][DK]; q, k [S][B][H][DK]; v [S][B][H][DV]; alpha, beta [S][B][H].
    Returns (o [S][B][H][DV], S [B][H][DV][DK])."""
    St = np.array(S0, dtype=np.float64, order="C", copy=True)
    q, k, v, alpha, beta = (_c(a, np.float64) for a in (q, k, v, alpha, beta))
    S, B, H, DK = q.shape
    DV = v.shape[3]
    o = np.full((S, B, H, DV), np.nan)
    ns = None if nsteps is None else _c(nsteps, np.int32)
    rc = _load().orc_gdn_recurrence(B, H, DK, DV, S, float(scale), _ptr(St), _ptr(q), _ptr(k),
                                    _ptr(v), _ptr(alpha), _ptr(beta), _ptr(ns), _ptr(o), threads)
    if rc:
        raise ValueError("orc_gdn_recurrence: invalid arguments")
    return o, St


# --------------------------------------------------------------------------
# Quantisers
# --------------------------------------------------------------------------
def gdn_speculative(S0, q, k, v, alpha, beta, accepted, scale=1.0, threads=0):
    """Speculative rounds on the Gated DeltaNet recurrence (the GDN form of
    m2_speculative). q, k [R][T][B][H][d_k], v [R][T][B][H][d_v],
    alpha, beta [R][T][B][H] are the T draft tokens of each of R rounds;
    accepted [R][B] in 0..T. Each round's draft outputs continue the
    recurrence from the committed state (on a copy); then the committed
    state advances by accepted[r][b] of those tokens. Returns
    (o [R][T][B][H][d_v], committed state after the last round)."""
    S = np.array(S0, dtype=np.float64, copy=True)
    R, T = q.shape[0], q.shape[1]
    os_ = []
    for r in range(R):
        o, _ = gdn_recurrence(S, q[r], k[r], v[r], alpha[r], beta[r], scale=scale, threads=threads)
        os_.append(o)
        for b in range(S.shape[0]):
            a = int(accepted[r][b])
            if a:
                sl = slice(b, b + 1)
                _, Sb = gdn_recurrence(S[sl], q[r][:a, sl], k[r][:a, sl], v[r][:a, sl], alpha[r][:a, sl],
                                       beta[r][:a, sl], scale=scale, threads=threads)
                S[b] = Sb[0]
    return np.stack(os_), S


def gdn_speculative_readcopy(S0, q, k, v, alpha, beta, accepted, kflush, fmt, scale=1.0, threads=0):
    """Gated DeltaNet speculative rounds whose drafts read the low-precision
    copy of the checkpoint ("NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu",
    sections "Durum trafigini azaltma ve rollback'in basitlestirilmesi" and
    "Kuantizasyon hatasinin sinirlandirilmasi"; the GDN form of
    m2_speculative_readcopy). Each sequence keeps its checkpoint (its state at
    its last fold; S0 at the start) and the tokens committed since. A round's
    draft outputs are the recurrence continued from the copy of the checkpoint
    (gdn_copy) through the committed tokens and the drafts; after the verify a
    sequence whose tokens since its checkpoint reach kflush folds them with
    the exact recurrence from the checkpoint. Rejected drafts touch nothing.

    q, k [R][T][B][H][d_k], v [R][T][B][H][d_v], alpha, beta [R][T][B][H];
    accepted [R][B]. Returns (o [R][T][B][H][d_v], committed state,
    checkpoint)."""
    ck = np.array(S0, dtype=np.float64, copy=True)
    R, T, B = np.shape(q)[0], np.shape(q)[1], np.shape(q)[2]
    hist = [[] for _ in range(B)]     # per sequence: (round, accepted) since the fold
    outs = np.empty((R, T) + (B,) + np.shape(v)[3:])
    args = (q, k, v, alpha, beta)

    def tokens(b, r, n):
        return [a[r][:n, b:b + 1] for a in args]

    for r in range(R):
        for b in range(B):
            pre = [tokens(b, rr, n) for rr, n in hist[b]]
            seq = [np.concatenate([p[i] for p in pre] + [a[r][:, b:b + 1]]) for i, a in enumerate(args)]
            o, _ = gdn_recurrence(gdn_copy(ck[b:b + 1], fmt), *seq, scale=scale, threads=threads)
            outs[r, :, b] = o[-T:, 0]
        for b in range(B):
            n = int(accepted[r][b])
            if n:
                hist[b].append((r, n))
            if sum(x for _, x in hist[b]) >= kflush:
                seq = [np.concatenate([tokens(b, rr, m)[i] for rr, m in hist[b]]) for i in range(5)]
                _, Sb = gdn_recurrence(ck[b:b + 1], *seq, scale=scale, threads=threads)
                ck[b] = Sb[0]
                hist[b] = []
    state = ck.copy()
    for b in range(B):
        if hist[b]:
            seq = [np.concatenate([tokens(b, rr, m)[i] for rr, m in hist[b]]) for i in range(5)]
            _, Sb = gdn_recurrence(ck[b:b + 1], *seq, scale=scale, threads=threads)
            state[b] = Sb[0]
    return outs, state, ck


def gdn_copy(S, fmt) -> np.ndarray:
    """The low-precision read copy of a Gated DeltaNet state [B][H][d_v][d_k],
    dequantised: each 64-row half of a (sequence, head) tile is one tile of
    the read-copy format (its values rounded to float32 first)."""
    S = np.asarray(S, np.float64)
    B, H, DV, DK = S.shape
    halves = S.reshape(B * H * DV // 64, 64, DK).astype(np.float32)
    if fmt == "fp8":
        d = dequant_fp8(*quant_fp8(halves))
    else:
        d = dequant_nvfp4(*quant_nvfp4(halves))
    return d.reshape(S.shape)


def gdn_ckpt16(S0, q, k, v, alpha, beta, kflush, scale=1.0, windows=None, threads=0):
    """Gated DeltaNet replay with an FP16 checkpoint ("NVIDIA ve Dao AI Lab,
    ... ReplaySSM'i sundu", section "Kuantizasyon hatasinin
    sinirlandirilmasi": an FP16 recurrence checkpoint). The stored
    checkpoint is the state rounded to binary16 at the start and after every
    commit; within a window every output is the recurrence continued from the
    stored checkpoint (float64 arithmetic), the flush token's included, and
    the commit stores the window's end state rounded to binary16.

    windows: lengths of the successive commit windows as in gdn_readcopy.
    Returns (o [S][B][H][d_v], stored checkpoint after the last commit, as
    float64 values)."""
    steps = np.shape(q)[0]
    if windows is None:
        windows = [kflush] * (steps // kflush)
    else:
        windows = list(windows)
        if any(n < 1 or n > kflush for n in windows):
            raise ValueError("gdn_ckpt16: bad windows")
    tail = steps - sum(windows)
    if tail < 0 or tail >= kflush:
        raise ValueError("gdn_ckpt16: bad windows")
    S = round_f16(S0)
    out, start = [], 0
    for n, commit in [(n, True) for n in windows] + ([(tail, False)] if tail else []):
        sl = slice(start, start + n)
        o, S_end = gdn_recurrence(S, q[sl], k[sl], v[sl], alpha[sl], beta[sl], scale=scale, threads=threads)
        out.append(o)
        if commit:
            S = round_f16(S_end)
        start += n
    return np.concatenate(out), S


def gdn_qrecurrence(S0, q, k, v, alpha, beta, fmt, scale=1.0, threads=0):
    """The quantised-recurrence baseline for Gated DeltaNet ("NVIDIA ve Dao AI
    Lab, ... ReplaySSM'i sundu", section "Kuantizasyon hatasinin
    sinirlandirilmasi": a quantised state recurs, so its rounding error
    accumulates with length). The state [B][H][d_v][d_k] lives in the
    read-copy tile format (fmt 'fp8' or 'nvfp4'), one tile per 64-row half of
    each (sequence, head) state, as the GDN read copy is laid out. It is
    quantised at the start; then every token dequantises it, applies the
    decode step in float64 (gdn_recurrence over that one token), emits its
    output from the updated state, and quantises the updated state (rounded
    to float32, the quantisers' input type) for the next token.
    Returns o [S][B][H][d_v]."""
    St = np.asarray(S0, np.float64)
    B, H, DV, DK = St.shape
    steps = np.shape(q)[0]

    def quant(t):
        halves = t.reshape(B * H * DV // 64, 64, DK).astype(np.float32)
        return quant_fp8(halves) if fmt == "fp8" else quant_nvfp4(halves)

    def dequant(c):
        d = dequant_fp8(*c) if fmt == "fp8" else dequant_nvfp4(*c)
        return d.reshape(B, H, DV, DK)

    cur = quant(St)
    out = np.empty((steps, B, H, DV))
    for s in range(steps):
        sl = slice(s, s + 1)
        o, St = gdn_recurrence(dequant(cur), q[sl], k[sl], v[sl], alpha[sl], beta[sl], scale=scale,
                               threads=threads)
        out[s] = o[0]
        cur = quant(St)
    return out


def gdn_readcopy(S0, q, k, v, alpha, beta, kflush, fmt, scale=1.0, windows=None, threads=0):
    """Gated DeltaNet replay decode whose outputs read a low-precision copy of
    the checkpoint ("NVIDIA ve Dao AI Lab, ... ReplaySSM'i sundu", section
    "Kuantizasyon hatasinin sinirlandirilmasi": the high-precision checkpoint
    carries the recurrence, the low-precision copy serves reads). The copy
    (gdn_copy) is made at the start of each commit window. A token's output
    is that of the recurrence continued from the copy through the window's
    tokens so far; the token that completes a k-token window is the flush
    token and reads the checkpoint itself. The checkpoint follows the float64
    recurrence exactly.

    windows: lengths of the successive commit windows (each <= kflush; one of
    length kflush ends in the automatic flush, a shorter one in an explicit
    flush). Default: windows of kflush, any remainder uncommitted.
    Returns (o [S][B][H][d_v], checkpoint after the last commit)."""
    S = np.array(S0, dtype=np.float64, copy=True)
    steps = np.shape(q)[0]
    if windows is None:
        windows = [kflush] * (steps // kflush)
        tail = steps - kflush * len(windows)
    else:
        windows = list(windows)
        tail = steps - sum(windows)
        if tail < 0 or tail >= kflush or any(n < 1 or n > kflush for n in windows):
            raise ValueError("gdn_readcopy: bad windows")
    out = []
    start = 0
    for n, commit in [(n, True) for n in windows] + ([(tail, False)] if tail else []):
        sl = slice(start, start + n)
        args = (q[sl], k[sl], v[sl], alpha[sl], beta[sl])
        o_ex, S_end = gdn_recurrence(S, *args, scale=scale, threads=threads)
        o, _ = gdn_recurrence(gdn_copy(S, fmt), *args, scale=scale, threads=threads)
        if n == kflush:
            o[-1] = o_ex[-1]
        out.append(o)
        if commit:
            S = S_end
        start += n
    return np.concatenate(out), S


def e4m3_encode(a) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().orc_e4m3_encode_array(a.size, _ptr(a), _ptr(out))
    return out


def e2m1_encode(a) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint8)
    _load().orc_e2m1_encode_array(a.size, _ptr(a), _ptr(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, np.uint8)
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c.ravel()]).reshape(c.shape)


def e2m1_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, np.uint8)
    return np.array([lib.orc_e2m1_decode(int(v)) for v in c.ravel()]).reshape(c.shape)


def quant_fp8(tiles: np.ndarray):
    """tiles [T][...] float32 -> (codes uint8 same shape, scale float32 [T])."""
    t = _c(tiles, np.float32)
    n = t[0].size if t.shape[0] else 0
    codes = np.empty(t.shape, np.uint8)
    scale = np.empty(t.shape[0], np.float32)
    _load().orc_quant_fp8(t.shape[0], n, _ptr(t), _ptr(codes), _ptr(scale))
    return codes, scale


def dequant_fp8(codes, scale) -> np.ndarray:
    codes, scale = _c(codes, np.uint8), _c(scale, np.float32)
    out = np.empty(codes.shape)
    n = codes[0].size if codes.shape[0] else 0
    _load().orc_dequant_fp8(codes.shape[0], n, _ptr(codes), _ptr(scale), _ptr(out))
    return out


def quant_nvfp4(tiles: np.ndarray):
    """tiles [T][rows][cols] float32 -> (codes uint8 [T][rows][cols/2],
    block scales uint8 [T][rows][cols/16], tile scale float32 [T])."""
    t = _c(tiles, np.float32)
    T, rows, cols = t.shape
    codes = np.empty((T, rows, cols // 2), np.uint8)
    bsc = np.empty((T, rows, cols // 16), np.uint8)
    ts = np.empty(T, np.float32)
    if _load().orc_quant_nvfp4(T, rows, cols, _ptr(t), _ptr(codes), _ptr(bsc), _ptr(ts)):
        raise ValueError("cols must be a multiple of 16")
    return codes, bsc, ts


def dequant_nvfp4(codes, bsc, ts) -> np.ndarray:
    codes, bsc, ts = _c(codes, np.uint8), _c(bsc, np.uint8), _c(ts, np.float32)
    T, rows, half = codes.shape
    out = np.empty((T, rows, half * 2))
    _load().orc_dequant_nvfp4(T, rows, half * 2, _ptr(codes), _ptr(bsc), _ptr(ts), _ptr(out))
    return out
