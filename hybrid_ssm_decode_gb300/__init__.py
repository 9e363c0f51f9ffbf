"""Python binding of librssm, the ReplaySSM decode step for GB300 (sm_103a).

Argument marshalling only. Every step of the decode path runs in the CUDA
kernels behind the C ABI declared in ``include/rssm.h``. There is no CPU
fallback: ``load()`` raises if the library has not been built.

The functions keep the C names (``rssm_create``, ``rssm_decode_step``, ...)
and take torch CUDA tensors, or raw device addresses, where the C ABI takes
device pointers. ``Layer`` bundles a workspace tensor and a handle for
convenience.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_BUILD = os.path.join(_PKG, "_build")
LIB_PATH = os.path.join(_PKG, "librssm.so")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-I" + _INCLUDE]

# status codes and enums (include/rssm.h)
RSSM_OK, RSSM_ERR_INVALID_ARG, RSSM_ERR_UNSUPPORTED, RSSM_ERR_CAPACITY, RSSM_ERR_CUDA, \
    RSSM_ERR_STATE = range(6)
RSSM_MAMBA2, RSSM_GDN = 1, 2
RSSM_REPLAY, RSSM_CONVENTIONAL = 1, 2
RSSM_F32, RSSM_BF16, RSSM_F16 = 1, 2, 3
RSSM_CKPT_FP8, RSSM_CKPT_NVFP4 = 4, 5
CKPT_DTYPE = {"f32": RSSM_F32, "f16": RSSM_F16, "fp8": RSSM_CKPT_FP8, "nvfp4": RSSM_CKPT_NVFP4}
RSSM_READ_NONE, RSSM_READ_FP8, RSSM_READ_NVFP4 = 0, 1, 2
RSSM_DEV_OK, RSSM_DEV_ACCEPTED_RANGE, RSSM_DEV_COUNT_RANGE, RSSM_DEV_TIMEOUT = 0, 1, 2, 3

READ_FMT = {"none": RSSM_READ_NONE, "fp8": RSSM_READ_FP8, "nvfp4": RSSM_READ_NVFP4}
DTYPE = {"f32": RSSM_F32, "bf16": RSSM_BF16}


class RssmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({status_string(status)})")


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kind", "mode", "batch", "heads", "head_dim", "state_dim", "groups", "k",
                 "max_draft", "in_dtype", "out_dtype", "read_fmt")] + [("gdn_scale", ctypes.c_float),
                                                                       ("ckpt_dtype", ctypes.c_int32)]


class Inputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "Bm", "C", "dt", "q", "k", "v", "alpha", "beta")]


_LAYOUT_REGIONS = ("ckpt", "counts", "err", "buf_x", "buf_b", "buf_dt", "buf_k", "buf_u",
                   "buf_a", "rc_codes", "rc_bscale", "rc_tscale", "snap", "buf_v", "buf_beta",
                   "ckpt_bscale", "ckpt_tscale", "cnt_hist")


class Layout(ctypes.Structure):
    _fields_ = ([(f, ctypes.c_size_t) for r in _LAYOUT_REGIONS for f in (r, r + "_bytes")]
                + [("total_bytes", ctypes.c_size_t), ("capacity", ctypes.c_int32)])


# --------------------------------------------------------------------------
# build / load
# --------------------------------------------------------------------------
def _sources():
    return sorted(os.path.join(_CSRC, f) for f in os.listdir(_CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(_INCLUDE, f) for f in os.listdir(_INCLUDE) if f.endswith(".h")]
    return _sources() + hdrs


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a (one translation unit per process, in
    parallel) and link librssm.so in the package directory."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(_BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = ["nvcc", *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, len(_sources()))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run(["nvcc", "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_lib = None
_lock = threading.Lock()


def load():
    """Load librssm.so. Raises if it is missing or older than its sources:
    the CUDA path has no fallback."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"librssm.so is not built ({LIB_PATH}); run "
                              "hybrid_ssm_decode_gb300.build() or __graft_entry__.build()")
        if is_stale():
            raise ImportError("librssm.so is older than its sources; rebuild it with "
                              "hybrid_ssm_decode_gb300.build()")
        lib = ctypes.CDLL(LIB_PATH)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "rssm_abi_version": ([], i32),
            "rssm_status_string": ([i32], ctypes.c_char_p),
            "rssm_workspace_size": ([ctypes.POINTER(Config), ctypes.POINTER(sz)], i32),
            "rssm_layout_for": ([ctypes.POINTER(Config), ctypes.POINTER(Layout)], i32),
            "rssm_create": ([ctypes.POINTER(Config), p, sz, p, p, p, p, ctypes.POINTER(p)], i32),
            "rssm_get_layout": ([p, ctypes.POINTER(Layout)], i32),
            "rssm_decode_step": ([p, i32, ctypes.POINTER(Inputs), p, p], i32),
            "rssm_verify_rollback": ([p, p, p], i32),
            "rssm_flush": ([p, p], i32),
            "rssm_get_error": ([p, ctypes.POINTER(ctypes.c_int32), p], i32),
            "rssm_check_bounded_wait": ([ctypes.c_int64, p, p], i32),
            "rssm_quantize": ([i32, i64, i32, i32, p, p, p, p, p], i32),
            "rssm_state_bytes": ([p, ctypes.POINTER(sz)], i32),
            "rssm_export_state": ([p, p, sz, p], i32),
            "rssm_import_state": ([p, p, sz, p], i32),
            "rssm_sync_counts": ([p, p], i32),
            "rssm_count_summary": ([p, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32)], i32),
            "rssm_destroy": ([p], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != RSSM_OK:
        raise RssmError(fn, status)


def _addr(t) -> int | None:
    """Device address of a torch tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# --------------------------------------------------------------------------
# C ABI, same names
# --------------------------------------------------------------------------
def status_string(status: int) -> str:
    return load().rssm_status_string(status).decode()


def make_config(kind="mamba2", mode="replay", batch=1, heads=1, head_dim=64, state_dim=128,
                groups=1, k=16, max_draft=1, in_dtype="bf16", out_dtype=None, read_fmt="none",
                gdn_scale=1.0, ckpt_dtype="f32") -> Config:
    return Config(kind={"mamba2": RSSM_MAMBA2, "gdn": RSSM_GDN}[kind],
                  mode={"replay": RSSM_REPLAY, "conventional": RSSM_CONVENTIONAL}[mode],
                  batch=batch, heads=heads, head_dim=head_dim, state_dim=state_dim,
                  groups=groups, k=k, max_draft=max_draft, in_dtype=DTYPE[in_dtype],
                  out_dtype=0 if out_dtype is None else DTYPE[out_dtype],
                  read_fmt=READ_FMT[read_fmt], gdn_scale=gdn_scale,
                  ckpt_dtype=CKPT_DTYPE[ckpt_dtype])


def rssm_workspace_size(cfg: Config) -> int:
    n = ctypes.c_size_t(0)
    _check("rssm_workspace_size", load().rssm_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def rssm_layout_for(cfg: Config) -> Layout:
    lay = Layout()
    _check("rssm_layout_for", load().rssm_layout_for(ctypes.byref(cfg), ctypes.byref(lay)))
    return lay


def rssm_create(cfg: Config, workspace, workspace_bytes: int, A=None, D=None, state0=None,
                stream=None) -> int:
    h = ctypes.c_void_p(0)
    _check("rssm_create", load().rssm_create(ctypes.byref(cfg), _addr(workspace), workspace_bytes,
                                             _addr(A), _addr(D), _addr(state0), _stream(stream),
                                             ctypes.byref(h)))
    return h.value


def rssm_get_layout(handle: int) -> Layout:
    lay = Layout()
    _check("rssm_get_layout", load().rssm_get_layout(handle, ctypes.byref(lay)))
    return lay


def rssm_decode_step(handle: int, T: int, inputs: Inputs, y, stream=None) -> None:
    _check("rssm_decode_step", load().rssm_decode_step(handle, T, ctypes.byref(inputs), _addr(y),
                                                       _stream(stream)))


def rssm_verify_rollback(handle: int, accepted, stream=None) -> None:
    _check("rssm_verify_rollback",
           load().rssm_verify_rollback(handle, _addr(accepted), _stream(stream)))


def rssm_flush(handle: int, stream=None) -> None:
    _check("rssm_flush", load().rssm_flush(handle, _stream(stream)))


def rssm_get_error(handle: int, stream=None) -> tuple:
    err = (ctypes.c_int32 * 4)()
    _check("rssm_get_error", load().rssm_get_error(handle, err, _stream(stream)))
    return tuple(err)


def rssm_check_bounded_wait(limit_ns: int, err4, stream=None) -> None:
    """Run the device bounded-wait check; the timeout lands in err4 (device int32[4])."""
    _check("rssm_check_bounded_wait", load().rssm_check_bounded_wait(limit_ns, _addr(err4), _stream(stream)))


def rssm_quantize(fmt: int, tiles: int, rows: int, cols: int, src, codes, bscale, tscale,
                  stream=None) -> None:
    _check("rssm_quantize", load().rssm_quantize(fmt, tiles, rows, cols, _addr(src), _addr(codes),
                                                 _addr(bscale), _addr(tscale), _stream(stream)))


def rssm_state_bytes(handle: int) -> int:
    n = ctypes.c_size_t(0)
    _check("rssm_state_bytes", load().rssm_state_bytes(handle, ctypes.byref(n)))
    return n.value


def rssm_export_state(handle: int, dst, nbytes: int, stream=None) -> None:
    _check("rssm_export_state", load().rssm_export_state(handle, _addr(dst), nbytes, _stream(stream)))


def rssm_import_state(handle: int, src, nbytes: int, stream=None) -> None:
    _check("rssm_import_state", load().rssm_import_state(handle, _addr(src), nbytes, _stream(stream)))


def rssm_sync_counts(handle: int, stream=None) -> None:
    _check("rssm_sync_counts", load().rssm_sync_counts(handle, _stream(stream)))


def rssm_count_summary(handle: int) -> tuple:
    """(known, min_count, max_count) as the handle knows them on the host."""
    known, lo, hi = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    _check("rssm_count_summary", load().rssm_count_summary(handle, ctypes.byref(known), ctypes.byref(lo),
                                                           ctypes.byref(hi)))
    return known.value, lo.value, hi.value


def rssm_destroy(handle: int) -> None:
    _check("rssm_destroy", load().rssm_destroy(handle))


# --------------------------------------------------------------------------
# convenience: a layer owning its workspace tensor
# --------------------------------------------------------------------------
class Layer:
    """One SSM layer on a caller-owned (torch) workspace.

    Tensors are torch CUDA tensors in the layouts of include/rssm.h; inputs of
    one step are [B][T][...] (T = 1 may be omitted).
    """

    def __init__(self, cfg: Config, A=None, D=None, state0=None, device="cuda", stream=None):
        import torch
        self.cfg = cfg
        self.bytes = rssm_workspace_size(cfg)
        # 256-byte aligned by the caching allocator
        self.workspace = torch.empty(self.bytes, dtype=torch.uint8, device=device)
        self._keep = (A, D)
        self.handle = rssm_create(cfg, self.workspace, self.bytes, A, D, state0, stream)
        self.layout = rssm_get_layout(self.handle)

    def close(self):
        if self.handle:
            rssm_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- steps ----
    def decode_step(self, y, T=1, x=None, Bm=None, C=None, dt=None, q=None, k=None, v=None,
                    alpha=None, beta=None, stream=None):
        inp = Inputs(*[_addr(t) for t in (x, Bm, C, dt, q, k, v, alpha, beta)])
        rssm_decode_step(self.handle, T, inp, y, stream)

    def verify_rollback(self, accepted, stream=None):
        rssm_verify_rollback(self.handle, accepted, stream)

    def flush(self, stream=None):
        rssm_flush(self.handle, stream)

    def get_error(self, stream=None):
        return rssm_get_error(self.handle, stream)

    def sync_counts(self, stream=None):
        rssm_sync_counts(self.handle, stream)

    def count_summary(self):
        return rssm_count_summary(self.handle)

    def export_state(self, stream=None):
        """The state image (checkpoint, records, counts, read copy) in a new
        uint8 CUDA tensor."""
        import torch
        n = rssm_state_bytes(self.handle)
        img = torch.empty(n, dtype=torch.uint8, device=self.workspace.device)
        rssm_export_state(self.handle, img, n, stream)
        return img

    def import_state(self, image, stream=None):
        rssm_import_state(self.handle, image, image.numel() * image.element_size(), stream)

    # ---- views of the workspace (for tests and inspection) ----
    def region(self, name: str, dtype, shape):
        import torch
        off = getattr(self.layout, name)
        nbytes = getattr(self.layout, name + "_bytes")
        if nbytes == 0:
            return None
        return self.workspace[off:off + nbytes].view(dtype).view(*shape)

    def ckpt(self):
        """The checkpoint region as a tensor: float32, float16 for an FP16
        checkpoint, or the uint8 codes of a tile-format checkpoint ([..][N]
        FP8, [..][N/2] NVFP4; scales in ckpt_bscale / ckpt_tscale)."""
        import torch
        c = self.cfg
        shape = (c.batch, c.heads, c.head_dim, c.state_dim)
        if c.ckpt_dtype == RSSM_CKPT_FP8:
            return self.region("ckpt", torch.uint8, shape)
        if c.ckpt_dtype == RSSM_CKPT_NVFP4:
            return self.region("ckpt", torch.uint8, shape[:3] + (c.state_dim // 2,))
        dt = torch.float16 if c.ckpt_dtype == RSSM_F16 else torch.float32
        return self.region("ckpt", dt, shape)

    def counts(self):
        import torch
        return self.region("counts", torch.int32, (self.cfg.batch, self.cfg.heads))
