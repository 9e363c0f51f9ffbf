"""The C ABI without a GPU: the library loads, exports every function that
include/rssm.h declares, its structs match the Python mirror byte for byte,
and host-checkable errors come back as status codes (no CUDA call made)."""
import ctypes
import os
import re
import subprocess

import pytest

import hybrid_ssm_decode_gb300 as rssm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rssm.h")


@pytest.fixture(scope="module")
def lib():
    rssm.build()
    return rssm.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:rssm_status|int32_t|const char\s*\*)\s*(rssm_\w+)\s*\(",
                                 text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert lib.rssm_abi_version() == 5


def test_struct_layouts_match_header(tmp_path):
    """Compile a probe against include/rssm.h and compare sizes and offsets
    with the ctypes mirror used by the binding."""
    probe = tmp_path / "probe.c"
    fields = {
        "rssm_config": [f for f, _ in rssm.Config._fields_],
        "rssm_inputs": [f for f, _ in rssm.Inputs._fields_],
        "rssm_layout": [f for f, _ in rssm.Layout._fields_],
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "rssm.h"', "int main(void){"]
    for s, fs in fields.items():
        lines.append(f'printf("{s} size %zu\\n", sizeof({s}));')
        for f in fs:
            lines.append(f'printf("{s} {f} %zu\\n", offsetof({s}, {f}));')
    lines.append("return 0;}")
    probe.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(probe), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l}
    for s, cls in (("rssm_config", rssm.Config), ("rssm_inputs", rssm.Inputs), ("rssm_layout", rssm.Layout)):
        assert got[(s, "size")] == ctypes.sizeof(cls)
        for f, _ in cls._fields_:
            assert got[(s, f)] == getattr(cls, f).offset, (s, f)


def _cfg(**kw):
    base = dict(kind="mamba2", mode="replay", batch=256, heads=128, head_dim=64, state_dim=128,
                groups=8, k=16, max_draft=1, in_dtype="bf16")
    base.update(kw)
    return rssm.make_config(**base)


def _status(cfg):
    n = ctypes.c_size_t(0)
    return rssm.load().rssm_workspace_size(ctypes.byref(cfg), ctypes.byref(n))


def test_layout_regions(lib):
    cfg = _cfg()
    lay = rssm.rssm_layout_for(cfg)
    B, H, P, N, G, cap = 256, 128, 64, 128, 8, 16
    assert lay.capacity == cap
    assert lay.ckpt_bytes == B * H * P * N * 4
    assert lay.counts_bytes == B * H * 4
    assert lay.buf_x_bytes == B * H * cap * P * 2
    assert lay.buf_b_bytes == B * G * cap * N * 2
    assert lay.buf_dt_bytes == B * H * cap * 2
    regions = sorted((getattr(lay, r), getattr(lay, r + "_bytes")) for r in rssm._LAYOUT_REGIONS
                     if getattr(lay, r + "_bytes"))
    for (o1, s1), (o2, _) in zip(regions, regions[1:]):
        assert o1 % 256 == 0 and o1 + s1 <= o2
    assert regions[-1][0] + regions[-1][1] <= lay.total_bytes == rssm.rssm_workspace_size(cfg)
    # read copies and snapshots
    nv = rssm.rssm_layout_for(_cfg(read_fmt="nvfp4"))
    assert nv.rc_codes_bytes == B * H * P * N // 2 and nv.rc_bscale_bytes == B * H * P * N // 16
    fp8 = rssm.rssm_layout_for(_cfg(read_fmt="fp8"))
    assert fp8.rc_codes_bytes == B * H * P * N and fp8.rc_bscale_bytes == 0
    snap = rssm.rssm_layout_for(_cfg(mode="conventional", max_draft=4))
    assert snap.snap_bytes == 4 * B * H * P * N * 4 and snap.buf_x_bytes == 0
    gdn = rssm.rssm_layout_for(_cfg(kind="gdn", heads=32, head_dim=128, state_dim=128, groups=1))
    assert gdn.buf_u_bytes == B * 32 * cap * 128 * 4 and gdn.buf_k_bytes == B * 32 * cap * 128 * 2
    g8 = rssm.rssm_layout_for(_cfg(kind="gdn", heads=32, head_dim=128, state_dim=128, groups=1, read_fmt="nvfp4"))
    assert g8.rc_codes_bytes == B * 32 * 128 * 64 and g8.rc_bscale_bytes == B * 32 * 128 * 8
    assert g8.rc_tscale_bytes == B * 32 * 2 * 4                 # one scale per 64-row half
    assert g8.buf_v_bytes == B * 32 * cap * 128 * 2 and g8.buf_beta_bytes == B * 32 * cap * 4
    assert gdn.buf_v_bytes == 0 and gdn.buf_beta_bytes == 0 and lay.buf_v_bytes == 0
    c8 = rssm.rssm_layout_for(_cfg(ckpt_dtype="fp8", read_fmt="nvfp4"))
    assert c8.ckpt_bytes == B * H * P * N and c8.ckpt_tscale_bytes == B * H * 4 and c8.ckpt_bscale_bytes == 0
    assert c8.rc_codes_bytes == B * H * P * N // 2
    c4 = rssm.rssm_layout_for(_cfg(ckpt_dtype="nvfp4"))
    assert c4.ckpt_bytes == B * H * P * N // 2 and c4.ckpt_bscale_bytes == B * H * P * N // 16
    assert c4.rc_codes_bytes == 0 and lay.ckpt_tscale_bytes == 0
    f16 = rssm.rssm_layout_for(_cfg(ckpt_dtype="f16", read_fmt="fp8"))
    assert f16.ckpt_bytes == B * H * P * N * 2 and f16.rc_codes_bytes == B * H * P * N
    # the record-count summary: one entry per count 0..32 and one for out-of-range counts
    assert lay.cnt_hist_bytes == (32 + 2) * 4 and lay.cnt_hist % 256 == 0


def test_ckpt_dtype_must_be_f32_or_f16(lib):
    for v, status in ((0, rssm.RSSM_OK), (rssm.RSSM_F32, rssm.RSSM_OK), (rssm.RSSM_BF16, rssm.RSSM_ERR_INVALID_ARG),
                      (rssm.RSSM_CKPT_NVFP4, rssm.RSSM_OK), (7, rssm.RSSM_ERR_INVALID_ARG)):
        cfg = _cfg()
        cfg.ckpt_dtype = v
        assert _status(cfg) == status, v


@pytest.mark.parametrize("kw,status", [
    (dict(k=0), rssm.RSSM_ERR_INVALID_ARG),
    (dict(k=33), rssm.RSSM_ERR_INVALID_ARG),
    (dict(k=30, max_draft=4), rssm.RSSM_ERR_UNSUPPORTED),      # capacity 33 > 32
    (dict(k=32, max_draft=1), rssm.RSSM_OK),
    (dict(groups=3), rssm.RSSM_ERR_INVALID_ARG),
    (dict(head_dim=96), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(batch=0), rssm.RSSM_ERR_INVALID_ARG),
    (dict(max_draft=9), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(read_fmt="fp8", mode="conventional", max_draft=2), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(read_fmt="nvfp4", max_draft=4), rssm.RSSM_OK),      # Mamba-2 drafts read the copy
    (dict(read_fmt="fp8", max_draft=8, in_dtype="f32"), rssm.RSSM_OK),
    (dict(read_fmt="fp8", max_draft=4, ckpt_dtype="f16"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(kind="gdn", groups=1, mode="conventional", max_draft=4), rssm.RSSM_OK),      # GDN snapshot baseline
    (dict(kind="gdn", groups=1, read_fmt="fp8"), rssm.RSSM_OK),
    (dict(kind="gdn", groups=1, read_fmt="nvfp4", max_draft=4), rssm.RSSM_OK),   # GDN drafts read the copy
    (dict(kind="gdn", groups=1, read_fmt="fp8", max_draft=4, mode="conventional"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(kind="gdn", groups=1, read_fmt="fp8", mode="conventional"), rssm.RSSM_OK),   # quantised recurrence
    (dict(kind="gdn", groups=1, read_fmt="nvfp4", mode="conventional", in_dtype="f32"), rssm.RSSM_OK),
    (dict(kind="gdn", groups=1, read_fmt="fp8", in_dtype="f32"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="f16"), rssm.RSSM_OK),
    (dict(ckpt_dtype="f16", read_fmt="nvfp4"), rssm.RSSM_OK),
    (dict(ckpt_dtype="f16", max_draft=4), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="f16", mode="conventional"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="f16", in_dtype="f32"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="f16", kind="gdn", groups=1), rssm.RSSM_OK),
    (dict(ckpt_dtype="f16", kind="gdn", groups=1, read_fmt="nvfp4"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="fp8", kind="gdn", groups=1), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="fp8"), rssm.RSSM_OK),
    (dict(ckpt_dtype="fp8", read_fmt="nvfp4"), rssm.RSSM_OK),
    (dict(ckpt_dtype="fp8", read_fmt="fp8"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="nvfp4"), rssm.RSSM_OK),
    (dict(ckpt_dtype="nvfp4", read_fmt="fp8"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="nvfp4", mode="conventional"), rssm.RSSM_ERR_UNSUPPORTED),
    (dict(ckpt_dtype="fp8", max_draft=2), rssm.RSSM_ERR_UNSUPPORTED),
])
def test_config_validation(lib, kw, status):
    assert _status(_cfg(**kw)) == status


def test_host_checked_errors_make_no_cuda_call(lib):
    cfg = _cfg(batch=2, heads=8, groups=1)
    need = rssm.rssm_workspace_size(cfg)
    h = ctypes.c_void_p(0)
    create = lib.rssm_create
    # null workspace, misaligned workspace, too small
    assert create(ctypes.byref(cfg), None, need, 16, 16, None, None, ctypes.byref(h)) == rssm.RSSM_ERR_INVALID_ARG
    assert create(ctypes.byref(cfg), 4096 + 16, need, 16, 16, None, None, ctypes.byref(h)) == rssm.RSSM_ERR_INVALID_ARG
    assert create(ctypes.byref(cfg), 4096, need - 1, 16, 16, None, None, ctypes.byref(h)) == rssm.RSSM_ERR_CAPACITY
    # Mamba-2 needs A and D
    assert create(ctypes.byref(cfg), 4096, need, None, 16, None, None, ctypes.byref(h)) == rssm.RSSM_ERR_INVALID_ARG
    assert h.value is None
    # null handles
    inp = rssm.Inputs()
    assert lib.rssm_decode_step(None, 1, ctypes.byref(inp), 4096, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_verify_rollback(None, 4096, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_flush(None, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_destroy(None) == rssm.RSSM_ERR_INVALID_ARG
    err = (ctypes.c_int32 * 4)()
    assert lib.rssm_get_error(None, err, None) == rssm.RSSM_ERR_INVALID_ARG
    # state image and count summary need a handle
    n = ctypes.c_size_t(0)
    i32 = ctypes.c_int32
    known, lo, hi = i32(0), i32(0), i32(0)
    assert lib.rssm_state_bytes(None, ctypes.byref(n)) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_export_state(None, 4096, 1 << 20, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_import_state(None, 4096, 1 << 20, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_sync_counts(None, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_count_summary(None, ctypes.byref(known), ctypes.byref(lo),
                                  ctypes.byref(hi)) == rssm.RSSM_ERR_INVALID_ARG
    # quantiser argument checks
    assert lib.rssm_quantize(3, 1, 64, 128, 4096, 4096, 4096, 4096, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_quantize(1, 1, 96, 128, 4096, 4096, 4096, 4096, None) == rssm.RSSM_ERR_UNSUPPORTED
    assert lib.rssm_quantize(2, 1, 64, 128, 4096, 4096, None, 4096, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_quantize(1, 0, 64, 128, None, None, None, None, None) == rssm.RSSM_OK
    # bounded-wait check: argument checks come before any device work
    assert lib.rssm_check_bounded_wait(1000, None, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_check_bounded_wait(0, 4096, None) == rssm.RSSM_ERR_INVALID_ARG
    assert lib.rssm_check_bounded_wait(2_000_000_000, 4096, None) == rssm.RSSM_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(6):
        assert rssm.status_string(s)
    assert rssm.status_string(99) == "unknown status"


def test_load_refuses_missing_library(monkeypatch, tmp_path):
    monkeypatch.setattr(rssm, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(rssm, "_lib", None)
    with pytest.raises(ImportError):
        rssm.load()
