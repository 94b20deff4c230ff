"""The C-ABI library loads here (no GPU) and exports every declared symbol;
host-side helpers and argument checks answer without touching a device."""

import os
import re

import pytest

from combine_moe_layout_02_gb300 import build as moe_build
from combine_moe_layout_02_gb300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.lib()


def _declared(profile=False):
    """Entry points declared in include/*.h; those under #ifdef MOE_PROFILE
    only when profile is set."""
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            if not profile:
                text = re.sub(r"#ifdef MOE_PROFILE.*?#endif", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"moe_layout", "moe_notify", "moe_dispatch", "moe_combine"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(moe.EXPORTS) >= names


def test_profile_entry_point_only_in_the_profile_build(lib):
    """The default library carries no profile symbol; the -DMOE_PROFILE build
    exports moe_profile_attach next to every other entry point."""
    import ctypes

    assert not hasattr(lib, "moe_profile_attach")
    assert "moe_profile_attach" in _declared(profile=True) - _declared()
    prof = ctypes.CDLL(moe_build.build(variant="profile"))
    for n in _declared(profile=True):
        assert hasattr(prof, n), n


def test_slot_stride_and_limits(lib):
    assert moe.moe_slot_stride(7168, 0) == 14848
    assert moe.moe_slot_stride(7168, 1) == 7680
    assert moe.moe_slot_stride(256, 0) == 1024
    assert moe.moe_slot_stride(0, 0) == -1
    ok = moe.make_shape(8, 256, 32768, 8, 7168)
    assert moe.moe_check_shape(ok) == moe.MOE_OK
    assert moe.moe_max_recv_rows(ok) == 32768 * 8
    assert moe.moe_scratch_bytes(ok) >= 8 * 16 * 8 * 4
    assert moe.moe_check_shape(moe.make_shape(8, 250, 32768, 8, 7168)) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_shape(moe.make_shape(8, 256, 32767, 8, 7168)) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_shape(moe.make_shape(8, 256, 32768, 17, 7168)) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_shape(moe.make_shape(8, 256, 32768, 8, 7164)) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_shape(moe.make_shape(8, 256, 32768, 8, 7176, quant=1)) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_shape(moe.make_shape(2048, 4096, 2048, 8, 64)) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_shape(moe.make_shape(8, 256, 0, 8, 7168)) == moe.MOE_OK
    # row counts are int32: S*K + E*(alignment-1) must fit
    assert moe.moe_check_shape(moe.make_shape(8, 256, 32768, 8, 7168, expert_alignment=8_000_000)) == moe.MOE_OK
    assert moe.moe_check_shape(moe.make_shape(8, 256, 32768, 8, 7168,
                                              expert_alignment=8_388_608)) == moe.MOE_ERR_UNSUPPORTED


def test_null_pointers_rejected_before_any_launch(lib):
    s = moe.make_shape(4, 16, 256, 2, 256)
    assert lib.moe_layout(s, None, None, None, None, None, None, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_notify(s, *([None] * 12), 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(s, None, None, None, None, None, None, 0, None, None, None, None,
                            None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(s, None, 512, None, 0, None, None, None, None, None,
                           None) == moe.MOE_ERR_INVALID_ARG
    # Misaligned (non-NULL) pointers are rejected on the host as well.
    assert lib.moe_combine(s, 8, 512, 16, 1, 16, 16, None, 16, None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.status_string(moe.MOE_ERR_CAPACITY) == "MOE_ERR_CAPACITY"


def test_static_scratch_size_guard_runs_on_the_host(lib):
    """moe_layout_static_scratch's built-in buffer holds one flag per source rank
    of the largest accepted shape; larger shapes are refused before any device
    is touched (the fake pointers below are never dereferenced)."""
    assert moe.MOE_LAYOUT_STATIC_SCRATCH_BYTES == 4 * 1024  # MOE_MAX_RANKS int32 flags
    too_big = moe.make_shape(2048, 4096, 2048 * 64, 8, 64)
    fake = 1 << 20
    assert lib.moe_layout_static_scratch(too_big, fake, fake, fake, fake, fake, fake,
                                         None) == moe.MOE_ERR_UNSUPPORTED
    ok = moe.make_shape(1024, 4096, 1024 * 64, 8, 64)
    assert lib.moe_layout_static_scratch(ok, None, fake, fake, fake, None, None,
                                         None) == moe.MOE_ERR_INVALID_ARG


def test_run_host_checks_arguments_on_the_host(lib):
    """moe_run_host validates everything before it touches a device (the fake
    device pointers below are never dereferenced)."""
    import ctypes

    s = moe.make_shape(4, 16, 64, 2, 64)
    n = 2
    arr = (ctypes.c_void_p * n)(*([1 << 20] * n))
    need = moe.moe_run_host_workspace_bytes(s, n)
    assert need > 0 and moe.moe_run_host_workspace_bytes(s, -1) == -1
    ws = 1 << 24
    args = lambda **k: dict(dict(x=arr, i=arr, w=None, o=arr, y=None, ys=0, fl=0, wsp=ws, wsb=need), **k)

    def call(shape=s, nb=n, **k):
        a = args(**k)
        return lib.moe_run_host(shape, nb, a["x"], a["i"], a["w"], a["o"], a["y"], a["ys"], a["fl"],
                                a["wsp"], a["wsb"], None)

    assert call(nb=0) == moe.MOE_OK                       # nothing to run
    assert call(nb=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(fl=4) == moe.MOE_ERR_INVALID_ARG          # unknown flag
    assert call(fl=moe.MOE_RUN_FUSED | moe.MOE_RUN_EXPERT) == moe.MOE_ERR_INVALID_ARG  # fused is rank-major
    assert call(wsb=need - 1) == moe.MOE_ERR_INVALID_ARG  # workspace too small
    assert call(wsp=ws + 16) == moe.MOE_ERR_INVALID_ARG   # workspace not 256-byte aligned
    assert call(x=None) == moe.MOE_ERR_INVALID_ARG
    q = moe.make_shape(4, 16, 64, 2, 64, quant=1)
    need_q = moe.moe_run_host_workspace_bytes(q, n)
    assert call(shape=q, wsb=need_q) == moe.MOE_ERR_INVALID_ARG  # int8 slots need expert outputs y
    assert call(shape=q, wsb=need_q, y=1 << 20, ys=64) == moe.MOE_ERR_INVALID_ARG       # y rows shorter than 2H
    assert call(shape=q, wsb=need_q, y=1 << 20, ys=136) == moe.MOE_ERR_INVALID_ARG      # stride not a multiple of 16
    assert call(shape=q, wsb=need_q, y=(1 << 20) + 8, ys=128) == moe.MOE_ERR_INVALID_ARG  # y not 16-byte aligned
    holes = (ctypes.c_void_p * n)(1 << 20, None)
    assert call(o=holes) == moe.MOE_ERR_INVALID_ARG      # a batch without an output buffer
