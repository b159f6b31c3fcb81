"""Host-side checks of the C ABI that need no GPU.

The library is compiled for sm_103a with the CUDA runtime linked statically, so
it loads on a machine without a GPU.  These tests check that it exports every
function include/*.h declares, and that argument validation rejects
bad calls before any CUDA call is made (so they run here, on the CPU).
"""
from __future__ import annotations

import glob
import os
import re
import subprocess

import pytest

import prompt_lookup_speculative_gb300 as pkg
from prompt_lookup_speculative_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return pkg.load_library()


def declared_functions() -> set[str]:
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(lookup_\w*)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("lookup_draft", "lookup_draft_ex", "lookup_draft_scan", "lookup_draft_fill",
                 "lookup_draft_host", "lookup_draft_workspace_bytes", "lookup_draft_strerror",
                 "lookup_draft_last_cuda_error", "lookup_draft_set_wait_limit_ns", "lookup_draft_noalloc",
                 "lookup_fuse", "lookup_schedule", "lookup_verify", "lookup_append", "lookup_index_slots_for",
                 "lookup_index_bytes", "lookup_index_build", "lookup_index_append", "lookup_index_draft",
                 "lookup_ctx_slots_for", "lookup_ctx_bytes", "lookup_ctx_build", "lookup_ctx_append",
                 "lookup_ctx_draft", "lookup_draft_read_floor", "lookup_draft_read_floor_bulk"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in sorted(declared_functions()):
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_exported_symbols_are_c_linkage(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_build.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for name in declared_functions():
        assert name in exported, f"{name} is not an unmangled dynamic symbol"


def test_built_for_sm103a():
    cmd = lib_build.compile_command("x.so")
    assert "arch=compute_103a,code=sm_103a" in cmd


def test_strerror(lib):
    assert lib.lookup_draft_strerror(0) == b"ok"
    assert lib.lookup_draft_strerror(-1) == b"invalid argument"
    assert lib.lookup_draft_strerror(-2) == b"CUDA error"
    assert lib.lookup_draft_strerror(12345)


FAKE = 0x10000        # a non-null, aligned address; never dereferenced by the host checks


@pytest.mark.parametrize("B,min_m,max_m,K", [
    (-1, 4, 12, 15),        # negative batch
    (4, 0, 12, 15),         # min_m < 1
    (4, 5, 4, 15),          # min_m > max_m
    (4, 4, 33, 15),         # max_m above LOOKUP_DRAFT_MAX_M
    (4, 4, 12, -1),         # K < 0
    (4, 4, 12, 65),         # K above LOOKUP_DRAFT_MAX_K
])
def test_rejects_bad_parameters(lib, B, min_m, max_m, K):
    rc = lib.lookup_draft(FAKE, FAKE, B, min_m, max_m, K, FAKE, FAKE, FAKE, None)
    assert rc == -1


def test_rejects_null_and_misaligned_pointers(lib):
    assert lib.lookup_draft(None, FAKE, 4, 4, 12, 15, FAKE, FAKE, FAKE, None) == -1
    assert lib.lookup_draft(FAKE, None, 4, 4, 12, 15, FAKE, FAKE, FAKE, None) == -1
    assert lib.lookup_draft(FAKE, FAKE, 4, 4, 12, 15, None, FAKE, FAKE, None) == -1
    assert lib.lookup_draft(FAKE, FAKE, 4, 4, 12, 15, FAKE, None, FAKE, None) == -1
    assert lib.lookup_draft(FAKE, FAKE, 4, 4, 12, 15, FAKE, FAKE, None, None) == -1
    assert lib.lookup_draft(FAKE + 2, FAKE, 4, 4, 12, 15, FAKE, FAKE, FAKE, None) == -1
    assert lib.lookup_draft(FAKE, FAKE + 4, 4, 4, 12, 15, FAKE, FAKE, FAKE, None) == -1
    assert lib.lookup_draft_scan(FAKE, FAKE, 4, 4, 12, None, 1 << 20, None) == -1
    assert lib.lookup_draft_scan(FAKE, FAKE, 4, 4, 12, FAKE + 4, 1 << 20, None) == -1
    assert lib.lookup_draft_fill(FAKE, FAKE, 4, 4, 12, 15, None, 1 << 20, FAKE, FAKE, FAKE, None, None) == -1


def test_bulk_read_floor_checks_its_arguments(lib):
    assert lib.lookup_draft_read_floor_bulk(FAKE, 1 << 20, None, None) == -1          # no output word
    assert lib.lookup_draft_read_floor_bulk(FAKE, 1 << 20, FAKE + 2, None) == -1      # misaligned word
    assert lib.lookup_draft_read_floor_bulk(None, 1 << 20, FAKE, None) == -1          # no data
    assert lib.lookup_draft_read_floor_bulk(FAKE + 4, 1 << 20, FAKE, None) == -1      # data not 16-byte aligned
    assert lib.lookup_draft_read_floor_bulk(FAKE, (1 << 20) + 4, FAKE, None) == -1    # size not a multiple of 16
    assert lib.lookup_draft_read_floor_bulk(None, 0, FAKE, None) == 0                 # nothing to read


def test_read_floor_checks_its_arguments(lib):
    assert lib.lookup_draft_read_floor(FAKE, 1 << 20, 4, 256, None, None) == -1
    assert lib.lookup_draft_read_floor(FAKE, 1 << 20, 4, 256, FAKE + 2, None) == -1
    assert lib.lookup_draft_read_floor(None, 1 << 20, 4, 256, FAKE, None) == -1
    assert lib.lookup_draft_read_floor(FAKE + 4, 1 << 20, 4, 256, FAKE, None) == -1
    assert lib.lookup_draft_read_floor(FAKE, (1 << 20) + 4, 4, 256, FAKE, None) == -1
    assert lib.lookup_draft_read_floor(FAKE, 1 << 20, 0, 256, FAKE, None) == -1
    assert lib.lookup_draft_read_floor(FAKE, 1 << 20, 33, 256, FAKE, None) == -1
    assert lib.lookup_draft_read_floor(FAKE, 1 << 20, 4, 100, FAKE, None) == -1
    assert lib.lookup_draft_read_floor(FAKE, 1 << 20, 4, 2048, FAKE, None) == -1
    assert lib.lookup_draft_read_floor(None, 0, 4, 256, FAKE, None) == 0     # nothing to read


def test_empty_batch_is_a_no_op(lib):
    # B == 0 enqueues nothing and needs no valid pointer or device.
    assert lib.lookup_draft(None, None, 0, 4, 12, 15, None, None, None, None) == 0
    assert lib.lookup_draft_ex(None, None, 0, 4, 12, 15, None, None, None, None, None) == 0
    assert lib.lookup_draft_host(None, None, 0, 4, 12, 15, None, None, None, None) == 0


def test_host_entry_checks_host_offsets(lib):
    import numpy as np
    tok = np.zeros(16, np.int32)
    out_d, out_l, out_p = np.zeros(8, np.int32), np.zeros(2, np.int32), np.zeros(2, np.int32)
    for bad in ([0, 5, 3], [-1, 4, 8], [0, 4, 4 + (1 << 31)]):
        off = np.array(bad, np.int64)
        rc = lib.lookup_draft_host(tok.ctypes.data, off.ctypes.data, 2, 4, 12, 4,
                                   out_d.ctypes.data, out_l.ctypes.data, out_p.ctypes.data, None)
        assert rc == -1, bad


def test_package_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError):
        pkg.load_library(str(tmp_path / "missing.so"))


def test_loop_steps_reject_bad_parameters(lib):
    F = FAKE
    # fuse: K < H + T, H < 1, agree_n > H, H + T above the limit, a null output
    assert lib.lookup_fuse(F, F, F, None, 4, 14, 7, 8, 8, 6, 2, 4, F, F, F, None) == -1
    assert lib.lookup_fuse(F, F, F, None, 4, 15, 0, 8, 8, 6, 0, 4, F, F, F, None) == -1
    assert lib.lookup_fuse(F, F, F, None, 4, 15, 7, 8, 8, 6, 8, 4, F, F, F, None) == -1
    assert lib.lookup_fuse(F, F, F, None, 4, 1 << 20, 1 << 16, 8, 8, 6, 2, 4, F, F, F, None) == -1
    assert lib.lookup_fuse(F, F, F, None, 4, 15, 7, 8, 8, 6, 2, 4, F, None, F, None) == -1
    # schedule: enter_steps < 1, sticky < 0, null state
    assert lib.lookup_schedule(F, F, 4, 7, 8, 4, 1, 0, 3, F, F, None) == -1
    assert lib.lookup_schedule(F, F, 4, 7, 8, 4, 1, 2, -1, F, F, None) == -1
    assert lib.lookup_schedule(F, F, 4, 7, 8, 4, 1, 2, 3, None, F, None) == -1
    # verify: negative P, P above the limit, probs without u
    assert lib.lookup_verify(F, F, F, None, None, None, None, 4, -1, F, F, F, None) == -1
    assert lib.lookup_verify(F, F, F, None, None, None, None, 4, 1 << 17, F, F, F, None) == -1
    assert lib.lookup_verify(F, F, F, F, None, None, None, 4, 15, F, F, F, None) == -1
    # append: negative W, null offsets
    assert lib.lookup_append(F, F, F, F, 4, -1, F, F, None) == -1
    assert lib.lookup_append(F, None, F, F, 4, 16, F, F, None) == -1


def test_loop_steps_empty_batch(lib):
    # B == 0: fuse, schedule and verify enqueue nothing and need no pointer.
    assert lib.lookup_fuse(None, None, None, None, 0, 15, 7, 8, 8, 6, 2, 4, None, None, None, None) == 0
    assert lib.lookup_schedule(None, None, 0, 7, 8, 4, 1, 2, 3, None, None, None) == 0
    assert lib.lookup_verify(None, None, None, None, None, None, None, 0, 15, None, None, None, None) == 0


def test_index_sizes(lib):
    # 2 * (12 - 4 + 1) * 1000 = 18000 -> 32768 slots; 128 + 8 * slots bytes
    assert lib.lookup_index_slots_for(1000, 4, 12) == 32768
    assert lib.lookup_index_slots_for(0, 4, 12) == 16
    assert lib.lookup_index_slots_for(1000, 5, 4) == 0
    assert lib.lookup_index_slots_for(1000, 4, 33) == 0
    assert lib.lookup_index_bytes(32768) == 128 + 8 * 32768
    assert lib.lookup_index_bytes(1000) == 0 and lib.lookup_index_bytes(8) == 0


def test_index_rejects_bad_parameters(lib):
    F = FAKE
    # build: min_m > max_m, hash_bits 0, slots not a power of two, misaligned index
    assert lib.lookup_index_build(F, F, F, 4, 5, 4, F, 1024, 64, None) == -1
    assert lib.lookup_index_build(F, F, F, 4, 4, 12, F, 1024, 0, None) == -1
    assert lib.lookup_index_build(F, F, F, 4, 4, 12, F, 1000, 64, None) == -1
    assert lib.lookup_index_build(F, F, F, 4, 4, 12, F + 8, 1024, 64, None) == -1
    # append: negative W, null cap
    assert lib.lookup_index_append(F, F, F, F, F, F, 4, -1, 4, 12, F, 1024, 64, None, None) == -1
    assert lib.lookup_index_append(F, F, F, None, F, F, 4, 16, 4, 12, F, 1024, 64, None, None) == -1
    # draft: K above the limit, null index
    assert lib.lookup_index_draft(F, F, F, 4, 4, 12, 65, F, 1024, 64, F, F, F, None, None, None) == -1
    assert lib.lookup_index_draft(F, F, F, 4, 4, 12, 15, None, 1024, 64, F, F, F, None, None, None) == -1
    # B == 0: append and draft enqueue nothing
    assert lib.lookup_index_append(None, None, None, None, None, None, 0, 16, 4, 12, None, 1024, 64, None, None) == 0
    assert lib.lookup_index_draft(None, None, None, 0, 4, 12, 15, None, 1024, 64, None, None, None, None, None,
                                  None) == 0


def test_ctx_sizes_and_argument_checks(lib):
    import numpy as np
    assert lib.lookup_ctx_slots_for(1000, 1, 4) == 16384          # 4 * 4 * 1000 = 16000 -> 16384
    assert lib.lookup_ctx_slots_for(1000, 0, 4) == 0 and lib.lookup_ctx_slots_for(1000, 1, 5) == 0
    assert lib.lookup_ctx_bytes(16384) == 128 + 32 * 16384 and lib.lookup_ctx_bytes(100) == 0
    F = FAKE
    mc = np.ones(4, np.int32)
    num = np.ones(4, np.int32)
    den = np.full(4, 2, np.int32)
    bad_den = np.zeros(4, np.int32)
    args = (mc.ctypes.data, num.ctypes.data)
    assert lib.lookup_ctx_build(F, F, F, 4, 2, 1, F, 1024, None) == -1                 # n_min > n_max
    assert lib.lookup_ctx_build(F, F, F, 70000, 1, 4, F, 1024, None) == -1             # B above 65536
    assert lib.lookup_ctx_draft(F, F, F, 4, 1, 4, 8, *args, bad_den.ctypes.data, F, 1024, F, F, None) == -1
    assert lib.lookup_ctx_draft(F, F, F, 4, 1, 4, 65, *args, den.ctypes.data, F, 1024, F, F, None) == -1
    assert lib.lookup_ctx_draft(None, None, None, 0, 1, 4, 8, *args, den.ctypes.data, None, 1024, None, None,
                                None) == 0
    assert lib.lookup_ctx_append(F, F, F, F, F, F, 4, -1, 1, 4, F, 1024, None, None) == -1


# ------------------------------------------------------------ checked build ----
def declared_in(header: str) -> set[str]:
    text = open(os.path.join(ROOT, "include", header), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return {m.group(1) for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(lookup_\w*)\s*\(", text, flags=re.M)}


@pytest.fixture(scope="module")
def checked_lib():
    lib_build.build()
    return pkg.load_checked_library()


def test_checked_library_exports_the_drafting_entry_points(checked_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_build.CHECKED_LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    names = declared_in("lookup_draft.h")
    assert {"lookup_draft", "lookup_draft_check_word", "lookup_draft_checked_build"} <= names
    for name in names:
        assert name in exported, f"{name} missing from the checked library"


def test_checked_build_flag_and_word_without_a_gpu(lib, checked_lib):
    import ctypes
    assert lib.lookup_draft_checked_build() == 0
    assert checked_lib.lookup_draft_checked_build() == 1
    out = ctypes.c_uint32(99)
    assert lib.lookup_draft_check_word(ctypes.byref(out), 1) == 0 and out.value == 0   # no device call
    assert lib.lookup_draft_check_word(None, 0) == -1
    assert checked_lib.lookup_draft_check_word(None, 0) == -1
    # the checked library validates its arguments like the regular one
    assert checked_lib.lookup_draft(FAKE, FAKE, 4, 5, 4, 15, FAKE, FAKE, FAKE, None) == -1
    assert checked_lib.lookup_draft(None, None, 0, 4, 12, 15, None, None, None, None) == 0


def test_checked_build_command():
    cmd = lib_build.compile_command("x.so", checked=True)
    assert "-DLOOKUP_DRAFT_CHECKED=1" in cmd and "arch=compute_103a,code=sm_103a" in cmd
    assert "-DLOOKUP_DRAFT_CHECKED=1" not in lib_build.compile_command("x.so")


def test_plan_rejects_bad_parameters(lib):
    F = FAKE
    # K < H + T, agree_n > H, enter_steps < 1, sticky < 0, slack < 0, a null state or output
    assert lib.lookup_plan(F, F, F, F, 4, 14, 7, 8, 8, 6, 2, 4, 1, 2, 3, F, F, F, F, F, None) == -1
    assert lib.lookup_plan(F, F, F, F, 4, 15, 7, 8, 8, 6, 8, 4, 1, 2, 3, F, F, F, F, F, None) == -1
    assert lib.lookup_plan(F, F, F, F, 4, 15, 7, 8, 8, 6, 2, 4, 1, 0, 3, F, F, F, F, F, None) == -1
    assert lib.lookup_plan(F, F, F, F, 4, 15, 7, 8, 8, 6, 2, 4, 1, 2, -1, F, F, F, F, F, None) == -1
    assert lib.lookup_plan(F, F, F, F, 4, 15, 7, 8, 8, 6, 2, 4, -1, 2, 3, F, F, F, F, F, None) == -1
    assert lib.lookup_plan(F, F, F, F, 4, 15, 7, 8, 8, 6, 2, 4, 1, 2, 3, None, F, F, F, F, None) == -1
    assert lib.lookup_plan(F, F, F, F, 4, 15, 7, 8, 8, 6, 2, 4, 1, 2, 3, F, F, F, F, None, None) == -1
    # B == 0 enqueues nothing
    assert lib.lookup_plan(None, None, None, None, 0, 15, 7, 8, 8, 6, 2, 4, 1, 2, 3, None, None, None, None, None,
                           None) == 0


def test_draft_plan_rejects_bad_parameters(lib):
    F = FAKE
    ok = [F, F, 4, 4, 12, F, F, 7, 8, 8, 6, 2, 4, 1, 2, 3, F, F, F, F, F, None, None, None]
    assert len(ok) == 24

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.lookup_draft_plan(*a)

    assert call(a7=0) == -1                 # H < 1
    assert call(a8=-1) == -1                # T < 0
    assert call(a7=40, a8=25) == -1         # H + T above LOOKUP_DRAFT_MAX_K
    assert call(a11=8) == -1                # agree_n > H
    assert call(a14=0) == -1                # enter_steps < 1
    assert call(a15=-1) == -1               # sticky < 0
    assert call(a13=-1) == -1               # slack < 0
    assert call(a3=5, a4=4) == -1           # min_m > max_m
    assert call(a5=None) == -1              # no model draft
    assert call(a16=None) == -1             # no state
    assert call(a16=F + 2) == -1            # misaligned state
    assert call(a0=F + 2) == -1             # misaligned tokens
    assert lib.lookup_draft_plan(None, None, 0, 4, 12, None, None, 7, 8, 8, 6, 2, 4, 1, 2, 3, None, None, None, None,
                                 None, None, None, None) == 0


def _gpu_present() -> bool:
    try:
        import torch
        return bool(torch.cuda.is_available())
    except Exception:  # pragma: no cover
        return False


@pytest.mark.skipif(_gpu_present(), reason="with a GPU the fake pointers would be launched on")
def test_cuda_failure_is_reported_without_a_gpu(lib):
    """With no usable device the first CUDA call of a valid-looking step fails: the
    entry point returns LOOKUP_DRAFT_ECUDA and lookup_draft_last_cuda_error names
    the call and the CUDA error."""
    rc = lib.lookup_draft(FAKE, FAKE, 4, 4, 12, 15, FAKE, FAKE, FAKE, None)
    assert rc == -2
    msg = lib.lookup_draft_last_cuda_error().decode()
    assert msg and "cuda" in msg.lower()
    assert lib.lookup_draft_strerror(rc) == b"CUDA error"
    assert lib.lookup_draft_noalloc(FAKE, FAKE, 4, 4, 12, 15, FAKE, FAKE, FAKE, None) == -2


def test_launch_counter_needs_no_gpu_and_counts_no_failed_call(lib):
    """lookup_draft_launch_count answers without a device; calls refused on their
    arguments or failing on CUDA enqueue nothing and leave it unchanged."""
    n0 = lib.lookup_draft_launch_count()
    assert lib.lookup_draft(FAKE, FAKE, 4, 4, 12, 15, FAKE, FAKE, FAKE, None) == -2
    assert lib.lookup_draft(FAKE, FAKE, 4, 4, 3, 15, FAKE, FAKE, FAKE, None) == -1
    assert lib.lookup_draft_plan(FAKE, FAKE, 4, 4, 12, FAKE, FAKE, 7, 8, 8, 6, 2, 4, 1, 2, 3, FAKE, FAKE, FAKE, FAKE,
                                 FAKE, FAKE, None, None) != 0
    assert lib.lookup_draft_launch_count() == n0
    assert pkg.launch_count(lib) == n0


def test_policy_rejects_bad_parameters(lib):
    F = FAKE
    ok = [F, F, 4, 7, 3, 1.0, 1.0, 1.0, 0.125, 0.05, 6, 8, 12, F, F, F, None]

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.lookup_policy(*a)

    assert call(a2=-1) == -1                # B < 0
    assert call(a3=-1) == -1                # n_lookup < 0
    assert call(a6=0.0) == -1               # t_model not positive
    assert call(a7=-1.0) == -1              # t_plain negative
    assert call(a8=1.5) == -1               # alpha above 1
    assert call(a9=-0.1) == -1              # negative margin
    assert call(a10=9) == -1                # edges decreasing
    assert call(a13=None) == -1             # no acceptance state
    assert lib.lookup_policy(None, None, 0, 7, 3, 1.0, 1.0, 1.0, 0.125, 0.05, 6, 8, 12, None, None, None, None) == 0


def test_binding_declares_argument_types_of_every_entry_point(lib, checked_lib):
    """ctypes passes undeclared integer arguments as C ints: a 64-bit device
    pointer would be cut to 32 bits.  Every function the headers declare has its
    argument types set in the binding, for both builds."""
    for name in sorted(declared_functions()):
        assert getattr(lib, name).argtypes is not None, f"{name}: argument types not declared"
    for name in sorted(declared_in("lookup_draft.h") | {"lookup_draft_plan"}):
        assert getattr(checked_lib, name).argtypes is not None, f"checked {name}: argument types not declared"
    with pytest.raises(AttributeError):
        checked_lib.lookup_policy                       # not in the checked build at all


def test_index_draft_plan_rejects_bad_parameters(lib):
    F = FAKE
    ok = [F, F, F, 4, 4, 12, F, 1024, 64, F, F, 7, 8, 8, 6, 2, 4, 1, 2, 3, F, F, F, F, F, None, None, None, None]
    assert len(ok) == 29

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.lookup_index_draft_plan(*a)

    assert call(a11=0) == -1                # H < 1
    assert call(a11=40, a12=25) == -1       # H + T above LOOKUP_DRAFT_MAX_K
    assert call(a15=8) == -1                # agree_n > H
    assert call(a18=0) == -1                # enter_steps < 1
    assert call(a7=1000) == -1              # slots not a power of two
    assert call(a20=None) == -1             # no state
    assert call(a6=F + 8) == -1             # misaligned index
    assert lib.lookup_index_draft_plan(None, None, None, 0, 4, 12, None, 1024, 64, None, None, 7, 8, 8, 6, 2, 4, 1, 2,
                                       3, None, None, None, None, None, None, None, None, None) == 0


def test_index_verify_append_rejects_bad_parameters(lib):
    F = FAKE
    # block, block_len, target, probs, qprobs, point_mass, u, B, P, tokens, base, len, cap, min_m, max_m, index,
    # slots, hash_bits, out_accepted, out_commit, out_ncommit, out_status, stream
    ok = [F, F, F, None, None, None, None, 4, 15, F, F, F, F, 4, 12, F, 1024, 64, F, F, F, None, None]
    assert len(ok) == 23

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.lookup_index_verify_append(*a)

    assert call(a8=-1) == -1                # P < 0
    assert call(a8=(1 << 16) + 1) == -1     # P above the verify block limit
    assert call(a3=F) == -1                 # probs without u
    assert call(a0=None) == -1              # no block with P > 0
    assert call(a19=None) == -1             # no commit output
    assert call(a12=None) == -1             # no cap
    assert call(a16=1000) == -1             # slots not a power of two
    assert call(a14=3) == -1                # max_m < min_m
    assert call(a15=F + 8) == -1            # misaligned index
    assert call(a7=-1) == -1                # B < 0
    assert call(a7=0, a0=None, a1=None, a2=None, a9=None, a15=None) == 0   # B == 0: nothing to do


def test_index_verify_append_draft_rejects_bad_parameters(lib):
    F = FAKE
    # block, block_len, target, probs, qprobs, point_mass, u, B, P, tokens, base, len, cap, min_m, max_m, index,
    # slots, hash_bits, K, out_accepted, out_commit, out_ncommit, out_status, out_draft, out_draft_len, out_pos,
    # out_mlen, out_fallback, stream
    ok = [F, F, F, None, None, None, None, 4, 15, F, F, F, F, 4, 12, F, 1024, 64, 15, F, F, F, None, F, F, F, None,
          None, None]
    assert len(ok) == 29

    def call(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return lib.lookup_index_verify_append_draft(*a)

    assert call(a18=-1) == -1               # K < 0
    assert call(a18=65) == -1               # K above LOOKUP_DRAFT_MAX_K
    assert call(a23=None) == -1             # no draft rows with K > 0
    assert call(a24=None) == -1             # no draft lengths
    assert call(a25=None) == -1             # no positions
    assert call(a8=-1) == -1                # P < 0
    assert call(a3=F) == -1                 # probs without u
    assert call(a16=1000) == -1             # slots not a power of two
    assert call(a15=F + 8) == -1            # misaligned index
    assert call(a7=0, a0=None, a9=None) == 0   # B == 0: nothing to do
