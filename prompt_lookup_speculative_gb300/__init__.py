"""GB300 prompt-lookup (n-gram) speculative drafting.

Python binding of the C ABI in ``include/lookup_draft.h``,
``include/lookup_loop.h``, ``include/lookup_index.h`` and
``include/lookup_ctxcache.h`` (ctypes; argument marshalling only -- every step
runs in the library's CUDA kernels).
PyTorch tensors supply device memory and the current CUDA stream.

    draft, length, pos = lookup_draft(tokens, offsets, min_m=4, max_m=12, K=15)

``tokens`` is an int32 CUDA tensor of concatenated histories and ``offsets`` an
int64 CUDA tensor of B+1 CSR boundaries.  For each request the result is the
longest current suffix (max_m .. min_m tokens) with a most recent earlier
occurrence in the request's own history, overlap allowed, and the K tokens
following it read from the self-extended history (HyperQwen lookup-drafting
article, section "第1步").  There is no CPU fallback: if the compiled library is
missing, importing the binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "LookupDraftError", "load_library", "lookup_draft", "lookup_draft_ex", "lookup_draft_host",
    "lookup_draft_scan", "lookup_draft_fill", "lookup_draft_noalloc", "workspace_bytes",
    "set_wait_limit_ns", "lookup_fuse", "lookup_schedule", "lookup_plan", "lookup_draft_plan", "lookup_verify",
    "lookup_append", "lookup_policy",
    "NgramIndex", "index_slots_for", "index_bytes", "lookup_index_build", "lookup_index_append",
    "lookup_index_draft", "lookup_index_draft_plan", "lookup_index_verify_append",
    "lookup_index_verify_append_draft", "ContextCache",
    "load_checked_library", "check_word",
    "launch_count",
    "MAX_M", "MAX_K", "LEN_FAILED", "CHECK_BITS",
]

MAX_M = 32
MAX_K = 64
LEN_FAILED = -1
# bits of the checked build's check word (LOOKUP_DRAFT_CHECK_* in include/lookup_draft.h)
CHECK_BITS = {"offsets": 0x01, "tile": 0x02, "suffix": 0x04, "tokens": 0x08, "slots": 0x10,
              "copy": 0x20, "index": 0x40, "output": 0x80}

_lib = None
_checked_lib = None
_lib_lock = threading.Lock()


class LookupDraftError(RuntimeError):
    def __init__(self, code: int, lib):
        msg = lib.lookup_draft_strerror(code).decode()
        cuda = lib.lookup_draft_last_cuda_error().decode()
        super().__init__(f"lookup_draft failed ({code}: {msg}){': ' + cuda if cuda else ''}")
        self.code = code


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled library (building it first if nvcc is available and it is stale)."""
    global _lib
    with _lib_lock:
        if _lib is not None and path is None:
            return _lib
        if path is None:
            path = _build.LIB_PATH
            if not _build.up_to_date():
                try:
                    _build.build()
                except Exception as exc:  # no toolchain: fail loudly, never fall back
                    if not os.path.exists(path):
                        raise RuntimeError(
                            f"the CUDA library {path} is missing and could not be built: {exc}") from exc
        if not os.path.exists(path):
            raise RuntimeError(f"the CUDA library {path} is missing; run build() first")
        lib = ctypes.CDLL(path)
        _declare(lib)
        if path == _build.LIB_PATH:
            _lib = lib
        return lib


def load_checked_library() -> ctypes.CDLL:
    """The checked build of the drafting step (include/lookup_draft.h, "Checked
    build"): the entry points of lookup_draft.h with device-side index checks.
    It is built beside the regular library; a debugging aid, not the product path."""
    global _checked_lib
    load_library()                       # builds both libraries when stale
    with _lib_lock:
        if _checked_lib is None:
            path = _build.CHECKED_LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"the checked CUDA library {path} is missing; run build() first")
            lib = ctypes.CDLL(path)
            _declare_draft(lib)
            _checked_lib = _Declared(lib)
        return _checked_lib


class _Declared:
    """A library whose entry points can only be called once their argument types
    are declared: ctypes would otherwise pass 64-bit pointers as 32-bit ints."""

    def __init__(self, lib: ctypes.CDLL):
        self._lib = lib

    def __getattr__(self, name):
        fn = getattr(self._lib, name)
        if name.startswith("lookup_") and fn.argtypes is None:
            raise AttributeError(f"{name}: no argument types declared for this library")
        return fn


def check_word(lib: ctypes.CDLL, clear: bool = False) -> int:
    """The current device's check word of `lib` (0 in the regular build); device
    memory is synchronised first.  clear=True clears it after reading."""
    out = ctypes.c_uint32(0)
    _check(lib.lookup_draft_check_word(ctypes.byref(out), 1 if clear else 0), lib)
    return int(out.value)


def launch_count(lib: ctypes.CDLL | None = None) -> int:
    """Kernel launches the library has enqueued since it was loaded (a capture
    counts each captured launch once; replays are not counted)."""
    return int((lib or load_library()).lookup_draft_launch_count())


def _declare(lib: ctypes.CDLL) -> None:
    _declare_draft(lib)
    _declare_loop(lib)


def _declare_draft(lib: ctypes.CDLL) -> None:
    """Argument types of the entry points in include/lookup_draft.h."""
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.lookup_draft.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.lookup_draft.restype = ctypes.c_int
    lib.lookup_draft_ex.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.lookup_draft_ex.restype = ctypes.c_int
    lib.lookup_draft_workspace_bytes.argtypes = [i32]
    lib.lookup_draft_workspace_bytes.restype = sz
    lib.lookup_draft_scan.argtypes = [vp, vp, i32, i32, i32, vp, sz, vp]
    lib.lookup_draft_scan.restype = ctypes.c_int
    lib.lookup_draft_fill.argtypes = [vp, vp, i32, i32, i32, i32, vp, sz, vp, vp, vp, vp, vp]
    lib.lookup_draft_fill.restype = ctypes.c_int
    lib.lookup_draft_host.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.lookup_draft_host.restype = ctypes.c_int
    lib.lookup_draft_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.lookup_draft_noalloc.restype = ctypes.c_int
    lib.lookup_draft_strerror.argtypes = [ctypes.c_int]
    lib.lookup_draft_strerror.restype = ctypes.c_char_p
    lib.lookup_draft_last_cuda_error.argtypes = []
    lib.lookup_draft_last_cuda_error.restype = ctypes.c_char_p
    lib.lookup_draft_launch_count.argtypes = []
    lib.lookup_draft_launch_count.restype = ctypes.c_uint64
    lib.lookup_draft_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.lookup_draft_set_wait_limit_ns.restype = None
    lib.lookup_draft_read_floor.argtypes = [vp, sz, i32, i32, vp, vp]
    lib.lookup_draft_read_floor.restype = ctypes.c_int
    lib.lookup_draft_read_floor_bulk.argtypes = [vp, sz, vp, vp]
    lib.lookup_draft_read_floor_bulk.restype = ctypes.c_int
    lib.lookup_draft_checked_build.argtypes = []
    lib.lookup_draft_checked_build.restype = ctypes.c_int
    lib.lookup_draft_check_word.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    lib.lookup_draft_check_word.restype = ctypes.c_int
    # declared in lookup_loop.h, defined beside the draft step (so both builds export it)
    lib.lookup_draft_plan.argtypes = [vp, vp, i32, i32, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                      vp, vp, vp, vp, vp, vp, vp, vp]
    lib.lookup_draft_plan.restype = ctypes.c_int


def _declare_loop(lib: ctypes.CDLL) -> None:
    """Argument types of the entry points in include/lookup_loop.h,
    include/lookup_index.h and include/lookup_ctxcache.h."""
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.lookup_fuse.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.lookup_fuse.restype = ctypes.c_int
    lib.lookup_schedule.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    lib.lookup_schedule.restype = ctypes.c_int
    lib.lookup_plan.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp,
                                vp, vp, vp]
    lib.lookup_plan.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.lookup_policy.argtypes = [vp, vp, i32, i32, i32, f32, f32, f32, f32, f32, i32, i32, i32, vp, vp, vp, vp]
    lib.lookup_policy.restype = ctypes.c_int
    lib.lookup_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp]
    lib.lookup_verify.restype = ctypes.c_int
    lib.lookup_append.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp]
    lib.lookup_append.restype = ctypes.c_int
    i64 = ctypes.c_int64
    lib.lookup_index_slots_for.argtypes = [i64, i32, i32]
    lib.lookup_index_slots_for.restype = i64
    lib.lookup_index_bytes.argtypes = [i64]
    lib.lookup_index_bytes.restype = sz
    lib.lookup_index_build.argtypes = [vp, vp, vp, i32, i32, i32, vp, i64, i32, vp]
    lib.lookup_index_build.restype = ctypes.c_int
    lib.lookup_index_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, i64, i32, vp, vp]
    lib.lookup_index_append.restype = ctypes.c_int
    lib.lookup_index_verify_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, i32, i32, vp,
                                               i64, i32, vp, vp, vp, vp, vp]
    lib.lookup_index_verify_append.restype = ctypes.c_int
    lib.lookup_index_verify_append_draft.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, i32, i32,
                                                     vp, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.lookup_index_verify_append_draft.restype = ctypes.c_int
    lib.lookup_index_draft.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, i64, i32, vp, vp, vp, vp, vp, vp]
    lib.lookup_index_draft.restype = ctypes.c_int
    lib.lookup_index_draft_plan.argtypes = [vp, vp, vp, i32, i32, i32, vp, i64, i32, vp, vp, i32, i32, i32, i32, i32,
                                            i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.lookup_index_draft_plan.restype = ctypes.c_int
    lib.lookup_ctx_slots_for.argtypes = [i64, i32, i32]
    lib.lookup_ctx_slots_for.restype = i64
    lib.lookup_ctx_bytes.argtypes = [i64]
    lib.lookup_ctx_bytes.restype = sz
    lib.lookup_ctx_build.argtypes = [vp, vp, vp, i32, i32, i32, vp, i64, vp]
    lib.lookup_ctx_build.restype = ctypes.c_int
    lib.lookup_ctx_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, i64, vp, vp]
    lib.lookup_ctx_append.restype = ctypes.c_int
    lib.lookup_ctx_draft.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, i64, vp, vp, vp]
    lib.lookup_ctx_draft.restype = ctypes.c_int


def _check(rc: int, lib) -> None:
    if rc != 0:
        raise LookupDraftError(rc, lib)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _as_batch(tokens, offsets):
    import torch
    if not (isinstance(tokens, torch.Tensor) and isinstance(offsets, torch.Tensor)):
        raise TypeError("tokens and offsets must be torch tensors")
    if tokens.dtype != torch.int32 or offsets.dtype != torch.int64:
        raise TypeError("tokens must be int32 and offsets int64")
    if not (tokens.is_cuda and offsets.is_cuda) or tokens.device != offsets.device:
        raise ValueError("tokens and offsets must be CUDA tensors on the same device")
    if not (tokens.is_contiguous() and offsets.is_contiguous()) or offsets.dim() != 1:
        raise ValueError("tokens and offsets must be contiguous; offsets one-dimensional")
    if offsets.numel() < 1:
        raise ValueError("offsets needs B + 1 >= 1 entries")
    return offsets.numel() - 1


def _outputs(B: int, K: int, device, out, with_mlen: bool):
    import torch
    if out is None:
        draft = torch.empty((B, K), dtype=torch.int32, device=device)
        length = torch.empty(B, dtype=torch.int32, device=device)
        pos = torch.empty(B, dtype=torch.int32, device=device)
        mlen = torch.empty(B, dtype=torch.int32, device=device) if with_mlen else None
        return draft, length, pos, mlen
    draft, length, pos = out[:3]
    mlen = out[3] if len(out) > 3 else None
    for t, shape in ((draft, (B, K)), (length, (B,)), (pos, (B,))):
        if t.dtype != torch.int32 or tuple(t.shape) != shape or not t.is_contiguous() or t.device != device:
            raise ValueError("output tensors must be contiguous int32 [B, K], [B], [B] on the input device")
    return draft, length, pos, mlen


def lookup_draft(tokens, offsets, min_m: int = 4, max_m: int = 12, K: int = 15,
                 out=None, stream=None):
    """One batched draft step on the current (or given) stream; returns (draft, length, pos)."""
    import torch
    lib = load_library()
    B = _as_batch(tokens, offsets)
    draft, length, pos, _ = _outputs(B, K, tokens.device, out, False)
    with torch.cuda.device(tokens.device):
        rc = lib.lookup_draft(tokens.data_ptr(), offsets.data_ptr(), B, min_m, max_m, K,
                              draft.data_ptr(), length.data_ptr(), pos.data_ptr(),
                              _stream_handle(stream))
    _check(rc, lib)
    return draft, length, pos


def lookup_draft_ex(tokens, offsets, min_m: int = 4, max_m: int = 12, K: int = 15,
                    out=None, stream=None):
    """lookup_draft plus the match length; returns (draft, length, pos, mlen)."""
    import torch
    lib = load_library()
    B = _as_batch(tokens, offsets)
    draft, length, pos, mlen = _outputs(B, K, tokens.device, out, True)
    with torch.cuda.device(tokens.device):
        rc = lib.lookup_draft_ex(tokens.data_ptr(), offsets.data_ptr(), B, min_m, max_m, K,
                                 draft.data_ptr(), length.data_ptr(), pos.data_ptr(),
                                 mlen.data_ptr() if mlen is not None else None,
                                 _stream_handle(stream))
    _check(rc, lib)
    return draft, length, pos, mlen


def lookup_draft_noalloc(tokens, offsets, min_m: int = 4, max_m: int = 12, K: int = 15,
                         out=None, stream=None):
    """lookup_draft for callers that must not allocate device memory during a step.

    Same results as lookup_draft; the scan's scratch lives in a fixed array inside
    the library (B + 16 * SMs <= 65,536), so the call allocates nothing.  Pass
    preallocated ``out`` tensors to keep the whole call allocation-free on the
    Python side too.  Calls whose GPU work overlaps in time share that array and
    race: keep them on one stream.
    """
    import torch
    lib = load_library()
    B = _as_batch(tokens, offsets)
    draft, length, pos, _ = _outputs(B, K, tokens.device, out, False)
    with torch.cuda.device(tokens.device):
        rc = lib.lookup_draft_noalloc(tokens.data_ptr(), offsets.data_ptr(), B, min_m, max_m, K,
                                      draft.data_ptr(), length.data_ptr(), pos.data_ptr(),
                                      _stream_handle(stream))
    _check(rc, lib)
    return draft, length, pos


def workspace_bytes(B: int, device=None) -> int:
    """Scratch bytes the staged calls need for B requests on a device."""
    import torch
    lib = load_library()
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        n = lib.lookup_draft_workspace_bytes(B)
    if n == 0 and B >= 0:
        raise LookupDraftError(-2, lib)
    return int(n)


def lookup_draft_scan(tokens, offsets, min_m: int, max_m: int, workspace, stream=None) -> None:
    """Stage 1 (the scan) into a caller-owned uint8/any CUDA workspace tensor."""
    import torch
    lib = load_library()
    B = _as_batch(tokens, offsets)
    with torch.cuda.device(tokens.device):
        rc = lib.lookup_draft_scan(tokens.data_ptr(), offsets.data_ptr(), B, min_m, max_m,
                                   workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                   _stream_handle(stream))
    _check(rc, lib)


def lookup_draft_fill(tokens, offsets, min_m: int, max_m: int, K: int, workspace,
                      out=None, stream=None, with_mlen: bool = False):
    """Stage 2 (reduce + draft fill) from a workspace written by lookup_draft_scan."""
    import torch
    lib = load_library()
    B = _as_batch(tokens, offsets)
    draft, length, pos, mlen = _outputs(B, K, tokens.device, out, with_mlen)
    with torch.cuda.device(tokens.device):
        rc = lib.lookup_draft_fill(tokens.data_ptr(), offsets.data_ptr(), B, min_m, max_m, K,
                                   workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                   draft.data_ptr(), length.data_ptr(), pos.data_ptr(),
                                   mlen.data_ptr() if mlen is not None else None,
                                   _stream_handle(stream))
    _check(rc, lib)
    return (draft, length, pos, mlen) if with_mlen else (draft, length, pos)


def lookup_draft_host(tokens, offsets, min_m: int = 4, max_m: int = 12, K: int = 15,
                      out=None, stream=None, device=None):
    """The step on host (numpy or CPU torch) buffers; copies in, runs, copies out, syncs.

    Returns numpy arrays (draft [B, K], length [B], pos [B]) unless ``out`` gives
    host arrays to fill.
    """
    import numpy as np
    import torch
    lib = load_library()
    tok = np.ascontiguousarray(tokens.numpy() if isinstance(tokens, torch.Tensor) else tokens,
                               dtype=np.int32)
    off = np.ascontiguousarray(offsets.numpy() if isinstance(offsets, torch.Tensor) else offsets,
                               dtype=np.int64)
    B = off.shape[0] - 1
    if out is None:
        out = (np.empty((B, K), np.int32), np.empty(B, np.int32), np.empty(B, np.int32))
    draft, length, pos = out
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        rc = lib.lookup_draft_host(tok.ctypes.data, off.ctypes.data, B, min_m, max_m, K,
                                   _host_ptr(draft), _host_ptr(length), _host_ptr(pos),
                                   _stream_handle(stream))
    _check(rc, lib)
    return draft, length, pos


def _host_ptr(a) -> int:
    import torch
    if isinstance(a, torch.Tensor):
        if a.is_cuda or not a.is_contiguous() or a.dtype != torch.int32:
            raise ValueError("host outputs must be contiguous int32 CPU tensors or arrays")
        return a.data_ptr()
    if a.dtype.name != "int32" or not a.flags["C_CONTIGUOUS"]:
        raise ValueError("host outputs must be contiguous int32 arrays")
    return a.ctypes.data


def read_floor(data, ctas_per_sm: int = 4, threads: int = 256, out=None, stream=None) -> None:
    """Measurement aid: one launch that only streams ``data`` (a CUDA tensor whose
    byte size is a multiple of 16, 16-byte aligned) on the stream, with 16-byte
    loads (``ctas_per_sm`` x ``threads``) or, with ``ctas_per_sm`` = 0, with bulk
    copies into shared memory (lookup_draft_read_floor_bulk).  ``out`` is a
    one-element int32 CUDA tensor the kernel may write (a fold of the data, in the
    rare case it equals a fixed pattern; -1 from the bulk read whose wait ran out)."""
    import torch
    lib = load_library()
    if not (isinstance(data, torch.Tensor) and data.is_cuda and data.is_contiguous()):
        raise ValueError("data must be a contiguous CUDA tensor")
    if out is None:
        out = torch.zeros(1, dtype=torch.int32, device=data.device)
    nbytes = data.numel() * data.element_size()
    if ctas_per_sm == 0:                 # the bulk-copy (TMA) read: one CTA per SM, threads ignored
        _check(lib.lookup_draft_read_floor_bulk(data.data_ptr(), nbytes, out.data_ptr(), _stream_handle(stream)),
               lib)
        return
    _check(lib.lookup_draft_read_floor(data.data_ptr(), nbytes, ctas_per_sm, threads, out.data_ptr(),
                                       _stream_handle(stream)), lib)


def set_wait_limit_ns(ns: int) -> None:
    """Diagnostics: limit on each bounded wait inside the scan and the bulk read
    floor (0 = default 1 s)."""
    load_library().lookup_draft_set_wait_limit_ns(int(ns))


# ------------------------------------------------------------- loop steps ----
def _dev(t, dtype, shape, device, name, optional=False):
    """Check a device tensor argument; return its pointer (None for an absent optional)."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")
    return t.data_ptr()


def lookup_fuse(lookup_draft, lookup_mlen, model_draft, long_block=None, H: int = 7, T: int = 8,
                replace_min: int = 8, agree_min: int = 6, agree_n: int = 2, tail_min: int = 4,
                out=None, stream=None):
    """Merge lookup drafts with the draft model's head proposals (HyperQwen
    lookup-drafting article, section "第2步").  Returns (block [B, H+T], len [B],
    point_mass [B, H+T]), int32 tensors on the inputs' device."""
    import torch
    lib = load_library()
    dev = lookup_draft.device
    B, K = lookup_draft.shape
    args = (_dev(lookup_draft, torch.int32, (B, K), dev, "lookup_draft"),
            _dev(lookup_mlen, torch.int32, (B,), dev, "lookup_mlen"),
            _dev(model_draft, torch.int32, (B, H), dev, "model_draft"),
            _dev(long_block, torch.int32, (B,), dev, "long_block", optional=True))
    if out is None:
        out = (torch.empty((B, H + T), dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty((B, H + T), dtype=torch.int32, device=dev))
    block, ln, pm = out
    optr = (_dev(block, torch.int32, (B, H + T), dev, "block"), _dev(ln, torch.int32, (B,), dev, "len"),
            _dev(pm, torch.int32, (B, H + T), dev, "point_mass"))
    with torch.cuda.device(dev):
        rc = lib.lookup_fuse(*args, B, K, H, T, replace_min, agree_min, agree_n, tail_min, *optr,
                             _stream_handle(stream))
    _check(rc, lib)
    return block, ln, pm


def lookup_schedule(lookup_mlen, committed, state, H: int = 7, T: int = 8, tail_min: int = 4, slack: int = 1,
                    enter_steps: int = 2, sticky: int = 3, out=None, stream=None):
    """One long-block scheduling update ("第3步"); ``state`` (int32 [B, 3], zeros at
    the start) is updated in place.  Returns out_long [B]."""
    import torch
    lib = load_library()
    dev = lookup_mlen.device
    B = lookup_mlen.shape[0]
    args = (_dev(lookup_mlen, torch.int32, (B,), dev, "lookup_mlen"),
            _dev(committed, torch.int32, (B,), dev, "committed"))
    sp = _dev(state, torch.int32, (B, 3), dev, "state")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=dev)
    op = _dev(out, torch.int32, (B,), dev, "out_long")
    with torch.cuda.device(dev):
        rc = lib.lookup_schedule(*args, B, H, T, tail_min, slack, enter_steps, sticky, sp, op,
                                 _stream_handle(stream))
    _check(rc, lib)
    return out


def lookup_plan(lookup_draft, lookup_mlen, model_draft, committed, state, H: int = 7, T: int = 8,
                replace_min: int = 8, agree_min: int = 6, agree_n: int = 2, tail_min: int = 4, slack: int = 1,
                enter_steps: int = 2, sticky: int = 3, out=None, stream=None):
    """lookup_schedule, then lookup_fuse with the new long flags, in one launch
    ("第3步", "第2步").  ``state`` (int32 [B, 3]) is updated in place.  Returns
    (long [B], block [B, H+T], len [B], point_mass [B, H+T])."""
    import torch
    lib = load_library()
    dev = lookup_draft.device
    B, K = lookup_draft.shape
    args = (_dev(lookup_draft, torch.int32, (B, K), dev, "lookup_draft"),
            _dev(lookup_mlen, torch.int32, (B,), dev, "lookup_mlen"),
            _dev(model_draft, torch.int32, (B, H), dev, "model_draft"),
            _dev(committed, torch.int32, (B,), dev, "committed"))
    sp = _dev(state, torch.int32, (B, 3), dev, "state")
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, H + T), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, H + T), dtype=torch.int32, device=dev))
    lng, block, ln, pm = out
    optr = (_dev(lng, torch.int32, (B,), dev, "long"), _dev(block, torch.int32, (B, H + T), dev, "block"),
            _dev(ln, torch.int32, (B,), dev, "len"), _dev(pm, torch.int32, (B, H + T), dev, "point_mass"))
    with torch.cuda.device(dev):
        rc = lib.lookup_plan(*args, B, K, H, T, replace_min, agree_min, agree_n, tail_min, slack, enter_steps, sticky,
                             sp, *optr, _stream_handle(stream))
    _check(rc, lib)
    return lng, block, ln, pm


def lookup_draft_plan(tokens, offsets, model_draft, committed, state, min_m: int = 4, max_m: int = 12, H: int = 7,
                      T: int = 8, replace_min: int = 8, agree_min: int = 6, agree_n: int = 2, tail_min: int = 4,
                      slack: int = 1, enter_steps: int = 2, sticky: int = 3, out=None, stream=None):
    """A draft step followed by lookup_plan, in two launches ("第1步", "第3步",
    "第2步"); ``state`` (int32 [B, 3]) is updated in place.  Returns (long [B],
    block [B, H+T], len [B], point_mass [B, H+T], mlen [B], draft_len [B])."""
    import torch
    lib = load_library()
    B = _as_batch(tokens, offsets)
    t, o = tokens, offsets
    dev = t.device
    args = (_dev(model_draft, torch.int32, (B, H), dev, "model_draft"),
            _dev(committed, torch.int32, (B,), dev, "committed"))
    sp = _dev(state, torch.int32, (B, 3), dev, "state")
    W = H + T
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, W), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, W), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    lng, block, ln, pm, ml, dl = out
    optr = (_dev(lng, torch.int32, (B,), dev, "long"), _dev(block, torch.int32, (B, W), dev, "block"),
            _dev(ln, torch.int32, (B,), dev, "len"), _dev(pm, torch.int32, (B, W), dev, "point_mass"),
            _dev(ml, torch.int32, (B,), dev, "mlen"), _dev(dl, torch.int32, (B,), dev, "draft_len"))
    with torch.cuda.device(dev):
        rc = lib.lookup_draft_plan(t.data_ptr(), o.data_ptr(), B, min_m, max_m, *args, H, T, replace_min, agree_min,
                                   agree_n, tail_min, slack, enter_steps, sticky, sp, *optr, _stream_handle(stream))
    _check(rc, lib)
    return lng, block, ln, pm, ml, dl


def lookup_policy(lookup_mlen, accepted, acc, prev, n_lookup: int, n_model: int, t_lookup: float, t_model: float,
                  t_plain: float, alpha: float = 0.125, margin: float = 0.05, edges=(6, 8, 12), out=None,
                  stream=None):
    """Draft-source controller (Strata engine article, section 五): 0 plain decoding,
    1 the draft model, 2 the lookup draft, per request.  ``acc`` (float32 [B, 5])
    and ``prev`` (int32 [B, 3]) are updated in place.  Returns the choices [B]."""
    import torch
    lib = load_library()
    dev = lookup_mlen.device
    B = lookup_mlen.shape[0]
    args = (_dev(lookup_mlen, torch.int32, (B,), dev, "lookup_mlen"), _dev(accepted, torch.int32, (B,), dev, "accepted"))
    ap = _dev(acc, torch.float32, (B, 5), dev, "acc")
    pp = _dev(prev, torch.int32, (B, 3), dev, "prev")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=dev)
    op = _dev(out, torch.int32, (B,), dev, "choice")
    with torch.cuda.device(dev):
        rc = lib.lookup_policy(*args, B, n_lookup, n_model, t_lookup, t_model, t_plain, alpha, margin,
                               int(edges[0]), int(edges[1]), int(edges[2]), ap, pp, op, _stream_handle(stream))
    _check(rc, lib)
    return out


def lookup_verify(block, length, target, probs=None, qprobs=None, point_mass=None, u=None,
                  out=None, stream=None):
    """Greedy (``probs`` None) or sampled verification of proposal blocks
    ("第3步").  Returns (accepted [B], commit [B, P+1], ncommit [B])."""
    import torch
    lib = load_library()
    dev = block.device
    B, P = block.shape
    f32 = torch.float32
    args = (_dev(block, torch.int32, (B, P), dev, "block"), _dev(length, torch.int32, (B,), dev, "len"),
            _dev(target, torch.int32, (B, P + 1), dev, "target"),
            _dev(probs, f32, (B, P), dev, "probs", optional=True),
            _dev(qprobs, f32, (B, P), dev, "qprobs", optional=True),
            _dev(point_mass, torch.int32, (B, P), dev, "point_mass", optional=True),
            _dev(u, f32, (B, P), dev, "u", optional=probs is None))
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, P + 1), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
    acc, commit, nc = out
    optr = (_dev(acc, torch.int32, (B,), dev, "accepted"), _dev(commit, torch.int32, (B, P + 1), dev, "commit"),
            _dev(nc, torch.int32, (B,), dev, "ncommit"))
    with torch.cuda.device(dev):
        rc = lib.lookup_verify(*args, B, P, *optr, _stream_handle(stream))
    _check(rc, lib)
    return acc, commit, nc


def lookup_append(tokens, offsets, commit, ncommit, out=None, stream=None):
    """The next step's CSR batch: every history followed by its committed tokens.

    Returns (new_tokens, new_offsets).  Without ``out`` the token buffer holds
    offsets[B] - offsets[0] + B * W tokens, enough for any counts, so the call
    never reads the counts back to the host; the batch is
    new_tokens[new_offsets[0] .. new_offsets[B]).
    """
    import torch
    lib = load_library()
    B = _as_batch(tokens, offsets)
    dev = tokens.device
    W = commit.shape[1]
    cp = _dev(commit, torch.int32, (B, W), dev, "commit")
    np_ = _dev(ncommit, torch.int32, (B,), dev, "ncommit")
    if out is None:
        out = (torch.empty(tokens.numel() + B * W, dtype=torch.int32, device=dev),
               torch.empty(B + 1, dtype=torch.int64, device=dev))
    out_t, out_o = out
    if out_t.dtype != torch.int32 or not out_t.is_contiguous() or out_t.device != dev:
        raise ValueError("out tokens must be a contiguous int32 tensor on the inputs' device")
    op = _dev(out_o, torch.int64, (B + 1,), dev, "out_offsets")
    # an empty tensor has no address; with no history token and nothing to write the
    # kernel dereferences neither pointer, so any valid aligned address will do
    tp = tokens.data_ptr() if tokens.numel() else offsets.data_ptr()
    otp = out_t.data_ptr() if out_t.numel() else out_o.data_ptr()
    with torch.cuda.device(dev):
        rc = lib.lookup_append(tp, offsets.data_ptr(), cp, np_, B, W, otp, op, _stream_handle(stream))
    _check(rc, lib)
    return out_t, out_o


# ----------------------------------------------------------- n-gram index ----
def index_slots_for(capacity_tokens: int, min_m: int = 4, max_m: int = 12) -> int:
    """Recommended slot count (a power of two, load factor <= 1/2)."""
    n = load_library().lookup_index_slots_for(int(capacity_tokens), min_m, max_m)
    if n <= 0:
        raise ValueError("invalid index parameters")
    return int(n)


def index_bytes(slots: int) -> int:
    n = load_library().lookup_index_bytes(int(slots))
    if n == 0:
        raise ValueError("slots must be a power of two >= 16")
    return int(n)


def _slab_args(tokens, base, length, cap=None):
    import torch
    dev = tokens.device
    B = base.shape[0]
    if tokens.dtype != torch.int32 or not tokens.is_contiguous() or not tokens.is_cuda:
        raise ValueError("tokens must be a contiguous int32 CUDA tensor")
    ptrs = (_dev(base, torch.int64, (B,), dev, "base"), _dev(length, torch.int32, (B,), dev, "len"))
    if cap is not None:
        ptrs += (_dev(cap, torch.int32, (B,), dev, "cap"),)
    return dev, B, ptrs


def lookup_index_build(tokens, base, length, min_m: int, max_m: int, index, slots: int, hash_bits: int = 64,
                       stream=None) -> None:
    """Build the n-gram index of the slab histories tokens[base[r] .. base[r] + len[r])."""
    import torch
    lib = load_library()
    dev, B, (bp, lp) = _slab_args(tokens, base, length)
    with torch.cuda.device(dev):
        rc = lib.lookup_index_build(tokens.data_ptr(), bp, lp, B, min_m, max_m, index.data_ptr(), int(slots),
                                    hash_bits, _stream_handle(stream))
    _check(rc, lib)


def lookup_index_append(tokens, base, length, cap, commit, ncommit, min_m: int, max_m: int, index, slots: int,
                        hash_bits: int = 64, status=None, stream=None):
    """Append each request's committed tokens in place, index them, grow len.
    Returns the per-request status tensor (0 ok, 1 slab full, 2 index mismatch)."""
    import torch
    lib = load_library()
    dev, B, (bp, lp, cp) = _slab_args(tokens, base, length, cap)
    W = commit.shape[1]
    cm = _dev(commit, torch.int32, (B, W), dev, "commit")
    nc = _dev(ncommit, torch.int32, (B,), dev, "ncommit")
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    sp = _dev(status, torch.int32, (B,), dev, "status")
    with torch.cuda.device(dev):
        rc = lib.lookup_index_append(tokens.data_ptr(), bp, lp, cp, cm, nc, B, W, min_m, max_m, index.data_ptr(),
                                     int(slots), hash_bits, sp, _stream_handle(stream))
    _check(rc, lib)
    return status


def lookup_index_verify_append(block, length, target, tokens, base, slab_len, cap, min_m: int, max_m: int, index,
                               slots: int, probs=None, qprobs=None, point_mass=None, u=None, hash_bits: int = 64,
                               out=None, status=None, stream=None):
    """lookup_verify followed by lookup_index_append of its commit rows, in one
    launch when the batch fits one wave of per-request CTAs.  ``length`` is the
    blocks' lengths, ``slab_len`` the histories' (grown in place).  Returns
    (accepted [B], commit [B, P+1], ncommit [B], status [B])."""
    import torch
    lib = load_library()
    dev, B, (bp, lp, cp) = _slab_args(tokens, base, slab_len, cap)
    P = block.shape[1]
    f32 = torch.float32
    args = (_dev(block, torch.int32, (B, P), dev, "block"), _dev(length, torch.int32, (B,), dev, "len"),
            _dev(target, torch.int32, (B, P + 1), dev, "target"),
            _dev(probs, f32, (B, P), dev, "probs", optional=True),
            _dev(qprobs, f32, (B, P), dev, "qprobs", optional=True),
            _dev(point_mass, torch.int32, (B, P), dev, "point_mass", optional=True),
            _dev(u, f32, (B, P), dev, "u", optional=probs is None))
    if out is None:
        out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty((B, P + 1), dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev))
    acc, commit, nc = out
    optr = (_dev(acc, torch.int32, (B,), dev, "accepted"), _dev(commit, torch.int32, (B, P + 1), dev, "commit"),
            _dev(nc, torch.int32, (B,), dev, "ncommit"))
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    sp = _dev(status, torch.int32, (B,), dev, "status")
    with torch.cuda.device(dev):
        rc = lib.lookup_index_verify_append(*args, B, P, tokens.data_ptr(), bp, lp, cp, min_m, max_m,
                                            index.data_ptr(), int(slots), hash_bits, *optr, sp,
                                            _stream_handle(stream))
    _check(rc, lib)
    return acc, commit, nc, status


def lookup_index_verify_append_draft(block, length, target, tokens, base, slab_len, cap, min_m: int, max_m: int,
                                     index, slots: int, K: int, probs=None, qprobs=None, point_mass=None, u=None,
                                     hash_bits: int = 64, out=None, stream=None):
    """lookup_index_verify_append, then lookup_index_draft (K tokens) on the grown
    histories: one launch when the batch fits one wave of per-request CTAs.
    Returns (accepted, commit [B, P+1], ncommit, status, draft [B, K], draft_len,
    pos, mlen, fallback)."""
    import torch
    lib = load_library()
    dev, B, (bp, lp, cp) = _slab_args(tokens, base, slab_len, cap)
    P = block.shape[1]
    f32 = torch.float32
    args = (_dev(block, torch.int32, (B, P), dev, "block"), _dev(length, torch.int32, (B,), dev, "len"),
            _dev(target, torch.int32, (B, P + 1), dev, "target"),
            _dev(probs, f32, (B, P), dev, "probs", optional=True),
            _dev(qprobs, f32, (B, P), dev, "qprobs", optional=True),
            _dev(point_mass, torch.int32, (B, P), dev, "point_mass", optional=True),
            _dev(u, f32, (B, P), dev, "u", optional=probs is None))
    shapes = ((B,), (B, P + 1), (B,), (B,), (B, K), (B,), (B,), (B,), (B,))
    names = ("accepted", "commit", "ncommit", "status", "draft", "draft_len", "pos", "mlen", "fallback")
    if out is None:
        out = tuple(torch.empty(sh, dtype=torch.int32, device=dev) for sh in shapes)
    optr = tuple(_dev(t, torch.int32, sh, dev, nm) for t, sh, nm in zip(out, shapes, names))
    with torch.cuda.device(dev):
        rc = lib.lookup_index_verify_append_draft(*args, B, P, tokens.data_ptr(), bp, lp, cp, min_m, max_m,
                                                  index.data_ptr(), int(slots), hash_bits, K, *optr[:4], *optr[4:],
                                                  _stream_handle(stream))
    _check(rc, lib)
    return out


def lookup_index_draft(tokens, base, length, min_m: int, max_m: int, K: int, index, slots: int,
                       hash_bits: int = 64, out=None, with_fallback: bool = False, stream=None):
    """The draft step from the index; exactly lookup_draft_ex's results for the slab
    histories.  Returns (draft, len, pos, mlen) and, with with_fallback, the
    per-request flag of the brute-force path."""
    import torch
    lib = load_library()
    dev, B, (bp, lp) = _slab_args(tokens, base, length)
    if out is None:
        out = (torch.empty((B, K), dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev),
               torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    draft, ln, pos, mlen = out
    fb = torch.empty(B, dtype=torch.int32, device=dev) if with_fallback else None
    optr = (_dev(draft, torch.int32, (B, K), dev, "draft"), _dev(ln, torch.int32, (B,), dev, "len"),
            _dev(pos, torch.int32, (B,), dev, "pos"), _dev(mlen, torch.int32, (B,), dev, "mlen"),
            _dev(fb, torch.int32, (B,), dev, "fallback", optional=True))
    with torch.cuda.device(dev):
        rc = lib.lookup_index_draft(tokens.data_ptr(), bp, lp, B, min_m, max_m, K, index.data_ptr(), int(slots),
                                    hash_bits, *optr, _stream_handle(stream))
    _check(rc, lib)
    return (draft, ln, pos, mlen, fb) if with_fallback else (draft, ln, pos, mlen)


def lookup_index_draft_plan(tokens, base, length, min_m: int, max_m: int, index, slots: int, model_draft, committed,
                            state, H: int = 7, T: int = 8, replace_min: int = 8, agree_min: int = 6, agree_n: int = 2,
                            tail_min: int = 4, slack: int = 1, enter_steps: int = 2, sticky: int = 3,
                            hash_bits: int = 64, out=None, stream=None):
    """lookup_index_draft (K = H + T) followed by lookup_plan, in one launch;
    ``state`` (int32 [B, 3]) is updated in place.  Returns (long, block, len,
    point_mass, mlen, draft_len, fallback)."""
    import torch
    lib = load_library()
    dev, B, (bp, lp) = _slab_args(tokens, base, length)
    W = H + T
    args = (_dev(model_draft, torch.int32, (B, H), dev, "model_draft"),
            _dev(committed, torch.int32, (B,), dev, "committed"))
    sp = _dev(state, torch.int32, (B, 3), dev, "state")
    shapes = ((B,), (B, W), (B,), (B, W), (B,), (B,), (B,))
    if out is None:
        out = tuple(torch.empty(sh, dtype=torch.int32, device=dev) for sh in shapes)
    names = ("long", "block", "len", "point_mass", "mlen", "draft_len", "fallback")
    optr = tuple(_dev(t, torch.int32, sh, dev, nm) for t, sh, nm in zip(out, shapes, names))
    with torch.cuda.device(dev):
        rc = lib.lookup_index_draft_plan(tokens.data_ptr(), bp, lp, B, min_m, max_m, index.data_ptr(), int(slots),
                                         hash_bits, *args, H, T, replace_min, agree_min, agree_n, tail_min, slack,
                                         enter_steps, sticky, sp, *optr, _stream_handle(stream))
    _check(rc, lib)
    return out


class NgramIndex:
    """A device-resident n-gram index over slab histories (include/lookup_index.h).

    Holds the index memory and its parameters; every method is one library call.
    """

    def __init__(self, capacity_tokens: int, min_m: int = 4, max_m: int = 12, device=None,
                 hash_bits: int = 64, slots: int | None = None):
        import torch
        self.min_m, self.max_m, self.hash_bits = min_m, max_m, hash_bits
        self.slots = int(slots) if slots is not None else index_slots_for(capacity_tokens, min_m, max_m)
        nbytes = index_bytes(self.slots)
        self.memory = torch.empty(nbytes, dtype=torch.uint8,
                                  device=device if device is not None else torch.cuda.current_device())

    def build(self, tokens, base, length, stream=None) -> None:
        lookup_index_build(tokens, base, length, self.min_m, self.max_m, self.memory, self.slots,
                           self.hash_bits, stream)

    def append(self, tokens, base, length, cap, commit, ncommit, status=None, stream=None):
        return lookup_index_append(tokens, base, length, cap, commit, ncommit, self.min_m, self.max_m,
                                   self.memory, self.slots, self.hash_bits, status, stream)

    def verify_append(self, block, block_len, target, tokens, base, length, cap, stream=None, **sampled):
        """Verify the blocks, then append what they commit (lookup_index_verify_append);
        ``sampled`` takes probs, qprobs, point_mass and u for sampled verification."""
        return lookup_index_verify_append(block, block_len, target, tokens, base, length, cap, self.min_m,
                                          self.max_m, self.memory, self.slots, hash_bits=self.hash_bits,
                                          stream=stream, **sampled)

    def verify_append_draft(self, block, block_len, target, tokens, base, length, cap, K: int = 15, stream=None,
                            **sampled):
        """Verify the blocks, append what they commit, and draft K tokens from the
        grown histories (lookup_index_verify_append_draft)."""
        return lookup_index_verify_append_draft(block, block_len, target, tokens, base, length, cap, self.min_m,
                                                self.max_m, self.memory, self.slots, K, hash_bits=self.hash_bits,
                                                stream=stream, **sampled)

    def draft_plan(self, tokens, base, length, model_draft, committed, state, H: int = 7, T: int = 8, stream=None,
                   **rules):
        """The draft from the index, then scheduling and fusion, in one launch
        (lookup_index_draft_plan)."""
        return lookup_index_draft_plan(tokens, base, length, self.min_m, self.max_m, self.memory, self.slots,
                                       model_draft, committed, state, H, T, hash_bits=self.hash_bits, stream=stream,
                                       **rules)

    def draft(self, tokens, base, length, K: int = 15, out=None, with_fallback: bool = False, stream=None):
        return lookup_index_draft(tokens, base, length, self.min_m, self.max_m, K, self.memory, self.slots,
                                  self.hash_bits, out, with_fallback, stream)


# ---------------------------------------------------------- context cache ----
class ContextCache:
    """Context-cache drafting (include/lookup_ctxcache.h): n-gram statistics of
    the slab histories, n in [n_min, n_max] (1..4), on the device.

    min_count and share ((num, den) per n, index n - 1) are the acceptance
    thresholds; the defaults take the llama.cpp article's 4-gram example (seen at
    least once, the top next token at least half of the time) for every n.
    """

    def __init__(self, capacity_tokens: int, n_min: int = 1, n_max: int = 4, device=None, slots: int | None = None,
                 min_count=(1, 1, 1, 1), share=((1, 2), (1, 2), (1, 2), (1, 2))):
        import torch
        lib = load_library()
        self.n_min, self.n_max = n_min, n_max
        self.slots = int(slots) if slots is not None else int(lib.lookup_ctx_slots_for(int(capacity_tokens), n_min,
                                                                                      n_max))
        nbytes = int(lib.lookup_ctx_bytes(self.slots))
        if nbytes == 0:
            raise ValueError("invalid context-cache parameters")
        self.memory = torch.empty(nbytes, dtype=torch.uint8,
                                  device=device if device is not None else torch.cuda.current_device())
        self.set_thresholds(min_count, share)

    def set_thresholds(self, min_count, share) -> None:
        import numpy as np
        self._mc = np.ascontiguousarray(min_count, dtype=np.int32)
        self._num = np.ascontiguousarray([s[0] for s in share], dtype=np.int32)
        self._den = np.ascontiguousarray([s[1] for s in share], dtype=np.int32)
        if self._mc.shape != (4,) or self._num.shape != (4,) or self._den.shape != (4,):
            raise ValueError("min_count and share need 4 entries (n = 1..4)")

    def build(self, tokens, base, length, stream=None) -> None:
        import torch
        lib = load_library()
        dev, B, (bp, lp) = _slab_args(tokens, base, length)
        with torch.cuda.device(dev):
            rc = lib.lookup_ctx_build(tokens.data_ptr(), bp, lp, B, self.n_min, self.n_max, self.memory.data_ptr(),
                                      self.slots, _stream_handle(stream))
        _check(rc, lib)

    def append(self, tokens, base, length, cap, commit, ncommit, status=None, stream=None):
        import torch
        lib = load_library()
        dev, B, (bp, lp, cp) = _slab_args(tokens, base, length, cap)
        W = commit.shape[1]
        cm = _dev(commit, torch.int32, (B, W), dev, "commit")
        nc = _dev(ncommit, torch.int32, (B,), dev, "ncommit")
        if status is None:
            status = torch.empty(B, dtype=torch.int32, device=dev)
        sp = _dev(status, torch.int32, (B,), dev, "status")
        with torch.cuda.device(dev):
            rc = lib.lookup_ctx_append(tokens.data_ptr(), bp, lp, cp, cm, nc, B, W, self.n_min, self.n_max,
                                       self.memory.data_ptr(), self.slots, sp, _stream_handle(stream))
        _check(rc, lib)
        return status

    def draft(self, tokens, base, length, K: int = 8, out=None, stream=None):
        """Returns (draft [B, K] int32, -1 past the end; len [B] int32)."""
        import torch
        lib = load_library()
        dev, B, (bp, lp) = _slab_args(tokens, base, length)
        if out is None:
            out = (torch.empty((B, K), dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
        d, ln = out
        dp = _dev(d, torch.int32, (B, K), dev, "draft")
        lnp = _dev(ln, torch.int32, (B,), dev, "len")
        with torch.cuda.device(dev):
            rc = lib.lookup_ctx_draft(tokens.data_ptr(), bp, lp, B, self.n_min, self.n_max, K, self._mc.ctypes.data,
                                      self._num.ctypes.data, self._den.ctypes.data, self.memory.data_ptr(),
                                      self.slots, dp, lnp, _stream_handle(stream))
        _check(rc, lib)
        return d, ln
