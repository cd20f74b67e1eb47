"""Thin ctypes binding of libmoments.so (argument marshalling only).

Every step of the operator runs in the library's CUDA kernels; PyTorch only provides device
memory and the current CUDA stream.  There is no CPU fallback: if the library is missing or
the tensors are not on a CUDA device, the calls raise.

Functions mirror the C ABI in ``include/moments.h``:

* :func:`moments_fwd`  -> (m2 [b,h,r,r], m1 [b,h,r])
* :func:`moments_bwd`  -> dict of d_xhat, d_bhat, d_da, d_rot, d_initial
* :class:`Moments` / :func:`moments` -- a ``torch.autograd.Function`` that saves only the
  five leaf inputs and recomputes everything in the backward.
"""
from __future__ import annotations

import ctypes
import os
import threading
import warnings
from dataclasses import dataclass

import torch

from . import build as _build

MM_F32, MM_BF16 = 0, 1
ROT = {"none": 0, "pairwise": 1, "half": 2, "quat": 3}
MM_FLAG_FORCE_GENERIC = 0x1
MM_FLAG_REUSE_CARRIES = 0x2
MM_FLAG_CHECK_FINITE = 0x4  # debug: outputs checked for NaN / inf, reported by device_status()
MM_FLAG_ROT_STEPS = 0x8  # rot holds per-token steps; the library builds the cumulative rotation
MM_FLAG_TEST_WAIT_TIMEOUT = 0x80000000  # testing only: see include/moments.h
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace", 4: "cuda", 5: "nonfinite",
          6: "timeout"}


class MomentsError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: status {code} ({STATUS.get(code, '?')})")
        self.code = code


class Problem(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("s", ctypes.c_int64), ("C", ctypes.c_int64), ("h", ctypes.c_int64),
                ("p", ctypes.c_int64), ("r", ctypes.c_int64), ("chunk_len", ctypes.c_int64),
                ("xb_dtype", ctypes.c_int32), ("rot", ctypes.c_int32), ("rope_dim", ctypes.c_int64),
                ("quat_blocks", ctypes.c_int64), ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmoments.so (building it first when absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libmoments.so not found at {_build.LIB}; run the build first")
            lib = ctypes.CDLL(_build.LIB)
            vp, i64p, fp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p
            pp = ctypes.POINTER(Problem)
            lib.mm_workspace_bytes.argtypes = [pp, ctypes.c_int]
            lib.mm_workspace_bytes.restype = ctypes.c_size_t
            lib.mm_path.argtypes = [pp, ctypes.c_int]
            lib.mm_path.restype = ctypes.c_int
            lib.mm_status_string.argtypes = [ctypes.c_int]
            lib.mm_status_string.restype = ctypes.c_char_p
            lib.moments_fwd.argtypes = [pp, vp, vp, fp, fp, fp, i64p, fp, fp, vp, ctypes.c_size_t, vp]
            lib.moments_fwd.restype = ctypes.c_int
            lib.moments_bwd.argtypes = [pp, vp, vp, fp, fp, fp, i64p, fp, fp, vp, vp, fp, fp, fp, vp,
                                        ctypes.c_size_t, vp]
            lib.moments_bwd.restype = ctypes.c_int
            lib.mm_device_status.argtypes = [vp, vp]
            lib.mm_device_status.restype = ctypes.c_int
            lib.moments_fwd_noalloc.argtypes = [pp, vp, vp, fp, fp, fp, i64p, fp, fp, vp]
            lib.moments_fwd_noalloc.restype = ctypes.c_int
            _lib = lib
    return _lib


@dataclass(frozen=True)
class Spec:
    """Static description of a call: shapes plus rotation flags."""
    b: int
    s: int
    C: int
    h: int
    p: int
    r: int
    chunk_len: int
    rot: str = "none"
    rope_dim: int = 0
    quat_blocks: int = 0
    dtype: str = "bf16"
    force_generic: bool = False
    rot_steps: bool = False  # rot is per-token steps (MM_FLAG_ROT_STEPS); d_rot is w.r.t. the steps

    def problem(self, extra_flags: int = 0) -> Problem:
        flags = (MM_FLAG_FORCE_GENERIC if self.force_generic else 0) | \
            (MM_FLAG_ROT_STEPS if self.rot_steps else 0) | extra_flags
        return Problem(self.b, self.s, self.C, self.h, self.p, self.r, self.chunk_len,
                       MM_BF16 if self.dtype == "bf16" else MM_F32, ROT[self.rot], self.rope_dim,
                       self.quat_blocks, flags, 0)

    @staticmethod
    def from_tensors(xhat, bhat, chunk_len, rot="none", rope_dim=0, quat_blocks=0, force_generic=False,
                     rot_steps=False):
        b, s, C, h, p = xhat.shape
        r = bhat.shape[-1]
        dt = "bf16" if xhat.dtype == torch.bfloat16 else "f32"
        return Spec(b, s, C, h, p, r, chunk_len, rot, rope_dim, quat_blocks, dt, force_generic, rot_steps)


def workspace_bytes(spec: Spec, backward: bool) -> int:
    return int(load().mm_workspace_bytes(ctypes.byref(spec.problem()), 1 if backward else 0))


def path(spec: Spec, backward: bool) -> int:
    """0 = SIMT fp32 kernels, 1 = tcgen05 tensor-core kernels."""
    return int(load().mm_path(ctypes.byref(spec.problem()), 1 if backward else 0))


_warned = set()

TC_RULES = ("bf16 operands, p a multiple of 8 below 64 or of 64 up to 512, r a multiple of 16 up to 128 "
            "(64 or 128 for half-split), "
            "C <= 8, "
            "rotation width (rope_dim/2 or 4 J) a multiple of 4 and at most 128")


def _note_path(spec: Spec, backward: bool):
    """Warn (once per problem shape) when a bf16 call falls to the SIMT kernels, which are about
    65x slower than the tensor-core kernels; mm_path() gives the same answer programmatically."""
    if spec.dtype != "bf16" or spec.force_generic:
        return
    key = (spec, backward)
    if key in _warned:
        return
    _warned.add(key)
    if path(spec, backward) == 0:
        warnings.warn(f"moments_{'bwd' if backward else 'fwd'}: this bf16 problem runs on the SIMT kernels; "
                      f"the tensor-core kernels need {TC_RULES}", RuntimeWarning, stacklevel=3)


def alloc_workspace(spec: Spec, backward: bool, device) -> torch.Tensor:
    n = max(workspace_bytes(spec, backward), 256)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise RuntimeError("libmoments runs on CUDA tensors only (no CPU fallback)")
        if t is not None and not t.is_contiguous():
            raise RuntimeError("libmoments expects contiguous tensors")


def _valid_host(valid_len, b):
    v = torch.as_tensor(valid_len, dtype=torch.int64).reshape(-1).cpu()
    if v.numel() == 1 and b != 1:
        v = v.expand(b)
    return v.contiguous()


def moments_fwd(spec: Spec, xhat, bhat, da, rot, initial, valid_len, *, workspace=None, stream=None,
                out=None, extra_flags=0, check_finite=False):
    """Forward call; returns (m2, m1) fp32 on the inputs' device.  ``extra_flags`` are OR-ed into the
    problem's flags (MM_FLAG_TEST_WAIT_TIMEOUT for the failure-path test); ``check_finite`` sets
    MM_FLAG_CHECK_FINITE (read the result with :func:`device_status` on the same workspace)."""
    lib = load()
    _check_dev(xhat, bhat, da, rot, initial)
    _note_path(spec, False)
    if check_finite:
        extra_flags |= MM_FLAG_CHECK_FINITE
    dev = xhat.device
    m2, m1 = out if out is not None else (
        torch.empty((spec.b, spec.h, spec.r, spec.r), dtype=torch.float32, device=dev),
        torch.empty((spec.b, spec.h, spec.r), dtype=torch.float32, device=dev))
    ws = workspace if workspace is not None else alloc_workspace(spec, False, dev)
    vh = _valid_host(valid_len, spec.b)
    with torch.cuda.device(dev):  # the kernels launch on the current device
        st = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
        rc = lib.moments_fwd(ctypes.byref(spec.problem(extra_flags)), _ptr(xhat), _ptr(bhat), _ptr(da), _ptr(rot),
                             _ptr(initial), ctypes.cast(vh.data_ptr(), ctypes.POINTER(ctypes.c_int64)),
                             _ptr(m2), _ptr(m1), _ptr(ws), ws.numel(), ctypes.c_void_p(st))
    if rc:
        raise MomentsError(rc, "moments_fwd")
    return m2, m1


def device_status(workspace, stream=None, device=None) -> int:
    """mm_device_status of the call that last used ``workspace`` (synchronises the stream); with
    ``workspace=None``, of the last :func:`moments_fwd_noalloc` call on ``device``."""
    lib = load()
    dev = workspace.device if workspace is not None else torch.device(device if device is not None else "cuda")
    with torch.cuda.device(dev):
        st = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
        return int(lib.mm_device_status(_ptr(workspace), ctypes.c_void_p(st)))


def moments_bwd(spec: Spec, xhat, bhat, da, rot, initial, valid_len, d_m2, d_m1, *, workspace=None,
                stream=None, out=None, reuse_carries=False, check_finite=False):
    """Backward call; returns dict d_xhat, d_bhat, d_da, d_rot, d_initial.  ``reuse_carries``:
    ``workspace`` (sized for the backward) went through :func:`moments_fwd` of the same spec and
    unchanged inputs, whose chunk carries the backward then takes instead of recomputing them.
    ``check_finite`` sets MM_FLAG_CHECK_FINITE over the five gradients."""
    if reuse_carries and workspace is None:
        raise ValueError("reuse_carries needs the workspace the forward wrote")
    lib = load()
    _check_dev(xhat, bhat, da, rot, initial, d_m2, d_m1)
    _note_path(spec, True)
    dev = xhat.device
    if out is None:
        out = dict(d_xhat=torch.empty_like(xhat), d_bhat=torch.empty_like(bhat), d_da=torch.empty_like(da),
                   d_rot=torch.empty_like(rot) if rot is not None else None,
                   d_initial=torch.empty_like(initial))
    ws = workspace if workspace is not None else alloc_workspace(spec, True, dev)
    vh = _valid_host(valid_len, spec.b)
    prob = spec.problem((MM_FLAG_REUSE_CARRIES if reuse_carries else 0) |
                        (MM_FLAG_CHECK_FINITE if check_finite else 0))
    with torch.cuda.device(dev):  # the kernels launch on the current device
        st = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
        rc = lib.moments_bwd(ctypes.byref(prob), _ptr(xhat), _ptr(bhat), _ptr(da), _ptr(rot),
                             _ptr(initial), ctypes.cast(vh.data_ptr(), ctypes.POINTER(ctypes.c_int64)),
                             _ptr(d_m2), _ptr(d_m1), _ptr(out["d_xhat"]), _ptr(out["d_bhat"]),
                             _ptr(out["d_da"]), _ptr(out["d_rot"]), _ptr(out["d_initial"]), _ptr(ws),
                             ws.numel(), ctypes.c_void_p(st))
    if rc:
        raise MomentsError(rc, "moments_bwd")
    return out


def moments_fwd_noalloc(spec: Spec, xhat, bhat, da, rot, initial, valid_len, *, stream=None, out=None):
    """Forward through ``moments_fwd_noalloc``: no workspace is passed or allocated; the library
    uses its fixed 16 MiB device scratch (for callers that cannot allocate).  Runs with the
    inputs' device current.  Calls that could overlap on the GPU must be serialised by the
    caller; :func:`device_status` with ``workspace=None`` reads the call's device status."""
    lib = load()
    _check_dev(xhat, bhat, da, rot, initial)
    dev = xhat.device
    m2, m1 = out if out is not None else (
        torch.empty((spec.b, spec.h, spec.r, spec.r), dtype=torch.float32, device=dev),
        torch.empty((spec.b, spec.h, spec.r), dtype=torch.float32, device=dev))
    vh = _valid_host(valid_len, spec.b)
    with torch.cuda.device(dev):  # the library takes the scratch of the current device
        st = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
        rc = lib.moments_fwd_noalloc(ctypes.byref(spec.problem()), _ptr(xhat), _ptr(bhat), _ptr(da), _ptr(rot),
                                     _ptr(initial), ctypes.cast(vh.data_ptr(), ctypes.POINTER(ctypes.c_int64)),
                                     _ptr(m2), _ptr(m1), ctypes.c_void_p(st))
    if rc:
        raise MomentsError(rc, "moments_fwd_noalloc")
    return m2, m1


class Moments(torch.autograd.Function):
    """(m2, m1) with the recompute backward: the five leaf inputs are saved, and the forward's
    workspace, whose chunk carries (1/chunk of the state trajectory) the backward reuses."""

    @staticmethod
    def forward(ctx, xhat, bhat, da, rot, initial, valid_len, spec):
        ws = alloc_workspace(spec, True, xhat.device)
        m2, m1 = moments_fwd(spec, xhat, bhat, da, rot, initial, valid_len, workspace=ws)
        ctx.save_for_backward(xhat, bhat, da, rot, initial)
        ctx.valid_len = valid_len
        ctx.spec = spec
        ctx.ws = ws
        return m2, m1

    @staticmethod
    def backward(ctx, d_m2, d_m1):
        xhat, bhat, da, rot, initial = ctx.saved_tensors
        sp = ctx.spec
        d_m2 = torch.zeros((sp.b, sp.h, sp.r, sp.r), device=xhat.device) if d_m2 is None else d_m2.contiguous()
        d_m1 = torch.zeros((sp.b, sp.h, sp.r), device=xhat.device) if d_m1 is None else d_m1.contiguous()
        g = moments_bwd(ctx.spec, xhat, bhat, da, rot, initial, ctx.valid_len, d_m2, d_m1, workspace=ctx.ws,
                        reuse_carries=True)
        ctx.ws = None
        return g["d_xhat"], g["d_bhat"], g["d_da"], g["d_rot"], g["d_initial"], None, None


def moments(xhat, bhat, da, rot, initial, valid_len, chunk_len, rot_kind="none", rope_dim=0, quat_blocks=0,
            rot_steps=False):
    """Differentiable (m2, m1); see :class:`Moments`.  ``rot_steps``: ``rot`` holds per-token
    steps (angle increments or per-token quaternions) and its gradient is w.r.t. them."""
    spec = Spec.from_tensors(xhat, bhat, chunk_len, rot_kind, rope_dim, quat_blocks, rot_steps=rot_steps)
    return Moments.apply(xhat, bhat, da, rot, initial, valid_len, spec)
