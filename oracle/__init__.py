"""fp64 CPU oracle for the physical-frame state-moments operator.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` -- never by the product package, which
shares no code with it.

* ``moments_oracle.c`` -- the plain definition: token-by-token recurrence in fp64 with
  explicit rotation and moment sums, and its reverse-mode backward (burn-mamba,
  "mamba3/moments/backward.rs", module header "Gradient math";
  "mamba3/moments/recalculated.rs", ``moments_phys_fwd``).
* ``chunked_ref.py`` -- a NumPy restatement of the pages' own chunkwise algorithm
  (``chunk_decay``, ``chunk_states``, ``rotate_chunk``, ``boundary_carries``,
  ``moments_phys_bwd``), used only to pin the token-level oracle.
* ``rotation_steps.py`` -- the per-token cumulative rotation built from per-token steps (angle
  steps summed, quaternion steps multiplied) and that build's gradient, for calls that pass the
  rotation as steps.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moments_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmoments_oracle.so")
_lock = threading.Lock()
_lib = None

ROT_KINDS = {"none": 0, "pairwise": 1, "half": 2, "quat": 3}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O3, OpenMP over (b,h)); returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            i64, dp, ip = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)
            common = [dp, dp, dp, dp, dp, ip] + [i64] * 6 + [ctypes.c_int, i64, i64, i64, i64]
            lib.moments_oracle_fwd.argtypes = common + [dp, dp]
            lib.moments_oracle_fwd.restype = ctypes.c_int
            lib.moments_oracle_bwd.argtypes = common + [dp, dp] + [dp] * 5
            lib.moments_oracle_bwd.restype = ctypes.c_int
            lib.moments_oracle_threads.argtypes = []
            lib.moments_oracle_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    return int(_load().moments_oracle_threads())


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _prep(xhat, bhat, da, rot, initial, valid_len, rot_kind, rope_dim, quat_blocks):
    xhat, bhat, da, initial = _f64(xhat), _f64(bhat), _f64(da), _f64(initial)
    b, s, C, h, p = xhat.shape
    r = bhat.shape[-1]
    assert bhat.shape == (b, s, C, h, r) and da.shape == (b, s, h) and initial.shape == (b, h, p, r)
    kind = ROT_KINDS[rot_kind]
    if kind in (1, 2):
        a = rope_dim // 2
        rot = _f64(rot) if a > 0 else np.zeros((b, s, h, 0))
        assert rot.shape == (b, s, h, a), rot.shape
    elif kind == 3:
        rot = _f64(rot)
        assert rot.shape == (b, s, h, quat_blocks, 4), rot.shape
    else:
        rot = np.zeros((b, s, h, 0))
    vl = np.ascontiguousarray(np.broadcast_to(np.asarray(valid_len, dtype=np.int64), (b,)))
    return xhat, bhat, da, rot, initial, vl, (b, s, C, h, p, r), kind


def moments_fwd(xhat, bhat, da, rot, initial, valid_len, rot_kind="pairwise", rope_dim=0,
                quat_blocks=0, bh_range=None):
    """Oracle forward. Returns (m2 [b,h,r,r], m1 [b,h,r]) in float64."""
    xhat, bhat, da, rot, initial, vl, (b, s, C, h, p, r), kind = _prep(
        xhat, bhat, da, rot, initial, valid_len, rot_kind, rope_dim, quat_blocks)
    m2 = np.zeros((b, h, r, r))
    m1 = np.zeros((b, h, r))
    lo, hi = (0, b * h) if bh_range is None else bh_range
    rc = _load().moments_oracle_fwd(
        _ptr(xhat), _ptr(bhat), _ptr(da), _ptr(rot), _ptr(initial),
        vl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        b, s, C, h, p, r, kind, rope_dim, quat_blocks, lo, hi, _ptr(m2), _ptr(m1))
    if rc:
        raise ValueError(f"oracle forward rejected its arguments (code {rc})")
    return m2, m1


def moments_bwd(xhat, bhat, da, rot, initial, valid_len, d_m2, d_m1, rot_kind="pairwise",
                rope_dim=0, quat_blocks=0, bh_range=None):
    """Oracle backward. Returns dict of float64 grads: d_xhat, d_bhat, d_da, d_rot, d_initial."""
    xhat, bhat, da, rot, initial, vl, (b, s, C, h, p, r), kind = _prep(
        xhat, bhat, da, rot, initial, valid_len, rot_kind, rope_dim, quat_blocks)
    d_m2, d_m1 = _f64(d_m2), _f64(d_m1)
    assert d_m2.shape == (b, h, r, r) and d_m1.shape == (b, h, r)
    out = dict(d_xhat=np.zeros_like(xhat), d_bhat=np.zeros_like(bhat), d_da=np.zeros_like(da),
               d_rot=np.zeros_like(rot), d_initial=np.zeros_like(initial))
    lo, hi = (0, b * h) if bh_range is None else bh_range
    rc = _load().moments_oracle_bwd(
        _ptr(xhat), _ptr(bhat), _ptr(da), _ptr(rot), _ptr(initial),
        vl.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
        b, s, C, h, p, r, kind, rope_dim, quat_blocks, lo, hi, _ptr(d_m2), _ptr(d_m1),
        _ptr(out["d_xhat"]), _ptr(out["d_bhat"]), _ptr(out["d_da"]), _ptr(out["d_rot"]),
        _ptr(out["d_initial"]))
    if rc:
        raise ValueError(f"oracle backward rejected its arguments (code {rc})")
    return out
