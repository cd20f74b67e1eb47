"""Host-side checks of libmoments.so that need no GPU: it builds for sm_103a, loads, exports
every symbol include/moments.h declares, sizes workspaces, and rejects bad arguments before
enqueuing anything."""
import ctypes
import os
import re

import pytest

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Problem, Spec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    names = declared_functions()
    assert {"moments_fwd", "moments_bwd", "mm_workspace_bytes", "mm_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    lib = binding.load()
    for code in range(7):
        assert lib.mm_status_string(code)
    assert lib.mm_status_string(99) == b"unknown status"


def base_spec(**kw):
    d = dict(b=2, s=64, C=1, h=2, p=8, r=16, chunk_len=16, rot="pairwise", rope_dim=8, dtype="f32")
    d.update(kw)
    return Spec(**d)


@pytest.mark.parametrize("bad", [
    dict(s=60),                      # chunk_len does not divide s
    dict(rope_dim=7),                # odd rope_dim
    dict(rope_dim=18),               # pairwise wider than r
    dict(rot="half", r=15, rope_dim=2),   # half-split needs even r
    dict(rot="half", rope_dim=18),   # rope_dim / 2 > r / 2
    dict(rot="quat", quat_blocks=5), # 4 J > r
    dict(b=0), dict(p=0), dict(chunk_len=0),
])
def test_workspace_query_rejects_invalid(bad):
    assert binding.workspace_bytes(base_spec(**bad), False) == 0
    assert binding.workspace_bytes(base_spec(**bad), True) == 0
    assert binding.path(base_spec(**bad), True) == -1


def test_workspace_grows_with_backward_and_is_aligned():
    f, b = binding.workspace_bytes(base_spec(), False), binding.workspace_bytes(base_spec(), True)
    assert 0 < f < b and f % 256 == 0 and b % 256 == 0


def _call_fwd(spec, ptrs, valid, ws_bytes):
    lib = binding.load()
    v = (ctypes.c_int64 * spec.b)(*valid)
    return lib.moments_fwd(ctypes.byref(spec.problem()), *ptrs[:5], v, ptrs[5], ptrs[6],
                           ptrs[7], ws_bytes, None)


FAKE = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(8)]  # never dereferenced


def test_fwd_rejects_before_enqueue():
    lib = binding.load()
    spec = base_spec()
    ws = binding.workspace_bytes(spec, False)
    bad = Spec(**{**spec.__dict__, "s": 60})
    assert _call_fwd(bad, FAKE, [60, 60], ws) == 1
    assert _call_fwd(spec, FAKE, [60, -1], ws) == 1               # negative valid_len
    nul = list(FAKE)
    nul[0] = None
    assert _call_fwd(spec, nul, [60, 60], ws) == 1               # null xhat
    assert _call_fwd(spec, FAKE, [60, 60], ws - 256) == 3        # workspace too small
    mis = list(FAKE)
    mis[7] = ctypes.c_void_p(0x1010)                              # misaligned workspace
    assert _call_fwd(spec, mis, [60, 60], ws) == 3
    norot = list(FAKE)
    norot[3] = None                                               # rot missing but rope_dim > 0
    assert _call_fwd(spec, norot, [60, 60], ws) == 1
    for i in (0, 1, 2, 4, 5, 6):                                  # a tensor off a 16-byte boundary
        odd = list(FAKE)
        odd[i] = ctypes.c_void_p(0x1000 * (i + 1) + 8)
        assert _call_fwd(spec, odd, [60, 60], ws) == 1
    big = Spec(**{**spec.__dict__, "b": 600})                      # beyond the parameter block
    assert _call_fwd(big, FAKE, [1] * 600, binding.workspace_bytes(big, False)) == 2


def test_bwd_rejects_before_enqueue():
    lib = binding.load()
    spec = base_spec()
    ws = binding.workspace_bytes(spec, True)
    v = (ctypes.c_int64 * 2)(60, 60)
    args = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(14)]
    args[9] = None  # d_xhat missing
    rc = lib.moments_bwd(ctypes.byref(spec.problem()), *args[:5], v, *args[5:12], None, ws, None)
    assert rc in (1, 3)
    rc = lib.moments_bwd(ctypes.byref(Spec(**{**spec.__dict__, "rope_dim": 3}).problem()),
                         *[ctypes.c_void_p(0x1000)] * 5, v, *[ctypes.c_void_p(0x1000)] * 7,
                         ctypes.c_void_p(0x100000), ws, None)
    assert rc == 1
    args = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(14)]
    args[7] = ctypes.c_void_p(0x1000 * 8 + 4)  # d_xhat off a 16-byte boundary
    rc = lib.moments_bwd(ctypes.byref(spec.problem()), *args[:5], v, *args[5:12], ctypes.c_void_p(0x100000),
                         ws, None)
    assert rc == 1


def test_no_cpu_fallback():
    """The product path refuses CPU tensors instead of computing anything on the host."""
    import torch
    x = torch.zeros(1, 16, 1, 1, 8)
    b = torch.zeros(1, 16, 1, 1, 16)
    with pytest.raises(RuntimeError):
        binding.moments_fwd(base_spec(b=1, s=16), x, b, torch.zeros(1, 16, 1), torch.zeros(1, 16, 1, 4),
                            torch.zeros(1, 1, 8, 16), [16])


def test_flag_values_match_the_header():
    text = open(os.path.join(ROOT, "include", "moments.h")).read()
    flags = dict(re.findall(r"#define\s+(MM_FLAG_[A-Z_]+)\s+(0x[0-9a-fA-F]+)u", text))
    assert int(flags["MM_FLAG_FORCE_GENERIC"], 16) == binding.MM_FLAG_FORCE_GENERIC
    assert int(flags["MM_FLAG_REUSE_CARRIES"], 16) == binding.MM_FLAG_REUSE_CARRIES
    assert int(flags["MM_FLAG_TEST_WAIT_TIMEOUT"], 16) == binding.MM_FLAG_TEST_WAIT_TIMEOUT
    assert int(flags["MM_FLAG_CHECK_FINITE"], 16) == binding.MM_FLAG_CHECK_FINITE
    assert int(flags["MM_FLAG_ROT_STEPS"], 16) == binding.MM_FLAG_ROT_STEPS
    spec = Spec(1, 64, 1, 2, 8, 16, 16)
    assert spec.problem(binding.MM_FLAG_REUSE_CARRIES).flags == binding.MM_FLAG_REUSE_CARRIES


def test_reuse_carries_needs_the_forward_workspace():
    """The binding refuses a carry-reusing backward without the workspace the forward wrote."""
    import torch
    spec = Spec(1, 64, 1, 2, 8, 16, 16, dtype="f32")
    x = torch.zeros((1, 64, 1, 2, 8))
    with pytest.raises(ValueError):
        binding.moments_bwd(spec, x, x, x, None, x, [60], x, x, reuse_carries=True)


def test_check_finite_flag_is_accepted_and_changes_no_sizing():
    """MM_FLAG_CHECK_FINITE (0x4) is a valid flag: the workspace size and the kernel path of a
    problem do not depend on it (the check runs in the workspace header)."""
    lib = binding.load()
    for spec in (base_spec(), Spec(2, 256, 2, 4, 64, 128, 64, "pairwise", 64)):
        for bwd in (0, 1):
            plain = lib.mm_workspace_bytes(ctypes.byref(spec.problem()), bwd)
            flagged = lib.mm_workspace_bytes(ctypes.byref(spec.problem(binding.MM_FLAG_CHECK_FINITE)), bwd)
            assert plain == flagged > 0
            assert lib.mm_path(ctypes.byref(spec.problem()), bwd) == \
                lib.mm_path(ctypes.byref(spec.problem(binding.MM_FLAG_CHECK_FINITE)), bwd)
    assert lib.mm_status_string(5) == b"non-finite values detected"


def test_rotation_steps_flag_sizes_the_build():
    """MM_FLAG_ROT_STEPS adds the cumulative rotation (both calls), its gradient (backward) and the
    scans' scratch to the workspace of a rotated problem, leaves a problem without rotation alone,
    and does not change the kernel path."""
    lib = binding.load()
    for spec in (base_spec(), Spec(2, 256, 2, 4, 64, 128, 64, "pairwise", 64),
                 Spec(2, 256, 1, 4, 64, 128, 64, "quat", 0, 8)):
        flagged = spec.problem(binding.MM_FLAG_ROT_STEPS)
        nrot = 4 * spec.b * spec.s * spec.h * (spec.rope_dim // 2 if spec.rot != "quat" else 4 * spec.quat_blocks)
        for bwd in (0, 1):
            plain = lib.mm_workspace_bytes(ctypes.byref(spec.problem()), bwd)
            more = lib.mm_workspace_bytes(ctypes.byref(flagged), bwd)
            assert more >= plain + (2 if bwd else 1) * nrot and more % 256 == 0
            assert lib.mm_path(ctypes.byref(spec.problem()), bwd) == lib.mm_path(ctypes.byref(flagged), bwd)
    none = Spec(2, 256, 2, 4, 64, 128, 64)
    for bwd in (0, 1):
        assert lib.mm_workspace_bytes(ctypes.byref(none.problem(binding.MM_FLAG_ROT_STEPS)), bwd) == \
            lib.mm_workspace_bytes(ctypes.byref(none.problem()), bwd)
    assert Spec(**{**base_spec().__dict__, "rot_steps": True}).problem().flags & binding.MM_FLAG_ROT_STEPS
