"""The forward entry point that allocates nothing (moments_fwd_noalloc).

Callers embedded in a framework that owns all device memory, or in loops where cudaMalloc /
cudaFree would synchronise the device, or plain C callers with only their own buffers, cannot
hand the library a workspace.  For them the library keeps a fixed 16 MiB scratch array on the
device.  These tests call that entry point through the C ABI and check it against the ordinary
workspace-taking forward, twice in a row (the second call reuses the array the first one left
behind), and check that a problem too large for the array is refused up front.

This file is collected last on purpose, so a stop-at-first-failure run has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Spec
from state_space_model_chunk_gb300.synthetic import WORKLOADS, make_inputs

from helpers import rel_err, tolerance

pytestmark = pytest.mark.gpu

CASES = [
    WORKLOADS["tiny_fp32"],                                                  # SIMT kernels
    WORKLOADS["large_s4096"].scaled(name="noalloc_tc", b=2, s=256, h=4, valid="fixed:200"),  # tensor-core kernels
    WORKLOADS["halfsplit_s1024"],
]


def spec_of(w):
    return Spec(w.b, w.s, w.C, w.h, w.p, w.r, w.chunk_len, w.rot, w.rope_dim, w.quat_blocks, w.dtype)


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_forward_matches_workspace_forward_twice(w):
    spec = spec_of(w)
    assert 0 < binding.workspace_bytes(spec, False) <= 16 << 20
    inp = make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items() if k != "valid_len"}
    rot = d["rot"] if d["rot"].numel() else None
    ref2, ref1 = binding.moments_fwd(spec, d["xhat"], d["bhat"], d["da"], rot, d["initial"], inp["valid_len"])
    torch.cuda.synchronize()
    tol = tolerance(w)
    for call in range(2):
        m2, m1 = binding.moments_fwd_noalloc(spec, d["xhat"], d["bhat"], d["da"], rot, d["initial"],
                                             inp["valid_len"])
        torch.cuda.synchronize()
        e2 = rel_err(m2.double().cpu().numpy(), ref2.double().cpu().numpy())
        e1 = rel_err(m1.double().cpu().numpy(), ref1.double().cpu().numpy())
        assert e2 <= tol and e1 <= tol, (w.name, call, e2, e1)


def test_noalloc_refuses_problems_beyond_its_scratch():
    w = WORKLOADS["large_s4096"]
    spec = spec_of(w)
    assert binding.workspace_bytes(spec, False) > 16 << 20
    lib = binding.load()
    fn = lib.moments_fwd_noalloc
    fn.argtypes = [ctypes.POINTER(binding.Problem)] + [ctypes.c_void_p] * 5 + [ctypes.POINTER(ctypes.c_int64)] + \
        [ctypes.c_void_p] * 3
    fn.restype = ctypes.c_int
    valid = (ctypes.c_int64 * w.b)(*([w.s] * w.b))
    fake = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(7)]  # never dereferenced: refused first
    rc = fn(ctypes.byref(spec.problem()), *fake[:5], valid, fake[5], fake[6], None)
    assert rc == 3  # MM_ERR_WORKSPACE
