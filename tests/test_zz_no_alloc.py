"""The forward entry point that allocates nothing (moments_fwd_noalloc).

Callers embedded in a framework that owns all device memory, or in loops where cudaMalloc /
cudaFree would synchronise the device, or plain C callers with only their own buffers, cannot
hand the library a workspace.  For them the library keeps a fixed 16 MiB scratch array on the
device.  These tests call that entry point through the C ABI and check it against the ordinary
workspace-taking forward (the same kernels, so the two agree up to the order of floating-point
additions), twice, with a different problem run through the same array in between, so that a
call that read scratch left by an earlier call instead of setting it would show; they also check
that a problem too large for the array is refused up front, and that the array's device status
words are readable.

This file is collected last on purpose, so a stop-at-first-failure run has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Spec
from state_space_model_chunk_gb300.synthetic import WORKLOADS, make_inputs

from helpers import max_rel_err, rel_err

pytestmark = pytest.mark.gpu

TOL = 1e-5  # same kernels on both sides: only the order of the additions may differ

CASES = [
    WORKLOADS["tiny_fp32"],                                                  # SIMT kernels
    WORKLOADS["large_s4096"].scaled(name="noalloc_tc", b=2, s=256, h=4, valid="fixed:200"),  # tensor-core kernels
    WORKLOADS["halfsplit_s1024"],
    # two 64-row groups per head: the groups' moments go through the array too
    WORKLOADS["quat_s2048"].scaled(name="noalloc_p128", b=2, s=256, h=2, p=128, valid="fixed:190"),
]
# run through the array between the two compared calls: other shapes, values and valid lengths
OTHER = WORKLOADS["quat_s2048"].scaled(name="noalloc_other", b=2, s=512, h=4, valid="fixed:333", seed=17)


def spec_of(w):
    return Spec(w.b, w.s, w.C, w.h, w.p, w.r, w.chunk_len, w.rot, w.rope_dim, w.quat_blocks, w.dtype)


def _args(w):
    inp = make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items() if k != "valid_len"}
    rot = d["rot"] if d["rot"].numel() else None
    return (spec_of(w), d["xhat"], d["bhat"], d["da"], rot, d["initial"], inp["valid_len"])


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_forward_matches_workspace_forward_twice(w):
    spec = spec_of(w)
    assert 0 < binding.workspace_bytes(spec, False) <= 16 << 20
    assert 0 < binding.workspace_bytes(spec_of(OTHER), False) <= 16 << 20
    args = _args(w)
    other = _args(OTHER)
    ref2, ref1 = binding.moments_fwd(*args)
    oref2, _ = binding.moments_fwd(*other)
    torch.cuda.synchronize()
    for call in range(2):
        m2, m1 = binding.moments_fwd_noalloc(*args)
        torch.cuda.synchronize()
        assert binding.device_status(None) == 0  # MM_OK in the array's status words
        for name, got, ref in (("m2", m2, ref2), ("m1", m1, ref1)):
            g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
            e, em = rel_err(g, r), max_rel_err(g, r)
            assert e <= TOL and em <= TOL, (w.name, call, name, e, em)
        # another problem through the same array before the next compared call
        o2, _ = binding.moments_fwd_noalloc(*other)
        torch.cuda.synchronize()
        assert rel_err(o2.double().cpu().numpy(), oref2.double().cpu().numpy()) <= TOL


def test_noalloc_refuses_problems_beyond_its_scratch():
    w = WORKLOADS["large_s4096"]
    spec = spec_of(w)
    assert binding.workspace_bytes(spec, False) > 16 << 20
    lib = binding.load()
    valid = (ctypes.c_int64 * w.b)(*([w.s] * w.b))
    fake = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(7)]  # never dereferenced: refused first
    rc = lib.moments_fwd_noalloc(ctypes.byref(spec.problem()), *fake[:5], valid, fake[5], fake[6], None)
    assert rc == 3  # MM_ERR_WORKSPACE
