"""GPU parity of the operator with the rotation given as per-token steps (MM_FLAG_ROT_STEPS): the
library builds the cumulative rotation, runs the operator on it, and returns the gradient w.r.t.
the steps.  Compared element by element with the fp64 oracle (the build and its gradient from
``oracle/rotation_steps.py`` around the token-level oracle), on the tensor-core and the SIMT
kernels, every rotation kind, several chunks of the build's scans and ragged valid lengths."""
import numpy as np
import pytest
import torch

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Spec
from state_space_model_chunk_gb300.synthetic import WORKLOADS, make_inputs, make_rot_steps

import oracle
from oracle import rotation_steps
from helpers import GRADS, compare, f64, tolerance

pytestmark = pytest.mark.gpu

CASES = [
    # (workload, force the SIMT kernels)
    (WORKLOADS["tiny_fp32"], False),
    (WORKLOADS["large_s4096"].scaled(name="steps_pairwise", b=2, s=448, h=4, valid="fixed:400"), False),
    (WORKLOADS["halfsplit_s1024"].scaled(name="steps_half", b=3, s=512, h=2, valid="ragged"), False),
    (WORKLOADS["quat_s2048"].scaled(name="steps_quat", b=2, s=384, h=3, quat_blocks=20, valid="ragged"), False),
    (WORKLOADS["quat_s2048"].scaled(name="steps_quat_simt", b=1, s=256, h=2, quat_blocks=8), True),
    (WORKLOADS["large_s4096"].scaled(name="steps_pairwise_simt", b=1, s=320, h=2, rope_dim=24), True),
    # the scans' last 64-token chunk partial (s = 80), fp32 on the SIMT kernels
    (WORKLOADS["tiny_fp32"].scaled(name="steps_partial_chunk", b=2, s=80, h=3, valid="fixed:71"), False),
    (WORKLOADS["tiny_fp32"].scaled(name="steps_quat_partial", b=1, s=80, h=2, rot="quat", rope_dim=0,
                                   quat_blocks=3, valid="fixed:80"), False),
    # two 64-row groups per head on the tensor cores
    (WORKLOADS["quat_s2048"].scaled(name="steps_quat_p128", b=2, s=192, h=2, p=128, quat_blocks=12,
                                    valid="ragged"), False),
    (WORKLOADS["large_s4096"].scaled(name="steps_pairwise_p192", b=1, s=256, h=3, p=192, C=2), False),
    # a sequence length that is not a multiple of 64 (the scans' and the kernels' last chunk partial)
    (WORKLOADS["large_s4096"].scaled(name="steps_pairwise_s200", b=2, s=200, h=2, chunk_len=40, valid="ragged"),
     False),
    # nothing valid: every output and gradient is zero
    (WORKLOADS["large_s4096"].scaled(name="steps_none_valid", b=1, s=128, h=4, valid="fixed:0"), False),
]


def _spec(w, force_generic):
    return Spec(w.b, w.s, w.C, w.h, w.p, w.r, w.chunk_len, w.rot, w.rope_dim, w.quat_blocks, w.dtype,
                force_generic, rot_steps=True)


def _oracle(w, inp, steps):
    cum = rotation_steps.build(f64(steps), w.rot)
    args = (f64(inp["xhat"]), f64(inp["bhat"]), f64(inp["da"]), cum, f64(inp["initial"]), inp["valid_len"].numpy())
    kw = dict(rot_kind=w.rot, rope_dim=w.rope_dim, quat_blocks=w.quat_blocks)
    m2, m1 = oracle.moments_fwd(*args, **kw)
    g = oracle.moments_bwd(*args, f64(inp["d_m2"]), f64(inp["d_m1"]), **kw)
    g["d_rot"] = rotation_steps.build_vjp(f64(steps), g["d_rot"], w.rot)
    g.update(m2=m2, m1=m1)
    return g


@pytest.mark.parametrize("w,simt", CASES, ids=[c[0].name + ("_simt" if c[1] else "") for c in CASES])
def test_rotation_steps_against_oracle(w, simt):
    inp = make_inputs(w)
    steps = make_rot_steps(w)
    spec = _spec(w, simt)
    plain = Spec(**{**spec.__dict__, "rot_steps": False})
    # the flag adds the build's buffers to the workspace and leaves the kernel path alone
    assert binding.workspace_bytes(spec, True) > binding.workspace_bytes(plain, True)
    assert binding.path(spec, True) == binding.path(plain, True)
    d = {k: v.cuda() for k, v in inp.items() if k != "valid_len"}
    st = steps.cuda()
    m2, m1 = binding.moments_fwd(spec, d["xhat"], d["bhat"], d["da"], st, d["initial"], inp["valid_len"])
    g = binding.moments_bwd(spec, d["xhat"], d["bhat"], d["da"], st, d["initial"], inp["valid_len"],
                            d["d_m2"], d["d_m1"])
    torch.cuda.synchronize()
    got = dict(m2=m2.cpu(), m1=m1.cpu(), **{k: g[k].cpu() for k in GRADS})
    assert got["d_rot"].shape == steps.shape
    ref = _oracle(w, inp, steps)
    compare(w.name + ("_simt" if simt else "") + "/steps", tolerance(w), [(k, got[k], ref[k]) for k in ref])
    # steps past valid_len get exactly zero gradient
    for bb in range(w.b):
        v = int(min(inp["valid_len"][bb], w.s))
        if v < w.s:
            assert torch.count_nonzero(got["d_rot"][bb, v:]) == 0


def test_rotation_steps_with_reused_carries_and_autograd():
    """The autograd wrapper (forward workspace reused by the backward) with steps: same numbers
    as separate calls."""
    w = WORKLOADS["large_s4096"].scaled(name="steps_autograd", b=1, s=256, h=4)
    inp = make_inputs(w)
    steps = make_rot_steps(w).cuda().requires_grad_(True)
    d = {k: v.cuda() for k, v in inp.items() if k != "valid_len"}
    m2, m1 = binding.moments(d["xhat"], d["bhat"], d["da"], steps, d["initial"], inp["valid_len"], w.chunk_len,
                             w.rot, w.rope_dim, rot_steps=True)
    ((m2 * d["d_m2"]).sum() + (m1 * d["d_m1"]).sum()).backward()
    ref = _oracle(w, inp, steps.detach().cpu())
    compare("steps_autograd", tolerance(w), [("m2", m2.detach(), ref["m2"]), ("m1", m1.detach(), ref["m1"]),
                                             ("d_rot", steps.grad, ref["d_rot"])])
