"""MM_FLAG_CHECK_FINITE: with the flag, a call whose outputs hold a NaN or infinity leaves
MM_ERR_NONFINITE in its workspace (read by mm_device_status); without it, or with finite
outputs, the status stays MM_OK.  A NaN input is an ordinary value here (it propagates through
the arithmetic), not a fault."""
import pytest
import torch

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Spec
from state_space_model_chunk_gb300.synthetic import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

MM_OK, MM_ERR_NONFINITE = 0, 5

CASES = [WORKLOADS["large_s4096"].scaled(name="finite_tc", b=2, s=256, h=4, C=2),  # tensor-core kernels
         # tensor-core kernels with two 64-row groups per head (outputs summed from group slices)
         WORKLOADS["large_s4096"].scaled(name="finite_tc_p128", b=1, s=128, h=2, C=2, p=128),
         WORKLOADS["tiny_fp32"]]                                                       # SIMT kernels


def _setup(w):
    spec = Spec(w.b, w.s, w.C, w.h, w.p, w.r, w.chunk_len, w.rot, w.rope_dim, w.quat_blocks, w.dtype)
    inp = make_inputs(w)
    d = {k: v.to("cuda") for k, v in inp.items() if k != "valid_len"}
    return spec, inp, d


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_forward_flag_reports_nonfinite_outputs(w):
    spec, inp, d = _setup(w)
    ws = binding.alloc_workspace(spec, False, torch.device("cuda"))
    args = (spec, d["xhat"], d["bhat"], d["da"], d["rot"])
    m2, m1 = binding.moments_fwd(*args, d["initial"], inp["valid_len"], workspace=ws, check_finite=True)
    assert binding.device_status(ws) == MM_OK and torch.isfinite(m2).all()
    bad_init = d["initial"].clone()
    bad_init[0, 0, 0, 0] = float("nan")
    m2, _ = binding.moments_fwd(*args, bad_init, inp["valid_len"], workspace=ws, check_finite=True)
    assert binding.device_status(ws) == MM_ERR_NONFINITE
    assert not torch.isfinite(m2).all()
    # the flag off: the same outputs, no check, status clean
    binding.moments_fwd(*args, bad_init, inp["valid_len"], workspace=ws)
    assert binding.device_status(ws) == MM_OK
    # and the next checked call on finite inputs clears it
    binding.moments_fwd(*args, d["initial"], inp["valid_len"], workspace=ws, check_finite=True)
    assert binding.device_status(ws) == MM_OK


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_backward_flag_reports_nonfinite_gradients(w):
    spec, inp, d = _setup(w)
    ws = binding.alloc_workspace(spec, True, torch.device("cuda"))
    args = (spec, d["xhat"], d["bhat"], d["da"], d["rot"], d["initial"], inp["valid_len"])
    g = binding.moments_bwd(*args, d["d_m2"], d["d_m1"], workspace=ws, check_finite=True)
    assert binding.device_status(ws) == MM_OK
    assert all(torch.isfinite(t.float()).all() for t in g.values() if t is not None)
    bad_dm1 = d["d_m1"].clone()
    bad_dm1[0, 0, 3] = float("inf")
    binding.moments_bwd(*args, d["d_m2"], bad_dm1, workspace=ws, check_finite=True)
    assert binding.device_status(ws) == MM_ERR_NONFINITE
    binding.moments_bwd(*args, d["d_m2"], bad_dm1, workspace=ws)
    assert binding.device_status(ws) == MM_OK
