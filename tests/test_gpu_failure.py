"""Device failure path: a bounded wait in a tensor-core kernel gives up, the call reports
MM_ERR_TIMEOUT through the workspace's device status word, and the GPU context stays usable.
The failing wait is one that nothing completes (MM_FLAG_TEST_WAIT_TIMEOUT): no fault, trap or hang
is involved."""
import pytest
import torch

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Spec
from state_space_model_chunk_gb300.synthetic import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

MM_OK, MM_ERR_TIMEOUT = 0, 6


def test_bounded_wait_gives_up_and_reports_timeout():
    w = WORKLOADS["halfsplit_s1024"]
    spec = Spec(w.b, w.s, w.C, w.h, w.p, w.r, w.chunk_len, w.rot, w.rope_dim, w.quat_blocks, w.dtype)
    assert binding.path(spec, False) == 1  # the tensor-core kernels, whose waits are bounded
    inp = make_inputs(w)
    d = {k: v.to("cuda") for k, v in inp.items() if k != "valid_len"}
    args = (spec, d["xhat"], d["bhat"], d["da"], d["rot"], d["initial"], inp["valid_len"])
    ws = binding.alloc_workspace(spec, False, torch.device("cuda"))

    m2_ref, m1_ref = (t.clone() for t in binding.moments_fwd(*args, workspace=ws))
    assert binding.device_status(ws) == MM_OK

    binding.moments_fwd(*args, workspace=ws, extra_flags=binding.MM_FLAG_TEST_WAIT_TIMEOUT)
    assert binding.device_status(ws) == MM_ERR_TIMEOUT

    # the context is still usable: the next call runs normally and reproduces the first result
    m2, m1 = binding.moments_fwd(*args, workspace=ws)
    assert binding.device_status(ws) == MM_OK
    torch.testing.assert_close(m2, m2_ref, rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(m1, m1_ref, rtol=1e-5, atol=1e-5)
