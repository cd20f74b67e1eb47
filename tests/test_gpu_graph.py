"""CUDA graph capture of a whole fwd+bwd step through the C ABI.

After a first (eager) call of a problem, the library's calls issue only stream work -- kernel
launches and memsets on the caller's stream, no allocation, no synchronisation, no attribute
changes -- so a caller can record a training step once and replay it.  Captured here: the forward
and the backward reusing its carries, on the tensor-core kernels and on the SIMT kernels.  The
replay must give the eager results (bit for bit on the tensor-core path, whose reductions run in a
fixed order; to fp32 rounding on the SIMT path, which adds m2 / m1 with atomics), and again after
new values are written into the captured input buffers."""
import pytest
import torch

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Spec
from state_space_model_chunk_gb300.synthetic import WORKLOADS, make_inputs

from helpers import GRADS

pytestmark = pytest.mark.gpu

CASES = [
    (WORKLOADS["large_s4096"].scaled(name="graph_tc", b=2, s=256, h=4, valid="fixed:200"), True),
    (WORKLOADS["quat_s2048"].scaled(name="graph_tc_p128", b=1, s=192, h=2, p=128), True),
    (WORKLOADS["tiny_fp32"], False),
]


def _spec(w):
    return Spec(w.b, w.s, w.C, w.h, w.p, w.r, w.chunk_len, w.rot, w.rope_dim, w.quat_blocks, w.dtype)


def _step(spec, d, valid, ws):
    args = (spec, d["xhat"], d["bhat"], d["da"], d["rot"] if d["rot"].numel() else None, d["initial"], valid)
    m2, m1 = binding.moments_fwd(*args, workspace=ws)
    g = binding.moments_bwd(*args, d["d_m2"], d["d_m1"], workspace=ws, reuse_carries=True)
    return dict(m2=m2, m1=m1, **{k: g[k] for k in GRADS if g[k] is not None})


def _same(a, b, exact):
    for k in a:
        x, y = a[k].float().cpu(), b[k].float().cpu()
        if exact:
            assert torch.equal(x, y), k
        else:
            assert torch.allclose(x, y, rtol=1e-5, atol=1e-6 * max(1.0, float(y.abs().max()))), k


@pytest.mark.parametrize("w,tc", CASES, ids=[c[0].name for c in CASES])
def test_captured_step_replays_the_eager_step(w, tc):
    spec = _spec(w)
    assert binding.path(spec, True) == int(tc)
    inp = make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items() if k != "valid_len"}
    valid = inp["valid_len"]
    ws = binding.alloc_workspace(spec, True, torch.device("cuda"))
    eager = {k: v.clone() for k, v in _step(spec, d, valid, ws).items()}  # first call: eager
    torch.cuda.synchronize()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on a side stream, as capture wants
        _step(spec, d, valid, ws)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = _step(spec, d, valid, ws)
    graph.replay()
    torch.cuda.synchronize()
    _same(out, eager, tc)

    # new values in the captured input buffers: the replay follows them
    w2 = w.scaled(name=w.name + "_2", seed=w.seed + 77)
    inp2 = make_inputs(w2)
    for k, v in d.items():
        v.copy_(inp2[k].to(v.device))
    graph.replay()
    torch.cuda.synchronize()
    ws2 = binding.alloc_workspace(spec, True, torch.device("cuda"))
    eager2 = _step(spec, {k: v.clone() for k, v in d.items()}, valid, ws2)
    torch.cuda.synchronize()
    _same(out, eager2, tc)
