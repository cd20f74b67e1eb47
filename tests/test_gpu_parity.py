"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, per output tensor both
normwise (||gpu - ref|| / ||ref||) and element-wise (max |gpu - ref| / max |ref|), with the bar
1e-4 for fp32 inputs and 2e-2 for bf16 inputs, plus exact zeros for every gradient position at
or past valid_len."""
import numpy as np
import pytest
import torch

from state_space_model_chunk_gb300 import binding
from state_space_model_chunk_gb300.binding import Spec
from state_space_model_chunk_gb300.synthetic import WORKLOADS, Workload, make_inputs, slice_bh

from helpers import GRADS, compare, oracle_bwd, oracle_fwd, tolerance

pytestmark = pytest.mark.gpu

DEV = "cuda"


def spec_of(w, force_generic=False):
    return Spec(w.b, w.s, w.C, w.h, w.p, w.r, w.chunk_len, w.rot, w.rope_dim, w.quat_blocks, w.dtype,
                force_generic)


def expected_fast(w, backward):
    """Whether the tensor-core kernels implement this workload (else the SIMT kernels run)."""
    rw = w.rope_dim // 2 if w.rot in ("pairwise", "half") else (4 * w.quat_blocks if w.rot == "quat" else 0)
    r_ok = w.r in (64, 128) if w.rot == "half" else (w.r % 16 == 0 and 16 <= w.r <= 128)
    p_ok = (w.p % 64 == 0 and 64 <= w.p <= 512) or (w.p % 8 == 0 and 8 <= w.p < 64)
    return (w.dtype == "bf16" and p_ok and r_ok and 1 <= w.C <= 8
            and rw % 4 == 0 and rw <= 128)


def run_gpu(w, inp, force_generic=False):
    d = {k: v.to(DEV) for k, v in inp.items() if k != "valid_len"}
    spec = spec_of(w, force_generic)
    assert binding.path(spec, False) == (0 if force_generic else int(expected_fast(w, False))), w.name
    assert binding.path(spec, True) == (0 if force_generic else int(expected_fast(w, True))), w.name
    rot = d["rot"] if d["rot"].numel() else None
    m2, m1 = binding.moments_fwd(spec, d["xhat"], d["bhat"], d["da"], rot, d["initial"], inp["valid_len"])
    g = binding.moments_bwd(spec, d["xhat"], d["bhat"], d["da"], rot, d["initial"], inp["valid_len"],
                            d["d_m2"], d["d_m1"])
    torch.cuda.synchronize()
    out = dict(m2=m2.cpu(), m1=m1.cpu())
    for k in GRADS:
        out[k] = g[k].cpu() if g[k] is not None else torch.zeros(0)
    return out


def check_against_oracle(w, inp, got, label=""):
    tol = tolerance(w)
    m2, m1 = oracle_fwd(w, inp)
    ref = oracle_bwd(w, inp)
    ref.update(m2=m2, m1=m1)
    errs = compare(label or w.name, tol, [(k, got[k], ref[k]) for k in ("m2", "m1") + GRADS])
    # positions at or past valid_len carry exactly zero gradient
    for bb in range(w.b):
        v = int(min(inp["valid_len"][bb], w.s))
        for k in ("d_xhat", "d_bhat", "d_da", "d_rot"):
            t = got[k]
            if t.numel() and v < w.s:
                assert torch.count_nonzero(t[bb, v:]) == 0, (label, k, bb)
    return errs


SMALL = [
    WORKLOADS["tiny_fp32"],
    WORKLOADS["halfsplit_s1024"],
    WORKLOADS["quat_s2048"].scaled(name="quat_small", b=2, s=256, h=4),
    WORKLOADS["large_s4096"].scaled(name="large_small", b=2, s=256, h=4, valid="fixed:200"),
    WORKLOADS["ragged_s16384"].scaled(name="ragged_small", b=3, s=512, h=4),
    WORKLOADS["large_s4096"].scaled(name="large_fp32_small", b=1, s=128, h=2, dtype="f32", xb_scale="unit"),
    WORKLOADS["halfsplit_s1024"].scaled(name="half_partial_rope", b=2, s=192, h=3, rope_dim=20, chunk_len=32),
    WORKLOADS["large_s4096"].scaled(name="pairwise_r96_c3", b=2, s=128, C=3, h=2, r=96, rope_dim=40),
    # r below 128 on the tensor cores (the tiles' tail columns load as zeros)
    WORKLOADS["quat_s2048"].scaled(name="quat_r32", b=2, s=192, h=3, r=32, quat_blocks=8),
    WORKLOADS["large_s4096"].scaled(name="pairwise_r48_c5", b=1, s=256, h=3, C=5, r=48, rope_dim=24,
                                    valid="fixed:200"),
    WORKLOADS["large_s4096"].scaled(name="norot_r112", b=2, s=128, h=2, r=112, rot="none", rope_dim=0),
    # half-split with r = 96 pairs columns 48 apart: the SIMT kernels
    WORKLOADS["halfsplit_s1024"].scaled(name="half_r96_simt", b=1, s=128, h=2, r=96, rope_dim=32),
    WORKLOADS["quat_s2048"].scaled(name="quat_partial_blocks", b=2, s=128, h=4, quat_blocks=20, C=2),
    WORKLOADS["tiny_fp32"].scaled(name="norot_odd", b=2, s=48, C=3, h=3, p=5, r=12, chunk_len=12, rot="none",
                                  rope_dim=0, valid="fixed:37"),
    # head counts that are not multiples of 4 (da rows not 16-byte multiples) on the tensor-core kernels
    WORKLOADS["large_s4096"].scaled(name="pairwise_h6", b=2, s=256, h=6, C=3, valid="fixed:230"),
    WORKLOADS["quat_s2048"].scaled(name="quat_h5", b=1, s=192, h=5),
    WORKLOADS["halfsplit_s1024"].scaled(name="half_r64_h3", b=2, s=256, h=3, chunk_len=32),
    WORKLOADS["ragged_s16384"].scaled(name="ragged_h1", b=3, s=384, h=1, chunk_len=64),
    # five to eight channels (the correction kernel's 16-token stages)
    WORKLOADS["large_s4096"].scaled(name="pairwise_c8", b=1, s=256, h=4, C=8, valid="fixed:241"),
    WORKLOADS["quat_s2048"].scaled(name="quat_c5", b=2, s=192, h=2, C=5),
    WORKLOADS["halfsplit_s1024"].scaled(name="half_r64_c7", b=1, s=320, h=3, C=7),
    # p above 64 on the tensor cores: each head's state rows run as groups of 64, whose moments
    # and d_bhat / d_da / d_rot are summed afterwards
    WORKLOADS["large_s4096"].scaled(name="pairwise_p128_h3", b=2, s=192, h=3, p=128, valid="fixed:150"),
    WORKLOADS["quat_s2048"].scaled(name="quat_p128_h4", b=1, s=256, h=4, p=128, quat_blocks=20),
    WORKLOADS["halfsplit_s1024"].scaled(name="half_p192_r64", b=2, s=128, h=2, p=192, C=2),
    WORKLOADS["large_s4096"].scaled(name="norot_p256_r32", b=1, s=128, h=2, p=256, r=32, rot="none", rope_dim=0),
    WORKLOADS["ragged_s16384"].scaled(name="ragged_p128_c5", b=3, s=256, h=2, p=128, C=5, r=80, rot="pairwise",
                                      rope_dim=48, chunk_len=64),
    # sequence lengths that are not a multiple of 64: the last chunk of every row is partial --
    # paired after a full chunk (s = 200, 100, 72) or alone in its pair (s = 136) -- and the
    # copies of its missing tokens run past the row (into the next row, or past the tensor)
    WORKLOADS["large_s4096"].scaled(name="pairwise_s200", b=2, s=200, h=4, chunk_len=8, valid="ragged"),
    WORKLOADS["quat_s2048"].scaled(name="quat_s100_h3_p128", b=2, s=100, h=3, p=128, chunk_len=20,
                                   quat_blocks=20),
    WORKLOADS["halfsplit_s1024"].scaled(name="half_s72", b=3, s=72, h=2, chunk_len=8),
    WORKLOADS["ragged_s16384"].scaled(name="ragged_s136_h5", b=3, s=136, h=5, chunk_len=8),
    # p below 64: the kernels run 64 rows, the rows past p zero (padded initial state, no d_xhat
    # stores past p)
    WORKLOADS["large_s4096"].scaled(name="pairwise_p32", b=2, s=192, h=4, p=32, valid="fixed:170"),
    WORKLOADS["quat_s2048"].scaled(name="quat_p16_h3", b=1, s=128, h=3, p=16),
    WORKLOADS["halfsplit_s1024"].scaled(name="half_p48_s100", b=2, s=100, h=2, p=48, chunk_len=4),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_parity_small(w):
    inp = make_inputs(w)
    got = run_gpu(w, inp)
    check_against_oracle(w, inp, got, w.name)


@pytest.mark.parametrize("w", [SMALL[2], SMALL[3], SMALL[4]], ids=["quat", "large", "ragged"])
def test_parity_generic_path_bf16(w):
    """The SIMT path on bf16 inputs (forced), same bar."""
    inp = make_inputs(w)
    got = run_gpu(w, inp, force_generic=True)
    check_against_oracle(w, inp, got, w.name + "/generic")


@pytest.mark.parametrize("valid", [(0, 256), (256, 0), (1, 255), (64, 65), (1000, 129)])
def test_parity_valid_len_edges(valid):
    w = WORKLOADS["large_s4096"].scaled(name="edges", b=2, s=256, h=4, C=2)
    inp = make_inputs(w)
    inp["valid_len"] = torch.tensor(valid, dtype=torch.int64)
    got = run_gpu(w, inp)
    check_against_oracle(w, inp, got, f"edges{valid}")
    if valid[0] == 0:
        assert torch.count_nonzero(got["m2"][0]) == 0 and torch.count_nonzero(got["d_initial"][0]) == 0


@pytest.mark.parametrize("l", [1, 8, 256])
def test_parity_chunk_len_extremes(l):
    w = WORKLOADS["large_s4096"].scaled(name=f"l{l}", b=1, s=256, h=4, C=2, chunk_len=l, valid="fixed:250")
    inp = make_inputs(w)
    got = run_gpu(w, inp)
    check_against_oracle(w, inp, got, w.name)


def test_parity_steep_decay_spans():
    """Decays far outside the usual range: two heads with per-token log-decay near -25, single
    reset tokens (da = -70) in another, the last head unchanged, so the backward sees spans
    whose prefix decay factors around the span midpoint would leave the safe exponent range
    next to spans where they do not."""
    w = WORKLOADS["large_s4096"].scaled(name="steep", b=2, s=256, h=4, C=2, valid="fixed:250")
    inp = make_inputs(w)
    da = inp["da"].clone()
    da[:, :, 0:2] *= 50.0
    da[:, 37, 2] = -70.0
    da[:, 101, 2] = -70.0
    da[1, 200:204, 2] = -35.0
    inp["da"] = da.contiguous()
    got = run_gpu(w, inp)
    check_against_oracle(w, inp, got, w.name)


@pytest.mark.parametrize("w", [SMALL[3], SMALL[0],
                               WORKLOADS["large_s4096"].scaled(name="tc_c6", b=1, s=128, h=4, C=6),
                               WORKLOADS["large_s4096"].scaled(name="tc_p128", b=2, s=192, h=2, p=128,
                                                               valid="fixed:130"),
                               WORKLOADS["large_s4096"].scaled(name="tc_p24", b=2, s=192, h=2, p=24,
                                                               valid="fixed:130")],
                         ids=["tensor_core", "simt", "tensor_core_c6", "tensor_core_p128", "tensor_core_p24"])
def test_backward_reusing_forward_carries(w):
    """MM_FLAG_REUSE_CARRIES: forward then backward on one workspace gives the gradients of a
    backward that recomputes the carries (on the tensor-core path with four and six channels, and on
    the SIMT path)."""
    inp = make_inputs(w)
    d = {k: v.to(DEV) for k, v in inp.items() if k != "valid_len"}
    spec = spec_of(w)
    rot = d["rot"] if d["rot"].numel() else None
    args = (spec, d["xhat"], d["bhat"], d["da"], rot, d["initial"], inp["valid_len"])
    ref = binding.moments_bwd(*args, d["d_m2"], d["d_m1"])
    ws = binding.alloc_workspace(spec, True, torch.device(DEV))
    m2, m1 = binding.moments_fwd(*args, workspace=ws)
    got = binding.moments_bwd(*args, d["d_m2"], d["d_m1"], workspace=ws, reuse_carries=True)
    torch.cuda.synchronize()
    for k in GRADS:
        if ref[k] is None:
            continue
        a_, b_ = got[k].float().cpu(), ref[k].float().cpu()
        assert torch.allclose(a_, b_, rtol=1e-5, atol=1e-6 * max(1.0, float(b_.abs().max()))), k
    out = dict(m2=m2.cpu(), m1=m1.cpu())
    for k in GRADS:
        out[k] = got[k].cpu() if got[k] is not None else torch.zeros(0)
    check_against_oracle(w, inp, out, w.name + "/reuse")


def full_size_pairs(w):
    """(batch row, head) pairs the oracle checks at full size: every pair of the quaternion
    workload; eight distinct pairs of the others, the first and the last among them and, for
    the ragged workload, pairs from every batch row (each row ends at its own valid length)."""
    if w.name == "quat_s2048":
        return [(bb, hh) for bb in range(w.b) for hh in range(w.h)]
    rng = np.random.default_rng(1234)
    pairs = {(0, 0), (w.b - 1, w.h - 1)}
    for bb in range(w.b):  # at least one pair per batch row where there are few rows
        if len(pairs) < 8 and w.b <= 4:
            pairs.add((bb, int(rng.integers(w.h))))
    while len(pairs) < 8:
        pairs.add((int(rng.integers(w.b)), int(rng.integers(w.h))))
    return sorted(pairs)


FULL = ["quat_s2048", "large_s4096", "ragged_s16384"]


@pytest.mark.parametrize("name", FULL)
def test_parity_full_size_sampled(name):
    """Full-size workloads in the bench's launch configuration; the oracle checks the pairs of
    `full_size_pairs` one by one (each pair is an independent problem), over the whole sequence,
    so the ragged rows' last valid chunks and their zero tails are compared too."""
    w = WORKLOADS[name]
    inp = make_inputs(w)
    got = run_gpu(w, inp)
    pairs = full_size_pairs(w)
    assert len(set(pairs)) == len(pairs) and len(pairs) >= min(8, w.b * w.h)
    subs = [slice_bh(inp, bb, hh) for bb, hh in pairs]
    stacked = {k: torch.cat([s[k] for s in subs], dim=0) for k in subs[0]}
    ws = w.scaled(b=len(pairs), h=1)
    m2, m1 = oracle_fwd(ws, stacked)
    ref = oracle_bwd(ws, stacked)
    ref.update(m2=m2, m1=m1)
    tol = tolerance(w)
    for i, (bb, hh) in enumerate(pairs):
        mine = dict(m2=got["m2"][bb, hh], m1=got["m1"][bb, hh], d_xhat=got["d_xhat"][bb, :, :, hh],
                    d_bhat=got["d_bhat"][bb, :, :, hh], d_da=got["d_da"][bb, :, hh],
                    d_rot=got["d_rot"][bb, :, hh], d_initial=got["d_initial"][bb, hh])
        theirs = dict(m2=ref["m2"][i, 0], m1=ref["m1"][i, 0], d_xhat=ref["d_xhat"][i, :, :, 0],
                      d_bhat=ref["d_bhat"][i, :, :, 0], d_da=ref["d_da"][i, :, 0],
                      d_rot=ref["d_rot"][i, :, 0], d_initial=ref["d_initial"][i, 0])
        compare(f"{name}/b{bb}h{hh}", tol, [(k, mine[k], theirs[k]) for k in theirs])
        v = int(min(inp["valid_len"][bb], w.s))
        for k in ("d_xhat", "d_bhat", "d_da", "d_rot"):
            if v < w.s:
                assert torch.count_nonzero(mine[k][v:]) == 0, (name, k)


def test_autograd_function_matches_direct_calls():
    w = SMALL[3]
    inp = make_inputs(w)
    d = {k: v.to(DEV) for k, v in inp.items() if k != "valid_len"}
    leaves = {k: d[k].clone().float().requires_grad_(True) if k in ("da", "rot", "initial")
              else d[k].clone().requires_grad_(True) for k in ("xhat", "bhat", "da", "rot", "initial")}
    m2, m1 = binding.moments(leaves["xhat"], leaves["bhat"], leaves["da"], leaves["rot"], leaves["initial"],
                             inp["valid_len"], w.chunk_len, w.rot, w.rope_dim, w.quat_blocks)
    (m2 * d["d_m2"]).sum().add((m1 * d["d_m1"]).sum()).backward()
    direct = run_gpu(w, inp)
    assert torch.allclose(m2.detach().cpu(), direct["m2"], rtol=1e-5, atol=1e-5)
    for k in ("xhat", "bhat", "da", "rot", "initial"):
        a = leaves[k].grad.float().cpu()
        b = direct["d_" + k].float()
        assert torch.allclose(a, b, rtol=1e-5, atol=1e-5), k
