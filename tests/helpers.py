"""Shared test helpers: the oracle on torch inputs, and the normwise error metric."""
import numpy as np
import torch

import oracle

GRADS = ("d_xhat", "d_bhat", "d_da", "d_rot", "d_initial")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_fwd(w, inp, bh_range=None):
    return oracle.moments_fwd(f64(inp["xhat"]), f64(inp["bhat"]), f64(inp["da"]), f64(inp["rot"]),
                              f64(inp["initial"]), inp["valid_len"].numpy(), rot_kind=w.rot,
                              rope_dim=w.rope_dim, quat_blocks=w.quat_blocks, bh_range=bh_range)


def oracle_bwd(w, inp, bh_range=None):
    return oracle.moments_bwd(f64(inp["xhat"]), f64(inp["bhat"]), f64(inp["da"]), f64(inp["rot"]),
                              f64(inp["initial"]), inp["valid_len"].numpy(), f64(inp["d_m2"]),
                              f64(inp["d_m1"]), rot_kind=w.rot, rope_dim=w.rope_dim,
                              quat_blocks=w.quat_blocks, bh_range=bh_range)


def rel_err(got, ref):
    """Normwise relative error ||got - ref||_F / ||ref||_F (0/0 -> 0)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)


def tolerance(w):
    """fp32 inputs: 1e-4; bf16 inputs: 2e-2 (normwise, per output tensor)."""
    return 1e-4 if w.dtype == "f32" else 2e-2
