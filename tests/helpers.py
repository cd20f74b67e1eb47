"""Shared test helpers: the oracle on torch inputs, the error metrics, and the parity report."""
import json
import os

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


def max_rel_err(got, ref):
    """Element-wise error against the tensor's scale: max |got - ref| / max |ref| (0/0 -> 0).

    Unlike the normwise figure, one wrong element (an angle, a chunk-boundary d_da) cannot hide
    behind the rest of the tensor: it shows at its own size relative to the largest value."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    den = float(np.max(np.abs(ref)))
    num = float(np.max(np.abs(got - ref)))
    if den == 0.0:
        return num
    return num / den


def tolerance(w):
    """fp32 inputs: 1e-4; bf16 inputs: 2e-2 -- both normwise and element-wise (max-abs error over
    the tensor's max |value|), per output tensor."""
    return 1e-4 if w.dtype == "f32" else 2e-2


def report(label, errs):
    """Append one line of per-tensor errors to the file named by $PARITY_REPORT, if set."""
    path = os.environ.get("PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": label, "errors": errs}) + "\n")


def compare(label, tol, pairs):
    """Check every (name, got, ref) pair normwise and element-wise against `tol`; returns
    {name: {"norm": e, "max": e}} and asserts with the full table on failure."""
    errs = {}
    for name, got, ref in pairs:
        ref = np.asarray(ref, dtype=np.float64)
        if ref.size == 0:
            continue
        g = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
        assert g.shape == ref.shape, (label, name, g.shape, ref.shape)
        assert np.all(np.isfinite(g)), (label, name, "non-finite values")
        errs[name] = {"norm": rel_err(g, ref), "max": max_rel_err(g, ref)}
    report(label, errs)
    bad = {k: v for k, v in errs.items() if not (v["norm"] <= tol and v["max"] <= tol)}
    assert not bad, f"{label}: errors above {tol}: {bad} (all: {errs})"
    return errs
