"""Seeded synthetic inputs for the state-moments operator.

This module only draws random numbers and lays them out; it holds none of the
operator's arithmetic, and it is the one module the CUDA path's tests and the CPU
oracle share.  Every draw comes from a ``torch.Generator('cpu')`` seeded per workload,
in the fixed order of :func:`make_inputs`, so the GPU path and the oracle see the
identical values (bf16 operands are drawn in fp32 and rounded once; the oracle reads
the rounded values, which convert to fp64 exactly).

Workloads (shapes from the five seeded configurations the operator is measured on):

=====================  ====  =====  ==  ==  ==  ===  ===  =========================  =====
name                   b     s      C   h   p   r    l    rotation                   dtype
=====================  ====  =====  ==  ==  ==  ===  ===  =========================  =====
tiny_fp32              1     64     1   2   8   16   16   pairwise, rope_dim 8       f32
halfsplit_s1024        2     1024   2   8   64  64   64   half-split, rope_dim 32    bf16
quat_s2048             4     2048   1   16  64  128  64   quaternion, 32 blocks      bf16
large_s4096            8     4096   4   32  64  128  64   pairwise, rope_dim 64      bf16
ragged_s16384          2     16384  2   16  64  128  128  half-split, rope_dim 128   bf16
=====================  ====  =====  ==  ==  ==  ===  ===  =========================  =====
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    s: int
    C: int
    h: int
    p: int
    r: int
    chunk_len: int
    rot: str                 # "none" | "pairwise" | "half" | "quat"
    rope_dim: int = 0        # complex kinds: rotated width (angles per token = rope_dim // 2)
    quat_blocks: int = 0     # quaternion kind: number of 4-blocks
    dtype: str = "bf16"      # dtype of xhat / bhat
    valid: str = "full"      # "full" | "fixed:<n>" | "ragged" (U[s/2, s] per batch row)
    xb_scale: str = "rsqrt_r"  # "unit": N(0,1); "rsqrt_r": N(0,1)/sqrt(r)
    da_kind: str = "softplus_m1"  # "softplus_half": -softplus(N(0,1))*0.5 ; "softplus_m1": -softplus(N(-1,1))
    init_std: float = 0.1
    seed: int = 0

    @property
    def n_angles(self) -> int:
        return self.rope_dim // 2 if self.rot in ("pairwise", "half") else 0

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_fp32", 1, 64, 1, 2, 8, 16, 16, "pairwise", rope_dim=8, dtype="f32",
                 valid="fixed:60", xb_scale="unit", da_kind="softplus_half", init_std=1.0, seed=0),
        Workload("halfsplit_s1024", 2, 1024, 2, 8, 64, 64, 64, "half", rope_dim=32, seed=1),
        Workload("quat_s2048", 4, 2048, 1, 16, 64, 128, 64, "quat", quat_blocks=32, seed=2),
        Workload("large_s4096", 8, 4096, 4, 32, 64, 128, 64, "pairwise", rope_dim=64, seed=3),
        Workload("ragged_s16384", 2, 16384, 2, 16, 64, 128, 128, "half", rope_dim=128,
                 valid="ragged", seed=4),
    ]
}

QUAT_STEP_STD = 0.05  # per-component std of the quaternion random-walk step


def _valid_lengths(w: Workload, g: torch.Generator) -> torch.Tensor:
    if w.valid == "full":
        return torch.full((w.b,), w.s, dtype=torch.int64)
    if w.valid.startswith("fixed:"):
        return torch.full((w.b,), int(w.valid.split(":")[1]), dtype=torch.int64)
    if w.valid == "ragged":
        return torch.randint(w.s // 2, w.s + 1, (w.b,), generator=g, dtype=torch.int64)
    raise ValueError(w.valid)


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw every input of one forward + backward call, on the CPU.

    Returns a dict of CPU tensors: xhat [b,s,C,h,p], bhat [b,s,C,h,r] (in the workload's
    dtype), da [b,s,h] f32, rot ([b,s,h,rope_dim/2] angles or [b,s,h,J,4] quaternions,
    f32), initial [b,h,p,r] f32, valid_len [b] int64, d_m2 [b,h,r,r] f32, d_m1 [b,h,r] f32.
    """
    g = torch.Generator("cpu")
    g.manual_seed(w.seed if seed is None else seed)
    b, s, C, h, p, r = w.b, w.s, w.C, w.h, w.p, w.r
    xdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    xs = 1.0 if w.xb_scale == "unit" else r ** -0.5
    xhat = (torch.randn((b, s, C, h, p), generator=g) * xs).to(xdt)
    bhat = (torch.randn((b, s, C, h, r), generator=g) * xs).to(xdt)
    if w.da_kind == "softplus_half":
        da = -torch.nn.functional.softplus(torch.randn((b, s, h), generator=g)) * 0.5
    else:
        da = -torch.nn.functional.softplus(torch.randn((b, s, h), generator=g) - 1.0)
    if w.rot in ("pairwise", "half"):
        steps = torch.rand((b, s, h, w.n_angles), generator=g) * 0.6 - 0.3
        rot = torch.cumsum(steps, dim=1)
    elif w.rot == "quat":
        rot = _quat_walk(b, s, h, w.quat_blocks, g)
    else:
        rot = torch.zeros((b, s, h, 0))
    initial = torch.randn((b, h, p, r), generator=g) * w.init_std
    valid_len = _valid_lengths(w, g)
    d_m2 = torch.randn((b, h, r, r), generator=g)
    d_m1 = torch.randn((b, h, r), generator=g)
    return dict(xhat=xhat.contiguous(), bhat=bhat.contiguous(), da=da.contiguous(),
                rot=rot.to(torch.float32).contiguous(), initial=initial.contiguous(),
                valid_len=valid_len, d_m2=d_m2.contiguous(), d_m1=d_m1.contiguous())


def _quat_walk(b, s, h, J, g):
    """Cumulative unit quaternions as a normalised random walk on the 3-sphere.

    q_{-1} = (1,0,0,0); q_t = normalise(q_{t-1} + 0.05 * N(0,1)^4).  Each step turns
    the block by a small angle (about 0.17 rad on average), the same scale as the
    complex workloads' angle increments.  Drawn and normalised in fp64, stored fp32.
    """
    steps = torch.randn((b, s, h, J, 4), generator=g, dtype=torch.float64) * QUAT_STEP_STD
    out = torch.empty((b, s, h, J, 4), dtype=torch.float64)
    q = torch.zeros((b, h, J, 4), dtype=torch.float64)
    q[..., 0] = 1.0
    for t in range(s):
        q = q + steps[:, t]
        q = q / q.norm(dim=-1, keepdim=True)
        out[:, t] = q
    return out.to(torch.float32)


def make_rot_steps(w: Workload) -> torch.Tensor:
    """Per-token rotation steps for calls made with the rotation given as steps: angle steps
    [b,s,h,rope_dim/2] ~ U(-0.3, 0.3) (the distribution the cumulative angles above are summed
    from), or per-token unit quaternions [b,s,h,J,4] = normalise((1,0,0,0) + 0.05 N(0,1)^4),
    drawn and normalised in fp64 and stored fp32.  A generator of its own (seed + 1000), so the
    other inputs of the workload do not change."""
    g = torch.Generator("cpu")
    g.manual_seed(w.seed + 1000)
    b, s, h = w.b, w.s, w.h
    if w.rot in ("pairwise", "half"):
        return (torch.rand((b, s, h, w.n_angles), generator=g) * 0.6 - 0.3).contiguous()
    if w.rot == "quat":
        q = torch.randn((b, s, h, w.quat_blocks, 4), generator=g, dtype=torch.float64) * QUAT_STEP_STD
        q[..., 0] += 1.0
        return (q / q.norm(dim=-1, keepdim=True)).to(torch.float32).contiguous()
    return torch.zeros((b, s, h, 0))


def slice_bh(inp: dict, bsel: int, hsel: int) -> dict:
    """The inputs of one (batch row, head) pair as a b=1, h=1 problem."""
    out = {}
    for k, v in inp.items():
        if k in ("xhat", "bhat"):
            out[k] = v[bsel:bsel + 1, :, :, hsel:hsel + 1]
        elif k in ("da", "rot"):
            out[k] = v[bsel:bsel + 1, :, hsel:hsel + 1]
        elif k in ("initial", "d_m2", "d_m1"):
            out[k] = v[bsel:bsel + 1, hsel:hsel + 1]
        elif k == "valid_len":
            out[k] = v[bsel:bsel + 1]
    return {k: v.contiguous() for k, v in out.items()}
