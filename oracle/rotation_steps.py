"""fp64 CPU oracle: the per-token cumulative rotation built from per-token steps, and the
vector-Jacobian product of that build.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` -- never by the product package, which shares no code with it.

The operator takes the *cumulative* rotation of every token ("mamba3/moments/recalculated.rs",
``RotPrim``: cumulative angles ``[b, s, h, a]`` or cumulative unit quaternions ``[b, s, h, J, 4]``).
The producer that builds it (``RotationSeq``, ``rotation::quat_mul``) is named there but not given
on the pages.  Reading adopted (the plainest one the names support):

* complex kinds: ``theta[b, t, h, i] = sum_{u <= t} dtheta[b, u, h, i]`` -- an inclusive prefix sum
  of per-token angle steps along the sequence, per batch row, head and angle;
* quaternions: ``Q[b, t, h, j] = q[b, t, h, j] (x) Q[b, t-1, h, j]`` with ``Q[b, -1] = 1`` -- each
  token's step applied after the rotation accumulated so far, ``(x)`` the Hamilton product of
  ``quat_mul_prim`` on the packed ``(w, x, y, z)`` axis.

Positions past ``valid_len`` are included in the build; they never reach an output of the
operator, so their steps get exactly zero gradient.

Gradients, by plain reverse mode of the two definitions:

* complex: ``d_dtheta[u] = sum_{t >= u} d_theta[t]``;
* quaternions: with ``G_t`` the total cotangent of ``Q_t``,
  ``G_t = dQ_t + conj(q_{t+1}) (x) G_{t+1}`` (``G`` past the end is 0) and
  ``d_q_t = G_t (x) conj(Q_{t-1})``: ``Q_t`` is linear in ``q_t`` through right multiplication by
  ``Q_{t-1}`` and in ``Q_{t-1}`` through left multiplication by ``q_t``, whose transposes are the
  multiplications by the conjugates.
"""
from __future__ import annotations

import numpy as np


def qmul(a, b):
    """Hamilton product a (x) b on the trailing (w, x, y, z) axis ("recalculated.rs",
    ``quat_mul_prim``)."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    aw, ax, ay, az = a[..., 0], a[..., 1], a[..., 2], a[..., 3]
    bw, bx, by, bz = b[..., 0], b[..., 1], b[..., 2], b[..., 3]
    return np.stack([aw * bw - ax * bx - ay * by - az * bz,
                     aw * bx + ax * bw + ay * bz - az * by,
                     aw * by - ax * bz + ay * bw + az * bx,
                     aw * bz + ax * by - ay * bx + az * bw], axis=-1)


def qconj(q):
    """Quaternion conjugate (w, -x, -y, -z) ("recalculated.rs", ``quat_conj_prim``)."""
    q = np.asarray(q, dtype=np.float64)
    return q * np.array([1.0, -1.0, -1.0, -1.0])


def cum_angles(dtheta):
    """Cumulative angles of per-token angle steps ``[b, s, h, a]`` (sequence axis 1)."""
    return np.cumsum(np.asarray(dtheta, dtype=np.float64), axis=1)


def cum_angles_vjp(d_theta):
    """Gradient w.r.t. the angle steps given the gradient w.r.t. the cumulative angles: the sum
    over every later-or-equal token."""
    g = np.asarray(d_theta, dtype=np.float64)
    return np.flip(np.cumsum(np.flip(g, axis=1), axis=1), axis=1)


def cum_quats(q):
    """Cumulative quaternions of per-token quaternion steps ``[b, s, h, J, 4]``: token by token,
    ``Q_t = q_t (x) Q_{t-1}`` from the identity."""
    q = np.asarray(q, dtype=np.float64)
    out = np.empty_like(q)
    prev = np.zeros(q.shape[:1] + q.shape[2:], dtype=np.float64)
    prev[..., 0] = 1.0
    for t in range(q.shape[1]):
        prev = qmul(q[:, t], prev)
        out[:, t] = prev
    return out


def cum_quats_vjp(q, dQ):
    """Gradient w.r.t. the quaternion steps ``q`` given ``dQ``, the gradient w.r.t. the
    cumulative quaternions; walks the tokens in reverse, carrying the cotangent of ``Q_t``."""
    q = np.asarray(q, dtype=np.float64)
    dQ = np.asarray(dQ, dtype=np.float64)
    Q = cum_quats(q)
    s = q.shape[1]
    dq = np.empty_like(q)
    G = np.zeros(q.shape[:1] + q.shape[2:], dtype=np.float64)
    one = np.zeros_like(G)
    one[..., 0] = 1.0
    for t in range(s - 1, -1, -1):
        G = dQ[:, t] + (qmul(qconj(q[:, t + 1]), G) if t + 1 < s else 0.0)
        prev = Q[:, t - 1] if t > 0 else one
        dq[:, t] = qmul(G, qconj(prev))
    return dq


def build(rot_steps, rot_kind):
    """The cumulative rotation the operator consumes, from the steps of ``rot_kind``."""
    if rot_kind == "quat":
        return cum_quats(rot_steps)
    if rot_kind in ("pairwise", "half"):
        return cum_angles(rot_steps)
    return np.asarray(rot_steps, dtype=np.float64)


def build_vjp(rot_steps, d_cum, rot_kind):
    """Gradient w.r.t. the steps, given the operator's gradient w.r.t. the cumulative rotation."""
    if rot_kind == "quat":
        return cum_quats_vjp(rot_steps, d_cum)
    if rot_kind in ("pairwise", "half"):
        return cum_angles_vjp(d_cum)
    return np.asarray(d_cum, dtype=np.float64)
