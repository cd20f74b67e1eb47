"""Pins of the oracle's cumulative-rotation build (``oracle/rotation_steps.py``) against things it
does not compute itself: brute-force sums, closed forms, the adjoint identity, the golden Hamilton
table, the planar case that reduces quaternions to angles, and central finite differences, both of
the build alone and of the whole operator fed with steps.  CPU only."""
import os

import numpy as np
import pytest

import oracle
from oracle import rotation_steps as rs

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_angle_steps_brute_force_and_closed_form():
    rng = np.random.default_rng(3)
    d = rng.uniform(-0.3, 0.3, size=(2, 7, 3, 4))
    th = rs.cum_angles(d)
    for b in range(2):
        for t in range(7):
            for h in range(3):
                for i in range(4):
                    assert th[b, t, h, i] == pytest.approx(sum(d[b, u, h, i] for u in range(t + 1)), abs=1e-15)
    const = np.full((1, 9, 1, 2), 0.25)
    assert np.array_equal(rs.cum_angles(const)[0, :, 0, 0], 0.25 * np.arange(1, 10))


def test_angle_steps_vjp_is_the_adjoint():
    """<build(d), g> == <d, vjp(g)> for every d, g: the gradient of a linear map is its transpose."""
    rng = np.random.default_rng(4)
    d = rng.normal(size=(2, 11, 2, 3))
    g = rng.normal(size=(2, 11, 2, 3))
    assert np.sum(rs.cum_angles(d) * g) == pytest.approx(np.sum(d * rs.cum_angles_vjp(g)), rel=1e-13)
    # the last step only moves the last angle; the first moves all of them
    e = np.zeros((1, 5, 1, 1))
    e[0, :, 0, 0] = 1.0
    assert np.array_equal(rs.cum_angles_vjp(e)[0, :, 0, 0], np.array([5.0, 4.0, 3.0, 2.0, 1.0]))


def test_qmul_matches_golden_hamilton_table():
    basis = {"1": [1, 0, 0, 0], "i": [0, 1, 0, 0], "j": [0, 0, 1, 0], "k": [0, 0, 0, 1]}
    rows = [l.split() for l in open(os.path.join(GOLD, "quaternion_basis.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for row in rows:
        got = rs.qmul(np.array(basis[row[0]], float), np.array(basis[row[1]], float))
        assert np.array_equal(got, np.array([float(v) for v in row[2:]])), row


def test_quaternion_steps_in_one_plane_reduce_to_angle_steps():
    """Steps (cos phi, 0, 0, -sin phi) commute; their running product is (cos theta, 0, 0,
    -sin theta) with theta the running sum of phi."""
    rng = np.random.default_rng(5)
    phi = rng.uniform(-0.3, 0.3, size=(2, 9, 3, 2))
    q = np.stack([np.cos(phi), np.zeros_like(phi), np.zeros_like(phi), -np.sin(phi)], axis=-1)
    Q = rs.cum_quats(q)
    th = np.cumsum(phi, axis=1)
    ref = np.stack([np.cos(th), np.zeros_like(th), np.zeros_like(th), -np.sin(th)], axis=-1)
    assert np.allclose(Q, ref, atol=1e-14)


def test_quaternion_step_order():
    """The reading: each step applies after the accumulated rotation, Q_t = q_t (x) Q_{t-1};
    with steps i then j the product is j i = -k (not i j = k)."""
    q = np.zeros((1, 2, 1, 1, 4))
    q[0, 0, 0, 0] = [0, 1, 0, 0]
    q[0, 1, 0, 0] = [0, 0, 1, 0]
    Q = rs.cum_quats(q)
    assert np.array_equal(Q[0, 0, 0, 0], [0, 1, 0, 0])
    assert np.array_equal(Q[0, 1, 0, 0], [0, 0, 0, -1])


def test_quaternion_steps_keep_unit_norm():
    rng = np.random.default_rng(6)
    q = rng.normal(size=(2, 50, 2, 3, 4))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    assert np.allclose(np.linalg.norm(rs.cum_quats(q), axis=-1), 1.0, atol=1e-13)


def test_quaternion_steps_vjp_finite_differences():
    """L = sum_t <W_t, Q_t> with random W; non-unit steps (the build is a plain product)."""
    rng = np.random.default_rng(7)
    q = rng.normal(size=(1, 5, 1, 2, 4))
    W = rng.normal(size=q.shape)
    ana = rs.cum_quats_vjp(q, W)
    eps = 1e-6
    num = np.zeros_like(q)
    it = np.nditer(q, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        p, m = q.copy(), q.copy()
        p[idx] += eps
        m[idx] -= eps
        num[idx] = (np.sum(W * rs.cum_quats(p)) - np.sum(W * rs.cum_quats(m))) / (2 * eps)
    assert np.abs(ana - num).max() <= 1e-8 * max(1.0, np.abs(num).max())


@pytest.mark.parametrize("kind,rope,J", [("pairwise", 4, 0), ("half", 4, 0), ("quat", 0, 2)])
def test_operator_fed_with_steps_finite_differences(kind, rope, J):
    """The whole operator with the rotation given as steps: the gradient w.r.t. the steps (the
    oracle's d_rot through the build's VJP) against central differences of <d_m2, m2> + <d_m1, m1>,
    valid_len < s on one row."""
    rng = np.random.default_rng(8 + J)
    b, s, C, h, p, r = 2, 6, 1, 1, 2, 8
    xhat, bhat = rng.normal(size=(b, s, C, h, p)), rng.normal(size=(b, s, C, h, r))
    da = -np.abs(rng.normal(size=(b, s, h))) * 0.5
    initial = rng.normal(size=(b, h, p, r))
    valid = np.array([s, s - 2])
    d_m2, d_m1 = rng.normal(size=(b, h, r, r)), rng.normal(size=(b, h, r))
    if kind == "quat":
        steps = rng.normal(size=(b, s, h, J, 4))
    else:
        steps = rng.uniform(-0.5, 0.5, size=(b, s, h, rope // 2))
    kw = dict(rot_kind=kind, rope_dim=rope, quat_blocks=J)

    def loss(st):
        m2, m1 = oracle.moments_fwd(xhat, bhat, da, rs.build(st, kind), initial, valid, **kw)
        return float(np.sum(d_m2 * m2) + np.sum(d_m1 * m1))

    g = oracle.moments_bwd(xhat, bhat, da, rs.build(steps, kind), initial, valid, d_m2, d_m1, **kw)
    ana = rs.build_vjp(steps, g["d_rot"], kind)
    eps = 1e-6
    num = np.zeros_like(steps)
    it = np.nditer(steps, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        pl, mi = steps.copy(), steps.copy()
        pl[idx] += eps
        mi[idx] -= eps
        num[idx] = (loss(pl) - loss(mi)) / (2 * eps)
    scale = max(1.0, np.abs(num).max())
    assert np.abs(ana - num).max() <= 2e-6 * scale, (np.abs(ana - num).max(), scale)
    # steps past valid_len on the short row get exactly zero gradient
    assert np.count_nonzero(ana[1, valid[1]:]) == 0
