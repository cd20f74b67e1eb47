"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle (token-level C, ``oracle/moments_oracle.c``) against a fact the
source pages or the mathematics fix: central finite differences, an exact computer-algebra
derivative on a tiny case, a brute-force closed form of the recurrence, the pages' own
chunked algorithm restated independently (``oracle/chunked_ref.py``), rotation identities
and permutations, symmetry / scaling laws, masking invariants, and the golden tables under
``tests/golden/``.  A dropped term, wrong sign, wrong index or transposed operand in the
oracle fails at least one of them.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import chunked_ref

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
KINDS = [("pairwise", 6, 0), ("half", 6, 0), ("quat", 0, 1), ("quat", 0, 2), ("none", 0, 0)]


def rand_problem(rng, b=2, s=7, C=2, h=2, p=3, r=8, kind="pairwise", rope_dim=6, J=0,
                 valid=(5, 7), unit_quat=False, da_scale=0.5):
    xhat = rng.standard_normal((b, s, C, h, p))
    bhat = rng.standard_normal((b, s, C, h, r))
    da = -np.log1p(np.exp(rng.standard_normal((b, s, h)))) * da_scale
    if kind in ("pairwise", "half"):
        rot = np.cumsum(rng.uniform(-0.6, 0.6, (b, s, h, rope_dim // 2)), axis=1)
    elif kind == "quat":
        rot = rng.standard_normal((b, s, h, J, 4))
        if unit_quat:
            rot /= np.linalg.norm(rot, axis=-1, keepdims=True)
    else:
        rot = np.zeros((b, s, h, 0))
    initial = rng.standard_normal((b, h, p, r))
    d_m2 = rng.standard_normal((b, h, r, r))
    d_m1 = rng.standard_normal((b, h, r))
    return dict(xhat=xhat, bhat=bhat, da=da, rot=rot, initial=initial,
                valid_len=np.array(valid, dtype=np.int64), d_m2=d_m2, d_m1=d_m1,
                kind=kind, rope_dim=rope_dim, J=J)


def fwd(P, **over):
    q = dict(P, **over)
    return oracle.moments_fwd(q["xhat"], q["bhat"], q["da"], q["rot"], q["initial"], q["valid_len"],
                              rot_kind=q["kind"], rope_dim=q["rope_dim"], quat_blocks=q["J"])


def bwd(P, **over):
    q = dict(P, **over)
    return oracle.moments_bwd(q["xhat"], q["bhat"], q["da"], q["rot"], q["initial"], q["valid_len"],
                              q["d_m2"], q["d_m1"], rot_kind=q["kind"], rope_dim=q["rope_dim"],
                              quat_blocks=q["J"])


def loss(P, **over):
    q = dict(P, **over)
    m2, m1 = fwd(q)
    return float(np.sum(q["d_m2"] * m2) + np.sum(q["d_m1"] * m1))


# --------------------------------------------------------------- finite differences
@pytest.mark.parametrize("kind,rope,J", KINDS)
def test_central_finite_differences(kind, rope, J):
    """All five gradients vs central differences (fp64, step 1e-6), valid_len < s on one row.
    Quaternions are left non-unit: the pages state the quaternion VJP is exact for all."""
    rng = np.random.default_rng(11 + rope + J)
    P = rand_problem(rng, kind=kind, rope_dim=rope, J=J)
    G = bwd(P)
    eps = 1e-6
    names = ["xhat", "bhat", "da", "initial"] + (["rot"] if P["rot"].size else [])
    for name in names:
        base = P[name]
        num = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus, minus = base.copy(), base.copy()
            plus[idx] += eps
            minus[idx] -= eps
            num[idx] = (loss(P, **{name: plus}) - loss(P, **{name: minus})) / (2 * eps)
        ana = G["d_" + name]
        scale = max(1.0, np.abs(num).max())
        assert np.abs(ana - num).max() <= 2e-6 * scale, (name, np.abs(ana - num).max(), scale)


# --------------------------------------------------------- exact symbolic derivative
def test_sympy_exact_two_tokens():
    """s=2, C=1, p=1 with r=4: forward and every gradient from computer algebra (exact
    differentiation of the loss written out by hand), complex-pairwise and quaternion."""
    sp = pytest.importorskip("sympy")
    rng = np.random.default_rng(5)
    for kind in ("pairwise", "half", "quat"):
        r = 4
        x = sp.symbols("x0:2")
        bb = sp.symbols("b0:8")
        a = sp.symbols("a0:2")
        h0 = sp.symbols("h0:4")
        if kind == "quat":
            th = sp.symbols("q0:8")
        else:
            th = sp.symbols("t0:2")   # one angle per token (rope_dim = 2)
        Dm = sp.Matrix(4, 4, list(sp.symbols("D0:16")))
        dm1 = sp.Matrix(1, 4, list(sp.symbols("e0:4")))

        def derot(v, t):
            v = list(v)
            if kind == "quat":
                Q = th[4 * t:4 * t + 4]
                w, xx, yy, zz = v
                return [Q[0] * w - Q[1] * xx - Q[2] * yy - Q[3] * zz,
                        Q[0] * xx + Q[1] * w + Q[2] * zz - Q[3] * yy,
                        Q[0] * yy - Q[1] * zz + Q[2] * w + Q[3] * xx,
                        Q[0] * zz + Q[1] * yy - Q[2] * xx + Q[3] * w]
            ix, iy = (0, 1) if kind == "pairwise" else (0, 2)
            c, s_ = sp.cos(th[t]), sp.sin(th[t])
            out = list(v)
            out[ix] = c * v[ix] + s_ * v[iy]
            out[iy] = -s_ * v[ix] + c * v[iy]
            return out

        hstate = list(h0)
        L = 0
        for t in range(2):
            hstate = [sp.exp(a[t]) * hstate[j] + x[t] * bb[4 * t + j] for j in range(4)]
            c = sp.Matrix(1, 4, derot(hstate, t))
            L += (c * Dm * c.T)[0, 0] + (dm1 * c.T)[0, 0]
        vals = {}
        xv, bv, av, hv = rng.standard_normal(2), rng.standard_normal(8), -rng.random(2), rng.standard_normal(4)
        thv = rng.standard_normal(8) if kind == "quat" else rng.uniform(-1, 1, 2)
        Dv, ev = rng.standard_normal(16), rng.standard_normal(4)
        for syms, v in ((x, xv), (bb, bv), (a, av), (h0, hv), (th, thv), (Dm, Dv), (dm1, ev)):
            for sym, val in zip(list(syms), v):
                vals[sym] = float(val)
        P = dict(xhat=xv.reshape(1, 2, 1, 1, 1), bhat=bv.reshape(1, 2, 1, 1, 4), da=av.reshape(1, 2, 1),
                 rot=thv.reshape(1, 2, 1, 1, 4) if kind == "quat" else thv.reshape(1, 2, 1, 1),
                 initial=hv.reshape(1, 1, 1, 4), valid_len=np.array([2]), d_m2=Dv.reshape(1, 1, 4, 4),
                 d_m1=ev.reshape(1, 1, 4), kind=kind, rope_dim=0 if kind == "quat" else 2,
                 J=1 if kind == "quat" else 0)
        ref_loss = float(L.subs(vals))
        assert abs(loss(P) - ref_loss) <= 1e-12 * max(1, abs(ref_loss))
        G = bwd(P)
        checks = [("d_xhat", x, G["d_xhat"].ravel()), ("d_bhat", bb, G["d_bhat"].ravel()),
                  ("d_da", a, G["d_da"].ravel()), ("d_initial", h0, G["d_initial"].ravel()),
                  ("d_rot", th, G["d_rot"].ravel())]
        for name, syms, got in checks:
            exact = np.array([float(sp.diff(L, sym).subs(vals)) for sym in syms])
            assert np.allclose(got, exact, rtol=1e-11, atol=1e-11), (kind, name, got, exact)


# ----------------------------------------------- brute-force closed form of the recurrence
def closed_form_states(P):
    """h_t = exp(A_t) initial + sum_{j<=t} exp(A_t - A_j) W_j with A the cumulative da
    from the first token, written as an explicit double sum (no recurrence)."""
    xhat, bhat, da, init = P["xhat"], P["bhat"], P["da"], P["initial"]
    b, s, C, h, p = xhat.shape
    A = np.cumsum(da, axis=1)  # [b,s,h]
    W = np.einsum("btchp,btchr->bthpr", xhat, bhat)
    H = np.zeros((b, s, h, p, bhat.shape[-1]))
    for t in range(s):
        H[:, t] = np.exp(A[:, t])[..., None, None] * init
        for j in range(t + 1):
            H[:, t] += np.exp(A[:, t] - A[:, j])[..., None, None] * W[:, j]
    return H


@pytest.mark.parametrize("da_zero", [False, True])
def test_identity_rotation_equals_unrotated_closed_form(da_zero):
    """theta = 0, Q = 1 and rope_dim = 0 all reproduce the un-rotated moments, which are
    computed here from the closed form of the states (da = 0 gives plain prefix sums)."""
    rng = np.random.default_rng(3)
    P = rand_problem(rng, kind="none", rope_dim=0, valid=(5, 7))
    if da_zero:
        P["da"] = np.zeros_like(P["da"])
    H = closed_form_states(P)
    m2_ref = np.zeros((2, 2, 8, 8))
    m1_ref = np.zeros((2, 2, 8))
    for bb in range(2):
        T = P["valid_len"][bb]
        m2_ref[bb] = np.einsum("thpr,thps->hrs", H[bb, :T], H[bb, :T])
        m1_ref[bb] = H[bb, :T].sum(axis=(0, 2))
    for kind, rope, J, rot in [("none", 0, 0, np.zeros((2, 7, 2, 0))),
                               ("pairwise", 0, 0, np.zeros((2, 7, 2, 0))),
                               ("pairwise", 8, 0, np.zeros((2, 7, 2, 4))),
                               ("half", 8, 0, np.zeros((2, 7, 2, 4))),
                               ("quat", 0, 2, np.tile(np.array([1.0, 0, 0, 0]), (2, 7, 2, 2, 1)))]:
        m2, m1 = fwd(P, kind=kind, rope_dim=rope, J=J, rot=rot)
        assert np.allclose(m2, m2_ref, rtol=1e-12, atol=1e-12), kind
        assert np.allclose(m1, m1_ref, rtol=1e-12, atol=1e-12), kind


@pytest.mark.parametrize("kind,rope,J", [("pairwise", 8, 0), ("half", 8, 0), ("quat", 0, 2), ("pairwise", 4, 0)])
def test_norm_preservation(kind, rope, J):
    """trace(m2) = sum_{t,p} |h_t[p]|^2 is invariant to the angles and to unit quaternions."""
    rng = np.random.default_rng(4)
    P = rand_problem(rng, kind=kind, rope_dim=rope, J=J, unit_quat=True)
    m2, _ = fwd(P)
    zero_rot = np.zeros_like(P["rot"])
    if kind == "quat":
        zero_rot[..., 0] = 1.0
    m2_0, _ = fwd(P, rot=zero_rot)
    tr = np.trace(m2, axis1=2, axis2=3)
    assert np.allclose(tr, np.trace(m2_0, axis1=2, axis2=3), rtol=1e-12)
    assert not np.allclose(m2, m2_0)  # the rotation does act


@pytest.mark.parametrize("kind,rope,J", [("pairwise", 8, 0), ("half", 4, 0), ("quat", 0, 2)])
def test_single_token_closed_form(kind, rope, J):
    """s = 1: c_0 = derot_0(e^{da_0} initial + sum_c xhat (x) bhat) with the de-rotation
    written as an explicit r x r matrix (R(-theta) per pair; the Hamilton left-multiplication
    matrix of Q per block), m2 = c_0^T c_0 summed over p, m1 = column sums."""
    rng = np.random.default_rng(6)
    P = rand_problem(rng, b=1, s=1, C=3, h=1, p=4, r=8, kind=kind, rope_dim=rope, J=J, valid=(1,))
    h0 = np.exp(P["da"][0, 0, 0]) * P["initial"][0, 0] + np.einsum(
        "cp,cr->pr", P["xhat"][0, 0, :, 0], P["bhat"][0, 0, :, 0])
    R = np.eye(8)   # c_row = R @ h_row
    if kind in ("pairwise", "half"):
        for i in range(rope // 2):
            ix, iy = (2 * i, 2 * i + 1) if kind == "pairwise" else (i, i + 4)
            th = P["rot"][0, 0, 0, i]
            R[ix, ix], R[ix, iy], R[iy, ix], R[iy, iy] = np.cos(th), np.sin(th), -np.sin(th), np.cos(th)
    else:
        for k in range(J):
            w, x, y, z = P["rot"][0, 0, 0, k]
            R[4 * k:4 * k + 4, 4 * k:4 * k + 4] = [[w, -x, -y, -z], [x, w, -z, y], [y, z, w, -x], [z, -y, x, w]]
    c = h0 @ R.T
    m2, m1 = fwd(P)
    assert np.allclose(m2[0, 0], c.T @ c, rtol=1e-12, atol=1e-12)
    assert np.allclose(m1[0, 0], c.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_full_decay_reset():
    """da = -inf: every step forgets the past, h_t = W_t.  With C = 1 and initial = 0 this
    gives m2 = sum_t |xhat_t|^2 (R_t bhat_t)(R_t bhat_t)^T."""
    rng = np.random.default_rng(7)
    P = rand_problem(rng, b=1, s=5, C=1, h=1, p=3, r=8, kind="pairwise", rope_dim=8, valid=(5,))
    P["da"] = np.full_like(P["da"], -np.inf)
    P["initial"] = np.zeros_like(P["initial"])
    m2_ref = np.zeros((8, 8))
    for t in range(5):
        v = P["bhat"][0, t, 0, 0].copy()
        out = v.copy()
        for i in range(4):
            th = P["rot"][0, t, 0, i]
            out[2 * i] = np.cos(th) * v[2 * i] + np.sin(th) * v[2 * i + 1]
            out[2 * i + 1] = -np.sin(th) * v[2 * i] + np.cos(th) * v[2 * i + 1]
        m2_ref += np.sum(P["xhat"][0, t, 0, 0] ** 2) * np.outer(out, out)
    m2, _ = fwd(P)
    assert np.allclose(m2[0, 0], m2_ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ chunked == unchunked
@pytest.mark.parametrize("kind,rope,J", KINDS)
@pytest.mark.parametrize("l,valid", [(1, 12), (3, 7), (4, 12), (12, 12), (4, 0), (4, 1), (4, 9), (6, 20), (12, 5)])
def test_chunked_pages_algorithm_matches_token_oracle(kind, rope, J, l, valid):
    """The pages' chunkwise forward and recompute backward (restated in NumPy) equal the
    token-level oracle for any chunk length and any valid_len (scalar, as on the pages)."""
    rng = np.random.default_rng(100 + l + valid)
    P = rand_problem(rng, b=2, s=12, kind=kind, rope_dim=rope, J=J, valid=(valid, valid))
    m2, m1 = fwd(P)
    c2, c1 = chunked_ref.fwd(P["xhat"], P["bhat"], P["da"], P["rot"], P["initial"], valid, l,
                             kind=kind, rope_dim=rope)
    assert np.allclose(m2, c2, rtol=1e-11, atol=1e-11)
    assert np.allclose(m1, c1, rtol=1e-11, atol=1e-11)
    G = bwd(P)
    Gc = chunked_ref.bwd(P["xhat"], P["bhat"], P["da"], P["rot"], P["initial"], valid, l,
                         P["d_m2"], P["d_m1"], kind=kind, rope_dim=rope)
    for k in ("d_xhat", "d_bhat", "d_da", "d_initial") + (("d_rot",) if P["rot"].size else ()):
        assert np.allclose(G[k], Gc[k], rtol=1e-10, atol=1e-10), k


# ------------------------------------------------------------------- permutation pins
def test_half_split_is_pairwise_on_permuted_rank():
    """Half-split pairs (i, i + r/2) = pairwise pairs (2i, 2i+1) after permuting the rank
    axis by pi = [0, r/2, 1, r/2+1, ...] (rest of the dims in order)."""
    rng = np.random.default_rng(8)
    r, na = 8, 3
    P = rand_problem(rng, r=r, kind="half", rope_dim=2 * na)
    pi = []
    for i in range(na):
        pi += [i, i + r // 2]
    pi += [i for i in range(r) if i not in pi]
    pi = np.array(pi)
    m2h, m1h = fwd(P)
    Q = dict(P, kind="pairwise", bhat=P["bhat"][..., pi], initial=P["initial"][..., pi],
             d_m2=P["d_m2"][..., pi][..., pi, :], d_m1=P["d_m1"][..., pi])
    m2p, m1p = fwd(Q)
    assert np.allclose(m2p, m2h[..., pi][..., pi, :], rtol=1e-12, atol=1e-12)
    assert np.allclose(m1p, m1h[..., pi], rtol=1e-12, atol=1e-12)
    Gh, Gp = bwd(P), bwd(Q)
    assert np.allclose(Gp["d_bhat"], Gh["d_bhat"][..., pi], rtol=1e-11, atol=1e-11)
    assert np.allclose(Gp["d_initial"], Gh["d_initial"][..., pi], rtol=1e-11, atol=1e-11)
    for k in ("d_xhat", "d_da", "d_rot"):
        assert np.allclose(Gp[k], Gh[k], rtol=1e-11, atol=1e-11), k


def test_quaternion_as_complex_pairs():
    """Q = (cos t, 0, 0, -sin t) acting on a block (w,x,y,z) equals the complex pairwise
    de-rotation with angle t on both pairs of the block reordered as [w, z, x, y]; the
    angle gradient is then d_t = -sin(t) d_Qw - cos(t) d_Qz (chain rule)."""
    rng = np.random.default_rng(9)
    P = rand_problem(rng, r=8, kind="quat", J=2)
    th = np.cumsum(rng.uniform(-0.5, 0.5, (2, 7, 2, 2)), axis=1)  # one angle per block
    Qr = np.zeros((2, 7, 2, 2, 4))
    Qr[..., 0], Qr[..., 3] = np.cos(th), -np.sin(th)
    perm = np.array([0, 3, 1, 2, 4, 7, 5, 6])            # [w,z,x,y] per block
    Pq = dict(P, rot=Qr)
    ang = np.repeat(th, 2, axis=-1)                       # both pairs of block k use th[k]
    Pc = dict(P, kind="pairwise", rope_dim=8, J=0, rot=ang, bhat=P["bhat"][..., perm],
              initial=P["initial"][..., perm], d_m2=P["d_m2"][..., perm][..., perm, :],
              d_m1=P["d_m1"][..., perm])
    m2q, m1q = fwd(Pq)
    m2c, m1c = fwd(Pc)
    assert np.allclose(m2c, m2q[..., perm][..., perm, :], rtol=1e-12, atol=1e-12)
    assert np.allclose(m1c, m1q[..., perm], rtol=1e-12, atol=1e-12)
    Gq, Gc = bwd(Pq), bwd(Pc)
    dq = Gq["d_rot"]
    dth_from_q = -np.sin(th) * dq[..., 0] - np.cos(th) * dq[..., 3]
    dth_c = Gc["d_rot"].reshape(2, 7, 2, 2, 2).sum(-1)
    assert np.allclose(dth_c, dth_from_q, rtol=1e-10, atol=1e-10)


def test_golden_quaternion_basis_table():
    """The Hamilton product seen through the operator: p = 1, C = 1, initial = 0, xhat = 1,
    bhat = right factor, Q = left factor, one token -> m1 = Q (x) v."""
    basis = {"1": [1, 0, 0, 0], "i": [0, 1, 0, 0], "j": [0, 0, 1, 0], "k": [0, 0, 0, 1]}
    rows = [l.split() for l in open(os.path.join(GOLD, "quaternion_basis.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for row in rows:
        left, right, prod = basis[row[0]], basis[row[1]], np.array([float(v) for v in row[2:]])
        P = dict(xhat=np.ones((1, 1, 1, 1, 1)), bhat=np.array(right, float).reshape(1, 1, 1, 1, 4),
                 da=np.zeros((1, 1, 1)), rot=np.array(left, float).reshape(1, 1, 1, 1, 4),
                 initial=np.zeros((1, 1, 1, 4)), valid_len=np.array([1]), d_m2=np.zeros((1, 1, 4, 4)),
                 d_m1=np.zeros((1, 1, 4)), kind="quat", rope_dim=0, J=1)
        _, m1 = fwd(P)
        assert np.array_equal(m1[0, 0], prod), row


def test_golden_chunk_bookkeeping():
    """processed-chunk counts and per-chunk valid rows (pages' chunk_mask / processed)."""
    rows = [l for l in open(os.path.join(GOLD, "chunk_masks.txt")) if l.strip() and not l.startswith("#")]
    for line in rows:
        head, proc, masks = line.split("|")
        valid, l, n = (int(v) for v in head.split())
        want = [int(v) for v in masks.split()]
        got = [int(chunked_ref._mask(l, k * l, valid).sum()) for k in range(n)]
        assert got == want, line
        processed = min(-(-valid // l), n) if valid > 0 else 0
        assert processed == int(proc)
        # the token oracle consumes exactly sum(want) tokens: m1 with unit writes counts them
        P = dict(xhat=np.ones((1, l * n, 1, 1, 1)), bhat=np.ones((1, l * n, 1, 1, 1)),
                 da=np.full((1, l * n, 1), -np.inf), rot=np.zeros((1, l * n, 1, 0)),
                 initial=np.zeros((1, 1, 1, 1)), valid_len=np.array([valid]), kind="none",
                 rope_dim=0, J=0, d_m2=None, d_m1=None)
        _, m1 = fwd(P)
        assert m1[0, 0, 0] == sum(want)


# ------------------------------------------------------------ symmetry and scaling
def test_antisymmetric_cotangent_gives_zero_grads():
    rng = np.random.default_rng(10)
    for kind, rope, J in KINDS:
        P = rand_problem(rng, kind=kind, rope_dim=rope, J=J)
        A = rng.standard_normal((2, 2, 8, 8))
        G = bwd(P, d_m2=A - np.swapaxes(A, 2, 3), d_m1=np.zeros((2, 2, 8)))
        for k, v in G.items():
            assert v.size == 0 or np.abs(v).max() == 0.0, (kind, k)


def test_m2_symmetric_psd_and_scaling():
    rng = np.random.default_rng(12)
    for kind, rope, J in KINDS:
        P = rand_problem(rng, kind=kind, rope_dim=rope, J=J)
        m2, m1 = fwd(P)
        assert np.array_equal(m2, np.swapaxes(m2, 2, 3))
        assert np.linalg.eigvalsh(m2).min() > -1e-9 * np.abs(m2).max()
        m2s, m1s = fwd(P, xhat=2.5 * P["xhat"], initial=2.5 * P["initial"])
        assert np.allclose(m2s, 6.25 * m2, rtol=1e-12, atol=1e-12)
        assert np.allclose(m1s, 2.5 * m1, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- masking invariants
@pytest.mark.parametrize("kind,rope,J", KINDS)
def test_masking_invariants(kind, rope, J):
    rng = np.random.default_rng(13)
    P = rand_problem(rng, s=9, kind=kind, rope_dim=rope, J=J, valid=(4, 9))
    m2, m1 = fwd(P)
    G = bwd(P)
    Q = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in P.items()}
    for name in ("xhat", "bhat", "da", "rot"):
        if Q[name].size:
            Q[name][0, 4:] = rng.standard_normal(Q[name][0, 4:].shape)
    m2q, m1q = fwd(Q)
    Gq = bwd(Q)
    assert np.array_equal(m2, m2q) and np.array_equal(m1, m1q)
    for k in G:
        assert np.array_equal(G[k], Gq[k]), k
        if k != "d_initial" and G[k].size:
            assert np.abs(G[k][0, 4:]).max() == 0.0, k
    # per-batch valid_len == independent single-row calls
    for bb in range(2):
        R = {k: (v[bb:bb + 1] if isinstance(v, np.ndarray) else v) for k, v in P.items()}
        m2r, m1r = fwd(R)
        assert np.array_equal(m2r[0], m2[bb]) and np.array_equal(m1r[0], m1[bb])
    # valid_len = 0: nothing contributes, every gradient is zero
    Z = bwd(P, valid_len=np.array([0, 0]))
    z2, z1 = fwd(P, valid_len=np.array([0, 0]))
    assert not z2.any() and not z1.any() and all(not v.any() for v in Z.values())
    # valid_len > s clamps to s
    c2, _ = fwd(P, valid_len=np.array([4, 50]))
    assert np.array_equal(c2, m2)
