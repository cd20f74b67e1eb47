"""The pages' chunkwise algorithm, restated in NumPy fp64 (TEST INFRASTRUCTURE ONLY).

This is a second, independent statement of the same operator, organised the way the
source pages organise it, so that the token-level C oracle can be pinned against it
("chunked == unchunked"):

* forward: burn-mamba "mamba3/moments/recalculated.rs", ``moments_phys_fwd`` -- a serial
  loop over chunks that stops at the first chunk starting at or past ``valid_len``;
  per chunk ``chunk_decay`` (inclusive cumsum, d_t = exp(a_t), the lower-triangular
  L[t,j] = exp(a_t - a_j)), ``chunk_states`` (channels folded into the write index of one
  contraction, plus the carried d_t * h_-), the carry = last state of the chunk,
  ``rotate_chunk`` (de-rotation), ``chunk_mask`` and the moment sums over the l*p rows.
* backward: "mamba3/moments/backward.rs", ``moments_phys_bwd`` -- ``boundary_carries``
  (decay-to-chunk-end contraction + serial accumulation), then a reverse chunk loop:
  recompute states, the moments VJP, the rotation transpose + ``d_theta_chunk`` /
  ``d_quat_chunk``, ``scatter_last`` of the carry cotangent, the new carry
  sum_t d_t G[t], d_W = L^T G, d_xhat / d_bhat, and d_da through the reverse-cumsum
  identity of the module header.  Skipped chunks get zero gradients.

Here ``valid_len`` is one scalar for the whole batch, as on the pages.  Shapes follow the
pages' pre-chunked layout: xhat [b,n,l,C,h,p] is the same memory as [b,s,C,h,p].
"""
from __future__ import annotations

import numpy as np


def _decay(da_blh):
    """d [b,h,l] and L [b,h,l,l] of one chunk (zero strictly above the diagonal)."""
    a = np.cumsum(np.transpose(da_blh, (0, 2, 1)), axis=2)
    l = a.shape[2]
    lower = np.tril(np.ones((l, l), dtype=bool))
    diff = a[:, :, :, None] - a[:, :, None, :]
    L = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
    return np.exp(a), L


def _states(x_blchp, b_blchr, d_bhl, L_bhll, hin_bhpr):
    """Cache-frame states of one chunk [b,h,l,p,r]; channels folded into the K index."""
    bsz, l, C, h, p = x_blchp.shape
    r = b_blchr.shape[-1]
    xw = np.einsum("bhtj,bjchp->bhtjcp", L_bhll, x_blchp).reshape(bsz, h, l, l * C, p)
    bk = np.transpose(b_blchr, (0, 3, 1, 2, 4)).reshape(bsz, h, l * C, r)
    intra = np.einsum("bhtkp,bhkr->bhtpr", xw, bk)
    return d_bhl[:, :, :, None, None] * hin_bhpr[:, :, None, :, :] + intra


def _writes(x_blchp, b_blchr):
    return np.einsum("bjchp,bjchr->bhjpr", x_blchp, b_blchr)


def _qmul(a, b):
    aw, ax, ay, az = (a[..., i] for i in range(4))
    bw, bx, by, bz = (b[..., i] for i in range(4))
    return np.stack([aw * bw - ax * bx - ay * by - az * bz,
                     aw * bx + ax * bw + ay * bz - az * by,
                     aw * by - ax * bz + ay * bw + az * bx,
                     aw * bz + ax * by - ay * bx + az * bw], axis=-1)


def _qconj(q):
    return q * np.array([1.0, -1.0, -1.0, -1.0])


def _rotate(v_bhlpr, rot, kind, rope_dim, start, transpose):
    """De-rotation (transpose=False: R(-theta) / Q (x) .) or its transpose of a chunk."""
    bsz, h, l, p, r = v_bhlpr.shape
    if kind == "none" or (kind in ("pairwise", "half") and rope_dim == 0):
        return v_bhlpr.copy()
    out = v_bhlpr.copy()
    if kind in ("pairwise", "half"):
        th = np.transpose(rot[:, start:start + l], (0, 2, 1, 3))[:, :, :, None, :]  # [b,h,l,1,a]
        phi = th if transpose else -th
        cs, sn = np.cos(phi), np.sin(phi)
        na = rope_dim // 2
        if kind == "pairwise":
            ix, iy = np.arange(na) * 2, np.arange(na) * 2 + 1
        else:
            ix, iy = np.arange(na), np.arange(na) + r // 2
        x, y = v_bhlpr[..., ix], v_bhlpr[..., iy]
        out[..., ix] = cs * x - sn * y
        out[..., iy] = sn * x + cs * y
        return out
    J = rot.shape[3]
    q = np.transpose(rot[:, start:start + l], (0, 2, 1, 3, 4))[:, :, :, None, :, :]  # [b,h,l,1,J,4]
    if transpose:
        q = _qconj(q)
    blocks = v_bhlpr[..., :4 * J].reshape(bsz, h, l, p, J, 4)
    out[..., :4 * J] = _qmul(np.broadcast_to(q, blocks.shape), blocks).reshape(bsz, h, l, p, 4 * J)
    return out


def _mask(l, start, valid_len):
    valid = min(max(valid_len - start, 0), l)
    m = np.zeros(l)
    m[:valid] = 1.0
    return m


def _chunked(a, l):
    b, s = a.shape[:2]
    return a.reshape((b, s // l, l) + a.shape[2:])


def fwd(xhat, bhat, da, rot, initial, valid_len, chunk_len, kind="pairwise", rope_dim=0):
    """Serial chunkwise forward; returns (m2 [b,h,r,r], m1 [b,h,r])."""
    x, bb, dd = _chunked(xhat, chunk_len), _chunked(bhat, chunk_len), _chunked(da, chunk_len)
    bsz, n, l, C, h, p = x.shape
    r = bb.shape[-1]
    hcar = np.array(initial, dtype=np.float64)
    m2 = np.zeros((bsz, h, r, r))
    m1 = np.zeros((bsz, h, r))
    for k in range(n):
        start = k * l
        if start >= valid_len:
            break
        d, L = _decay(dd[:, k])
        st = _states(x[:, k], bb[:, k], d, L, hcar)
        hcar = st[:, :, l - 1]
        ph = _rotate(st, rot, kind, rope_dim, start, False)
        ph = ph * _mask(l, start, valid_len)[None, None, :, None, None]
        rows = ph.reshape(bsz, h, l * p, r)
        m2 += np.einsum("bhkr,bhks->bhrs", rows, rows)
        m1 += rows.sum(axis=2)
    return m2, m1


def _carries(x, bb, dd, initial, processed):
    """Entry states of the first ``processed`` chunks (decay-to-end contraction + scan)."""
    bsz, n, l, C, h, p = x.shape
    hcar = np.array(initial, dtype=np.float64)
    out = []
    for k in range(processed):
        out.append(hcar)
        if k + 1 == processed:
            break
        a = np.cumsum(np.transpose(dd[:, k], (0, 2, 1)), axis=2)  # [b,h,l]
        scale = np.exp(a[:, :, -1:] - a)
        contrib = np.einsum("bhj,bjchp,bjchr->bhpr", scale, x[:, k], bb[:, k])
        hcar = np.exp(a[:, :, -1])[:, :, None, None] * hcar + contrib
    return out


def _rev_cumsum(t, axis):
    return np.flip(np.cumsum(np.flip(t, axis), axis), axis)


def bwd(xhat, bhat, da, rot, initial, valid_len, chunk_len, d_m2, d_m1, kind="pairwise", rope_dim=0):
    """The pages' recompute backward; returns dict d_xhat, d_bhat, d_da, d_rot, d_initial."""
    x, bb, dd = _chunked(xhat, chunk_len), _chunked(bhat, chunk_len), _chunked(da, chunk_len)
    bsz, n, l, C, h, p = x.shape
    r = bb.shape[-1]
    processed = min(-(-valid_len // l), n) if valid_len > 0 else 0
    hins = _carries(x, bb, dd, initial, processed)
    dsym = d_m2 + np.swapaxes(d_m2, 2, 3)
    dx = np.zeros_like(x)
    db = np.zeros_like(bb)
    dda = np.zeros_like(dd)
    drot = np.zeros_like(rot) if rot is not None else None
    dcar = np.zeros((bsz, h, p, r))
    for k in reversed(range(processed)):
        start = k * l
        d, L = _decay(dd[:, k])
        st = _states(x[:, k], bb[:, k], d, L, hins[k])
        ph = _rotate(st, rot, kind, rope_dim, start, False)
        msk = _mask(l, start, valid_len)[None, None, :, None, None]
        dph = (np.einsum("bhlpr,bhrs->bhlps", ph, dsym) + d_m1[:, :, None, None, :]) * msk
        dst = _rotate(dph, rot, kind, rope_dim, start, True)
        if kind in ("pairwise", "half") and rope_dim > 0:
            na = rope_dim // 2
            if kind == "pairwise":
                ix, iy = np.arange(na) * 2, np.arange(na) * 2 + 1
            else:
                ix, iy = np.arange(na), np.arange(na) + r // 2
            dth = (dph[..., ix] * ph[..., iy] - dph[..., iy] * ph[..., ix]).sum(axis=3)  # [b,h,l,a]
            drot[:, start:start + l] = np.transpose(dth, (0, 2, 1, 3))
        elif kind == "quat":
            J = rot.shape[3]
            dq = _qmul(dph[..., :4 * J].reshape(bsz, h, l, p, J, 4),
                       _qconj(st[..., :4 * J].reshape(bsz, h, l, p, J, 4))).sum(axis=3)
            drot[:, start:start + l] = np.transpose(dq, (0, 2, 1, 3, 4))
        G = dst.copy()
        G[:, :, l - 1] += dcar                                  # scatter_last
        dcar = np.einsum("bhl,bhlpr->bhpr", d, G)
        dW = np.einsum("bhtj,bhtpr->bhjpr", L, G)
        dx[:, k] = np.einsum("bjchr,bhjpr->bjchp", bb[:, k], dW)
        db[:, k] = np.einsum("bjchp,bhjpr->bjchr", x[:, k], dW)
        W = _writes(x[:, k], bb[:, k])
        scal = np.einsum("bhlpr,bhpr->bhl", G, hins[k]) * d
        A = np.einsum("bhtpr,bhjpr->bhtj", G, W) * L
        row, col = A.sum(axis=3), A.sum(axis=2)
        dda[:, k] = np.transpose(_rev_cumsum(scal + row, 2) - _rev_cumsum(col, 2), (0, 2, 1))
    return dict(d_xhat=dx.reshape(xhat.shape), d_bhat=db.reshape(bhat.shape),
                d_da=dda.reshape(da.shape), d_rot=drot, d_initial=dcar)
