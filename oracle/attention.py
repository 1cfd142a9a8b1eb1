"""Plain float64 definitions of exact attention, its tiled online-softmax
schedule and its gradients.  Test infrastructure only (see the package
docstring for who may import it).

Conventions
-----------
* Tensors are ``[..., N, d]`` (normally ``[B, H, N, d]``); every leading index
  is an independent head.  Inputs of any float dtype are widened to float64
  before any arithmetic, so bf16 inputs are taken at their exact bf16 values.
* ``scale`` multiplies the raw scores.  NOTES, "The Standard Attention
  Problem" prints ``P = softmax(S / d_k)``, but its worked example divides
  ``1`` by "2" and gets ``0.707`` for ``d = 2``; only ``1/sqrt(d)`` gives that
  number, so the square root was lost when the page was extracted.  Callers
  pass ``1/sqrt(d)`` for the pages' attention; the oracle itself takes any
  positive scale.
* ``window``: ``<= 0`` means unmasked.  A positive ``window = w`` (odd) lets
  query ``i`` attend to key ``j`` iff ``|i - j| <= (w - 1) / 2``, following
  NOTES, "Worked example Local Attention Window" (``w = 3``: the token itself
  and one neighbour on each side).  The band always contains the diagonal, so
  no query row with a matching key is ever fully masked.
* ``lse`` is the natural logarithm of the row sum of ``exp`` over the scaled,
  masked scores.
"""

from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def window_radius(window: int) -> int | None:
    """Half-width ``r`` of a symmetric window of full width ``window``.

    NOTES, "Worked example Local Attention Window": ``w = 3`` means the token
    itself plus one neighbour each side, i.e. ``r = (w - 1) / 2``.  Returns
    ``None`` for an unmasked call (``window <= 0``).  Even widths have no
    reading on the page and are rejected.
    """
    if window <= 0:
        return None
    if window % 2 == 0:
        raise ValueError("window width must be odd (self plus r neighbours per side)")
    return (window - 1) // 2


def window_mask(n_q: int, n_k: int, window: int) -> np.ndarray:
    """Boolean ``[n_q, n_k]`` matrix: True where query ``i`` may see key ``j``.

    NOTES, "Worked example Local Attention Window": for ``N = 6, w = 3`` this
    is the printed tridiagonal 0/1 matrix.
    """
    r = window_radius(window)
    if r is None:
        return np.ones((n_q, n_k), dtype=bool)
    i = np.arange(n_q)[:, None]
    j = np.arange(n_k)[None, :]
    return np.abs(i - j) <= r


def dense_scores(q, k, scale: float, window: int = 0) -> np.ndarray:
    """Scaled, masked score matrix ``S = Q K^T * scale`` (masked entries -inf).

    NOTES, "The Standard Attention Problem", first line of the computational
    flow (``S = Q K^T``), with the scale applied as in that section's second
    line and the window of "Worked example Local Attention Window".
    """
    q, k = _f64(q), _f64(k)
    s = np.matmul(q, np.swapaxes(k, -1, -2)) * float(scale)
    if window > 0:
        s = np.where(window_mask(q.shape[-2], k.shape[-2], window), s, NEG_INF)
    return s


def dense_forward(q, k, v, scale: float, window: int = 0):
    """Exact attention by its definition: ``O = softmax(S) V`` and ``lse``.

    NOTES, "The Standard Attention Problem" (S, P = softmax, O = P V) with the
    max-shift of "Derivation: Incremental Softmax", Step 1 (subtracting the
    row maximum changes no softmax value and keeps ``exp`` finite); TVIZ step
    "dense" (all N x N scores materialised, each row normalised over every
    key).  Returns ``(O [..., N, d], lse [..., N])`` in float64.
    """
    v = _f64(v)
    s = dense_scores(q, k, scale, window)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=-1, keepdims=True)
    p = e / l
    o = np.matmul(p, v)
    lse = m[..., 0] + np.log(l[..., 0])
    return o, lse


def dense_forward_rows(q, k, v, scale: float, rows, window: int = 0):
    """``dense_forward`` restricted to the query rows ``rows`` of one head.

    ``q, k, v`` are ``[N, d]``; returns ``(O[rows], lse[rows])``.  Each output
    row of the definition depends on its own query row and on all keys and
    values only, so this is the same definition evaluated row by row, used to
    check sampled rows of very large problems.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    rows = np.asarray(rows, dtype=np.int64)
    s = np.matmul(q[rows], k.T) * float(scale)
    r = window_radius(window)
    if r is not None:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(np.abs(rows[:, None] - j) <= r, s, NEG_INF)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=-1, keepdims=True)
    o = np.matmul(e / l, v)
    return o, m[:, 0] + np.log(l[:, 0])


def banded_forward_rows(q, k, v, scale: float, rows, window: int):
    """Windowed attention for the rows ``rows`` touching only in-band keys.

    NOTES, "Worked example Local Attention Window" (cost O(N w) instead of
    O(N^2)): row ``i`` reads keys ``max(0, i - r) .. min(N - 1, i + r)`` only.
    ``q, k, v`` are ``[N, d]`` of one head.  Agrees with
    ``dense_forward_rows(..., window)``; the tests check that.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    r = window_radius(window)
    if r is None:
        raise ValueError("banded_forward_rows needs a positive window")
    n = k.shape[0]
    outs, lses = [], []
    for i in np.asarray(rows, dtype=np.int64):
        lo, hi = max(0, i - r), min(n, i + r + 1)
        s = (k[lo:hi] @ q[i]) * float(scale)
        m = np.max(s)
        e = np.exp(s - m)
        l = np.sum(e)
        outs.append((e / l) @ v[lo:hi])
        lses.append(m + np.log(l))
    return np.array(outs), np.array(lses)


def block_statistics(x, v):
    """Per-block statistics of NOTES, "Derivation: Incremental Softmax", Step 2.

    For a block of scores ``x`` (``[..., b]``, already scaled; masked entries
    -inf) and the block's value rows ``v`` (``[b, d]``) returns
    ``m = max x``, ``l = sum_j exp(x_j - m)`` and the unnormalised block output
    ``O~ = sum_j exp(x_j - m) v_j``.  A block whose scores are all -inf has
    ``m = -inf, l = 0, O~ = 0``.
    """
    x, v = _f64(x), _f64(v)
    m = np.max(x, axis=-1)
    finite = np.isfinite(m)
    ref = np.where(finite, m, 0.0)
    e = np.exp(x - ref[..., None])  # exp(-inf) = 0 for masked entries
    l = np.sum(e, axis=-1)
    o = np.matmul(e, v)
    return m, l, o


def _shift(m_old, m_new):
    """``exp(m_old - m_new)`` with the convention that an empty block
    (``m_old = -inf``) contributes with factor 0."""
    m_old, m_new = _f64(m_old), _f64(m_new)
    out = np.zeros(np.broadcast(m_old, m_new).shape)
    ok = np.isfinite(m_old)
    np.exp(m_old - m_new, out=out, where=ok)
    return out


def merge_statistics(m1, l1, o1, m2, l2, o2):
    """Merge two blocks' ``(m, l, O~)``: NOTES, "Derivation: Incremental
    Softmax", Step 3.

    ``m_new = max(m1, m2)``; both sums and both unnormalised outputs are moved
    to the common reference point ``m_new`` by ``exp(m_b - m_new)`` and added.
    The returned ``O~`` is still unnormalised; the page's ``O_new`` is
    ``O~ / l_new`` (done once, at the end, by ``tiled_forward``).
    """
    m_new = np.maximum(_f64(m1), _f64(m2))
    a1 = _shift(m1, m_new)
    a2 = _shift(m2, m_new)
    l_new = a1 * _f64(l1) + a2 * _f64(l2)
    o_new = a1[..., None] * _f64(o1) + a2[..., None] * _f64(o2)
    return m_new, l_new, o_new


def tiled_forward(q, k, v, scale: float, block_rows: int, block_cols: int, window: int = 0,
                  trace=None):
    """Exact attention one tile at a time with running statistics.

    TVIZ step "tiles": a query-major loop; for each ``block_rows`` x
    ``block_cols`` score tile, the running maximum, running denominator and
    weighted numerator of every query row in the tile are updated (earlier
    contributions are rescaled whenever the running maximum rises), and the
    numerator is divided by the denominator once all key tiles are seen.  The
    per-tile update is NOTES Step 3's merge of the running state with the
    tile's Step 2 statistics ("generalises to any number of blocks").  The
    last tile in either direction may be short (TVIZ numerical checks:
    "uneven final tiles").  The full score matrix is never formed.

    ``trace`` (optional list): for every tile, appends a dict with the tile's
    query/key ranges, its score tile and the running ``m``, ``l`` and partial
    output ``O~ / l`` of its query rows, as in the TVIZ tile replay.
    Returns ``(O, lse)`` like ``dense_forward``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = q.shape[:-2]
    n_q, d = q.shape[-2:]
    n_k = k.shape[-2]
    dv = v.shape[-1]
    o_out = np.empty(lead + (n_q, dv))
    lse_out = np.empty(lead + (n_q,))
    for idx in np.ndindex(*lead):
        qh, kh, vh = q[idx], k[idx], v[idx]
        for i0 in range(0, n_q, block_rows):
            i1 = min(n_q, i0 + block_rows)
            m = np.full(i1 - i0, NEG_INF)
            l = np.zeros(i1 - i0)
            acc = np.zeros((i1 - i0, dv))
            for j0 in range(0, n_k, block_cols):
                j1 = min(n_k, j0 + block_cols)
                s = (qh[i0:i1] @ kh[j0:j1].T) * float(scale)
                if window > 0:
                    s = np.where(window_mask(n_q, n_k, window)[i0:i1, j0:j1], s, NEG_INF)
                mb, lb, ob = block_statistics(s, vh[j0:j1])
                m, l, acc = merge_statistics(m, l, acc, mb, lb, ob)
                if trace is not None:
                    with np.errstate(invalid="ignore", divide="ignore"):
                        part = acc / l[:, None]
                    trace.append(dict(head=idx, rows=(i0, i1), cols=(j0, j1), scores=s.copy(),
                                      m=m.copy(), l=l.copy(), partial=part))
            o_out[idx][i0:i1] = acc / l[:, None]
            lse_out[idx][i0:i1] = m + np.log(l)
    return o_out, lse_out


def dense_backward(q, k, v, do, scale: float, window: int = 0):
    """Gradients of ``O = softmax(S) V`` with respect to Q, K and V.

    The pages only say that the backward pass recomputes S and P instead of
    reading them (NOTES, "Backward Pass: Recomputation"); they print no
    formulas, so this is the derivative of the definition above, written out:

    * ``dV = P^T dO`` and ``dP = dO V^T``  (O = P V is bilinear);
    * row-wise softmax Jacobian: ``dS_ij = P_ij (dP_ij - D_i)`` with
      ``D_i = sum_j P_ij dP_ij``;
    * ``S = scale * Q K^T``: ``dQ = scale * dS K`` and ``dK = scale * dS^T Q``.

    Masked scores have ``P = 0`` and so receive no gradient.  Returns
    ``(dQ, dK, dV)`` in float64.
    """
    v, do = _f64(v), _f64(do)
    q, k = _f64(q), _f64(k)
    s = dense_scores(q, k, scale, window)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    p = e / np.sum(e, axis=-1, keepdims=True)
    dv = np.matmul(np.swapaxes(p, -1, -2), do)
    dp = np.matmul(do, np.swapaxes(v, -1, -2))
    dsum = np.sum(p * dp, axis=-1, keepdims=True)
    ds = p * (dp - dsum)
    dq = float(scale) * np.matmul(ds, k)
    dk = float(scale) * np.matmul(np.swapaxes(ds, -1, -2), q)
    return dq, dk, dv
