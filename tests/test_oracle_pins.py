"""Pins of the float64 oracle's forward pass against things other than itself.

Each test pins the oracle to one of: values printed on the pages (fixtures in
tests/golden/, each naming its page and section), closed forms, invariants of
the mathematics, or a library routine (torch's float64 CPU attention).  The
mutation tests at the end plant plausible mistakes in copies of the oracle's
arithmetic (on the CPU) and check that the pins catch each of them.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Flash attention and efficient attention -- Hinglish notes, worked example
# ---------------------------------------------------------------------------

def check_worked_example(forward, golden):
    """The example's query row 0 output, to the page's 3 printed decimals."""
    q = np.array(golden["Q"], float)[None, None]
    k = np.array(golden["K"], float)[None, None]
    v = np.array(golden["V"], float)[None, None]
    o, _ = forward(q, k, v, 1.0 / math.sqrt(2.0))
    return np.allclose(o[0, 0, 0], golden["merge"]["O_row0"], atol=5e-4, rtol=0)


def test_worked_example_row0(golden_dir):
    g = _load(golden_dir, "notes_worked_example.json")
    assert check_worked_example(oracle.dense_forward, g)
    assert check_worked_example(lambda q, k, v, s: oracle.tiled_forward(q, k, v, s, 1, 2), g)
    # the exact value behind the printed [0.830, 1.170]
    q = np.array(g["Q"], float)
    o, _ = oracle.dense_forward(q, q, np.array(g["V"], float), 1 / math.sqrt(2))
    assert abs(o[0, 0] - 0.8302385) < 1e-7 and abs(o[0, 1] - 1.1697615) < 1e-7


def test_worked_example_block_statistics(golden_dir):
    g = _load(golden_dir, "notes_worked_example.json")
    q = np.array(g["Q"], float)
    k = np.array(g["K"], float)
    v = np.array(g["V"], float)
    tol = dict(atol=5e-4, rtol=0)
    scale = 1.0 / math.sqrt(2.0)
    stats = []
    for blk, (j0, j1) in (("block1", (0, 2)), ("block2", (2, 4))):
        s = oracle.dense_scores(q[0:1], k[j0:j1], scale)[0]
        np.testing.assert_allclose(s, g[blk]["scores"], **tol)
        m, l, ot = oracle.block_statistics(s, v[j0:j1])
        np.testing.assert_allclose(np.exp(s - m), g[blk]["exponents"], **tol)
        np.testing.assert_allclose(m, g[blk]["m"], **tol)
        np.testing.assert_allclose(l, g[blk]["l"], **tol)
        np.testing.assert_allclose(ot, g[blk]["O_tilde"], **tol)
        stats.append((m, l, ot))
    m, l, num = oracle.merge_statistics(*stats[0], *stats[1])
    np.testing.assert_allclose(m, g["merge"]["m_new"], **tol)
    np.testing.assert_allclose(l, g["merge"]["l_new"], **tol)
    np.testing.assert_allclose(num, g["merge"]["numerator"], **tol)
    np.testing.assert_allclose(num / l, g["merge"]["O_row0"], **tol)


def test_worked_example_scale_is_inverse_sqrt_d(golden_dir):
    """The page prints '/2' but its 0.707 needs 1/sqrt(2); a literal 1/d fails."""
    g = _load(golden_dir, "notes_worked_example.json")
    q = np.array(g["Q"], float)
    assert abs(oracle.dense_scores(q[:1], q[:1], 1 / math.sqrt(2))[0, 0] - 0.707) < 5e-4
    assert abs(oracle.dense_scores(q[:1], q[:1], 1 / 2)[0, 0] - 0.707) > 0.1


def test_worked_example_rescale_aside(golden_dir):
    """The section's aside: block maxima 1/sqrt(2) and sqrt(2) give block 1 a
    rescale factor of about 0.493 in the merge."""
    a = _load(golden_dir, "notes_worked_example.json")["aside"]
    m1, m2 = a["m1"], a["m2"]
    # l1 = 1 and l2 = 0 isolate block 1's factor in l_new
    _, l_new, _ = oracle.merge_statistics(np.array(m1), np.array(1.0), np.zeros(1),
                                          np.array(m2), np.array(0.0), np.zeros(1))
    assert abs(float(l_new) - a["factor1"]) < 5e-4


# ---------------------------------------------------------------------------
# Compute attention one tile at a time (TensorViz): tile replay
# ---------------------------------------------------------------------------

def replay_running_stats(merge, golden):
    """Feed the page's printed score tiles through Step 2 / Step 3 and return
    the worst deviation from its printed running max and denominators."""
    m = np.full(2, -np.inf)
    l = np.zeros(2)
    acc = np.zeros((2, 1))
    worst = 0.0
    for t in golden["tiles"]:
        s = np.array(t["scores"], float).reshape(2, 2)
        mb, lb, ob = oracle.block_statistics(s, np.zeros((2, 1)))
        m, l, acc = merge(m, l, acc, mb, lb, ob)
        worst = max(worst, np.max(np.abs(m - t["running_max"])),
                    np.max(np.abs(l - t["running_denominator"])))
    return worst


def test_tviz_replay_running_statistics(golden_dir):
    g = _load(golden_dir, "tviz_tile_replay.json")
    assert replay_running_stats(oracle.merge_statistics, g) <= 1e-14
    # tile 3 raises row 0's maximum (0.599 -> 1.050): the rescale path is exercised
    assert g["tiles"][2]["running_max"][0] > g["tiles"][1]["running_max"][0]


def test_tviz_replay_final_equals_dense(golden_dir):
    """After the last tile the page's partial output is the dense output
    (difference 2.2e-16 on the page); the oracle's tiled schedule must reach
    the dense definition to the same order on its own inputs."""
    g = _load(golden_dir, "tviz_tile_replay.json")
    last = np.array(g["tiles"][-1]["partial_output_q0"])
    assert np.max(np.abs(last - g["final_dense_output_q0"])) <= 1e-15
    rng = np.random.default_rng(0)
    q, k, v = (rng.standard_normal((1, 6, 4)) for _ in range(3))
    trace = []
    o_t, _ = oracle.tiled_forward(q, k, v, 0.5, 2, 2, trace=trace)
    o_d, _ = oracle.dense_forward(q, k, v, 0.5)
    assert np.max(np.abs(o_t - o_d)) <= 1e-14
    rows01 = [t for t in trace if t["rows"] == (0, 2)]
    assert [t["cols"] for t in rows01] == [(0, 2), (2, 4), (4, 6)]
    np.testing.assert_allclose(rows01[-1]["partial"], o_d[0, 0:2], atol=1e-14, rtol=0)


# ---------------------------------------------------------------------------
# tiled == dense across tile sizes (TVIZ numerical checks: five tile sizes,
# uneven final tiles) and large logits (running-max correction stays finite)
# ---------------------------------------------------------------------------

TILES = [(1, 1), (2, 2), (2, 3), (3, 5), (4, 4), (None, None)]


@pytest.mark.parametrize("n", [6, 7, 13])
@pytest.mark.parametrize("window", [0, 3, 5])
def test_tiled_equals_dense(n, window):
    rng = np.random.default_rng(100 + n + window)
    q, k, v = (rng.standard_normal((2, 2, n, 4)) for _ in range(3))
    o_d, lse_d = oracle.dense_forward(q, k, v, 0.5, window)
    for br, bc in TILES:
        o_t, lse_t = oracle.tiled_forward(q, k, v, 0.5, br or n, bc or n, window)
        assert np.max(np.abs(o_t - o_d)) <= 1e-13, (br, bc)
        assert np.max(np.abs(lse_t - lse_d)) <= 1e-13, (br, bc)


def test_large_logits_stay_finite():
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((1, 1, 13, 4)) for _ in range(3))
    q, k = q * 40.0, k * 40.0  # scores of order +-1000: exp overflows without the max-shift
    s = oracle.dense_scores(q, k, 0.5)
    assert np.abs(s).max() > 800
    with np.errstate(over="ignore", invalid="ignore"):
        naive = np.exp(s) @ v[0, 0] / np.exp(s).sum(-1, keepdims=True)
    assert not np.all(np.isfinite(naive))
    o_d, lse_d = oracle.dense_forward(q, k, v, 0.5)
    assert np.all(np.isfinite(o_d)) and np.all(np.isfinite(lse_d))
    for br, bc in TILES:
        o_t, lse_t = oracle.tiled_forward(q, k, v, 0.5, br or 13, bc or 13)
        assert np.all(np.isfinite(o_t))
        assert np.max(np.abs(o_t - o_d)) <= 1e-12
        assert np.max(np.abs(lse_t - lse_d) / np.abs(lse_d)) <= 1e-12


# ---------------------------------------------------------------------------
# window (NOTES, Worked example Local Attention Window)
# ---------------------------------------------------------------------------

def test_window_mask_matches_page(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "notes_window_n6_w3.txt"))
            if l.strip() and not l.startswith("#")]
    page = np.array(rows, dtype=int).astype(bool)
    assert page.shape == (6, 6)
    assert np.array_equal(oracle.window_mask(6, 6, 3), page)


def test_window_radius_and_even_width():
    assert oracle.window_radius(0) is None and oracle.window_radius(-4) is None
    assert oracle.window_radius(3) == 1 and oracle.window_radius(257) == 128
    with pytest.raises(ValueError):
        oracle.window_radius(4)


@pytest.mark.parametrize("n", [1, 5, 9])
def test_wide_window_is_unmasked(n):
    rng = np.random.default_rng(n)
    q, k, v = (rng.standard_normal((1, 1, n, 3)) for _ in range(3))
    o0, l0 = oracle.dense_forward(q, k, v, 0.7)
    o1, l1 = oracle.dense_forward(q, k, v, 0.7, window=2 * n - 1)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


@pytest.mark.parametrize("n,w", [(37, 5), (200, 33), (512, 257)])
def test_banded_equals_dense_masked(n, w):
    rng = np.random.default_rng(n)
    q, k, v = (rng.standard_normal((n, 16)) for _ in range(3))
    rows = np.arange(n)
    o_b, l_b = oracle.banded_forward_rows(q, k, v, 0.25, rows, w)
    o_d, l_d = oracle.dense_forward(q, k, v, 0.25, window=w)
    assert np.max(np.abs(o_b - o_d)) <= 1e-13 and np.max(np.abs(l_b - l_d)) <= 1e-12


def test_rows_variant_matches_full():
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((50, 8)) for _ in range(3))
    for w in (0, 9):
        o, l = oracle.dense_forward(q, k, v, 0.3, window=w)
        rows = np.array([0, 7, 49, 23])
        o_r, l_r = oracle.dense_forward_rows(q, k, v, 0.3, rows, window=w)
        assert np.max(np.abs(o_r - o[rows])) <= 1e-15 and np.max(np.abs(l_r - l[rows])) <= 1e-15


# ---------------------------------------------------------------------------
# library routine: torch's float64 CPU scaled-dot-product attention
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("window", [0, 1, 3, 9])
def test_against_torch_sdpa_float64(window):
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(11)
    q, k, v = (torch.randn(2, 3, 17, 8, generator=g, dtype=torch.float64) for _ in range(3))
    mask = None
    if window > 0:
        r = (window - 1) // 2
        i = torch.arange(17)
        mask = (i[:, None] - i[None, :]).abs() <= r
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=0.35)
    o, lse = oracle.dense_forward(q.numpy(), k.numpy(), v.numpy(), 0.35, window)
    assert np.max(np.abs(o - ref.numpy())) <= 1e-13
    s = (q @ k.transpose(-1, -2)) * 0.35
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) <= 1e-13


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def test_equal_scores_average_values():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((9, 4))
    v = rng.standard_normal((9, 4))
    o, lse = oracle.dense_forward(q, np.zeros((9, 4)), v, 1.3)
    assert np.max(np.abs(o - v.mean(0))) <= 1e-15
    assert np.max(np.abs(lse - math.log(9))) <= 1e-15


def test_constant_values_pass_through():
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal((2, 11, 5)), rng.standard_normal((2, 11, 5))
    c = rng.standard_normal(5)
    o, _ = oracle.dense_forward(q, k, np.broadcast_to(c, (2, 11, 5)), 0.9, window=5)
    assert np.max(np.abs(o - c)) <= 1e-14


def test_two_key_closed_form():
    """With two keys, row i's output is v0 + (v1 - v0) * sigmoid(scale q_i.(k1 - k0))
    and lse is log(exp(s0) + exp(s1))."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal((5, 3))
    k = rng.standard_normal((2, 3))
    v = rng.standard_normal((2, 4))
    scale = 0.8
    o, lse = oracle.dense_forward(q, k, v, scale)
    sig = 1.0 / (1.0 + np.exp(-scale * q @ (k[1] - k[0])))
    assert np.max(np.abs(o - (v[0] + np.outer(sig, v[1] - v[0])))) <= 1e-14
    assert np.max(np.abs(lse - np.logaddexp(scale * q @ k[0], scale * q @ k[1]))) <= 1e-14


def test_identity_values_expose_probabilities():
    """With V = I the output row is the probability row: non-negative, summing
    to one, and ordered like the scores (softmax is monotone)."""
    rng = np.random.default_rng(9)
    n = 12
    q, k = rng.standard_normal((n, 6)), rng.standard_normal((n, 6))
    p, _ = oracle.dense_forward(q, k, np.eye(n), 0.4)
    assert np.all(p >= 0) and np.max(np.abs(p.sum(-1) - 1)) <= 1e-15
    s = q @ k.T
    for i in range(n):
        assert np.array_equal(np.argsort(p[i], kind="stable"), np.argsort(s[i], kind="stable"))
    # and the masked entries are exactly zero
    pw, _ = oracle.dense_forward(q, k, np.eye(n), 0.4, window=3)
    assert np.array_equal(pw > 0, oracle.window_mask(n, n, 3))


def test_one_hot_limit():
    """Orthogonal, very large queries and keys: each query sees only its own key."""
    n = 6
    q = 30.0 * np.eye(n)
    v = np.arange(n * 3, dtype=float).reshape(n, 3)
    o, lse = oracle.dense_forward(q, q, v, 1.0)
    assert np.max(np.abs(o - v)) <= 1e-12
    assert np.max(np.abs(lse - 900.0)) <= 1e-12


def test_convex_hull_and_lse_bounds():
    rng = np.random.default_rng(10)
    q, k, v = (rng.standard_normal((3, 20, 7)) for _ in range(3))
    o, lse = oracle.dense_forward(q, k, v, 0.6, window=7)
    assert np.all(o <= v.max(axis=-2, keepdims=True) + 1e-15)
    assert np.all(o >= v.min(axis=-2, keepdims=True) - 1e-15)
    s = oracle.dense_scores(q, k, 0.6, 7)
    mx = s.max(-1)
    cnt = np.isfinite(s).sum(-1)
    assert np.all(lse >= mx) and np.all(lse <= mx + np.log(cnt) + 1e-15)


def test_permutation_equivariance():
    rng = np.random.default_rng(12)
    q, k, v = (rng.standard_normal((10, 5)) for _ in range(3))
    o, lse = oracle.dense_forward(q, k, v, 0.5)
    pk = rng.permutation(10)
    o2, l2 = oracle.dense_forward(q, k[pk], v[pk], 0.5)
    assert np.max(np.abs(o2 - o)) <= 1e-14 and np.max(np.abs(l2 - lse)) <= 1e-14
    pq = rng.permutation(10)
    o3, l3 = oracle.dense_forward(q[pq], k, v, 0.5)
    assert np.max(np.abs(o3 - o[pq])) <= 1e-15 and np.max(np.abs(l3 - lse[pq])) <= 1e-15


# ---------------------------------------------------------------------------
# mutation tests: plausible mistakes, planted in copies on the CPU, are caught
# ---------------------------------------------------------------------------

def _fwd_transposed(q, k, v, scale, window=0):
    s = np.matmul(np.asarray(k, float), np.swapaxes(np.asarray(q, float), -1, -2)) * scale
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    return p @ v, None


def _fwd_scale_over_d(q, k, v, scale, window=0):
    d = np.asarray(q).shape[-1]
    return oracle.dense_forward(q, k, v, 1.0 / d)


def _merge_without_rescale(m1, l1, o1, m2, l2, o2):
    m_new = np.maximum(m1, m2)
    return m_new, np.asarray(l1) + l2, np.asarray(o1) + o2


def _merge_wrong_sign(m1, l1, o1, m2, l2, o2):
    m_new = np.maximum(m1, m2)
    f1 = np.where(np.isfinite(m1), np.exp(np.where(np.isfinite(m1), m_new - m1, 0.0)), 0.0)
    f2 = np.where(np.isfinite(m2), np.exp(np.where(np.isfinite(m2), m_new - m2, 0.0)), 0.0)
    return m_new, f1 * l1 + f2 * l2, f1[..., None] * o1 + f2[..., None] * o2


def test_mutants_are_caught(golden_dir):
    g = _load(golden_dir, "notes_worked_example.json")
    tv = _load(golden_dir, "tviz_tile_replay.json")
    assert check_worked_example(oracle.dense_forward, g)
    # a query/key transposition: the worked example has Q = K, so it needs the
    # torch cross-check or the permutation test; check against the library here
    torch = pytest.importorskip("torch")
    gen = torch.Generator().manual_seed(1)
    q, k, v = (torch.randn(1, 1, 6, 4, generator=gen, dtype=torch.float64) for _ in range(3))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=0.5).numpy()
    bad, _ = _fwd_transposed(q.numpy(), k.numpy(), v.numpy(), 0.5)
    assert np.max(np.abs(bad - ref)) > 1e-3
    # the literal 1/d reading of the garbled scale
    assert not check_worked_example(_fwd_scale_over_d, g)
    # a merge that forgets to rescale, or rescales with the wrong sign
    assert replay_running_stats(oracle.merge_statistics, tv) <= 1e-14
    assert replay_running_stats(_merge_without_rescale, tv) > 1e-3
    assert replay_running_stats(_merge_wrong_sign, tv) > 1e-3
