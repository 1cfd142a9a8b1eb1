"""GPU parity of the backward pass (recomputation) against the float64 oracle's
analytic gradients, through the C ABI.

The forward's O and lse come from the library's own forward (as in training);
the oracle differentiates the definition from Q, K, V and dO alone.  Bar:
relative L2 error <= 1e-2 for each of dQ, dK, dV.
"""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_02_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _fa():
    from exact_tiled_attention_02_gb300 import binding
    return binding


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _check_grad(name, g, r, what):
    """Relative L2 <= 1e-2; where the exact gradient is identically zero (one
    key: every softmax row is [1], so dS = 0 and dQ = dK = 0) a relative error
    is undefined and the bar is an absolute 1e-5 instead."""
    assert np.all(np.isfinite(g)), (name, what)
    if np.linalg.norm(r) == 0.0:
        assert np.max(np.abs(g)) <= 1e-5, (name, np.max(np.abs(g)), what)
    else:
        assert _rel(g, r) <= 1e-2, (name, _rel(g, r), what)


def _run(q, k, v, do, scale, window, dev):
    fa = _fa()
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = fa.fa_fwd(qd, kd, vd, scale=scale, window=window)
    dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, lse, dod, scale=scale, window=window)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    return dq, dk, dv


BWD_CASES = [
    # B, H, N, d, window, qk_mult
    (1, 1, 1, 128, 0, 1.0),
    (1, 2, 5, 128, 0, 1.0),
    (1, 1, 64, 128, 0, 1.0),
    (1, 2, 65, 128, 0, 1.0),
    (2, 1, 200, 128, 0, 1.0),
    (1, 2, 300, 128, 0, 8.0),
    (1, 1, 513, 128, 0, 1.0),
    (1, 2, 300, 128, 3, 1.0),
    (1, 1, 700, 128, 65, 1.0),
    (1, 1, 1000, 128, 257, 1.0),
    (1, 1, 640, 128, 257, 8.0),
    (1, 1, 1, 64, 0, 1.0),
    (1, 2, 65, 64, 0, 1.0),
    (2, 2, 300, 64, 0, 8.0),
    (1, 1, 513, 64, 0, 1.0),
    (1, 2, 700, 64, 65, 1.0),
    (1, 2, 300, 64, 1, 1.0),  # window 1: P = I, so dQ = dK = 0 and dV = dO
    (1, 1, 129, 64, 3, 8.0),
    # d = 64 adds -lse/scale and -D in the tensor core as three bf16 terms:
    # large logits (large lse) over many query tiles, with and without a band
    (1, 1, 2048, 64, 0, 8.0),
    (1, 1, 1500, 64, 257, 8.0),
    (1, 1, 1, 96, 0, 1.0),
    (1, 2, 200, 96, 0, 1.0),
    (1, 1, 513, 96, 0, 8.0),
    (1, 2, 700, 96, 65, 1.0),
    # bands wider than one key tile each side: each key tile meets several
    # query tiles through the band-limited loop
    (1, 1, 2000, 128, 1025, 1.0),
    (1, 2, 1500, 96, 513, 8.0),
    (1, 1, 1800, 64, 769, 1.0),
]


@pytest.mark.parametrize("B,H,N,d,window,qk", BWD_CASES)
def test_bwd_elementwise(B, H, N, d, window, qk):
    dev = _dev()
    q, k, v, do = inputs.make_inputs(B, H, N, d, "bf16", seed=3 * N + window, qk_mult=qk, with_do=True)
    scale = 1 / np.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, scale, window, dev)
    refs = oracle.dense_backward(_np(q), _np(k), _np(v), _np(do), scale, window)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        _check_grad(name, _np(g), r, (B, H, N, d, window, qk))


@pytest.mark.parametrize("d", [64, 96, 128])
def test_bwd_deterministic_dk_dv(d):
    """dK and dV of a whole key tile are reduced on chip.  The key tiles of a
    partly filled last wave run as two CTAs whose fp32 partial rows are added
    into zeroed memory, and two addends sum the same in either order.  So dK
    and dV are bitwise repeatable either way; dQ (fp32 reductions from many
    CTAs) is repeatable to rounding.  1 x 2 x 333 has 6 key tiles, so on a
    GPU with 12 or more SMs every tile is split (3 query tiles: halves of 1
    and 2)."""
    dev = _dev()
    q, k, v, do = inputs.make_inputs(1, 2, 333, d, "bf16", seed=4, with_do=True)
    a = _run(q, k, v, do, 1 / np.sqrt(d), 0, dev)
    b = _run(q, k, v, do, 1 / np.sqrt(d), 0, dev)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert _rel(_np(a[0]), _np(b[0])) <= 1e-3


def test_bwd_split_last_wave_mixed():
    """80 heads x 2 key tiles = 160 CTAs: on a 152-SM GB300 that is 152 whole
    key tiles and a last wave of 8 tiles split in two.  Every head against
    the oracle, and dK / dV bitwise repeatable."""
    dev = _dev()
    B, H, N, d = 1, 80, 256, 128
    q, k, v, do = inputs.make_inputs(B, H, N, d, "bf16", seed=21, with_do=True)
    scale = 1 / np.sqrt(d)
    a = _run(q, k, v, do, scale, 0, dev)
    b = _run(q, k, v, do, scale, 0, dev)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    refs = oracle.dense_backward(_np(q), _np(k), _np(v), _np(do), scale, 0)
    for name, g, r in zip(("dq", "dk", "dv"), a, refs):
        _check_grad(name, _np(g), r, (B, H, N, d, 0, 1.0))


@pytest.mark.parametrize("d", [64, 96, 128])
def test_bwd_guard_bands(d):
    """dQ, dK and dV are written exactly inside [B,H,N,d]: canaries around
    them stay untouched for a ragged N."""
    dev = _dev()
    fa = _fa()
    B, H, N = 1, 2, 200
    q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, H, N, d, "bf16", seed=21, with_do=True))
    o, lse = fa.fa_fwd(q, k, v)
    pad = 4096
    n = B * H * N * d
    bufs = [torch.full((2 * pad + n,), 5.0, device=dev, dtype=torch.bfloat16) for _ in range(3)]
    dq, dk, dv = (b[pad:pad + n].view(B, H, N, d) for b in bufs)
    fa.fa_bwd(q, k, v, o, lse, do, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.all(b[:pad] == 5.0) and torch.all(b[-pad:] == 5.0)
    refs = oracle.dense_backward(_np(q), _np(k), _np(v), _np(do), 1 / np.sqrt(d))
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        _check_grad(name, _np(g), r, d)


@pytest.mark.parametrize("d", [64, 96, 128])
def test_bwd_workspace_rows(d):
    """White-box check of the element-wise passes around the main kernel, on a
    workspace the caller supplies (its layout is the one fa.h documents).
    Every row's lse term is -lse log2 e (d = 64: -lse / scale) and its D term is
    -D_i = -sum_k dO_ik O_ik, computed here in float64 from the same O, lse
    and dO.  The padding rows past N hold the values that make their P (and
    so their dS) zero.  And dQ is exactly bf16(scale * accumulator).  A wrong
    term on a few rows would barely move the gradients' relative L2 error;
    here every row is checked."""
    dev = _dev()
    fa = _fa()
    B, H, N = 2, 3, 300  # Npad = 384: 84 padding rows per head
    q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, H, N, d, "bf16", seed=31, with_do=True))
    scale = 1 / np.sqrt(d)
    o, lse = fa.fa_fwd(q, k, v, scale=scale)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), device=dev, dtype=torch.uint8)
    dq, _, _ = fa.fa_bwd(q, k, v, o, lse, do, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    raw = ws.cpu().numpy()
    npad = (N + 127) // 128 * 128
    acc_bytes = (B * H * N * d * 4 + 255) // 256 * 256
    per = 16 if d == 64 else 4
    vec_bytes = (B * H * npad * per + 255) // 256 * 256

    def section(off):
        if d == 64:  # three bf16 terms and five zeros per 16-byte row
            u16 = raw[off:off + B * H * npad * 16].view(np.uint16).reshape(B * H, npad, 8)
            assert np.all(u16[..., 3:] == 0)
            terms = (u16[..., :3].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            return terms.sum(-1)
        return raw[off:off + B * H * npad * 4].view(np.float32).reshape(B * H, npad).astype(np.float64)

    lterm, dterm = section(acc_bytes), section(acc_bytes + vec_bytes)
    od, dod = _np(o).reshape(B * H, N, d), _np(do).reshape(B * H, N, d)
    want_d = -(od * dod).sum(-1)
    mag = (np.abs(od) * np.abs(dod)).sum(-1)
    L = lse.cpu().numpy().astype(np.float64).reshape(B * H, N)
    want_l = -L / np.float32(scale) if d == 64 else -L * np.log2(np.e)
    assert np.all(np.abs(lterm[:, :N] - want_l) <= 2e-6 * np.abs(want_l) + 1e-6)
    assert np.all(np.abs(dterm[:, :N] - want_d) <= 1e-5 * mag + 1e-7)
    if d == 64:
        assert np.all(np.abs(lterm[:, N:] + 1e30) <= 1e-6 * 1e30)
    else:
        assert np.all(lterm[:, N:] == -np.inf)
    assert np.all(dterm[:, N:] == 0.0)
    acc = torch.from_numpy(raw[:B * H * N * d * 4].view(np.float32).reshape(B, H, N, d).copy())
    assert torch.equal((acc * np.float32(scale)).to(torch.bfloat16), dq.cpu())


@pytest.mark.parametrize("d", [64, 96])
def test_bwd_large_sampled_heads(d):
    """d = 64 and 96 at a size with many key and query tiles (B=2, H=8,
    N=2048), two whole heads against the oracle."""
    dev = _dev()
    q, k, v, do = inputs.make_inputs(2, 8, 2048, d, "bf16", seed=d, with_do=True)
    dq, dk, dv = _run(q, k, v, do, 1 / np.sqrt(d), 0, dev)
    for b, h in ((0, 0), (1, 7)):
        refs = oracle.dense_backward(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), _np(do[b, h]), 1 / np.sqrt(d))
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), refs):
            assert _rel(_np(g), r) <= 1e-2, (name, b, h, _rel(_np(g), r))


def test_workload5_full_size_sampled_heads():
    """The full-size backward workload, launched as the bench launches it:
    three whole heads against the oracle, plus identities of the exact
    gradient over every head."""
    dev = _dev()
    w = configs.WORKLOADS[5]
    q, k, v, do = inputs.workload_inputs(w, with_do=True)
    dq, dk, dv = _run(q, k, v, do, w.scale, w.window, dev)
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()
    rng = np.random.default_rng(5)
    heads = [(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))]
    for b, h in heads:
        refs = oracle.dense_backward(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), _np(do[b, h]), w.scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), refs):
            assert _rel(_np(g), r) <= 1e-2, (name, b, h, _rel(_np(g), r))
    # sum over keys of dK vanishes; sum over keys of dV equals the sum over queries of dO
    sk = dk.float().sum(dim=2)
    assert float(sk.abs().max()) <= 2e-2 * float(dk.float().abs().sum(dim=2).max())
    sv = dv.float().sum(dim=2)
    sdo = do.to(dev).float().sum(dim=2)
    assert float((sv - sdo).norm() / sdo.norm()) <= 1e-2


def test_workload2_full_size_sampled_heads():
    """Workload 2 (d = 64) at full size, launched as the bench launches it:
    three whole heads against the oracle, plus identities of the exact
    gradient over every head."""
    dev = _dev()
    w = configs.WORKLOADS[2]
    q, k, v, do = inputs.workload_inputs(w, with_do=True)
    dq, dk, dv = _run(q, k, v, do, w.scale, w.window, dev)
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()
    rng = np.random.default_rng(2)
    heads = [(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))]
    for b, h in heads:
        refs = oracle.dense_backward(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), _np(do[b, h]), w.scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), refs):
            assert _rel(_np(g), r) <= 1e-2, (name, b, h, _rel(_np(g), r))
    # sum over keys of dK vanishes; sum over keys of dV equals the sum over queries of dO
    sk = dk.float().sum(dim=2)
    assert float(sk.abs().max()) <= 2e-2 * float(dk.float().abs().sum(dim=2).max())
    sv = dv.float().sum(dim=2)
    sdo = do.to(dev).float().sum(dim=2)
    assert float((sv - sdo).norm() / sdo.norm()) <= 1e-2


def test_workload3_backward_full_size_heads():
    """The bench's own backward (workload 3: N = 8192, d = 128, Q,K x8, so
    large logits), launched as the bench launches it: two whole heads
    against the oracle, plus finiteness everywhere."""
    dev = _dev()
    w = configs.WORKLOADS[3]
    q, k, v, do = inputs.workload_inputs(w, with_do=True)
    dq, dk, dv = _run(q, k, v, do, w.scale, w.window, dev)
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        refs = oracle.dense_backward(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), _np(do[b, h]), w.scale)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), refs):
            assert _rel(_np(g), r) <= 1e-2, (name, b, h, _rel(_np(g), r))


def test_workload4_backward_full_size_slices():
    """Workload 4 (N = 16384, window 257) at full size.  With a band of radius
    r, dQ of query i needs keys within r of i, and dK, dV of key j need the
    rows within r of j, whose lse and D need keys within 2r of j; so the
    oracle's gradients of a slice [s, e) of the sequence are exact for queries
    in [s + r, e - r) and keys in [s + 2r, e - 2r) (no margin at the
    sequence's own ends).  Three slices of two heads are checked."""
    dev = _dev()
    w = configs.WORKLOADS[4]
    r = (w.window - 1) // 2
    q, k, v, do = inputs.workload_inputs(w, with_do=True)
    dq, dk, dv = _run(q, k, v, do, w.scale, w.window, dev)
    for g in (dq, dk, dv):
        assert torch.isfinite(g.float()).all()
    n = w.N
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        for s0, e0 in ((0, 1024), (n // 2 - 512, n // 2 + 512), (n - 1024, n)):
            refs = oracle.dense_backward(_np(q[b, h, s0:e0]), _np(k[b, h, s0:e0]), _np(v[b, h, s0:e0]),
                                         _np(do[b, h, s0:e0]), w.scale, w.window)
            qa, qb = (s0 + r if s0 > 0 else s0), (e0 - r if e0 < n else e0)
            ka, kb = (s0 + 2 * r if s0 > 0 else s0), (e0 - 2 * r if e0 < n else e0)
            for name, g, ref, (a, z) in zip(("dq", "dk", "dv"), (dq, dk, dv), refs, ((qa, qb), (ka, kb), (ka, kb))):
                got = _np(g[b, h, a:z])
                want = ref[a - s0:z - s0]
                assert _rel(got, want) <= 1e-2, (name, b, h, s0, _rel(got, want))


def test_bwd_unsupported_requests():
    dev = _dev()
    fa = _fa()
    x = torch.zeros(1, 1, 8, 80, device=dev, dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 8, device=dev, dtype=torch.float32)
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd(x, x, x, x, lse, x)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED  # bf16 head dimensions are 64, 96 and 128
    z = torch.zeros(1, 1, 8, 256, device=dev, dtype=torch.bfloat16)
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd(z, z, z, z, lse, z)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED  # d = 256 has a forward only
    y = torch.zeros(1, 1, 8, 132, device=dev, dtype=torch.float32)
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd(y, y, y, y, lse, y)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED  # float32 head dimensions are 1..128


# float32 backward (CUDA cores, accurate expf).  Each gradient element is a
# sum of at most N + d fp32 products, so its rounding error is of the order
# sqrt(N + d) * 2^-24 relative to the sum of the magnitudes (worst case
# (N + d) * 2^-24 = 6e-5 at N + d = 1000).  Bar: relative L2 <= 2e-5 per
# gradient; an exactly zero gradient (N = 1) within 1e-6 absolute.
F32_BWD_CASES = [
    # B, H, N, d, window
    (1, 1, 1, 4, 0), (1, 2, 5, 4, 0), (2, 1, 33, 17, 0), (1, 3, 100, 64, 0), (1, 1, 77, 128, 0),
    (1, 2, 50, 8, 3), (1, 1, 200, 32, 65), (2, 2, 129, 4, 257), (1, 1, 600, 128, 0),
    (1, 1, 130, 65, 0), (1, 2, 300, 96, 0), (1, 1, 1000, 127, 129),
]


def _check_f32_grad(name, g, r, what):
    assert np.all(np.isfinite(g)), (name, what)
    if np.linalg.norm(r) == 0.0:
        assert np.max(np.abs(g)) <= 1e-6, (name, np.max(np.abs(g)), what)
    else:
        assert _rel(g, r) <= 2e-5, (name, _rel(g, r), what)


@pytest.mark.parametrize("B,H,N,d,window", F32_BWD_CASES)
def test_bwd_f32_elementwise(B, H, N, d, window):
    dev = _dev()
    q, k, v, do = inputs.make_inputs(B, H, N, d, "f32", seed=11 * N + d + window, with_do=True)
    scale = 1 / np.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, scale, window, dev)
    refs = oracle.dense_backward(_np(q), _np(k), _np(v), _np(do), scale, window)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        _check_f32_grad(name, _np(g), r, (B, H, N, d, window))


def test_bwd_f32_workload1_and_repeatable():
    """The float32 [1, 1, 6, 4] workload with a dO drawn after q, k, v from
    the same generator; no atomics anywhere, so two runs agree bit for bit."""
    dev = _dev()
    w = configs.WORKLOADS[1]
    q, k, v, do = inputs.workload_inputs(w, with_do=True)
    a = _run(q, k, v, do, w.scale, w.window, dev)
    b = _run(q, k, v, do, w.scale, w.window, dev)
    refs = oracle.dense_backward(_np(q), _np(k), _np(v), _np(do), w.scale, w.window)
    for name, g, g2, r in zip(("dq", "dk", "dv"), a, b, refs):
        assert torch.equal(g, g2), name
        assert np.abs(_np(g) - r).max() <= 1e-5, (name, np.abs(_np(g) - r).max())
