"""GPU parity of the float32 tensor-core forward (3xTF32 split) against the
float64 oracle, through the C ABI.  Bar: the float32 bar, max-abs 1e-5 on O and
on lse.  Derivation: each product keeps 22 significant bits of each operand
and drops terms below 2^-21 relative; with |q_c k_c| = O(1), d <= 128 and
scale = 1/sqrt(d), S is off by at most 2^-21 sum_c |q_c k_c| scale (a few
1e-6 at d = 128, typically a few 1e-7) and P by as much relative, and O (a
convex combination of V rows, |V| = O(1)) by about 1e-6.  d <= 64 and
64 < d <= 128 run different kernels (Q in shared memory, or split into
tensor memory), so both ranges are covered."""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_02_gb300 import inputs

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
    return t.detach().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,H,N,d,window", [
    (1, 1, 1, 4, 0), (1, 2, 5, 4, 0), (2, 1, 33, 17, 0), (1, 3, 100, 64, 0), (1, 1, 129, 64, 0),
    (1, 2, 50, 8, 3), (1, 1, 300, 32, 65), (2, 2, 129, 4, 257), (1, 1, 1000, 64, 0), (1, 2, 777, 48, 129),
    # 64 < d <= 128: one tile, ragged tails, head dimensions that are not a
    # multiple of 4, windows across several 64-key tiles
    (1, 1, 1, 65, 0), (1, 2, 5, 128, 0), (2, 1, 129, 100, 0), (1, 3, 300, 128, 0), (1, 1, 1000, 96, 0),
    (1, 2, 200, 127, 3), (1, 1, 700, 128, 129), (2, 2, 333, 80, 65), (1, 1, 2048, 128, 0),
])
def test_3xtf32_elementwise(B, H, N, d, window):
    dev = _dev()
    q, k, v = inputs.make_inputs(B, H, N, d, "f32", seed=7 * N + d + window)
    o, lse = _fa().fa_fwd_f32_3xtf32(q.to(dev), k.to(dev), v.to(dev), window=window)
    torch.cuda.synchronize()
    assert _fa().fa_last_device_status() == 0
    o_ref, lse_ref = oracle.dense_forward(_np(q), _np(k), _np(v), 1 / np.sqrt(d), window)
    assert np.abs(_np(o) - o_ref).max() <= 1e-5, np.abs(_np(o) - o_ref).max()
    assert np.abs(_np(lse) - lse_ref).max() <= 1e-5, np.abs(_np(lse) - lse_ref).max()


def test_3xtf32_large_sampled_and_guard_bands():
    """B=2, H=4, N=4096, d=64: sampled rows of every head against the oracle;
    canaries around O and lse stay untouched."""
    dev = _dev()
    B, H, N, d = 2, 4, 4096, 64
    q, k, v = (t.to(dev) for t in inputs.make_inputs(B, H, N, d, "f32", seed=64))
    pad = 4096
    obuf = torch.full((2 * pad + B * H * N * d,), 7.0, device=dev, dtype=torch.float32)
    lbuf = torch.full((2 * pad + B * H * N,), -3.0, device=dev, dtype=torch.float32)
    o = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    _fa().fa_fwd_f32_3xtf32(q, k, v, o=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[-pad:] == 7.0)
    assert torch.all(lbuf[:pad] == -3.0) and torch.all(lbuf[-pad:] == -3.0)
    rng = np.random.default_rng(4096)
    for b in range(B):
        for h in range(H):
            rows = np.sort(rng.choice(N, 24, replace=False))
            o_ref, lse_ref = oracle.dense_forward_rows(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), 0.125, rows)
            assert np.abs(_np(o[b, h, rows]) - o_ref).max() <= 1e-5
            assert np.abs(_np(lse[b, h, rows]) - lse_ref).max() <= 1e-5


def test_3xtf32_d128_large_sampled_and_guard_bands():
    """B=2, H=8, N=4096, d=128 (many CTAs, 64 key tiles each): sampled rows of
    every head against the oracle; canaries around O and lse stay untouched."""
    dev = _dev()
    B, H, N, d = 2, 8, 4096, 128
    q, k, v = (t.to(dev) for t in inputs.make_inputs(B, H, N, d, "f32", seed=128))
    pad = 4096
    obuf = torch.full((2 * pad + B * H * N * d,), 7.0, device=dev, dtype=torch.float32)
    lbuf = torch.full((2 * pad + B * H * N,), -3.0, device=dev, dtype=torch.float32)
    o = obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = lbuf[pad:pad + B * H * N].view(B, H, N)
    _fa().fa_fwd_f32_3xtf32(q, k, v, o=o, lse=lse)
    torch.cuda.synchronize()
    assert _fa().fa_last_device_status() == 0
    assert torch.all(obuf[:pad] == 7.0) and torch.all(obuf[-pad:] == 7.0)
    assert torch.all(lbuf[:pad] == -3.0) and torch.all(lbuf[-pad:] == -3.0)
    rng = np.random.default_rng(128)
    for b in range(B):
        for h in range(H):
            rows = np.sort(np.concatenate([[0, 127, 128, N - 1], rng.choice(N, 20, replace=False)]))
            o_ref, lse_ref = oracle.dense_forward_rows(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), 1 / np.sqrt(d),
                                                       rows)
            assert np.abs(_np(o[b, h, rows]) - o_ref).max() <= 1e-5
            assert np.abs(_np(lse[b, h, rows]) - lse_ref).max() <= 1e-5


def test_3xtf32_agrees_with_cuda_core_path_d128():
    """The two float32 paths at d = 128 on one problem: both within 1e-5 of
    the oracle, so within 2e-5 of each other everywhere."""
    dev = _dev()
    q, k, v = (t.to(dev) for t in inputs.make_inputs(1, 4, 1500, 128, "f32", seed=1500))
    o1, l1 = _fa().fa_fwd_f32_3xtf32(q, k, v, window=257)
    o2, l2 = _fa().fa_fwd(q, k, v, window=257)
    torch.cuda.synchronize()
    assert float((o1 - o2).abs().max()) <= 2e-5
    assert float((l1 - l2).abs().max()) <= 2e-5


def test_3xtf32_rejects():
    dev = _dev()
    fa = _fa()
    x = torch.zeros(1, 1, 8, 129, device=dev, dtype=torch.float32)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_f32_3xtf32(x, x, x)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    y = torch.zeros(1, 1, 8, 64, device=dev, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.fa_fwd_f32_3xtf32(y, y, y)
