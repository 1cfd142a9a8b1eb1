"""GPU parity of the key-major forward schedule (the comparison schedule) against
the float64 oracle, through the C ABI.  Same bars as the query-major bf16
forward: O max-abs 2e-2 and mean-abs 2e-3; lse max-abs 1e-3."""

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


def _check(o, lse, o_ref, lse_ref, what):
    err = np.abs(_np(o) - o_ref)
    assert np.all(np.isfinite(_np(o))), what
    assert err.max() <= 2e-2, (what, err.max())
    assert err.mean() <= 2e-3, (what, err.mean())
    le = np.abs(_np(lse) - lse_ref)
    assert le.max() <= 1e-3, (what, le.max())


@pytest.mark.parametrize("B,H,N,d,window,qk", [
    (1, 1, 1, 128, 0, 1.0), (1, 2, 7, 64, 0, 1.0), (2, 1, 129, 128, 0, 1.0), (1, 2, 513, 64, 0, 8.0),
    (1, 1, 1000, 128, 0, 8.0), (1, 2, 300, 128, 3, 1.0), (1, 1, 700, 64, 65, 1.0), (1, 1, 640, 128, 257, 8.0),
    (1, 1, 257, 128, 513, 1.0),
])
def test_key_major_elementwise(B, H, N, d, window, qk):
    dev = _dev()
    q, k, v = inputs.make_inputs(B, H, N, d, "bf16", seed=5 * N + d + window, qk_mult=qk)
    o, lse = _fa().fa_fwd_key_major(q.to(dev), k.to(dev), v.to(dev), window=window)
    torch.cuda.synchronize()
    assert _fa().fa_last_device_status() == 0
    o_ref, lse_ref = oracle.dense_forward(_np(q), _np(k), _np(v), 1 / np.sqrt(d), window)
    _check(o, lse, o_ref, lse_ref, (B, H, N, d, window, qk))


def test_key_major_workload3_sampled_and_agrees_with_query_major():
    """Workload 3's full size: sampled rows against the oracle, and every
    output within the bf16 bar of the query-major kernel's."""
    dev = _dev()
    w = configs.WORKLOADS[3]
    q, k, v = inputs.workload_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = _fa().fa_fwd_key_major(qd, kd, vd, scale=w.scale)
    o2, lse2 = _fa().fa_fwd(qd, kd, vd, scale=w.scale)
    torch.cuda.synchronize()
    assert _fa().fa_last_device_status() == 0
    assert float((o.float() - o2.float()).abs().max()) <= 4e-2
    assert float((lse - lse2).abs().max()) <= 2e-3
    rng = np.random.default_rng(33)
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        rows = np.sort(rng.choice(w.N, 48, replace=False))
        o_ref, lse_ref = oracle.dense_forward_rows(_np(q[b, h]), _np(k[b, h]), _np(v[b, h]), w.scale, rows)
        _check(o[b, h, rows], lse[b, h, rows], o_ref, lse_ref, (b, h))


def test_key_major_rejects():
    dev = _dev()
    fa = _fa()
    x = torch.zeros(1, 1, 8, 96, device=dev, dtype=torch.bfloat16)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_key_major(x, x, x)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    y = torch.zeros(1, 1, 8, 64, device=dev, dtype=torch.bfloat16)
    ws = torch.empty(16, device=dev, dtype=torch.uint8)
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_key_major(y, y, y, workspace=ws)
    assert e.value.status == fa.FA_ERR_INVALID
