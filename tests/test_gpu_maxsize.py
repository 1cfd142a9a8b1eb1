"""GPU parity beyond 32-bit element offsets: B*H*N*d just over 2^31 per
tensor, forward and backward through the C ABI, in bf16 at every head
dimension, with and without a window (4 GB per tensor, about 45 GB on the
device; d = 256 forward only) and in float32 on both float32 forward paths (8.6 GB per tensor).

Heads at the start, middle and end of the batch are compared with the
float64 oracle (O, lse, dQ, dK, dV), and every output is checked finite.  An
offset computed in 32 bits anywhere would put the last heads' rows in the
wrong place or read the wrong rows.

Inputs: 64 seeded heads from the shared input generator.  Head h of the large
problem is base head h mod 64, rotated by h // 64 positions along the sequence,
so every head differs.  The oracle rebuilds the sampled heads on the CPU from
the same base.
"""

import numpy as np
import pytest

import oracle
from exact_tiled_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N = 256
BASE_HEADS = 64


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("d,window", [(64, 0), (96, 0), (128, 0), (128, 257), (256, 0)])
def test_more_than_2_31_elements_per_tensor(d, window):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_02_gb300 import binding as fa
    dev = torch.device("cuda:0")
    H = (1 << 31) // (N * d) + 1  # B*H*N*d = 2^31 + N*d
    base = inputs.make_inputs(1, BASE_HEADS, N, d, "bf16", seed=77, with_do=True)

    hs = torch.arange(H, device=dev)
    idx = (torch.arange(N, device=dev)[None, :] - (hs // BASE_HEADS)[:, None]) % N

    def expand(t):
        return t[0].to(dev)[(hs % BASE_HEADS)[:, None], idx].unsqueeze(0)

    def head(t, h):
        return torch.roll(t[0, h % BASE_HEADS], shifts=h // BASE_HEADS, dims=0)

    q, k, v, do = (expand(t) for t in base)
    assert q.numel() > (1 << 31)
    scale = 1 / np.sqrt(d)
    with_bwd = d != 256  # bf16 d = 256 is forward only
    o, lse = fa.fa_fwd(q, k, v, scale=scale, window=window)
    grads = fa.fa_bwd(q, k, v, o, lse, do, scale=scale, window=window) if with_bwd else ()
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for t in (o, lse, *grads):
        assert bool(torch.isfinite(t).all())
    for h in (0, H // 2, H - 1):
        qh, kh, vh, doh = (_np(head(t, h)) for t in base)
        o_ref, lse_ref = oracle.dense_forward(qh, kh, vh, scale, window)
        err = np.abs(_np(o[0, h]) - o_ref)
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (h, err.max(), err.mean())
        assert np.abs(lse[0, h].cpu().numpy().astype(np.float64) - lse_ref).max() <= 1e-3, h
        if with_bwd:
            refs = oracle.dense_backward(qh, kh, vh, doh, scale, window)
            for name, g, r in zip(("dq", "dk", "dv"), (t[0, h] for t in grads), refs):
                assert _rel(_np(g), r) <= 1e-2, (name, h, _rel(_np(g), r))
    del q, k, v, do, o, lse, grads, idx, hs
    torch.cuda.empty_cache()


def test_f32_more_than_2_31_elements_per_tensor():
    """The float32 paths at B*H*N*d = 2^31 + N*d (8.6 GB per tensor, about
    120 GB on the device at the peak): the exact CUDA-core forward and
    backward, then the 3xTF32 tensor-core forward with its split copies.
    Bars as for float32 everywhere: max-abs 1e-5 on O and lse, relative L2
    2e-5 on each gradient."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_02_gb300 import binding as fa
    dev = torch.device("cuda:0")
    d = 128
    H = (1 << 31) // (N * d) + 1
    base = inputs.make_inputs(1, BASE_HEADS, N, d, "f32", seed=78, with_do=True)
    hs = torch.arange(H, device=dev)
    idx = (torch.arange(N, device=dev)[None, :] - (hs // BASE_HEADS)[:, None]) % N

    def expand(t):
        return t[0].to(dev)[(hs % BASE_HEADS)[:, None], idx].unsqueeze(0)

    def head(t, h):
        return torch.roll(t[0, h % BASE_HEADS], shifts=h // BASE_HEADS, dims=0)

    q, k, v, do = (expand(t) for t in base)
    assert q.numel() > (1 << 31)
    scale = 1 / np.sqrt(d)
    sampled = (0, H // 2, H - 1)
    refs = {}
    for h in sampled:
        qh, kh, vh, doh = (_np(head(t, h)) for t in base)
        refs[h] = (oracle.dense_forward(qh, kh, vh, scale), oracle.dense_backward(qh, kh, vh, doh, scale))

    o, lse = fa.fa_fwd(q, k, v, scale=scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, do, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    for h in sampled:
        (o_ref, lse_ref), grads = refs[h]
        assert np.abs(_np(o[0, h]) - o_ref).max() <= 1e-5, h
        assert np.abs(_np(lse[0, h]) - lse_ref).max() <= 1e-5, h
        for name, g, r in zip(("dq", "dk", "dv"), (dq[0, h], dk[0, h], dv[0, h]), grads):
            assert _rel(_np(g), r) <= 2e-5, (name, h, _rel(_np(g), r))
    del dq, dk, dv, o, lse
    torch.cuda.empty_cache()

    o, lse = fa.fa_fwd_f32_3xtf32(q, k, v, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    for h in sampled:
        (o_ref, lse_ref), _ = refs[h]
        assert np.abs(_np(o[0, h]) - o_ref).max() <= 1e-5, h
        assert np.abs(_np(lse[0, h]) - lse_ref).max() <= 1e-5, h
    del q, k, v, do, o, lse, idx, hs
    torch.cuda.empty_cache()
