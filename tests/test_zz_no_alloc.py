"""The allocation-free backward entry point, fa_bwd_static_workspace.

It exists for callers that cannot allocate device memory: its scratch is a
fixed array inside the library instead of a caller-provided workspace.  This
file checks, through the C ABI, that two calls in a row on different problems
give the same gradients as fa_bwd with an ordinary workspace (within the
backward bar: relative L2 <= 1e-2), so contents left in the shared array by
one call do not leak into the next.  It is named so that pytest collects it
last, and it needs no state from other test files.
"""

import numpy as np
import pytest

from exact_tiled_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _rel(a, b):
    a = a.detach().float().cpu().numpy().astype(np.float64)
    b = b.detach().float().cpu().numpy().astype(np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_static_workspace_matches_fa_bwd_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_02_gb300 import binding as fa
    dev = torch.device("cuda:0")
    for B, H, N, window, seed in ((1, 2, 700, 0, 31), (2, 1, 333, 65, 32)):
        q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, H, N, 128, "bf16", seed=seed, with_do=True))
        o, lse = fa.fa_fwd(q, k, v, window=window)
        ref = fa.fa_bwd(q, k, v, o, lse, do, window=window)
        out = tuple(torch.full_like(q, float("nan")) for _ in range(3))
        fa.fa_bwd_static_workspace(q, k, v, o, lse, do, *out, window=window)
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        for name, g, r in zip(("dq", "dk", "dv"), out, ref):
            assert torch.isfinite(g.float()).all(), name
            assert _rel(g, r) <= 1e-2, (name, B, H, N, _rel(g, r))


def test_static_workspace_refuses_oversized_problems():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_02_gb300 import binding as fa
    dev = torch.device("cuda:0")
    # B*H*N*d*4 bytes of dQ accumulator alone exceed 64 MiB: refused before any launch
    assert fa.fa_bwd_workspace_bytes(1, 16, 16384, 128) > 64 << 20
    x = torch.zeros(1, 16, 16384, 128, device=dev, dtype=torch.bfloat16)
    lse = torch.zeros(1, 16, 16384, device=dev, dtype=torch.float32)
    with pytest.raises(fa.FaError) as e:
        fa.fa_bwd_static_workspace(x, x, x, x, lse, x, x, x, x)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


def test_static_workspace_binding_checks_lse():
    """The wrapper rejects an lse of the wrong dtype, layout or size before
    the library sees it (the kernels would read past a short one)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_02_gb300 import binding as fa
    dev = torch.device("cuda:0")
    x = torch.zeros(1, 2, 256, 128, device=dev, dtype=torch.bfloat16)
    good = torch.zeros(1, 2, 256, device=dev, dtype=torch.float32)
    for bad in (good.half(), good[:, :1], torch.zeros(1, 256, 2, device=dev).transpose(1, 2)):
        with pytest.raises(ValueError):
            fa.fa_bwd_static_workspace(x, x, x, x, bad, x, x, x, x)


def test_static_workspace_in_a_cuda_graph():
    """What the entry point is for: a backward inside a captured CUDA graph
    with nothing allocated for it.  Captured once after a warm-up call,
    replayed on new inputs, it matches fa_bwd with an ordinary workspace (dK,
    dV bit for bit, dQ to rounding)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_02_gb300 import binding as fa
    dev = torch.device("cuda:0")
    B, H, N, d = 1, 2, 700, 128
    q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, H, N, d, "bf16", seed=60, with_do=True))
    o, lse = fa.fa_fwd(q, k, v)
    out = tuple(torch.empty_like(q) for _ in range(3))
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fa.fa_bwd_static_workspace(q, k, v, o, lse, do, *out)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_bwd_static_workspace(q, k, v, o, lse, do, *out)
    new = [t.to(dev) for t in inputs.make_inputs(B, H, N, d, "bf16", seed=61, with_do=True)]
    o_new, lse_new = fa.fa_fwd(*new[:3])
    for dst, src in zip((q, k, v, do, o, lse), (*new, o_new, lse_new)):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == fa.FA_OK
    ref = fa.fa_bwd(*new[:3], o_new, lse_new, new[3])
    torch.cuda.synchronize()
    assert torch.equal(out[1], ref[1]) and torch.equal(out[2], ref[2])  # dK, dV: reduced on chip
    assert _rel(out[0], ref[0]) <= 1e-3
