"""The library inside a CUDA graph.

A forward and a backward (caller-owned outputs and workspace) are captured
once into a ``torch.cuda.CUDAGraph`` and replayed with new inputs copied into
the captured buffers.  Every replay must give what eager calls give on the
same inputs: O, lse, dK and dV bit for bit, dQ (summed by reductions in any
order) to rounding.  The host work of a call (argument checks, tensor maps)
happens at capture; a replay only launches the kernels.
"""

import pytest

from exact_tiled_attention_02_gb300 import inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("window", [0, 257])
def test_forward_and_backward_replay_in_a_graph(window):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_tiled_attention_02_gb300 import binding as fa
    dev = torch.device("cuda:0")
    B, H, N, d = 1, 4, 700, 128
    q, k, v, do = (t.to(dev) for t in inputs.make_inputs(B, H, N, d, "bf16", seed=50, with_do=True))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), device=dev, dtype=torch.uint8)

    def step():
        fa.fa_fwd(q, k, v, window=window, o=o, lse=lse)
        fa.fa_bwd(q, k, v, o, lse, do, window=window, dq=dq, dk=dk, dv=dv, workspace=ws)

    side = torch.cuda.Stream(device=dev)  # warm up off the capturing stream, as torch recommends
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (51, 52):
        new = [t.to(dev) for t in inputs.make_inputs(B, H, N, d, "bf16", seed=seed, with_do=True)]
        for dst, src in zip((q, k, v, do), new):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        o_ref, lse_ref = fa.fa_fwd(*new[:3], window=window)
        dq_ref, dk_ref, dv_ref = fa.fa_bwd(*new[:3], o_ref, lse_ref, new[3], window=window)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), seed
        assert torch.equal(dk, dk_ref) and torch.equal(dv, dv_ref), seed
        assert float((dq.float() - dq_ref.float()).norm() / dq_ref.float().norm()) <= 1e-3, seed
