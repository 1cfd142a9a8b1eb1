"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every function include/fa.h declares, and rejects invalid requests on the host
before any CUDA call (so these calls are safe with fake, never-dereferenced
pointers)."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fa.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def b():
    from exact_tiled_attention_02_gb300 import binding
    return binding


def test_library_loads_and_exports_header_symbols(b):
    names = _declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names
    for n in names:
        assert hasattr(b.lib, n), n
    assert set(names) <= set(b.EXPORTS) | set(names)
    assert set(b.EXPORTS) == set(names)


def test_version_and_strings(b):
    assert b.fa_version() >= 100
    for s in range(5):
        assert b.fa_status_string(s).startswith("FA_")
    assert "unknown" in b.fa_status_string(99)


def test_workspace_size(b):
    assert b.fa_bwd_workspace_bytes(0, 1, 1, 1) == 0
    n = b.fa_bwd_workspace_bytes(4, 16, 4096, 128)
    rows = 4 * 16 * 4096
    assert n >= rows * 128 * 4 + rows * 4 and n % 256 == 0
    # dQ accumulator (15 floats -> 256 B), lse2 and D (128 padded rows each -> 512 B)
    assert b.fa_bwd_workspace_bytes(1, 1, 3, 5) == 256 + 512 + 512
    # d = 128: dV and dK partial rows of the 2 * 2 key tiles follow
    assert b.fa_bwd_workspace_bytes(2, 1, 129, 128) == 2 * 129 * 128 * 4 + 2 * (2 * 256 * 4) + 4 * 2 * 128 * 128 * 4
    assert b.fa_bwd_workspace_bytes(1, 1, 128, 96) == 128 * 96 * 4 + 2 * 512 + 1 * 2 * 128 * 96 * 4
    # ... for at most 128 key tiles
    assert b.fa_bwd_workspace_bytes(4, 16, 4096, 128) == 4 * 16 * 4096 * (128 * 4 + 2 * 4) + 128 * 2 * 128 * 128 * 4
    # d = 64: 16 bytes per padded row in the two row arrays
    assert b.fa_bwd_workspace_bytes(2, 1, 129, 64) == 2 * 129 * 64 * 4 + 2 * (2 * 256 * 16) + 4 * 2 * 128 * 64 * 4
    # other head dimensions (fp32 only): no partial rows
    assert b.fa_bwd_workspace_bytes(2, 1, 129, 32) == 2 * 129 * 32 * 4 + 2 * (2 * 256 * 4)


def test_wait_limit_roundtrip(b):
    old = b.fa_set_wait_limit_us(12345)
    assert b.fa_set_wait_limit_us(old) == 12345
    assert b.fa_set_wait_limit_us(0) == old  # <= 0 restores the default
    b.fa_set_wait_limit_us(old)


P = 1 << 20  # a fake, 16-byte-aligned pointer value; never dereferenced


def fwd(b, q=P, k=P, v=P, o=P, lse=0, B=1, H=1, N=8, d=64, scale=0.125, window=0, dt=1):
    vp = ctypes.c_void_p
    return b.lib.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, N, d, scale, window, dt, vp(0))


def bwd(b, ws=P, ws_bytes=1 << 30, dt=1, d=128, N=8, window=0, lse=P, scale=0.1):
    vp = ctypes.c_void_p
    return b.lib.fa_bwd(vp(P), vp(P), vp(P), vp(P), vp(lse), vp(P), vp(P), vp(P), vp(P), 1, 1, N, d, scale, window,
                        dt, vp(ws), ws_bytes, vp(0))


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1),
    (dict(q=P + 8), 1), (dict(o=P + 2), 1), (dict(lse=P + 2), 1),
    (dict(B=0), 1), (dict(H=-1), 1), (dict(N=0), 1), (dict(d=0), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(window=4), 1), (dict(window=256), 1), (dict(dt=7), 1),
    (dict(d=80), 2), (dict(d=32), 2), (dict(d=192), 2), (dict(d=512), 2), (dict(dt=0, d=129), 2),
])
def test_fwd_rejects_on_host(b, kw, code):
    assert fwd(b, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), 1), (dict(ws=P + 16), 1), (dict(ws_bytes=100), 1), (dict(lse=0), 1),
    (dict(window=2), 1), (dict(scale=0.0), 1), (dict(d=80), 2), (dict(d=256), 2), (dict(d=32), 2), (dict(dt=0, d=129), 2),
])
def test_bwd_rejects_on_host(b, kw, code):
    assert bwd(b, **kw) == code


def bwd_static(b, q=P, lse=P, dt=1, B=1, H=1, N=8, d=128, window=0, scale=0.1):
    vp = ctypes.c_void_p
    return b.lib.fa_bwd_static_workspace(vp(q), vp(P), vp(P), vp(P), vp(lse), vp(P), vp(P), vp(P), vp(P), B, H, N, d,
                                         scale, window, dt, vp(0))


BIG = dict(B=4, H=16, N=16384)  # needs far more than the 64 MiB static scratch


@pytest.mark.parametrize("kw,code", [
    # invalid arguments get fa_bwd's status whatever the problem's size
    (dict(q=0, **BIG), 1), (dict(lse=0, **BIG), 1), (dict(q=P + 8, **BIG), 1), (dict(dt=7, **BIG), 1),
    (dict(window=4, **BIG), 1), (dict(scale=0.0, **BIG), 1), (dict(B=0), 1),
    (dict(q=0), 1), (dict(dt=7), 1),
    # backward not implemented for these head dimensions, whatever the size
    (dict(d=256, **BIG), 2), (dict(d=80, **BIG), 2), (dict(d=256), 2),
    # valid arguments, workspace larger than the static scratch: refused before any device access
    (dict(**BIG), 2), (dict(dt=0, d=100, **BIG), 2),
])
def test_bwd_static_workspace_rejects_on_host(b, kw, code):
    assert bwd_static(b, **kw) == code


def km(b, ws=P, ws_bytes=1 << 30, dt=1, d=128, N=8, window=0, scale=0.1, o=P):
    vp = ctypes.c_void_p
    return b.lib.fa_fwd_key_major(vp(P), vp(P), vp(P), vp(o), vp(0), 1, 1, N, d, scale, window, dt, vp(ws), ws_bytes,
                                  vp(0))


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), 1), (dict(ws=P + 16), 1), (dict(ws_bytes=100), 1), (dict(o=0), 1), (dict(o=P + 4), 1),
    (dict(window=2), 1), (dict(scale=0.0), 1), (dict(d=96), 2), (dict(d=256), 2), (dict(dt=0, d=64), 2),
])
def test_key_major_rejects_on_host(b, kw, code):
    assert km(b, **kw) == code


def test_key_major_workspace_size(b):
    assert b.fa_fwd_key_major_workspace_bytes(1, 0, 1, 1) == 0
    # O~ (2 * 129 rows x 128 fp32), then m and l (258 floats -> 1280 B each)
    assert b.fa_fwd_key_major_workspace_bytes(2, 1, 129, 128) == 2 * 129 * 128 * 4 + 2 * 1280


def tf(b, ws=P, ws_bytes=1 << 30, d=64, N=8, window=0, scale=0.1, o=P, lse=0):
    vp = ctypes.c_void_p
    return b.lib.fa_fwd_f32_3xtf32(vp(P), vp(P), vp(P), vp(o), vp(lse), 1, 1, N, d, scale, window, vp(ws), ws_bytes,
                                   vp(0))


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), 1), (dict(ws=P + 16), 1), (dict(ws_bytes=100), 1), (dict(o=0), 1), (dict(o=P + 4), 1),
    (dict(lse=P + 2), 1), (dict(window=2), 1), (dict(scale=0.0), 1), (dict(N=0), 1), (dict(d=129), 2),
    (dict(d=256), 2),
])
def test_3xtf32_rejects_on_host(b, kw, code):
    assert tf(b, **kw) == code


def test_3xtf32_workspace_size(b):
    assert b.fa_fwd_f32_3xtf32_workspace_bytes(1, 1, 0, 8) == 0
    # Q, K hi/lo: 4 x (2*100 rows x 64 fp32); V^T hi/lo: 2 x (2 x 64 x 128 fp32), each rounded to 256 B
    rows = (2 * 100 * 64 * 4 + 255) // 256 * 256
    vt = 2 * 64 * 128 * 4
    assert b.fa_fwd_f32_3xtf32_workspace_bytes(2, 1, 100, 16) == 4 * rows + 2 * vt
    # 64 < d <= 128: K hi/lo rows of 128 and V^T hi/lo with 128 rows; Q is split in the kernel
    rows = (2 * 100 * 128 * 4 + 255) // 256 * 256
    vt = 2 * 128 * 128 * 4
    assert b.fa_fwd_f32_3xtf32_workspace_bytes(2, 1, 100, 100) == 2 * rows + 2 * vt


def test_selftest_rejects_bad_limit(b):
    assert b.lib.fa_selftest_wait_timeout(0, ctypes.c_void_p(0)) == 1
    assert b.lib.fa_selftest_wait_timeout(100001, ctypes.c_void_p(0)) == 1


def test_workloads_and_inputs():
    from exact_tiled_attention_02_gb300 import configs, inputs
    w = configs.WORKLOADS
    assert [w[i].N for i in range(1, 6)] == [6, 2048, 8192, 16384, 4096]
    assert w[4].pairs_per_head() == 257 * 16384 - 128 * 129 == 4194176
    small = configs.Workload(9, "t", 1, 1, 300, 8, "bf16", window=65)
    r = 32
    assert small.pairs_per_head() == sum(min(299, i + r) - max(0, i - r) + 1 for i in range(300))
    assert w[3].fwd_flops() == 4.0 * 2 * 16 * 8192 * 8192 * 128
    q, k, v = inputs.workload_inputs(w[1])
    assert q.shape == (1, 1, 6, 4) and str(q.dtype) == "torch.float32"
    q2, _, _ = inputs.workload_inputs(w[1])
    assert (q == q2).all()
    q, k, v, do = inputs.make_inputs(1, 2, 5, 64, "bf16", seed=3, qk_mult=8.0, with_do=True)
    assert str(q.dtype) == "torch.bfloat16" and do.shape == (1, 2, 5, 64)
