"""Host-side checks of the C ABI (no GPU): the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything.

The device pointers here are fake addresses. Every call must stop at argument validation or at
an empty-shape early return, so that none reaches a launch or a copy even where a GPU is
present: a call that passed validation would hand the fake address to a kernel."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_io_aware_fa_gb300 import build
    build.build()
    from exact_io_aware_fa_gb300 import api
    return api.library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_expected_api():
    from exact_io_aware_fa_gb300 import api
    assert set(header_functions()) == set(api.EXPORTS)


def test_library_exports_every_header_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    from exact_io_aware_fa_gb300 import api
    assert api.status_string(0) == "FA_OK"
    assert api.status_string(3) == "FA_ERR_ALIGNMENT"
    assert api.status_string(99) == "FA_ERR_UNKNOWN"


A = 1 << 20  # a fake, 16-byte-aligned device address: never dereferenced by these checks


def fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_forward(q, k, v, o, lse, B, H, N, d, causal, scale, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), 1), (dict(H=-2), 1), (dict(N=-5), 1),
    (dict(causal=2), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(d=32), 2), (dict(d=96), 2), (dict(d=256), 2),
    (dict(q=0), 1), (dict(lse=0), 1),
    (dict(q=A + 8), 3), (dict(o=A + 2), 3), (dict(lse=A + 2), 3),
])
def test_forward_rejects(lib, kw, status):
    assert fwd(lib, **kw) == status


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(N=0), dict(N=0, q=0, k=0, v=0, o=0, lse=0)])
def test_forward_empty_is_ok(lib, kw):
    assert fwd(lib, **kw) == 0


def bwd(lib, B=1, H=1, N=128, d=64, causal=0, scale=0.125, ws=0, **ptrs):
    p = {n: A for n in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv")}
    p.update(ptrs)
    return lib.fa_backward(p["q"], p["k"], p["v"], p["o"], p["lse"], p["do"], p["dq"], p["dk"],
                           p["dv"], B, H, N, d, causal, scale, ws, None)


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), 1), (dict(causal=3), 1), (dict(scale=0.0), 1), (dict(d=80), 2),
    (dict(dq=0), 1), (dict(do=0), 1), (dict(dk=A + 4), 3), (dict(lse=A + 1), 3),
    (dict(ws=A + 16), 3),
])
def test_backward_rejects(lib, kw, status):
    assert bwd(lib, **kw) == status


def test_backward_empty_is_ok(lib):
    assert bwd(lib, N=0) == 0 and bwd(lib, B=0) == 0


def test_workspace_bytes(lib):
    from exact_io_aware_fa_gb300 import api
    # two 16-byte fold records and d fp32 dQ partial sums per padded query row
    assert api.backward_workspace_bytes(1, 1, 128, 64) == 128 * (32 + 4 * 64) + 256
    # N is padded to a multiple of 128
    assert api.backward_workspace_bytes(2, 3, 129, 128) == 6 * 256 * (32 + 4 * 128) + 256
    assert api.backward_workspace_bytes(0, 1, 128, 64) == 0
    assert api.backward_workspace_bytes(1, 1, 128, 48) == 0


def test_missing_library_fails_loudly(tmp_path):
    from exact_io_aware_fa_gb300 import api
    saved = api._LIB
    try:
        api._LIB = None
        with pytest.raises(api.FaLibraryMissing):
            api.library(str(tmp_path / "nope.so"))
    finally:
        api._LIB = saved


def fwd_ex(lib, B=1, Hq=4, Hkv=2, Tq=128, Tk=256, d=64, causal=1, window=-1, scale=0.125, **ptrs):
    p = {n: A for n in ("q", "k", "v", "o", "lse")}
    p.update(ptrs)
    return lib.fa_forward_ex(p["q"], p["k"], p["v"], p["o"], p["lse"], B, Hq, Hkv, Tq, Tk, d,
                             causal, window, scale, None)


def bwd_ex(lib, B=1, Hq=4, Hkv=2, Tq=128, Tk=256, d=64, causal=1, window=-1, scale=0.125, ws=0,
           **ptrs):
    p = {n: A for n in ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv")}
    p.update(ptrs)
    return lib.fa_backward_ex(p["q"], p["k"], p["v"], p["o"], p["lse"], p["do"], p["dq"],
                              p["dk"], p["dv"], B, Hq, Hkv, Tq, Tk, d, causal, window, scale, ws,
                              None)


EX_REJECT = [
    (dict(Hq=3, Hkv=2), 1),               # Hq not a multiple of Hkv
    (dict(Hq=4, Hkv=0), 1), (dict(Hq=0, Hkv=2), 1),
    (dict(Hkv=-1), 1), (dict(Tq=-1), 1), (dict(Tk=-3), 1),
    (dict(causal=0, window=10), 1),       # a window needs the causal diagonal
    (dict(window=-2), 1),
    (dict(Tq=300, Tk=200), 1),            # causal with more queries than keys: empty rows
    (dict(causal=0, Tk=0), 1),            # no keys at all
    (dict(d=96), 2), (dict(scale=0.0), 1), (dict(causal=2), 1),
    (dict(k=0), 1), (dict(v=A + 2), 3), (dict(lse=A + 1), 3),
]


@pytest.mark.parametrize("kw,status", EX_REJECT)
def test_forward_ex_rejects(lib, kw, status):
    assert fwd_ex(lib, **kw) == status


@pytest.mark.parametrize("kw,status", EX_REJECT + [(dict(dk=0), 1), (dict(ws=A + 32), 3)])
def test_backward_ex_rejects(lib, kw, status):
    assert bwd_ex(lib, **kw) == status


def test_ex_empty_is_ok(lib):
    assert fwd_ex(lib, Tq=0) == 0
    assert fwd_ex(lib, B=0) == 0
    assert fwd_ex(lib, Hq=0, Hkv=0, q=0, k=0, v=0, o=0, lse=0) == 0
    # non-causal Tq > Tk is a valid shape: it passes the shape checks and stops at the next
    # one, the misaligned output pointer (FA_ERR_ALIGNMENT, not FA_ERR_INVALID_ARG). A call with
    # a valid shape and well-formed fake pointers would launch a kernel on a machine with a GPU.
    assert fwd_ex(lib, causal=0, Tq=500, Tk=200, o=A + 2) == 3
    assert bwd_ex(lib, B=0) == 0
    assert bwd_ex(lib, Tq=0, Tk=0) == 0


def fwd_split(lib, nsplit=4, ws=0, B=1, Hq=4, Hkv=2, Tq=1, Tk=1024, d=64, causal=1, window=-1,
              scale=0.125, **ptrs):
    p = {n: A for n in ("q", "k", "v", "o", "lse")}
    p.update(ptrs)
    return lib.fa_forward_splitkv(p["q"], p["k"], p["v"], p["o"], p["lse"], B, Hq, Hkv, Tq, Tk, d,
                                  causal, window, scale, nsplit, ws, None)


@pytest.mark.parametrize("kw,status", EX_REJECT + [
    (dict(nsplit=0), 1), (dict(nsplit=-2), 1), (dict(nsplit=65), 1), (dict(ws=A + 64), 3)])
def test_forward_splitkv_rejects(lib, kw, status):
    assert fwd_split(lib, **kw) == status


def test_splitkv_workspace_bytes(lib):
    from exact_io_aware_fa_gb300 import api
    # nsplit partial rows of d fp32 values plus one fp32 LSE each, both parts 256-byte aligned
    rows = 2 * 3 * 5 * 4
    assert api.splitkv_workspace_bytes(2, 3, 5, 64, 4) == (rows * 64 * 4 + 255) // 256 * 256 + \
        (rows * 4 + 255) // 256 * 256
    assert api.splitkv_workspace_bytes(1, 1, 1, 128, 1) == 0   # no split, no workspace
    assert api.splitkv_workspace_bytes(1, 1, 1, 128, 65) == 0
    assert api.splitkv_workspace_bytes(1, 1, 1, 96, 4) == 0


def test_split_choice():
    from exact_io_aware_fa_gb300 import api
    c = api.choose_splits
    assert c(4, 16, 16, 2048, 2048, 152) == 1        # 512 blocks fill the GPU
    assert c(8, 32, 32, 1, 16384, 152) == 1          # 256 decode rows fill it too
    assert c(1, 8, 8, 1, 16384, 152) == 16           # 8 rows x 16 chunks = 128 units
    assert c(1, 32, 32, 1, 16384, 152) == 4          # 32 rows x 4 chunks, one round
    assert c(1, 32, 32, 512, 16384, 152) == 2        # chunked prefill, 64 blocks
    assert c(1, 32, 32, 1024, 16384, 152) == 1       # 128 blocks: no split
    assert c(1, 8, 8, 1, 300, 152) == 1              # too few key tiles to split
    assert c(1, 1, 1, 1, 1 << 20, 152) == api.MAX_SPLITS
    # grouped heads with short query blocks are packed: one block per KV head
    assert c(1, 32, 8, 1, 16384, 152) == 16          # 8 packed blocks x 16 chunks
    assert c(8, 32, 8, 1, 16384, 152) == 2           # 64 packed blocks x 2 chunks
    assert c(1, 32, 8, 512, 16384, 152) == 2         # Tq > 64: not packed, as MHA
    assert c(0, 32, 8, 1, 16384, 152) == 1 and c(1, 32, 5, 1, 16384, 152) == 1  # invalid


def host_step(lib, q=A, k=A, v=A, do=A, o=A, lse=A, dq=A, dk=A, dv=A, B=1, Hq=2, Hkv=1, Tq=128,
              Tk=256, d=64, causal=1, window=-1, scale=0.125, nchunks=0, buf=None):
    return lib.fa_forward_backward_host(q, k, v, do, o, lse, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d,
                                        causal, window, scale, nchunks, buf, None)


@pytest.mark.parametrize("kw,status", [
    (dict(nchunks=-1), 1), (dict(nchunks=17), 1), (dict(q=0), 1), (dict(do=0), 1),
    (dict(lse=0), 1), (dict(dq=0), 1), (dict(k=0), 1), (dict(dv=0), 1),
    (dict(buf=A + 16), 1), (dict(Hq=3, Hkv=2), 1), (dict(Tq=300), 1), (dict(window=5, causal=0), 1),
    (dict(d=96), 2),
])
def test_host_step_rejects(lib, kw, status):
    # every one of these is refused before any CUDA call (no GPU here)
    assert host_step(lib, **kw) == status


def test_host_step_empty_is_ok(lib):
    assert host_step(lib, B=0) == 0
    assert host_step(lib, Hq=0, Hkv=0, q=0, k=0, v=0, do=0, o=0, lse=0, dq=0, dk=0, dv=0) == 0


def test_host_step_device_bytes():
    from exact_io_aware_fa_gb300 import api
    r = lambda x: (x + 255) // 256 * 256

    def expect(B, Hq, Hkv, Tq, Tk, d, nch):
        nkv = B * Hkv
        nch = min(nch or 4, nkv)
        starts = [nkv * c // nch for c in range(nch + 1)]
        per = max(b - a for a, b in zip(starts, starts[1:])) * (Hq // Hkv)  # largest chunk
        ws = api.backward_workspace_bytes(1, per, Tq, d)
        q = B * Hq * Tq * d * 2
        kv = B * Hkv * Tk * d * 2
        return 4 * r(q) + 4 * r(kv) + r(B * Hq * Tq * 4) + 2 * r(ws)

    for args in [(1, 2, 1, 128, 256, 64, 0), (4, 16, 16, 2048, 2048, 64, 0),
                 (2, 8, 2, 100, 300, 128, 3), (1, 4, 4, 1, 777, 64, 16), (3, 6, 3, 50, 50, 128, 1)]:
        assert api.host_step_device_bytes(*args) == expect(*args), args
    assert api.host_step_device_bytes(1, 2, 1, 128, 256, 64, 0) == 411136
    assert api.host_step_device_bytes(1, 2, 1, 128, 256, 64, 17) == 0
    assert api.host_step_device_bytes(1, 2, 1, 128, 256, 96, 0) == 0


def test_naive_softmax_argument_checks(lib):
    """fa_naive_softmax validates before launching anything (no GPU needed)."""
    from exact_io_aware_fa_gb300 import api
    A = 1 << 20
    assert lib.fa_naive_softmax(A, A, A, -1, 16, 0, 0.125, None) == api.FA_ERR_INVALID_ARG
    assert lib.fa_naive_softmax(A, A, A, 16, 16, 2, 0.125, None) == api.FA_ERR_INVALID_ARG
    assert lib.fa_naive_softmax(A, A, A, 16, 16, 0, 0.0, None) == api.FA_ERR_INVALID_ARG
    assert lib.fa_naive_softmax(A, A, A, 16, 16, 0, float("nan"), None) == api.FA_ERR_INVALID_ARG
    assert lib.fa_naive_softmax(None, A, A, 16, 16, 0, 0.125, None) == api.FA_ERR_INVALID_ARG
    assert lib.fa_naive_softmax(A + 2, A, A, 16, 16, 0, 0.125, None) == api.FA_ERR_ALIGNMENT
    assert lib.fa_naive_softmax(None, None, None, 0, 16, 0, 0.125, None) == api.FA_OK
