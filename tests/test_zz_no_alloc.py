"""fa_backward_noalloc: the backward for callers that may not allocate device memory at call
time (runtimes with a fixed start-up memory plan, hosts without allocator access). It uses
the library's own fixed device workspace instead of a caller buffer or cudaMallocAsync, so
its results must match the allocating entry point's, also when the shared workspace still
holds an earlier call's contents.

Collected last on purpose: if it fails, a run that stops at the first failure has already
run every other test."""
import math
import os

import pytest

from parity_util import same_up_to_summation_order, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api as fa_api
    return fa_api


def _case(api, B, H, N, d, causal, seed):
    """Inputs, the forward's O/LSE, and the allocating entry point's gradients (bf16)."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    bits = synthetic.attention_inputs(B, H, N, d, seed=seed, with_dout=True)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = api.forward(q, k, v, causal=causal, scale=scale)
    ws = torch.empty(api.backward_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    ref = api.backward(q, k, v, o, lse, do, causal=causal, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    return dict(q=q, k=k, v=v, do=do, o=o, lse=lse, scale=scale, ref=ref)


def _noalloc(api, c, B, H, N, d, causal):
    import torch
    dq, dk, dv = (torch.full_like(c["q"], float("nan")) for _ in range(3))
    stream = torch.cuda.current_stream().cuda_stream
    st = api.backward_noalloc_raw(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(),
                                  c["o"].data_ptr(), c["lse"].data_ptr(), c["do"].data_ptr(),
                                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                  int(causal), c["scale"], stream)
    assert st == api.FA_OK, api.status_string(st)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    return dq, dk, dv


def _assert_same(api, got, ref, what):
    """The two entry points run the same kernels on the same inputs: dK and dV are bit-identical
    and dQ differs at most by the order in which its fp32 partial sums were added."""
    import torch
    dq, dk, dv = got
    assert torch.isfinite(dq.float()).all(), what
    assert same_up_to_summation_order(dq, ref[0]), f"{what}: dQ differs from fa_backward"
    assert torch.equal(dk, ref[1]), f"{what}: dK differs from fa_backward"
    assert torch.equal(dv, ref[2]), f"{what}: dV differs from fa_backward"


def test_noalloc_matches_allocating_backward_twice(api):
    import torch
    # Calls in a row with different shapes: each reuses the workspace the call before left
    # behind (larger head dim, more heads, causal first; then a ragged non-causal case; then
    # the first shape again over the second's leftovers).
    limit = api.noalloc_scratch_bytes()
    cases = [(2, 4, 300, 128, True, 31), (1, 3, 1000, 64, False, 32), (2, 4, 300, 128, True, 31)]
    first = None
    for n, (B, H, N, d, causal, seed) in enumerate(cases):
        assert api.backward_workspace_bytes(B, H, N, d) <= limit
        c = _case(api, B, H, N, d, causal, seed)
        got = _noalloc(api, c, B, H, N, d, causal)
        _assert_same(api, got, c["ref"], f"call {n + 1}: B{B} H{H} N{N} d{d}")
        if n == 0:
            first = got
    # the repeated shape gives the first call's dK and dV bit for bit
    assert torch.equal(first[1], got[1]) and torch.equal(first[2], got[2])


def test_noalloc_size_matches_header(api):
    # The library reports the size its header promises.
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "fa.h")).read()
    m = re.search(r"#define FA_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", hdr)
    assert m, "FA_NOALLOC_SCRATCH_BYTES not found in include/fa.h"
    assert api.noalloc_scratch_bytes() == int(m.group(1)) * int(m.group(2)) * int(m.group(3))


def test_noalloc_rejects_sizes_beyond_its_workspace(api):
    # B*H = 64, N = 4096, d = 128 needs 143 MB of workspace: rejected before any launch
    # (the pointers are never used, so fake aligned addresses are enough).
    B, H, N, d = 4, 16, 4096, 128
    assert api.backward_workspace_bytes(B, H, N, d) > api.noalloc_scratch_bytes()
    A = 1 << 20
    st = api.backward_noalloc_raw(A, A, A, A, A, A, A, A, A, B, H, N, d, 1, 0.088, 0)
    assert st == api.FA_ERR_UNSUPPORTED
