"""Parity of the extended entry points (grouped KV heads, query offset, sliding window):
fa_forward_ex / fa_backward_ex against the fp64 oracle's forward_ex / backward_ex on the same
seeded bf16 inputs. Query row i sits at key position Tk - Tq + i; a window W keeps keys at
positions >= position - W. Sizes span several tiles with ragged tails; the backward is fed
the CUDA forward's O and LSE."""
import numpy as np
import pytest

import oracle
from parity_util import (assert_close_grad, assert_close_lse, assert_close_o, default_scale,
                         same_up_to_summation_order, to_dev, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import __graft_entry__
    __graft_entry__.build()
    from exact_io_aware_fa_gb300 import api
    return api, oracle.oracle()


# (B, Hq, Hkv, Tq, Tk, d, causal, window)
CASES = [
    (1, 4, 1, 200, 200, 64, False, -1),     # multi-query, non-causal
    (2, 8, 2, 300, 300, 128, True, -1),     # grouped, causal
    (1, 2, 2, 100, 513, 64, True, -1),      # chunked prefill: offset 413
    (1, 4, 2, 1, 1000, 128, True, -1),      # decode: one query row
    (1, 3, 1, 5, 300, 64, True, -1),        # a few query rows, offset not tile-aligned
    (1, 2, 2, 130, 257, 64, False, -1),     # Tq != Tk, non-causal
    (1, 2, 1, 600, 600, 64, True, 100),     # window inside one key tile
    (1, 2, 2, 300, 700, 128, True, 0),      # window 0: each row sees its own key only
    (1, 4, 2, 512, 512, 64, True, 256),     # window on a tile multiple
    (1, 2, 2, 1000, 1000, 128, True, 129),  # window straddling two key tiles
    (2, 4, 4, 384, 1200, 64, True, 300),    # offset and window together
    (1, 8, 1, 257, 257, 128, True, 1000),   # window wider than the sequence
    # grouped heads with Tq <= 64 run packed (a KV head's query heads as one block of rows)
    (2, 8, 2, 33, 700, 128, True, 50),      # packed rows 132 straddle the first tile, window
    (1, 16, 1, 64, 256, 64, True, -1),      # MQA, 1024 packed rows, causal boundary tile
    (1, 4, 2, 64, 300, 64, False, -1),      # packed exactly one tile per KV head
    (1, 4, 2, 65, 300, 64, True, -1),       # Tq = 65: not packed
    # MQA with short causal blocks: every key row sums 16 heads' rows, |dV| reaches ~14
    (1, 16, 1, 64, 64, 64, True, -1),       # packed forward, 1024 rows
    (1, 16, 1, 65, 65, 64, True, -1),       # unpacked
]


def ids(c):
    B, Hq, Hkv, Tq, Tk, d, causal, w = c
    return f"B{B}Hq{Hq}Hkv{Hkv}Tq{Tq}Tk{Tk}d{d}{'c' if causal else 'n'}w{w}"


def run_fwd(api, bits, causal, window, scale):
    import torch
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    o, lse = api.forward(q, k, v, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    return q, k, v, o, lse


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_forward_ex(env, case):
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d, causal, window = case
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=Tq * 7 + Tk)
    scale = default_scale(d)
    _, _, _, o, lse = run_fwd(api, bits, causal, window, scale)
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], causal, scale, window)
    small = Tq * Tk < 4096 or 0 <= window < 16
    assert_close_o(to_f64(o), o_ref, ids(case), small_case=small)
    assert_close_lse(to_f64(lse), lse_ref, ids(case))


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_backward_ex(env, case):
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d, causal, window = case
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=Tq * 7 + Tk + 1,
                                         with_dout=True)
    scale = default_scale(d)
    q, k, v, o, lse = run_fwd(api, bits, causal, window, scale)
    do = to_dev(bits["do"])
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=causal, scale=scale, window=window)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    ref, sens = orc.backward_ex_sens(bits["q"], bits["k"], bits["v"], bits["do"], causal, scale,
                                     window)
    for name, a, b, s in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref, sens):
        assert_close_grad(to_f64(a), b, name, ids(case), sens=s)


def test_mha_call_matches_ex_call(env):
    """fa_forward / fa_backward are the extended calls with Hq = Hkv, Tq = Tk, no window:
    bit-identical results."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, _ = env
    B, H, N, d = 1, 3, 333, 64
    bits = synthetic.attention_inputs(B, H, N, d, seed=5, with_dout=True)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    scale = default_scale(d)
    o1 = torch.empty_like(q)
    l1 = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    st = api.forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), l1.data_ptr(),
                         B, H, N, d, 1, scale, 0)
    assert st == api.FA_OK
    o2, l2 = api.forward(q, k, v, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = [torch.empty_like(q) for _ in range(3)]
    st = api.backward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), l1.data_ptr(),
                          do.data_ptr(), *(t.data_ptr() for t in g1), B, H, N, d, 1, scale, 0, 0)
    assert st == api.FA_OK
    g2 = api.backward(q, k, v, o2, l2, do, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert same_up_to_summation_order(g1[0], g2[0])  # dQ
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])


def test_no_query_rows_zeroes_kv_gradients(env):
    """Tq = 0: nothing attends to the keys, so dK = dV = 0 (written, not left as they were)."""
    import torch
    api, _ = env
    B, H, Tk, d = 1, 2, 300, 64
    dk = torch.full((B, H, Tk, d), 3.0, dtype=torch.bfloat16, device="cuda")
    dv = torch.full_like(dk, 3.0)
    st = api.backward_ex_raw(0, 0, 0, 0, 0, 0, 0, dk.data_ptr(), dv.data_ptr(), B, H, H, 0, Tk, d,
                             1, -1, 0.125, 0, 0)
    assert st == api.FA_OK
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(dk)) == 0 and int(torch.count_nonzero(dv)) == 0


def test_window_covers_unseen_key_tiles(env):
    """Key tiles that no query row can see (window far behind a short query block) get zero
    gradient from their CTA, which runs no step."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d, window = 1, 2, 1, 64, 1024, 128, 50
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=91, with_dout=True)
    scale = default_scale(d)
    q, k, v, o, lse = run_fwd(api, bits, True, window, scale)
    do = to_dev(bits["do"])
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=True, scale=scale, window=window,
                              dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    first_seen = Tk - Tq - window
    assert int(torch.count_nonzero(dk[:, :, : first_seen // 128 * 128])) == 0
    assert int(torch.count_nonzero(dv[:, :, : first_seen // 128 * 128])) == 0
    ref = orc.backward_ex(bits["q"], bits["k"], bits["v"], bits["do"], True, scale, window)
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_close_grad(to_f64(a), b, name, "unseen tiles")


def test_autograd_wrapper_matches_raw_calls(env):
    """api.attention (torch.autograd) gives the same O and the same gradients as the direct
    forward / backward calls."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, _ = env
    bits = synthetic.attention_inputs_ex(1, 4, 2, 200, 300, 64, seed=17, with_dout=True)
    q, k, v = (to_dev(bits[n]).requires_grad_(True) for n in ("q", "k", "v"))
    do = to_dev(bits["do"])
    o = api.attention(q, k, v, causal=True)
    o.backward(do)
    o2, lse2 = api.forward(q.detach(), k.detach(), v.detach(), causal=True)
    dq2, dk2, dv2 = api.backward(q.detach(), k.detach(), v.detach(), o2, lse2, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o2)
    assert same_up_to_summation_order(q.grad, dq2)
    assert torch.equal(k.grad, dk2) and torch.equal(v.grad, dv2)


def test_calls_from_a_new_host_thread(env):
    """A host thread that never touched CUDA before (as a framework's worker thread) can call
    forward and backward: the library binds the device's context itself."""
    import threading
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, _ = env
    bits = synthetic.attention_inputs(1, 2, 300, 128, seed=23, with_dout=True)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    ref_o, ref_lse = api.forward(q, k, v, causal=True)
    ref_g = api.backward(q, k, v, ref_o, ref_lse, do, causal=True)
    torch.cuda.synchronize()
    out = {}

    def work():
        try:
            o, lse = api.forward(q, k, v, causal=True)
            out["g"] = api.backward(q, k, v, o, lse, do, causal=True)
            out["o"] = o
            torch.cuda.synchronize()
        except Exception as e:  # reported below
            out["err"] = e

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert "err" not in out, out.get("err")
    assert torch.equal(out["o"], ref_o)
    assert same_up_to_summation_order(out["g"][0], ref_g[0])  # dQ
    assert torch.equal(out["g"][1], ref_g[1]) and torch.equal(out["g"][2], ref_g[2])


def test_backward_many_units_with_empty_tiles(env):
    """Persistent backward over more units than SMs where most key tiles see no query (window
    far behind a short query block): zero-step units interleave with working ones in every
    CTA's walk."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d, window = 1, 32, 16, 150, 1400, 64, 90
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=77, with_dout=True)
    scale = default_scale(d)
    q, k, v, o, lse = run_fwd(api, bits, True, window, scale)
    do = to_dev(bits["do"])
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=True, scale=scale, window=window)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    ref = orc.backward_ex(bits["q"], bits["k"], bits["v"], bits["do"], True, scale, window)
    for name, a, b in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_close_grad(to_f64(a), b, name, "many units, empty tiles")
