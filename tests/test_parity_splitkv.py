"""Parity of the split-KV ("flash-decoding") forward: fa_forward_splitkv cuts every query
block's key range into chunks, writes per-chunk partials and merges them; O and LSE must match
the fp64 oracle's unsplit forward_ex on the same seeded bf16 inputs. Includes decode (one query
row), chunks that some rows cannot see, chunks with no key tile at all, and the equality of
nsplit = 1 with fa_forward_ex."""
import pytest

import oracle
from parity_util import assert_close_lse, assert_close_o, default_scale, to_dev, to_f64

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


# (B, Hq, Hkv, Tq, Tk, d, causal, window, nsplit)
# Grouped heads with Tq <= 64 run packed (a KV head's query heads as one block of rows).
CASES = [
    (1, 8, 2, 50, 2000, 64, True, -1, 4),     # packed rows 200: tiles straddle packed heads
    (1, 8, 1, 64, 3000, 128, True, 600, 3),   # MQA packed into 512 rows (two blocks), window
    (2, 6, 3, 7, 999, 64, False, -1, 2),      # packed, non-causal, ragged keys
    (2, 8, 2, 1, 3000, 128, True, -1, 8),     # decode against a long cache
    (1, 4, 4, 1, 777, 64, False, -1, 3),      # decode, ragged cache, non-causal
    (1, 2, 2, 300, 1000, 64, True, -1, 3),    # chunked prefill
    (1, 3, 3, 700, 700, 64, False, -1, 4),    # plain multi-head attention
    (1, 2, 1, 500, 900, 128, True, 200, 5),   # window: many rows see nothing in some chunks
    (1, 2, 2, 129, 200, 64, True, -1, 7),     # more splits than key tiles: empty chunks
    (1, 4, 2, 64, 4096, 128, True, -1, 16),   # short query block, many splits
    (2, 2, 2, 256, 256, 128, True, -1, 2),    # causal square: tile 0 empty in split 1
    # at most 8 query rows per KV head (group * Tq <= 8): decode shapes
    (1, 8, 1, 1, 5000, 128, True, -1, 7),     # 8 rows per KV head, ragged cache
    (1, 5, 1, 1, 3000, 64, False, -1, 4),     # 5 rows (padded to 8), non-causal
    (2, 4, 2, 3, 1000, 128, True, 100, 3),    # 6 rows at 3 positions, window
    (1, 2, 2, 1, 20, 64, True, -1, 1),        # cache shorter than one 32-key tile, no split
    (1, 4, 1, 2, 90, 128, True, 5, 64),       # 64 splits of 3 tiles: empty chunks, window 5
    (3, 6, 3, 4, 4097, 64, True, -1, 16),     # 8 rows at 4 positions
    (1, 1, 1, 8, 512, 128, True, -1, 5),      # one head, 8 consecutive causal rows
    (1, 2, 1, 4, 300, 64, False, -1, 2),      # 8 rows, non-causal
]


def ids(c):
    B, Hq, Hkv, Tq, Tk, d, causal, w, ns = c
    return f"B{B}Hq{Hq}Hkv{Hkv}Tq{Tq}Tk{Tk}d{d}{'c' if causal else 'n'}w{w}s{ns}"


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_splitkv_matches_oracle(env, case):
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d, causal, window, nsplit = case
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=3 * Tk + Tq + nsplit)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    scale = default_scale(d)
    o, lse = api.forward(q, k, v, causal=causal, scale=scale, window=window, nsplit=nsplit)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], causal, scale, window)
    assert_close_o(to_f64(o), o_ref, ids(case), small_case=Tq * Tk < 4096)
    assert_close_lse(to_f64(lse), lse_ref, ids(case))


@pytest.mark.parametrize("d", [64, 128])
def test_runs_of_empty_key_chunks(env, d):
    """Many more key splits than key tiles, and several units per SM: most units of every SM
    are key chunks with no tile for either Q tile, often several in a row. Such units release
    their Q buffer at once; the kernel must not lose track of the buffer's phases."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, nsplit = 2, 40, 8, 256, 640, 16   # 5 key tiles, 16 splits
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=77 + d)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    scale = default_scale(d)
    o, lse = api.forward(q, k, v, causal=True, scale=scale, nsplit=nsplit)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], True, scale)
    assert_close_o(to_f64(o), o_ref, f"empty chunks d={d}")
    assert_close_lse(to_f64(lse), lse_ref, f"empty chunks d={d}")


def test_one_split_is_the_plain_forward(env):
    """nsplit = 1 runs fa_forward_ex: bit-identical output."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, _ = env
    bits = synthetic.attention_inputs_ex(1, 4, 2, 300, 600, 64, seed=8)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    o1, l1 = api.forward(q, k, v, causal=True, nsplit=1)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    st = api.forward_ex_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(),
                            1, 4, 2, 300, 600, 64, 1, -1, default_scale(64), 0)
    assert st == api.FA_OK
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_library_allocated_split_workspace(env):
    """workspace = NULL: the library allocates the partials on the stream."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d = 1, 2, 1, 3, 2500, 128
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=12)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device="cuda")
    st = api.forward_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, Hq, Hkv, Tq, Tk, d, 1, -1, default_scale(d), 6, 0,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == api.FA_OK
    torch.cuda.synchronize()
    assert api.device_error() == 0
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], True, default_scale(d))
    assert_close_o(to_f64(o), o_ref, "ws=NULL", small_case=True)
    assert_close_lse(to_f64(lse), lse_ref, "ws=NULL")


def test_automatic_split_choice_for_decode(env):
    """api.forward picks splits by itself for a decode shape and stays exact."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d = 2, 4, 1, 1, 4000, 64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert api.choose_splits(B, Hq, Hkv, Tq, Tk, sms) > 1
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=21)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    o, lse = api.forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], True, default_scale(d))
    assert_close_o(to_f64(o), o_ref, "auto", small_case=True)
    assert_close_lse(to_f64(lse), lse_ref, "auto")


def test_split_decode_in_several_head_chunks(env):
    """Split launches use the sorted order over chunks of heads: one query row against 65536
    keys reads 32 MB of K/V per head, so 10 heads form chunks of 4, 4 and 2."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    B, Hq, Hkv, Tq, Tk, d = 1, 10, 10, 1, 65536, 128
    bits = synthetic.attention_inputs_ex(B, Hq, Hkv, Tq, Tk, d, seed=65)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    scale = default_scale(d)
    o, lse = api.forward(q, k, v, causal=True, scale=scale, nsplit=8)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    o_ref, lse_ref = orc.forward_ex(bits["q"], bits["k"], bits["v"], True, scale)
    assert_close_o(to_f64(o), o_ref, "decode head chunks", small_case=True)
    assert_close_lse(to_f64(lse), lse_ref, "decode head chunks")
