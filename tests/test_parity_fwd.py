"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle on the same
seeded bf16 inputs. Small and ragged sizes are compared in full; the full-size
configurations on seeded samples of query rows (plus tile-boundary rows)."""
import math

import numpy as np
import pytest

import oracle
from parity_util import (assert_close_lse, assert_close_o, default_scale, to_dev, to_f64)

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


def run_fwd(api, bits, causal, scale):
    import torch
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    o, lse = api.forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    return to_f64(o), lse.cpu().numpy().astype(np.float64)


def test_worked_example_unit_case(env):
    """Scores [0,1,2,-1] against values [2,4,1,3] give 1.8619 ("15. FlashAttention",
    section "Worked example"): q = e_0, k_j = s_j e_0, v_j = value_j e_0, scale 1, N = 4."""
    api, orc = env
    d, N = 64, 4
    q = np.zeros((1, 1, N, d), np.float32)
    k = np.zeros((1, 1, N, d), np.float32)
    v = np.zeros((1, 1, N, d), np.float32)
    q[0, 0, 0, 0] = 1.0
    k[0, 0, :, 0] = [0, 1, 2, -1]
    v[0, 0, :, 0] = [2, 4, 1, 3]
    bits = {n: (a.view(np.uint32) >> 16).astype(np.uint16) for n, a in (("q", q), ("k", k), ("v", v))}
    o, lse = run_fwd(api, bits, False, 1.0)
    assert abs(o[0, 0, 0, 0] - 1.8619) <= 5e-3  # bf16 output: 1.8619 rounds to 1.859375
    assert abs(lse[0, 0, 0] - math.log(math.exp(0) + math.exp(1) + math.exp(2) + math.exp(-1))) <= 1e-3
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], False, 1.0)
    assert_close_o(o, o_ref, "unit", small_case=True)
    assert_close_lse(lse, lse_ref, "unit")


SMALL_N = [1, 4, 17, 127, 128, 129, 255, 256, 257, 383, 513, 1000]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", SMALL_N)
def test_small_and_ragged_full(env, d, causal, N):
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(1, 2, N, d, seed=100 + N, qk_sigma=1.5)
    o, lse = run_fwd(api, bits, causal, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], causal, default_scale(d))
    assert_close_o(o, o_ref, f"N={N} d={d} causal={causal}", small_case=True)
    assert_close_lse(lse, lse_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_closed_form(env, causal):
    """Q = 0: every visible score is 0, so LSE_i = ln(#visible) and O_i is the mean of the
    visible V rows (oracle pin reused on the GPU)."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    N, d = 300, 128
    bits = synthetic.attention_inputs(1, 1, N, d, seed=5)
    bits["q"] = np.zeros_like(bits["q"])
    o, lse = run_fwd(api, bits, causal, default_scale(d))
    nvis = np.arange(1, N + 1) if causal else np.full(N, N)
    assert np.max(np.abs(lse[0, 0] - np.log(nvis))) <= 1e-3
    o_ref, _ = orc.forward_bf16(bits["q"], bits["k"], bits["v"], causal, default_scale(d))
    assert_close_o(o, o_ref, "zero q")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_row_max_jump_beyond_exp2_range(env, d, causal):
    """Keys of the last quarter scaled by 100: the first key tile there raises a row's max by
    hundreds (log2 units of the scaled scores), far past the lagging reference's threshold and
    the fp32 exponent range of exp2, so that tile's weights are taken against the moved
    reference and O is rescaled by a factor that underflows to 0. N = 1000 (ragged)."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    N = 1000
    bits = synthetic.attention_inputs(1, 2, N, d, seed=300 + d + int(causal))
    k = synthetic.bf16_bits_to_float64(bits["k"])
    k[:, :, 3 * N // 4:] *= 100.0
    bits["k"] = synthetic.float32_to_bf16_bits(k.astype(np.float32))
    o, lse = run_fwd(api, bits, causal, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], causal, default_scale(d))
    what = f"key jump d={d} causal={causal}"
    assert_close_o(o, o_ref, what, small_case=True)
    assert_close_lse(lse, lse_ref, what)


def test_output_bounds_untouched(env):
    """Ragged N: nothing is written past the end of O or LSE."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, _ = env
    B, H, N, d = 1, 3, 200, 64
    bits = synthetic.attention_inputs(B, H, N, d, seed=9)
    q, k, v = (to_dev(bits[n]) for n in ("q", "k", "v"))
    n_el = B * H * N * d
    obuf = torch.full((n_el + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((B * H * N + 1024,), 7.0, dtype=torch.float32, device="cuda")
    o = obuf[:n_el].view(B, H, N, d)
    lse = lbuf[: B * H * N].view(B, H, N)
    api.forward(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(obuf[n_el:] == 7.0)
    assert torch.all(lbuf[B * H * N:] == 7.0)


def test_forward_full_b1_h1_n256_d64(env):
    """B=1 H=1 N=256 d=64, non-causal, N(0,1), scale 1/8."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(1, 1, 256, 64, seed=1001)
    o, lse = run_fwd(api, bits, False, 0.125)
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], False, 0.125)
    assert_close_o(o, o_ref, "B1 H1 N256 d64")
    assert_close_lse(lse, lse_ref, "B1 H1 N256 d64")


def test_forward_full_b4_h16_n2048_d64(env):
    """B=4 H=16 N=2048 d=64, non-causal, N(0,1), scale 1/sqrt(d): compared in full."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(4, 16, 2048, 64, seed=1002)
    o, lse = run_fwd(api, bits, False, default_scale(64))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], False, default_scale(64))
    assert_close_o(o, o_ref, "B4 H16 N2048 d64")
    assert_close_lse(lse, lse_ref, "B4 H16 N2048 d64")


def _sampled(env, B, H, N, d, causal, seed, qk_sigma):
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(B, H, N, d, seed=seed, qk_sigma=qk_sigma)
    o, lse = run_fwd(api, bits, causal, default_scale(d))
    rows = synthetic.sample_rows(N, 32, seed)
    o_ref, lse_ref = orc.forward_rows_bf16(bits["q"], bits["k"], bits["v"], causal,
                                           default_scale(d), rows)
    what = f"B{B} H{H} N{N} d{d} causal={causal}"
    assert_close_o(o[:, :, rows], o_ref, what)
    assert_close_lse(lse[:, :, rows], lse_ref, what)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_forward_sampled_b8_h32_n8192_d128_causal(env):
    """B=8 H=32 N=8192 d=128, causal, N(0,1)."""
    _sampled(env, 8, 32, 8192, 128, True, 1003, 1.0)


@pytest.mark.parametrize("N", [16384, 16000])
def test_forward_sampled_b1_h64_d128_causal_qk_sd3(env, N):
    """B=1 H=64 d=128 causal, Q and K ~ N(0, 3^2) (large score ranges), V ~ N(0,1)."""
    _sampled(env, 1, 64, N, 128, True, 1004, 3.0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [100, 300])
def test_persistent_many_units_per_cta(env, d, causal, N):
    """More (head, 256-row block) units than SMs, so every persistent CTA runs several units
    back to back; with N = 100 the second Q tile of every unit is empty (its buffer release
    must not run ahead of the other tile's epilogue)."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(2, 200, N, d, seed=300 + N + d)
    o, lse = run_fwd(api, bits, causal, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], causal, default_scale(d))
    assert_close_o(o, o_ref, f"many units N={N} d={d} causal={causal}", small_case=True)
    assert_close_lse(lse, lse_ref, f"many units N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [200, 300])
def test_half_units_in_last_round(env, d, N):
    """Non-causal launches whose last round of (head, 256-row block) units would fill at most
    half of the SMs run that round as half units, one 128-row Q tile each. Sizes chosen from
    the device's SM count so that a few units are left over; with N = 300 the second tile of
    every block is ragged and one half unit of each leftover block is past the end (empty)."""
    import torch
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nqb = -(-N // 256)
    H = (sms + 8 + nqb - 1) // nqb          # units = H * nqb = sms + (a few)
    units = H * nqb
    assert units > sms and 0 < units % sms <= sms // 2
    bits = synthetic.attention_inputs(1, H, N, d, seed=700 + N + d)
    o, lse = run_fwd(api, bits, False, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], False, default_scale(d))
    assert_close_o(o, o_ref, f"half units N={N} d={d}", small_case=True)
    assert_close_lse(lse, lse_ref, f"half units N={N} d={d}")


def test_sorted_causal_order_in_several_head_chunks(env):
    """A causal launch of at most 16 units per SM deals its units heaviest first inside chunks
    of heads whose K/V fits in 128 MB of L2. B1 H36 N16384 d128 reads 8 MB of K/V per head:
    chunks of 16, 16 and 4 heads (the last one ragged); 2304 units, under 16 per SM on 152."""
    _sampled(env, 1, 36, 16384, 128, True, 4041, 1.0)


def test_long_sequence_sampled(env):
    """N = 131072 keys and queries (causal, d=64): 1024 key tiles per row block, positions and
    row offsets well past 2^16; 32 seeded rows plus the tile-boundary rows against the oracle."""
    _sampled(env, 1, 1, 131072, 64, True, 4099, 1.0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [513, 700, 2048])
def test_softmax_stress_peaked_rows(env, d, causal, N):
    """Q, K ~ N(0, 3^2): scaled scores with a spread of ~9 make many rows peaked (one weight
    close to 1), where the rounding of the dominant weight to bf16 matters."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    bits = synthetic.attention_inputs(1, 4, N, d, seed=300 + N + d, qk_sigma=3.0)
    o, lse = run_fwd(api, bits, causal, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], causal, default_scale(d))
    assert_close_o(o, o_ref, f"stress N={N} d={d} causal={causal}")
    assert_close_lse(lse, lse_ref, f"stress N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_row_max_growing_along_the_keys(env, d, causal):
    """Key rows scaled by a factor growing from 1 to 8 along the sequence: every row's maximum
    keeps growing from key tile to key tile, by more than exp2(8) over a few tiles, so the
    online rescale runs many times within one row."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    N = 1500
    bits = synthetic.attention_inputs(1, 2, N, d, seed=77 + d)
    k = synthetic.bf16_bits_to_float64(bits["k"])
    k = k * (1.0 + 7.0 * np.arange(N) / N)[None, None, :, None]
    bits["k"] = synthetic.float32_to_bf16_bits(k.astype(np.float32))
    o, lse = run_fwd(api, bits, causal, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], causal, default_scale(d))
    assert_close_o(o, o_ref, f"growing max d={d} causal={causal}")
    assert_close_lse(lse, lse_ref, f"growing max d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_single_dominant_key(env, d):
    """One key per row far above the others (its weight ~1): O must be that key's value row
    up to output rounding, whichever tile it sits in."""
    from exact_io_aware_fa_gb300 import synthetic
    api, orc = env
    N = 1000
    bits = synthetic.attention_inputs(1, 1, N, d, seed=91 + d)
    q = synthetic.bf16_bits_to_float64(bits["q"])
    k = synthetic.bf16_bits_to_float64(bits["k"]) * 0.25
    for i in range(N):
        # key (7919 i) mod N (a permutation) aligned with query i: its scaled score is about
        # 6 |q_i|^2 / (max|q_i| sqrt(d)) ~ 15-20 above the others' spread of ~0.25
        k[0, 0, (i * 7919) % N] += 6.0 * q[0, 0, i] / max(1.0, np.abs(q[0, 0, i]).max())
    bits["k"] = synthetic.float32_to_bf16_bits(k.astype(np.float32))
    o, lse = run_fwd(api, bits, False, default_scale(d))
    o_ref, lse_ref = orc.forward_bf16(bits["q"], bits["k"], bits["v"], False, default_scale(d))
    assert_close_o(o, o_ref, f"dominant key d={d}")
    assert_close_lse(lse, lse_ref, f"dominant key d={d}")
