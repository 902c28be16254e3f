"""Helpers shared by the GPU parity tests: moving the shared seeded bf16 bits to the device
and comparing against the oracle with the tolerances the attention path is held to."""
from __future__ import annotations

import math

import numpy as np

# Tolerances (absolute): O max <= 1e-2 and mean <= 1e-3; LSE <= 1e-3; dQ/dK/dV max <= 2e-2.
O_MAX, O_MEAN, LSE_MAX, GRAD_MAX = 1e-2, 1e-3, 1e-3, 2e-2


def to_dev(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_bits_of(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_rounding_error(x_ref: np.ndarray) -> np.ndarray:
    """|RNE_bf16(x) - x| elementwise: the error any bf16 output of the exact value carries."""
    from exact_io_aware_fa_gb300 import synthetic
    r = synthetic.bf16_bits_to_float64(synthetic.float32_to_bf16_bits(x_ref.astype(np.float32)))
    return np.abs(r - x_ref)


def assert_close_o(o, o_ref, what="", small_case=False):
    """O within max-abs 1e-2 and mean-abs 1e-3 of the oracle.

    The max-abs bound is applied to the error beyond the unavoidable rounding of the exact
    result to the bf16 output: |O - O_ref| <= 1e-2 + |bf16(O_ref) - O_ref| elementwise.
    (With |O| >= 4, reachable in the softmax-stress configuration, the bf16 spacing is 2^-5
    and the correctly rounded exact value itself can be 0.0156 away.)

    ``small_case``: for a handful of keys O is an average of very few V rows, so |O| is
    O(1) and the bf16 rounding of the output alone (spacing 2^-8 for |O| in [0.5, 1),
    mean error a quarter of that) reaches 1e-3; such edge cases use a mean bound of
    max(1e-3, 2^-8 * mean|O_ref|). The configurations always use the plain bounds."""
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    excess = err - bf16_rounding_error(o_ref)
    assert excess.max() <= O_MAX, (f"{what}: O max-abs {err.max():.3g}, beyond output rounding "
                                   f"{excess.max():.3g}")
    mean_bound = O_MEAN
    if small_case:
        mean_bound = max(O_MEAN, 2.0 ** -8 * float(np.abs(o_ref).mean()))
    assert err.mean() <= mean_bound, f"{what}: O mean-abs {err.mean():.3g} (bound {mean_bound:.3g})"


def assert_close_lse(lse, lse_ref, what=""):
    err = np.abs(lse - lse_ref)
    assert np.all(np.isfinite(lse)), f"{what}: non-finite LSE"
    assert err.max() <= LSE_MAX, f"{what}: LSE max-abs {err.max():.3g}"


# Unit roundoff of bf16 (8 significant bits, round to nearest even): |bf16(x) - x| <= 2^-8 |x|.
BF16_U = 2.0 ** -8


def assert_close_grad(g, g_ref, name, what="", sens=None):
    """Gradient within max-abs 2e-2 of the oracle beyond the bf16 rounding of the exact value.

    ``sens`` (optional, from the oracle's backward_ex_sens) adds, per element, the first-order
    bound of the error that rounding P to bf16 (before dV = P^T dO) or dS to bf16 (before
    dK = scale dS^T Q and dQ = scale dS K) introduces: each rounded operand is off by at most
    BF16_U of itself, so the element moves by at most BF16_U * sens with sens the sum of the
    absolute products it adds up (sum_i P_ij |dO_ie| for dV). That bound grows with the number of
    query rows summed into one key row -- e.g. 16 query heads on one KV head -- where the
    absolute 2e-2 alone, stated for gradients of a few units, no longer covers bf16 operands."""
    err = np.abs(g - g_ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
    excess = err - bf16_rounding_error(g_ref)
    if sens is not None:
        excess = excess - BF16_U * sens
    assert excess.max() <= GRAD_MAX, (f"{what}: {name} max-abs {err.max():.3g}, beyond output "
                                      f"rounding{' and operand rounding' if sens is not None else ''}"
                                      f" {excess.max():.3g}")


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def same_up_to_summation_order(a, b) -> bool:
    """dQ of two runs (torch tensors): its fp32 partial sums from different key tiles are added
    by atomic reductions in whatever order the tiles finish. That moves a result by about 2^-24
    of the partials' size, which after bf16 rounding is at most one unit in the last place -- or,
    where partials cancel to near zero, a small absolute amount (bounded here by 2^-16 of the
    largest |dQ|). Everything else the kernels compute is deterministic and compared exactly."""
    a, b = a.float(), b.float()
    floor = 2.0 ** -16 * float(b.abs().max())
    return bool(((a - b).abs() <= 2.0 ** -7 * b.abs() + floor).all())
