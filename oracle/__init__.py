"""ctypes wrapper around the fp64 CPU oracle in ``fa_oracle.c``.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by the bench's
CPU-baseline leg, never by the product path. The oracle shares no code with the CUDA
path; it is compiled by gcc from ``fa_oracle.c`` alone.

Functions take bf16 bit arrays (``numpy.uint16``, from the shared seeded generator) or
float64 arrays, in the [B, H, N, d] layout, and return float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict = {}


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_HERE, "_build", name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake variant of it) with gcc."""
    out = lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-fno-fast-math",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutant: int = 0):
    with _LOCK:
        if mutant in _LIBS:
            return _LIBS[mutant]
        lib = ctypes.CDLL(build(mutant))
        P = ctypes.c_void_p
        L = ctypes.c_long
        I = ctypes.c_int
        D = ctypes.c_double
        lib.fa_oracle_forward_bf16.argtypes = [P, P, P, P, P, L, L, L, L, I, D, I]
        lib.fa_oracle_forward_rows_bf16.argtypes = [P, P, P, P, P, L, L, L, L, I, D, P, L, I]
        lib.fa_oracle_forward_f64.argtypes = [P, P, P, P, P, L, L, L, L, I, D, I]
        lib.fa_oracle_probs_f64.argtypes = [P, P, P, L, L, L, L, I, D, I]
        lib.fa_oracle_backward_bf16.argtypes = [P, P, P, P, P, P, P, L, L, L, L, I, D, I]
        lib.fa_oracle_backward_f64.argtypes = [P, P, P, P, P, P, P, L, L, L, L, I, D, I]
        lib.fa_oracle_backward_rows_bf16.argtypes = [P, P, P, P, P, P, P, L, L, L, L, I, D,
                                                     P, L, P, L, I]
        lib.fa_oracle_forward_ex_f64.argtypes = [P, P, P, P, P, L, L, L, L, L, L, I, L, D, I]
        lib.fa_oracle_forward_ex_bf16.argtypes = [P, P, P, P, P, L, L, L, L, L, L, I, L, D, I]
        lib.fa_oracle_backward_ex_f64.argtypes = [P, P, P, P, P, P, P, L, L, L, L, L, L, I, L, D, I]
        lib.fa_oracle_backward_ex_bf16.argtypes = [P, P, P, P, P, P, P, L, L, L, L, L, L, I, L, D,
                                                   I]
        lib.fa_oracle_backward_ex_sens_bf16.argtypes = [P, P, P, P, P, P, P, P, P, P, L, L, L, L,
                                                        L, L, I, L, D, I]
        lib.fa_oracle_mutant_id.argtypes = []
        for fn in ("fa_oracle_forward_bf16", "fa_oracle_forward_rows_bf16",
                   "fa_oracle_forward_f64", "fa_oracle_probs_f64", "fa_oracle_backward_bf16",
                   "fa_oracle_backward_f64", "fa_oracle_backward_rows_bf16",
                   "fa_oracle_forward_ex_f64", "fa_oracle_forward_ex_bf16",
                   "fa_oracle_backward_ex_f64", "fa_oracle_backward_ex_bf16",
                   "fa_oracle_backward_ex_sens_bf16", "fa_oracle_mutant_id"):
            getattr(lib, fn).restype = ctypes.c_int
        _LIBS[mutant] = lib
        return lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _shape4(q: np.ndarray):
    if q.ndim != 4:
        raise ValueError("expected [B, H, N, d]")
    return q.shape


class Oracle:
    """Handle on one build of the oracle (``mutant=0`` is the real one)."""

    def __init__(self, mutant: int = 0, threads: int | None = None):
        self.mutant = mutant
        self.threads = threads or default_threads()
        self.lib = _lib(mutant)

    # -- forward ----------------------------------------------------------------------
    def forward_bf16(self, q, k, v, causal: bool, scale: float):
        B, H, N, d = _shape4(q)
        q, k, v = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v))
        o = np.empty((B, H, N, d), dtype=np.float64)
        lse = np.empty((B, H, N), dtype=np.float64)
        _check(self.lib.fa_oracle_forward_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                               B, H, N, d, int(causal), float(scale),
                                               self.threads), "forward")
        return o, lse

    def forward_rows_bf16(self, q, k, v, causal: bool, scale: float, rows):
        B, H, N, d = _shape4(q)
        q, k, v = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v))
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nr = rows.shape[0]
        o = np.empty((B, H, nr, d), dtype=np.float64)
        lse = np.empty((B, H, nr), dtype=np.float64)
        _check(self.lib.fa_oracle_forward_rows_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                                    _ptr(lse), B, H, N, d, int(causal),
                                                    float(scale), _ptr(rows), nr,
                                                    self.threads), "forward_rows")
        return o, lse

    def forward_f64(self, q, k, v, causal: bool, scale: float):
        B, H, N, d = _shape4(q)
        q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
        o = np.empty((B, H, N, d), dtype=np.float64)
        lse = np.empty((B, H, N), dtype=np.float64)
        _check(self.lib.fa_oracle_forward_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                              B, H, N, d, int(causal), float(scale),
                                              self.threads), "forward_f64")
        return o, lse

    def probs_f64(self, q, k, causal: bool, scale: float):
        B, H, N, d = _shape4(q)
        q, k = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k))
        P = np.empty((B, H, N, N), dtype=np.float64)
        _check(self.lib.fa_oracle_probs_f64(_ptr(q), _ptr(k), _ptr(P), B, H, N, d,
                                            int(causal), float(scale), self.threads), "probs")
        return P

    # -- backward ---------------------------------------------------------------------
    def backward_bf16(self, q, k, v, dout, causal: bool, scale: float):
        B, H, N, d = _shape4(q)
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v, dout))
        dq, dk, dv = (np.empty((B, H, N, d), dtype=np.float64) for _ in range(3))
        _check(self.lib.fa_oracle_backward_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                                _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                                int(causal), float(scale), self.threads),
               "backward")
        return dq, dk, dv

    def backward_f64(self, q, k, v, dout, causal: bool, scale: float):
        B, H, N, d = _shape4(q)
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, dout))
        dq, dk, dv = (np.empty((B, H, N, d), dtype=np.float64) for _ in range(3))
        _check(self.lib.fa_oracle_backward_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                               _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                               int(causal), float(scale), self.threads),
               "backward_f64")
        return dq, dk, dv

    def backward_rows_bf16(self, q, k, v, dout, causal: bool, scale: float, rows_q, rows_k):
        B, H, N, d = _shape4(q)
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v, dout))
        rq = np.ascontiguousarray(rows_q, dtype=np.int64)
        rk = np.ascontiguousarray(rows_k, dtype=np.int64)
        dq = np.empty((B, H, rq.shape[0], d), dtype=np.float64)
        dk = np.empty((B, H, rk.shape[0], d), dtype=np.float64)
        dv = np.empty((B, H, rk.shape[0], d), dtype=np.float64)
        _check(self.lib.fa_oracle_backward_rows_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                                     _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
                                                     int(causal), float(scale), _ptr(rq),
                                                     rq.shape[0], _ptr(rk), rk.shape[0],
                                                     self.threads), "backward_rows")
        return dq, dk, dv


class NoVisibleKey(ValueError):
    """A query row sees no key (the attention of that row is undefined)."""


def _check_ex(rc: int, what: str) -> None:
    if rc == -3:
        raise NoVisibleKey(f"oracle {what}: a query row has no visible key")
    _check(rc, what)


def _ex_shapes(q, k):
    if q.ndim != 4 or k.ndim != 4 or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("expected q [B,Hq,Tq,d] and k/v [B,Hkv,Tk,d]")
    B, Hq, Tq, d = q.shape
    _, Hkv, Tk, _ = k.shape
    return B, Hq, Hkv, Tq, Tk, d


def _ex_methods():
    def forward_ex(self, q, k, v, causal: bool, scale: float, window: int = -1):
        """Grouped KV heads, query rows at positions (Tk - Tq) + i, optional left window."""
        B, Hq, Hkv, Tq, Tk, d = _ex_shapes(q, k)
        f64 = q.dtype != np.uint16
        conv = (lambda x: np.ascontiguousarray(x, dtype=np.float64)) if f64 else \
               (lambda x: np.ascontiguousarray(x, dtype=np.uint16))
        q, k, v = conv(q), conv(k), conv(v)
        o = np.empty((B, Hq, Tq, d), dtype=np.float64)
        lse = np.empty((B, Hq, Tq), dtype=np.float64)
        fn = self.lib.fa_oracle_forward_ex_f64 if f64 else self.lib.fa_oracle_forward_ex_bf16
        _check_ex(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tq, Tk, d,
                     int(causal), int(window), float(scale), self.threads), "forward_ex")
        return o, lse

    def backward_ex(self, q, k, v, dout, causal: bool, scale: float, window: int = -1):
        B, Hq, Hkv, Tq, Tk, d = _ex_shapes(q, k)
        f64 = q.dtype != np.uint16
        conv = (lambda x: np.ascontiguousarray(x, dtype=np.float64)) if f64 else \
               (lambda x: np.ascontiguousarray(x, dtype=np.uint16))
        q, k, v, dout = conv(q), conv(k), conv(v), conv(dout)
        dq = np.empty((B, Hq, Tq, d), dtype=np.float64)
        dk = np.empty((B, Hkv, Tk, d), dtype=np.float64)
        dv = np.empty((B, Hkv, Tk, d), dtype=np.float64)
        fn = self.lib.fa_oracle_backward_ex_f64 if f64 else self.lib.fa_oracle_backward_ex_bf16
        _check_ex(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq,
                     Hkv, Tq, Tk, d, int(causal), int(window), float(scale), self.threads),
                  "backward_ex")
        return dq, dk, dv

    def backward_ex_sens(self, q, k, v, dout, causal: bool, scale: float, window: int = -1):
        """backward_ex on bf16 bits plus the gradients' sensitivities to relative errors in the
        operands the products consume: (dq, dk, dv), (sq, sk, sv) with
        sv_je = sum_i P_ij |dO_ie| (over the group's query rows), sk_je = scale sum_i |dS_ij|
        |q_ie|, sq_ie = scale sum_j |dS_ij| |k_je|. If every P_ij (dS_ij) entering dV (dK, dQ)
        carries a relative error of at most u, each gradient element moves by at most u times
        its sensitivity (the triangle inequality on the sums that define it)."""
        B, Hq, Hkv, Tq, Tk, d = _ex_shapes(q, k)
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.uint16) for x in (q, k, v, dout))
        dq = np.empty((B, Hq, Tq, d), dtype=np.float64)
        dk = np.empty((B, Hkv, Tk, d), dtype=np.float64)
        dv = np.empty((B, Hkv, Tk, d), dtype=np.float64)
        sq, sk, sv = np.empty_like(dq), np.empty_like(dk), np.empty_like(dv)
        _check_ex(self.lib.fa_oracle_backward_ex_sens_bf16(
            _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(sq), _ptr(sk),
            _ptr(sv), B, Hq, Hkv, Tq, Tk, d, int(causal), int(window), float(scale), self.threads),
            "backward_ex_sens")
        return (dq, dk, dv), (sq, sk, sv)

    Oracle.forward_ex = forward_ex
    Oracle.backward_ex = backward_ex
    Oracle.backward_ex_sens = backward_ex_sens


_ex_methods()


# ---- flash-decoding partials and their merge --------------------------------------------
#
# "15. FlashAttention" (inference.shantanugoel.com), section "Decode is different:
# flash-decoding": the key sequence is cut into chunks; each chunk i yields a partial
# (m_i, l_i, a_i) -- the running max, the sum of exp(s - m_i) and the unnormalised accumulator
# sum of exp(s - m_i) v over the chunk's visible keys -- and the partials combine by
#   m = max_i m_i,  l = sum_i exp(m_i - m) l_i,  a = sum_i exp(m_i - m) a_i,  O = a / l,
# a rule that is associative (any grouping gives the same triple). Plain numpy in fp64, for
# small cases; the visibility rule is that of forward_ex.

def _visible_ex(pos: int, j: int, causal: bool, window: int) -> bool:
    if causal and j > pos:
        return False
    if window >= 0 and j < pos - window:
        return False
    return True


def partials_f64(q, k, v, causal: bool, scale: float, window: int, bounds):
    """Partials (m, l, a) of every key chunk [bounds[i], bounds[i+1]) for every query row.

    Returns m [C, B, Hq, Tq], l [C, B, Hq, Tq], a [C, B, Hq, Tq, d] (m = -inf, l = 0, a = 0
    for a chunk in which the row sees no key)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    B, Hq, Hkv, Tq, Tk, d = _ex_shapes(q, k)
    group = Hq // Hkv
    C = len(bounds) - 1
    m = np.full((C, B, Hq, Tq), -np.inf)
    l = np.zeros((C, B, Hq, Tq))
    a = np.zeros((C, B, Hq, Tq, d))
    for b in range(B):
        for h in range(Hq):
            kh, vh = k[b, h // group], v[b, h // group]
            for i in range(Tq):
                pos = Tk - Tq + i
                for c in range(C):
                    js = [j for j in range(bounds[c], bounds[c + 1])
                          if _visible_ex(pos, j, causal, window)]
                    if not js:
                        continue
                    s = scale * (kh[js] @ q[b, h, i])
                    m[c, b, h, i] = s.max()
                    e = np.exp(s - m[c, b, h, i])
                    l[c, b, h, i] = e.sum()
                    a[c, b, h, i] = e @ vh[js]
    return m, l, a


def merge_partials(m, l, a):
    """Combine partials along axis 0 by the flash-decoding rule; returns the merged partial
    (m, l, a) and O = a / l, LSE = m + ln l. A row whose chunks all lack keys is an error."""
    m, l, a = (np.asarray(x, dtype=np.float64) for x in (m, l, a))
    mm = m.max(axis=0)
    if np.any(np.isneginf(mm)):
        raise NoVisibleKey("merge: a query row has no visible key in any chunk")
    w = np.where(np.isneginf(m), 0.0, np.exp(m - mm[None]))
    ll = (w * l).sum(axis=0)
    aa = (w[..., None] * a).sum(axis=0)
    return mm, ll, aa, aa / ll[..., None], mm + np.log(ll)


def oracle(threads: int | None = None) -> Oracle:
    return Oracle(0, threads)
