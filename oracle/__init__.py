"""CPU oracle for the BitNet b1.58 W2A8 path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never imports it and shares no code with it.

This module is argument marshalling (numpy arrays in, numpy arrays out) around
``bitnet_oracle.c``; every step of the arithmetic is in that C file, which
cites the passage of the pages each function follows.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    from .build import build_oracle

    return build_oracle(force=force)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH) or _stale():
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    sig = {
        "oracle_bf16_to_f32": (None, [_p, _i64, _p]),
        "oracle_abs_sum": (ctypes.c_double, [_p, _i64]),
        "oracle_absmean": (_f32, [_p, _i64]),
        "oracle_gamma": (_f32, [_f32, _f32, _f32]),
        "oracle_ternarize": (ctypes.c_int, [_f32, _f32]),
        "oracle_pack_codes": (None, [_p, _i64, _p]),
        "oracle_unpack_codes": (None, [_p, _i64, _p]),
        "oracle_pack_weights": (None, [_p, _i64, _i64, _f32, _f32, _p, _p, _p]),
        "oracle_quant_act": (None, [_p, _i64, _i64, _p, _p]),
        "oracle_contract": (None, [_p, _p, _i64, _i64, _i64, _i64, _i64, _p]),
        "oracle_epilogue": (None, [_p, _p, _f32, _i64, _i64, _p]),
        "oracle_swiglu": (None, [_p, _p, _p, _f32, _f32, _i64, _i64, _p]),
        "oracle_silu": (ctypes.c_double, [ctypes.c_double]),
        "oracle_pack_weights_grouped": (None, [_p, _i64, _i64, _i64, _f32, _f32, _p, _p, _p]),
        "oracle_contract_grouped": (None, [_p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _p]),
        "oracle_epilogue_grouped": (None, [_p, _p, _p, _i64, _i64, _i64, _p, _p]),
        "oracle_sum_squares": (ctypes.c_double, [_p, _i64]),
        "oracle_rmsnorm_apply": (None, [_p, _p, _i64, _f32, _f32, _p, _p]),
        "oracle_rmsnorm": (None, [_p, _p, _i64, _i64, _f32, _p, _p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _stale() -> bool:
    src = os.path.join(_HERE, "bitnet_oracle.c")
    return os.path.getmtime(src) > os.path.getmtime(_LIB_PATH)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().oracle_bf16_to_f32(_ptr(bits), bits.size, _ptr(out))
    return out


def abs_sum(w: np.ndarray) -> float:
    w = np.ascontiguousarray(w, dtype=np.float32)
    return _load().oracle_abs_sum(_ptr(w), w.size)


def absmean(w: np.ndarray) -> np.float32:
    w = np.ascontiguousarray(w, dtype=np.float32)
    return np.float32(_load().oracle_absmean(_ptr(w), w.size))


def gamma(mean: float, alpha: float = 1.0, eps: float = 1e-8) -> np.float32:
    return np.float32(_load().oracle_gamma(mean, alpha, eps))


def ternarize(g: float, w: float) -> int:
    return int(_load().oracle_ternarize(g, w))


def pack_codes(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8).ravel()
    out = np.empty((q.size + 3) // 4, dtype=np.uint8)
    _load().oracle_pack_codes(_ptr(q), q.size, _ptr(out))
    return out


def unpack_codes(packed: np.ndarray, n: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8).ravel()
    assert packed.size * 4 >= n
    out = np.empty(n, dtype=np.int8)
    _load().oracle_unpack_codes(_ptr(packed), n, _ptr(out))
    return out


def pack_weights(W: np.ndarray, alpha: float = 1.0, eps: float = 1e-8):
    """Returns (packed uint8 [ceil(N*K/4)], beta float32, absmean float32)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    assert W.ndim == 2
    N, K = W.shape
    packed = np.empty((N * K + 3) // 4, dtype=np.uint8)
    beta = np.zeros(1, dtype=np.float32)
    am = np.zeros(1, dtype=np.float32)
    _load().oracle_pack_weights(_ptr(W), N, K, alpha, eps, _ptr(packed), _ptr(beta), _ptr(am))
    return packed, beta[0], am[0]


def quant_act(x: np.ndarray):
    """x fp32 [M, K] -> (x_q int8 [M, K], scale fp32 [M] = per-token absmax)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.ndim == 2
    M, K = x.shape
    xq = np.empty((M, K), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    _load().oracle_quant_act(_ptr(x), M, K, _ptr(xq), _ptr(s))
    return xq, s


def contract(xq: np.ndarray, packed: np.ndarray, N: int, K: int, rows=None, threads: int = 1):
    """int32 acc [M, N]; only rows in ``rows`` (range or None = all) are filled.

    ``threads`` > 1 splits the row range over a thread pool; the C routine
    releases the GIL, each thread computes a disjoint block of rows.
    """
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    M = xq.shape[0]
    assert xq.shape == (M, K) and packed.size * 4 >= N * K
    acc = np.zeros((M, N), dtype=np.int32)
    r0, r1 = (0, N) if rows is None else (rows[0], rows[1])
    lib = _load()
    if threads <= 1 or r1 - r0 < 2:
        lib.oracle_contract(_ptr(xq), _ptr(packed), M, N, K, r0, r1, _ptr(acc))
        return acc
    from concurrent.futures import ThreadPoolExecutor

    bounds = np.linspace(r0, r1, threads + 1).astype(np.int64)
    with ThreadPoolExecutor(threads) as ex:
        futs = [
            ex.submit(lib.oracle_contract, _ptr(xq), _ptr(packed), M, N, K, int(a), int(b), _ptr(acc))
            for a, b in zip(bounds[:-1], bounds[1:]) if b > a
        ]
        for f in futs:
            f.result()
    return acc


def epilogue(acc: np.ndarray, scale: np.ndarray, w_scale: float) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    M, N = acc.shape
    y = np.empty((M, N), dtype=np.float32)
    _load().oracle_epilogue(_ptr(acc), _ptr(scale), w_scale, M, N, _ptr(y))
    return y


def bitlinear(x: np.ndarray, packed: np.ndarray, beta: float, N: int, K: int, threads: int = 1):
    """Whole decode/prefill path: quant_act -> contraction -> epilogue."""
    xq, s = quant_act(x)
    acc = contract(xq, packed, N, K, threads=threads)
    return epilogue(acc, s, beta), acc, xq, s


def silu(z: float) -> float:
    return float(_load().oracle_silu(float(z)))


def swiglu(acc_gate: np.ndarray, acc_up: np.ndarray, scale: np.ndarray, w_scale_gate: float,
           w_scale_up: float) -> np.ndarray:
    """fp64 [M, I]: silu(y_gate) * y_up from the exact BitLinear outputs."""
    acc_gate = np.ascontiguousarray(acc_gate, dtype=np.int32)
    acc_up = np.ascontiguousarray(acc_up, dtype=np.int32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    M, I = acc_gate.shape
    assert acc_up.shape == (M, I)
    out = np.empty((M, I), dtype=np.float64)
    _load().oracle_swiglu(_ptr(acc_gate), _ptr(acc_up), _ptr(scale), w_scale_gate, w_scale_up, M, I, _ptr(out))
    return out


def bitlinear_swiglu(x: np.ndarray, packed_gate: np.ndarray, beta_gate: float, packed_up: np.ndarray,
                     beta_up: float, I: int, K: int, threads: int = 1):
    """The FFN front half: quant_act -> two contractions -> silu(gate) * up (fp64)."""
    xq, s = quant_act(x)
    acc_g = contract(xq, packed_gate, I, K, threads=threads)
    acc_u = contract(xq, packed_up, I, K, threads=threads)
    return swiglu(acc_g, acc_u, s, beta_gate, beta_up), acc_g, acc_u, xq, s


def pack_weights_grouped(W: np.ndarray, G: int, alpha: float = 1.0, eps: float = 1e-8):
    """Group-wise ternarisation: every G consecutive weights of a row are one
    group with its own gamma and beta.  Returns (packed uint8 [N*K/4],
    w_scale float32 [N, K/G] (beta per group), absmean float32 [N, K/G])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    assert G > 0 and G % 4 == 0 and K % G == 0
    packed = np.empty(N * K // 4, dtype=np.uint8)
    ws = np.empty((N, K // G), dtype=np.float32)
    am = np.empty((N, K // G), dtype=np.float32)
    _load().oracle_pack_weights_grouped(_ptr(W), N, K, G, alpha, eps, _ptr(packed), _ptr(ws), _ptr(am))
    return packed, ws, am


def contract_grouped(xq: np.ndarray, packed: np.ndarray, N: int, K: int, G: int, threads: int = 1) -> np.ndarray:
    """int32 [M, N, K/G]: the integer product of each weight group."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    M = xq.shape[0]
    assert xq.shape == (M, K) and packed.size * 4 >= N * K and K % G == 0
    acc = np.empty((M, N, K // G), dtype=np.int32)
    lib = _load()
    if threads <= 1 or N < 2 * threads:
        lib.oracle_contract_grouped(_ptr(xq), _ptr(packed), M, N, K, G, 0, N, _ptr(acc))
        return acc
    from concurrent.futures import ThreadPoolExecutor

    bounds = np.linspace(0, N, threads + 1).astype(np.int64)
    with ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(lib.oracle_contract_grouped, _ptr(xq), _ptr(packed), M, N, K, G, int(a), int(b),
                          _ptr(acc)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        for f in futs:
            f.result()
    return acc


def epilogue_grouped(acc_g: np.ndarray, scale: np.ndarray, w_scale: np.ndarray):
    """(y, cond), fp64 [M, N]: y = s/127 * sum_g w_scale[n, g] * acc_g, and
    cond = s/127 * sum_g |w_scale[n, g] * acc_g| (the rounding condition)."""
    acc_g = np.ascontiguousarray(acc_g, dtype=np.int32)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    w_scale = np.ascontiguousarray(w_scale, dtype=np.float32)
    M, N, ng = acc_g.shape
    assert w_scale.shape == (N, ng)
    y = np.empty((M, N), dtype=np.float64)
    cond = np.empty((M, N), dtype=np.float64)
    _load().oracle_epilogue_grouped(_ptr(acc_g), _ptr(scale), _ptr(w_scale), M, N, ng, _ptr(y), _ptr(cond))
    return y, cond


def bitlinear_grouped(x: np.ndarray, packed: np.ndarray, w_scale: np.ndarray, N: int, K: int, G: int,
                      threads: int = 1):
    """BitLinear forward with group scales: quant_act -> per-group products
    -> y (fp64), cond, acc_g, x_q, s."""
    xq, s = quant_act(x)
    acc_g = contract_grouped(xq, packed, N, K, G, threads=threads)
    y, cond = epilogue_grouped(acc_g, s, w_scale)
    return y, cond, acc_g, xq, s


def bitlinear_fake_quant(W: np.ndarray, x: np.ndarray, weight_scale=None, alpha: float = 1.0, eps: float = 1e-8,
                         threads: int = 1):
    """The training-time BitLinear forward of [Deep-dive] section 3.1: the fp32
    shadow weights are ternarised on every call (absmean, section 2.2), the
    activations absmax-quantised, the integer product rescaled by act_scale
    (absmax / 127) and by the per-output weight_scale (a learned [N] vector;
    beta when None).  The straight-through estimator of section 2.4 only
    changes the backward pass.  Returns (y, cond, acc, xq, s, packed, beta):
    y fp64 with cond = |y| bound input as in epilogue_grouped when
    weight_scale is given, else y fp32 rounded once (epilogue) and cond None."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    packed, beta, _ = pack_weights(W, alpha, eps)
    if weight_scale is None:
        y, acc, xq, s = bitlinear(x, packed, beta, N, K, threads=threads)
        return y, None, acc, xq, s, packed, beta
    ws = np.ascontiguousarray(weight_scale, dtype=np.float32).reshape(N, 1)
    y, cond, acc_g, xq, s = bitlinear_grouped(x, packed, ws, N, K, K, threads=threads)
    return y, cond, acc_g[:, :, 0], xq, s, packed, beta


# nn.RMSNorm's default eps for fp32 inputs: the machine epsilon of fp32
RMS_EPS = 2.0 ** -23


def sum_squares(x: np.ndarray) -> float:
    """S = sum x_k^2 of one token, fp64, left to right."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return float(_load().oracle_sum_squares(_ptr(x), x.size))


def rmsnorm(x: np.ndarray, g=None, eps: float = RMS_EPS):
    """RMSNorm per token of x fp32 [M, K] with weight g [K] (None = ones):
    returns (h fp32 [M, K], ms fp32 [M], the mean squares)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.ndim == 2
    M, K = x.shape
    h = np.empty((M, K), dtype=np.float32)
    ms = np.empty(M, dtype=np.float32)
    gp = None
    if g is not None:
        g = np.ascontiguousarray(g, dtype=np.float32).ravel()
        assert g.size == K
        gp = _ptr(g)
    _load().oracle_rmsnorm(_ptr(x), gp, M, K, eps, _ptr(h), _ptr(ms))
    return h, ms


def rmsnorm_apply(x_row: np.ndarray, ms: float, g=None, eps: float = RMS_EPS):
    """One token normalised with a given fp32 mean square: (h [K], r)."""
    x_row = np.ascontiguousarray(x_row, dtype=np.float32).ravel()
    K = x_row.size
    h = np.empty(K, dtype=np.float32)
    r = np.zeros(1, dtype=np.float32)
    gp = None
    if g is not None:
        g = np.ascontiguousarray(g, dtype=np.float32).ravel()
        assert g.size == K
        gp = _ptr(g)
    _load().oracle_rmsnorm_apply(_ptr(x_row), gp, K, np.float32(ms), eps, _ptr(h), _ptr(r))
    return h, np.float32(r[0])


def bitlinear_rmsnorm(x: np.ndarray, g, packed: np.ndarray, beta: float, N: int, K: int, eps: float = RMS_EPS,
                      threads: int = 1):
    """RMSNorm, then the BitLinear forward: returns (y, acc, xq, s, h, ms)."""
    h, ms = rmsnorm(x, g, eps)
    y, acc, xq, s = bitlinear(h, packed, beta, N, K, threads=threads)
    return y, acc, xq, s, h, ms
