"""BitNet b1.58 W2A8 ternary matmul for NVIDIA B300 (sm_103a).

Thin Python binding over the C ABI of libbitnet_w2a8.so: torch tensors supply
device memory and the current CUDA stream; every step of the computation runs
in the library's CUDA kernels.  Function names follow the C entry points.

    packed, beta, absmean = pack_weights(W)          # offline, W [N, K]
    x_q, scale = quant_act(x)                         # x [M, K] bf16/fp32
    y = w2a8_gemv(x_q, scale, packed, beta, N, K)     # decode, M <= 64
    y = w2a8_gemm(x_q, scale, packed, beta, N, K)     # prefill
    y = bitlinear(x, packed, beta, N, K)              # fused quant + matmul
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import BitnetError

__all__ = [
    "BitnetError", "pack_weights", "quant_act", "w2a8_gemv", "w2a8_gemm", "bitlinear", "bitlinear_workspace_bytes",
    "pack_workspace_bytes", "gemv_workspace_bytes", "gemm_workspace_bytes", "check_device_error",
    "set_pdl", "GEMV_MAX_M", "library_path", "w2a8_gemv_static_scratch", "GEMV_STATIC_SCRATCH_BYTES",
    "rmsnorm_quant_act", "bitlinear_rmsnorm", "RMS_EPS", "w2a8_grouped", "bitlinear_grouped", "pack_weights_grouped",
    "grouped_workspace_bytes",
]

GEMV_MAX_M = 64
GEMV_STATIC_SCRATCH_BYTES = 4 << 20
F32, BF16 = 0, 1
library_path = _lib.LIB_PATH


def _L():
    return _lib.load()


try:  # the raw handle of the current stream, without building a Stream object
    _raw_stream = torch._C._cuda_getCurrentRawStream
except AttributeError:  # pragma: no cover
    _raw_stream = None


def _stream(dev: torch.device) -> int:
    if _raw_stream is not None:
        return _raw_stream(dev.index if dev.index is not None else torch.cuda.current_device())
    return torch.cuda.current_stream(dev).cuda_stream


# Workspace sizes answered by the library, per (query, shape): the size
# queries are pure functions of the shape, so each is asked once.
_ws_sizes = {}


def _ws_bytes(query: str, *shape) -> int:
    key = (query, shape)
    v = _ws_sizes.get(key)
    if v is None:
        v = int(getattr(_L(), query)(*shape))
        _ws_sizes[key] = v
    return v


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def pack_workspace_bytes(N: int, K: int) -> int:
    """Bytes of device scratch pack_weights needs for an [N, K] matrix."""
    return int(_L().bitnet_pack_workspace_bytes(N, K))


def gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    """Bytes of device scratch w2a8_gemv needs (M <= 64 tokens, N x K weights)."""
    return int(_L().bitnet_gemv_workspace_bytes(M, N, K))


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    """Bytes of device scratch w2a8_gemm needs (M tokens, N x K weights)."""
    return int(_L().bitnet_gemm_workspace_bytes(M, N, K))


def set_pdl(enable: bool) -> None:
    """Launch this thread's kernels with programmatic dependent launch (each
    kernel still waits for its predecessor before touching its outputs)."""
    _L().bitnet_set_pdl(1 if enable else 0)


def check_device_error(stream=None) -> None:
    """Synchronise `stream` (default: the current one) and raise if a kernel's
    bounded wait expired since the last check."""
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _lib.check("bitnet_check_device_error", _L().bitnet_check_device_error(s))


class _WorkspaceCache:
    """Device workspaces for calls made without an explicit one, keyed by
    (device, kind, stream).

    Every entry point takes its workspace with any contents (the kernels
    zero, in stream order, whatever they accumulate into), so one buffer per
    key is reused across shapes; calls on different streams get different
    buffers.  A buffer is replaced by a larger one when a larger shape
    arrives, and the old one is freed: a CUDA-graph capture must therefore
    pass an explicit workspace that outlives the graph.
    """

    def __init__(self):
        self._bufs = {}

    def get(self, dev: torch.device, kind: str, nbytes: int, stream_id: int) -> torch.Tensor:
        key = (dev.index, kind, stream_id)
        buf = self._bufs.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
            self._bufs[key] = buf
        return buf


_ws = _WorkspaceCache()


def pack_weights(W: torch.Tensor, alpha: float = 1.0, eps: float = 1e-8):
    """Absmean-ternarise and 2-bit pack W [N, K] (fp32 or bf16, on the GPU).

    Returns (packed uint8 [N, K//4], beta float32 [1], absmean float32 [1]).
    """
    _dev(W, "W")
    if W.dim() != 2:
        raise ValueError("W must be 2-D [N, K]")
    N, K = W.shape
    dev = W.device
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=dev)
    beta = torch.empty(1, dtype=torch.float32, device=dev)
    absmean = torch.empty(1, dtype=torch.float32, device=dev)
    nbytes = max(pack_workspace_bytes(N, K), 256)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = _L().bitnet_pack_weights(W.data_ptr(), _dtype_code(W), N, K, alpha, eps, packed.data_ptr(),
                                  beta.data_ptr(), absmean.data_ptr(), ws.data_ptr(), nbytes, _stream(dev))
    _lib.check("bitnet_pack_weights", st)
    return packed, beta, absmean


def quant_act(x: torch.Tensor, out=None):
    """Per-token absmax int8 quantisation of x [M, K]: returns (x_q int8, scale f32 [M])."""
    _dev(x, "x")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    if out is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=x.device)
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
    else:
        x_q, scale = out
    st = _L().bitnet_quant_act(x.data_ptr(), _dtype_code(x), M, K, x_q.data_ptr(), scale.data_ptr(),
                               _stream(x.device))
    _lib.check("bitnet_quant_act", st)
    return x_q, scale


def _matmul(fn_name, ws_fn, kind, x_q, scale, packed, w_scale, N, K, want_acc, out, workspace):
    for t, nm in ((x_q, "x_q"), (scale, "scale"), (packed, "packed"), (w_scale, "w_scale")):
        _dev(t, nm)
    M = x_q.shape[0]
    dev = x_q.device
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N), dtype=torch.int32, device=dev) if want_acc else None
    stream = _stream(dev)
    if workspace is None:
        workspace = _ws.get(dev, kind, _ws_bytes(ws_fn, M, N, K), stream)
    st = getattr(_L(), fn_name)(x_q.data_ptr(), scale.data_ptr(), M, packed.data_ptr(), w_scale.data_ptr(), N, K,
                                y.data_ptr(), acc.data_ptr() if acc is not None else None,
                                workspace.data_ptr(), workspace.numel(), stream)
    _lib.check(fn_name, st)
    return (y, acc) if want_acc else y


def w2a8_gemv(x_q, scale, packed, w_scale, N: int, K: int, want_acc: bool = False, out=None, workspace=None):
    """Decode GEMV (M <= 64): y [M, N] fp32 (and the exact int32 acc if asked)."""
    return _matmul("bitnet_w2a8_gemv", "bitnet_gemv_workspace_bytes", "gemv", x_q, scale, packed, w_scale, N, K,
                   want_acc, out, workspace)


def w2a8_gemm(x_q, scale, packed, w_scale, N: int, K: int, want_acc: bool = False, out=None, workspace=None):
    """Prefill GEMM (any M): y [M, N] fp32 (and the exact int32 acc if asked)."""
    return _matmul("bitnet_w2a8_gemm", "bitnet_gemm_workspace_bytes", "gemm", x_q, scale, packed, w_scale, N, K,
                   want_acc, out, workspace)


def w2a8_gemv_static_scratch(x_q, scale, packed, w_scale, N: int, K: int, want_acc: bool = False, out=None):
    """Decode GEMV like w2a8_gemv, for callers that cannot allocate device
    scratch: the library's fixed 4 MiB device array is used instead of a
    workspace (shapes that need more raise BitnetError TOO_LARGE).  Calls
    that may overlap on the GPU share that array and must not run
    concurrently.  The output tensors are still allocated here by torch
    unless `out` is given."""
    for t, nm in ((x_q, "x_q"), (scale, "scale"), (packed, "packed"), (w_scale, "w_scale")):
        _dev(t, nm)
    M = x_q.shape[0]
    dev = x_q.device
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N), dtype=torch.int32, device=dev) if want_acc else None
    st = _L().bitnet_w2a8_gemv_static_scratch(x_q.data_ptr(), scale.data_ptr(), M, packed.data_ptr(),
                                              w_scale.data_ptr(), N, K, y.data_ptr(),
                                              acc.data_ptr() if acc is not None else None, _stream(dev))
    _lib.check("bitnet_w2a8_gemv_static_scratch", st)
    return (y, acc) if want_acc else y


def bitlinear_workspace_bytes(M: int, N: int, K: int) -> int:
    """Bytes of device scratch bitlinear needs."""
    return int(_L().bitnet_bitlinear_workspace_bytes(M, N, K))


def bitlinear(x: torch.Tensor, packed: torch.Tensor, w_scale: torch.Tensor, N: int, K: int, want_acc: bool = False,
              want_xq: bool = False, out=None, workspace=None):
    """Fused BitLinear forward (absmax quantisation inside the matmul kernels).

    x [M, K] bf16/fp32 -> y fp32 [M, N]; with want_acc / want_xq also the exact
    int32 accumulators and (x_q int8 [M, K], scale fp32 [M]).
    """
    for t, nm in ((x, "x"), (packed, "packed"), (w_scale, "w_scale")):
        _dev(t, nm)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M = x.shape[0]
    dev = x.device
    if out is not None:
        _dev(out, "out")
        y = out
    else:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N), dtype=torch.int32, device=dev) if want_acc else None
    xq = torch.empty((M, K), dtype=torch.int8, device=dev) if want_xq else None
    sc = torch.empty(M, dtype=torch.float32, device=dev) if want_xq else None
    stream = _stream(dev)
    if workspace is None:
        workspace = _ws.get(dev, "bitlinear", _ws_bytes("bitnet_bitlinear_workspace_bytes", M, N, K), stream)
    st = _L().bitnet_bitlinear(x.data_ptr(), _dtype_code(x), M, packed.data_ptr(), w_scale.data_ptr(), N, K,
                               y.data_ptr(), xq.data_ptr() if want_xq else None,
                               sc.data_ptr() if want_xq else None, acc.data_ptr() if want_acc else None,
                               workspace.data_ptr(), workspace.numel(), stream)
    if st:
        _lib.check("bitnet_bitlinear", st)
    res = (y,)
    if want_acc:
        res += (acc,)
    if want_xq:
        res += (xq, sc)
    return res[0] if len(res) == 1 else res


RMS_EPS = 2.0 ** -23  # nn.RMSNorm's default eps for fp32


def rmsnorm_quant_act(x: torch.Tensor, g=None, eps: float = RMS_EPS, want_h: bool = False, want_ms: bool = False):
    """RMSNorm of x [M, K] (bf16/fp32, K % 8 == 0) with weight g [K] (None:
    ones), then per-token absmax int8 quantisation of the normalised h.

    Returns (x_q int8 [M, K], scale f32 [M]) and, if asked, h f32 [M, K] and
    the mean squares f32 [M]."""
    _dev(x, "x")
    if g is not None:
        _dev(g, "g")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    dev = x.device
    xq = torch.empty((M, K), dtype=torch.int8, device=dev)
    sc = torch.empty(M, dtype=torch.float32, device=dev)
    h = torch.empty((M, K), dtype=torch.float32, device=dev) if want_h else None
    ms = torch.empty(M, dtype=torch.float32, device=dev) if want_ms else None
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    st = _L().bitnet_rmsnorm_quant_act(x.data_ptr(), _dtype_code(x), M, K, ptr(g), eps, xq.data_ptr(), sc.data_ptr(),
                                       ptr(h), ptr(ms), _stream(dev))
    _lib.check("bitnet_rmsnorm_quant_act", st)
    res = (xq, sc)
    if want_h:
        res += (h,)
    if want_ms:
        res += (ms,)
    return res


def bitlinear_rmsnorm(x: torch.Tensor, g, packed: torch.Tensor, w_scale: torch.Tensor, N: int, K: int,
                      eps: float = RMS_EPS, want_acc: bool = False, want_xq: bool = False, want_ms: bool = False,
                      out=None, workspace=None):
    """BitLinear forward on RMSNorm(x): y fp32 [M, N]; g [K] fp32 or None;
    with want_acc the exact int32 products, want_xq (x_q, scale), want_ms the
    mean squares."""
    for t, nm in ((x, "x"), (packed, "packed"), (w_scale, "w_scale")):
        _dev(t, nm)
    if g is not None:
        _dev(g, "g")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M = x.shape[0]
    dev = x.device
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N), dtype=torch.int32, device=dev) if want_acc else None
    xq = torch.empty((M, K), dtype=torch.int8, device=dev) if want_xq else None
    sc = torch.empty(M, dtype=torch.float32, device=dev) if want_xq else None
    ms = torch.empty(M, dtype=torch.float32, device=dev) if want_ms else None
    stream = _stream(dev)
    if workspace is None:
        workspace = _ws.get(dev, "bitlinear", _ws_bytes("bitnet_bitlinear_workspace_bytes", M, N, K), stream)
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    st = _L().bitnet_bitlinear_rmsnorm(x.data_ptr(), _dtype_code(x), M, ptr(g), eps, packed.data_ptr(),
                                       w_scale.data_ptr(), N, K, y.data_ptr(), ptr(xq), ptr(sc), ptr(ms), ptr(acc),
                                       workspace.data_ptr(), workspace.numel(), stream)
    _lib.check("bitnet_bitlinear_rmsnorm", st)
    res = (y,)
    if want_acc:
        res += (acc,)
    if want_xq:
        res += (xq, sc)
    if want_ms:
        res += (ms,)
    return res[0] if len(res) == 1 else res


def bitlinear_swiglu_workspace_bytes(M: int, I: int, K: int) -> int:
    """Bytes of device scratch bitlinear_swiglu needs (I rows in each of gate and up)."""
    return int(_L().bitnet_bitlinear_swiglu_workspace_bytes(M, I, K))


def bitlinear_swiglu(x: torch.Tensor, packed_gate: torch.Tensor, w_scale_gate: torch.Tensor,
                     packed_up: torch.Tensor, w_scale_up: torch.Tensor, I: int, K: int, want_acc: bool = False,
                     want_xq: bool = False, out=None, workspace=None):
    """Front half of the BitLinear feed-forward: silu(gate(x)) * up(x), fp32 [M, I].

    packed_gate / packed_up are [I, K/4] uint8 (two views of one [2I, K/4]
    fused gate+up matrix work too); with want_acc also the exact int32
    products (acc_gate, acc_up), with want_xq the int8 activations and scales.
    """
    for t, nm in ((x, "x"), (packed_gate, "packed_gate"), (w_scale_gate, "w_scale_gate"),
                  (packed_up, "packed_up"), (w_scale_up, "w_scale_up")):
        _dev(t, nm)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M = x.shape[0]
    dev = x.device
    a = out if out is not None else torch.empty((M, I), dtype=torch.float32, device=dev)
    acc_g = torch.empty((M, I), dtype=torch.int32, device=dev) if want_acc else None
    acc_u = torch.empty((M, I), dtype=torch.int32, device=dev) if want_acc else None
    xq = torch.empty((M, K), dtype=torch.int8, device=dev) if want_xq else None
    sc = torch.empty(M, dtype=torch.float32, device=dev) if want_xq else None
    nbytes = bitlinear_swiglu_workspace_bytes(M, I, K)
    stream = _stream(dev)
    if workspace is None:
        workspace = _ws.get(dev, "bitlinear_swiglu", nbytes, stream)
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    st = _L().bitnet_bitlinear_swiglu(x.data_ptr(), _dtype_code(x), M, packed_gate.data_ptr(),
                                      w_scale_gate.data_ptr(), packed_up.data_ptr(), w_scale_up.data_ptr(), I, K,
                                      a.data_ptr(), ptr(xq), ptr(sc), ptr(acc_g), ptr(acc_u), workspace.data_ptr(),
                                      workspace.numel(), stream)
    _lib.check("bitnet_bitlinear_swiglu", st)
    res = (a,)
    if want_acc:
        res += (acc_g, acc_u)
    if want_xq:
        res += (xq, sc)
    return res[0] if len(res) == 1 else res


def pack_weights_grouped(W: torch.Tensor, G: int, alpha: float = 1.0, eps: float = 1e-8):
    """Group-wise absmean ternarisation of W [N, K] (fp32 / bf16, on the GPU):
    every G consecutive weights of a row form a group with its own gamma and
    beta (G = K: per output channel).

    Returns (packed uint8 [N, K//4], w_scale float32 [N, K//G] (beta per
    group), absmean float32 [N, K//G])."""
    _dev(W, "W")
    if W.dim() != 2:
        raise ValueError("W must be 2-D [N, K]")
    N, K = W.shape
    dev = W.device
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=dev)
    ng = K // G if G > 0 else 0
    w_scale = torch.empty((N, ng), dtype=torch.float32, device=dev)
    absmean = torch.empty((N, ng), dtype=torch.float32, device=dev)
    st = _L().bitnet_pack_weights_grouped(W.data_ptr(), _dtype_code(W), N, K, G, alpha, eps, packed.data_ptr(),
                                          w_scale.data_ptr(), absmean.data_ptr(), _stream(dev))
    _lib.check("bitnet_pack_weights_grouped", st)
    return packed, w_scale, absmean


def grouped_workspace_bytes(M: int, N: int, K: int, G: int) -> int:
    """Bytes of device scratch the group-scaled calls need on their tensor-core path."""
    return int(_L().bitnet_grouped_workspace_bytes(M, N, K, G))


def w2a8_grouped(x_q, scale, packed, w_scale, N: int, K: int, G: int, want_acc: bool = False, out=None,
                 workspace=None):
    """Ternary matmul with group scales w_scale [N, K//G], any M: y fp32 [M, N]
    (and the exact per-group int32 products [M, N, K//G] if asked).  Three or
    more tokens run on the tensor cores when the shape allows (a workspace
    is taken from the cache unless given)."""
    for t, nm in ((x_q, "x_q"), (scale, "scale"), (packed, "packed"), (w_scale, "w_scale")):
        _dev(t, nm)
    M = x_q.shape[0]
    dev = x_q.device
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N, K // G), dtype=torch.int32, device=dev) if want_acc else None
    stream = _stream(dev)
    if workspace is None:
        workspace = _ws.get(dev, "grouped", _ws_bytes("bitnet_grouped_workspace_bytes", M, N, K, G), stream)
    st = _L().bitnet_w2a8_grouped_ws(x_q.data_ptr(), scale.data_ptr(), M, packed.data_ptr(), w_scale.data_ptr(), N,
                                     K, G, y.data_ptr(), acc.data_ptr() if acc is not None else None,
                                     workspace.data_ptr(), workspace.numel(), stream)
    _lib.check("bitnet_w2a8_grouped_ws", st)
    return (y, acc) if want_acc else y


def bitlinear_grouped(x: torch.Tensor, packed: torch.Tensor, w_scale: torch.Tensor, N: int, K: int, G: int,
                      want_acc: bool = False, want_xq: bool = False, out=None, workspace=None):
    """BitLinear forward with group scales: x [M, K] bf16/fp32 -> y fp32 [M, N];
    with want_acc also the per-group products, with want_xq (x_q, scale)."""
    for t, nm in ((x, "x"), (packed, "packed"), (w_scale, "w_scale")):
        _dev(t, nm)
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M = x.shape[0]
    dev = x.device
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N, K // G), dtype=torch.int32, device=dev) if want_acc else None
    xq = torch.empty((M, K), dtype=torch.int8, device=dev) if want_xq else None
    sc = torch.empty(M, dtype=torch.float32, device=dev) if want_xq else None
    stream = _stream(dev)
    if workspace is None:
        workspace = _ws.get(dev, "bitlinear_grouped", _ws_bytes("bitnet_grouped_workspace_bytes", M, N, K, G), stream)
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    st = _L().bitnet_bitlinear_grouped(x.data_ptr(), _dtype_code(x), M, packed.data_ptr(), w_scale.data_ptr(), N, K,
                                       G, y.data_ptr(), ptr(xq), ptr(sc), ptr(acc), workspace.data_ptr(),
                                       workspace.numel(), stream)
    _lib.check("bitnet_bitlinear_grouped", st)
    res = (y,)
    if want_acc:
        res += (acc,)
    if want_xq:
        res += (xq, sc)
    return res[0] if len(res) == 1 else res


def bitlinear_grouped_workspace_bytes(M: int, K: int) -> int:
    """Bytes of device scratch bitlinear_grouped needs."""
    return int(_L().bitnet_bitlinear_grouped_workspace_bytes(M, K))


def bitlinear_fake_quant(W: torch.Tensor, x: torch.Tensor, weight_scale=None, alpha: float = 1.0, eps: float = 1e-8,
                         want_acc: bool = False, want_packed: bool = False, out=None, workspace=None):
    """Training-time BitLinear forward: the shadow weights W [N, K] (fp32/bf16)
    are ternarised on this call, x [M, K] quantised per token, y fp32 [M, N]
    rescaled by weight_scale [N] (learned per-output scale) or by beta.
    With want_acc also the exact int32 products, with want_packed the packed
    weights and beta of this call."""
    for t, nm in ((W, "W"), (x, "x")):
        _dev(t, nm)
    if weight_scale is not None:
        _dev(weight_scale, "weight_scale")
    if W.dim() != 2 or x.dim() != 2:
        raise ValueError("W must be [N, K] and x [M, K]")
    N, K = W.shape
    M = x.shape[0]
    dev = x.device
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=dev)
    acc = torch.empty((M, N), dtype=torch.int32, device=dev) if want_acc else None
    packed = torch.empty((N, K // 4), dtype=torch.uint8, device=dev) if want_packed else None
    beta = torch.empty(1, dtype=torch.float32, device=dev) if want_packed else None
    nbytes = bitlinear_fake_quant_workspace_bytes(M, N, K)
    stream = _stream(dev)
    if workspace is None:
        workspace = _ws.get(dev, "bitlinear_fake_quant", nbytes, stream)
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    st = _L().bitnet_bitlinear_fake_quant(W.data_ptr(), _dtype_code(W), x.data_ptr(), _dtype_code(x), M, N, K, alpha,
                                          eps, ptr(weight_scale), y.data_ptr(), ptr(packed), ptr(beta), None, None,
                                          ptr(acc), workspace.data_ptr(), workspace.numel(), stream)
    _lib.check("bitnet_bitlinear_fake_quant", st)
    res = (y,)
    if want_acc:
        res += (acc,)
    if want_packed:
        res += (packed, beta)
    return res[0] if len(res) == 1 else res


def bitlinear_fake_quant_workspace_bytes(M: int, N: int, K: int) -> int:
    """Bytes of device scratch bitlinear_fake_quant needs (the packed copy of W included)."""
    return int(_L().bitnet_bitlinear_fake_quant_workspace_bytes(M, N, K))


def selftest_wait_timeout(limit_ns: int = 2_000_000, stream=None) -> None:
    """Run the failure-path self-test: a kernel whose bounded on-chip wait
    expires after limit_ns records a timeout in the device error word (the
    next check_device_error raises BitnetError TIMEOUT)."""
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _lib.check("bitnet_selftest_wait_timeout", _L().bitnet_selftest_wait_timeout(int(limit_ns), s))
