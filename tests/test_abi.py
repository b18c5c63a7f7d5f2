"""The C-ABI library loads, exports every declared symbol and rejects bad
arguments on the host before touching the GPU (no GPU needed)."""
import glob
import os
import re

import pytest

from conftest import ROOT

INVALID_ARG, SHAPE, WORKSPACE = 1, 2, 7


@pytest.fixture(scope="module")
def clib():
    from ternary_weight_05_b300 import _lib, build

    build.build()
    return _lib.load()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(bitnet_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ["bitnet_pack_weights", "bitnet_quant_act", "bitnet_w2a8_gemv", "bitnet_w2a8_gemm"]:
        assert required in names


def test_library_exports_every_declared_symbol(clib):
    from ternary_weight_05_b300 import _lib

    for name in declared_symbols():
        assert hasattr(clib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(clib):
    assert clib.bitnet_status_string(0) == b"BITNET_OK"
    assert clib.bitnet_status_string(6) == b"BITNET_ERR_TIMEOUT"
    assert clib.bitnet_status_string(99) == b"BITNET_ERR_UNKNOWN"
    assert clib.bitnet_version() >= 100


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def test_quant_act_validation(clib):
    assert clib.bitnet_quant_act(None, 0, 1, 8, FAKE, FAKE, None) == INVALID_ARG
    assert clib.bitnet_quant_act(FAKE, 3, 1, 8, FAKE, FAKE, None) == INVALID_ARG
    assert clib.bitnet_quant_act(FAKE, 0, 0, 8, FAKE, FAKE, None) == SHAPE
    assert clib.bitnet_quant_act(FAKE, 1, 4, -1, FAKE, FAKE, None) == SHAPE


def test_pack_validation(clib):
    ws = clib.bitnet_pack_workspace_bytes(16, 64)
    assert ws >= 256 + 8
    assert clib.bitnet_pack_workspace_bytes(16, 6) == 0
    args = lambda **kw: dict(dict(W=FAKE, dt=0, N=16, K=64, a=1.0, e=1e-8, p=FAKE, b=FAKE, am=None, ws=FAKE,
                                  wsb=ws), **kw)

    def call(**kw):
        a = args(**kw)
        return clib.bitnet_pack_weights(a["W"], a["dt"], a["N"], a["K"], a["a"], a["e"], a["p"], a["b"], a["am"],
                                        a["ws"], a["wsb"], None)

    assert call(W=None) == INVALID_ARG
    assert call(p=None) == INVALID_ARG
    assert call(dt=5) == INVALID_ARG
    assert call(a=float("nan")) == INVALID_ARG
    assert call(e=float("inf")) == INVALID_ARG
    assert call(K=6) == SHAPE
    assert call(N=0) == SHAPE
    assert call(ws=None) == WORKSPACE
    assert call(wsb=ws - 1) == WORKSPACE


@pytest.mark.parametrize("fn", ["bitnet_w2a8_gemv", "bitnet_w2a8_gemm"])
def test_matmul_validation(clib, fn):
    f = getattr(clib, fn)

    def call(xq=FAKE, s=FAKE, M=1, p=FAKE, ws_=FAKE, N=8, K=64, y=FAKE, work=FAKE, wb=1 << 20):
        return f(xq, s, M, p, ws_, N, K, y, None, work, wb, None)

    assert call(xq=None) == INVALID_ARG
    assert call(y=None) == INVALID_ARG
    assert call(ws_=None) == INVALID_ARG
    assert call(K=10) == SHAPE
    assert call(M=0) == SHAPE
    assert call(N=-3) == SHAPE
    assert call(work=None) == WORKSPACE
    if fn == "bitnet_w2a8_gemv":
        assert call(M=65) == SHAPE


ALIGNMENT = 3


def test_bitlinear_validation(clib):
    nb = clib.bitnet_bitlinear_workspace_bytes(1, 8, 64)
    assert nb > 0 and clib.bitnet_bitlinear_workspace_bytes(1, 8, 6) == 0

    def call(x=FAKE, dt=1, M=1, p=FAKE, w=FAKE, N=8, K=64, y=FAKE, work=FAKE, wb=nb):
        return clib.bitnet_bitlinear(x, dt, M, p, w, N, K, y, None, None, None, work, wb, None)

    assert call(x=None) == INVALID_ARG
    assert call(y=None) == INVALID_ARG
    assert call(dt=2) == INVALID_ARG
    assert call(M=0) == SHAPE
    assert call(K=10) == SHAPE
    assert call(x=FAKE + 1) == ALIGNMENT
    assert call(work=None) == WORKSPACE
    assert call(wb=nb - 1) == WORKSPACE
    assert call(work=FAKE + 16) == WORKSPACE  # not 256-byte aligned


def test_grouped_ws_validation(clib):
    nb = clib.bitnet_grouped_workspace_bytes(16, 300, 2560, 128)
    assert nb >= clib.bitnet_bitlinear_grouped_workspace_bytes(16, 2560) and nb > 0
    assert clib.bitnet_grouped_workspace_bytes(16, 300, 2560, 100) == 0  # G does not divide K

    def call(xq=FAKE, M=16, N=300, K=2560, G=128, y=FAKE, work=FAKE, wb=nb):
        return clib.bitnet_w2a8_grouped_ws(xq, FAKE, M, FAKE, FAKE, N, K, G, y, None, work, wb, None)

    assert call(xq=None) == INVALID_ARG
    assert call(y=None) == INVALID_ARG
    assert call(M=0) == SHAPE
    assert call(G=100) == SHAPE
    assert call(y=FAKE + 2) == ALIGNMENT
    assert call(work=None) == WORKSPACE
    assert call(wb=nb - 1) == WORKSPACE
    assert call(work=FAKE + 64) == WORKSPACE


def test_rmsnorm_validation(clib):
    def quant(x=FAKE, dt=1, M=1, K=64, g=None, eps=2.0 ** -23, xq=FAKE, s=FAKE, h=None):
        return clib.bitnet_rmsnorm_quant_act(x, dt, M, K, g, eps, xq, s, h, None, None)

    assert quant(x=None) == INVALID_ARG
    assert quant(s=None) == INVALID_ARG
    assert quant(dt=5) == INVALID_ARG
    assert quant(eps=-1.0) == INVALID_ARG
    assert quant(eps=float("nan")) == INVALID_ARG
    assert quant(M=0) == SHAPE
    assert quant(K=12) == SHAPE  # K % 8 != 0
    assert quant(x=FAKE + 8) == ALIGNMENT
    assert quant(g=FAKE + 4) == ALIGNMENT
    assert quant(h=FAKE + 4) == ALIGNMENT
    nb = clib.bitnet_bitlinear_workspace_bytes(2, 8, 64)

    def bl(x=FAKE, g=None, eps=2.0 ** -23, K=64, y=FAKE, work=FAKE, wb=nb):
        return clib.bitnet_bitlinear_rmsnorm(x, 1, 2, g, eps, FAKE, FAKE, 8, K, y, None, None, None, None, work, wb,
                                             None)

    assert bl(x=None) == INVALID_ARG
    assert bl(y=None) == INVALID_ARG
    assert bl(eps=float("inf")) == INVALID_ARG
    assert bl(K=60) == SHAPE  # K % 8 != 0
    assert bl(g=FAKE + 8) == ALIGNMENT
    assert bl(work=None) == WORKSPACE
    assert bl(wb=nb - 1) == WORKSPACE


def test_bitlinear_swiglu_validation(clib):
    nb = clib.bitnet_bitlinear_swiglu_workspace_bytes(2, 8, 64)
    # the fallback's two [M, I] fp32 outputs come on top of the BitLinear's
    assert nb >= clib.bitnet_bitlinear_workspace_bytes(2, 8, 64) + 2 * 2 * 8 * 4
    assert clib.bitnet_bitlinear_swiglu_workspace_bytes(0, 8, 64) == 0

    def call(x=FAKE, dt=0, M=2, pg=FAKE, wg=FAKE, pu=FAKE, wu=FAKE, I=8, K=64, out=FAKE, work=FAKE, wb=nb):
        return clib.bitnet_bitlinear_swiglu(x, dt, M, pg, wg, pu, wu, I, K, out, None, None, None, None, work, wb,
                                            None)

    for kw in ("x", "pg", "wg", "pu", "wu", "out"):
        assert call(**{kw: None}) == INVALID_ARG, kw
    assert call(dt=7) == INVALID_ARG
    assert call(M=-1) == SHAPE
    assert call(I=0) == SHAPE
    assert call(K=66) == SHAPE
    assert call(wu=FAKE + 2) == ALIGNMENT
    assert call(work=None) == WORKSPACE
    assert call(wb=nb - 1) == WORKSPACE


def test_grouped_validation(clib):
    def pack(W=FAKE, dt=0, N=4, K=256, G=128, p=FAKE, w=FAKE):
        return clib.bitnet_pack_weights_grouped(W, dt, N, K, G, 1.0, 1e-8, p, w, None, None)

    assert pack(W=None) == INVALID_ARG
    assert pack(w=None) == INVALID_ARG
    assert pack(dt=9) == INVALID_ARG
    assert pack(G=0) == SHAPE
    assert pack(G=6) == SHAPE      # not a multiple of 4
    assert pack(G=96) == SHAPE     # does not divide K
    assert pack(w=FAKE + 2) == ALIGNMENT

    def mm(xq=FAKE, s=FAKE, M=1, p=FAKE, w=FAKE, N=8, K=256, G=64, y=FAKE):
        return clib.bitnet_w2a8_grouped(xq, s, M, p, w, N, K, G, y, None, None)

    assert mm(xq=None) == INVALID_ARG
    assert mm(w=None) == INVALID_ARG
    assert mm(M=0) == SHAPE
    assert mm(G=48) == SHAPE
    assert mm(y=FAKE + 1) == ALIGNMENT

    nb = clib.bitnet_bitlinear_grouped_workspace_bytes(2, 256)
    assert nb >= 2 * 256 + 8 and clib.bitnet_bitlinear_grouped_workspace_bytes(0, 256) == 0

    def bl(x=FAKE, dt=1, M=2, G=64, work=FAKE, wb=nb):
        return clib.bitnet_bitlinear_grouped(x, dt, M, FAKE, FAKE, 8, 256, G, FAKE, None, None, None, work, wb, None)

    assert bl(x=None) == INVALID_ARG
    assert bl(dt=3) == INVALID_ARG
    assert bl(G=100) == SHAPE
    assert bl(x=FAKE + 1) == ALIGNMENT
    assert bl(work=None) == WORKSPACE
    assert bl(wb=nb - 1) == WORKSPACE


def test_fake_quant_validation(clib):
    nb = clib.bitnet_bitlinear_fake_quant_workspace_bytes(2, 8, 64)
    assert nb >= 8 * 64 // 4 + clib.bitnet_bitlinear_workspace_bytes(2, 8, 64)
    assert clib.bitnet_bitlinear_fake_quant_workspace_bytes(2, 8, 6) == 0

    def call(W=FAKE, wd=0, x=FAKE, xd=1, M=2, N=8, K=64, a=1.0, e=1e-8, wsc=None, y=FAKE, work=FAKE, wb=nb):
        return clib.bitnet_bitlinear_fake_quant(W, wd, x, xd, M, N, K, a, e, wsc, y, None, None, None, None, None,
                                                work, wb, None)

    assert call(W=None) == INVALID_ARG
    assert call(x=None) == INVALID_ARG
    assert call(wd=4) == INVALID_ARG
    assert call(a=float("nan")) == INVALID_ARG
    assert call(K=62) == SHAPE
    assert call(M=0) == SHAPE
    assert call(wsc=FAKE + 1) == ALIGNMENT
    assert call(work=None) == WORKSPACE
    assert call(wb=nb - 1) == WORKSPACE


def test_workspace_sizes_cover_partials(clib):
    for M, N, K in [(1, 2560, 2560), (16, 28672, 8192), (64, 13824, 2560), (3, 129, 1000)]:
        nb = clib.bitnet_gemv_workspace_bytes(M, N, K)
        assert nb >= ((N + 127) // 128) * 128 * M * 4
    assert clib.bitnet_gemv_workspace_bytes(65, 8, 64) == 0
    assert clib.bitnet_gemm_workspace_bytes(2048, 6912, 2560) > 0


def test_gemm_workspace_covers_the_split_tail(clib):
    # 2048 tokens x 2560 rows: 8 x 20 = 160 tiles of 256 x 128 on 148 SMs,
    # a last wave of 12 tiles whose K loops are split across the CTAs: the
    # workspace holds their int32 partial sums (256 x 128 each) and tickets
    xb = 2048 * 6912 * 2
    split = clib.bitnet_gemm_workspace_bytes(2048, 2560, 6912)
    assert split >= xb + 2048 * 8 + 12 * 256 * 128 * 4 + 12 * 16 * 4
    # 2048 x 6912: 432 tiles, a last wave of 136 (over half full): no split
    whole = clib.bitnet_gemm_workspace_bytes(2048, 6912, 2560)
    assert whole == ((2048 * 2560 * 2 + 1023) // 1024) * 1024 + ((2048 * 8 + 255) // 256) * 256 + 1024


def test_selftest_wait_validation(clib):
    assert clib.bitnet_selftest_wait_timeout(10, None) == INVALID_ARG          # below 1 us
    assert clib.bitnet_selftest_wait_timeout(2_000_000_000, None) == INVALID_ARG  # above 1 s


def test_package_fails_loudly_without_library(tmp_path, monkeypatch):
    from ternary_weight_05_b300 import _lib

    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError):
        _lib.load()


def test_binding_rejects_host_tensors():
    """The Python binding never computes on the host: every entry point
    raises on CPU tensors before anything reaches the library."""
    import torch

    import ternary_weight_05_b300 as tw

    W = torch.zeros((8, 64))
    x = torch.zeros((1, 64), dtype=torch.bfloat16)
    xq = torch.zeros((1, 64), dtype=torch.int8)
    s = torch.ones(1)
    packed = torch.zeros((8, 16), dtype=torch.uint8)
    beta = torch.ones(1)
    calls = [
        lambda: tw.pack_weights(W),
        lambda: tw.quant_act(x),
        lambda: tw.w2a8_gemv(xq, s, packed, beta, 8, 64),
        lambda: tw.w2a8_gemm(xq, s, packed, beta, 8, 64),
        lambda: tw.w2a8_gemv_static_scratch(xq, s, packed, beta, 8, 64),
        lambda: tw.bitlinear(x, packed, beta, 8, 64),
        lambda: tw.bitlinear_swiglu(x, packed, beta, packed, beta, 8, 64),
        lambda: tw.pack_weights_grouped(W, 32),
        lambda: tw.w2a8_grouped(xq, s, packed, torch.ones((8, 2)), 8, 64, 32),
        lambda: tw.bitlinear_grouped(x, packed, torch.ones((8, 2)), 8, 64, 32),
        lambda: tw.bitlinear_fake_quant(W, x),
    ]
    for i, call in enumerate(calls):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()


def test_injected_cuda_failure_reaches_every_caller(clib):
    """Host-side failure path: with failures injected at the device query,
    every entry point that enqueues work returns BITNET_ERR_CUDA after its
    argument checks, before any other CUDA call, one injected failure each
    (the composite calls stop at their first device query)."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("the calls below pass placeholder pointers: host-only test")
    CUDA = 5
    nb_bl = clib.bitnet_bitlinear_workspace_bytes(2, 8, 64)
    nb_sw = clib.bitnet_bitlinear_swiglu_workspace_bytes(2, 8, 64)
    nb_gr = clib.bitnet_bitlinear_grouped_workspace_bytes(2, 256)
    nb_fq = clib.bitnet_bitlinear_fake_quant_workspace_bytes(2, 8, 64)
    nb_pk = clib.bitnet_pack_workspace_bytes(16, 64)
    calls = {
        "pack_weights": lambda: clib.bitnet_pack_weights(FAKE, 0, 16, 64, 1.0, 1e-8, FAKE, FAKE, None, FAKE, nb_pk,
                                                         None),
        "quant_act": lambda: clib.bitnet_quant_act(FAKE, 0, 1, 8, FAKE, FAKE, None),
        "w2a8_gemv": lambda: clib.bitnet_w2a8_gemv(FAKE, FAKE, 1, FAKE, FAKE, 8, 64, FAKE, None, FAKE, 1 << 20, None),
        "w2a8_gemm": lambda: clib.bitnet_w2a8_gemm(FAKE, FAKE, 300, FAKE, FAKE, 8, 64, FAKE, None, FAKE, 1 << 22,
                                                   None),
        "static_scratch": lambda: clib.bitnet_w2a8_gemv_static_scratch(FAKE, FAKE, 1, FAKE, FAKE, 8, 64, FAKE, None,
                                                                      None),
        "bitlinear": lambda: clib.bitnet_bitlinear(FAKE, 1, 1, FAKE, FAKE, 8, 64, FAKE, None, None, None, FAKE, nb_bl,
                                                   None),
        "swiglu": lambda: clib.bitnet_bitlinear_swiglu(FAKE, 0, 2, FAKE, FAKE, FAKE, FAKE, 8, 64, FAKE, None, None,
                                                       None, None, FAKE, nb_sw, None),
        "pack_grouped": lambda: clib.bitnet_pack_weights_grouped(FAKE, 0, 4, 256, 128, 1.0, 1e-8, FAKE, FAKE, None,
                                                                 None),
        "w2a8_grouped": lambda: clib.bitnet_w2a8_grouped(FAKE, FAKE, 1, FAKE, FAKE, 8, 256, 64, FAKE, None, None),
        "bitlinear_grouped": lambda: clib.bitnet_bitlinear_grouped(FAKE, 1, 2, FAKE, FAKE, 8, 256, 64, FAKE, None,
                                                                   None, None, FAKE, nb_gr, None),
        "fake_quant": lambda: clib.bitnet_bitlinear_fake_quant(FAKE, 0, FAKE, 1, 2, 8, 64, 1.0, 1e-8, None, FAKE,
                                                               None, None, None, None, None, FAKE, nb_fq, None),
        "selftest": lambda: clib.bitnet_selftest_wait_timeout(2_000_000, None),
        "w2a8_grouped_ws": lambda: clib.bitnet_w2a8_grouped_ws(FAKE, FAKE, 4, FAKE, FAKE, 8, 512, 128, FAKE, None,
                                                               FAKE, 1 << 22, None),
        "rmsnorm_quant": lambda: clib.bitnet_rmsnorm_quant_act(FAKE, 1, 2, 64, None, 2.0 ** -23, FAKE, FAKE, None,
                                                               None, None),
        "bitlinear_rmsnorm": lambda: clib.bitnet_bitlinear_rmsnorm(FAKE, 1, 2, FAKE, 2.0 ** -23, FAKE, FAKE, 8, 64,
                                                                   FAKE, None, None, None, None, FAKE, nb_bl, None),
    }
    n = len(calls) + 3
    assert clib.bitnet_test_inject_cuda_failures(n) == 0
    try:
        for i, (name, call) in enumerate(calls.items()):
            assert call() == CUDA, name
            # exactly one injected failure consumed: the call went no further
            left = clib.bitnet_test_inject_cuda_failures(n - i - 1)
            assert left == n - i - 1, (name, left)
    finally:
        assert clib.bitnet_test_inject_cuda_failures(0) == 3
