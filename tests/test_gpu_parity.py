"""GPU (CUDA library, through the C ABI) versus the CPU oracle, element by
element, on seeded inputs: bit-exact for packed bytes, int8 activations,
scales, beta and int32 accumulators; fp32 outputs within 1e-6 relative."""
import numpy as np
import pytest

from conftest import load_golden
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu

RTOL = 1e-6  # fp32 output tolerance (three fp32 roundings, < 2e-7 relative)


def to_dev(a, dev, dtype=None):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return t if dtype is None else t.view(dtype)


def assert_y_close(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    zero = y_ref == 0
    assert np.all(y[zero] == 0)
    rel = np.abs(y[~zero] - y_ref[~zero]) / np.abs(y_ref[~zero])
    assert rel.size == 0 or rel.max() <= RTOL, rel.max()


# ------------------------------------------------------------- quant_act ---

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
# K spans every kernel variant: scalar (K % 8 != 0), rows held in registers
# with 1, 2, 4 or 8 vectors per thread (K <= 2048, 4096, 8192, 16384), and
# the two-pass loop for longer rows.
@pytest.mark.parametrize("M,K", [(1, 1), (1, 7), (3, 100), (2, 2560), (5, 6912), (17, 8192), (64, 1000), (1, 2048),
                                 (1, 2056), (2, 12288), (1, 16384), (3, 20000), (1, 28672)])
def test_quant_act_random(lib, oracle_mod, cuda_dev, dtype, M, K):
    import torch

    bits, xf = synth.acts_np(M, K, "student_t4", seed=M * 7 + K, outlier_p=0.01, bf16=(dtype == "bf16"))
    if M > 2:
        xf[1] = 0.0
        if bits is not None:
            bits[1] = 0
    x = to_dev(bits, cuda_dev, torch.bfloat16) if dtype == "bf16" else to_dev(xf, cuda_dev)
    xq, s = lib.quant_act(x)
    xq_ref, s_ref = oracle_mod.quant_act(xf)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)


def test_quant_act_every_bf16_value(lib, oracle_mod, cuda_dev):
    # every finite bf16 value, in rows whose absmax is fixed: all roundings
    import torch

    bits_all = np.arange(1 << 16, dtype=np.uint16)
    f = synth.bf16_bits_to_f32(bits_all)
    keep = np.isfinite(f) & (np.abs(f) <= 3.0)
    bits_v = bits_all[keep]
    K = 256
    n = bits_v.size
    M = (n + K - 2) // (K - 1)
    bits = np.zeros((M, K), dtype=np.uint16)
    flat = np.zeros(M * (K - 1), dtype=np.uint16)
    flat[:n] = bits_v
    bits[:, 1:] = flat.reshape(M, K - 1)
    bits[:, 0] = synth.f32_to_bf16_bits(np.float32([3.0]))[0]
    xq, s = lib.quant_act(to_dev(bits, cuda_dev, torch.bfloat16))
    xq_ref, s_ref = oracle_mod.quant_act(synth.bf16_bits_to_f32(bits))
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)


def test_quant_act_golden(lib, cuda_dev):
    g = load_golden("quant_act_worked.json")
    xq, s = lib.quant_act(to_dev(np.array(g["x"], dtype=np.float32), cuda_dev))
    assert xq.cpu().numpy().tolist() == g["x_q"]
    assert s.cpu().numpy().tolist() == [float(np.float32(v)) for v in g["scale"]]


# ------------------------------------------------------------------ pack ---

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,K,dist", [(1, 4, "normal"), (3, 12, "normal"), (7, 100, "laplace"),
                                      (129, 1024, "normal"), (64, 4100, "laplace"), (300, 2560, "normal")])
def test_pack_random(lib, oracle_mod, cuda_dev, dtype, N, K, dist):
    import torch

    W = synth.weights_np(N, K, dist, 0.02, seed=N + K)
    if dtype == "bf16":
        bits = synth.f32_to_bf16_bits(W)
        W = synth.bf16_bits_to_f32(bits)
        Wd = to_dev(bits, cuda_dev, torch.bfloat16)
    else:
        Wd = to_dev(W, cuda_dev)
    packed, beta, am = lib.pack_weights(Wd)
    p_ref, b_ref, am_ref = oracle_mod.pack_weights(W)
    assert np.array_equal(packed.cpu().numpy().ravel(), p_ref)
    assert beta.item() == float(b_ref)
    assert am.item() == float(am_ref)


@pytest.mark.parametrize("name", ["ternarize_worked.json", "ternarize_reciprocal.json"])
def test_pack_golden(lib, cuda_dev, name):
    g = load_golden(name)
    packed, beta, _ = lib.pack_weights(to_dev(np.array(g["W"], dtype=np.float32), cuda_dev))
    assert packed.cpu().numpy().ravel().tolist() == g["packed"]
    assert beta.item() == g["beta"]


def test_pack_all_zero_and_ties(lib, oracle_mod, cuda_dev):
    W = np.zeros((4, 64), dtype=np.float32)
    packed, beta, am = lib.pack_weights(to_dev(W, cuda_dev))
    assert np.all(packed.cpu().numpy() == 0x55) and beta.item() == 0.0 and am.item() == 0.0
    # exact ties at +-0.5 and +-1.5 times 1/gamma, and huge values
    W = np.tile(np.float32([0.5, 1.5, -0.5, -1.5, 1e30, -1e30, 0.0, -0.0]), (8, 2)) * np.float32(0.37)
    p, b, _ = lib.pack_weights(to_dev(W, cuda_dev))
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    assert np.array_equal(p.cpu().numpy().ravel(), p_ref) and b.item() == float(b_ref)


def test_pack_with_pdl_enabled(lib, oracle_mod, cuda_dev):
    """The four pack kernels launched with programmatic dependent launch:
    each waits for its predecessor (absmean sums -> gamma -> codes -> beta),
    repeated back to back on one stream."""
    W = synth.weights_np(1000, 4096, "laplace", 0.01, seed=3)
    p_ref, b_ref, am_ref = oracle_mod.pack_weights(W)
    Wd = to_dev(W, cuda_dev)
    lib.set_pdl(True)
    try:
        outs = [lib.pack_weights(Wd) for _ in range(4)]
    finally:
        lib.set_pdl(False)
    for packed, beta, am in outs:
        assert np.array_equal(packed.cpu().numpy().ravel(), p_ref)
        assert beta.item() == float(b_ref) and am.item() == float(am_ref)


# ------------------------------------------------------------------ GEMV ---

def gemv_case(lib, oracle_mod, dev, M, N, K, seed, offset=0):
    import torch

    rng = np.random.default_rng(seed)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    packed = oracle_mod.pack_codes(q)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    if M > 1:
        xq[-1] = 127  # extreme accumulator magnitudes
    s = (rng.random(M) * 5 + 0.01).astype(np.float32)
    beta = np.float32(rng.random() * 0.5 + 0.4)
    acc_ref = oracle_mod.contract(xq, packed, N, K, threads=8)
    y_ref = oracle_mod.epilogue(acc_ref, s, float(beta))
    pk = torch.zeros(packed.size + 64, dtype=torch.uint8, device=dev)
    pk[offset:offset + packed.size] = to_dev(packed, dev)
    y, acc = lib.w2a8_gemv(to_dev(xq, dev), to_dev(s, dev), pk[offset:offset + packed.size],
                           to_dev(np.array([beta]), dev), N, K, want_acc=True)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_y_close(y.cpu().numpy(), y_ref)


@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16, 17, 32, 33, 64])
@pytest.mark.parametrize("N,K", [(1, 512), (129, 1024), (300, 2560), (257, 2624), (128, 6912)])
def test_gemv_tma_path(lib, oracle_mod, cuda_dev, M, N, K):
    gemv_case(lib, oracle_mod, cuda_dev, M, N, K, seed=M * 1000 + N + K)


@pytest.mark.parametrize("M,N,K", [(1, 7, 4), (3, 5, 12), (2, 33, 100), (5, 64, 448), (64, 9, 1000)])
def test_gemv_generic_path(lib, oracle_mod, cuda_dev, M, N, K):
    gemv_case(lib, oracle_mod, cuda_dev, M, N, K, seed=M + N + K)


@pytest.mark.parametrize("fn", ["gemv", "gemm"])
@pytest.mark.parametrize("M", [1, 3, 20])
def test_matmul_beyond_fp32_exact_k(lib, oracle_mod, cuda_dev, fn, M):
    # K = 66048: every weight +1, every activation 127, so sum code * x reaches
    # 2 * 127 * K > 2^24, past what fp32 tensor-core accumulation holds
    # exactly; such shapes must take an exact path.
    import torch

    N, K = 40, 66048
    q = np.ones((N, K), dtype=np.int8)
    q[1::2, ::3] = -1
    packed = oracle_mod.pack_codes(q)
    xq = np.full((M, K), 127, dtype=np.int8)
    xq[-1, ::5] = -127
    s = np.full(M, 3.0, dtype=np.float32)
    acc_ref = oracle_mod.contract(xq, packed, N, K, threads=8)
    y_ref = oracle_mod.epilogue(acc_ref, s, 0.5)
    f = lib.w2a8_gemv if fn == "gemv" else lib.w2a8_gemm
    y, acc = f(to_dev(xq, cuda_dev), to_dev(s, cuda_dev), to_dev(packed, cuda_dev),
               to_dev(np.array([0.5], np.float32), cuda_dev), N, K, want_acc=True)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_y_close(y.cpu().numpy(), y_ref)


@pytest.mark.parametrize("fn", ["gemv", "gemm"])
@pytest.mark.parametrize("M", [1, 3, 20])
def test_matmul_at_the_fp32_exact_limit(lib, oracle_mod, cuda_dev, fn, M):
    # K = 65536, the longest row the tensor-core paths take: every weight +1
    # and every activation 127 give sum code * x = 2 * 127 * 65536 =
    # 16,646,144 < 2^24, still exact in the fp32 accumulators
    N, K = 40, 65536
    q = np.ones((N, K), dtype=np.int8)
    q[1::2, ::7] = -1
    packed = oracle_mod.pack_codes(q)
    xq = np.full((M, K), 127, dtype=np.int8)
    if M > 1:
        xq[-1, ::5] = -127
    s = np.full(M, 2.0, dtype=np.float32)
    acc_ref = oracle_mod.contract(xq, packed, N, K, threads=8)
    assert acc_ref.max() == K * 127  # the extreme magnitude is reached
    y_ref = oracle_mod.epilogue(acc_ref, s, 0.5)
    f = lib.w2a8_gemv if fn == "gemv" else lib.w2a8_gemm
    y, acc = f(to_dev(xq, cuda_dev), to_dev(s, cuda_dev), to_dev(packed, cuda_dev),
               to_dev(np.array([0.5], np.float32), cuda_dev), N, K, want_acc=True)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_y_close(y.cpu().numpy(), y_ref)


def test_gemv_workspace_any_contents(lib, oracle_mod, cuda_dev):
    # one workspace, filled with garbage, shared by calls of different shapes
    # and paths (tensor-core stream-K, row-range, mma.sync stream-K for
    # K > 65536): each call zeroes what it accumulates into
    import torch

    cases = [(64, 1, 512), (3, 129, 1024), (16, 300, 2560), (1, 257, 2624), (40, 2000, 1024), (5, 24, 66048),
             (3, 129, 1024)]
    nbytes = max(lib.gemv_workspace_bytes(M, N, K) for M, N, K in cases)
    ws = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device=cuda_dev)
    for i, (M, N, K) in enumerate(cases):
        rng = np.random.default_rng(i)
        q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
        packed = oracle_mod.pack_codes(q)
        xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        s = (rng.random(M) + 0.5).astype(np.float32)
        acc_ref = oracle_mod.contract(xq, packed, N, K, threads=8)
        y, acc = lib.w2a8_gemv(to_dev(xq, cuda_dev), to_dev(s, cuda_dev), to_dev(packed, cuda_dev),
                               to_dev(np.array([0.75], np.float32), cuda_dev), N, K, want_acc=True, workspace=ws)
        assert np.array_equal(acc.cpu().numpy(), acc_ref), (M, N, K)
        assert_y_close(y.cpu().numpy(), oracle_mod.epilogue(acc_ref, s, 0.75))


def test_gemv_unaligned_packed_pointer(lib, oracle_mod, cuda_dev):
    gemv_case(lib, oracle_mod, cuda_dev, 4, 100, 1024, seed=5, offset=3)


@pytest.mark.parametrize("M", [1, 16])
def test_gemv_many_ctas_share_row_tiles(lib, oracle_mod, cuda_dev, M):
    # few rows, long K: every row tile is split across CTAs (workspace path),
    # run twice to check the workspace is left zeroed
    for rep in range(2):
        gemv_case(lib, oracle_mod, cuda_dev, M, 200, 16384, seed=77 + rep)


def test_gemv_pipeline_golden(lib, cuda_dev):
    g = load_golden("bitlinear_worked.json")
    # pad K to 512 with zero activations so the TMA path runs
    K = 512
    q = np.zeros((2, K), dtype=np.int8)
    xq = np.zeros((2, K), dtype=np.int8)
    codes = [[1, -1, 0, 1], [0, 0, -1, 1]]
    q[:, :4] = codes
    xq[:, :4] = g["x_q"]
    import oracle

    packed = oracle.pack_codes(q)
    y, acc = lib.w2a8_gemv(to_dev(xq, cuda_dev), to_dev(np.array(g["scale"], np.float32), cuda_dev),
                           to_dev(packed, cuda_dev), to_dev(np.array([g["beta"]], np.float32), cuda_dev),
                           2, K, want_acc=True)
    assert acc.cpu().numpy().tolist() == g["acc"]
    assert y.cpu().numpy().tolist() == g["y"]


def test_bitlinear_end_to_end_small(lib, oracle_mod, cuda_dev):
    import torch

    W = synth.weights_np(384, 1536, "normal", 0.02, seed=3)
    bits, xf = synth.acts_np(5, 1536, "normal", seed=4, outlier_p=0.001)
    packed, beta, _ = lib.pack_weights(to_dev(W, cuda_dev))
    y = lib.bitlinear(to_dev(bits, cuda_dev, torch.bfloat16), packed, beta, 384, 1536)
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    y_ref, _, _, _ = oracle_mod.bitlinear(xf, p_ref, b_ref, 384, 1536)
    assert_y_close(y.cpu().numpy(), y_ref)


def test_no_device_error_after_suite(lib, cuda_dev):
    lib.check_device_error()
