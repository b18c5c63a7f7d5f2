"""Group-wise and per-channel weight scales on the GPU against the oracle.

Packing (bitnet_pack_weights_grouped) is compared bit for bit: packed bytes,
beta per group and mean|W_g|.  The matmul (bitnet_w2a8_grouped,
bitnet_bitlinear_grouped) is compared bit for bit on the int8 activations,
scales and per-group int32 products; y is compared with the bound of its
fp32 arithmetic: y = fl(F * fl(s / 127)) where F adds K/G group terms
acc_g * scale_g with one rounding per term and per addition (at most K/G + 5
roundings on the streaming path: J <= 4 terms per lane and 5 shuffle
additions; K/G on the generic path; K/G fused multiply-adds plus at most a
few fp32 atomic additions of split row tiles on the tensor-core path), each
at most 2^-24 of the running sum of magnitudes, so |y - y_exact| <=
(K/G + 8) * 2^-24 * cond with cond = (s / 127) * sum_g |acc_g * scale_g|
(computed by the oracle).
"""
import numpy as np
import pytest

from test_gpu_parity import to_dev
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def assert_grouped_close(y, y_ref, cond, ng):
    y = np.asarray(y, dtype=np.float64)
    tol = (ng + 8) * U * cond + 1e-30
    err = np.abs(y - y_ref)
    assert np.all(err <= tol), float((err / tol).max())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,K,G", [(3, 16, 4), (7, 256, 64), (129, 2560, 128), (40, 6912, 6912), (33, 8192, 8192),
                                   (20, 2880, 192), (5, 20000, 5000)])
def test_pack_grouped_vs_oracle(lib, oracle_mod, cuda_dev, dtype, N, K, G):
    import torch

    W = synth.weights_np(N, K, "laplace", 0.01, seed=N + K + G)
    W *= np.exp(np.random.default_rng(G).standard_normal((N, 1))).astype(np.float32)  # rows of different scale
    if dtype == "bf16":
        bits = synth.f32_to_bf16_bits(W)
        W = synth.bf16_bits_to_f32(bits)
        Wd = to_dev(bits, cuda_dev, torch.bfloat16)
    else:
        Wd = to_dev(W, cuda_dev)
    packed, ws, am = lib.pack_weights_grouped(Wd, G)
    p_ref, ws_ref, am_ref = oracle_mod.pack_weights_grouped(W, G)
    assert np.array_equal(packed.cpu().numpy().ravel(), p_ref)
    assert np.array_equal(ws.cpu().numpy(), ws_ref)
    assert np.array_equal(am.cpu().numpy(), am_ref)


def test_pack_grouped_golden(lib, cuda_dev):
    from conftest import load_golden

    g = load_golden("grouped_worked.json")
    packed, ws, am = lib.pack_weights_grouped(to_dev(np.array(g["W"], dtype=np.float32), cuda_dev), g["G"])
    assert packed.cpu().numpy().ravel().tolist() == g["packed"]
    assert ws.cpu().numpy().tolist() == g["w_scale"]
    assert am.cpu().numpy().tolist() == g["absmean"]


def grouped_case(lib, oracle_mod, dev, M, N, K, G, seed, learned=False):
    """Random ternary codes, int8 activations and scales: group scales from
    the pack, or arbitrary signed 'learned' scales."""
    rng = np.random.default_rng(seed)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    packed = oracle_mod.pack_codes(q)
    if learned:
        ws = (rng.standard_normal((N, K // G)) * 0.05).astype(np.float32)
    else:
        ws = (rng.integers(1, G + 1, size=(N, K // G)) / G).astype(np.float32)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    if M > 1:
        xq[-1] = 127  # one token at the extreme magnitude
    s = (rng.random(M) * 4 + 0.01).astype(np.float32)
    y, acc = lib.w2a8_grouped(to_dev(xq, dev), to_dev(s, dev), to_dev(packed, dev), to_dev(ws, dev), N, K, G,
                              want_acc=True)
    acc_ref = oracle_mod.contract_grouped(xq, packed, N, K, G, threads=8)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    y_ref, cond = oracle_mod.epilogue_grouped(acc_ref, s, ws)
    assert_grouped_close(y.cpu().numpy(), y_ref, cond, K // G)


# streaming kernel: M <= 2, G a power of two up to 2048 or G = K; generic
# kernel: more tokens, other G, K % 64 != 0
@pytest.mark.parametrize("M", [1, 2, 3, 9])
@pytest.mark.parametrize("N,K,G", [(300, 2560, 64), (300, 2560, 128), (129, 4096, 2048), (257, 2560, 2560),
                                   (64, 8192, 128), (70, 2880, 192), (33, 1000, 200)])
def test_w2a8_grouped_vs_oracle(lib, oracle_mod, cuda_dev, M, N, K, G):
    if M == 2 and K == 8192:
        pytest.skip("covered by M=1 (two tokens stream rows up to 4096)")
    grouped_case(lib, oracle_mod, cuda_dev, M, N, K, G, seed=M * 1000 + N + K + G)


@pytest.mark.parametrize("M,N,K,G", [(1, 500, 2560, 2560), (2, 500, 4096, 128), (5, 100, 2560, 640)])
def test_w2a8_grouped_learned_signed_scales(lib, oracle_mod, cuda_dev, M, N, K, G):
    grouped_case(lib, oracle_mod, cuda_dev, M, N, K, G, seed=7 + M, learned=True)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("N,K,G", [(300, 2560, 128), (129, 4096, 4096), (100, 2880, 192)])
def test_bitlinear_grouped_vs_oracle(lib, oracle_mod, cuda_dev, dtype, M, N, K, G):
    """Pack on the GPU, then the fused grouped BitLinear, against the oracle's
    pack -> quant_act -> per-group products -> epilogue; and bitwise equal to
    quant_act followed by w2a8_grouped."""
    import torch

    W = synth.weights_np(N, K, "normal", 0.02, seed=N + K)
    bits, xf = synth.acts_np(M, K, "student_t4", seed=M + K, outlier_p=0.002, bf16=(dtype == "bf16"))
    if M > 2:
        xf[1] = 0.0  # an all-zero token
        if bits is not None:
            bits[1] = 0
    x = to_dev(bits, cuda_dev, torch.bfloat16) if dtype == "bf16" else to_dev(xf, cuda_dev)
    packed, ws, _ = lib.pack_weights_grouped(to_dev(W, cuda_dev), G)
    y, acc, xq, s = lib.bitlinear_grouped(x, packed, ws, N, K, G, want_acc=True, want_xq=True)
    p_ref, ws_ref, _ = oracle_mod.pack_weights_grouped(W, G)
    y_ref, cond, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear_grouped(xf, p_ref, ws_ref, N, K, G, threads=8)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_grouped_close(y.cpu().numpy(), y_ref, cond, K // G)
    xq2, s2 = lib.quant_act(x)
    y2 = lib.w2a8_grouped(xq2, s2, packed, ws, N, K, G)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    lib.check_device_error()


@pytest.mark.parametrize("M", [1, 2])
def test_grouped_gateup_layer_full(lib, oracle_mod, cuda_dev, M):
    """The 13824 x 2560 fused gate+up layer with groups of 128, full size."""
    import torch

    N, K, G = 13824, 2560, 128
    W = synth.weights_np(N, K, "normal", 0.02, seed=30)
    bits, xf = synth.acts_np(M, K, "normal", seed=31)
    packed, ws, _ = lib.pack_weights_grouped(to_dev(W, cuda_dev), G)
    p_ref, ws_ref, _ = oracle_mod.pack_weights_grouped(W, G)
    assert np.array_equal(packed.cpu().numpy().ravel(), p_ref) and np.array_equal(ws.cpu().numpy(), ws_ref)
    y, acc = lib.bitlinear_grouped(to_dev(bits, cuda_dev, torch.bfloat16), packed, ws, N, K, G, want_acc=True)
    y_ref, cond, acc_ref, _, _ = oracle_mod.bitlinear_grouped(xf, p_ref, ws_ref, N, K, G, threads=8)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_grouped_close(y.cpu().numpy(), y_ref, cond, K // G)


def test_grouped_graph_pdl(lib, oracle_mod, cuda_dev):
    """Grouped BitLinears captured in a CUDA graph with programmatic dependent
    launch (the benchmark's launch configuration), replayed three times."""
    import torch

    N, K, G = 2560, 2560, 128
    layers = []
    for i in range(3):
        W = synth.weights_np(N, K, "normal", 0.02, seed=60 + i)
        bits, xf = synth.acts_np(1, K, "normal", seed=70 + i, outlier_p=0.001)
        packed, ws, _ = lib.pack_weights_grouped(to_dev(W, cuda_dev), G)
        layers.append(dict(W=W, xf=xf, packed=packed, ws=ws, x=to_dev(bits, cuda_dev, torch.bfloat16),
                           y=torch.empty((1, N), dtype=torch.float32, device=cuda_dev)))
    wsp = torch.zeros(lib.bitlinear_grouped_workspace_bytes(1, K), dtype=torch.uint8, device=cuda_dev)
    stream = torch.cuda.Stream(cuda_dev)
    lib.set_pdl(True)
    try:
        with torch.cuda.stream(stream):
            def step():
                for e in layers:
                    lib.bitlinear_grouped(e["x"], e["packed"], e["ws"], N, K, G, out=e["y"], workspace=wsp)

            step()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            for e in layers:
                e["y"].fill_(float("nan"))
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(cuda_dev)
    finally:
        lib.set_pdl(False)
    for e in layers:
        p_ref, ws_ref, _ = oracle_mod.pack_weights_grouped(e["W"], G)
        y_ref, cond, _, _, _ = oracle_mod.bitlinear_grouped(e["xf"], p_ref, ws_ref, N, K, G, threads=8)
        assert_grouped_close(e["y"].cpu().numpy(), y_ref, cond, K // G)
    lib.check_device_error()


# the tensor-core path (3..64 tokens per chunk, M > 64 in chunks of <= 64):
# G in {64, 128, 256, 512} or one group per row of <= 512 weights, ragged N
# across 128-row tiles and split row tiles (stream-K over 512-K units)
@pytest.mark.parametrize("M", [3, 8, 16, 33, 64, 65, 130])
@pytest.mark.parametrize("N,K,G", [(300, 2560, 64), (1000, 2560, 128), (129, 8192, 256), (257, 4096, 512),
                                   (200, 512, 512)])
def test_w2a8_grouped_tensor_core(lib, oracle_mod, cuda_dev, M, N, K, G):
    assert lib.grouped_workspace_bytes(M, N, K, G) > lib.bitlinear_grouped_workspace_bytes(M, K)
    grouped_case(lib, oracle_mod, cuda_dev, M, N, K, G, seed=M * 77 + N + K + G, learned=(M % 2 == 1))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M", [3, 16, 64, 100])
def test_bitlinear_grouped_tensor_core(lib, oracle_mod, cuda_dev, dtype, M):
    """The fused grouped BitLinear on the tensor-core path (the prep kernel
    quantises, lays out and sums the groups) against the oracle, and bitwise
    equal to quant_act + the int8 grouped matmul on the same path; a
    garbage-filled workspace."""
    import torch

    N, K, G = 700, 2560, 128
    W = synth.weights_np(N, K, "laplace", 0.01, seed=M + 5)
    bits, xf = synth.acts_np(M, K, "student_t4", seed=M + 6, outlier_p=0.002, bf16=(dtype == "bf16"))
    xf[1] = 0.0
    if bits is not None:
        bits[1] = 0
    x = to_dev(bits, cuda_dev, torch.bfloat16) if dtype == "bf16" else to_dev(xf, cuda_dev)
    packed, ws, _ = lib.pack_weights_grouped(to_dev(W, cuda_dev), G)
    work = torch.empty(lib.grouped_workspace_bytes(M, N, K, G), dtype=torch.uint8, device=cuda_dev)
    work.fill_(0xC3)
    y, acc, xq, s = lib.bitlinear_grouped(x, packed, ws, N, K, G, want_acc=True, want_xq=True, workspace=work)
    p_ref, ws_ref, _ = oracle_mod.pack_weights_grouped(W, G)
    y_ref, cond, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear_grouped(xf, p_ref, ws_ref, N, K, G, threads=8)
    assert np.array_equal(xq.cpu().numpy(), xq_ref) and np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_grouped_close(y.cpu().numpy(), y_ref, cond, K // G)
    y2 = lib.w2a8_grouped(xq, s, packed, ws, N, K, G)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    lib.check_device_error()

