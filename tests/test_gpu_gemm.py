"""tcgen05 prefill GEMM (through the C ABI) versus the CPU oracle: exact int32
accumulators, fp32 outputs within 1e-6 relative; plus GEMM == GEMV where both
apply."""
import numpy as np
import pytest

from test_gpu_parity import assert_y_close, to_dev

pytestmark = pytest.mark.gpu


def gemm_case(lib, oracle_mod, dev, M, N, K, seed, extreme=False):
    rng = np.random.default_rng(seed)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    if extreme:
        q[: N // 2] = 1
    packed = oracle_mod.pack_codes(q)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    if extreme:
        xq[: M // 2] = 127
        xq[M // 2:] = -127
    s = (rng.random(M) * 5 + 0.01).astype(np.float32)
    beta = np.float32(0.6899)
    acc_ref = oracle_mod.contract(xq, packed, N, K, threads=8)
    y_ref = oracle_mod.epilogue(acc_ref, s, float(beta))
    y, acc = lib.w2a8_gemm(to_dev(xq, dev), to_dev(s, dev), to_dev(packed, dev), to_dev(np.array([beta]), dev),
                           N, K, want_acc=True)
    a = acc.cpu().numpy()
    if not np.array_equal(a, acc_ref):
        bad = np.argwhere(a != acc_ref)
        raise AssertionError(f"{len(bad)} accumulator mismatches, first {bad[:5].tolist()}: "
                             f"{a[tuple(bad[0])]} vs {acc_ref[tuple(bad[0])]}")
    assert_y_close(y.cpu().numpy(), y_ref)


@pytest.mark.parametrize("M,N,K", [(128, 128, 512), (1, 128, 512), (256, 1024, 1024), (200, 300, 2560),
                                   (129, 257, 2624), (384, 256, 576), (512, 512, 6912), (1000, 130, 1536)])
def test_gemm_tensor_core_path(lib, oracle_mod, cuda_dev, M, N, K):
    gemm_case(lib, oracle_mod, cuda_dev, M, N, K, seed=M + 7 * N + 13 * K)


# more tiles than SMs with a last wave under half full: the tail tiles are
# split by K across all CTAs (stream-K) and summed in the workspace.  150
# tiles (2 split, K = 1024: 32 units over 148 CTAs, most CTAs one 64-K block),
# 160 tiles (12 split, K = 2560: segments crossing tile boundaries), ragged M
# and N, and the extreme-magnitude accumulators through the split.
@pytest.mark.parametrize("M,N,K", [(300, 9600, 1024), (512, 10240, 2560), (300, 9500, 1088)])
def test_gemm_stream_k_tail(lib, oracle_mod, cuda_dev, M, N, K):
    gemm_case(lib, oracle_mod, cuda_dev, M, N, K, seed=M + N + K)


def test_gemm_stream_k_extreme_and_workspace_reuse(lib, oracle_mod, cuda_dev):
    import torch

    M, N, K = 300, 9600, 2048
    ws = torch.full((lib.gemm_workspace_bytes(M, N, K),), 0xAB, dtype=torch.uint8, device=cuda_dev)
    rng = np.random.default_rng(11)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    q[: N // 2] = 1
    packed = oracle_mod.pack_codes(q)
    for rep in range(2):  # the workspace starts with garbage, then holds the previous call's leftovers
        xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
        xq[: M // 3] = 127
        s = (rng.random(M) * 5 + 0.01).astype(np.float32)
        y, acc = lib.w2a8_gemm(to_dev(xq, cuda_dev), to_dev(s, cuda_dev), to_dev(packed, cuda_dev),
                               to_dev(np.array([np.float32(0.5)]), cuda_dev), N, K, want_acc=True, workspace=ws)
        acc_ref = oracle_mod.contract(xq, packed, N, K, threads=8)
        assert np.array_equal(acc.cpu().numpy(), acc_ref), rep
        assert_y_close(y.cpu().numpy(), oracle_mod.epilogue(acc_ref, s, 0.5))
    lib.check_device_error()


def test_gemm_extreme_accumulators(lib, oracle_mod, cuda_dev):
    # |acc| = 127 * K = 1,040,384 at K = 8192: the largest magnitude the fp32
    # accumulation must still hold exactly
    gemm_case(lib, oracle_mod, cuda_dev, 256, 256, 8192, seed=3, extreme=True)


@pytest.mark.parametrize("M,N,K", [(3, 5, 12), (130, 33, 100), (64, 40, 448)])
def test_gemm_generic_path(lib, oracle_mod, cuda_dev, M, N, K):
    gemm_case(lib, oracle_mod, cuda_dev, M, N, K, seed=M + N + K)


@pytest.mark.parametrize("M", [1, 7, 64])
def test_gemm_equals_gemv(lib, oracle_mod, cuda_dev, M):
    import torch

    rng = np.random.default_rng(M)
    N, K = 700, 2560
    packed = oracle_mod.pack_codes(rng.integers(-1, 2, size=(N, K)).astype(np.int8))
    xq = to_dev(rng.integers(-127, 128, size=(M, K)).astype(np.int8), cuda_dev)
    s = to_dev((rng.random(M) + 0.5).astype(np.float32), cuda_dev)
    b = to_dev(np.array([0.7], np.float32), cuda_dev)
    pk = to_dev(packed, cuda_dev)
    y1, a1 = lib.w2a8_gemm(xq, s, pk, b, N, K, want_acc=True)
    y2, a2 = lib.w2a8_gemv(xq, s, pk, b, N, K, want_acc=True)
    assert torch.equal(a1, a2)
    assert torch.equal(y1, y2)
