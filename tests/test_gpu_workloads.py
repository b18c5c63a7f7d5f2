"""The five workloads at full size on the GPU, against the oracle.

Small workloads are compared element by element; the large ones on sampled
outputs the oracle computes row by row (every sampled row for every token):
  bitlinear-1024  1024x1024, M=1, fp32 activations              full
  2b-decode       q/o 2560^2, gate/up 6912x2560, down 2560x6912  full
  gateup-sweep    13824x2560, M in {1,2,4,8,16,32,64}            full
  prefill-2048    M=2048 x (6912x2560, 2560x6912)                256 sampled rows
  100b-stream     30 x (28672x8192), M in {1,2,16}               pack of layers 0/29
                                                                 byte-exact, beta of
                                                                 all 30, 256 rows
  ffn-2b-decode   gate+up 13824x2560 -> SwiGLU -> down 2560x6912 full (graph, PDL)
Also the decode stack in the launch configuration the benchmark times
(CUDA graph replay with programmatic dependent launch).
"""
import numpy as np
import pytest

from test_gpu_parity import assert_y_close, to_dev
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu


def host_layer(L, M):
    W = synth.weights_np(L.N, L.K, L.w_dist, L.w_scale, seed=L.w_seed)
    bits, xf = synth.acts_np(M, L.K, L.x_dist, seed=L.x_seed, outlier_p=L.outlier_p, bf16=L.x_bf16)
    return W, bits, xf


def run_layer(lib, dev, W, bits, xf, N, K, path):
    import torch

    packed, beta, am = lib.pack_weights(to_dev(W, dev))
    x = to_dev(bits, dev, torch.bfloat16) if bits is not None else to_dev(xf, dev)
    xq, s = lib.quant_act(x)
    fn = lib.w2a8_gemv if path == "gemv" else lib.w2a8_gemm
    y, acc = fn(xq, s, packed, beta, N, K, want_acc=True)
    return packed, beta, xq, s, y, acc


def check_full(oracle_mod, lib, dev, L, M, path="gemv"):
    W, bits, xf = host_layer(L, M)
    packed, beta, xq, s, y, acc = run_layer(lib, dev, W, bits, xf, L.N, L.K, path)
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    assert np.array_equal(packed.cpu().numpy().ravel(), p_ref)
    assert beta.item() == float(b_ref)
    y_ref, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear(xf, p_ref, b_ref, L.N, L.K, threads=8)
    assert np.array_equal(xq.cpu().numpy(), xq_ref) and np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_y_close(y.cpu().numpy(), y_ref)


def test_bitlinear_1024(lib, oracle_mod, cuda_dev):
    wl = synth.workload("bitlinear-1024")
    check_full(oracle_mod, lib, cuda_dev, wl.layers[0], 1)


@pytest.mark.parametrize("idx", range(5))
def test_2b_decode_layers(lib, oracle_mod, cuda_dev, idx):
    wl = synth.workload("2b-decode")
    check_full(oracle_mod, lib, cuda_dev, wl.layers[idx], 1)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_gateup_sweep(lib, oracle_mod, cuda_dev, M):
    wl = synth.workload("gateup-sweep")
    check_full(oracle_mod, lib, cuda_dev, wl.layers[0], M)


def sampled_check(oracle_mod, xq, s, packed_h, beta, y, acc, N, K, rows):
    xq_h = xq.cpu().numpy()
    s_h = s.cpu().numpy()
    y_h = y.cpu().numpy()
    acc_h = acc.cpu().numpy()
    kb = K // 4
    for r in rows:
        a_ref = oracle_mod.contract(xq_h, packed_h[r * kb:(r + 1) * kb], 1, K)[:, 0]
        assert np.array_equal(acc_h[:, r], a_ref), r
        y_ref = oracle_mod.epilogue(a_ref[:, None].astype(np.int32), s_h, beta)[:, 0]
        assert_y_close(y_h[:, r], y_ref)


@pytest.mark.parametrize("idx", [0, 1])
def test_prefill_2048_sampled(lib, oracle_mod, cuda_dev, idx):
    wl = synth.workload("prefill-2048")
    L = wl.layers[idx]
    W, bits, xf = host_layer(L, 2048)
    packed, beta, xq, s, y, acc = run_layer(lib, cuda_dev, W, bits, xf, L.N, L.K, "gemm")
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    assert np.array_equal(packed.cpu().numpy().ravel(), p_ref) and beta.item() == float(b_ref)
    xq_ref, s_ref = oracle_mod.quant_act(xf)
    assert np.array_equal(xq.cpu().numpy(), xq_ref) and np.array_equal(s.cpu().numpy(), s_ref)
    rows = np.random.default_rng(idx).choice(L.N, 256, replace=False)
    rows = np.concatenate([rows, [0, L.N - 1]])
    sampled_check(oracle_mod, xq, s, p_ref, float(b_ref), y, acc, L.N, L.K, rows)


@pytest.mark.slow
def test_100b_stream(lib, oracle_mod, cuda_dev):
    import torch

    wl = synth.workload("100b-stream")
    rng = np.random.default_rng(5)
    for li, L in enumerate(wl.layers):
        W = synth.weights_np(L.N, L.K, L.w_dist, L.w_scale, seed=L.w_seed)
        packed, beta, _ = lib.pack_weights(to_dev(W, cuda_dev))
        p_ref, b_ref, _ = oracle_mod.pack_weights(W)
        assert beta.item() == float(b_ref), li
        if li not in (0, 29):
            continue
        assert np.array_equal(packed.cpu().numpy().ravel(), p_ref), li
        # M = 2 on this matrix runs on the tensor-core GEMV (two tokens, long
        # rows, a large matrix); the fused BitLinear must give the same bits
        for M in (1, 2, 16):
            bits, xf = synth.acts_np(M, L.K, L.x_dist, seed=L.x_seed)
            x = to_dev(bits, cuda_dev, torch.bfloat16)
            xq, s = lib.quant_act(x)
            y, acc = lib.w2a8_gemv(xq, s, packed, beta, L.N, L.K, want_acc=True)
            rows = np.concatenate([rng.choice(L.N, 256, replace=False), [0, L.N - 1]])
            sampled_check(oracle_mod, xq, s, p_ref, float(b_ref), y, acc, L.N, L.K, rows)
            yf, accf = lib.bitlinear(x, packed, beta, L.N, L.K, want_acc=True)
            assert np.array_equal(accf.cpu().numpy(), acc.cpu().numpy()), (li, M)
            assert np.array_equal(yf.cpu().numpy().view(np.uint32), y.cpu().numpy().view(np.uint32)), (li, M)


@pytest.mark.parametrize("pdl", [True, False])
def test_decode_stack_graph_launch(lib, oracle_mod, cuda_dev, pdl):
    """Two layers of the 2b-decode stack captured in a CUDA graph (the
    benchmark's launch configuration) and replayed three times."""
    import torch

    wl = synth.workload("2b-decode")
    entries = []
    for rep in range(2):
        for L in wl.layers:
            W = synth.weights_np(L.N, L.K, L.w_dist, L.w_scale, seed=L.w_seed + 1000 * rep)
            bits, xf = synth.acts_np(1, L.K, L.x_dist, seed=L.x_seed + 1000 * rep, outlier_p=L.outlier_p)
            packed, beta, _ = lib.pack_weights(to_dev(W, cuda_dev))
            entries.append(dict(L=L, W=W, xf=xf, packed=packed, beta=beta,
                                x=to_dev(bits, cuda_dev, torch.bfloat16),
                                xq=torch.empty((1, L.K), dtype=torch.int8, device=cuda_dev),
                                s=torch.empty(1, dtype=torch.float32, device=cuda_dev),
                                y=torch.full((1, L.N), float("nan"), dtype=torch.float32, device=cuda_dev)))
    ws = torch.zeros(max(lib.gemv_workspace_bytes(1, e["L"].N, e["L"].K) for e in entries), dtype=torch.uint8,
                     device=cuda_dev)
    stream = torch.cuda.Stream(cuda_dev)
    lib.set_pdl(pdl)
    try:
        with torch.cuda.stream(stream):
            def step():
                for e in entries:
                    lib.quant_act(e["x"], out=(e["xq"], e["s"]))
                    lib.w2a8_gemv(e["xq"], e["s"], e["packed"], e["beta"], e["L"].N, e["L"].K, out=e["y"],
                                  workspace=ws)

            step()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            for e in entries:
                e["y"].fill_(float("nan"))
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(cuda_dev)
    finally:
        lib.set_pdl(False)
    for e in entries:
        L = e["L"]
        p_ref, b_ref, _ = oracle_mod.pack_weights(e["W"])
        y_ref, _, _, _ = oracle_mod.bitlinear(e["xf"], p_ref, b_ref, L.N, L.K, threads=8)
        assert_y_close(e["y"].cpu().numpy(), y_ref)
    lib.check_device_error()


@pytest.mark.parametrize("M", [1, 2, 4])
def test_ffn_2b_decode_graph_launch(lib, oracle_mod, cuda_dev, M):
    """Two layers of the feed-forward decode workload (fused gate+up matrix,
    SwiGLU, down) captured in a CUDA graph with programmatic dependent launch
    and replayed three times, against the oracle: the SwiGLU product within
    its bound, the down output within its bound given the near-midpoint
    positions of its quantisation."""
    import torch
    from test_gpu_swiglu import assert_down_close, assert_swiglu_close, down_reference

    wl = synth.workload("ffn-2b-decode")
    gu, dn = wl.layers
    I, D = gu.N // 2, gu.K
    h = I * D // 4
    layers = []
    for rep in range(2):
        Wgu = synth.weights_np(gu.N, gu.K, gu.w_dist, gu.w_scale, seed=gu.w_seed + 1000 * rep)
        Wd = synth.weights_np(dn.N, dn.K, dn.w_dist, dn.w_scale, seed=dn.w_seed + 1000 * rep)
        bits, xf = synth.acts_np(M, D, gu.x_dist, seed=gu.x_seed + 1000 * rep, outlier_p=gu.outlier_p)
        pgu, bgu, _ = lib.pack_weights(to_dev(Wgu, cuda_dev))
        pd, bd, _ = lib.pack_weights(to_dev(Wd, cuda_dev))
        layers.append(dict(Wgu=Wgu, Wd=Wd, xf=xf, pg=pgu[:I], pu=pgu[I:], bgu=bgu, pd=pd, bd=bd,
                           x=to_dev(bits, cuda_dev, torch.bfloat16),
                           a=torch.empty((M, I), dtype=torch.float32, device=cuda_dev),
                           y=torch.empty((M, D), dtype=torch.float32, device=cuda_dev)))
    ws = torch.zeros(max(lib.bitlinear_swiglu_workspace_bytes(M, I, D), lib.bitlinear_workspace_bytes(M, D, I)),
                     dtype=torch.uint8, device=cuda_dev)
    stream = torch.cuda.Stream(cuda_dev)
    lib.set_pdl(True)
    try:
        with torch.cuda.stream(stream):
            def step():
                for e in layers:
                    lib.bitlinear_swiglu(e["x"], e["pg"], e["bgu"], e["pu"], e["bgu"], I, D, out=e["a"],
                                         workspace=ws)
                    lib.bitlinear(e["a"], e["pd"], e["bd"], D, I, out=e["y"], workspace=ws)

            step()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            for e in layers:
                e["a"].fill_(float("nan"))
                e["y"].fill_(float("nan"))
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(cuda_dev)
    finally:
        lib.set_pdl(False)
    for e in layers:
        pgu_ref, b_ref, _ = oracle_mod.pack_weights(e["Wgu"])
        pd_ref, bd_ref, _ = oracle_mod.pack_weights(e["Wd"])
        a_ref, accg_ref, _, _, s_ref = oracle_mod.bitlinear_swiglu(e["xf"], pgu_ref[:h], b_ref, pgu_ref[h:], b_ref,
                                                                   I, D, threads=8)
        assert_swiglu_close(e["a"].cpu().numpy(), a_ref, accg_ref, s_ref, float(b_ref))
        dref = down_reference(oracle_mod, dict(a=a_ref, acc_g=accg_ref, s=s_ref, beta_g=float(b_ref)), pd_ref,
                              bd_ref, D, I)
        assert_down_close(e["y"].cpu().numpy(), dref, dref["near"].sum(axis=1))
    lib.check_device_error()
