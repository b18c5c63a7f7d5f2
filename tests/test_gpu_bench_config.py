"""The exact configurations bench.py times, against the oracle.

  * the 100B-class layer stream (28672 x 8192 Laplace weights, bf16
    activations): the fused BitLinear call, the kernels the default line
    times, on layers 0 and 29 at M = 1 (the streaming kernel with the bf16
    prologue at its full-register edge, K = 8192) and M = 16 (the fused prep
    kernel + the tensor-core GEMV), on sampled rows that include rows 0 and
    N - 1;
  * the benchmark's launch configuration: bench.build_stack and
    bench.capture_passes (fused BitLinears, CUDA graph of several passes,
    programmatic dependent launch), replayed, every layer checked after the
    replays -- the 100B stream (3 layers) and the whole 150-BitLinear 2B
    decode stack (every output).
Packed bytes are checked byte for byte where the oracle packs the same W;
int32 products and int8 activations exactly; fp32 outputs within 1e-6
relative.
"""
import os
import sys

import numpy as np
import pytest

from conftest import ROOT
from test_gpu_parity import assert_y_close, to_dev
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu

if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _rows(N, n, seed):
    rows = np.random.default_rng(seed).choice(N, n, replace=False)
    return np.unique(np.concatenate([rows, [0, N - 1]]))


def _check_rows(oracle_mod, xf, p_ref, beta, K, y, acc, rows):
    """y and acc ([M, N] host arrays) on `rows` against the oracle's BitLinear
    of those rows (the oracle quantises x itself)."""
    kb = K // 4
    xq_ref, s_ref = oracle_mod.quant_act(xf)
    sub = np.concatenate([p_ref[r * kb:(r + 1) * kb] for r in rows])
    a_ref = oracle_mod.contract(xq_ref, sub, len(rows), K, threads=8)
    y_ref = oracle_mod.epilogue(a_ref, s_ref, beta)
    if acc is not None:
        assert np.array_equal(acc[:, rows], a_ref)
    assert_y_close(y[:, rows], y_ref)
    return xq_ref, s_ref


@pytest.mark.parametrize("li", [0, 29])
def test_100b_stream_fused_bitlinear(lib, oracle_mod, cuda_dev, li):
    import torch

    L = synth.workload("100b-stream").layers[li]
    W = synth.weights_np(L.N, L.K, L.w_dist, L.w_scale, seed=L.w_seed)
    packed, beta, _ = lib.pack_weights(to_dev(W, cuda_dev))
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    del W
    assert np.array_equal(packed.cpu().numpy().ravel(), p_ref) and beta.item() == float(b_ref)
    rows = _rows(L.N, 384, seed=li)
    for M in (1, 16):
        bits, xf = synth.acts_np(M, L.K, L.x_dist, seed=L.x_seed + M)
        ws = torch.empty(lib.bitlinear_workspace_bytes(M, L.N, L.K), dtype=torch.uint8, device=cuda_dev)
        ws.fill_(0xA5)  # any contents
        y, acc, xq, s = lib.bitlinear(to_dev(bits, cuda_dev, torch.bfloat16), packed, beta, L.N, L.K,
                                      want_acc=True, want_xq=True, workspace=ws)
        xq_ref, s_ref = _check_rows(oracle_mod, xf, p_ref, float(b_ref), L.K, y.cpu().numpy(), acc.cpu().numpy(),
                                    rows)
        assert np.array_equal(xq.cpu().numpy(), xq_ref) and np.array_equal(s.cpu().numpy(), s_ref)
    lib.check_device_error()


def _bench_stack(args, dev):
    import bench

    wl, stack, M = bench.build_stack(args, dev, rank=0, world=1)
    ws_bytes = max(max(lib_ws(M, e) for e in stack), 256)
    return stack, M, ws_bytes


def lib_ws(M, e):
    import ternary_weight_05_b300 as tw

    return max(tw.gemv_workspace_bytes(M, e["n"], e["L"].K), tw.bitlinear_workspace_bytes(M, e["n"], e["L"].K))


def _replay_bench_graph(lib, dev, argv):
    """Builds the stack as bench.py does, captures its graph of passes with
    PDL on, fills every output with NaN, replays twice; returns the stack
    and the bench arguments."""
    import torch

    import bench

    args = bench.parse(argv)
    stack, M, ws_bytes = _bench_stack(args, dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws.fill_(0x5A)
    stream = torch.cuda.Stream(dev)
    lib.set_pdl(True)
    try:
        with torch.cuda.stream(stream):
            ppg = bench.passes_per_graph(args.tokens)
            graph = bench.capture_passes(stack, ws, True, 0, ppg, stream)
            for e in stack:
                e["y"].fill_(float("nan"))
            for _ in range(2):
                graph.replay()
        torch.cuda.synchronize(dev)
    finally:
        lib.set_pdl(False)
    lib.check_device_error()
    return args, stack, M


def _host_weights(L, rep, dev):
    return synth.weights_torch(L.N, L.K, L.w_dist, L.w_scale, L.w_seed + 1000 * rep, dev).cpu().numpy()


def test_bench_graph_100b_stream(lib, oracle_mod, cuda_dev):
    """bench.py's default decode step (fused BitLinears in a graph of 8
    passes, PDL) on the first 3 layers of the 100B stream."""
    args, stack, M = _replay_bench_graph(lib, cuda_dev, ["--workload", "100b-stream", "--layers", "3",
                                                         "--tokens", "8"])
    assert M == 1 and len(stack) == 3
    for i, e in enumerate(stack):
        L = e["L"]
        W = _host_weights(L, 0, cuda_dev)
        p_ref, b_ref, _ = oracle_mod.pack_weights(W)
        del W
        assert np.array_equal(e["packed"].cpu().numpy().ravel(), p_ref), i
        xf = e["x"].float().cpu().numpy()
        _check_rows(oracle_mod, xf, p_ref, float(b_ref), L.K, e["y"].cpu().numpy(), None, _rows(L.N, 256, 7 + i))


def test_bench_graph_2b_decode_stack(lib, oracle_mod, cuda_dev):
    """bench.py's 2b-decode step: all 150 fused BitLinears of the 30-layer
    stack in one graph with PDL, every output against the oracle."""
    args, stack, M = _replay_bench_graph(lib, cuda_dev, ["--workload", "2b-decode"])
    assert len(stack) == 150 and M == 1
    wl = synth.workload("2b-decode")
    for i, e in enumerate(stack):
        L, rep = e["L"], i // len(wl.layers)
        W = _host_weights(L, rep, cuda_dev)
        p_ref, b_ref, _ = oracle_mod.pack_weights(W)
        assert np.array_equal(e["packed"].cpu().numpy().ravel(), p_ref), i
        assert e["beta"].item() == float(b_ref), i
        xf = e["x"].float().cpu().numpy()
        y_ref, _, _, _ = oracle_mod.bitlinear(xf, p_ref, b_ref, L.N, L.K, threads=8)
        assert_y_close(e["y"].cpu().numpy(), y_ref)
