"""The row split of a BitLinear across ranks (ternary_weight_05_b300.shard):
the bounds cover every output row once, and the ranks' slices, each computed
on its own rows of the packed matrix with the whole matrix's scale, assemble
into the unsplit result -- checked with the oracle as the per-rank worker, on
two gloo ranks on the CPU."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

from conftest import ROOT
from ternary_weight_05_b300 import shard, synth


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("N", [0, 1, 5, 127, 128, 129, 1000, 2560, 6912, 28672, 28673])
def test_row_bounds_partition(N, world):
    b = [shard.row_bounds(N, world, r) for r in range(world)]
    assert b[0][0] == 0 and b[-1][1] == N
    for (a0, a1), (c0, c1) in zip(b, b[1:]):
        assert a1 == c0  # contiguous, in rank order
    sizes = [r1 - r0 for r0, r1 in b]
    assert all(s >= 0 for s in sizes) and sum(sizes) == N
    if N >= 128 * world:
        # whole 128-row tiles except the last range's tail; at most one tile apart
        assert all(r0 % 128 == 0 for r0, _ in b)
        full = [s for s in sizes[:-1]]
        assert max(sizes) - min(sizes) <= 128
        assert all(s % 128 == 0 for s in full)
    else:
        assert max(sizes) - min(sizes) <= 1


def test_row_bounds_rejects_bad_rank():
    with pytest.raises(ValueError):
        shard.row_bounds(10, 2, 2)
    with pytest.raises(ValueError):
        shard.row_bounds(10, 0, 0)


def test_packed_rows_are_the_rows(oracle_mod):
    """The byte range of rows [r0, r1) is the packed matrix of those rows:
    its products are the unsplit products' columns r0..r1."""
    import torch

    N, K = 300, 1024
    W = synth.weights_np(N, K, "laplace", 0.01, seed=3)
    p, beta, _ = oracle_mod.pack_weights(W)
    _, xf = synth.acts_np(3, K, "normal", seed=4)
    xq, s = oracle_mod.quant_act(xf)
    full = oracle_mod.contract(xq, p, N, K)
    for world in (2, 3):
        for r in range(world):
            r0, r1 = shard.row_bounds(N, world, r, align=64)
            sub = shard.packed_rows(torch.from_numpy(p), K, r0, r1).numpy()
            assert sub.size == (r1 - r0) * K // 4
            assert np.array_equal(oracle_mod.contract(xq, sub, r1 - r0, K), full[:, r0:r1])
            sub2 = shard.packed_rows(torch.from_numpy(p.reshape(N, K // 4)), K, r0, r1).numpy().ravel()
            assert np.array_equal(sub2, sub)


_RANK_CODE = r"""
import os, sys, json
sys.path.insert(0, os.environ["BENCH_ROOT"])
import numpy as np
import torch
import torch.distributed as dist
dist.init_process_group("gloo")
import oracle
from ternary_weight_05_b300 import shard, synth
rank, world = dist.get_rank(), dist.get_world_size()
N, K, M = 1000, 2048, 4
W = synth.weights_np(N, K, "laplace", 0.01, seed=11)
p, beta, _ = oracle.pack_weights(W)        # the whole matrix's pack and beta
_, xf = synth.acts_np(M, K, "normal", seed=12)
r0, r1 = shard.row_bounds(N, world, rank)
mine = shard.packed_rows(torch.from_numpy(p), K, r0, r1).numpy()
y_loc, acc_loc, _, _ = oracle.bitlinear(xf, mine, beta, r1 - r0, K)
y = shard.gather_rows(torch.from_numpy(y_loc), N, world, rank)
acc = shard.gather_rows(torch.from_numpy(acc_loc), N, world, rank)
y_ref, acc_ref, _, _ = oracle.bitlinear(xf, p, beta, N, K)
ok = bool(np.array_equal(acc.numpy(), acc_ref)) and bool(np.array_equal(y.numpy().view(np.uint32),
                                                                           y_ref.view(np.uint32)))
print(json.dumps({"rank": rank, "rows": [r0, r1], "ok": ok}), flush=True)
dist.barrier()
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_row_split_two_gloo_ranks(oracle_mod):
    import json

    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), BENCH_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_CODE], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE))
    outs = []
    for p in procs:
        so, se = p.communicate(timeout=180)
        assert p.returncode == 0, se.decode()[-2000:]
        outs.append(json.loads(so.decode().strip().splitlines()[-1]))
    outs.sort(key=lambda o: o["rank"])
    assert outs[0]["rows"] == [0, 512] and outs[1]["rows"] == [512, 1000]
    assert all(o["ok"] for o in outs)
