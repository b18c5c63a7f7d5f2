"""The seeded input generators (host side): bf16 rounding to nearest even,
the documented distributions, determinism, and the workload table."""
import numpy as np
import pytest
import torch

from ternary_weight_05_b300 import synth


def test_bf16_rounding_is_nearest_even_like_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32),
                        np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 65504.0, 1e-30, 0.0, -0.0])])
    bits = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert synth.bf16_bits_to_f32(bits[200000:200001])[0] == 1.0
    back = synth.bf16_bits_to_f32(bits)
    assert np.all(np.abs(back[:200000] - x[:200000]) <= np.abs(x[:200000]) * 2 ** -8)


@pytest.mark.parametrize("dist,scale,p0", [("normal", 0.02, 0.3101), ("laplace", 0.01, 0.3935)])
def test_weight_distributions(dist, scale, p0):
    W = synth.weights_np(512, 1024, dist, scale, seed=3).astype(np.float64)
    assert abs(W.mean()) < 5 * scale / np.sqrt(W.size)
    sd = np.sqrt(2) * scale if dist == "laplace" else scale
    assert abs(W.std() / sd - 1) < 0.01
    # fraction below half the absmean: the zero fraction of the ternarisation
    frac = np.mean(np.abs(W) < 0.5 * np.abs(W).mean())
    assert abs(frac - p0) < 0.005


def test_activation_outliers_and_determinism():
    bits, x = synth.acts_np(64, 4096, "normal", seed=5, outlier_p=0.001)
    bits2, x2 = synth.acts_np(64, 4096, "normal", seed=5, outlier_p=0.001)
    assert np.array_equal(bits, bits2) and np.array_equal(x, x2)
    assert np.array_equal(synth.bf16_bits_to_f32(bits), x)
    big = np.mean(np.abs(x) > 8.0)  # |N(0,1)| > 8 is ~1e-15: these are the x20 outliers
    assert 0.0005 < big < 0.0015
    _, t = synth.acts_np(64, 4096, "student_t4", seed=6, bf16=False)
    assert t.dtype == np.float32 and abs(np.var(t.astype(np.float64)) - 2.0) < 0.3  # Var t(4) = 2


def test_workload_table():
    assert set(synth.WORKLOADS) == {"bitlinear-1024", "2b-decode", "gateup-sweep", "prefill-2048", "100b-stream",
                                    "ffn-2b-decode"}
    wl = synth.workload("100b-stream")
    assert len(wl.layers) == 30 and all(L.N == 28672 and L.K == 8192 for L in wl.layers)
    assert sum(L.N * L.K // 4 for L in wl.layers) == 1761607680
    gu, dn = synth.workload("ffn-2b-decode").layers
    assert (gu.N, gu.K, dn.N, dn.K) == (13824, 2560, 2560, 6912)
    with pytest.raises(KeyError):
        synth.workload("nope")
