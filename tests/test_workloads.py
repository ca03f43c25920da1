"""The seeded synthetic inputs: deterministic, the stated shapes and statistics."""
import torch

from bit_weight_quantization_02_b300 import workloads as wl


def test_weights_are_deterministic_and_bf16():
    a = wl.gen_weight(64, 128, seed=5, outliers=True)
    b = wl.gen_weight(64, 128, seed=5, outliers=True)
    c = wl.gen_weight(64, 128, seed=6, outliers=True)
    assert a.dtype == torch.bfloat16 and a.shape == (64, 128)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_weight_statistics_and_outliers():
    w = wl.gen_weight(1024, 1024, seed=1).float()
    assert abs(w.std().item() - 0.02) < 5e-4
    wo = wl.gen_weight(1024, 1024, seed=1, outliers=True).float()
    frac = (wo != w).float().mean().item()
    assert 0.0007 < frac < 0.0013  # Bernoulli(0.001) mask, each hit scaled by 10
    ratio = (wo[wo != w] / w[wo != w])
    assert torch.allclose(ratio, torch.full_like(ratio, 10.0), rtol=1e-2)


def test_activations():
    x = wl.gen_activation(8, 4096, seed=3).float()
    assert abs(x.std().item() - 1.0) < 0.02


def test_configs_match_the_stated_workloads():
    assert [(c.N, c.K, c.group_size, c.M) for c in wl.config1()] == [(512, 512, 32, 1)]
    c2 = wl.config2()
    assert [(c.N, c.K) for c in c2] == [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),
                                        (14336, 4096), (14336, 4096), (4096, 14336)]
    assert all(c.group_size == 32 and c.M == 1 and c.outliers for c in c2)
    c3 = wl.config3()
    assert sorted({c.M for c in c3}) == [2, 4, 8, 16, 32] and all(c.group_size == 64 for c in c3)
    c4 = wl.config4()
    assert sorted({c.M for c in c4}) == [2048, 8192] and all(c.group_size == 32 for c in c4)
    c5 = wl.config5(1)
    assert len(c5) == 224 and all(c.group_size == 128 for c in c5)
    assert wl.config5_weight_count() == 6_979_321_856
    assert len({c.w_seed for c in c5}) == 224
