"""The seeded input generator: published SplitMix64 outputs, determinism,
independence of streams, and the distributions the workloads ask for."""
import numpy as np

import synth


def test_splitmix64_published_outputs():
    # SplitMix64 seeded with 0 (Vigna's splitmix64.c): first three outputs
    z = synth.u64(0, 3)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_chunked_equals_unchunked():
    n = (1 << 20) * 2 + 12345
    a = synth.u64(99, n)
    b = synth.u64(99, 1000)
    assert np.array_equal(a[:1000], b)
    # element i is the stream's output i, independent of how it was chunked
    i = (1 << 20) + 7
    assert a[i] == synth.u64(99, i + 1)[i]


def test_keys_independent_and_deterministic():
    wl = synth.WORKLOADS["tiny"]
    assert np.array_equal(synth.expert_slab(wl, 3), synth.expert_slab(wl, 3))
    assert not np.array_equal(synth.expert_slab(wl, 3), synth.expert_slab(wl, 4))
    assert not np.array_equal(synth.expert_slab(wl, 3, layer=1), synth.expert_slab(wl, 3))
    assert not np.array_equal(synth.tokens(wl, stream=0), synth.tokens(wl, stream=1))


def test_distributions():
    key = synth.derive_key(1, 0, 0, 0)
    n = synth.normal(key, 200_000, 0.0, 0.5).astype(np.float64)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 0.5) < 0.01
    u = synth.uniform(key, 200_000, 0.005, 0.02)
    assert u.min() >= 0.005 and u.max() <= 0.02 and abs(u.mean() - 0.0125) < 1e-4
    b = synth.random_bytes(key, 1 << 16)
    lo, hi = b & 15, b >> 4
    for nib in (lo, hi):
        counts = np.bincount(nib, minlength=16)
        assert counts.min() > 0.8 * (1 << 12) and counts.max() < 1.2 * (1 << 12)


def test_workload_shapes():
    W = synth.WORKLOADS
    g = W["glm_decode"]
    assert (g.T, g.H, g.E, g.K, g.I, g.n_shared, g.I_shared, g.routed_scale, g.seed) == \
        (1, 6144, 256, 8, 2048, 1, 2048, 2.5, 2)
    assert W["glm_batched"].T == 512 and W["glm_batched"].bias_dist == ("normal", 0.0, 0.5)
    assert W["stack35b"].n_layers == 40 and W["stack35b"].prenorm_residual
    assert W["olmoe"].n_shared == 0
    li = synth.layer_inputs(W["tiny"])
    assert li.slabs.shape == (16, W["tiny"].slab_bytes) and li.scales.dtype == np.float32
    assert li.router_w.shape == (16, 256) and abs(float(li.router_w.std()) - 0.02) < 0.002
