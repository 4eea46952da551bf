"""The seeded input generators: determinism and the configured distributions."""
import numpy as np

import synth


def _keys(s, V):
    k = np.zeros(s.shape[0], np.int64)
    for j in range(s.shape[1]):
        k = k * V + s[:, j]
    return k


def test_deterministic_and_seeded():
    cfg = synth.CONFIGS["tiny"]
    a = synth.make_catalogue(cfg, 0)
    b = synth.make_catalogue(cfg, 0)
    c = synth.make_catalogue(cfg, 1)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    m1 = synth.make_model(3, 16, 8, "bf16", 0)
    m2 = synth.make_model(3, 16, 8, "bf16", 0)
    assert all(np.array_equal(x, y) for x, y in zip(m1.W, m2.W))


def test_tiny_uniform_distinct():
    cfg = synth.CONFIGS["tiny"]
    s = synth.make_catalogue(cfg)
    assert s.shape == (20_000, 3) and s.dtype == np.int32
    assert s.min() >= 0 and s.max() < 256
    assert np.unique(_keys(s, 256)).size == 20_000


def test_mid_sparse_shape():
    cfg = synth.CONFIGS["mid_sparse"]
    s = synth.make_catalogue(cfg)
    V = cfg.V
    k = np.unique(_keys(s, V))
    assert k.size == 1_000_000
    t1, n1 = np.unique(s[:, 0], return_counts=True)
    assert t1.size == V                                  # every step-1 token is legal
    assert 150_000 < n1.max() < 190_000                  # Zipf(1.1) head ~ 169k items
    p2 = np.unique(k // V)
    fan2 = np.unique(p2 // V, return_counts=True)[1]
    # round(n/8) children clamped to V: the Zipf head saturates the codebook,
    # which pulls the mean from ~61 down to ~43 and pushes the head's
    # children to ~83 leaves each
    assert 35 < fan2.mean() < 70 and fan2.max() == V
    fan3 = k.size / p2.size
    assert 7 < fan3 < 13


def test_distinct_per_group_uniform():
    rng = synth.rng_for(0, "level", 0)
    counts = np.full(20000, 3)
    out = synth.distinct_per_group(rng, counts, 10).reshape(-1, 3)
    assert (np.diff(out, axis=1) > 0).all()
    # each of the C(10,3) = 120 subsets appears about equally often
    codes = out[:, 0] * 100 + out[:, 1] * 10 + out[:, 2]
    _, c = np.unique(codes, return_counts=True)
    assert c.size == 120 and c.min() > 100 and c.max() < 240


def test_model_moments():
    d = 256
    m = synth.make_model(2, 4096, d, "f32", 0)
    assert abs(m.C[0].var() - 1 / d) < 0.02 / d
    assert abs(m.W[0].var() - d ** -0.5) < 0.02 * d ** -0.5
    u = synth.make_requests(4096, d)
    assert abs(u.var() - 1 / d) < 0.02 / d


def test_half_storage():
    m = synth.make_model(1, 64, 32, "bf16", 0)
    assert m.W[0].dtype == np.uint16
    w32 = synth.bf16_bits_to_f32(m.W[0])
    assert np.array_equal(synth.f32_to_bf16_bits(w32), m.W[0])
    m16 = synth.make_model(1, 64, 32, "f16", 0)
    assert m16.W[0].dtype == np.float16
