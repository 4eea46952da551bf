"""Pins of the oracle's light causal decoder (the per-step hidden-state
producer of "Separating Thinking from Spelling", AI Papers Daily digest: a
fixed-size concept from the backbone, a 2-layer 256-wide causal decoder over
the concept and the generated prefix running the trie-constrained beam
search).  CPU only.

Each part is pinned to something other than the oracle: the normalisation and
the causal attention to PyTorch's own CPU routines, the whole decoder to closed
forms of special cases (residual branches switched off; attention made
uniform), to causality, and the beam search over it to exhaustive enumeration.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.zerogr_oracle as Z
import synth
from _helpers import tiny_catalogue

torch = pytest.importorskip("torch")


def rms_matches_torch() -> bool:
    x = np.random.default_rng(1).normal(0, 2, (7, 48))
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (48,), eps=Z.RMS_EPS).numpy()
    return np.allclose(Z.rms_norm(x), want, rtol=1e-12, atol=1e-12)


def attention_matches_torch() -> bool:
    rng = np.random.default_rng(2)
    n, d, heads = 6, 32, 4
    Q, K, V = (rng.normal(0, 1.5, (n, d)) for _ in range(3))
    split = lambda X: torch.from_numpy(X).reshape(n, heads, d // heads).transpose(0, 1)
    want = torch.nn.functional.scaled_dot_product_attention(split(Q), split(K), split(V), is_causal=True)
    want = want.transpose(0, 1).reshape(n, d).numpy()
    return np.allclose(Z.causal_attention(Q, K, V, heads), want, rtol=1e-10, atol=1e-12)


def zero_residual_closed_form() -> bool:
    """Attention and MLP outputs weighted by zero: every layer is the identity,
    so the hidden vector is the normalised last input row (concept M-1 plus its
    position embedding with no prefix; the last token's embedding plus its
    position embedding otherwise)."""
    w = synth.make_deco(3, 12, 16, M=2, heads=2, ffn=32, seed=3, zero_residual=True)
    c = synth.make_concepts(1, 2, 16, 3)[0]
    ok = np.allclose(oracle.deco_hidden(w, c, ()),
                     oracle.rms_norm((c[1].astype(np.float64) + w.P[1])[None])[0], atol=1e-12)
    for pre in [(5,), (5, 7)]:
        j = len(pre) - 1
        last = w.E[j][pre[-1]].astype(np.float64) + w.P[2 + j]
        ok = ok and np.allclose(oracle.deco_hidden(w, c, pre), oracle.rms_norm(last[None])[0], atol=1e-12)
    return ok


def uniform_attention_is_running_mean() -> bool:
    """All scores equal (zero queries): row i averages the values of rows 0..i."""
    V = np.random.default_rng(4).normal(0, 1, (5, 8))
    got = Z.causal_attention(np.zeros((5, 8)), np.random.default_rng(5).normal(0, 1, (5, 8)), V, 2)
    want = np.cumsum(V, axis=0) / np.arange(1, 6)[:, None]
    return np.allclose(got, want, atol=1e-12)


def causal() -> bool:
    """A position's output does not depend on later positions."""
    w = synth.make_deco(4, 10, 16, M=2, heads=4, ffn=32, seed=6)
    c = synth.make_concepts(1, 2, 16, 6)[0]
    a = oracle.deco_forward(w, c, (1, 2, 3))
    b = oracle.deco_forward(w, c, (1, 9, 0))
    return np.allclose(a[:3], b[:3], atol=1e-12) and not np.allclose(a[3:], b[3:])


def test_rms_norm_matches_torch():
    assert rms_matches_torch()


def test_causal_attention_matches_torch_sdpa():
    assert attention_matches_torch()


def test_zero_residual_closed_form():
    assert zero_residual_closed_form()


def test_uniform_attention_is_running_mean():
    assert uniform_attention_is_running_mean()


def test_causality():
    assert causal()


@pytest.mark.parametrize("seed,L,V,n", [(0, 3, 6, 40), (1, 2, 9, 30), (2, 3, 5, 60)])
def test_deco_beam_search_equals_exhaustive(seed, L, V, n):
    """With beam >= catalogue size, the beam search over the decoder's hidden
    vectors returns every item with its exact filter-first score, which form
    a probability distribution over the catalogue."""
    sids = tiny_catalogue(L, V, n, seed)
    trie = oracle.Trie(sids, L, V)
    m = synth.make_model(L, V, 16, "f32", seed)
    w = synth.make_deco(L, V, 16, M=2, heads=2, ffn=32, seed=seed)
    c = synth.make_concepts(2, 2, 16, seed)
    res = oracle.decode(trie, m, c, beam=n, K=n, deco=w)
    for q in range(2):
        bs, bsc = oracle.brute_force(trie, m, c[q], deco=w)
        assert np.array_equal(res.sids[q], bs)
        assert np.max(np.abs(res.scores[q] - bsc)) < 1e-9
        assert abs(np.exp(res.scores[q]).sum() - 1.0) < 1e-9
        for i in range(0, n, 7):
            assert abs(oracle.path_score(trie, m, c[q], bs[i], deco=w) - bsc[i]) < 1e-9


def test_decoder_changes_the_hidden_vectors():
    """The decoder is a different model than the token tables: decodes differ."""
    sids = tiny_catalogue(3, 8, 60, 4)
    trie = oracle.Trie(sids, 3, 8)
    m = synth.make_model(3, 8, 16, "f32", 4)
    w = synth.make_deco(3, 8, 16, M=2, heads=2, ffn=32, seed=4)
    c = synth.make_concepts(1, 2, 16, 4)
    a = oracle.decode(trie, m, c, beam=4, K=4, deco=w)
    b = oracle.decode(trie, m, synth.make_requests(1, 16, 4), beam=4, K=4)
    assert not np.allclose(a.scores, b.scores)
