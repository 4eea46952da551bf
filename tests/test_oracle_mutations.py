"""Planted mistakes in the oracle (CPU only): each plausible error must make at
least one pin fail, which shows the pins constrain the oracle and do not just
restate it."""
import numpy as np
import pytest

import oracle
import oracle.zerogr_oracle as Z
import synth
from _helpers import tiny_catalogue


def _exhaustive_pin_holds():
    """The brute-force pin of test_oracle_pins, as a predicate."""
    for seed, L, V, n, dtype in [(1, 3, 4, 20, "bf16"), (4, 3, 8, 40, "f32")]:
        sids = tiny_catalogue(L, V, n, seed)
        m = synth.make_model(L, V, 5, dtype, seed)
        u = synth.make_requests(2, 5, seed)
        trie = Z.Trie(sids, L, V)
        res = Z.decode(trie, m, u, beam=n, K=n)
        for q in range(2):
            bs, bsc = Z.brute_force(trie, m, u[q])
            if not np.array_equal(res.sids[q], bs) or np.max(np.abs(res.scores[q] - bsc)) > 1e-9:
                return False
            if abs(np.exp(res.scores[q]).sum() - 1.0) > 1e-6:
                return False
    return True


def _membership_pin_holds():
    cfg = synth.CONFIGS["tiny"]
    sids = synth.make_catalogue(cfg)
    m = synth.make_model(cfg.L, cfg.V, cfg.d)
    u = synth.make_requests(1, cfg.d)
    trie = Z.Trie(sids, cfg.L, cfg.V)
    res = Z.decode(trie, m, u, beam=cfg.beam, K=cfg.topk)
    return all(trie.contains(res.sids[0, i]) for i in range(cfg.topk))


def _tie_pin_holds():
    m = synth.make_model(1, 6, 4)
    m.W[0][4] = m.W[0][1]
    sids = np.array([[1], [4], [5]], dtype=np.int32)
    res = Z.decode(Z.Trie(sids, 1, 6), m, synth.make_requests(1, 4), beam=3, K=3)
    order = [int(t) for t in res.sids[0, :, 0]]
    return order.index(1) < order.index(4)


def _normalised_pin_holds():
    z = np.random.default_rng(3).normal(0, 3, 300)
    return abs(np.exp(Z.filtered_log_softmax(z)).sum() - 1.0) < 1e-6


def test_pins_hold_on_the_real_oracle():
    assert _exhaustive_pin_holds()
    assert _membership_pin_holds()
    assert _tie_pin_holds()
    assert _normalised_pin_holds()


def test_mistake_softmax_without_normaliser(monkeypatch):
    monkeypatch.setattr(Z, "filtered_log_softmax", lambda z: np.asarray(z) - np.max(z))
    assert not _normalised_pin_holds()
    assert not _exhaustive_pin_holds()


def test_mistake_softmax_over_full_codebook(monkeypatch):
    """Normalising over all V tokens (score-first order) instead of the legal set."""
    real = Z.decode

    def score_first(trie, model, u, beam, K, requests=None):
        orig = Z.step_logits
        full = {}

        def logits(Wd, s, T, h):
            full["z"] = Wd[s - 1] @ h
            return Wd[s - 1][T] @ h

        def lsm(z):
            zf = full["z"]
            m = zf.max()
            return np.asarray(z) - (m + np.log(np.exp(zf - m).sum()))

        monkeypatch.setattr(Z, "step_logits", logits)
        monkeypatch.setattr(Z, "filtered_log_softmax", lsm)
        try:
            return real(trie, model, u, beam, K, requests)
        finally:
            monkeypatch.setattr(Z, "step_logits", orig)

    monkeypatch.setattr(Z, "decode", score_first)
    assert not _exhaustive_pin_holds()


def test_mistake_wrong_weight_step(monkeypatch):
    monkeypatch.setattr(Z, "step_logits", lambda Wd, s, T, h: Wd[s % len(Wd)][T] @ h)
    assert not _exhaustive_pin_holds()


def test_mistake_sign_flip(monkeypatch):
    monkeypatch.setattr(Z, "step_logits", lambda Wd, s, T, h: -(Wd[s - 1][T] @ h))
    assert not _exhaustive_pin_holds()


def test_mistake_hidden_not_advanced(monkeypatch):
    monkeypatch.setattr(Z, "advance_hidden", lambda h, Cd, s, t: h)
    assert not _exhaustive_pin_holds()


def test_mistake_hidden_wrong_table(monkeypatch):
    monkeypatch.setattr(Z, "advance_hidden", lambda h, Cd, s, t: h + Cd[-s][t])
    assert not _exhaustive_pin_holds()


def test_mistake_tie_break_reversed(monkeypatch):
    monkeypatch.setattr(Z, "candidate_order", lambda vals, flat: np.lexsort((-flat, -vals)))
    assert not _tie_pin_holds()


def test_mistake_no_filter(monkeypatch):
    monkeypatch.setattr(Z.Trie, "children", lambda self, p: np.arange(self.V))
    assert not _membership_pin_holds()


def test_mistake_successor_off_by_one(monkeypatch):
    """A serializer whose rowptr is shifted by one entry breaks the index walk."""
    real = Z.serialize_index

    def shifted(sids, L, V, force_format=-1):
        tabs = real(sids, L, V, force_format)
        for t in tabs:
            t.rowptr = np.concatenate([[0], t.rowptr[:-1] + 1]).astype(np.uint32)
        return tabs

    monkeypatch.setattr(Z, "serialize_index", shifted)
    from conftest import read_golden
    from _helpers import golden_catalogue
    L, V, sids = golden_catalogue(read_golden("worked_example.txt"))
    tabs = Z.serialize_index(sids, L, V)
    with pytest.raises(Exception):
        row = 0
        for s, t in enumerate([3, 5]):
            toks = Z.table_row_tokens(tabs[s], row, V)
            j = int(np.nonzero(toks == t)[0][0])
            row = int(tabs[s].rowptr[row]) + j
        assert list(Z.table_row_tokens(tabs[2], row, V)) == [1, 4]


def _score_first_pin_holds():
    sids = tiny_catalogue(3, 4, 20, 1)
    m = synth.make_model(3, 4, 5, "bf16", 1)
    u = synth.make_requests(2, 5, 1)
    trie = Z.Trie(sids, 3, 4)
    res = Z.decode(trie, m, u, beam=20, K=20, order="score_first")
    for q in range(2):
        bs, bsc = Z.brute_force(trie, m, u[q], order="score_first")
        if not np.array_equal(res.sids[q], bs) or np.max(np.abs(res.scores[q] - bsc)) > 1e-9:
            return False
    return True


def test_score_first_pin_holds_on_the_real_oracle():
    assert _score_first_pin_holds()


def test_mistake_score_first_normalised_over_legal(monkeypatch):
    """A score-first order that (wrongly) renormalises over the legal tokens."""
    monkeypatch.setattr(Z, "score_first_log_probs", lambda z_all, T: Z.filtered_log_softmax(np.asarray(z_all)[T]))
    assert not _score_first_pin_holds()


def test_mistake_score_first_without_max_shift_sign(monkeypatch):
    """A normaliser with the wrong sign (z + lse)."""
    def wrong(z_all, T):
        z = np.asarray(z_all, dtype=np.float64)
        return z[T] + (z.max() + np.log(np.exp(z - z.max()).sum()))
    monkeypatch.setattr(Z, "score_first_log_probs", wrong)
    assert not _score_first_pin_holds()


def _trie_pin_holds():
    from test_oracle_pins import trie_children_match_recount
    return trie_children_match_recount()


def test_trie_pin_holds_on_the_real_oracle():
    assert _trie_pin_holds()


@pytest.mark.parametrize("delta", [1, -1])
def test_mistake_trie_range_span_off_by_one_power(monkeypatch, delta):
    """A key range under a prefix whose span is V**(L-s+delta) instead of V**(L-s)."""
    def wrong_range(self, prefix):
        s = len(prefix)
        p = 0
        for t in prefix:
            p = p * self.V + int(t)
        span = self.V ** max(self.L - s + delta, 0)
        lo = int(np.searchsorted(self.keys, p * span, side="left"))
        hi = int(np.searchsorted(self.keys, (p + 1) * span, side="left"))
        return lo, hi
    monkeypatch.setattr(Z.Trie, "_range", wrong_range)
    assert not _trie_pin_holds()


def test_mistake_trie_children_wrong_digit(monkeypatch):
    """children() reading the token one step too deep (the digit after the next one)."""
    def wrong_children(self, prefix):
        prefix = tuple(int(t) for t in prefix)
        lo, hi = self._range(prefix)
        div = self.V ** max(self.L - len(prefix) - 2, 0)
        return np.unique((self.keys[lo:hi] // div) % self.V)
    monkeypatch.setattr(Z.Trie, "children", wrong_children)
    assert not _trie_pin_holds()


# ---------------------------------------------------------------- light decoder

def test_decoder_pins_hold_on_the_real_oracle():
    import test_oracle_deco as P
    assert P.rms_matches_torch() and P.attention_matches_torch() and P.zero_residual_closed_form()
    assert P.uniform_attention_is_running_mean() and P.causal()


def test_mistake_attention_without_causal_mask(monkeypatch):
    import test_oracle_deco as P

    def full(Q, K, V, heads):
        n, d = Q.shape
        dh = d // heads
        out = np.zeros((n, d))
        for h in range(heads):
            c = slice(h * dh, (h + 1) * dh)
            S = Q[:, c] @ K[:, c].T / np.sqrt(dh)
            Pm = np.exp(S - S.max(axis=1, keepdims=True))
            out[:, c] = (Pm / Pm.sum(axis=1, keepdims=True)) @ V[:, c]
        return out
    monkeypatch.setattr(Z, "causal_attention", full)
    assert not P.causal()
    assert not P.attention_matches_torch()


def test_mistake_attention_unscaled(monkeypatch):
    import test_oracle_deco as P
    real = Z.causal_attention
    monkeypatch.setattr(Z, "causal_attention", lambda Q, K, V, heads: real(Q * np.sqrt(Q.shape[1] // heads), K, V, heads))
    assert not P.attention_matches_torch()


def test_mistake_position_embedding_off_by_one(monkeypatch):
    import test_oracle_deco as P
    real = Z.deco_forward

    def shifted(w, concepts_q, prefix):
        import copy
        w2 = copy.copy(w)
        w2.P = np.roll(w.P, 1, axis=0)
        return real(w2, concepts_q, prefix)
    monkeypatch.setattr(Z, "deco_forward", shifted)
    assert not P.zero_residual_closed_form()


def test_mistake_norm_by_sum_of_squares(monkeypatch):
    import test_oracle_deco as P
    monkeypatch.setattr(Z, "rms_norm", lambda X: np.asarray(X, np.float64) / np.sqrt(
        np.sum(np.asarray(X, np.float64) ** 2, axis=-1, keepdims=True) + Z.RMS_EPS))
    assert not P.rms_matches_torch()
    assert not P.zero_residual_closed_form()
