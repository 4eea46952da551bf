"""Pins of the CPU oracle to facts other than itself.

Each test checks the oracle against something the pages state (golden
fixtures with citations), a closed form, a library routine, an invariant, or
brute force on tiny inputs.  No GPU is needed.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
import oracle.zerogr_oracle as Z
import synth
from _helpers import golden_catalogue, tiny_catalogue
from conftest import read_golden


# ---------------------------------------------------------------- worked example

def test_worked_example_trie():
    fx = read_golden("worked_example.txt")
    L, V, sids = golden_catalogue(fx)
    trie = oracle.Trie(sids, L, V)
    prefix = tuple(fx["prefix"][0])
    assert list(trie.children(prefix)) == sorted(fx["legal"][0])


@pytest.mark.parametrize("fmt", [-1, oracle.SPARSE, oracle.DENSE])
def test_worked_example_index_walk(fmt):
    """Walk the step tables with the implicit-successor rule (entry position =
    next-step row) along 3 then 5; the row reached lists exactly {1, 4}."""
    fx = read_golden("worked_example.txt")
    L, V, sids = golden_catalogue(fx)
    tabs = oracle.serialize_index(sids, L, V, force_format=fmt)
    row = 0
    for s, t in enumerate(fx["prefix"][0]):
        toks = oracle.table_row_tokens(tabs[s], row, V)
        j = int(np.nonzero(toks == t)[0][0])
        row = int(tabs[s].rowptr[row]) + j
    assert list(oracle.table_row_tokens(tabs[2], row, V)) == sorted(fx["legal"][0])


# ---------------------------------------------------------------- index invariants

def _prefix_sets(sids, L):
    return [sorted({tuple(int(x) for x in r[:s]) for r in sids}) for s in range(L + 1)]


@pytest.mark.parametrize("seed,L,V,n", [(0, 3, 8, 60), (1, 2, 40, 300), (2, 4, 5, 200),
                                         (3, 1, 33, 20), (4, 3, 64, 500)])
@pytest.mark.parametrize("fmt", [-1, oracle.SPARSE, oracle.DENSE])
def test_index_brute_force_recount(seed, L, V, n, fmt):
    """Rows are the distinct (s-1)-prefixes in lexicographic order, each row's
    tokens are the distinct extensions; recounted with Python sets."""
    sids = tiny_catalogue(L, V, n, seed)
    dup = np.concatenate([sids, sids[: n // 3]])        # duplicates are merged
    tabs = oracle.serialize_index(dup, L, V, force_format=fmt)
    pre = _prefix_sets(sids, L)
    for s in range(1, L + 1):
        tab = tabs[s - 1]
        rows = pre[s - 1]
        assert tab.rows == len(rows)
        assert tab.nnz == len(pre[s])
        for r, p in enumerate(rows):
            want = sorted({q[s - 1] for q in pre[s] if q[:s - 1] == p})
            assert list(oracle.table_row_tokens(tab, r, V)) == want
        F = np.diff(tab.rowptr.astype(np.int64))
        assert F.sum() == tab.nnz and tab.rowptr[0] == 0
        assert tab.max_fanout == F.max()
        if s < L:
            assert tab.nnz == tabs[s].rows          # entries of s = rows of s+1
        else:
            assert tab.nnz == len(pre[L])           # one entry per distinct item
    # implicit successor: entry e of step s extends to the prefix of row e at s+1
    for s in range(1, L):
        for r, p in enumerate(pre[s - 1]):
            toks = oracle.table_row_tokens(tabs[s - 1], r, V)
            for j, t in enumerate(toks):
                e = int(tabs[s - 1].rowptr[r]) + j
                assert pre[s][e] == p + (int(t),)


TRIE_CASES = [(0, 3, 8, 60), (1, 2, 40, 300), (2, 4, 5, 200), (3, 1, 33, 20), (4, 3, 64, 500)]


def trie_children_match_recount(cases=TRIE_CASES) -> bool:
    """Trie.children at every prefix of every length (and at absent prefixes)
    equals the distinct next tokens recounted with Python sets over the raw
    SID rows; Trie.contains is true exactly for catalogue items."""
    for seed, L, V, n in cases:
        sids = tiny_catalogue(L, V, n, seed)
        trie = oracle.Trie(sids, L, V)
        items = {tuple(int(x) for x in r) for r in sids}
        for s in range(L):
            nxt = {}
            for it in items:
                nxt.setdefault(it[:s], set()).add(it[s])
            for p, toks in nxt.items():
                if list(trie.children(p)) != sorted(toks):
                    return False
            rng = np.random.default_rng(seed + 10 * s)
            for _ in range(20):          # prefixes that no item starts with
                p = tuple(int(x) for x in rng.integers(0, V, size=s))
                if p not in nxt and trie.children(p).size != 0:
                    return False
        for it in list(items)[:50]:
            if not trie.contains(it):
                return False
        rng = np.random.default_rng(seed)
        for _ in range(50):
            it = tuple(int(x) for x in rng.integers(0, V, size=L))
            if trie.contains(it) != (it in items):
                return False
    return True


def test_distinct_sorted_is_the_sorted_set():
    rng = np.random.default_rng(5)
    for n, hi in [(0, 3), (1, 3), (50, 4), (1000, 50), (5000, 1 << 40)]:
        x = rng.integers(0, hi, size=n)
        assert list(Z.distinct_sorted(x)) == sorted(set(int(v) for v in x))


def test_trie_from_keys_equals_trie():
    sids = tiny_catalogue(3, 16, 300, 7)
    a = oracle.Trie(sids, 3, 16)
    b = Z.Trie.from_keys(a.keys, 3, 16)
    for p in [(), (int(sids[0, 0]),), tuple(int(x) for x in sids[1, :2])]:
        assert list(a.children(p)) == list(b.children(p))
    assert b.contains(sids[3]) and b.n_unique == a.n_unique


def test_trie_children_brute_force_recount():
    """[Problem]: a token is legal after a prefix iff prefix + token starts a
    catalogue SID - checked at every prefix of every length, not only at the
    worked example's."""
    assert trie_children_match_recount()


def test_format_rule_closed_form():
    """Dense iff 4*rows*ceil(V/32) < 2*nnz, evaluated by hand."""
    assert oracle.choose_format(1, 256, 256) == oracle.DENSE      # 32 < 512
    assert oracle.choose_format(256, 4096, 256) == oracle.SPARSE  # 8192 >= 8192
    assert oracle.choose_format(256, 4097, 256) == oracle.DENSE   # 8192 < 8194
    assert oracle.choose_format(10, 5, 33) == oracle.SPARSE       # 80 >= 10
    assert oracle.choose_format(1, 1, 32) == oracle.SPARSE        # 4 >= 2


def test_format_choice_tiny_config():
    """Tiny config (20,000 uniform SIDs over 256^3): steps 1-2 dense, 3 sparse."""
    cfg = synth.CONFIGS["tiny"]
    tabs = oracle.serialize_index(synth.make_catalogue(cfg), cfg.L, cfg.V)
    assert [t.fmt for t in tabs] == [oracle.DENSE, oracle.DENSE, oracle.SPARSE]
    assert tabs[0].rows == 1 and tabs[0].nnz == 256


def test_export_layout():
    fx = read_golden("worked_example.txt")
    L, V, sids = golden_catalogue(fx)
    tabs = oracle.serialize_index(sids, L, V, force_format=oracle.SPARSE)
    b = tabs[2].export_bytes()
    head = np.frombuffer(b[:16], "<u4")
    assert list(head) == [oracle.SPARSE, tabs[2].rows, tabs[2].nnz, 1]
    assert len(b) == 16 + 4 * (tabs[2].rows + 1) + 4 * ((2 * tabs[2].nnz + 3) // 4)


# ---------------------------------------------------------------- slot figure

def test_slot_figure():
    fx = read_golden("slot_figure.txt")
    f = fx["fanouts"][0]
    comp = oracle.compact_layout(f)
    assert sum(f) == fx["compact_length"][0][0]
    assert comp[1] + 1 == fx["compact_first_of_B_1based"][0][0]
    S, tab = oracle.padded_slot_layout(f)
    assert S == fx["slots_per_beam"][0][0]
    assert tab.size == fx["total_slots"][0][0]
    assert tab[1, 0] == 0 and fx["first_of_B_slot_1based"][0][0] == 1
    assert int((tab[0] < 0).sum()) == fx["A_empty_slots"][0][0]
    # B's slot does not depend on A's count (unlike the compact list)
    S2, tab2 = oracle.padded_slot_layout([2, 3])
    assert tab2[1, 0] == tab[1, 0] and oracle.compact_layout([2, 3])[1] != comp[1]


# ---------------------------------------------------------------- filtered softmax

@pytest.mark.parametrize("n", [1, 2, 7, 300, 5000])
def test_filtered_log_softmax_normalised(n):
    z = np.random.default_rng(n).normal(0, 3, n)
    lp = oracle.filtered_log_softmax(z)
    assert abs(np.exp(lp).sum() - 1.0) < 1e-6


def test_fanout_one_is_zero():
    for z in [0.0, -12.5, 3e4, 1e-30]:
        assert oracle.filtered_log_softmax(np.array([z]))[0] == 0.0


def test_shift_invariance():
    z = np.random.default_rng(1).normal(0, 1, 50)
    a = oracle.filtered_log_softmax(z)
    b = oracle.filtered_log_softmax(z + 123.25)
    assert np.max(np.abs(a - b)) < 1e-12


def test_matches_library_log_softmax():
    z = np.random.default_rng(2).normal(0, 2, 777)
    assert np.max(np.abs(oracle.filtered_log_softmax(z) - scipy.special.log_softmax(z))) < 1e-12


# ---------------------------------------------------------------- beam search

def _model(L, V, d, dtype="f32", seed=0):
    return synth.make_model(L, V, d, dtype, seed)


def test_full_product_catalogue_equals_unconstrained():
    """When every SID exists, the filter admits every token: the constrained
    decode equals the unconstrained one exactly."""
    L, V, d = 2, 6, 8
    sids = synth.product_catalogue(L, V)
    m = _model(L, V, d)
    u = synth.make_requests(3, d, 5)
    trie = oracle.Trie(sids, L, V)
    a = oracle.decode(trie, m, u, beam=4, K=4)
    b = oracle.decode(None, m, u, beam=4, K=4)
    assert np.array_equal(a.sids, b.sids)
    assert np.array_equal(a.scores, b.scores)


@pytest.mark.parametrize("seed,L,V,n,dtype", [(0, 2, 5, 9, "f32"), (1, 3, 4, 20, "bf16"),
                                               (2, 3, 6, 30, "f16"), (3, 1, 7, 7, "f32"),
                                               (4, 3, 8, 40, "f32")])
def test_beam_search_equals_exhaustive(seed, L, V, n, dtype):
    """With beam >= number of items nothing is pruned: the decode returns every
    item with its summed filtered log-probabilities, best first."""
    sids = tiny_catalogue(L, V, n, seed)
    m = _model(L, V, 5, dtype, seed)
    u = synth.make_requests(2, 5, seed)
    trie = oracle.Trie(sids, L, V)
    res = oracle.decode(trie, m, u, beam=n, K=n)
    for q in range(2):
        bs, bsc = oracle.brute_force(trie, m, u[q])
        assert np.array_equal(res.sids[q], bs)
        assert np.max(np.abs(res.scores[q] - bsc)) < 1e-12
        # filter-first scores form a distribution over the catalogue
        assert abs(np.exp(bsc).sum() - 1.0) < 1e-6


def test_topk_below_beam_equals_exhaustive_prefix():
    sids = tiny_catalogue(3, 6, 50, 7)
    m = _model(3, 6, 4, "f32", 7)
    u = synth.make_requests(1, 4, 7)
    trie = oracle.Trie(sids, 3, 6)
    res = oracle.decode(trie, m, u, beam=50, K=3)
    bs, bsc = oracle.brute_force(trie, m, u[0])
    assert np.array_equal(res.sids[0], bs[:3])


def test_greedy_special_case():
    """beam = K = 1 is greedy: at each step take the argmax of W_s[T] . h."""
    cfg = synth.CONFIGS["tiny"]
    sids = synth.make_catalogue(cfg)
    m = _model(cfg.L, cfg.V, cfg.d)
    u = synth.make_requests(3, cfg.d, 1)
    trie = oracle.Trie(sids, cfg.L, cfg.V)
    res = oracle.decode(trie, m, u, beam=1, K=1)
    for q in range(3):
        h = u[q].astype(np.float64)
        p = ()
        for s in range(cfg.L):
            T = trie.children(p)
            z = m.W_as_f64(s)[T] @ h
            t = int(T[int(np.argmax(z))])
            p = p + (t,)
            if s < cfg.L - 1:
                h = h + m.C[s][t]
        assert tuple(res.sids[q, 0]) == p


def test_tiny_config_outputs_valid():
    cfg = synth.CONFIGS["tiny"]
    sids = synth.make_catalogue(cfg)
    m = _model(cfg.L, cfg.V, cfg.d)
    u = synth.make_requests(2, cfg.d)
    trie = oracle.Trie(sids, cfg.L, cfg.V)
    res = oracle.decode(trie, m, u, beam=cfg.beam, K=cfg.topk)
    for q in range(2):
        assert np.all(np.diff(res.scores[q]) <= 0)
        for i in range(cfg.topk):
            sid = res.sids[q, i]
            assert trie.contains(sid)
            assert abs(oracle.path_score(trie, m, u[q], sid) - res.scores[q, i]) < 1e-10


def test_dead_beams_and_padding():
    """Fewer candidates than the beam: surplus outputs are SID -1, score -inf."""
    sids = np.array([[0, 1], [2, 3]], dtype=np.int32)
    m = _model(2, 4, 4)
    u = synth.make_requests(1, 4)
    trie = oracle.Trie(sids, 2, 4)
    res = oracle.decode(trie, m, u, beam=8, K=8)
    assert (res.sids[0, :2] >= 0).all() and (res.sids[0, 2:] == -1).all()
    assert np.isneginf(res.scores[0, 2:]).all()
    assert res.n_cand[0].tolist() == [2, 2]
    # each first token has one child, so step 2 adds log(1) = 0 exactly
    assert abs(np.exp(res.scores[0, :2]).sum() - 1.0) < 1e-12


def test_tie_break_lower_slot_first():
    """Two tokens with identical weight rows score exactly alike; the lower
    token (lower slot) comes first, then the lower parent-beam rank."""
    L, V, d = 1, 6, 4
    m = _model(L, V, d)
    m.W[0][4] = m.W[0][1]
    sids = np.array([[1], [4], [5]], dtype=np.int32)
    u = synth.make_requests(1, d)
    res = oracle.decode(oracle.Trie(sids, L, V), m, u, beam=3, K=3)
    order = [int(t) for t in res.sids[0, :, 0]]
    assert res.scores[0, order.index(1)] == res.scores[0, order.index(4)]
    assert order.index(1) < order.index(4)


def test_unconstrained_single_step_is_log_softmax():
    """L = 1 unconstrained: scores are scipy's log_softmax over all V tokens."""
    V, d = 37, 6
    m = _model(1, V, d)
    u = synth.make_requests(2, d, 3)
    res = oracle.decode(None, m, u, beam=V, K=V)
    for q in range(2):
        ref = scipy.special.log_softmax(m.W_as_f64(0) @ u[q].astype(np.float64))
        assert np.max(np.abs(np.sort(res.scores[q]) - np.sort(ref))) < 1e-12
        assert list(res.sids[q, :, 0]) == list(np.lexsort((np.arange(V), -ref)))


def test_bf16_storage_roundtrip():
    x = np.array([1.0, 1.00390625, 1.005859375, -3.14159, 65504.0, 1e-30], np.float32)
    b = synth.f32_to_bf16_bits(x)
    y = synth.bf16_bits_to_f32(b)
    assert y[0] == 1.0 and y[1] == 1.0                  # tie rounds to even
    assert y[2] == np.float32(1.0078125)
    assert abs(y[3] - x[3]) <= abs(x[3]) * 2 ** -8


# ------------------------------------------------- score-first order (the conventional baseline)

@pytest.mark.parametrize("seed,L,V,n,dtype", [(0, 2, 5, 9, "f32"), (1, 3, 4, 20, "bf16"),
                                               (4, 3, 8, 40, "f32")])
def test_score_first_equals_exhaustive(seed, L, V, n, dtype):
    """Score-first with beam >= number of items: every item with the log of
    the product of its tokens' codebook-wide softmax probabilities (the
    brute-force walk), best first."""
    sids = tiny_catalogue(L, V, n, seed)
    m = _model(L, V, 5, dtype, seed)
    u = synth.make_requests(2, 5, seed)
    trie = oracle.Trie(sids, L, V)
    res = oracle.decode(trie, m, u, beam=n, K=n, order="score_first")
    for q in range(2):
        bs, bsc = oracle.brute_force(trie, m, u[q], order="score_first")
        assert np.array_equal(res.sids[q], bs)
        assert np.max(np.abs(res.scores[q] - bsc)) < 1e-12


def test_score_first_is_the_unconstrained_path_probability():
    """An item's score-first score is its path log-probability under the
    unconstrained model: the exhaustive unconstrained decode over all V^L
    sequences (a distribution: total mass 1) gives the same numbers, and the
    catalogue's score-first mass is the part of that distribution it covers,
    below 1 when some tokens are illegal."""
    L, V, n = 2, 5, 9
    sids = tiny_catalogue(L, V, n, 3)
    m = _model(L, V, 6, "f32", 3)
    u = synth.make_requests(2, 6, 3)
    trie = oracle.Trie(sids, L, V)
    unc = oracle.decode(None, m, u, beam=V ** L, K=V ** L)
    sf = oracle.decode(trie, m, u, beam=n, K=n, order="score_first")
    for q in range(2):
        assert abs(np.exp(unc.scores[q]).sum() - 1.0) < 1e-9
        full = {tuple(int(t) for t in s): float(v) for s, v in zip(unc.sids[q], unc.scores[q])}
        got = [full[tuple(int(t) for t in s)] for s in sf.sids[q]]
        assert np.max(np.abs(np.array(got) - sf.scores[q])) < 1e-12
        mass = np.exp(sf.scores[q]).sum()
        assert mass < 1.0 - 1e-3
        assert abs(mass - sum(math.exp(full[tuple(int(t) for t in s)]) for s in sids)) < 1e-12


def test_score_first_equals_filter_first_on_product_catalogue():
    """When every SID exists the legal set is the codebook: both orders
    normalise over the same tokens and agree exactly."""
    L, V, d = 2, 6, 8
    sids = synth.product_catalogue(L, V)
    m = _model(L, V, d)
    u = synth.make_requests(3, d, 5)
    trie = oracle.Trie(sids, L, V)
    a = oracle.decode(trie, m, u, beam=4, K=4)
    b = oracle.decode(trie, m, u, beam=4, K=4, order="score_first")
    assert np.array_equal(a.sids, b.sids)
    assert np.max(np.abs(a.scores - b.scores)) < 1e-12


def test_score_first_single_step_closed_form():
    """One step: score-first = filter-first + log(softmax mass of the legal
    tokens) with both log-sum-exps from scipy; the order is the same."""
    V, d = 40, 16
    m = _model(1, V, d, "f32", 9)
    u = synth.make_requests(1, d, 9)
    legal = np.array([2, 5, 11, 17, 23, 31, 38])
    sids = legal[:, None].astype(np.int32)
    trie = oracle.Trie(sids, 1, V)
    a = oracle.decode(trie, m, u, beam=7, K=7)
    b = oracle.decode(trie, m, u, beam=7, K=7, order="score_first")
    z = m.W_as_f64(0) @ u[0].astype(np.float64)
    shift = scipy.special.logsumexp(z[legal]) - scipy.special.logsumexp(z)
    assert shift < 0
    assert np.array_equal(a.sids, b.sids)
    assert np.max(np.abs(b.scores - (a.scores + shift))) < 1e-12


@pytest.mark.parametrize("order", ["filter_first", "score_first"])
def test_path_score_matches_exhaustive_walk(order):
    """The per-item path score (hidden vector rebuilt from scratch for every
    prefix) equals the brute-force walk's product of per-step softmax
    probabilities for every item of a tiny catalogue, in both orders."""
    sids = tiny_catalogue(3, 6, 40, 12)
    m = _model(3, 6, 5, "bf16", 12)
    u = synth.make_requests(1, 5, 12)
    trie = oracle.Trie(sids, 3, 6)
    bs, bsc = oracle.brute_force(trie, m, u[0], order=order)
    for sid, sc in zip(bs, bsc):
        assert abs(oracle.path_score(trie, m, u[0], sid, order) - sc) < 1e-12
    # an item outside the catalogue has no path
    missing = next(t for t in ((a, b, c) for a in range(6) for b in range(6) for c in range(6))
                   if not trie.contains(t))
    assert oracle.path_score(trie, m, u[0], missing, order) == -math.inf
