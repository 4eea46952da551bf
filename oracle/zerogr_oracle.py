"""CPU oracle for filtering-first constrained beam decoding over semantic IDs.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA library: it reads the same seeded arrays (from ``synth``) and
nothing else.  Everything is float64 numpy, written for a reader to check by
eye against the method's description, not for speed.

Source: "ZeroGR: Filtering-First Constrained Decoding for Generative
Recommendation" (paper-daily.com digest), sections cited per function:
  [Problem]   "What problem does it solve" - SIDs, beam search, the validity
              filter and the worked example 3-5-1 / 3-5-4 -> {1, 4}.
  [Order]     "Does filtering first change the result" - softmax normalised
              over the legal tokens only (filter-first); the conventional
              order normalises over every token and masks afterwards
              (score-first, the comparison of that section).
  [Pipeline]  "Overall flow" - the four stages of one decoding step.
  [Index]     "Why slice the index by decoding step" - one table per step,
              rows are prefixes, an entry's position is its next-step row,
              dense tables for steps with many legal tokens, sparse otherwise.
  [Speed]     "Why computing fewer scores is not automatically faster" and its
              figure "compact list vs padded slots" (paper section 4 /
              Figure 9) - every beam of a step gets the same number of slots,
              empty slots score -inf, a candidate's slot depends only on
              (beam, rank).
Readings taken where the pages are silent (listed with reasons in the design
notes): the softmax set is the legal set; sparse slots and table columns are
in ascending token order; step-s rows are the distinct length-(s-1) prefixes in
lexicographic order; a step is stored dense iff its bitmap is smaller than its
CSR column array; ties order by lower parent-beam rank, then lower slot; one
root beam per request; beams beyond the number of candidates are dead and
outputs are padded with SID -1 and score -inf.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(worked example, slot figure, closed forms, brute force).  The quality claim
of the [Order] section (99.85-99.90 % overlap with score-first on a trained
MovieLens model) needs a dataset and a trained model: parity unpinned, not
tested.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

SPARSE = 0
DENSE = 1


# ---------------------------------------------------------------------------
# catalogue trie  [Problem], [Index]
# ---------------------------------------------------------------------------

def sid_keys(sids: np.ndarray, V: int) -> np.ndarray:
    """Base-V integer key of each SID; numeric order = lexicographic order.
    Requires V**L < 2**63."""
    sids = np.asarray(sids, dtype=np.int64)
    L = sids.shape[1]
    if V ** L >= 2 ** 63:
        raise ValueError("oracle keys need V**L < 2**63")
    k = np.zeros(sids.shape[0], dtype=np.int64)
    for s in range(L):
        k = k * V + sids[:, s]
    return k


def distinct_sorted(x: np.ndarray) -> np.ndarray:
    """The distinct values of x in ascending order: a library sort, then every
    value equal to its predecessor dropped (the definition of a set's sorted
    listing; np.unique computes the same but is far slower on 10^8 keys)."""
    x = np.sort(np.asarray(x).ravel())
    if x.size == 0:
        return x
    keep = np.empty(x.size, dtype=bool)
    keep[0] = True
    np.not_equal(x[1:], x[:-1], out=keep[1:])
    return x[keep]


def keys_to_sids(keys: np.ndarray, L: int, V: int) -> np.ndarray:
    out = np.empty((keys.size, L), dtype=np.int64)
    k = keys.copy()
    for s in range(L - 1, -1, -1):
        out[:, s] = k % V
        k //= V
    return out


class Trie:
    """The catalogue as a prefix tree, held implicitly as the sorted list of
    distinct SID keys: the SIDs under a prefix form one contiguous key range.

    [Problem]: a token is legal after a prefix iff prefix+token starts some
    catalogue SID."""

    def __init__(self, sids: np.ndarray, L: int, V: int):
        sids = np.asarray(sids)
        if sids.ndim != 2 or sids.shape[1] != L:
            raise ValueError("sids must be [n, L]")
        if sids.size and (sids.min() < 0 or sids.max() >= V):
            raise ValueError("token out of range")
        self.L, self.V = L, V
        raw = sid_keys(sids, V)
        self.keys = distinct_sorted(raw)
        self.n_input = int(raw.size)
        self.n_unique = int(self.keys.size)
        self._cache = {}

    @classmethod
    def from_keys(cls, keys: np.ndarray, L: int, V: int) -> "Trie":
        """A trie over keys that are already the distinct ascending base-V SID
        keys of a catalogue (another Trie's ``keys``, e.g. memory-mapped in a
        worker process), without sorting again."""
        t = cls.__new__(cls)
        t.L, t.V = L, V
        t.keys = keys
        t.n_input = t.n_unique = int(keys.size)
        t._cache = {}
        return t

    def _range(self, prefix) -> tuple[int, int]:
        s = len(prefix)
        p = 0
        for t in prefix:
            p = p * self.V + int(t)
        span = self.V ** (self.L - s)
        lo = int(np.searchsorted(self.keys, p * span, side="left"))
        hi = int(np.searchsorted(self.keys, (p + 1) * span, side="left"))
        return lo, hi

    def children(self, prefix) -> np.ndarray:
        """Legal next tokens after ``prefix`` (a tuple of tokens), ascending."""
        prefix = tuple(int(t) for t in prefix)
        got = self._cache.get(prefix)
        if got is None:
            lo, hi = self._range(prefix)
            s = len(prefix)
            div = self.V ** (self.L - s - 1)
            got = distinct_sorted((self.keys[lo:hi] // div) % self.V)
            self._cache[prefix] = got
        return got

    def contains(self, sid) -> bool:
        lo, hi = self._range(tuple(sid))
        return hi > lo and len(sid) == self.L


# ---------------------------------------------------------------------------
# step-sliced index, canonical serialisation  [Index]
# ---------------------------------------------------------------------------

@dataclass
class StepTable:
    fmt: int                 # SPARSE or DENSE
    rows: int                # distinct length-(s-1) prefixes
    nnz: int                 # distinct length-s prefixes (= rows of step s+1)
    words: int               # 32-bit words per dense bitmap row
    rowptr: np.ndarray       # uint32 [rows+1]; entry e of row r is next-step row e
    col: np.ndarray | None   # uint16 [nnz] legal tokens, ascending within a row
    bitmap: np.ndarray | None  # uint32 [rows, words]
    max_fanout: int

    def export_bytes(self) -> bytes:
        """Canonical byte layout: u32 header {fmt, rows, nnz, words}, u32
        rowptr[rows+1], then the payload: u16 col[nnz] zero-padded to a
        multiple of 4 bytes (sparse) or u32 bitmap[rows][words] (dense)."""
        head = np.array([self.fmt, self.rows, self.nnz, self.words], dtype="<u4").tobytes()
        rp = self.rowptr.astype("<u4").tobytes()
        if self.fmt == SPARSE:
            pay = self.col.astype("<u2").tobytes()
            pay += b"\0" * ((-len(pay)) % 4)
        else:
            pay = self.bitmap.astype("<u4").tobytes()
        return head + rp + pay


def choose_format(rows: int, nnz: int, V: int) -> int:
    """[Index] says only that steps with many legal tokens are stored dense.
    Reading: the smaller table wins (the pages' goal for the index is memory);
    dense iff the bitmap (4*ceil(V/32) bytes a row) is smaller than the CSR
    column array (2 bytes an entry)."""
    words = (V + 31) // 32
    return DENSE if 4 * rows * words < 2 * nnz else SPARSE


def serialize_index(sids: np.ndarray, L: int, V: int, force_format: int = -1) -> list[StepTable]:
    """Build the per-step tables of [Index] from the catalogue.

    Step s (1-based) has one row per distinct length-(s-1) prefix, in
    lexicographic order (step 1 has the single empty prefix).  A row lists
    the legal tokens that extend it, ascending.  Enumerating all (row, token)
    entries of step s in order, entry e extends to the prefix that is row e of
    step s+1, so no successor array is stored; rowptr[r] is the position of
    row r's first entry."""
    keys = distinct_sorted(sid_keys(sids, V))
    words = (V + 31) // 32
    tables = []
    for s in range(1, L + 1):
        ent = distinct_sorted(keys // (V ** (L - s)))  # distinct s-prefixes, sorted
        parent = ent // V                              # their (s-1)-prefixes
        rows_val = distinct_sorted(parent)
        rowidx = np.searchsorted(rows_val, parent)
        F = np.bincount(rowidx, minlength=rows_val.size).astype(np.int64)
        rowptr = np.zeros(rows_val.size + 1, dtype=np.int64)
        rowptr[1:] = np.cumsum(F)
        tok = ent % V
        fmt = choose_format(rows_val.size, ent.size, V) if force_format < 0 else int(force_format)
        col = bitmap = None
        if fmt == SPARSE:
            col = tok.astype(np.uint16)
        else:
            widx = rowidx * words + tok // 32
            bit = (np.int64(1) << (tok % 32)).astype(np.float64)
            bm = np.bincount(widx, weights=bit, minlength=rows_val.size * words)
            bitmap = bm.astype(np.uint64).astype(np.uint32).reshape(rows_val.size, words)
        tables.append(StepTable(fmt, int(rows_val.size), int(ent.size), words,
                                rowptr.astype(np.uint32), col, bitmap,
                                int(F.max()) if F.size else 0))
    return tables


def table_row_tokens(tab: StepTable, r: int, V: int) -> np.ndarray:
    """Legal tokens of row r read back from a serialised table."""
    if tab.fmt == SPARSE:
        return tab.col[tab.rowptr[r]:tab.rowptr[r + 1]].astype(np.int64)
    bits = tab.bitmap[r]
    toks = [w * 32 + b for w in range(tab.words) for b in range(32) if (int(bits[w]) >> b) & 1]
    return np.array([t for t in toks if t < V], dtype=np.int64)


# ---------------------------------------------------------------------------
# padded candidate slots  [Speed], figure "compact list vs padded slots"
# ---------------------------------------------------------------------------

def padded_slot_layout(fanouts) -> tuple[int, np.ndarray]:
    """Every beam of a step gets S = max fan-out slots; beam b's j-th legal
    candidate (ascending token order) sits in slot (b, j), flat index b*S+j;
    slots j >= F_b are empty and score -inf.  Returns (S, rank table [n, S]
    holding j or -1 for an empty slot)."""
    f = np.asarray(fanouts, dtype=np.int64)
    S = int(f.max()) if f.size else 0
    tab = np.full((f.size, S), -1, dtype=np.int64)
    for b, fb in enumerate(f):
        tab[b, :fb] = np.arange(fb)
    return S, tab


def compact_layout(fanouts) -> np.ndarray:
    """The naive layout the [Speed] section contrasts with: all beams'
    candidates packed into one list; beam b starts at the sum of the
    fan-outs before it (so it depends on the other beams)."""
    f = np.asarray(fanouts, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(f)[:-1]]) if f.size else f


# ---------------------------------------------------------------------------
# filtered log-softmax  [Order], [Pipeline] stage 4
# ---------------------------------------------------------------------------

def filtered_log_softmax(z_legal: np.ndarray) -> np.ndarray:
    """log-softmax over the legal tokens only: lp_t = z_t - lse,
    lse = m + log(sum_t exp(z_t - m)), m = max_t z_t."""
    z = np.asarray(z_legal, dtype=np.float64)
    m = z.max()
    lse = m + math.log(float(np.exp(z - m).sum()))
    return z - lse


def score_first_log_probs(z_all: np.ndarray, T: np.ndarray) -> np.ndarray:
    """[Order], [Problem]: the conventional order scores every token, takes
    the log-softmax over the whole codebook and only then masks: the legal
    tokens T keep lp_t = z_t - lse_V, lse_V = m + log(sum_v exp(z_v - m))
    over all V tokens, m = max_v z_v.  The probability mass of the illegal
    tokens is dropped, not redistributed."""
    z = np.asarray(z_all, dtype=np.float64)
    m = z.max()
    lse_all = m + math.log(float(np.exp(z - m).sum()))
    return z[np.asarray(T, dtype=np.int64)] - lse_all


ORDERS = ("filter_first", "score_first")


# ---------------------------------------------------------------------------
# light causal decoder producing each step's hidden vector ("Separating
# Thinking from Spelling", AI Papers Daily digest: a backbone emits a fixed-size
# next-item concept once; a light 2-layer, 256-wide causal decoder conditioned
# on the concept and the generated prefix runs the trie-constrained beam
# search).  Readings (the digest gives only the above): inputs are the M
# concept vectors then the embeddings of the chosen tokens, each plus a
# position embedding; pre-norm layers x += attention(norm(x)), x += MLP(norm(x));
# RMS normalisation without gain, causal multi-head attention scaled by
# 1/sqrt(head width), ReLU MLP; the hidden vector is the normalised output of
# the last position.
# ---------------------------------------------------------------------------

RMS_EPS = 1e-6


def rms_norm(X: np.ndarray) -> np.ndarray:
    """Each row divided by the root of its mean square (plus RMS_EPS)."""
    X = np.asarray(X, dtype=np.float64)
    return X / np.sqrt(np.mean(X * X, axis=-1, keepdims=True) + RMS_EPS)


def causal_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, heads: int) -> np.ndarray:
    """Per head h (a contiguous block of d/heads columns): row i attends to
    rows j <= i with weights softmax_j(q_i . k_j / sqrt(d/heads))."""
    n, d = Q.shape
    dh = d // heads
    out = np.zeros((n, d))
    mask = np.tril(np.ones((n, n), dtype=bool))
    for h in range(heads):
        c = slice(h * dh, (h + 1) * dh)
        S = Q[:, c] @ K[:, c].T / math.sqrt(dh)
        S = np.where(mask, S, -np.inf)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        out[:, c] = P @ V[:, c]
    return out


def deco_forward(w, concepts_q: np.ndarray, prefix) -> np.ndarray:
    """Output rows of every position of the sequence [concepts, tokens of the
    prefix] after all layers (before the final normalisation)."""
    rows = [np.asarray(concepts_q[m], np.float64) + w.P[m] for m in range(w.M)]
    rows += [np.asarray(w.E[j][int(t)], np.float64) + w.P[w.M + j] for j, t in enumerate(prefix)]
    X = np.array(rows)
    for l in range(w.layers):
        A = rms_norm(X)
        Q = A @ np.asarray(w.Wq[l], np.float64).T
        K = A @ np.asarray(w.Wk[l], np.float64).T
        Vv = A @ np.asarray(w.Wv[l], np.float64).T
        X = X + causal_attention(Q, K, Vv, w.heads) @ np.asarray(w.Wo[l], np.float64).T
        H = np.maximum(rms_norm(X) @ np.asarray(w.W1[l], np.float64).T, 0.0)
        X = X + H @ np.asarray(w.W2[l], np.float64).T
    return X


def deco_hidden(w, concepts_q: np.ndarray, prefix) -> np.ndarray:
    """Hidden vector of a beam with the given prefix: the normalised output of
    the sequence's last position."""
    return rms_norm(deco_forward(w, concepts_q, prefix)[-1])


# ---------------------------------------------------------------------------
# beam search  [Pipeline]
# ---------------------------------------------------------------------------

@dataclass
class DecodeResult:
    sids: np.ndarray        # int64 [B, K, L], -1 for missing outputs
    scores: np.ndarray      # float64 [B, K], -inf for missing outputs
    gaps: np.ndarray        # float64 [B, L]: kept-vs-first-dropped score gap per step (inf if none dropped)
    n_cand: np.ndarray      # int64 [B, L]: candidates per step
    next_score: np.ndarray  # float64 [B]: best final candidate that was not returned (-inf if none)


def _weights_f64(model):
    return [model.W_as_f64(s) for s in range(model.L)]


def step_logits(Wd, s: int, T: np.ndarray, h: np.ndarray) -> np.ndarray:
    """[Speed]: score only the legal tokens, z_t = W_s[t] . h (s is 1-based)."""
    return Wd[s - 1][T] @ h


def advance_hidden(h: np.ndarray, Cd, s: int, t: int) -> np.ndarray:
    """Synthetic model: after choosing token t at step s, h += C_s[t]."""
    return h + Cd[s - 1][t]


def candidate_order(vals: np.ndarray, flat: np.ndarray) -> np.ndarray:
    """Best first: higher score, then lower flat slot index (parent-beam rank
    major, ascending token within a beam)."""
    return np.lexsort((flat, -vals))


def decode(trie: Trie | None, model, u: np.ndarray, beam: int, K: int,
           requests=None, order: str = "filter_first", deco=None) -> DecodeResult:
    """Filtering-first constrained beam search, one request at a time.

    Per request: one root beam (empty prefix, cumulative score 0, hidden u).
    Step s = 1..L, for every live beam b [Pipeline]:
      T_b  = legal next tokens of b's prefix (all V tokens if trie is None,
             the unconstrained decode of the [Results] section);
      z_t  = W_s[t] . h_b for t in T_b (only legal rows are touched);
      lp_t = z_t - lse over T_b                       [Order];
      cand = cum_b + lp_t.
    Keep the best `beam` candidates (the best K at the last step), ordered by
    score, then lower parent-beam rank, then lower slot (ascending token).
    A survivor's hidden vector is h_b + C_s[t] (the synthetic model's
    prefix state).  Output rows beyond the number of candidates are -1/-inf.
    order="score_first" replaces lp_t by the conventional order's
    score_first_log_probs (every token scored, normaliser over the codebook,
    then the mask); everything else is unchanged.
    deco: a light decoder's weights; then u holds each request's concept
    vectors [B, M, d] and a beam's hidden vector is deco_hidden of its prefix
    (the token tables C are not used).
    """
    if order not in ORDERS:
        raise ValueError(order)
    L, V = model.L, model.V
    u = np.asarray(u)
    B = u.shape[0]
    req = range(B) if requests is None else list(requests)
    Wd = _weights_f64(model)
    Cd = [np.asarray(c, dtype=np.float64) for c in model.C] if deco is None else None
    out_sids = np.full((B, K, L), -1, dtype=np.int64)
    out_scores = np.full((B, K), -np.inf)
    gaps = np.full((B, L), np.inf)
    n_cand = np.zeros((B, L), dtype=np.int64)
    next_score = np.full(B, -np.inf)
    all_tok = np.arange(V)
    for q in req:
        h0 = deco_hidden(deco, u[q], ()) if deco is not None else u[q].astype(np.float64)
        beams = [((), 0.0, h0)]
        for s in range(1, L + 1):
            keep = beam if s < L else K
            legal = [trie.children(p) if trie is not None else all_tok for p, _, _ in beams]
            S, slots = padded_slot_layout([t.size for t in legal])
            vals, flat, toks, ranks = [], [], [], []
            for rank, ((p, cum, h), T) in enumerate(zip(beams, legal)):
                if order == "score_first":
                    lp = score_first_log_probs(step_logits(Wd, s, all_tok, h), T)
                else:
                    lp = filtered_log_softmax(step_logits(Wd, s, T, h))
                vals.append(cum + lp)
                flat.append(rank * S + slots[rank, :T.size])
                toks.append(T)
                ranks.append(np.full(T.size, rank))
            vals = np.concatenate(vals)
            flat = np.concatenate(flat)
            toks = np.concatenate(toks)
            ranks = np.concatenate(ranks)
            best = candidate_order(vals, flat)
            n_cand[q, s - 1] = vals.size
            if vals.size > keep:
                gaps[q, s - 1] = vals[best[keep - 1]] - vals[best[keep]]
                if s == L:
                    next_score[q] = vals[best[keep]]
            chosen = best[:keep]
            new = []
            for i in chosen:
                p, cum, h = beams[ranks[i]]
                t = int(toks[i])
                if s == L:
                    h2 = None
                elif deco is not None:
                    h2 = deco_hidden(deco, u[q], p + (t,))
                else:
                    h2 = advance_hidden(h, Cd, s, t)
                new.append((p + (t,), float(vals[i]), h2))
            beams = new
        for i, (p, cum, _) in enumerate(beams):
            out_sids[q, i] = p
            out_scores[q, i] = cum
    return DecodeResult(out_sids, out_scores, gaps, n_cand, next_score)


def path_score(trie: Trie | None, model, u_q: np.ndarray, sid, order: str = "filter_first",
               Wd=None, deco=None) -> float:
    """Filter-first score of one item along its own path: the sum over steps
    of its token's log-probability among the legal tokens after its prefix
    (score-first: among all V tokens).  The hidden vector is recomputed from
    scratch as u + sum_{j<s} C_j[t_j].  Wd: the stored weights already widened
    to float64 (model.W_as_f64 of every step), to spare repeated widening."""
    L, V = model.L, model.V
    if Wd is None:
        Wd = _weights_f64(model)
    total = 0.0
    for s in range(1, L + 1):
        prefix = tuple(int(t) for t in sid[:s - 1])
        if deco is not None:
            h = deco_hidden(deco, u_q, prefix)
        else:
            h = np.asarray(u_q, dtype=np.float64).copy()
            for j, t in enumerate(prefix):
                h = h + np.asarray(model.C[j][t], dtype=np.float64)
        T = trie.children(prefix) if trie is not None else np.arange(V)
        t = int(sid[s - 1])
        pos = np.searchsorted(T, t)
        if pos >= T.size or T[pos] != t:
            return -math.inf
        if order == "score_first":
            z = Wd[s - 1] @ h
            total += float(z[t] - (z.max() + math.log(float(np.exp(z - z.max()).sum()))))
        else:
            z = Wd[s - 1][T] @ h
            total += float(filtered_log_softmax(z)[pos])
    return total


def brute_force(trie: Trie, model, u_q: np.ndarray, order: str = "filter_first", deco=None):
    """Exhaustive enumeration for tiny catalogues: every item with its
    filter-first score, computed as the log of the product of per-step
    probabilities softmax(z over legal tokens)[token] (score-first:
    softmax(z over all V tokens)[token]), walking the trie recursively
    (independent of ``decode``).  Returns (sids [n, L] ordered by score
    descending then SID ascending, scores)."""
    L, V = model.L, model.V
    Wd = _weights_f64(model)
    items, probs = [], []

    def walk(prefix, prob):
        s = len(prefix) + 1
        if deco is not None:
            h = deco_hidden(deco, u_q, prefix)
        else:
            h = np.asarray(u_q, dtype=np.float64) + sum(
                (np.asarray(model.C[j][t], dtype=np.float64) for j, t in enumerate(prefix)),
                np.zeros(model.d))
        T = trie.children(prefix)
        if order == "score_first":
            z = Wd[s - 1] @ h
            e = np.exp(z - z.max())
            p = (e / e.sum())[T]
        else:
            z = Wd[s - 1][T] @ h
            e = np.exp(z - z.max())
            p = e / e.sum()
        for t, pt in zip(T, p):
            if s == L:
                items.append(prefix + (int(t),))
                probs.append(prob + math.log(pt))
            else:
                walk(prefix + (int(t),), prob + math.log(pt))

    walk((), 0.0)
    sids = np.array(items, dtype=np.int64).reshape(-1, L)
    sc = np.array(probs)
    order = np.lexsort(tuple(sids[:, j] for j in range(L - 1, -1, -1)) + (-sc,))
    return sids[order], sc[order]
