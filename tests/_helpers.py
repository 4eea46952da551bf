"""Shared test helpers: tiny catalogues, golden fixtures and the top-K parity check."""
from __future__ import annotations

import math

import numpy as np

import synth

LAST_MAX_ERR = 0.0


def tiny_catalogue(L: int, V: int, n: int, seed: int) -> np.ndarray:
    return synth.catalogue_uniform(L, V, n, seed)


def golden_catalogue(fx):
    L = fx["L"][0][0]
    V = fx["V"][0][0]
    sids = np.array(fx["item"], dtype=np.int32)
    return L, V, sids


def check_topk(gpu_sids, gpu_scores, ref, trie, model, u, tol, window, requests=None, order="filter_first",
               deco=None):
    """Compare a decode's top-K output with the oracle's.

    Both sides compute the same beam search; floating-point rounding differs
    (fp32 vs fp64), so decisions between candidates whose exact scores lie
    within ``window`` of each other may go either way.  For every request:
      * output rows are valid: SIDs in the catalogue (constrained decode),
        distinct, scores non-increasing, padding (-1 / -inf) only at the end;
      * each returned score equals the exact path score of its SID (in the
        decode's order: filter-first or score-first) within ``tol``;
      * unless an intermediate beam boundary was a near-tie (gap <= window),
        the same number of outputs is returned, the sorted score lists agree
        within ``tol`` and every oracle item whose score clears the first
        dropped candidate by more than ``window`` is returned.
    deco: the light decoder's weights when it produces the hidden vectors (u
    then holds the concept vectors).
    Returns the number of requests that had only the first two checks; the
    largest |score - exact path score| seen is left in LAST_MAX_ERR."""
    global LAST_MAX_ERR
    gpu_sids = np.asarray(gpu_sids)
    gpu_scores = np.asarray(gpu_scores, dtype=np.float64)
    B, K, L = gpu_sids.shape
    req = range(B) if requests is None else list(requests)
    ambiguous = 0
    max_err = 0.0
    Wd = [model.W_as_f64(s) for s in range(model.L)]
    for q in req:
        valid = gpu_sids[q, :, 0] >= 0
        nv = int(valid.sum())
        assert valid[:nv].all(), f"request {q}: padding is not at the end"
        assert np.all(gpu_sids[q, nv:] == -1)
        assert np.all(np.isneginf(gpu_scores[q, nv:]))
        sc = gpu_scores[q, :nv]
        assert np.all(np.isfinite(sc))
        assert np.all(np.diff(sc) <= 1e-7 + 1e-7 * np.abs(sc[1:])), f"request {q}: not sorted"
        seen = set()
        for i in range(nv):
            sid = tuple(int(t) for t in gpu_sids[q, i])
            assert sid not in seen, f"request {q}: duplicate SID {sid}"
            seen.add(sid)
            if trie is not None:
                assert trie.contains(sid), f"request {q}: SID {sid} not in catalogue"
            exact = _path(trie, model, u[q], sid, order, Wd, deco)
            max_err = max(max_err, abs(exact - sc[i]))
            LAST_MAX_ERR = max_err
            assert abs(exact - sc[i]) <= tol, \
                f"request {q} rank {i}: score {sc[i]} vs exact {exact}"
        if np.any(ref.gaps[q, :L - 1] <= window):
            ambiguous += 1
            continue
        rv = ref.sids[q, :, 0] >= 0
        nr = int(rv.sum())
        assert nr == nv, f"request {q}: {nv} outputs vs oracle {nr}"
        ref_sc = ref.scores[q, :nr]
        assert np.max(np.abs(np.sort(sc) - np.sort(ref_sc)), initial=0.0) <= tol, \
            f"request {q}: sorted scores differ"
        cut = ref.next_score[q] + window
        for i in range(nr):
            if ref_sc[i] > cut:
                sid = tuple(int(t) for t in ref.sids[q, i])
                assert sid in seen, f"request {q}: oracle item {sid} ({ref_sc[i]}) missing"
    return ambiguous


def _path(trie, model, u_q, sid, order="filter_first", Wd=None, deco=None):
    from oracle import path_score
    return path_score(trie, model, u_q, sid, order, Wd, deco)


def isclose_inf(a, b, tol):
    if math.isinf(a) or math.isinf(b):
        return a == b
    return abs(a - b) <= tol
