"""Full steps whose scores never reach memory (chunk tops) and the single
rounding of the hidden vector, against the oracle and against the written
scores.

The full projection's epilogue keeps, per 32-token chunk of a beam row, the
legal (max, sum exp), the second-largest legal score and the position of the
largest; the select cuts on chunk maxima and re-scores only chunks whose
second-largest also clears the cut.  With fp32 weights the re-score repeats
the SIMT projection's arithmetic in the same order, so on dense-format steps a
decode is bit-identical to the one that writes every score (on sparse-format
steps the written path normalises with the standard exponential, so scores
agree to rounding); with half weights the re-score may differ from the tensor
cores by rounding, so results are checked against the oracle.  Mass exact ties drive the select through its narrowing
histograms and its ordered tie walk.
"""
import numpy as np
import pytest

import _helpers as _h
import oracle
import synth
from _helpers import check_topk, tiny_catalogue

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
WINDOW = 1e-4


@pytest.fixture(scope="module")
def zg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import generative_recommendation_constrained_gb300 as zg
    return zg


def _stream():
    return torch.cuda.current_stream().cuda_stream


def run(zg, idx, model, u, beam, K, variants=None, scores=0, hidden=0, fused=0, dm=None, uncon=False):
    """Decode with a forced plan; uncon: the unconstrained decode (no index)
    with the plan's full-projection settings."""
    from generative_recommendation_constrained_gb300.device import Decoder, DeviceModel
    dm = dm or DeviceModel(model)
    B = u.shape[0]
    plan = None
    if idx is not None:
        plan = zg.zg_plan_force(idx, B, beam, variants)
        zg.zg_plan_set_fusion(plan, fused)
        zg.zg_plan_set_full_projection(plan, hidden, scores)
    dec = Decoder(None if uncon else idx, plan, dm, B, beam, K)
    s, sc = dec(torch.from_numpy(np.ascontiguousarray(u)).cuda())
    torch.cuda.synchronize()
    zg.zg_check_device_status(0)
    return s.cpu().numpy(), sc.cpu().numpy()


@pytest.fixture(scope="module")
def mid(zg):
    cfg = synth.CONFIGS["mid_sparse"]
    sids = synth.make_catalogue(cfg)
    model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype)
    u = synth.make_requests(cfg.batch, cfg.d)
    trie = oracle.Trie(sids, cfg.L, cfg.V)
    ref = oracle.decode(trie, model, u, cfg.beam, cfg.topk)
    idx = zg.zg_index_build(sids, cfg.V, stream=_stream())
    return cfg, sids, model, u, trie, ref, idx


def same_results(a, b, ref, L, tol=2e-6, window=1e-5):
    """Equal SIDs wherever no oracle beam boundary is within the window, and
    equal scores to within the log-sum-exp's rounding (written scores of a
    sparse-format step are normalised from the scores with the standard
    exponential, chunk tops from the epilogue's partials)."""
    clean = ~np.any(ref.gaps[:, :L - 1] <= window, axis=1)
    assert np.array_equal(a[0][clean], b[0][clean])
    fin = np.isfinite(a[1])
    assert np.array_equal(fin, np.isfinite(b[1]))
    assert np.max(np.abs(a[1][fin] - b[1][fin]), initial=0.0) <= tol


@pytest.mark.parametrize("variants", [[1, 1, 1], [0, 1, 1], [1, 0, 1]])
def test_fp32_chunk_tops_equal_written(zg, mid, variants):
    cfg, sids, model, u, trie, ref, idx = mid
    a = run(zg, idx, model, u, cfg.beam, cfg.topk, variants, scores=zg.ZG_SCORES_WRITTEN)
    b = run(zg, idx, model, u, cfg.beam, cfg.topk, variants, scores=zg.ZG_SCORES_CHUNK_TOPS)
    same_results(a, b, ref, cfg.L)
    check_topk(b[0], b[1], ref, trie, model, u, 1e-4, WINDOW)


def test_fp32_dense_steps_bit_identical(zg):
    """On dense-format steps both paths normalise from the same partials and
    the re-score repeats the SIMT projection's arithmetic: bit-identical."""
    cfg = synth.CONFIGS["tiny"]
    sids = synth.make_catalogue(cfg)
    model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype)
    u = synth.make_requests(6, cfg.d)
    idx = zg.zg_index_build(sids, cfg.V, format_mode=zg.ZG_FORMAT_ALL_DENSE, stream=_stream())
    a = run(zg, idx, model, u, cfg.beam, cfg.topk, [1, 1, 1], scores=zg.ZG_SCORES_WRITTEN)
    b = run(zg, idx, model, u, cfg.beam, cfg.topk, [1, 1, 1], scores=zg.ZG_SCORES_CHUNK_TOPS)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_tiny_chunk_tops_every_format(zg, mode):
    """Few chunks per kept candidate (the cut takes every chunk) and sparse
    steps expanded into per-beam bitmaps."""
    cfg = synth.CONFIGS["tiny"]
    sids = synth.make_catalogue(cfg)
    model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype)
    u = synth.make_requests(6, cfg.d)
    idx = zg.zg_index_build(sids, cfg.V, format_mode=mode, stream=_stream())
    trie = oracle.Trie(sids, cfg.L, cfg.V)
    ref = oracle.decode(trie, model, u, cfg.beam, cfg.topk)
    a = run(zg, idx, model, u, cfg.beam, cfg.topk, [1, 1, 1], scores=zg.ZG_SCORES_WRITTEN)
    b = run(zg, idx, model, u, cfg.beam, cfg.topk, [1, 1, 1], scores=zg.ZG_SCORES_CHUNK_TOPS)
    same_results(a, b, ref, cfg.L)
    check_topk(b[0], b[1], ref, trie, model, u, 1e-4, WINDOW)


def test_fewer_candidates_than_keep(zg):
    """Fewer legal tokens than the beam at every step (dead beams, padding)."""
    sids = np.array([[0, 1, 2], [0, 1, 3], [5, 0, 0], [40, 7, 9]], np.int32)
    model = synth.make_model(3, 64, 16, "f32", 2)
    u = synth.make_requests(2, 16, 2)
    idx = zg.zg_index_build(sids, 64, stream=_stream())
    trie = oracle.Trie(sids, 3, 64)
    ref = oracle.decode(trie, model, u, 8, 8)
    s, sc = run(zg, idx, model, u, 8, 8, [1, 1, 1], scores=zg.ZG_SCORES_CHUNK_TOPS)
    assert np.array_equal(s, ref.sids)
    assert np.allclose(sc, ref.scores, atol=1e-5)


@pytest.mark.parametrize("g0", [32, 512, 4096])
def test_chunk_tops_exact_ties(zg, g0):
    """Identical weight rows in groups of g0 tokens: every chunk's maximum
    ties with its second (re-scored), with g0 = 4,096 every step-1 candidate
    ties (the list overflows, the histograms narrow to one key and the
    ordered tie walk picks the lowest slots)."""
    V, d, beam = 4096, 32, 16
    T2 = np.arange(0, V, 103)[:40]
    sids = np.stack(np.meshgrid(np.arange(V), T2, indexing="ij"), -1).reshape(-1, 2).astype(np.int32)
    model = synth.make_model(2, V, d, "f32", 11)
    model.W[0][:] = model.W[0][(np.arange(V) // g0) * g0]
    model.C[0][:] = model.C[0][(np.arange(V) // g0) * g0]
    model.W[1][:] = model.W[1][(np.arange(V) // 256) * 256]
    u = synth.make_requests(2, d, 11)
    idx = zg.zg_index_build(sids, V, stream=_stream())
    trie = oracle.Trie(sids, 2, V)
    ref = oracle.decode(trie, model, u, beam, beam)
    s, sc = run(zg, idx, model, u, beam, beam, [1, 1], scores=zg.ZG_SCORES_CHUNK_TOPS)
    assert np.array_equal(s, ref.sids)
    assert np.allclose(sc, ref.scores, atol=1e-4)


def _dense2(V, n1, p, seed):
    rng = np.random.default_rng(seed)
    first = rng.choice(V, n1, replace=False)
    rows = [np.stack([np.full(k.size, f), k], 1) for f in first for k in [np.nonzero(rng.random(V) < p)[0]]]
    return np.concatenate(rows).astype(np.int32)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_half_weights_chunk_tops_vs_oracle(zg, dtype):
    """Tensor-core full steps (hi + lo hidden) handing chunk tops to the
    select on a dense step and the unconstrained decode."""
    V, d = 4096, 64
    sids = _dense2(V, 40, 0.9, 5)
    model = synth.make_model(2, V, d, dtype, 5)
    u = synth.make_requests(3, d, 5)
    idx = zg.zg_index_build(sids, V, stream=_stream())
    trie = oracle.Trie(sids, 2, V)
    ref = oracle.decode(trie, model, u, 16, 16)
    a = run(zg, idx, model, u, 16, 16, [1, 1], scores=zg.ZG_SCORES_WRITTEN)
    b = run(zg, idx, model, u, 16, 16, [1, 1], scores=zg.ZG_SCORES_CHUNK_TOPS)
    check_topk(b[0], b[1], ref, trie, model, u, 2e-2, WINDOW)
    fin = np.isfinite(a[1])
    assert np.array_equal(fin, np.isfinite(b[1]))
    assert np.max(np.abs(a[1][fin] - b[1][fin]), initial=0.0) <= 1e-5
    # a large-vocabulary step without written scores in the unconstrained decode
    uref = oracle.decode(None, model, u, 16, 16)
    s, sc = run(zg, idx, model, u, 16, 16, [1, 1], scores=zg.ZG_SCORES_CHUNK_TOPS, uncon=True)
    check_topk(s, sc, uref, None, model, u, 2e-2, WINDOW)


@pytest.mark.parametrize("dtype,window", [("bf16", 1e-2), ("f16", 2e-3)])
@pytest.mark.parametrize("scores", [1, 2])
def test_single_rounding_hidden(zg, dtype, window, scores):
    """One rounding of the hidden vector: half the tensor work; every returned
    score must still equal its item's exact path score within 2e-2, and the
    top-K sets must match wherever the oracle's beam boundaries are clear of
    the rounding (window)."""
    V, d = 4096, 64
    sids = _dense2(V, 40, 0.9, 6)
    model = synth.make_model(2, V, d, dtype, 6)
    u = synth.make_requests(4, d, 6)
    idx = zg.zg_index_build(sids, V, stream=_stream())
    trie = oracle.Trie(sids, 2, V)
    ref = oracle.decode(trie, model, u, 16, 16)
    s, sc = run(zg, idx, model, u, 16, 16, [1, 1], scores=scores, hidden=zg.ZG_HIDDEN_SINGLE)
    amb = check_topk(s, sc, ref, trie, model, u, 2e-2, window)
    print(f"single rounding {dtype} scores={scores}: near-tie requests {amb} of 4, "
          f"max |score - exact| {_h.LAST_MAX_ERR:.2e}")
    assert _h.LAST_MAX_ERR < (5e-3 if dtype == "bf16" else 1e-3)
