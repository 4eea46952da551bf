"""Full-size configurations (10M-100M items) on the GPU against the oracle:
the codebook sweep (V = 2,048 .. 16,384, bf16), the dense-early catalogue
(50M items, fp16) and the large catalogue (100M items, bf16, beam 256) at
batch 64 and at the batch sweep's 1, 8 and 32.

  * Index: every step table of every configuration bit-exact against the
    oracle's serialisation.
  * Decode: the whole batch in the tuned plan and in forced all-selective and
    all-full plans; every request of the batch is checked against the
    oracle's beam search (check_topk: SIDs in the catalogue, each score equal
    to the exact path score within the tolerance, the same top-K set wherever
    no intermediate beam boundary is a near-tie).  The number of requests
    with such a near-tie is reported and bounded.
  * Unconstrained decode: eight requests against the oracle.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
import _helpers as _h
from _helpers import check_topk

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")

TOL = 2e-2        # bf16/fp16 weights, fp32 accumulation
# Decision window: every GPU path accumulates in fp32 (the tensor-core path
# with the hidden split into two halves), so candidate scores agree with the
# fp64 oracle to ~1e-6 and a beam boundary can only flip where the oracle's
# own gap is below ~1e-5.  With beam 256 such near-ties are not rare (6 of the
# 64 large-catalogue requests, 3 of 128 dense-early, none of the sweep's).
WINDOW = 1e-5
CASES = [("sweep_v2048", 0), ("sweep_v4096", 0), ("sweep_v8192", 0), ("sweep_v16384", 0),
         ("dense_early", 0), ("large", 0), ("large", 1), ("large", 8), ("large", 32)]
_DATA = {}        # the last configuration's inputs, trie and oracle results (one entry)


@pytest.fixture(scope="module")
def zg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import generative_recommendation_constrained_gb300 as zg
    return zg


def _inputs(name):
    """Catalogue, model, the full batch's requests, trie and the oracle's
    decode of every request of the full batch (cached across batch sizes)."""
    if name not in _DATA:
        _DATA.clear()
        cfg = synth.CONFIGS[name]
        sids = synth.make_catalogue(cfg, 0)
        model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype, 0)
        u = synth.make_requests(cfg.batch, cfg.d, 1000)
        trie = oracle.Trie(sids, cfg.L, cfg.V)
        ref = oracle.decode(trie, model, u, cfg.beam, cfg.topk)
        _DATA[name] = (sids, model, u, trie, ref)
    return _DATA[name]


def _head(ref, B):
    """The oracle's results of the first B requests."""
    return oracle.DecodeResult(ref.sids[:B], ref.scores[:B], ref.gaps[:B], ref.n_cand[:B], ref.next_score[:B])


@pytest.fixture(scope="module", params=CASES, ids=[f"{n}-b{b}" if b else n for n, b in CASES])
def full(request, zg):
    name, B = request.param
    cfg = synth.CONFIGS[name]
    sids, model, u, trie, ref = _inputs(name)
    if B:
        # requests 0..B-1 of the same seeded stream: the first B rows of the full batch
        cfg = dataclasses.replace(cfg, batch=B)
        u = synth.make_requests(B, cfg.d, 1000)
        assert np.array_equal(u, _DATA[name][2][:B])
        ref = _head(ref, B)
    stream = torch.cuda.current_stream().cuda_stream
    idx = zg.zg_index_build(sids, cfg.V, stream=stream)
    yield cfg, sids, model, u, idx, trie, ref, B
    del idx


def _decode(zg, cfg, idx, dm, u, plan):
    from generative_recommendation_constrained_gb300.device import Decoder
    dec = Decoder(idx, plan, dm, u.shape[0], cfg.beam, cfg.topk)
    s, sc = dec(torch.from_numpy(u).cuda())
    torch.cuda.synchronize()
    zg.zg_check_device_status(0)
    return s.cpu().numpy(), sc.cpu().numpy()


def test_fullsize_index(zg, full):
    cfg, sids, model, u, idx, trie, ref, B = full
    if B:
        pytest.skip("index checked once per catalogue")
    info = zg.zg_index_info_get(idx)
    assert info["n_unique"] == trie.n_unique
    tabs = oracle.serialize_index(sids, cfg.L, cfg.V)
    for s in range(1, cfg.L + 1):
        assert zg.zg_index_export(idx, s) == tabs[s - 1].export_bytes(), f"step {s}"


def test_fullsize_decode_plans(zg, full):
    cfg, sids, model, u, idx, trie, ref, B = full
    from generative_recommendation_constrained_gb300.device import DeviceModel
    dm = DeviceModel(model)
    stream = torch.cuda.current_stream().cuda_stream
    warm = torch.from_numpy(synth.make_requests(cfg.batch, cfg.d, 99)).cuda()
    tuned = zg.zg_tune(idx, dm.struct, warm, cfg.batch, cfg.beam, cfg.topk, 3, stream)
    plans = {"tuned": tuned,
             "selective": zg.zg_plan_force(idx, cfg.batch, cfg.beam, [0] * cfg.L),
             "full": zg.zg_plan_force(idx, cfg.batch, cfg.beam, [1] * cfg.L)}
    amb = {}
    outs = {}
    for name, plan in plans.items():
        s, sc = _decode(zg, cfg, idx, dm, u, plan)
        amb[name] = check_topk(s, sc, ref, trie, model, u, TOL, WINDOW)
        amb[name + "_max_err"] = _h.LAST_MAX_ERR
        outs[name] = sc
    print(f"{cfg.name} batch {cfg.batch}: near-tie requests (set check skipped) and max |score - exact|: {amb}")
    # every request is checked for validity and exact path scores; the set check
    # may be skipped only where the oracle's own beam boundary is a near-tie
    near = int(np.sum(np.any(ref.gaps[:, :cfg.L - 1] <= WINDOW, axis=1)))
    assert all(amb[n] == near for n in plans)
    assert near <= max(2, cfg.batch // 8), f"{near} of {cfg.batch} requests have near-ties"
    # where no beam boundary is a near-tie, every plan returns the same scores
    clean = ~np.any(ref.gaps[:, :cfg.L - 1] <= WINDOW, axis=1)
    for name in ("selective", "full"):
        a, b = outs["tuned"][clean], outs[name][clean]
        fin = np.isfinite(a)
        assert np.array_equal(fin, np.isfinite(b))
        assert np.max(np.abs(a[fin] - b[fin]), initial=0.0) <= TOL


def test_fullsize_unconstrained(zg, full):
    cfg, sids, model, u, idx, trie, ref, B = full
    if B:
        pytest.skip("unconstrained decode checked once per catalogue")
    from generative_recommendation_constrained_gb300.device import DeviceModel
    dm = DeviceModel(model)
    uu = np.ascontiguousarray(u[:8])
    s, sc = _decode(zg, cfg, None, dm, uu, None)
    uref = oracle.decode(None, model, uu, cfg.beam, cfg.topk)
    amb = check_topk(s, sc, uref, None, model, uu, TOL, WINDOW)
    assert amb <= 2
