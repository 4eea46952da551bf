"""The light causal decoder as the per-step hidden-state producer, on the GPU
against the oracle ("Separating Thinking from Spelling", AI Papers Daily
digest: a fixed concept from the backbone, a light 2-layer causal decoder
over the concept and the prefix running the trie-constrained beam search).

The decode's input is each request's concept vectors; every step runs the
decoder (embedding, normalisation, causal attention over the request's
concept rows and the beam's ancestors' rows, MLP) before the projection.
Scores are compared with the oracle's fp64 decoder and beam search within the
fp32 tolerance (2e-2 for half output heads).
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


def run(zg, idx, model, deco, concepts, beam, K, variants):
    from generative_recommendation_constrained_gb300.device import Decoder, DeviceModel
    dm = DeviceModel(model, deco=deco)
    B = concepts.shape[0]
    plan = zg.zg_plan_force(idx, B, beam, variants) if idx is not None else None
    dec = Decoder(idx, plan, dm, B, beam, K)
    s, sc = dec(torch.from_numpy(np.ascontiguousarray(concepts)).cuda())
    torch.cuda.synchronize()
    zg.zg_check_device_status(0)
    return s.cpu().numpy(), sc.cpu().numpy(), dec


@pytest.mark.parametrize("variants", [[0, 0, 0], [1, 1, 1], [1, 0, 1], [2, 0, 0]])
def test_decoder_hidden_vectors_vs_oracle(zg, variants):
    L, V, d = 3, 64, 64
    sids = tiny_catalogue(L, V, 600, 3)
    model = synth.make_model(L, V, d, "f32", 3)
    deco = synth.make_deco(L, V, d, M=2, heads=4, ffn=256, layers=2, seed=3)
    c = synth.make_concepts(5, 2, d, 3)
    idx = zg.zg_index_build(sids, V, stream=_stream())
    trie = oracle.Trie(sids, L, V)
    ref = oracle.decode(trie, model, c, 8, 8, deco=deco)
    s, sc, _ = run(zg, idx, model, deco, c, 8, 8, variants)
    amb = check_topk(s, sc, ref, trie, model, c, 1e-4, WINDOW, deco=deco)
    print(f"decoder {variants}: near-tie requests {amb}, max |score - exact| {_h.LAST_MAX_ERR:.2e}")
    assert amb <= 1


def test_decoder_width_256_half_heads(zg):
    """The digest's width (256), four heads, bf16 output heads."""
    L, V, d = 3, 256, 256
    sids = tiny_catalogue(L, V, 3000, 4)
    model = synth.make_model(L, V, d, "bf16", 4)
    deco = synth.make_deco(L, V, d, M=2, heads=4, ffn=1024, layers=2, seed=4)
    c = synth.make_concepts(3, 2, d, 4)
    idx = zg.zg_index_build(sids, V, stream=_stream())
    trie = oracle.Trie(sids, L, V)
    ref = oracle.decode(trie, model, c, 8, 8, deco=deco)
    for variants in ([0, 0, 0], [1, 1, 0]):
        s, sc, _ = run(zg, idx, model, deco, c, 8, 8, variants)
        check_topk(s, sc, ref, trie, model, c, 2e-2, WINDOW, deco=deco)


def test_decoder_unconstrained_and_trace(zg):
    """Unconstrained decode over the decoder; the trace reports the decoder's
    time per step beside the projection and select."""
    L, V, d = 3, 40, 32
    model = synth.make_model(L, V, d, "f32", 5)
    deco = synth.make_deco(L, V, d, M=3, heads=2, ffn=64, layers=2, seed=5)
    c = synth.make_concepts(2, 3, d, 5)
    ref = oracle.decode(None, model, c, 6, 6, deco=deco)
    s, sc, dec = run(zg, None, model, deco, c, 6, 6, None)
    check_topk(s, sc, ref, None, model, c, 1e-4, WINDOW, deco=deco)
    tr = dec.trace(torch.from_numpy(c).cuda())
    assert all(st["ms_model"] > 0 for st in tr["steps"])


def test_decoder_host_buffers(zg):
    """zg_decode_host copies the B x M concept vectors in."""
    L, V, d = 2, 32, 32
    sids = tiny_catalogue(L, V, 300, 6)
    model = synth.make_model(L, V, d, "f32", 6)
    deco = synth.make_deco(L, V, d, M=2, heads=2, ffn=64, layers=1, seed=6)
    c = synth.make_concepts(3, 2, d, 6)
    from generative_recommendation_constrained_gb300.device import DeviceModel
    dm = DeviceModel(model, deco=deco)
    idx = zg.zg_index_build(sids, V, stream=_stream())
    plan = zg.zg_plan_force(idx, 3, 4, [0, 0])
    n = zg.zg_decode_host_workspace_size(idx, plan, dm.struct, 3, 4, 4)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o_s = np.zeros((3, 4, 2), np.int32)
    o_sc = np.zeros((3, 4), np.float32)
    zg.zg_decode_host(idx, plan, dm.struct, np.ascontiguousarray(c), 3, 4, 4, o_s, o_sc, ws, n, _stream())
    trie = oracle.Trie(sids, L, V)
    ref = oracle.decode(trie, model, c, 4, 4, deco=deco)
    check_topk(o_s, o_sc, ref, trie, model, c, 1e-4, WINDOW, deco=deco)
