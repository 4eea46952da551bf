"""Failure paths exercised without a GPU fault.

Index build: a host-side injection makes the builder's pinned staging
allocation or a host-to-device copy report a failure; the build must return
the status, release what it holds, and the next build must work.

Tensor-core full projection: every mbarrier wait in the
kernel is bounded; when one gives up, the kernel records the timeout bit in
the device status word, drains its own copies and tensor-core operations,
frees its tensor memory and returns, leaving the context usable.

The test lowers the wait limit to a single poll (no operand load lands that
fast), so the pipeline waits expire on a small full-projection decode; it
checks that zg_check_device_status reports the timeout, and that with the
default limit restored the next decode is correct against the oracle.  No
kernel is made to fault or hang: the expiry is the kernel's own bounded wait.
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import check_topk, tiny_catalogue

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def zg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import generative_recommendation_constrained_gb300 as zg
    return zg


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tensor_core_wait_expiry_is_reported_and_recovers(zg, dtype):
    from generative_recommendation_constrained_gb300.device import Decoder, DeviceModel
    L, V, d, B, beam, K = 2, 640, 64, 3, 8, 8
    sids = tiny_catalogue(L, V, 5000, 11)
    model = synth.make_model(L, V, d, dtype, 11)
    u = synth.make_requests(B, d, 11)
    stream = torch.cuda.current_stream().cuda_stream
    idx = zg.zg_index_build(sids, V, stream=stream)
    dm = DeviceModel(model)
    plan = zg.zg_plan_force(idx, B, beam, [1] * L)      # tensor-core full projection at every step
    dec = Decoder(idx, plan, dm, B, beam, K)
    ud = torch.from_numpy(u).cuda()
    zg.zg_check_device_status(stream)                    # nothing pending
    zg.zg_debug_set_wait_limit(1)
    try:
        dec(ud)
        with pytest.raises(zg.ZgError) as e:
            zg.zg_check_device_status(stream)
        assert e.value.status == 6 and "tensor-core wait expired" in str(e.value)
    finally:
        zg.zg_debug_set_wait_limit(0)
    zg.zg_check_device_status(stream)                    # the flag was cleared by the read
    for _ in range(2):                                   # the context still works: correct decodes
        s, sc = dec(ud)
        torch.cuda.synchronize()
        zg.zg_check_device_status(stream)
        trie = oracle.Trie(sids, L, V)
        ref = oracle.decode(trie, model, u, beam, K)
        check_topk(s.cpu().numpy(), sc.cpu().numpy(), ref, trie, model, u, 2e-2, 1e-4)


@pytest.mark.parametrize("point,after,code", [(1, 0, 2), (1, 1, 2), (2, 0, 3), (2, 3, 3)])
def test_index_build_injected_failure_and_recovery(zg, point, after, code):
    V = 64
    sids = tiny_catalogue(3, V, 3000, 4)
    stream = torch.cuda.current_stream().cuda_stream
    zg.zg_debug_inject_build_failure(point, after)
    try:
        with pytest.raises(zg.ZgError) as e:
            zg.zg_index_build(sids, V, stream=stream, pinned_chunk_bytes=1 << 12)
        assert e.value.status == code
    finally:
        zg.zg_debug_inject_build_failure(0, 0)
    torch.cuda.synchronize()
    idx = zg.zg_index_build(sids, V, stream=stream, pinned_chunk_bytes=1 << 12)
    tabs = oracle.serialize_index(sids, 3, V)
    for s in (1, 2, 3):
        assert zg.zg_index_export(idx, s) == tabs[s - 1].export_bytes()
