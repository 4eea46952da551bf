"""zg_decode_static: the decode for callers that cannot allocate device
memory while they serve (device memory pre-reserved by another framework's
allocator, request threads where allocation is not allowed, statically
planned runtimes).  Its scratch is the library's fixed 16 MiB device array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import synth

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


def test_static_scratch_decode_matches_workspace_decode(zg):
    from generative_recommendation_constrained_gb300.device import Decoder, DeviceModel
    cfg = synth.CONFIGS["mid_sparse"]
    sids = synth.make_catalogue(cfg)
    model = synth.make_model(cfg.L, cfg.V, cfg.d, cfg.w_dtype)
    stream = torch.cuda.current_stream().cuda_stream
    idx = zg.zg_index_build(sids, cfg.V, stream=stream)
    dm = DeviceModel(model)
    plan = zg.zg_plan_force(idx, cfg.batch, cfg.beam, [1, 0, 0])
    assert zg.zg_decode_workspace_size(idx, plan, dm.struct, cfg.batch, cfg.beam, cfg.topk) \
        <= zg._lib.ZG_STATIC_SCRATCH_BYTES
    ref = Decoder(idx, plan, dm, cfg.batch, cfg.beam, cfg.topk)
    out_sids = torch.empty((cfg.batch, cfg.topk, cfg.L), dtype=torch.int32, device="cuda")
    out_scores = torch.empty((cfg.batch, cfg.topk), dtype=torch.float32, device="cuda")
    for call in range(2):          # two calls in a row share the static array
        u = torch.from_numpy(synth.make_requests(cfg.batch, cfg.d, 500 + call)).cuda()
        want_s, want_sc = ref(u)
        out_sids.fill_(-7)
        out_scores.fill_(7.0)
        zg.zg_decode_static(idx, plan, dm.struct, u, cfg.batch, cfg.beam, cfg.topk, out_sids, out_scores,
                            stream)
        torch.cuda.synchronize()
        zg.zg_check_device_status(stream)
        a, b = want_sc.cpu().numpy(), out_scores.cpu().numpy()
        fin = np.isfinite(a)
        assert np.array_equal(fin, np.isfinite(b))
        assert np.max(np.abs(a[fin] - b[fin]), initial=0.0) <= 1e-4
        assert np.array_equal(want_s.cpu().numpy(), out_sids.cpu().numpy())


def test_static_scratch_rejects_large_decodes(zg):
    from generative_recommendation_constrained_gb300.device import DeviceModel
    model = synth.make_model(2, 16384, 64, "bf16", 3)
    dm = DeviceModel(model)
    B, beam, K = 64, 64, 64                  # unconstrained: 64*64 x 16384 scores, far above 16 MiB
    u = torch.zeros((B, 64), dtype=torch.float32, device="cuda")
    s = torch.empty((B, K, 2), dtype=torch.int32, device="cuda")
    sc = torch.empty((B, K), dtype=torch.float32, device="cuda")
    with pytest.raises(zg.ZgError) as e:
        zg.zg_decode_static(None, None, dm.struct, u, B, beam, K, s, sc, 0)
    assert e.value.status == 1 and "static scratch" in str(e.value)
