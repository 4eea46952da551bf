"""The C-ABI library on the CPU: it builds, loads, exports every declared
symbol, and its host-side logic (index builder, argument checks, save/load)
matches the oracle.  No CUDA device is used."""
import os
import re

import numpy as np
import pytest

import oracle
import synth
from _helpers import golden_catalogue, tiny_catalogue
from conftest import ROOT, read_golden


@pytest.fixture(scope="module")
def zg():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_zg_build", os.path.join(ROOT, "generative_recommendation_constrained_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import generative_recommendation_constrained_gb300 as zg
    return zg


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^ZG_API\s+[\w\s\*]+?\b(zg_\w+)\s*\(", txt, flags=re.M))
    return sorted(names)


def test_exports_every_declared_symbol(zg):
    import ctypes
    names = _declared_symbols()
    assert len(names) >= 18
    lib = ctypes.CDLL(zg.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_version(zg):
    assert "sm_103a" in zg.zg_version()


CATS = [("tiny", None), ("uni_3_8_60", (3, 8, 60, 0)), ("uni_2_40_300", (2, 40, 300, 1)),
        ("uni_4_5_200", (4, 5, 200, 2)), ("uni_1_33_20", (1, 33, 20, 3)),
        ("uni_3_64_500", (3, 64, 500, 4)), ("uni_2_70_900", (2, 70, 900, 5))]


def _cat(spec):
    name, p = spec
    if p is None:
        cfg = synth.CONFIGS[name]
        return cfg.L, cfg.V, synth.make_catalogue(cfg)
    L, V, n, seed = p
    return L, V, tiny_catalogue(L, V, n, seed)


@pytest.mark.parametrize("spec", CATS, ids=[c[0] for c in CATS])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_host_index_bit_exact(zg, spec, mode):
    L, V, sids = _cat(spec)
    dup = np.concatenate([sids, sids[::7]])                     # duplicates merge
    rng = np.random.default_rng(0)
    dup = dup[rng.permutation(dup.shape[0])]
    idx = zg.zg_index_build(dup, V, format_mode=mode, residency=zg.ZG_RESIDENT_HOST, n_threads=3,
                            pinned_chunk_bytes=4096)
    fmt = -1 if mode == 0 else (oracle.SPARSE if mode == 1 else oracle.DENSE)
    tabs = oracle.serialize_index(dup, L, V, force_format=fmt)
    info = zg.zg_index_info_get(idx)
    assert info["n_input"] == dup.shape[0] and info["n_unique"] == sids.shape[0]
    assert info["dense_trie_bytes"] == sum(t.rows * V * 4 for t in tabs)
    for s in range(1, L + 1):
        assert zg.zg_index_export(idx, s) == tabs[s - 1].export_bytes(), f"step {s}"
        st = zg.zg_index_stats(idx, s)
        assert st["max_fanout"] == tabs[s - 1].max_fanout
        assert st["rows"] == tabs[s - 1].rows and st["nnz"] == tabs[s - 1].nnz


def test_worked_example_host_index(zg):
    L, V, sids = golden_catalogue(read_golden("worked_example.txt"))
    for mode in (1, 2):
        idx = zg.zg_index_build(sids, V, format_mode=mode, residency=zg.ZG_RESIDENT_HOST)
        fmt = oracle.SPARSE if mode == 1 else oracle.DENSE
        tabs = oracle.serialize_index(sids, L, V, force_format=fmt)
        for s in range(1, L + 1):
            assert zg.zg_index_export(idx, s) == tabs[s - 1].export_bytes()


def test_threads_do_not_change_the_index(zg):
    cfg = synth.CONFIGS["mid_sparse"]
    sids = synth.make_catalogue(cfg)
    a = zg.zg_index_build(sids, cfg.V, residency=zg.ZG_RESIDENT_HOST, n_threads=1)
    b = zg.zg_index_build(sids, cfg.V, residency=zg.ZG_RESIDENT_HOST, n_threads=8,
                          pinned_chunk_bytes=1 << 16)
    tabs = oracle.serialize_index(sids, cfg.L, cfg.V)
    for s in range(1, cfg.L + 1):
        ea = zg.zg_index_export(a, s)
        assert ea == zg.zg_index_export(b, s) == tabs[s - 1].export_bytes()
    assert [zg.zg_index_stats(a, s)["format"] for s in (1, 2, 3)] == [1, 0, 0]


def test_save_load_roundtrip_and_corruption(zg, tmp_path):
    L, V, sids = 3, 64, tiny_catalogue(3, 64, 500, 9)
    idx = zg.zg_index_build(sids, V, residency=zg.ZG_RESIDENT_HOST)
    p = str(tmp_path / "i.zgidx")
    zg.zg_index_save(idx, p)
    back = zg.zg_index_load(p, zg.ZG_RESIDENT_HOST)
    for s in range(1, L + 1):
        assert zg.zg_index_export(back, s) == zg.zg_index_export(idx, s)
    raw = bytearray(open(p, "rb").read())
    raw[len(raw) // 2] ^= 0xFF
    open(p, "wb").write(bytes(raw))
    with pytest.raises(zg.ZgError) as e:
        zg.zg_index_load(p, zg.ZG_RESIDENT_HOST)
    assert e.value.status == 7
    open(p, "wb").write(bytes(raw[:40]))
    with pytest.raises(zg.ZgError):
        zg.zg_index_load(p, zg.ZG_RESIDENT_HOST)
    with pytest.raises(zg.ZgError):
        zg.zg_index_load(str(tmp_path / "missing"), zg.ZG_RESIDENT_HOST)


@pytest.mark.parametrize("sids,V,code", [
    (np.zeros((0, 3), np.int32), 8, 1),                       # empty catalogue
    (np.array([[0, 8, 1]], np.int32), 8, 1),                  # token >= V
    (np.array([[0, -1, 1]], np.int32), 8, 1),                 # negative token
    (np.zeros((1, 9), np.int32), 8, 1),                       # L > 8
    (np.zeros((1, 3), np.int32), 0, 1),                       # V < 1
    (np.zeros((1, 3), np.int32), 65537, 1),                   # V > 65536
    (np.zeros((1, 5), np.int32), 65536, 4),                   # 5 * 16 key bits > 64
])
def test_build_rejects_bad_input(zg, sids, V, code):
    with pytest.raises(zg.ZgError) as e:
        zg.zg_index_build(sids, V, residency=zg.ZG_RESIDENT_HOST)
    assert e.value.status == code
    assert len(str(e.value)) > 20


def test_decode_argument_checks(zg):
    """Checks that happen before any CUDA call (unconstrained, fake pointers)."""
    fake = 1 << 20
    m = zg.make_model(3, 64, 32, zg.ZG_F32, [fake, fake], [fake, fake, fake])
    n = zg.zg_decode_workspace_size(None, None, m, 4, 8, 8)
    assert n > 4 * 8 * 32 * 4
    bad = [
        dict(B=0, beam=8, K=8), dict(B=4, beam=8, K=9), dict(B=4, beam=0, K=0),
        dict(B=4, beam=513, K=1),
    ]
    for kw in bad:
        with pytest.raises(zg.ZgError) as e:
            zg.zg_decode_workspace_size(None, None, m, kw["B"], kw["beam"], kw["K"])
        assert e.value.status == 1
    for dd in (12, 0, 1032):
        m2 = zg.make_model(3, 64, dd, zg.ZG_F32, [fake, fake], [fake, fake, fake])
        with pytest.raises(zg.ZgError):
            zg.zg_decode_workspace_size(None, None, m2, 4, 8, 8)
    m3 = zg.make_model(3, 64, 32, zg.ZG_F32, [fake, 0], [fake, fake, fake])   # C[1] missing
    with pytest.raises(zg.ZgError):
        zg.zg_decode_workspace_size(None, None, m3, 4, 8, 8)
    m4 = zg.make_model(3, 64, 32, 7, [fake, fake], [fake, fake, fake])        # bad dtype
    with pytest.raises(zg.ZgError):
        zg.zg_decode_workspace_size(None, None, m4, 4, 8, 8)
    # a host-resident index cannot be decoded
    idx = zg.zg_index_build(tiny_catalogue(3, 64, 100, 1), 64, residency=zg.ZG_RESIDENT_HOST)
    with pytest.raises(zg.ZgError) as e:
        zg.zg_decode_workspace_size(idx, None, m, 4, 8, 8)
    assert "host-resident" in str(e.value)
    # workspace too small / misaligned, before any launch
    with pytest.raises(zg.ZgError):
        zg.zg_decode(None, None, m, fake, 4, 8, 8, fake, fake, fake, 16, 0)
    with pytest.raises(zg.ZgError):
        zg.zg_decode(None, None, m, fake, 4, 8, 8, fake, fake, fake + 8, n, 0)


def test_plan_force_checks(zg):
    idx = zg.zg_index_build(tiny_catalogue(3, 16, 50, 2), 16, residency=zg.ZG_RESIDENT_HOST)
    p = zg.zg_plan_force(idx, 2, 4, [0, 1, 0])
    v, ms, g, fms = zg.zg_plan_describe(p)
    assert list(v) == [0, 1, 0] and (ms == -1).all() and g == 8 and (fms == -1).all()
    zg.zg_plan_set_fusion(p, 0)
    assert zg.zg_plan_describe(p)[2] == 0
    with pytest.raises(zg.ZgError):
        zg.zg_plan_set_fusion(p, 3)
    with pytest.raises(zg.ZgError):
        zg.zg_plan_force(idx, 2, 4, [0, 3, 0])


def test_plan_variants_and_order_checked(zg):
    """zg_plan_force takes ZG_SELECTIVE / ZG_FULL / ZG_NAIVE only; the order
    setter takes the two orders only (host-side checks, no GPU)."""
    idx = zg.zg_index_build(tiny_catalogue(3, 16, 50, 2), 16, residency=zg.ZG_RESIDENT_HOST)
    L = zg.zg_index_info_get(idx)["L"]
    p = zg.zg_plan_force(idx, 2, 4, [zg.ZG_NAIVE] * L)
    assert list(zg.zg_plan_describe(p)[0]) == [zg.ZG_NAIVE] * L
    zg.zg_plan_set_order(p, zg.ZG_ORDER_SCORE_FIRST)
    zg.zg_plan_set_order(p, zg.ZG_ORDER_FILTER_FIRST)
    with pytest.raises(zg.ZgError):
        zg.zg_plan_set_order(p, 2)
    with pytest.raises(zg.ZgError):
        zg.zg_plan_force(idx, 2, 4, [3] * L)


def _fnv1a(b: bytes) -> int:
    h = 1469598103934665603
    for x in b:
        h = ((h ^ x) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h


def _parse_index_file(raw: bytes):
    """Header fields and per-step metadata of a saved index, and where the
    table image starts (the layout zg_index_save writes)."""
    L, V = np.frombuffer(raw[8:16], "<i4")
    off = 8 + 8 + 16 + 8
    steps = []
    for _ in range(int(L)):
        fmt = int(np.frombuffer(raw[off:off + 4], "<i4")[0])
        rows, nnz, words, mf = (int(x) for x in np.frombuffer(raw[off + 4:off + 20], "<u4"))
        o_rp, o_pay, b_rp, b_pay = (int(x) for x in np.frombuffer(raw[off + 20:off + 52], "<u8"))
        steps.append(dict(fmt=fmt, rows=rows, nnz=nnz, words=words, mf=mf, o_rp=o_rp, o_pay=o_pay))
        off += 52
    return int(L), int(V), steps, off


@pytest.mark.parametrize("damage", ["rowptr_decreasing", "rowptr_end", "token_ge_v", "tokens_unsorted",
                                    "bitmap_extra_bit", "max_fanout"])
def test_load_rejects_inconsistent_tables(zg, tmp_path, damage):
    """A file whose checksum is intact but whose tables break the index's
    invariants (rowptr from 0 to nnz, non-decreasing; tokens below V and
    ascending in a row; a dense row's popcount = its fan-out; the stored
    largest fan-out) is refused on load, so no kernel can be pointed out of
    the tables' bounds by a loaded file."""
    L, V, sids = 3, 64, tiny_catalogue(3, 64, 500, 9)
    idx = zg.zg_index_build(sids, V, residency=zg.ZG_RESIDENT_HOST, format_mode=zg.ZG_FORMAT_AUTO)
    p = str(tmp_path / "i.zgidx")
    zg.zg_index_save(idx, p)
    raw = bytearray(open(p, "rb").read())
    L, V, steps, img0 = _parse_index_file(bytes(raw))
    assert [st["fmt"] for st in steps] == [1, 1, 0]    # dense, dense, sparse under the automatic rule
    dense, sparse = steps[1], steps[2]

    def u32(at, val=None):
        o = img0 + at
        if val is None:
            return int(np.frombuffer(raw[o:o + 4], "<u4")[0])
        raw[o:o + 4] = np.array([val], "<u4").tobytes()

    def u16(at, val=None):
        o = img0 + at
        if val is None:
            return int(np.frombuffer(raw[o:o + 2], "<u2")[0])
        raw[o:o + 2] = np.array([val], "<u2").tobytes()

    if damage == "rowptr_decreasing":
        u32(sparse["o_rp"] + 4 * 2, u32(sparse["o_rp"] + 4 * 1) - 1 if u32(sparse["o_rp"] + 4) else 5)
    elif damage == "rowptr_end":
        u32(sparse["o_rp"] + 4 * sparse["rows"], sparse["nnz"] + 3)
    elif damage == "token_ge_v":
        u16(sparse["o_pay"], V + 5)
    elif damage == "tokens_unsorted":
        r = next(r for r in range(sparse["rows"]) if u32(sparse["o_rp"] + 4 * (r + 1)) - u32(sparse["o_rp"] + 4 * r) >= 2)
        e = u32(sparse["o_rp"] + 4 * r)
        a, b = u16(sparse["o_pay"] + 2 * e), u16(sparse["o_pay"] + 2 * (e + 1))
        u16(sparse["o_pay"] + 2 * e, b)
        u16(sparse["o_pay"] + 2 * (e + 1), a)
    elif damage == "bitmap_extra_bit":
        w = u32(dense["o_pay"])
        bit = next(i for i in range(32) if not (w >> i) & 1)
        u32(dense["o_pay"], w | (1 << bit))
    elif damage == "max_fanout":
        o = 8 + 8 + 16 + 8 + 2 * 52 + 16          # step 3's stored max fan-out field
        raw[o:o + 4] = np.array([sparse["mf"] + 1], "<u4").tobytes()
    tot = len(raw) - img0 - 8
    raw[-8:] = np.array([_fnv1a(bytes(raw[img0:img0 + tot]))], "<u8").tobytes()
    open(p, "wb").write(bytes(raw))
    with pytest.raises(zg.ZgError) as e:
        zg.zg_index_load(p, zg.ZG_RESIDENT_HOST)
    assert e.value.status == 7


def test_static_scratch_size_matches_header(zg):
    txt = open(os.path.join(ROOT, "include", "zerogr.h")).read()
    m = re.search(r"#define ZG_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", txt)
    assert m and zg._lib.ZG_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_plan_save_load_roundtrip_and_damage(zg, tmp_path):
    """[Speed]: the per-step choice is kept until the next model update; a
    saved plan loads back identical, and short, corrupt or out-of-range files
    are refused."""
    sids = tiny_catalogue(3, 16, 300, 2)
    idx = zg.zg_index_build(sids, 16, residency=zg.ZG_RESIDENT_HOST)
    plan = zg.zg_plan_force(idx, 5, 8, [1, 0, 2])
    zg.zg_plan_set_fusion(plan, 4)
    zg.zg_plan_set_order(plan, zg.ZG_ORDER_SCORE_FIRST)
    zg.zg_plan_set_full_projection(plan, zg.ZG_HIDDEN_SINGLE, zg.ZG_SCORES_CHUNK_TOPS)
    p = str(tmp_path / "p.zgplan")
    zg.zg_plan_save(plan, p)
    back = zg.zg_plan_load(p)
    a, b = zg.zg_plan_describe(plan), zg.zg_plan_describe(back)
    for x, y in zip(a, b):
        assert np.array_equal(np.asarray(x), np.asarray(y))
    raw = open(p, "rb").read()
    for cut in range(0, len(raw)):                     # every truncation
        open(p, "wb").write(raw[:cut])
        with pytest.raises(zg.ZgError) as e:
            zg.zg_plan_load(p)
        assert e.value.status == 7
    bad = bytearray(raw)
    bad[20] ^= 0x40                                    # a flipped bit: checksum mismatch
    open(p, "wb").write(bytes(bad))
    with pytest.raises(zg.ZgError):
        zg.zg_plan_load(p)
    # a well-formed file with an invalid variant (checksum recomputed)
    body = bytearray(raw[8:-8])
    L = int.from_bytes(body[0:4], "little")
    body[4 * 7 + 4 + 20] = 7                           # first variant byte
    fixed = raw[:8] + bytes(body) + np.array([_fnv1a(bytes(body))], "<u8").tobytes()
    open(p, "wb").write(fixed)
    with pytest.raises(zg.ZgError):
        zg.zg_plan_load(p)
    assert L == 3
