"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every entry point the header declares, status strings, argument
validation and the planner's choices."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("tsgemm.h", "tsattn.h")]


@pytest.fixture(scope="module")
def ts():
    from hierarchical_gemm_gb300 import build
    build.build()
    from hierarchical_gemm_gb300 import tsgemm
    return tsgemm


def _declared():
    text = "".join(open(h).read() for h in HEADERS)
    return set(re.findall(r"TSGEMM_API\s+[\w\s\*]+?\b(ts(?:gemm|attn)_\w+)\s*\(", text))


def test_library_exports_every_declared_symbol(ts):
    names = _declared()
    assert {"tsgemm_plan", "tsgemm_run", "tsgemm_destroy"} <= names
    lib = ctypes.CDLL(ts.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(ts.EXPORTS)


def test_status_strings(ts):
    seen = set()
    for code in range(8):
        s = ts.status_string(code)
        assert s and s != "unknown status"
        seen.add(s)
    assert len(seen) == 8
    assert ts.status_string(99) == "unknown status"


@pytest.mark.parametrize("args,code", [
    ((0, 64, 64, "bf16", "bf16"), 1),
    ((64, -1, 64, "bf16", "bf16"), 1),
    ((64, 64, 0, "bf16", "bf16"), 1),
    ((64, 64, 64, "f16", "bf16"), 2),
    ((64, 64, 64, "bf16", "f16"), 2),
    ((64, 64, 64, "f32", "f32"), 2),
    ((64, 64, 12, "bf16", "bf16"), 3),   # A row = 24 bytes
    ((64, 12, 64, "bf16", "f32"), 3),    # B row = 24 bytes
    ((64, 64, 2 ** 31, "bf16", "bf16"), 2),
])
def test_choose_config_validation(ts, args, code):
    with pytest.raises(ts.TsgemmError) as e:
        ts.choose_config(*args, num_sms=152)
    assert e.value.status == code


def test_choose_config_rejects_bad_forced_values(ts):
    for force, code in [({"block_n": 96}, 2), ({"block_n": 320}, 2), ({"block_m": 64}, 2),
                        ({"block_m": 256, "block_n": 192}, 2), ({"block_m": 256, "block_n": 64}, 2),
                        ({"splits": 100}, 2), ({"stages": 1}, 2), ({"stages": 40}, 2),
                        ({"splits": -1}, 1), ({"units": 5}, 1), ({"split_tiles": 3}, 1),
                        ({"splits": 2, "split_tiles": 5}, 2)]:
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(128, 128, 1024, "bf16", "bf16", 152, **force)
        assert e.value.status == code, force


def test_bad_layout_and_null_output(ts):
    cfg = ts.Config()
    f = ts.Config()
    for layout in (0, 1, 2, 3):
        assert ts.lib.tsgemm_choose_config(64, 64, 64, 1, 1, layout, 152, ctypes.byref(f), ctypes.byref(cfg)) == 0
    assert ts.lib.tsgemm_choose_config(64, 64, 64, 1, 1, 4, 152, ctypes.byref(f), ctypes.byref(cfg)) == 1
    assert ts.lib.tsgemm_choose_config(64, 64, 64, 1, 1, -1, 152, ctypes.byref(f), ctypes.byref(cfg)) == 1
    assert ts.lib.tsgemm_choose_config(64, 64, 64, 1, 1, 0, 152, ctypes.byref(f), None) == 1
    assert ts.lib.tsgemm_choose_config(64, 64, 64, 1, 1, 0, 0, ctypes.byref(f), ctypes.byref(cfg)) == 1


def _ceil(a, b):
    return (a + b - 1) // b


@pytest.mark.parametrize("shape", [
    (256, 256, 256, "f16", "f32"), (4096, 4096, 4096, "bf16", "bf16"),
    (128, 28672, 8192, "bf16", "bf16"), (16384, 16384, 8192, "bf16", "bf16"),
    (1024, 1024, 65536, "bf16", "f32"), (129, 264, 72, "f16", "f16"), (1, 8, 8, "bf16", "bf16")])
@pytest.mark.parametrize("sms", [148, 152])
def test_planner_invariants(ts, shape, sms):
    M, N, K, din, dout = shape
    c = ts.choose_config(M, N, K, din, dout, sms)
    bm, bn = c["block_m"], c["block_n"]
    tiles = _ceil(M, bm) * _ceil(N, bn)
    assert (bm, bn) in [(128, 64), (128, 128), (128, 192), (128, 256), (256, 128), (256, 256), (256, 512)]
    st = c["split_tiles"]
    sk = c["stream_k_tiles"]
    per = bm // 128  # CTAs per unit
    assert 0 <= st <= tiles and (st == 0) == (c["splits"] == 1)
    assert 1 <= c["splits"] <= _ceil(K, 64)
    if sk:
        # stream-K: every slot takes a share of the last sk tiles' K slices
        assert c["splits"] == 1 and st == 0 and 0 < sk <= tiles
        assert c["units"] >= tiles and c["grid"] == per * (sms // per)
        # a contributor slot and an owner slot per CTA
        assert c["workspace_bytes"] == 2 * (sms // per) * bm * bn * 4
    else:
        assert c["units"] == (tiles - st) + st * c["splits"]
        assert c["grid"] % per == 0 and 1 <= c["grid"] <= per * min(sms // per, c["units"])
        assert c["workspace_bytes"] == st * c["splits"] * bm * bn * 4
    stage = 128 * 64 * 2 + (bn // per) * 64 * 2
    staging = 0 if dout == "f32" else 8 * 2 * 32 * 32 * 2  # 8 epilogue warps x 2 blocks (16-bit outputs)
    smem = 1024 + c["stages"] * stage + staging + 8 * (2 * c["stages"] + 5) + 16
    assert smem <= 232448
    # the ring is as deep as the shared memory allows
    assert smem + stage > 232448 or c["stages"] == 16
    assert c["timeout_ms"] == 1000


def test_wide_pair_tiles_rule(ts):
    # 256 x 512 pair tiles: chosen with at least four whole rounds and a last
    # round at least two thirds full, never split, never stream-K
    for M, N, K, din, lay in [(8192, 8192, 8192, "bf16", "rrr"), (16384, 16384, 8192, "bf16", "rrr"),
                              (16384, 16384, 8192, "e4m3", "rcr"), (16384, 16384, 8192, "bf16", "rcr")]:
        c = ts.choose_config(M, N, K, din, "bf16", 152, layout=lay)
        assert (c["block_m"], c["block_n"]) == (256, 512), (M, N, K, din, lay)
        assert c["splits"] == 1 and c["stream_k_tiles"] == 0 and c["workspace_bytes"] == 0
        assert c["stages"] == 4 and c["grid"] == 152 and c["units"] == _ceil(M, 256) * _ceil(N, 512)
    # too few rounds, a thin last round, the K x M layouts, forced fields
    for M, N, K, lay, force in [(4096, 4096, 4096, "rrr", {}), (8192, 8704, 8192, "rrr", {}),
                                (8192, 8192, 8192, "crr", {}), (8192, 8192, 8192, "rrr", dict(stages=6)),
                                (8192, 8192, 8192, "rrr", dict(stream_k_tiles=36)),
                                (8192, 8192, 8192, "rrr", dict(block_n=256))]:
        c = ts.choose_config(M, N, K, "bf16", "bf16", 152, layout=lay, **force)
        assert c["block_n"] != 512, (M, N, K, lay, force)
    # forced: whole tiles or stream-K, pairs only, no split
    c = ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152, block_m=256, block_n=512)
    assert c["block_n"] == 512 and c["stream_k_tiles"] == 0 and c["units"] == 128
    c = ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152, block_m=256, block_n=512, stream_k_tiles=52)
    assert c["stream_k_tiles"] == 52 and c["workspace_bytes"] == 2 * 76 * 256 * 512 * 4
    for force in [dict(block_m=128, block_n=512), dict(block_m=256, block_n=512, splits=2),
                  dict(block_n=512)]:
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152, **force)
        assert e.value.status == 2, force


def test_planner_choices_for_the_workloads(ts):
    # The skinny weight-streaming shape fills the GPU with one wave of
    # 128 x 192 tiles and no split; the long-K shape is split.
    c = ts.choose_config(128, 28672, 8192, "bf16", "bf16", 152)
    assert c["block_m"] == 128 and c["block_n"] == 192 and c["splits"] == 1 and c["grid"] == 150
    # the large square shapes use CTA pairs
    c = ts.choose_config(16384, 16384, 8192, "bf16", "bf16", 152)
    assert c["block_m"] == 256 and c["grid"] == 152
    c = ts.choose_config(1024, 1024, 65536, "bf16", "f32", 152)
    assert c["splits"] > 1
    # 4096^3 bf16: CTA pairs on 256 x 256 tiles, stream-K over the tiles
    # past two whole rounds (256 - 2 x 76 = 104), run between those rounds
    c = ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152)
    assert (c["block_m"], c["block_n"], c["splits"], c["stream_k_tiles"]) == (256, 256, 1, 104)
    # 4096^3 E4M3: a tile's mainloop is half as long, too short to hide the
    # stream-K add, so no split (measured faster)
    c = ts.choose_config(4096, 4096, 4096, "e4m3", "bf16", 152, layout="rcr")
    assert (c["block_m"], c["block_n"], c["splits"], c["stream_k_tiles"]) == (256, 256, 1, 0)


def test_forced_fields_are_honoured(ts):
    c = ts.choose_config(1000, 1000, 4096, "bf16", "bf16", 152, block_m=128, block_n=128, splits=5,
                         stages=3, group_m=4, grid=7, timeout_ms=50)
    assert (c["block_m"], c["block_n"], c["splits"], c["stages"], c["group_m"], c["grid"],
            c["timeout_ms"]) == (128, 128, 5, 3, 4, 7, 50)
    c = ts.choose_config(1000, 1000, 4096, "bf16", "bf16", 152, block_m=256, grid=7)
    assert c["block_m"] == 256 and c["grid"] == 6  # whole pairs only


def test_split_factor_may_exceed_the_grid(ts):
    # the S parts of a split tile never wait for one another, so S may be
    # larger than the grid's CTAs (pairs): the parts then run in turn
    c = ts.choose_config(512, 512, 4096, "bf16", "f32", 152, block_m=128, splits=4, grid=4)
    assert c["grid"] == 4
    for force, grid in [(dict(block_m=128, splits=4, grid=3), 3), (dict(block_m=256, splits=3, grid=4), 4),
                        (dict(block_m=128, splits=16, grid=2), 2)]:
        c = ts.choose_config(512, 512, 4096, "bf16", "f32", 152, **force)
        assert c["grid"] == grid and c["splits"] == force["splits"]
    # unforced plans still keep the parts of a tile within one round
    for sms in (2, 8, 152):
        for shape in [(1024, 1024, 65536), (4096, 4096, 4096), (128, 256, 65536)]:
            c = ts.choose_config(*shape, "bf16", "f32", sms)
            assert c["splits"] <= c["grid"] // (c["block_m"] // 128)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_plan_without_a_gpu_fails_cleanly(ts):
    with pytest.raises(ts.TsgemmError) as e:
        ts.Plan(128, 128, 128, "bf16", "bf16")
    assert e.value.status == ts.ERR_CUDA


def test_run_and_status_reject_null_plan(ts):
    assert ts.lib.tsgemm_run(None, 16, 16, 16, None) == ts.ERR_INVALID_ARG
    assert ts.lib.tsgemm_status(None) == ts.ERR_INVALID_ARG
    assert ts.lib.tsgemm_get_config(None, None) == ts.ERR_INVALID_ARG
    assert ts.lib.tsgemm_destroy(None) == ts.OK
    h = ctypes.c_void_p(1)
    assert ts.lib.tsgemm_plan(ctypes.byref(h), 0, 8, 8, 1, 1, 0) == ts.ERR_INVALID_ARG
    assert h.value is None  # *out is cleared on failure
    assert ts.lib.tsgemm_plan(None, 8, 8, 8, 1, 1, 0) == ts.ERR_INVALID_ARG


@pytest.mark.parametrize("layout,shape,code", [
    ("rrr", (12, 64, 64), 0),   # M is free when A is stored M x K
    ("crr", (12, 64, 64), 3),   # A stored K x M: a row of 12 bf16 is 24 bytes
    ("crr", (16, 64, 64), 0),
    ("rcr", (64, 12, 64), 3),   # N * 2 = 24: C rows misaligned in any layout
    ("rcr", (64, 64, 12), 3),   # B stored N x K: rows of K = 12
    ("ccr", (64, 64, 24), 0),
])
def test_alignment_rules_per_layout(ts, layout, shape, code):
    M, N, K = shape
    if code == 0:
        ts.choose_config(M, N, K, "bf16", "bf16", 152, layout=layout)
    else:
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(M, N, K, "bf16", "bf16", 152, layout=layout)
        assert e.value.status == ts.ERR_ALIGNMENT


# ------------------------------------------------------- 8-bit inputs --

@pytest.mark.parametrize("din", ["e4m3", "e5m2"])
def test_fp8_takes_the_k_major_layout_only(ts, din):
    for dout in ("f16", "bf16", "f32"):
        cfg = ts.choose_config(512, 512, 1024, din, dout, 152, layout="rcr")
        assert cfg["block_n"] in (64, 128, 192, 256)
    for layout in ("rrr", "crr", "ccr"):
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(512, 512, 1024, din, "bf16", 152, layout=layout)
        assert e.value.status == ts.ERR_UNSUPPORTED
    for dout in ("e4m3", "e5m2"):  # 8-bit formats are inputs only
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(512, 512, 1024, din, dout, 152, layout="rcr")
        assert e.value.status == ts.ERR_UNSUPPORTED


def test_fp8_alignment_is_in_bytes(ts):
    ts.choose_config(64, 64, 16, "e4m3", "f32", 152, layout="rcr")  # rows of 16 bytes
    for shape in [(64, 64, 8), (64, 64, 24)]:
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(*shape, "e4m3", "f32", 152, layout="rcr")
        assert e.value.status == ts.ERR_ALIGNMENT


def test_fp8_slices_are_128_deep(ts):
    # K = 256 is two 128-element slices: at most two K parts
    ts.choose_config(128, 128, 256, "e4m3", "f32", 152, layout="rcr", splits=2)
    with pytest.raises(ts.TsgemmError) as e:
        ts.choose_config(128, 128, 256, "e4m3", "f32", 152, layout="rcr", splits=3)
    assert e.value.status == ts.ERR_UNSUPPORTED
    # the 16-bit path at the same K has four 64-element slices
    ts.choose_config(128, 128, 256, "bf16", "f32", 152, layout="rcr", splits=4)


def test_fp8_dtype_names(ts):
    assert ts.dtype_code("e4m3") == ts.E4M3 == 3
    assert ts.dtype_code(torch.float8_e4m3fn) == ts.E4M3
    assert ts.dtype_code(torch.float8_e5m2) == ts.E5M2 == 4


# ----------------------------------------------- no multicast option --

def test_no_multicast_cluster_option(ts):
    # The CTA pair (2 x 1 cluster) is the only cluster shape of the GEMM:
    # there is no field that selects clusters of several pairs sharing
    # operand tiles by multicast.
    assert "cluster_n" not in ts.Config().as_dict()
    with pytest.raises(TypeError):
        ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152, cluster_n=2)
    cfg = ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152)
    assert cfg["block_m"] == 256 and cfg["grid"] % 2 == 0


def test_library_has_no_multicast_load():
    # No source of the library issues a multicast TMA load (the only
    # .multicast::cluster left is the pair's tcgen05.commit, an mbarrier
    # arrive addressed to both CTAs of the pair).
    import glob
    import os
    import re
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "hierarchical_gemm_gb300", "csrc")
    for path in glob.glob(os.path.join(csrc, "*")):
        with open(path) as f:
            for line in f:
                if "multicast::cluster" in line:
                    assert re.search(r"tcgen05\.commit", line), (path, line)


# ---------------------------------------------------------- stream-K --

def _sk_segments(w, slots, kb):
    segs = 0
    for g in range(slots):
        a, b = g * w // slots, (g + 1) * w // slots
        if b > a:
            segs += (b - 1) // kb - a // kb + 1
    return segs


def test_stream_k_plan(ts):
    c = ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152, block_m=256, block_n=256, stream_k_tiles=104)
    assert c["stream_k_tiles"] == 104 and c["splits"] == 1 and c["split_tiles"] == 0
    assert c["grid"] == 152 and c["workspace_bytes"] == 2 * 76 * 256 * 256 * 4
    assert c["units"] == (256 - 104) + _sk_segments(104 * 64, 76, 64)
    c = ts.choose_config(1000, 1288, 328, "bf16", "f32", 152, block_m=128, block_n=128, stream_k_tiles=30)
    assert c["grid"] == 152 and c["workspace_bytes"] == 2 * 152 * 128 * 128 * 4
    assert c["units"] == (8 * 11 - 30) + _sk_segments(30 * 6, 152, 6)
    for force, code in [(dict(stream_k_tiles=-2), 1), (dict(stream_k_tiles=10, splits=2), 1),
                        (dict(stream_k_tiles=10, splits=2, split_tiles=3), 1)]:
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152, **force)
        assert e.value.status == code, force
    # -1: no stream-K even where the planner would otherwise consider it
    assert ts.choose_config(4096, 4096, 4096, "bf16", "bf16", 152, stream_k_tiles=-1)["stream_k_tiles"] == 0


def test_stream_k_needs_a_slice_per_slot(ts):
    # 5 tiles x 6 K slices < 152 slots: some slots would get no slice
    with pytest.raises(ts.TsgemmError) as e:
        ts.choose_config(1000, 1288, 328, "bf16", "f32", 152, block_m=128, block_n=128, stream_k_tiles=5)
    assert e.value.status == ts.ERR_UNSUPPORTED


def _sk_walk(tiles_sk, kb, G, full=0):
    """The kernel's stream-K schedule, restated: each slot runs its whole
    tiles (g, g + G, ... below `full`) but the last, then the segments of
    its stream-K range, then its last whole tile.  Every K slice of every
    stream-K tile and every whole tile is covered once, contributors are
    their slot's first stream-K segment, each owner's contributors are the
    next m slots and come no later in their slots' order than the owner in
    its own, and the owner segment is the last of its slot's range (the
    slot's last unit only when no whole tile follows)."""
    W = tiles_sk * kb
    cover = [[0] * kb for _ in range(tiles_sk)]
    whole = [0] * full
    owners, contrib = {}, {}
    pos = {}  # (slot, tile) -> index of the unit in the slot's order
    for g in range(G):
        a, b = g * W // G, (g + 1) * W // G
        nsk = (b - 1) // kb - a // kb + 1 if b > a else 0
        ndp = (full - 1 - g) // G + 1 if g < full else 0
        first_dp = max(ndp - 1, 0)
        order = [("dp", d) for d in range(first_dp)] + [("sk", jj) for jj in range(nsk)]
        if ndp > 0:
            order.append(("dp", ndp - 1))
        for j, (kind, i) in enumerate(order):
            last = j == len(order) - 1
            if kind == "dp":
                whole[g + i * G] += 1
                continue
            start = a if i == 0 else (a // kb + i) * kb
            assert start < b
            t = start // kb
            end = min(b, (t + 1) * kb)
            for k in range(start - t * kb, end - t * kb):
                cover[t][k] += 1
            pos[(g, t)] = j
            if start > t * kb:
                assert i == 0
                contrib.setdefault(t, []).append(g)
            elif end < (t + 1) * kb:
                owners[t] = (g, ((t + 1) * kb * G - 1) // W - g)
                assert end == b and i == nsk - 1  # the owner segment ends the range
                assert last == (ndp == 0)
    assert all(c == 1 for row in cover for c in row)
    assert all(c == 1 for c in whole)
    assert set(contrib) == set(owners)
    for t, (g, m) in owners.items():
        assert contrib[t] == list(range(g + 1, g + m + 1))
        assert all(pos[(c, t)] <= pos[(g, t)] for c in contrib[t])


@pytest.mark.parametrize("args", [(16, 64, 76), (104, 16, 76), (64, 32, 152), (30, 6, 152), (20, 16, 36),
                                  (30, 40, 76), (104, 64, 76, 152), (16, 1024, 76), (68, 128, 76, 4028),
                                  (30, 40, 76, 100), (104, 64, 76, 76)])
def test_stream_k_decomposition(args):
    _sk_walk(*args)


# ------------------------------------------------ DSMEM cluster split --

def test_cluster_split_rules(ts):
    c = ts.choose_config(1024, 2048, 8192, "bf16", "bf16", 152, cluster_split=2)
    assert c["cluster_split"] == 2 and c["block_m"] == 128 and c["splits"] == 1
    assert c["units"] == 8 * 8 and c["grid"] == 128 and c["workspace_bytes"] == 0
    stage = 128 * 64 * 2 + c["block_n"] * 64 * 2
    smem = 1024 + c["stages"] * stage + 8 * 2 * 32 * 32 * 2 + (2 * 128 * 32 * 4 + 32) + 8 * (2 * c["stages"] + 7) + 16
    assert smem <= 232448 < smem + stage
    # the planner never proposes it by itself
    assert ts.choose_config(1024, 2048, 8192, "bf16", "bf16", 152)["cluster_split"] == 1
    for force, code in [(dict(cluster_split=2, block_m=256), 1), (dict(cluster_split=2, splits=2), 1),
                        (dict(cluster_split=4, stream_k_tiles=4), 1), (dict(cluster_split=3), 2),
                        (dict(cluster_split=6), 2), (dict(cluster_split=16), 2)]:
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(1024, 2048, 8192, "bf16", "bf16", 152, **force)
        assert e.value.status == code, force
    for args, code in [((1024, 2048, 8192, "bf16", "bf16", 152, "rcr"), 2), ((1024, 2048, 64, "bf16", "bf16", 152, "rrr"), 2),
                       ((1024, 2048, 8192, "e4m3", "bf16", 152, "rcr"), 2)]:
        with pytest.raises(ts.TsgemmError) as e:
            ts.choose_config(*args[:6], layout=args[6], cluster_split=2)
        assert e.value.status == code, args


@pytest.mark.parametrize("cs", [2, 4, 8])
def test_cluster_split_sizes(ts, cs):
    # cs CTAs per cluster, one tile per cluster at a time; every CTA needs a
    # K slice of its own
    c = ts.choose_config(1024, 2048, 8192, "bf16", "f32", 152, cluster_split=cs)
    assert c["cluster_split"] == cs and c["grid"] % cs == 0
    assert c["grid"] == min(64, 152 // cs) * cs
    c = ts.choose_config(128, 256, 64 * cs, "bf16", "f32", 152, cluster_split=cs)
    assert c["grid"] == cs and c["units"] == 1
    with pytest.raises(ts.TsgemmError) as e:
        ts.choose_config(128, 256, 64 * cs - 64, "bf16", "f32", 152, cluster_split=cs)
    assert e.value.status == 2
    with pytest.raises(ts.TsgemmError) as e:
        ts.choose_config(128, 256, 8192, "bf16", "f32", cs - 1, cluster_split=cs)
    assert e.value.status == 2


# ---------------------------------------------------------- attention --

def test_attention_argument_checks(ts):
    # host-side validation runs before any device query
    f = ts.lib.tsattn_forward
    p = 256  # a 16-byte aligned dummy address; nothing is launched
    assert f(0, 1, 1, 1, 128, ts.BF16, 1.0, 0, p, p, p, p, None, None) == ts.ERR_INVALID_ARG
    assert f(1, 1, 1, 1, 128, ts.BF16, 1.0, 0, None, p, p, p, None, None) == ts.ERR_INVALID_ARG
    assert f(1, 1, 1, 1, 64, ts.BF16, 1.0, 0, p, p, p, p + 4096, None, None) == ts.ERR_UNSUPPORTED
    assert f(1, 1, 1, 1, 128, ts.F32, 1.0, 0, p, p, p, p + 4096, None, None) == ts.ERR_UNSUPPORTED
    assert f(1, 1, 1, 1, 128, ts.BF16, float("nan"), 0, p, p, p, p + 4096, None, None) == ts.ERR_INVALID_ARG
    assert f(1, 1, 1, 1, 128, ts.BF16, 1.0, 0, p + 8, p, p, p + 4096, None, None) == ts.ERR_ALIGNMENT
    # O overlapping Q
    assert f(1, 1, 8, 8, 128, ts.BF16, 1.0, 0, p, p + 8192, p + 16384, p + 256, None, None) == ts.ERR_INVALID_ARG


# ------------------------------------------------- attention launch order --

def _causal_order(BH, nq, group):
    """The attention kernel's causal launch order, restated: CTA b takes
    chunk b // (group nq) of `group` (batch, head)s; within it the longest
    query tiles (largest qb) come first, one per (batch, head)."""
    out = []
    for b in range(BH * nq):
        span = group * nq
        chunk = b // span
        gc = min(group, BH - chunk * group)
        idx = b - chunk * span
        out.append((chunk * group + idx % gc, nq - 1 - idx // gc))
    return out


@pytest.mark.parametrize("BH,nq,group", [(1, 1, 1), (6, 2, 6), (128, 16, 32), (129, 16, 32), (33, 3, 7), (5, 16, 5)])
def test_causal_launch_order_covers_every_tile_once(BH, nq, group):
    order = _causal_order(BH, nq, group)
    assert sorted(order) == sorted((bh, qb) for bh in range(BH) for qb in range(nq))
    # within each chunk the query tiles never grow along the launch order
    span = group * nq
    for c0 in range(0, BH * nq, span):
        qbs = [qb for _, qb in order[c0:c0 + span]]
        assert qbs == sorted(qbs, reverse=True)
