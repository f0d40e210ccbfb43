"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every entry point the header declares, and validates arguments exactly as
documented, without launching anything (gg_heap_wrap + the *_check entry
points touch no device state)."""
import ctypes
import json
import os
import re

import pytest
import torch

import gemm_gather_gb300 as gg
from gemm_gather_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_gather.h")
BASE = 1 << 36          # fake device addresses: nothing is dereferenced
TABLE = 1 << 40
PART = 1 << 24


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:gg_status|const char \*|uint64_t|int)\s*\*?\s*(gg_\w+)\s*\(",
                                 text, flags=re.M)))


BUILDS = {"libgemm_gather.so": 0, "libgemm_gather_checked.so": 1}


@pytest.mark.parametrize("name", sorted(BUILDS))
def test_every_declared_symbol_is_exported(name):
    """Both builds (release and checked) export every declared call, and
    gg_checked_build tells them apart (a host-only call)."""
    names = declared_functions()
    assert len(names) >= 14
    lib = ctypes.CDLL(os.path.join(os.path.dirname(_lib.LIB_PATH), name))
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.EXPORTS) == names
    lib.gg_checked_build.restype = ctypes.c_int
    assert lib.gg_checked_build() == BUILDS[name]
    lib.gg_version.restype = ctypes.c_int
    assert lib.gg_version() == gg.lib.gg_version()


def test_loaded_build_follows_the_environment():
    assert gg.checked_build() == (os.environ.get("GEMM_GATHER_CHECKED", "0") == "1")


@pytest.fixture
def heap():
    return gg.heap_wrap(BASE, PART, 8, TABLE)


def test_heap_wrap_table(heap):
    assert gg.heap_info(heap) == (8, PART)
    assert gg.heap_bases(heap) == [BASE + h * PART for h in range(8)]


@pytest.mark.parametrize("args,status", [
    ((BASE + 8, PART, 4, TABLE), _lib.GG_ERR_ALIGNMENT),
    ((BASE, PART + 8, 4, TABLE), _lib.GG_ERR_INVALID_ARG),
    ((BASE, 0, 4, TABLE), _lib.GG_ERR_INVALID_ARG),
    ((BASE, PART, 0, TABLE), _lib.GG_ERR_INVALID_ARG),
    ((BASE, PART, 2000, TABLE), _lib.GG_ERR_INVALID_ARG),
    ((0, PART, 4, TABLE), _lib.GG_ERR_INVALID_ARG),
    ((BASE, PART, 4, TABLE + 4), _lib.GG_ERR_ALIGNMENT),
])
def test_heap_wrap_rejects(args, status):
    with pytest.raises(gg.GGError) as e:
        gg.heap_wrap(*args)
    assert e.value.status == status


def test_heap_workspace_accepts_and_clears(heap):
    slot = _lib.GG_WORKSPACE_SLOT_BYTES
    gg.heap_set_workspace(heap, BASE + (1 << 30), 64 * slot)
    gg.heap_set_workspace(heap, BASE + (1 << 30), slot)
    gg.heap_set_workspace(heap, None, 0)          # removed: fixed shares again
    assert ag(heap) == "tma"                      # validation is unaffected


@pytest.mark.parametrize("ptr,nbytes,status", [
    (BASE + 128, 512, _lib.GG_ERR_ALIGNMENT),     # not 256-byte aligned
    (BASE, 500, _lib.GG_ERR_INVALID_ARG),         # not whole slots
    (BASE, 0, _lib.GG_ERR_INVALID_ARG),           # pointer without a size
    (None, 512, _lib.GG_ERR_INVALID_ARG),         # size without a pointer
    (BASE, 512 * ((1 << 20) + 1), _lib.GG_ERR_INVALID_ARG),  # too many slots
])
def test_heap_workspace_rejects(heap, ptr, nbytes, status):
    with pytest.raises(gg.GGError) as e:
        gg.heap_set_workspace(heap, ptr, nbytes)
    assert e.value.status == status


def test_claim_policy_round_trip():
    assert gg.get_claim_policy() == "auto"
    for p in ("always", "never", "auto"):
        gg.set_claim_policy(p)
        assert gg.get_claim_policy() == p
    for bad in (-1, 3):
        assert _lib.lib.gg_set_claim_policy(bad) == _lib.GG_ERR_INVALID_ARG
    assert gg.get_claim_policy() == "auto"


def test_heap_workspace_needs_a_heap():
    assert _lib.lib.gg_heap_set_workspace(None, BASE, 512) == _lib.GG_ERR_INVALID_ARG


def ag(heap, **kw):
    a = dict(rank=-1, input=BASE + 4096, ld_in=256, output=BASE + (1 << 20), ld_out=256, M=64,
             N=256, dtype=torch.float16, tile=(8, 256), comm_programs=4, group=(0, 1, 2),
             path="auto")
    a.update(kw)
    return gg.all_gather_check(heap, a["rank"], a["input"], a["ld_in"], a["output"], a["ld_out"],
                               a["M"], a["N"], a["dtype"], a["tile"], a["comm_programs"],
                               a["group"], a["path"])


def test_gather_valid_calls(heap):
    assert ag(heap) == "tma"
    assert ag(heap, rank=1) == "tma"
    assert ag(heap, path="bulk") == "bulk"
    assert ag(heap, path="tma") == "tma"
    assert ag(heap, M=0) == "none"
    assert ag(heap, N=0) == "none"
    assert ag(heap, input=BASE + 4098) == "vector"
    assert ag(heap, path="vector") == "vector"
    assert ag(heap, group=(1, 2, 4), rank=5) == "tma"
    # a ragged N with 16-byte pitches still takes tensor maps (boxes clip); bulk
    # copies need whole 16-byte rows
    assert ag(heap, N=255, ld_in=256, ld_out=256) == "tma"
    assert ag(heap, N=255, ld_in=256, ld_out=256, path="auto", tile=(8, 264)) == "vector"
    # block_n above 256 elements is beyond a tensor-map box: bulk copies instead
    assert ag(heap, tile=(4, 512), N=1024, ld_in=1024, ld_out=1024,
              output=BASE + (4 << 20)) == "bulk"
    # an explicit 32x64 tile is accepted as given (never remapped)
    assert ag(heap, tile=(32, 64)) == "tma"


@pytest.mark.parametrize("kw,status", [
    (dict(group=(0, 1, 9)), _lib.GG_ERR_INVALID_ARG),          # member 8 is not a heap
    (dict(group=(0, 0, 2)), _lib.GG_ERR_INVALID_ARG),          # stride 0
    (dict(group=(0, 1, 0)), _lib.GG_ERR_INVALID_ARG),          # empty group
    (dict(group=(-1, 1, 2)), _lib.GG_ERR_INVALID_ARG),
    (dict(group=(0, 1, 65)), _lib.GG_ERR_INVALID_ARG),         # above GG_MAX_WORLD
    (dict(rank=3), _lib.GG_ERR_INVALID_ARG),                   # not a member
    (dict(rank=-2), _lib.GG_ERR_INVALID_ARG),
    (dict(group=(1, 2, 3), rank=2), _lib.GG_ERR_INVALID_ARG),  # between strided members
    (dict(ld_in=100), _lib.GG_ERR_INVALID_ARG),                # pitch below N
    (dict(ld_out=100), _lib.GG_ERR_INVALID_ARG),
    (dict(M=-1), _lib.GG_ERR_INVALID_ARG),
    (dict(tile=(0, 256)), _lib.GG_ERR_UNSUPPORTED),
    (dict(tile=(257, 8)), _lib.GG_ERR_UNSUPPORTED),
    (dict(tile=(64, 512)), _lib.GG_ERR_UNSUPPORTED),           # 64 KB tile
    (dict(comm_programs=0), _lib.GG_ERR_INVALID_ARG),
    (dict(comm_programs=70000), _lib.GG_ERR_INVALID_ARG),
    (dict(output=BASE - 256), _lib.GG_ERR_NOT_IN_HEAP),        # below the heap
    (dict(output=BASE + 8 * PART), _lib.GG_ERR_NOT_IN_HEAP),   # past the end
    (dict(output=BASE + PART - 1024), _lib.GG_ERR_NOT_IN_HEAP),  # overruns the partition
    (dict(input=BASE + 8 * PART + (1 << 20)), _lib.GG_ERR_NOT_IN_HEAP),
    (dict(input=BASE + (1 << 20) + 512), _lib.GG_ERR_INVALID_ARG),  # overlaps the output
    (dict(rank=0, input=BASE + PART + (1 << 20)), _lib.GG_ERR_INVALID_ARG),  # overlaps member 1
    (dict(input=BASE + 4098, path="bulk"), _lib.GG_ERR_ALIGNMENT),
    (dict(input=BASE + 4098, path="tma"), _lib.GG_ERR_ALIGNMENT),
    (dict(tile=(4, 512), N=1024, ld_in=1024, ld_out=1024, output=BASE + (4 << 20),
          path="tma"), _lib.GG_ERR_ALIGNMENT),
    (dict(dtype=7), _lib.GG_ERR_INVALID_ARG),
    (dict(output=0), _lib.GG_ERR_INVALID_ARG),
])
def test_gather_rejects(heap, kw, status):
    with pytest.raises(gg.GGError) as e:
        ag(heap, **kw)
    assert e.value.status == status, str(e.value)
    assert gg.lib.gg_last_error().decode()


def mag(heap, **kw):
    a = dict(rank=-1, A=BASE + 4096, lda=1024, B=TABLE + 4096, ldb=512, output=BASE + (4 << 20),
             ld_out=512, M=256, N=512, K=1024, dtype=torch.float16, tile=gg.FUSED_TILE,
             comm_programs=148, group=(0, 1, 4))
    a.update(kw)
    gg.matmul_all_gather_check(heap, a["rank"], a["A"], a["lda"], a["B"], a["ldb"], a["output"],
                               a["ld_out"], a["M"], a["N"], a["K"], a["dtype"], a["tile"],
                               a["comm_programs"], a["group"])


def plan(heap, path="auto", **kw):
    a = dict(rank=-1, A=BASE + 4096, lda=1024, B=TABLE + 4096, ldb=8192, output=BASE + (4 << 20),
             ld_out=8192, M=64, N=512, K=1024, dtype=torch.float16, tile=gg.FUSED_TILE,
             comm_programs=148, group=(0, 1, 4))
    a.update(kw)
    return gg.matmul_all_gather_plan(heap, a["rank"], a["A"], a["lda"], a["B"], a["ldb"],
                                     a["output"], a["ld_out"], a["M"], a["N"], a["K"], a["dtype"],
                                     a["tile"], a["comm_programs"], a["group"], path)


def test_fused_plan_variants(heap):
    """The tile is the CTA's output tile, never remapped; the path only picks
    one CTA or CTA pairs."""
    assert plan(heap) == "2sm"
    assert plan(heap, comm_programs=1) == "1sm"
    assert plan(heap, path="1sm") == "1sm"
    assert plan(heap, path="2sm") == "2sm"
    assert plan(heap, tile=gg.FUSED_TILE_WIDE) == "2sm"
    assert plan(heap, tile=gg.FUSED_TILE_WIDE, path="2sm", N=256) == "2sm"
    assert plan(heap, M=0) == "none"
    assert plan(heap, K=0) == "none"   # no matmul kernel: the output is filled with zeros


@pytest.mark.parametrize("kw,status", [
    (dict(tile=gg.FUSED_TILE_WIDE, path="1sm"), _lib.GG_ERR_UNSUPPORTED),   # pairs only
    (dict(tile=gg.FUSED_TILE_WIDE, comm_programs=1), _lib.GG_ERR_INVALID_ARG),
    (dict(path="2sm", comm_programs=1), _lib.GG_ERR_INVALID_ARG),
    (dict(tile=(256, 128)), _lib.GG_ERR_UNSUPPORTED),
    (dict(tile=(128, 384)), _lib.GG_ERR_UNSUPPORTED),
])
def test_fused_plan_rejects(heap, kw, status):
    with pytest.raises(gg.GGError) as e:
        plan(heap, **kw)
    assert e.value.status == status, str(e.value)


def test_fused_empty_contraction_validates_the_output_only(heap):
    """K == 0: C_r is the zero matrix; A and B are never read (NULL or unaligned
    is fine), but the output must still be an aligned buffer inside the heap."""
    mag(heap, K=0, A=None, B=None)
    mag(heap, K=0, A=BASE + 4100, lda=3)
    for kw, status in [(dict(output=BASE + (4 << 20) + 8), _lib.GG_ERR_ALIGNMENT),
                       (dict(output=BASE + PART - 4096), _lib.GG_ERR_NOT_IN_HEAP),
                       (dict(N=500, ldb=512, ld_out=512), _lib.GG_ERR_ALIGNMENT),
                       (dict(ld_out=8196), _lib.GG_ERR_ALIGNMENT)]:
        with pytest.raises(gg.GGError) as e:
            mag(heap, K=0, **kw)
        assert e.value.status == status, (kw, str(e.value))


def test_fused_valid_calls(heap):
    mag(heap)
    mag(heap, rank=2, A=TABLE + (1 << 20))
    mag(heap, dtype=torch.bfloat16)
    mag(heap, K=0)
    mag(heap, M=0)
    mag(heap, tile=gg.FUSED_TILE_WIDE)
    with pytest.raises(gg.GGError) as e:           # the wide tile needs CTA pairs
        mag(heap, tile=gg.FUSED_TILE_WIDE, comm_programs=1)
    assert e.value.status == _lib.GG_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,status", [
    (dict(tile=(256, 128)), _lib.GG_ERR_UNSUPPORTED),
    (dict(tile=(32, 64)), _lib.GG_ERR_UNSUPPORTED),    # never remapped to the supported tile
    (dict(tile=(8, 256)), _lib.GG_ERR_UNSUPPORTED),
    (dict(dtype=torch.float32), _lib.GG_ERR_UNSUPPORTED),
    (dict(N=500, ldb=512, ld_out=512), _lib.GG_ERR_ALIGNMENT),
    (dict(lda=1028), _lib.GG_ERR_ALIGNMENT),
    (dict(A=BASE + 4100), _lib.GG_ERR_ALIGNMENT),
    (dict(lda=1000), _lib.GG_ERR_INVALID_ARG),          # below K
    (dict(group=(0, 1, 9)), _lib.GG_ERR_INVALID_ARG),
    (dict(rank=5), _lib.GG_ERR_INVALID_ARG),
    (dict(output=BASE + PART - 4096), _lib.GG_ERR_NOT_IN_HEAP),
    (dict(A=TABLE), _lib.GG_ERR_NOT_IN_HEAP),           # group launch: A must be symmetric
    (dict(A=BASE + (4 << 20) + 4096), _lib.GG_ERR_INVALID_ARG),  # A overlaps the output
    (dict(B=BASE + (4 << 20)), _lib.GG_ERR_INVALID_ARG),         # B overlaps member 0's output
])
def test_fused_rejects(heap, kw, status):
    with pytest.raises(gg.GGError) as e:
        mag(heap, **kw)
    assert e.value.status == status, str(e.value)


def test_wait_limit_roundtrip():
    gg.set_wait_limit_ns(12345)
    assert gg.get_wait_limit_ns() == 12345
    gg.set_wait_limit_ns(0)
    assert gg.get_wait_limit_ns() == 2_000_000_000


def test_page_facts_tile_geometry():
    """The tile geometry the pages print (tests/golden/page_facts.json)."""
    facts = json.load(open(os.path.join(ROOT, "tests", "golden", "page_facts.json")))
    for t in facts["tiles"]:
        es = {"f16": 2}[t["dtype"]]
        assert t["block_m"] * t["block_n"] == t["elements"]
        assert t["block_n"] * es == t["row_bytes"]
    heap = gg.heap_wrap(BASE, PART, 8, TABLE)
    t = facts["explicit_tile_not_remapped"]
    # accepted as the 32x64 tile it is (128-byte rows: a tensor-map box of 32 x 64)
    assert ag(heap, tile=(t["block_m"], t["block_n"])) == "tma"
    s = facts["sweep"]
    assert len(s["M"]) * len(s["N"]) * len(s["dtypes"]) * len(s["comm_sms"]) == s["configurations"]
    p = facts["peers_per_tile"]
    assert p["world_size"] - 1 == p["peer_destinations"]
    r = facts["rotated_order"]
    assert [(r["rank"] + j) % r["world_size"] for j in range(r["world_size"])] == r["order"]


def coll(heap, kind, **kw):
    a = dict(rank=-1, input=BASE + 4096, ld_in=256, output=BASE + (1 << 20), ld_out=256, M=64,
             N=256, dtype=torch.float16, tile=(8, 256), comm_programs=16, group=(0, 1, 4),
             dests_per_wait=0, path="auto")
    a.update(kw)
    return gg.collective_check(kind, heap, a["rank"], a["input"], a["ld_in"], a["output"],
                               a["ld_out"], a["M"], a["N"], a["dtype"], a["tile"],
                               a["comm_programs"], a["group"], a["dests_per_wait"], a["path"])


def test_next_collectives_valid(heap):
    assert coll(heap, "all_gather", dests_per_wait=2) == "tma"
    assert coll(heap, "all_gather", dests_per_wait=2, path="bulk") == "bulk"
    assert coll(heap, "all_gather_partitioned") == "tma"
    assert coll(heap, "all_gather_partitioned", comm_programs=4) == "tma"
    assert coll(heap, "all_gather_partitioned", path="vector") == "vector"
    assert coll(heap, "all_to_all") == "tma"
    assert coll(heap, "all_to_all", input=BASE + 4098) == "vector"
    assert coll(heap, "all_to_all", rank=2, input=TABLE) == "tma"


@pytest.mark.parametrize("kind,kw,status", [
    ("all_gather", dict(dests_per_wait=-1), _lib.GG_ERR_INVALID_ARG),
    ("all_gather_partitioned", dict(comm_programs=3), _lib.GG_ERR_INVALID_ARG),  # < W
    ("all_gather_partitioned", dict(path="bulk"), _lib.GG_ERR_UNSUPPORTED),
    ("all_to_all", dict(path="bulk"), _lib.GG_ERR_UNSUPPORTED),
    # the all-to-all input is W*M rows: 4 x 64 rows of 512 B overlap the output at +1 MB
    ("all_to_all", dict(input=BASE + (1 << 20) - 4 * 64 * 512 + 512), _lib.GG_ERR_INVALID_ARG),
    ("all_to_all", dict(input=BASE + PART - 64 * 512), _lib.GG_ERR_NOT_IN_HEAP),
])
def test_next_collectives_reject(heap, kind, kw, status):
    with pytest.raises(gg.GGError) as e:
        coll(heap, kind, **kw)
    assert e.value.status == status, str(e.value)


def test_binding_stream_argument():
    """The binding passes an explicit stream through as its handle, and the
    legacy default stream (NULL) while torch has not initialised CUDA."""
    import torch
    from gemm_gather_gb300 import _stream
    assert _stream(0x1234) == 0x1234
    assert _stream(0) is None
    if not torch.cuda.is_initialized():
        assert _stream(None) is None


def test_store_policy_round_trip():
    assert gg.get_store_policy() == "evict_first"  # the library's default
    try:
        gg.set_store_policy("plain")
        assert gg.get_store_policy() == "plain"
        with pytest.raises(gg.GGError) as e:
            gg.check(gg.lib.gg_set_store_policy(7))
        assert e.value.status == _lib.GG_ERR_INVALID_ARG
        assert gg.get_store_policy() == "plain"
    finally:
        gg.set_store_policy("evict_first")
