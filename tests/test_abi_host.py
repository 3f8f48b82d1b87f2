"""The C-ABI library on the host (no GPU): it builds, loads, exports every
function the public header declares, and rejects bad arguments before
enqueuing anything.  No call here reaches a kernel launch."""
import ctypes

import pytest

from combine_moe_plan_02_gb300 import _abi, build

EINVAL, EALIGN, OK = _abi.MOE_EINVAL, _abi.MOE_EALIGN, _abi.MOE_OK
FAKE = 0x10000        # 16-byte aligned, never dereferenced: validation fails first
MIS = 0x10008         # 8-byte aligned only


@pytest.fixture(scope="module")
def L():
    build.build()
    return _abi.load()


def test_exports_every_header_function(L):
    names = _abi.header_functions()
    assert "moe_plan" in names and "moe_dispatch" in names and "moe_combine" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/moe_plan.h but not exported"
    assert set(names) == set(_abi.SIGNATURES), "binding and header disagree"


def test_version_and_status_strings(L):
    assert L.moe_version() == 2
    for s in (0, 1, 2, 3):
        assert L.moe_status_string(s)
    assert b"unknown" in L.moe_status_string(99)


def test_plan_workspace_size(L):
    assert L.moe_plan_workspace_size(128, 2, 8) == 0            # one tile: no scratch
    assert L.moe_plan_workspace_size(1024, 8, 64) == 0          # 8192 entries: one tile
    assert L.moe_plan_workspace_size(4096, 8, 64) == 0          # one launch, no scratch
    assert L.moe_plan_workspace_size(16384, 8, 64) == 0         # 131072 entries: still one launch
    ws = L.moe_plan_workspace_size(16385, 8, 64)                # beyond: tile histograms
    assert ws > 0 and ws % 256 == 0
    assert L.moe_plan_workspace_size(20000, 0, 64) == 0         # invalid K
    assert L.moe_group_plan_workspace_size(20000, 8, 64, 8) > 0
    assert L.moe_group_plan_workspace_size(128, 8, 64, 8) == 0     # one tile: no scratch
    gws = L.moe_group_plan_workspace_size(4096, 8, 64, 8)          # tiles counted once
    assert gws > 0 and gws % 256 == 0
    assert L.moe_group_plan_workspace_size(4096, 8, 64, 7) == 0  # 7 does not divide 64


@pytest.mark.parametrize("args,want", [
    (dict(S=-1), EINVAL), (dict(K=0), EINVAL), (dict(K=33), EINVAL), (dict(E=0), EINVAL),
    (dict(E=1025), EINVAL), (dict(S=1 << 28, K=8), EINVAL), (dict(cnt=None), EINVAL),
    (dict(tok_map=None), EINVAL), (dict(ws=None, S=20000, K=8), EINVAL),
    (dict(ws_bytes=16, S=20000, K=8), EINVAL),
])
def test_plan_rejects(L, args, want):
    a = dict(idx=FAKE, S=16, K=2, E=8, cnt=FAKE, off=FAKE, src=FAKE, tok_map=FAKE, ninv=FAKE,
             ws=FAKE, ws_bytes=0)
    a.update(args)
    assert L.moe_plan(a["idx"], a["S"], a["K"], a["E"], a["cnt"], a["off"], a["src"],
                      a["tok_map"], a["ninv"], a["ws"], a["ws_bytes"], None) == want


def test_plan_rejects_misaligned_workspace(L):
    assert L.moe_plan(FAKE, 20000, 8, 64, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 16, 1 << 20,
                      None) == EALIGN


def test_group_plan_rejects(L):
    assert L.moe_group_plan(FAKE, FAKE, 16, 2, 8, 3, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0,
                            None) == EINVAL
    assert L.moe_group_plan(FAKE, None, 16, 2, 8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0,
                            None) == EINVAL


def test_dispatch_validation(L):
    d = lambda **k: L.moe_dispatch(k.get("x", FAKE), k.get("S", 4), k.get("H", 64),
                                   k.get("dt", 0), k.get("K", 2), k.get("tm", FAKE),
                                   k.get("px", FAKE), k.get("rows", 8), k.get("xs", None),
                                   k.get("ns", 0), k.get("ps", None), None)
    assert d(S=0) == OK                      # nothing to do, nothing enqueued
    assert d(dt=7) == EINVAL
    assert d(K=0) == EINVAL
    assert d(x=None) == EINVAL
    assert d(rows=0) == EINVAL
    assert d(H=4) == EALIGN                  # 8-byte rows
    assert d(x=MIS) == EALIGN
    assert d(px=MIS) == EALIGN
    assert d(ns=48) == EINVAL                # scales without buffers
    assert d(ns=3, xs=FAKE, ps=FAKE) == EALIGN   # 12-byte scale rows
    dd = lambda **k: L.moe_dispatch_dedup(FAKE, 16, 64, 0, 8, 8, FAKE, FAKE, FAKE,
                                          k.get("gtm", FAKE), k.get("mr", 128),
                                          k.get("gx", FAKE), FAKE, k.get("prows", 128), None)
    assert dd(mr=100) == EINVAL              # max_rows < S*min(K,G)
    assert dd(gtm=None) == EINVAL            # no gtok_map
    assert dd(prows=0) == EINVAL             # no packed rows
    assert dd(gx=MIS) == EALIGN


def test_combine_validation(L):
    c = lambda **k: L.moe_combine(k.get("y", FAKE), k.get("rows", 8), k.get("idt", 0),
                                  k.get("w", FAKE), k.get("tm", FAKE), k.get("S", 4),
                                  k.get("H", 64), k.get("K", 2), k.get("out", FAKE),
                                  k.get("odt", 0), None)
    assert c(S=0) == OK
    assert c(idt=2) == EINVAL                # fp8 is a transport type, not a combine input
    assert c(odt=5) == EINVAL
    assert c(w=None) == EINVAL
    assert c(rows=0) == EINVAL
    assert c(rows=1 << 31) == EINVAL
    assert c(H=12) == EALIGN
    assert c(out=MIS) == EALIGN
    cd = lambda **k: L.moe_combine_dedup(FAKE, k.get("rows", 128), 1, FAKE, FAKE, 8, FAKE,
                                         FAKE, FAKE, 16, 64, 8, k.get("mr", 128), FAKE, FAKE,
                                         1, None)
    assert cd(mr=127) == EINVAL              # max_rows < S*min(K,G)
    assert cd(rows=0) == EINVAL              # no expert rows
    assert cd(rows=1 << 31) == EINVAL


def test_combine_fold_validation(L):
    c = lambda **k: L.moe_combine_fold(k.get("y", FAKE), k.get("rows", 8), k.get("idt", 0),
                                       k.get("w", FAKE), k.get("wt", 0), k.get("tm", FAKE),
                                       k.get("S", 4), k.get("H", 64), k.get("K", 2),
                                       k.get("out", FAKE), k.get("odt", 0), k.get("ow", FAKE),
                                       None)
    assert c(S=0) == OK
    assert c(wt=2) == EINVAL                 # weighted is 0 or 1
    assert c(w=None) == EINVAL               # the fold needs the weights
    assert c(w=None, wt=1, ow=None) == EINVAL
    assert c(idt=2) == EINVAL
    assert c(K=33) == EINVAL
    assert c(tm=None) == EINVAL
    assert c(ow=FAKE + 2) == EALIGN
    assert c(H=12) == EALIGN
    assert c(y=MIS) == EALIGN


def test_plan_dispatch_validation(L):
    f = lambda **k: L.moe_plan_dispatch(k.get("idx", FAKE), k.get("x", FAKE), k.get("S", 16),
                                        k.get("H", 64), k.get("dt", 0), k.get("K", 2),
                                        k.get("E", 8), k.get("xs", None), k.get("ns", 0),
                                        FAKE, FAKE, FAKE, FAKE, FAKE, k.get("px", FAKE),
                                        k.get("rows", 32), k.get("ps", None), None, 0, None)
    assert L.moe_plan_dispatch_fused_max() >= 256
    assert f(dt=3) == EINVAL
    assert f(E=0) == EINVAL and f(E=1025) == EINVAL
    assert f(K=33) == EINVAL
    assert f(rows=0) == EINVAL
    assert f(ns=4) == EINVAL                  # scales without buffers
    assert f(ns=257, xs=FAKE, ps=FAKE) == EINVAL
    assert f(ns=3, xs=FAKE, ps=FAKE) == EALIGN
    assert f(H=12) == EALIGN
    assert f(x=MIS) == EALIGN
    assert f(px=MIS) == EALIGN
    # above the crossover the plan needs its workspace (none given here)
    assert f(S=200000, K=8, E=64, rows=1600000) == EINVAL


def test_selftest_wait_limits(L):
    assert L.moe_selftest_wait_timeout(999, None) == EINVAL
    assert L.moe_selftest_wait_timeout(100_000_001, None) == EINVAL


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _abi.load()


def test_device_errors_rejects_null(L):
    assert L.moe_device_errors(None) == EINVAL
    _ = ctypes  # noqa


def test_quant_dispatch_validation(L):
    q = lambda **k: L.moe_dispatch_quant_fp8(k.get("x", FAKE), k.get("S", 4), k.get("H", 256),
                                             k.get("K", 2), k.get("tm", FAKE), k.get("block", 128),
                                             k.get("q", FAKE), k.get("sc", FAKE),
                                             k.get("rows", 8), None)
    assert q(S=0) == OK
    assert q(block=100) == EINVAL
    assert q(block=512) == EINVAL
    assert q(H=192) == EINVAL                 # not a multiple of the block
    assert q(K=0) == EINVAL
    assert q(tm=None) == EINVAL
    assert q(rows=0) == EINVAL
    assert q(x=MIS) == EALIGN
    assert q(q=MIS) == EALIGN
    assert q(sc=FAKE + 2) == EALIGN


def test_capacity_plan_validation(L):
    c = lambda **k: L.moe_plan_capacity(FAKE, k.get("S", 16), 2, k.get("E", 8), k.get("cap", 4),
                                        FAKE, FAKE, FAKE, FAKE, FAKE, k.get("nd", FAKE), None, 0,
                                        None)
    assert c(cap=0) == EINVAL
    assert c(cap=1 << 30, E=8) == EINVAL      # E * capacity >= 2^31
    assert c(nd=None) == EINVAL
    assert c(S=-1) == EINVAL


def test_selftest_convert_rejects_bad_ranges(L):
    f = L.moe_selftest_convert
    assert f(1, 4, FAKE, None, None) == EINVAL             # first not a multiple of 4
    assert f(0, 6, FAKE, None, None) == EINVAL             # count not a multiple of 4
    assert f(0, -4, FAKE, None, None) == EINVAL
    assert f(0xfffffffc, 8, FAKE, None, None) == EINVAL    # past 2^32
    assert f(0, 4, None, None, None) == EINVAL             # no output
    assert f(0, 4, MIS, None, None) == EALIGN
    assert f(0, 4, None, MIS, None) == EALIGN
    assert f(0, 0, FAKE, FAKE, None) == OK                 # nothing to do, nothing enqueued
