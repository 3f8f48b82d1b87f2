"""CPU oracle for single-GPU MoE dispatch and combine (ctypes wrapper).

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this package.  The product path (the CUDA library
and its Python binding) never imports it, and it never imports them.

The arithmetic lives in ``oracle.c`` (plain C, single-threaded, compiled
with -ffp-contract=off); this module only builds it with gcc and marshals
numpy arrays.  See ``oracle.c`` for the definitions and their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ODT_BF16, ODT_F32, ODT_FP8_E4M3 = 0, 1, 2
_DT = {"bf16": ODT_BF16, "f32": ODT_F32, "fp8_e4m3": ODT_FP8_E4M3}

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fvisibility=hidden"]


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile oracle.c into a shared library with gcc; returns its path."""
    cmd = ["gcc", *CFLAGS, *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


_lib: Optional[ctypes.CDLL] = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            build()
        _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f32.restype = ctypes.c_float
    lib.oracle_plan.argtypes = [P, I64, I32, I32, P, P, P, P, P]
    lib.oracle_plan.restype = I32
    lib.oracle_plan_capacity.argtypes = [P, I64, I32, I32, I64, P, P, P, P, P, P]
    lib.oracle_plan_capacity.restype = I32
    lib.oracle_group_plan.argtypes = [P, P, I64, I32, I32, I32, P, P, P, P, P]
    lib.oracle_group_plan.restype = I32
    lib.oracle_dispatch.argtypes = [P, I64, I64, I32, P, P]
    lib.oracle_dispatch.restype = None
    lib.oracle_dispatch_dedup.argtypes = [P, I64, I64, I32, P, P, P, P]
    lib.oracle_dispatch_dedup.restype = None
    lib.oracle_combine.argtypes = [P, I32, P, P, I64, I64, I32, P, I32]
    lib.oracle_combine.restype = None
    lib.oracle_combine_dedup.argtypes = [P, I32, P, I64, P, P, P, I64, I64, I32, P, P, I32]
    lib.oracle_combine_dedup.restype = None
    lib.oracle_combine_fold.argtypes = [P, I32, P, I32, P, I64, I64, I32, P, I32, P]
    lib.oracle_combine_fold.restype = None
    lib.oracle_expert_scale_bf16.argtypes = [P, P, I32, P, I64, P]
    lib.oracle_expert_scale_bf16.restype = None
    lib.oracle_expert_dequant_fp8.argtypes = [P, P, I64, I64, I32, P]
    lib.oracle_expert_dequant_fp8.restype = None
    lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_quant_fp8.argtypes = [P, I64, I64, I32, P, P]
    lib.oracle_quant_fp8.restype = None
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# Python-level calls (numpy in, numpy out)
# ---------------------------------------------------------------------------

def plan(topk_idx: np.ndarray, E: int, lib=None):
    """Returns dict(cnt i32[E], off i64[E+1], packed_src i32[n_valid],
    tok_map i64[S,K], n_invalid int)."""
    lib = lib or load()
    idx = _c(topk_idx, np.int32)
    S, K = idx.shape
    cnt = np.zeros(E, np.int32)
    off = np.zeros(E + 1, np.int64)
    src = np.full(max(S * K, 1), -7, np.int32)
    tmap = np.zeros((S, K), np.int64)
    ninv = np.zeros(1, np.int32)
    rc = lib.oracle_plan(_p(idx), S, K, E, _p(cnt), _p(off), _p(src), _p(tmap), _p(ninv))
    assert rc == 0
    return dict(cnt=cnt, off=off, packed_src=src[: int(off[E])], tok_map=tmap,
                n_invalid=int(ninv[0]))


def plan_capacity(topk_idx: np.ndarray, E: int, capacity: int, lib=None):
    """Returns dict(cnt, off, packed_src i32[E*capacity] (unwritten rows -7),
    tok_map, n_invalid, n_dropped)."""
    lib = lib or load()
    idx = _c(topk_idx, np.int32)
    S, K = idx.shape
    cnt = np.zeros(E, np.int32)
    off = np.zeros(E + 1, np.int64)
    src = np.full(max(E * capacity, 1), -7, np.int32)
    tmap = np.zeros((S, K), np.int64)
    ninv = np.zeros(1, np.int32)
    ndrop = np.zeros(1, np.int32)
    rc = lib.oracle_plan_capacity(_p(idx), S, K, E, capacity, _p(cnt), _p(off), _p(src),
                                  _p(tmap), _p(ninv), _p(ndrop))
    assert rc == 0
    return dict(cnt=cnt, off=off, packed_src=src[:E * capacity], tok_map=tmap,
                n_invalid=int(ninv[0]), n_dropped=int(ndrop[0]))


def group_plan(topk_idx: np.ndarray, tok_map: np.ndarray, E: int, group_size: int, lib=None):
    """Returns dict(gcnt i32[G], goff i64[G+1], gtok_map i64[S,K],
    grp_src i32[R], grp_tok_map i64[R,K])."""
    lib = lib or load()
    idx = _c(topk_idx, np.int32)
    tm = _c(tok_map, np.int64)
    S, K = idx.shape
    G = E // group_size
    rmax = max(S * min(K, G), 1)
    gcnt = np.zeros(G, np.int32)
    goff = np.zeros(G + 1, np.int64)
    gtm = np.zeros((S, K), np.int64)
    gsrc = np.full(rmax, -7, np.int32)
    gtk = np.full((rmax, K), -7, np.int64)
    rc = lib.oracle_group_plan(_p(idx), _p(tm), S, K, E, group_size, _p(gcnt), _p(goff),
                               _p(gtm), _p(gsrc), _p(gtk))
    assert rc == 0
    R = int(goff[G])
    return dict(gcnt=gcnt, goff=goff, gtok_map=gtm, grp_src=gsrc[:R], grp_tok_map=gtk[:R])


def dispatch(rows: np.ndarray, tok_map: np.ndarray, n_rows_out: int, fill: int = 0xFF, lib=None):
    """rows [S, ...] (any dtype) -> packed [n_rows_out, ...], unwritten rows
    keep the byte `fill`."""
    lib = lib or load()
    rows = np.ascontiguousarray(rows)
    tm = _c(tok_map, np.int64)
    S, K = tm.shape
    row_bytes = rows[0].nbytes if S > 0 else int(np.prod(rows.shape[1:])) * rows.itemsize
    packed = np.empty((n_rows_out,) + rows.shape[1:], rows.dtype)
    packed.view(np.uint8).reshape(-1)[:] = fill
    lib.oracle_dispatch(_p(rows), S, row_bytes, K, _p(tm), _p(packed))
    return packed


def dispatch_dedup(x: np.ndarray, grp_src: np.ndarray, grp_tok_map: np.ndarray, K: int,
                   n_rows_out: int, fill: int = 0xFF, lib=None):
    lib = lib or load()
    x = np.ascontiguousarray(x)
    gs = _c(grp_src, np.int32)
    gtk = _c(grp_tok_map, np.int64)
    R = gs.shape[0]
    row_bytes = int(np.prod(x.shape[1:])) * x.itemsize
    grp_x = np.empty((R,) + x.shape[1:], x.dtype)
    grp_x.view(np.uint8).reshape(-1)[:] = fill
    packed = np.empty((n_rows_out,) + x.shape[1:], x.dtype)
    packed.view(np.uint8).reshape(-1)[:] = fill
    lib.oracle_dispatch_dedup(_p(x), R, row_bytes, K, _p(gs),
                              _p(gtk if R > 0 else np.zeros((1, K), np.int64)),
                              _p(grp_x if R > 0 else np.zeros(1, np.uint8)), _p(packed))
    return grp_x, packed


def _np_dt(dt: str):
    return {"bf16": np.uint16, "f32": np.float32}[dt]


def combine(y: np.ndarray, in_dt: str, topk_w: np.ndarray, tok_map: np.ndarray, H: int,
            out_dt: str, lib=None):
    lib = lib or load()
    y = _c(y, _np_dt(in_dt))
    w = _c(topk_w, np.float32)
    tm = _c(tok_map, np.int64)
    S, K = tm.shape
    out = np.zeros((S, H), _np_dt(out_dt))
    lib.oracle_combine(_p(y) if y.size else None, _DT[in_dt], _p(w), _p(tm), S, H, K, _p(out),
                       _DT[out_dt])
    return out


def combine_dedup(y: np.ndarray, in_dt: str, topk_w: np.ndarray, grp_src: np.ndarray,
                  grp_tok_map: np.ndarray, gtok_map: np.ndarray, H: int, out_dt: str, lib=None):
    lib = lib or load()
    y = _c(y, _np_dt(in_dt))
    w = _c(topk_w, np.float32)
    gs = _c(grp_src, np.int32)
    gtk = _c(grp_tok_map, np.int64)
    gtm = _c(gtok_map, np.int64)
    S, K = gtm.shape
    R = gs.shape[0]
    gtok = np.zeros((max(R, 1), H), np.float32)
    out = np.zeros((S, H), _np_dt(out_dt))
    lib.oracle_combine_dedup(_p(y) if y.size else None, _DT[in_dt], _p(w), R,
                             _p(gs) if R else None, _p(gtk) if R else None, _p(gtm), S, H, K,
                             _p(gtok), _p(out), _DT[out_dt])
    return gtok[:R], out


def combine_fold(y: np.ndarray, in_dt: str, topk_w: np.ndarray, token_map: np.ndarray,
                 H: int, out_dt: str, weighted: bool = False, fold: bool = True, lib=None):
    """Combine over any token map, weighted or not, with the weight fold.
    Returns (out, out_weights or None)."""
    lib = lib or load()
    y = _c(y, _np_dt(in_dt))
    w = _c(topk_w, np.float32)
    tm = _c(token_map, np.int64)
    S, K = tm.shape
    out = np.zeros((S, H), _np_dt(out_dt))
    ow = np.zeros((S, K), np.float32) if fold else None
    lib.oracle_combine_fold(_p(y) if y.size else None, _DT[in_dt], _p(w), int(weighted), _p(tm),
                            S, H, K, _p(out), _DT[out_dt], _p(ow) if fold else None)
    return out, ow


def expert_scale_bf16(packed: np.ndarray, off: np.ndarray, c: np.ndarray, lib=None):
    lib = lib or load()
    packed = _c(packed, np.uint16)
    off = _c(off, np.int64)
    c = _c(c, np.float32)
    H = packed.shape[1]
    y = np.zeros_like(packed)
    lib.oracle_expert_scale_bf16(_p(packed), _p(off), len(c), _p(c), H, _p(y))
    return y


def quant_fp8(x_bf16: np.ndarray, block: int, lib=None):
    """Blockwise E4M3 codes and f32 scales of bf16 rows: (q uint8 [S,H],
    scales f32 [S, H/block])."""
    lib = lib or load()
    x = _c(x_bf16, np.uint16)
    S, H = x.shape
    q = np.zeros((S, H), np.uint8)
    sc = np.zeros((S, H // block), np.float32)
    if S:
        lib.oracle_quant_fp8(_p(x), S, H, block, _p(q), _p(sc))
    return q, sc


def f32_to_e4m3(v: float, lib=None) -> int:
    return int((lib or load()).oracle_f32_to_e4m3(float(v)))


def expert_dequant_fp8(q: np.ndarray, scales: np.ndarray, block: int, lib=None):
    lib = lib or load()
    q = _c(q, np.uint8)
    sc = _c(scales, np.float32)
    R, H = q.shape
    y = np.zeros((R, H), np.uint16)
    lib.oracle_expert_dequant_fp8(_p(q), _p(sc), R, H, block, _p(y))
    return y


def f32_to_bf16(v: float, lib=None) -> int:
    return int((lib or load()).oracle_f32_to_bf16(float(v)))


def bf16_to_f32(h: int, lib=None) -> float:
    return float((lib or load()).oracle_bf16_to_f32(int(h)))


def e4m3_to_f32(q: int, lib=None) -> float:
    return float((lib or load()).oracle_e4m3_to_f32(int(q)))


def run_workload(wl, lib=None):
    """Whole oracle path for one workload: plan, dispatch (and scales),
    the synthetic expert stage, combine.  Returns a dict of every output."""
    lib = lib or load()
    res = {}
    p = plan(wl.topk_idx, wl.E, lib=lib)
    res.update(p)
    V = int(p["off"][wl.E])
    packed = dispatch(wl.x, p["tok_map"], V, lib=lib)
    res["packed_x"] = packed
    if wl.x_scales is not None:
        res["packed_scales"] = dispatch(wl.x_scales, p["tok_map"], V, lib=lib)
    if wl.group_size:
        gp = group_plan(wl.topk_idx, p["tok_map"], wl.E, wl.group_size, lib=lib)
        res.update(gp)
        grp_x, packed_d = dispatch_dedup(wl.x, gp["grp_src"], gp["grp_tok_map"], wl.K, V, lib=lib)
        res["grp_x"] = grp_x
        res["packed_x_dedup"] = packed_d
    # expert stage
    if wl.dtype == "bf16":
        y = expert_scale_bf16(packed, p["off"], wl.expert_scale, lib=lib)
        in_dt = "bf16"
    elif wl.dtype == "f32":
        y = packed * wl.expert_scale[np.searchsorted(p["off"], np.arange(V), side="right") - 1][:, None] \
            if V else packed
        y = np.ascontiguousarray(y, np.float32)
        in_dt = "f32"
    else:
        y = expert_dequant_fp8(packed, res["packed_scales"], wl.scale_block, lib=lib)
        in_dt = "bf16"
    res["y"] = y
    res["out"] = combine(y, in_dt, wl.topk_w, p["tok_map"], wl.H, wl.out_dtype, lib=lib)
    if wl.group_size:
        gtok, out_d = combine_dedup(y, in_dt, wl.topk_w, res["grp_src"], res["grp_tok_map"],
                                    res["gtok_map"], wl.H, wl.out_dtype, lib=lib)
        res["gtok"] = gtok
        res["out_dedup"] = out_d
    return res
