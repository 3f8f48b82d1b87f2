"""Seeded synthetic inputs for single-GPU MoE token dispatch and combine.

This module is shared by the parity tests, the CPU oracle's callers and the
benchmark.  It holds no arithmetic of the dispatch/combine method itself:
it only draws routing decisions, gate weights, activations and per-expert
scales, and rounds them to the transport dtype with library casts.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used in counter mode, so every value is a
pure function of (seed, stream, index) and the inputs are identical on any
host.  Normal variates use the Box-Muller transform.

Workload shapes follow the pages' measured settings:
  * "MoonEP: Drop cooperative launch from the CTA-independent local kernels"
    (S=4096 tokens, K=8, H=7168: the measured-impact table);
  * "mori #448: cco + flydsl dispatch/combine" (EP8, hidden 7168, top-k 8;
    blockwise fp8 with one f32 scale per 128 elements);
  * "mori #625: EPv2 internode dispatch/combine" (hidden 6144, top-k 8,
    4..32 tokens; the small-token latency tables).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one independent counter stream per drawn quantity.
STREAM_ROUTING = 1
STREAM_LOGITS = 2
STREAM_X = 3
STREAM_EXPERT_SCALE = 4
STREAM_PERMUTATION = 5


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n raw 64-bit outputs of stream `stream` of generator `seed`, starting
    at counter `offset`."""
    with np.errstate(over="ignore"):
        key = _mix64(np.array([(seed * 0x632BE59BD9B4E019 + stream * 0x8CB92BA72F3D8DD7)
                               & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix64(key + ctr * _GAMMA)


def uniform01(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    z = splitmix64(seed, stream, n, offset)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """N(0,1) doubles by Box-Muller over pairs of uniforms."""
    m = (n + 1) // 2
    z = splitmix64(seed, stream, 2 * m)
    u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
    u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:n]


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def topk_uniform(seed: int, S: int, E: int, K: int) -> np.ndarray:
    """Per token, K distinct experts drawn uniformly without replacement, in
    draw order.  The first K entries of a uniformly random permutation of the
    E experts (random keys, argsort) have exactly this law."""
    if S == 0:
        return np.zeros((0, K), dtype=np.int32)
    keys = uniform01(seed, STREAM_ROUTING, S * E).reshape(S, E)
    order = np.argsort(keys, axis=1, kind="stable")
    return order[:, :K].astype(np.int32)


def topk_zipf(seed: int, S: int, E: int, K: int, alpha: float) -> np.ndarray:
    """Per token, K distinct experts drawn one after another without
    replacement, each draw proportional to (rank+1)^-alpha over the experts
    not yet drawn; ranks are assigned through a seeded permutation of the E
    experts.  Successive weighted sampling equals ordering the exponential
    race keys -log(U_e)/p_e ascending (Efraimidis and Spirakis, 2006)."""
    if S == 0:
        return np.zeros((0, K), dtype=np.int32)
    perm = np.argsort(uniform01(seed, STREAM_PERMUTATION, E), kind="stable")
    p = (np.arange(E, dtype=np.float64) + 1.0) ** (-alpha)
    p_expert = np.empty(E, dtype=np.float64)
    p_expert[perm] = p  # expert perm[i] has rank i
    u = uniform01(seed, STREAM_ROUTING, S * E).reshape(S, E)
    keys = -np.log1p(-u) / p_expert[None, :]
    order = np.argsort(keys, axis=1, kind="stable")
    return order[:, :K].astype(np.int32)


def softmax_weights(seed: int, S: int, K: int) -> np.ndarray:
    """Gate weights: softmax over the K selected entries of N(0,1) logits,
    computed in f64 and stored as f32."""
    if S == 0:
        return np.zeros((0, K), dtype=np.float32)
    logits = normal(seed, STREAM_LOGITS, S * K).reshape(S, K)
    ex = np.exp(logits - logits.max(axis=1, keepdims=True))
    return (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)


# ---------------------------------------------------------------------------
# activations
# ---------------------------------------------------------------------------

def activations_f32(seed: int, S: int, H: int) -> np.ndarray:
    return normal(seed, STREAM_X, S * H).astype(np.float32).reshape(S, H)


def to_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """Round to bf16 with torch's CPU cast (round to nearest even) and return
    the raw 16-bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


E4M3_MAX = 448.0


def fp8_blockwise_quantize(x_f32: np.ndarray, block: int):
    """Input preparation for the fp8 workload: per `block`-element block,
    scale = amax/448 (1 when the block is all zero) and code = e4m3(v/scale)
    saturated to the finite range, cast with torch's CPU float8_e4m3fn
    conversion.  Returns (codes uint8 [S,H], scales f32 [S, H/block])."""
    import torch
    S, H = x_f32.shape
    assert H % block == 0
    xb = x_f32.reshape(S, H // block, block).astype(np.float32)
    amax = np.abs(xb).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    v = np.clip(xb / scale[:, :, None], -E4M3_MAX, E4M3_MAX).astype(np.float32)
    q = torch.from_numpy(np.ascontiguousarray(v.reshape(S, H))).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), scale


# ---------------------------------------------------------------------------
# configurations
# ---------------------------------------------------------------------------

DT_BF16 = "bf16"
DT_F32 = "f32"
DT_FP8 = "fp8_e4m3"


@dataclass
class Workload:
    """One seeded input batch.

    x: the token rows as raw element bits (uint16 for bf16, float32 for f32,
    uint8 codes for fp8), shape [S, H].  x_scales: f32 [S, H/128] for fp8,
    else None.  topk_idx int32 [S, K], topk_w f32 [S, K].  expert_scale f32
    [E]: the per-expert factor c_e of the synthetic expert stage (all ones
    for identity experts).  group_size: experts per virtual group for the
    dedup path (0 = direct path).
    """
    name: str
    S: int
    H: int
    E: int
    K: int
    dtype: str
    out_dtype: str
    topk_idx: np.ndarray
    topk_w: np.ndarray
    x: np.ndarray
    expert_scale: np.ndarray
    x_scales: Optional[np.ndarray] = None
    scale_block: int = 0
    group_size: int = 0
    meta: Dict[str, object] = field(default_factory=dict)

    @property
    def elem_bytes(self) -> int:
        return {DT_BF16: 2, DT_F32: 4, DT_FP8: 1}[self.dtype]

    @property
    def row_bytes(self) -> int:
        return self.H * self.elem_bytes


def _expert_scale(seed: int, E: int, identity: bool) -> np.ndarray:
    if identity:
        return np.ones(E, dtype=np.float32)
    return (0.5 + uniform01(seed, STREAM_EXPERT_SCALE, E)).astype(np.float32)


def make(name: str, seed: int = 0, S: Optional[int] = None, H: Optional[int] = None,
         E: Optional[int] = None, K: Optional[int] = None) -> Workload:
    """Build a named workload; S/H/E/K override the named shape (used for
    small and ragged parity cases with the same recipe).

    Names:
      tiny      S=128 H=256 E=8 K=2 bf16, uniform routing, identity experts
      moonep    S=4096 H=7168 E=64 K=8 bf16, uniform, c_e ~ U(0.5, 1.5)
      zipf      S=8192 H=7168 E=256 K=8 bf16, Zipf(1.2) routing, identity
      dedup     S=4096 H=4096 E=64 (8 groups of 8) K=8 f32, uniform, identity
      fp8small  S=128 H=6144 E=256 K=8, fp8 e4m3 rows + f32 scales per 128
                elements, bf16 combine output, uniform, identity
    """
    shapes = {
        "tiny": (128, 256, 8, 2),
        "moonep": (4096, 7168, 64, 8),
        "zipf": (8192, 7168, 256, 8),
        "dedup": (4096, 4096, 64, 8),
        "fp8small": (128, 6144, 256, 8),
    }
    if name not in shapes:
        raise ValueError(f"unknown workload {name!r}")
    s0, h0, e0, k0 = shapes[name]
    S = s0 if S is None else S
    H = h0 if H is None else H
    E = e0 if E is None else E
    K = k0 if K is None else K

    if name == "zipf":
        idx = topk_zipf(seed, S, E, K, 1.2)
    else:
        idx = topk_uniform(seed, S, E, K)
    w = softmax_weights(seed, S, K)
    xf = activations_f32(seed, S, H)
    common = dict(name=name, S=S, H=H, E=E, K=K, topk_idx=idx, topk_w=w)
    if name in ("tiny", "moonep", "zipf"):
        return Workload(dtype=DT_BF16, out_dtype=DT_BF16, x=to_bf16_bits(xf),
                        expert_scale=_expert_scale(seed, E, identity=(name != "moonep")),
                        **common)
    if name == "dedup":
        return Workload(dtype=DT_F32, out_dtype=DT_F32, x=xf,
                        expert_scale=_expert_scale(seed, E, identity=True),
                        group_size=8, meta={"groups": E // 8}, **common)
    # fp8small
    q, sc = fp8_blockwise_quantize(xf, 128) if S > 0 else (
        np.zeros((0, H), np.uint8), np.zeros((0, H // 128), np.float32))
    return Workload(dtype=DT_FP8, out_dtype=DT_BF16, x=q, x_scales=sc, scale_block=128,
                    expert_scale=_expert_scale(seed, E, identity=True), **common)


FP8_SWEEP_TOKENS = (4, 8, 16, 32, 128, 1024)
