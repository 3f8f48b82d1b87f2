"""Quantising dispatch (bf16 rows -> blockwise E4M3 codes + f32 scales in the
packed rows) against the CPU oracle: codes, scales and untouched rows are
compared bit-exactly.  The divisions and the cast are IEEE f32 and
round-to-nearest-even on both sides, so no tolerance is needed."""
import os

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402


def _run(x_bits: np.ndarray, idx: np.ndarray, E: int, block: int, sc_offset: int = 0):
    import combine_moe_plan_02_gb300 as moe
    S, H = x_bits.shape
    K = idx.shape[1]
    dev = torch.device("cuda")
    x = torch.from_numpy(x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    plan = moe.moe_plan(torch.from_numpy(np.ascontiguousarray(idx)).to(dev), E)
    q = gpu_path.poisoned((max(S * K, 1), H), torch.uint8)
    n_sc = max(S * K, 1) * (H // block)
    # sc_offset floats into a larger buffer: a scale buffer that is only
    # 4-byte aligned takes the register kernel instead of the bulk one
    sc = gpu_path.poisoned((n_sc + sc_offset,), torch.float32)[sc_offset:].view(
        max(S * K, 1), H // block)
    moe.moe_dispatch_quant_fp8(x, plan.tok_map, block=block, packed_q=q, packed_scales=sc)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    return q.cpu().numpy(), sc.cpu().numpy(), int(plan.off[-1].item())


def _check(x_bits, idx, E, block, sc_offset=0):
    q, sc, V = _run(x_bits, idx, E, block, sc_offset)
    p = oracle.plan(idx, E)
    q0, sc0 = oracle.quant_fp8(x_bits, block)
    ref_q = oracle.dispatch(q0, p["tok_map"], V)
    ref_sc = oracle.dispatch(sc0, p["tok_map"], V)
    assert V == int(p["off"][-1])
    assert np.array_equal(q[:V], ref_q)
    assert np.array_equal(sc[:V].view(np.uint32), ref_sc.view(np.uint32))
    assert np.all(q[V:] == gpu_path.POISON)          # rows past off[E] untouched


@pytest.mark.timeout(600)
def test_moonep_shape():
    wl = workloads.make("moonep", seed=21, S=600)
    _check(wl.x, wl.topk_idx, wl.E, 128)


@pytest.mark.timeout(600)
@pytest.mark.parametrize("S", workloads.FP8_SWEEP_TOKENS)
def test_small_token_shape(S):
    """H=6144, E=256, K=8 (the fp8 latency workload), bf16 input rows."""
    wl = workloads.make("moonep", seed=S, S=S, H=6144, E=256, K=8)
    _check(wl.x, wl.topk_idx, wl.E, 128)


@pytest.mark.timeout(600)
@pytest.mark.parametrize("block", [16, 32, 64, 128, 256])
def test_block_sizes(block):
    wl = workloads.make("moonep", seed=block, S=257, H=768, E=16, K=3)
    _check(wl.x, wl.topk_idx, wl.E, block)


@pytest.mark.timeout(600)
@pytest.mark.parametrize("H", [4096, 2560, 1024])
@pytest.mark.parametrize("block", [16, 128, 256])
@pytest.mark.parametrize("sc_offset", [0, 1])
def test_both_kernels(H, block, sc_offset):
    """Rows that are whole multiples of 4 blocks with a 16-byte aligned scale
    buffer go through shared memory and bulk stores (2048-element chunks and
    a shorter last chunk); the others (H % (4*block) != 0, or a scale buffer
    that is only 4-byte aligned) through the register kernel.  Same bits."""
    wl = workloads.make("moonep", seed=H + block, S=131, H=H, E=32, K=6)
    _check(wl.x, wl.topk_idx, wl.E, block, sc_offset)


@pytest.mark.timeout(600)
def test_edge_rows():
    """All-zero blocks (scale 1), tiny blocks (subnormal codes), huge values,
    a ragged H (not a multiple of 256), unused entries."""
    wl = workloads.make("moonep", seed=3, S=90, H=384, E=8, K=4)
    xf = workloads.activations_f32(3, 90, 384)
    xf[0] = 0.0
    xf[1, :128] *= 1e-30
    xf[2, 128:256] *= 1e30
    xf[4, ::7] = 448.0
    x = workloads.to_bf16_bits(xf)
    idx = wl.topk_idx.copy()
    idx[::5, 2] = -1
    _check(x, idx, wl.E, 128)


@pytest.mark.timeout(600)
@pytest.mark.parametrize("H", [1024, 384])   # shared-memory kernel, register kernel
def test_tiny_blocks(H):
    """Blocks whose largest magnitude is near or below 2^-83, down to the
    smallest bf16 subnormal: their scale amax/448 reaches the f32 subnormal
    range, where the reciprocal-based division is not exact; the codes and
    scales must still be those of the oracle's plain divisions."""
    rng = np.random.default_rng(5)
    S, E, K = 64, 8, 3
    mags = [2.0 ** -82, 2.0 ** -83, 2.0 ** -84, 1e-30, 1e-35, 5.3e-36, 1e-37, 1e-38,
            2.0 ** -126, 2.0 ** -127, 2.0 ** -130, 2.0 ** -133]
    xf = np.zeros((S, H), np.float32)
    nb = H // 128
    for r in range(S):
        for b in range(nb):
            m = mags[(r * nb + b) % len(mags)]
            blk = rng.standard_normal(128).astype(np.float32) * np.float32(m)
            blk[rng.integers(0, 128)] = np.float32(m) * (1 if (r + b) % 2 else -1)
            xf[r, b * 128:(b + 1) * 128] = blk
    x = workloads.to_bf16_bits(xf)
    idx = workloads.topk_uniform(9, S, E, K)
    _check(x, idx, E, 128)


@pytest.mark.timeout(600)
def test_every_bf16_value_encodes_like_the_oracle():
    """Each 128-block holds 448 (so scale = 1 and the codes are the plain
    E4M3 encoding of the inputs) and 127 bf16 values; together the rows cover
    every finite bf16 value of magnitude <= 448."""
    allbits = np.arange(1 << 16, dtype=np.uint32)
    vals = (allbits << 16).view(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= 448)
    bits = allbits[keep].astype(np.uint16)
    per = 127
    nrows_blocks = -(-bits.size // per)
    pad = nrows_blocks * per - bits.size
    bits = np.concatenate([bits, np.zeros(pad, np.uint16)]).reshape(nrows_blocks, per)
    lead = np.full((nrows_blocks, 1), 0x43E0, np.uint16)     # bf16 448.0
    blocks = np.concatenate([lead, bits], axis=1)             # [nb, 128]
    H = 1024
    nb_row = H // 128
    nrows = -(-blocks.shape[0] // nb_row)
    extra = nrows * nb_row - blocks.shape[0]
    filler = np.tile(np.concatenate([[0x43E0], np.zeros(127, np.uint16)]).astype(np.uint16),
                     (extra, 1))
    x = np.concatenate([blocks, filler]).reshape(nrows, H)
    idx = np.zeros((nrows, 1), np.int32)
    q, sc, V = _run(x, idx, 1, 128)
    assert np.all(sc[:V] == 1.0)
    ref = np.array([oracle.f32_to_e4m3(float(v)) for v in
                    (x.astype(np.uint32) << 16).view(np.float32).reshape(-1)], np.uint8)
    assert np.array_equal(q[:V].reshape(-1), ref)


@pytest.mark.timeout(600)
def test_quantised_dispatch_matches_dispatch_of_quantised_rows():
    """The fused path equals quantising with the oracle and dispatching the
    codes and scales with the byte-copy dispatch (which forwards scales)."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=5, S=128, H=6144, E=256, K=8)
    q0, sc0 = oracle.quant_fp8(wl.x, 128)
    dev = torch.device("cuda")
    plan = moe.moe_plan(torch.from_numpy(wl.topk_idx).to(dev), wl.E)
    pq, ps = moe.moe_dispatch(torch.from_numpy(q0).to(dev).view(torch.float8_e4m3fn),
                              plan.tok_map, x_scales=torch.from_numpy(sc0).to(dev))
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    fq, fs = moe.moe_dispatch_quant_fp8(x, plan.tok_map)
    torch.cuda.synchronize()
    assert torch.equal(pq.view(torch.uint8), fq.view(torch.uint8))
    assert torch.equal(ps.view(torch.int32), fs.view(torch.int32))


def _oracle_quant_parallel(x_bf16, block):
    """oracle.quant_fp8 over row chunks in spawned worker processes (the
    quantisation is per row, so chunks are independent); the oracle itself
    stays single-threaded C."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    n = max(1, min(16, os.cpu_count() or 1))
    chunks = [c for c in np.array_split(np.arange(x_bf16.shape[0]), n) if c.size]
    with ProcessPoolExecutor(len(chunks), mp_context=mp.get_context("spawn")) as ex:
        parts = list(ex.map(oracle.quant_fp8, [np.ascontiguousarray(x_bf16[c]) for c in chunks],
                            [block] * len(chunks)))
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))


@pytest.mark.timeout(900)
def test_full_size_every_token():
    """The benchmarked launch (S=4096 H=7168 E=64 K=8, block 128): the codes
    and scales of every token, in each of its K packed rows, equal the
    oracle's quantisation of that token row."""
    import combine_moe_plan_02_gb300 as moe
    wl = workloads.make("moonep", seed=0)
    dev = torch.device("cuda")
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev).view(torch.bfloat16)
    plan = moe.moe_plan(torch.from_numpy(wl.topk_idx).to(dev), wl.E)
    q = gpu_path.poisoned((wl.S * wl.K, wl.H), torch.uint8)
    sc = gpu_path.poisoned((wl.S * wl.K, wl.H // 128), torch.float32)
    moe.moe_dispatch_quant_fp8(x, plan.tok_map, packed_q=q, packed_scales=sc)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    tm = plan.tok_map.cpu().numpy()
    assert np.array_equal(tm, oracle.plan(wl.topk_idx, wl.E)["tok_map"])
    q0, sc0 = _oracle_quant_parallel(wl.x, 128)
    qn = q.cpu().numpy()
    scn = sc.cpu().numpy().view(np.uint32)
    order = tm.reshape(-1)                   # packed row of entry s*K + k
    assert np.array_equal(qn[order], np.repeat(q0, wl.K, axis=0))
    assert np.array_equal(scn[order], np.repeat(sc0.view(np.uint32), wl.K, axis=0))
