"""Combine at batch sizes of tens of thousands of gathered rows against the
CPU oracle, bitwise: a ragged last lane step, K from 1 to 16, f32 output,
unweighted rows through the fold call, and unused and out-of-range expert
ids, including a token with no valid entry (its output row is zero)."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from tests import gpu_path  # noqa: E402


def _inputs(S, H, E, K, seed, holes):
    wl = workloads.make("moonep", seed=seed, S=S, H=H, E=E, K=K)
    idx = wl.topk_idx.copy()
    if holes:
        idx[::7, 0] = -1
        idx[::11, K - 1] = E        # out of range: no slot, counted invalid
        idx[5, :] = -1              # a token with no valid entry
    p = oracle.plan(idx, E)
    V = int(p["off"][-1])
    y = workloads.to_bf16_bits(workloads.activations_f32(seed + 1, V, H))
    return wl, idx, p, y


def _run(y, w, tok_map, H, out_dt, weighted):
    import combine_moe_plan_02_gb300 as moe
    dev = torch.device("cuda")
    yd = torch.from_numpy(y.view(np.int16)).to(dev).view(torch.bfloat16)
    wd = torch.from_numpy(w).to(dev)
    md = torch.from_numpy(tok_map).to(dev)
    tdt = torch.float32 if out_dt == "f32" else torch.bfloat16
    out = gpu_path.poisoned((tok_map.shape[0], H), tdt)
    if weighted:
        moe.moe_combine(yd, wd, md, out=out)
    else:
        moe.moe_combine_fold(yd, wd, md, weighted=False, fold=False, out=out)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() == 0
    got = out.cpu()
    return got.view(torch.int16).numpy().view(np.uint16) if out_dt == "bf16" else got.numpy()


@pytest.mark.timeout(600)
@pytest.mark.parametrize("S,H,E,K,out_dt,weighted,holes", [
    (2000, 4104, 64, 8, "bf16", True, False),    # 513 steps of 8 per row: one lane-step tail
    (2000, 4104, 64, 8, "f32", True, False),     # f32 output (quad layout)
    (16000, 1024, 16, 2, "bf16", True, False),   # K = 2
    (12000, 2048, 8, 1, "bf16", True, False),    # K = 1: a weighted copy
    (2000, 2048, 64, 16, "bf16", True, False),   # K = 16: two chunks of 8 gathers
    (2500, 3080, 64, 8, "bf16", True, True),     # unused and invalid ids
    (2500, 3080, 64, 8, "bf16", False, True),    # unweighted (fold call, no out_weights)
])
def test_large_combine_matches_oracle(S, H, E, K, out_dt, weighted, holes):
    wl, idx, p, y = _inputs(S, H, E, K, seed=S + H + K, holes=holes)
    got = _run(y, wl.topk_w, p["tok_map"], H, out_dt, weighted)
    if weighted:
        ref = oracle.combine(y, "bf16", wl.topk_w, p["tok_map"], H, out_dt)
    else:
        ref, _ = oracle.combine_fold(y, "bf16", wl.topk_w, p["tok_map"], H, out_dt,
                                     weighted=False, fold=False)
    assert np.array_equal(got.view(np.uint8), ref.view(np.uint8)), \
        f"{int((got != ref).sum())} elements differ"
    if holes:
        assert not got[5].view(np.uint8).any()   # +0.0 everywhere


@pytest.mark.timeout(300)
@pytest.mark.parametrize("out_dt", ["bf16", "f32"])
def test_out_of_range_map_entries_are_dropped_and_reported(out_dt):
    """Map entries outside [-1, y_rows) are never gathered: the term is
    dropped, bit 2 of the device error word is set, and every other term is
    summed as usual (bf16 output takes the K <= 8 bf16 kernel, f32 output the
    general one)."""
    import combine_moe_plan_02_gb300 as moe
    S, H, E, K = 600, 1032, 32, 8
    wl, idx, p, y = _inputs(S, H, E, K, seed=77, holes=False)
    V = y.shape[0]
    bad = p["tok_map"].copy()
    bad[3, 2] = V                 # one past the end of y
    bad[10, 0] = V + 12345
    bad[11, 7] = 1 << 40
    bad[20, 4] = -7
    dropped = bad.copy()
    dropped[(dropped >= V) | (dropped < -1)] = -1
    assert moe.moe_device_errors() == 0
    dev = torch.device("cuda")
    yd = torch.from_numpy(y.view(np.int16)).to(dev).view(torch.bfloat16)
    tdt = torch.float32 if out_dt == "f32" else torch.bfloat16
    out = gpu_path.poisoned((S, H), tdt)
    moe.moe_combine(yd, torch.from_numpy(wl.topk_w).to(dev), torch.from_numpy(bad).to(dev),
                    out=out)
    torch.cuda.synchronize()
    assert moe.moe_device_errors() & 4
    got = out.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if out_dt == "bf16" else got.numpy()
    ref = oracle.combine(y, "bf16", wl.topk_w, dropped, H, out_dt)
    assert np.array_equal(got.view(np.uint8), ref.view(np.uint8))
