"""Seeded input generators and the stored oracle fixture (no GPU)."""
import hashlib
import json
import os

import numpy as np

import oracle
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def test_splitmix64_known_values():
    # SplitMix64 reference outputs for state 0 (Vigna's splitmix64.c):
    # the first outputs are mix(1*gamma), mix(2*gamma), ...
    gamma = 0x9E3779B97F4A7C15

    def mix(z):
        z &= (1 << 64) - 1
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & ((1 << 64) - 1)
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & ((1 << 64) - 1)
        return z ^ (z >> 31)

    assert mix(gamma) == 0xE220A8397B1DCDAF   # published first output of SplitMix64 from seed 0
    key = mix((3 * 0x632BE59BD9B4E019 + 2 * 0x8CB92BA72F3D8DD7) & ((1 << 64) - 1))
    got = workloads.splitmix64(3, 2, 4)
    want = [mix(key + (i + 1) * gamma) for i in range(4)]
    assert [int(v) for v in got] == want


def test_deterministic_and_shaped():
    a = workloads.make("moonep", seed=0, S=64, H=128)
    b = workloads.make("moonep", seed=0, S=64, H=128)
    assert np.array_equal(a.topk_idx, b.topk_idx) and np.array_equal(a.x, b.x)
    assert a.topk_idx.shape == (64, 8) and a.topk_idx.dtype == np.int32
    assert a.x.shape == (64, 128) and a.x.dtype == np.uint16
    c = workloads.make("moonep", seed=1, S=64, H=128)
    assert not np.array_equal(a.topk_idx, c.topk_idx)


def test_routing_distinct_and_weights_normalised():
    for name in ("tiny", "moonep", "zipf", "dedup", "fp8small"):
        wl = workloads.make(name, seed=2, S=257, H=128 if name != "fp8small" else 256)
        idx = wl.topk_idx
        assert idx.min() >= 0 and idx.max() < wl.E
        assert all(len(set(r.tolist())) == wl.K for r in idx)
        assert np.allclose(wl.topk_w.sum(axis=1), 1.0, atol=1e-6)
        assert wl.topk_w.dtype == np.float32


def test_uniform_routing_is_balanced():
    wl = workloads.make("moonep", seed=0, S=4096, H=8)
    cnt = np.bincount(wl.topk_idx.reshape(-1), minlength=wl.E)
    assert cnt.sum() == 4096 * 8
    assert abs(cnt.mean() - 512) < 1e-9 and cnt.min() > 400 and cnt.max() < 630


def test_zipf_routing_is_skewed_with_empty_tail():
    wl = workloads.make("zipf", seed=0, S=8192, H=8)
    cnt = np.sort(np.bincount(wl.topk_idx.reshape(-1), minlength=wl.E))[::-1]
    assert cnt[0] > 0.9 * 8192           # the top experts are hit by nearly every token
    assert cnt[-1] < 60                  # the tail is almost empty
    assert cnt[:8].sum() > 0.4 * cnt.sum()


def test_fp8_quantisation_rule():
    wl = workloads.make("fp8small", seed=3, S=8)
    import torch
    q = torch.from_numpy(wl.x).view(torch.float8_e4m3fn).float().numpy()
    xf = workloads.activations_f32(3, 8, wl.H)
    blocks = xf.reshape(8, -1, 128)
    amax = np.abs(blocks).max(axis=2)
    assert np.array_equal(wl.x_scales, (amax / np.float32(448.0)).astype(np.float32))
    # the largest element of each block maps to the largest finite code
    assert np.all(np.abs(q.reshape(8, -1, 128)).max(axis=2) == 448.0)
    deq = q.reshape(8, -1, 128) * wl.x_scales[:, :, None]
    assert np.all(np.abs(deq - blocks) <= np.abs(blocks) * 2 ** -3 + wl.x_scales[:, :, None] * 2 ** -9)


def test_empty_workloads():
    for name in ("dedup", "fp8small", "tiny"):
        wl = workloads.make(name, seed=0, S=0)
        assert wl.topk_idx.shape == (0, wl.K) and wl.x.shape[0] == 0


def test_stored_tiny_fixture_matches_oracle():
    with open(os.path.join(HERE, "golden", "tiny_seed0.json")) as f:
        gold = json.load(f)
    res = oracle.run_workload(workloads.make("tiny", seed=0))
    assert res["cnt"].tolist() == gold["cnt"]
    assert res["off"].tolist() == gold["off"]
    assert res["n_invalid"] == gold["n_invalid"]
    assert res["tok_map"].reshape(-1).tolist() == gold["tok_map"]
    assert res["packed_src"].tolist() == gold["packed_src"]
    assert hashlib.sha256(res["packed_x"].tobytes()).hexdigest() == gold["sha256_packed_x"]
    assert hashlib.sha256(res["out"].tobytes()).hexdigest() == gold["sha256_out"]
