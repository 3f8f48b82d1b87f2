"""The two number-format conversions of the kernels, over every binary32 bit
pattern (moe_selftest_convert runs them exactly as the quantising dispatch
casts its quotients to E4M3 and as the combines store bf16): against torch's
CPU casts, library routines written from the same format definitions (OCP
OFP8 v1.0 E4M3; bfloat16 = the upper half of binary32, round to nearest
even), to which the oracle's own encoders are pinned in tests/pins.py
(ROCm/mori "Draft: cco + flydsl dispatch/combine #448", Fp8BlockwiseQuant
notes and accumulator note).

torch's E4M3 cast does not saturate: from 464 up (the midpoint between 448
and the 480 that E4M3 cannot hold) it returns the NaN code, where the
kernels' cast gives +-448, the largest finite code, as the quantisation rule
requires; those values are checked against that rule instead.  NaN inputs
must give a NaN code / a NaN bf16."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

CHUNK = 1 << 28


@pytest.mark.timeout(1800)
def test_every_binary32_pattern():
    import combine_moe_plan_02_gb300 as moe
    L = moe.lib()
    dev = torch.device("cuda")
    e8 = torch.empty(CHUNK, dtype=torch.uint8, device=dev)
    b16 = torch.empty(CHUNK, dtype=torch.int16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    base = np.arange(CHUNK, dtype=np.uint32)
    for first in range(0, 1 << 32, CHUNK):
        assert L.moe_selftest_convert(first, CHUNK, e8.data_ptr(), b16.data_ptr(), stream) == 0
        bits = base + np.uint32(first)                  # no wrap: first + CHUNK <= 2^32
        f = torch.from_numpy(bits.view(np.float32))
        got8 = e8.cpu()
        got16 = b16.cpu()
        nan = torch.isnan(f)
        sat = (f.abs() >= 464.0) & ~nan
        ref8 = f.to(torch.float8_e4m3fn).view(torch.uint8)
        ok8 = (got8 == ref8) | sat | nan
        assert bool(ok8.all()), f"E4M3 differs from bit pattern {first:#x} on"
        want_sat = torch.where(f[sat] < 0, 0xFE, 0x7E).to(torch.uint8)
        assert torch.equal(got8[sat], want_sat)
        assert bool(((got8[nan] & 0x7F) == 0x7F).all())
        ref16 = f.to(torch.bfloat16).view(torch.int16)
        ok16 = (got16 == ref16) | nan
        assert bool(ok16.all()), f"bf16 differs from bit pattern {first:#x} on"
        assert bool(((got16[nan].to(torch.int32) & 0x7FFF) > 0x7F80).all())
    assert moe.moe_device_errors() == 0
