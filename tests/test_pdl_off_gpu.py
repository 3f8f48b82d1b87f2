"""The full-size parity cases once more, on a build of the library whose
launches never overlap their predecessor (programmatic dependent launch
switched off at compile time, MOE_USE_PDL=0).

Every kernel of the library waits (griddepcontrol.wait) before it touches
memory that earlier stream work writes, and the plan's rank kernel reads
topk_idx before that wait only when its histogram kernel, launched without
the attribute, ran first.  With PDL on, the results depend on that ordering
being right; with PDL off, each launch starts only after the previous one
finished, so the ordering cannot matter.  Both builds must give the oracle's
bits (MoonEP "Drop cooperative launch ...", "New test": each case run with
PDL on and with PDL off).

The second build goes to a temporary directory and is loaded by a child
pytest process through MOE_GB300_LIB; the child runs the selected parity
tests unchanged.
"""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# the full-size workloads, the plan modes (one tile, one launch, two kernels,
# static scratch), the one-launch plan + dispatch, graphs, capacity, dedup and
# batches on several streams at once
PDL_OFF_CASES = [
    "tests/test_parity_gpu.py::test_moonep_full_size",
    "tests/test_parity_gpu.py::test_zipf_full_size",
    "tests/test_parity_gpu.py::test_dedup_full_size",
    "tests/test_parity_gpu.py::test_shapes",
    "tests/test_parity_gpu.py::test_fp8_small_token_sweep",
    "tests/test_plan_dispatch_gpu.py::test_tiled_one_launch_shapes",
    "tests/test_plan_dispatch_gpu.py::test_fp8_rows_and_scales",
    "tests/test_plan_dispatch_gpu.py::test_cuda_graph_replay",
    "tests/test_capacity_gpu.py::test_capacity_uniform",
    "tests/test_capacity_gpu.py::test_dedup_over_capacity_plan",
    "tests/test_combine_large_gpu.py",
    "tests/test_zz_no_alloc.py",
    "tests/test_graph_gpu.py",
    "tests/test_streams_gpu.py",
    "tests/test_pdl_off_gpu.py::test_loaded_library_is_the_requested_build",
]


def test_loaded_library_is_the_requested_build():
    """In the child process: the binding loaded the build named by
    MOE_GB300_LIB (in a normal run: the in-tree build)."""
    import combine_moe_plan_02_gb300 as moe
    from combine_moe_plan_02_gb300 import _abi
    want = os.environ.get("MOE_GB300_LIB") or os.path.join(_abi.PKG, "libmoe_gb300.so")
    assert os.path.samefile(moe.lib()._name, want)


@pytest.mark.timeout(1800)
def test_full_size_parity_with_pdl_off(tmp_path):
    from combine_moe_plan_02_gb300 import build
    lib = build.build(force=True, out=str(tmp_path / "libmoe_gb300_nopdl.so"),
                      build_dir=str(tmp_path / "obj"), defines=("MOE_USE_PDL=0",))
    env = dict(os.environ, MOE_GB300_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        "-p", "no:cacheprovider", *PDL_OFF_CASES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1700)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1]
