"""The mma.sync throughput probe (wq_debug_mma_peak) that bench.py times for
the int8 and bf16 warp-level peaks: every thread's checksum must be exactly
8 chains x 4 elements x K x iters, so a launch that skipped work fails."""

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402


@pytest.mark.parametrize("kind,k", [(0, 32), (1, 16)])
@pytest.mark.parametrize("iters,blocks", [(1, 1), (37, 3), (1000, 152)])
def test_mma_peak_checksums_are_exact(kind, k, iters, blocks):
    out = wq.debug_mma_peak(kind, iters, blocks)
    torch.cuda.synchronize()
    assert out.shape == (blocks * 256,)
    assert bool((out == 8 * 4 * k * iters).all())
    wq.check_status()
