"""The tensor-rate probe: dense FP16 FLOP per SM per clock, measured on the device.

The GEMM's per-clock roofline is SMs x (FLOP per SM per clock) x SM clock; the probe gives
the middle factor from the hardware itself.  It cannot exceed the Blackwell-class dense
rate of 8192 FLOP per SM per clock (a 128 x 256 x 16 MMA every 128 clocks) by more than the
timing's own noise, and the issue loop keeps the pipe busy enough to come close to it.
"""
import pytest

import tensor_core_tiled_gb300 as tct

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(tct_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def test_tensor_rate_probe_per_sm_per_clock():
    med, lo, hi = tct.gemm_tensor_rate_probe(1 << 16, torch.cuda.current_stream().cuda_stream)
    assert 0 < lo <= med <= hi
    assert 0.9 * 8192 <= med <= 1.01 * 8192, med
    assert tct.gemm_f16_f32_get_error() == tct.GEMM_OK


def test_tensor_rate_probe_rejects_bad_counts():
    for n in (0, -1, (1 << 22) + 1):
        with pytest.raises(tct.GemmError):
            tct.gemm_tensor_rate_probe(n)
