"""The tensor-core throughput probe behind the prefill roofline: it runs,
leaves the device status clean, and its measured rate is a plausible dense
FP4 rate for one GB300 (well above the bf16 rate of the same tensor cores,
below the nominal FP4 figure)."""
import pytest
import torch

from gpu_util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    return ensure_built()


@pytest.mark.parametrize("n", [64, 128, 256])
def test_mxf4_probe_rate(moe, n):
    s = torch.cuda.current_stream()
    moe.moe_mxf4_mma_probe(n, 1 << 12, s)  # warm
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    flops = moe.moe_mxf4_mma_probe(n, 1 << 16, s)
    e1.record(s)
    torch.cuda.synchronize()
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    assert moe.moe_device_status() == 0
    assert 100.0 < tflops < 20000.0, tflops
    print(f"kind::mxf4 M=128 N={n} K=64: {tflops:.0f} TFLOP/s")
