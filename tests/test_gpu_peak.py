"""The tensor-core throughput probe (hm_mma_peak_probe): every MMA kind runs to completion on
the GPU without a device error, reports the FLOPs it issued, and its rate is a plausible fraction
of the kind's nominal dense peak (above a tenth, below twice). The probe's numbers are the
denominators of the tensor-bound roofline fractions, so this only guards that it measures tensor
work at all; the values themselves are recorded by the benchmark."""
import pytest
import torch

pytestmark = pytest.mark.gpu

NOMINAL_TFLOPS = {0: 2250.0, 1: 4500.0, 2: 13500.0, 3: 4500.0, 4: 13500.0,   # bf16, fp8, fp4 dense
                  5: 2250.0, 6: 2250.0}


@pytest.fixture(scope="module")
def hm():
    import __graft_entry__
    __graft_entry__.build()
    from moe_hm_gemm_gb300 import hm as mod
    return mod


@pytest.mark.parametrize("kind", [0, 1, 2, 3, 4, 5, 6])
def test_peak_probe_runs_and_is_plausible(hm, kind):
    tflops, ms = hm.mma_peak(kind, iters=2000, repeats=2)
    assert hm.device_error() == 0
    assert ms > 0
    nominal = NOMINAL_TFLOPS[kind]
    assert 0.1 * nominal < tflops < 2.0 * nominal, f"kind {kind}: {tflops:.0f} TFLOP/s"
