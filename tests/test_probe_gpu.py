"""The tensor-rate probes, through the C-ABI.

The INT8 probe (the denominator of "% of dense INT8 peak") runs, synchronises
and reports a plausible rate for the legacy mma.sync s8 instruction of an
sm_103 part (on the order of 150 TOPS; the bound only rejects a probe that did
not run or timed nothing).

The FP16 pair-MMA probe times the hot GEMM's own instruction.  Its rate cannot
exceed what 152 SMs at the part's highest clock can do: 8192 operations per
clock and SM for dense FP16 (2.25 PFLOP/s nominal), so 152 * 8192 * 2.07e9 =
2.58 PFLOP/s; and a probe that ran reports well above the INT8 instruction's
rate."""
import pytest
import torch

pytestmark = pytest.mark.gpu

F16_CEILING_TFLOPS = 152 * 8192 * 2.07e9 / 1e12


def test_probe_mma_s8_reports_a_plausible_rate(lib):
    assert torch.cuda.is_available()
    t1 = lib.h3q_probe_mma_s8_tops()
    t2 = lib.h3q_probe_mma_s8_tops()
    assert 20.0 < t1 < 2000.0, t1
    # two runs of the same probe agree to within a few percent
    assert abs(t1 - t2) / max(t1, t2) < 0.1, (t1, t2)


@pytest.mark.parametrize("a_in_smem", [False, True])
def test_probe_mma_f16_pair_reports_a_plausible_rate(lib, a_in_smem):
    assert torch.cuda.is_available()
    t1 = lib.h3q_probe_mma_f16_pair_tflops(a_in_smem)
    t2 = lib.h3q_probe_mma_f16_pair_tflops(a_in_smem)
    assert 500.0 < t1 < 1.02 * F16_CEILING_TFLOPS, t1
    assert abs(t1 - t2) / max(t1, t2) < 0.1, (t1, t2)
