"""The INT8 tensor-rate probe (the denominator of "% of dense INT8 peak"):
through the C-ABI it runs, synchronises and reports a plausible rate for the
legacy mma.sync s8 instruction of an sm_103 part (on the order of 150 TOPS;
the bound below only rejects a probe that did not run or timed nothing)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_probe_mma_s8_reports_a_plausible_rate(lib):
    assert torch.cuda.is_available()
    t1 = lib.h3q_probe_mma_s8_tops()
    t2 = lib.h3q_probe_mma_s8_tops()
    assert 20.0 < t1 < 2000.0, t1
    # two runs of the same probe agree to within a few percent
    assert abs(t1 - t2) / max(t1, t2) < 0.1, (t1, t2)
