"""The device-side failure path: a bounded wait that runs out reports a
timeout in the status word the host reads, and the context stays usable.
The wait is made to run out without any fault (an mbarrier that nothing
arrives on), by the same helper every kernel of the library uses."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(lib, oracle):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    dev = torch.device("cuda:0")
    status = torch.full((4,), -1, dtype=torch.int32, device=dev)
    assert lib.h3q_selftest_bounded_wait(status) == lib.H3Q_ERR_TIMEOUT
    assert int(status[0]) != 0
    # the context is still usable: a Linear right after is correct and its own
    # status word is clean
    rng = np.random.default_rng(90)
    xb = oracle.round_to_bf16(rng.standard_normal((100, 512)))
    w = (rng.standard_normal((72, 512)) * 0.02).astype(np.float32)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    qw, sw = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
    out = lib.h3q_linear_w8a8(x, qw, sw, None, want_acc=True)
    torch.cuda.synchronize()
    assert lib.h3q_workspace_status(out["workspace"], 100, 512) == lib.H3Q_OK
    ref = oracle.linear(xb, *oracle.quantize_weights(w))
    assert np.array_equal(out["acc"].cpu().numpy(), ref["acc"])
