"""The allocation-free entry point, h3q_linear_w8a8_noalloc.

It serves callers that may not allocate device memory at call time (for
example an engine plugin handed only its input and output buffers); its
scratch is a fixed 16 MiB array inside the library.  Through the C-ABI, two
calls in a row must give the same results as h3q_linear_w8a8 with a
caller-provided workspace.  Both run the same kernels on the same operands, and
the library's outputs depend on the operands alone, so everything is compared
bit for bit: INT32 accumulators, activation scales and BF16 outputs (a shared-
scratch fault could otherwise hide inside a one-ulp tolerance).  After each
call the scratch's status word, read with h3q_linear_w8a8_noalloc_status, must
be clear.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _bf16(bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def test_noalloc_matches_workspace_entry_point_twice():
    import w8a8_int8_linear_h3q_gb300 as h3q
    h3q.load()
    dev = torch.device("cuda:0")
    for call, (M, N, K, seed) in enumerate([(300, 264, 5376, 71), (97, 136, 1040, 72)]):
        c = synth.make_linear(M, N, K, seed=seed, outlier_p=0.01, outlier_mul=20.0)
        qw, sw = h3q.h3q_quantize_weights(torch.from_numpy(c.w[0]).to(dev))
        x = _bf16(c.x_bits, dev)
        b = _bf16(c.bias_bits[0], dev)
        ref = h3q.h3q_linear_w8a8(x, qw, sw, b, want_acc=True, want_xq=True)
        got = h3q.h3q_linear_w8a8_noalloc(x, qw, sw, b, want_acc=True)
        torch.cuda.synchronize()
        assert torch.equal(got["acc"], ref["acc"]), f"call {call}: INT32 accumulators differ"
        assert torch.equal(got["xs"].view(torch.int32), ref["xs"].view(torch.int32))
        assert torch.equal(got["y"].view(torch.int16), ref["y"].view(torch.int16)), \
            f"call {call}: BF16 outputs differ"
        assert h3q.h3q_linear_w8a8_noalloc_status(M, K) == h3q.H3Q_OK
        # pre-quantised activations as well (the INT8 -> FP16 coding path)
        got2 = h3q.h3q_linear_w8a8_noalloc(None, qw, sw, b, xq=ref["xq"], xs=ref["xs"],
                                           want_acc=True)
        torch.cuda.synchronize()
        assert torch.equal(got2["acc"], ref["acc"])
        assert torch.equal(got2["y"].view(torch.int16), ref["y"].view(torch.int16))
        assert h3q.h3q_linear_w8a8_noalloc_status(M, K) == h3q.H3Q_OK


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import w8a8_int8_linear_h3q_gb300 as h3q
    h3q.load()
    dev = torch.device("cuda:0")
    M, N, K = 4096, 128, 5376          # needs ~44 MB of scratch
    assert h3q.h3q_linear_workspace_bytes(M, N, K) > 16 << 20
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=dev)
    qw = torch.zeros((N, K), dtype=torch.int8, device=dev)
    sw = torch.ones((N,), dtype=torch.float32, device=dev)
    with pytest.raises(h3q.H3QError) as e:
        h3q.h3q_linear_w8a8_noalloc(x, qw, sw)
    assert e.value.status == h3q.H3Q_ERR_UNSUPPORTED_SHAPE
