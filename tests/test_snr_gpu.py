"""Accuracy of the quantised Linear against the unquantised one (an INT8 SNR
check, as the "[feat] Add MiniMax H3 MLX T2VA inference" review's test
coverage lists), per profile of the converter's scope rule: dit_proj
quantises all six projections of a block, the narrower mlp profile only FC1
and FC2 ("feat(mps): support MiniMax-H3 INT8 inference on Apple M5", opening
description: optional narrower profiles for accuracy ablations).

On sampled token rows, the GPU's W8A8 outputs are compared with the float64
unquantised Linear; their SNR must equal the oracle's own W8A8 SNR on the same
rows (the GPU is within one BF16 ulp of the oracle), which this test also
reports.  The figures themselves are a property of symmetric per-token INT8,
not a pass mark; a floor of 15 dB only guards against a broken path."""
import numpy as np
import pytest
import torch

import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _rows(M, seed, n=256):
    return np.sort(np.random.default_rng(seed).choice(M, size=min(n, M), replace=False))


def _snr_pair(lib, oracle, dev, x_dev, x_bits_rows, w, b_dev, b_bits, rows):
    qw, sw = lib.h3q_quantize_weights(w if torch.is_tensor(w) else torch.from_numpy(w).to(dev))
    out = lib.h3q_linear_w8a8(x_dev, qw, sw, b_dev)
    w_np = w.cpu().numpy() if torch.is_tensor(w) else w
    ref = oracle.reference_linear(x_bits_rows, w_np, b_bits)
    y_gpu = oracle.widen_bf16(_bits(out["y"][torch.from_numpy(rows).to(dev)]))
    y_orc = oracle.widen_bf16(oracle.linear(x_bits_rows, *oracle.quantize_weights(w_np), b_bits)["y"])
    return oracle.snr_db(y_gpu, ref), oracle.snr_db(y_orc, ref)


@pytest.mark.parametrize("profile", ["dit_proj", "mlp"])
def test_sweep_block_snr_per_profile(lib, oracle, dev, profile):
    block, M = 0, synth.SWEEP_M
    rows = _rows(M, 700)
    xs = {K: synth.sweep_x(K, dev) for K in (synth.H3_WIDTH, synth.H3_MLP_WIDTH)}
    names = {"q": "attn.to_q", "k": "attn.to_k", "v": "attn.to_v", "o": "attn.to_out",
             "fc1": "mlp.fc1", "fc2": "mlp.fc2"}
    report = {}
    for j, (nm, N, K) in enumerate(synth.SWEEP_LINEARS):
        if not oracle.in_scope(f"blocks.{block}.{names[nm]}.weight", profile):
            continue                                 # stays unquantised under this profile
        w, b = synth.sweep_weight(block, j, dev)
        x = xs[K]
        xr = _bits(x[torch.from_numpy(rows).to(dev)])
        gpu, orc = _snr_pair(lib, oracle, dev, x, xr, w, b, _bits(b), rows)
        assert abs(gpu - orc) < 0.05, (nm, gpu, orc)
        assert gpu > 15.0, (nm, gpu)
        report[nm] = round(float(gpu), 2)
    expect = {"dit_proj": {"q", "k", "v", "o", "fc1", "fc2"}, "mlp": {"fc1", "fc2"}}[profile]
    assert set(report) == expect
    print(f"\nW8A8 vs float64 SNR (dB), sweep block {block}, profile {profile}: {report}")


def test_named_workloads_snr(lib, oracle, dev):
    report = {}
    for name in ("attn", "fc1", "fc2"):
        c = synth.WORKLOADS[name]()
        rows = _rows(c.M, 710)
        x = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        b = torch.from_numpy(c.bias_bits[0].view(np.int16)).view(torch.bfloat16).to(dev)
        gpu, orc = _snr_pair(lib, oracle, dev, x, c.x_bits[rows], c.w[0], b, c.bias_bits[0], rows)
        assert abs(gpu - orc) < 0.05, (name, gpu, orc)
        assert gpu > 15.0, (name, gpu)
        report[name] = round(float(gpu), 2)
    print(f"\nW8A8 vs float64 SNR (dB), first Linear of each workload: {report}")


def test_affine_comparison_snr(lib, oracle, dev):
    # The comparison scheme of "MLX implementation and experiment report"
    # (Operator tuning: Q8/g64, Q4/g64): weight-only group-wise affine.  Its
    # SNR against the float64 unquantised Linear, on the same rows as W8A8:
    # the GPU's Q8 and Q4 paths must match the oracle's SNR at the same width.
    # Weight-only Q8 keeps the BF16 activations, so it should sit well above
    # per-token INT8 activations; Q4's 17x coarser step puts it below both.
    report = {}
    for name in ("attn", "fc2", "image_qkv", "image_down"):
        c = synth.WORKLOADS[name]()
        rows = _rows(c.M, 720, n=128)
        cols = np.sort(np.random.default_rng(721).choice(c.w[0].shape[0], 1024, replace=False))
        x = torch.from_numpy(c.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        b = torch.from_numpy(c.bias_bits[0].view(np.int16)).view(torch.bfloat16).to(dev)
        w = c.w[0]
        ref = oracle.reference_linear(c.x_bits[rows], w[cols], c.bias_bits[0][cols])
        rt, ct = torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)
        # W8A8 on the GPU
        qw, sw = lib.h3q_quantize_weights(torch.from_numpy(w).to(dev))
        y8 = lib.h3q_linear_w8a8(x, qw, sw, b)["y"][rt][:, ct]
        snr = {"w8a8": oracle.snr_db(oracle.widen_bf16(_bits(y8)), ref)}
        # affine Q8 and Q4 on the GPU, and the oracle's at the same widths
        for bits in (8, 4):
            qa, ab = lib.h3q_quantize_weights_affine(torch.from_numpy(w).to(dev), bits=bits)
            ya = lib.h3q_linear_affine_w8(x, qa, ab, b)["y"][rt][:, ct]
            snr[f"affine_q{bits}"] = oracle.snr_db(oracle.widen_bf16(_bits(ya)), ref)
            oq, oa, ob = oracle.quantize_affine(w[cols], bits=bits)
            yo = oracle.linear_affine(c.x_bits[rows], oracle.dequant_affine(oq, oa, ob),
                                      c.bias_bits[0][cols])["y"]
            snr[f"oracle_q{bits}"] = oracle.snr_db(oracle.widen_bf16(yo), ref)
            assert abs(snr[f"affine_q{bits}"] - snr[f"oracle_q{bits}"]) < 0.05, (name, snr)
        assert snr["affine_q8"] > snr["w8a8"] > snr["affine_q4"], (name, snr)
        report[name] = {k: round(float(v), 2) for k, v in snr.items()}
    print(f"\nSNR vs float64 (dB), W8A8 against group-wise affine: {report}")
