"""Seeded synthetic inputs for the W8A8 INT8 projection Linear.

This module is the one thing the CPU oracle and the CUDA path share: it draws
random tensors and holds none of the method's arithmetic (no quantisation, no
GEMM, no epilogue).  Both sides consume the identical bytes it returns.

The shapes are the MiniMax-H3 DiT projection shapes at the model's native
hidden width 5376 (Q, K, V, attention-out 5376->5376; FC1 5376->21504;
FC2 21504->5376), as described in "feat(mps): support MiniMax-H3 INT8
inference on Apple M5" (ModelTC/LightX2V pull request #1672), opening
description: the ``dit_proj`` profile quantises FC1, FC2, Q, K, V and the
attention output of all 50 main blocks, 300 Linear operators.

Recipe (numpy ``default_rng(seed)``, PCG64), drawn in this order:
  1. X ~ N(0, 1) as float32 (or SiLU(z), z ~ N(0, 1), for the FC2 input);
  2. an outlier mask, Bernoulli(p) from ``rng.random`` (only where the
     workload has outliers), the masked entries multiplied by a factor;
  3. the FP32 weights ~ N(0, std), one per Linear, in the order given;
  4. the biases ~ N(0, 0.1), one per Linear, in the same order.
X and the biases are rounded to BF16 (round-to-nearest-even, done by torch's
CPU dtype conversion) and returned as uint16 bit patterns.

The 300-Linear sweep is too large to draw on a host in test time (17.3 G
weight elements), so its tensors come from torch's counter-based CUDA
generator instead; ``sweep_*`` below documents that recipe.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

H3_WIDTH = 5376          # MiniMax-H3 DiT hidden width (native K)
H3_MLP_WIDTH = 21504     # FC1 output / FC2 input width
H3_BLOCKS = 50           # main transformer blocks


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 (round-to-nearest-even) via torch's CPU cast; uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def sha256(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()[:16]


@dataclass
class LinearCase:
    """One Linear's inputs: X (BF16 bits), FP32 weight, BF16 bias bits."""
    name: str
    x_bits: np.ndarray            # uint16 [M, K]
    w: list                       # list of float32 [N, K], one per Linear
    bias_bits: list               # list of uint16 [N], one per Linear
    linear_names: list = field(default_factory=list)

    @property
    def M(self) -> int:
        return int(self.x_bits.shape[0])

    @property
    def K(self) -> int:
        return int(self.x_bits.shape[1])

    def hashes(self) -> dict:
        h = {"x": sha256(self.x_bits)}
        for nm, w, b in zip(self.linear_names, self.w, self.bias_bits):
            h[nm + ".w"] = sha256(w)
            h[nm + ".bias"] = sha256(b)
        return h


def _x_normal(rng, M, K, outlier_p, outlier_mul):
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outlier_p > 0:
        mask = rng.random((M, K), dtype=np.float32) < np.float32(outlier_p)
        x[mask] *= np.float32(outlier_mul)
    return x


def _x_silu(rng, M, K):
    z = rng.standard_normal((M, K), dtype=np.float32)
    # SiLU(z) = z * sigmoid(z), evaluated in float64 then cast (input prep only)
    z64 = z.astype(np.float64)
    return (z64 / (1.0 + np.exp(-z64))).astype(np.float32)


def _weights(rng, shapes_std):
    ws = [rng.standard_normal(shape, dtype=np.float32) * np.float32(std)
          for shape, std in shapes_std]
    bs = [to_bf16_bits(rng.standard_normal(shape[0], dtype=np.float32) * np.float32(0.1))
          for shape, _ in shapes_std]
    return ws, bs


def make_linear(M, N, K, seed, x_kind="normal", outlier_p=0.0, outlier_mul=1.0,
                w_std=0.02, n_linears=1, names=None) -> LinearCase:
    """Generic seeded case: any shape, same recipe as the named workloads."""
    rng = np.random.default_rng(seed)
    if x_kind == "silu":
        x = _x_silu(rng, M, K)
    else:
        x = _x_normal(rng, M, K, outlier_p, outlier_mul)
    ws, bs = _weights(rng, [((N, K), w_std)] * n_linears)
    names = names or [f"linear{i}" for i in range(n_linears)]
    return LinearCase("custom", to_bf16_bits(x), ws, bs, names)


# --- the five named workloads -------------------------------------------------

def tiny() -> LinearCase:
    """X [64, 5376] N(0,1) with 1% of entries x20; W [256, 5376] N(0, 0.02); seed 0."""
    c = make_linear(64, 256, H3_WIDTH, seed=0, outlier_p=0.01, outlier_mul=20.0, w_std=0.02)
    c.name = "tiny"
    return c


def attn(M: int = 8192) -> LinearCase:
    """X [8192, 5376] N(0,1) + 0.5% outliers x30; Q, K, V, O weights [5376, 5376]
    N(0, 0.02) drawn in that order, then the four biases; seed 1."""
    c = make_linear(M, H3_WIDTH, H3_WIDTH, seed=1, outlier_p=0.005, outlier_mul=30.0,
                    w_std=0.02, n_linears=4, names=["q", "k", "v", "o"])
    c.name = "attn"
    return c


def fc1(M: int = 32767) -> LinearCase:
    """X [32767, 5376] N(0,1) (ragged M); W [21504, 5376] N(0, 0.015); seed 2."""
    c = make_linear(M, H3_MLP_WIDTH, H3_WIDTH, seed=2, w_std=0.015, names=["fc1"])
    c.name = "fc1"
    return c


def fc2(M: int = 32768) -> LinearCase:
    """X [32768, 21504] = SiLU(z), z ~ N(0,1); W [5376, 21504] N(0, 0.01); seed 3."""
    c = make_linear(M, H3_WIDTH, H3_MLP_WIDTH, seed=3, x_kind="silu", w_std=0.01,
                    names=["fc2"])
    c.name = "fc2"
    return c


# --- H3-Image operator shapes at 4096 tokens (a secondary workload) ----------------
# "MLX implementation and experiment report" (MiniMax-H3-Image-mlx), Operator
# tuning: the QKV GEMM 5376 -> 21504, the fused gate/up GEMM 5376 -> 28672 and
# the down GEMM 14336 -> 5376, timed there at 4096 tokens on synthetic BF16
# inputs.  Here: X ~ N(0,1), W ~ N(0, 0.02), bias ~ N(0, 0.1).

IMAGE_TOKENS = 4096


def image_qkv(M: int = IMAGE_TOKENS) -> LinearCase:
    """X [4096, 5376] N(0,1); W [21504, 5376] N(0, 0.02); seed 5."""
    c = make_linear(M, 21504, H3_WIDTH, seed=5, w_std=0.02, names=["qkv"])
    c.name = "image_qkv"
    return c


def image_gate_up(M: int = IMAGE_TOKENS) -> LinearCase:
    """X [4096, 5376] N(0,1); W [28672, 5376] N(0, 0.02); seed 6."""
    c = make_linear(M, 28672, H3_WIDTH, seed=6, w_std=0.02, names=["gate_up"])
    c.name = "image_gate_up"
    return c


def image_down(M: int = IMAGE_TOKENS) -> LinearCase:
    """X [4096, 14336] N(0,1); W [5376, 14336] N(0, 0.02); seed 7."""
    c = make_linear(M, H3_WIDTH, 14336, seed=7, w_std=0.02, names=["down"])
    c.name = "image_down"
    return c


# --- the 300-Linear sweep (device-generated) -------------------------------------

SWEEP_M = 75647
SWEEP_LINEARS = (("q", H3_WIDTH, H3_WIDTH), ("k", H3_WIDTH, H3_WIDTH),
                 ("v", H3_WIDTH, H3_WIDTH), ("o", H3_WIDTH, H3_WIDTH),
                 ("fc1", H3_MLP_WIDTH, H3_WIDTH), ("fc2", H3_WIDTH, H3_MLP_WIDTH))


def _seed_of(*path: int) -> int:
    """A 63-bit torch generator seed from numpy's SeedSequence(path)."""
    ss = np.random.SeedSequence(list(path))
    return int(ss.generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def _sweep_seed(*path: int) -> int:
    return _seed_of(4, *path)


def sweep_x(K: int, device, M: int = SWEEP_M):
    """Sweep activations [M, K] (K = 5376 or 21504) as a torch BF16 tensor on
    ``device``: N(0,1) with 0.5% of entries x30, from a torch generator seeded
    by SeedSequence([4, K])."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(_sweep_seed(K))
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    mask = torch.rand((M, K), generator=g, device=device, dtype=torch.float32) < 0.005
    x = torch.where(mask, x * 30.0, x)
    return x.to(torch.bfloat16)


def sweep_weight(block: int, j: int, device):
    """Block ``block``, Linear ``j`` of SWEEP_LINEARS: FP32 weight [N, K] ~ N(0, 0.02)
    and BF16 bias [N] ~ N(0, 0.1), from a torch generator seeded by
    SeedSequence([4, block, j])."""
    import torch
    _, N, K = SWEEP_LINEARS[j]
    g = torch.Generator(device=device)
    g.manual_seed(_sweep_seed(block, j))
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * 0.02
    b = (torch.randn((N,), generator=g, device=device, dtype=torch.float32) * 0.1).to(torch.bfloat16)
    return w, b


# --- fc1 / fc2 drawn on the device (bench timing only) ----------------------------

def device_case(name: str, device):
    """The fc1 or fc2 workload with the same shapes and distributions as
    ``fc1()`` / ``fc2()``, drawn on ``device`` by torch's counter-based CUDA
    generator (seeded by SeedSequence([seed, 1]), seed 2 or 3) instead of
    numpy on the host, where a 32768 x 21504 draw takes tens of seconds.  Used
    where only the distribution matters (timing: the exactness checks of the
    GEMM depend on the norms of the coded rows, which these draws share with
    the host recipe); parity tests use the host recipe's bytes.  Returns
    (X BF16 [M, K], W FP32 [N, K], bias BF16 [N]) on ``device``."""
    import torch
    if name == "fc1":
        M, N, K, seed, std = 32767, H3_MLP_WIDTH, H3_WIDTH, 2, 0.015
    elif name == "fc2":
        M, N, K, seed, std = 32768, H3_WIDTH, H3_MLP_WIDTH, 3, 0.01
    else:
        raise ValueError(f"device_case: fc1 or fc2, not {name!r}")
    g = torch.Generator(device=device)
    g.manual_seed(_seed_of(seed, 1))
    z = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if name == "fc2":
        z = z * torch.sigmoid(z)            # SiLU of the normal draw (input preparation)
    x = z.to(torch.bfloat16)
    del z
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * std
    b = (torch.randn((N,), generator=g, device=device, dtype=torch.float32) * 0.1).to(torch.bfloat16)
    return x, w, b


WORKLOADS = {"tiny": tiny, "attn": attn, "fc1": fc1, "fc2": fc2, "image_qkv": image_qkv,
             "image_gate_up": image_gate_up, "image_down": image_down}
