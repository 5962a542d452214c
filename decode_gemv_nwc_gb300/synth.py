"""Seeded synthetic inputs shaped like the workloads the NWC pages describe.

This module draws random numbers and rounds them to BF16 bit patterns. It
holds none of the method's arithmetic (no ranking, coding, decoding or
matvec), so both the CUDA path and the CPU oracle may take their inputs from
it. Every function is deterministic for a given seed and device.

Weights and activations are returned as BF16 bit patterns (``uint16`` numpy
arrays on the host, ``int16`` torch tensors on a device). Values are drawn in
FP32 and rounded to BF16 by round-to-nearest-even (torch's conversion).

Workloads (named by what they are):
  * single 64x512 matrix, N(0, 0.02) plus 33 outliers of +-U(1, 8) and 8 exact
    zeros, activations N(0, 1) of length 512;
  * square 4096x4096 and odd 4095x4100 matrices, N(0, 0.02);
  * a 36-layer decoder stack shaped like a 4B model (q, k, v, o, gate, up,
    down) with a per-layer sigma of 0.02 * U(0.5, 2);
  * a 151936x2560 tied embedding / lm_head table and 4096 token ids;
  * gate 9728x2560 and down 2560x9728 matrices for the fp8 variant.
"""
from __future__ import annotations

import numpy as np
import torch

SIGMA = 0.02

# (name, N out features, K in features) of one decoder layer of the stack.
LAYER_SHAPES = (
    ("q", 4096, 2560),
    ("k", 1024, 2560),
    ("v", 1024, 2560),
    ("o", 2560, 4096),
    ("gate", 9728, 2560),
    ("up", 9728, 2560),
    ("down", 2560, 9728),
)
N_LAYERS = 36
VOCAB, HIDDEN = 151936, 2560


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _to_bits(t: torch.Tensor):
    """FP32 tensor -> BF16 bit patterns (RNE); numpy uint16 on the host."""
    b = t.to(torch.bfloat16).view(torch.int16)
    if b.device.type == "cpu":
        return b.numpy().view(np.uint16)
    return b


def normal_bf16(shape, sigma: float, seed: int, device="cpu"):
    """BF16 bit patterns of N(0, sigma^2) draws."""
    g = _gen(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return _to_bits(t * sigma)


def activations_bf16(k: int, seed: int, device="cpu"):
    """Activation vector x of length k, N(0, 1), as BF16 bit patterns."""
    return normal_bf16((k,), 1.0, seed, device)


def small_matrix_with_outliers(seed: int = 0):
    """64x512 N(0, 0.02) with 0.1% of entries (33) replaced by +-U(1, 8) and
    8 further distinct entries set to exact zero. Returns uint16 (64, 512)."""
    n, k = 64, 512
    g = _gen(seed)
    w = torch.randn(n, k, generator=g, dtype=torch.float32) * SIGMA
    perm = torch.randperm(n * k, generator=g)
    n_out = int(round(0.001 * n * k))  # 33
    out_pos = perm[:n_out]
    zero_pos = perm[n_out:n_out + 8]
    mag = 1.0 + 7.0 * torch.rand(n_out, generator=g)
    sgn = torch.where(torch.rand(n_out, generator=g) < 0.5, -1.0, 1.0)
    flat = w.view(-1)
    flat[out_pos] = mag * sgn
    flat[zero_pos] = 0.0
    return _to_bits(w)


def layer_sigmas(seed_base: int = 100):
    """Per-layer sigma = 0.02 * U(0.5, 2), one draw per layer (seed 100+layer)."""
    out = []
    for layer in range(N_LAYERS):
        g = _gen(seed_base + layer)
        u = torch.rand(1, generator=g).item()
        out.append(SIGMA * (0.5 + 1.5 * u))
    return out


def layer_matrix(layer: int, name: str, device="cpu"):
    """One matrix of the 36-layer stack, BF16 bits. Seed = 100 + layer, with
    the matrix's index in the layer added so the seven matrices differ."""
    idx = [s[0] for s in LAYER_SHAPES].index(name)
    _, n, k = LAYER_SHAPES[idx]
    sigma = layer_sigmas()[layer]
    return normal_bf16((n, k), sigma, 100 + layer + 1000 * (idx + 1), device)


def token_ids(n_ids: int, vocab: int, seed: int = 8):
    """Token ids drawn uniformly from [0, vocab), int32 numpy array."""
    g = _gen(seed)
    return torch.randint(0, vocab, (n_ids,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact: append 16 zero bits)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
