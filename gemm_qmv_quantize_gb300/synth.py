"""Seeded synthetic inputs for the quantized skinny matmul path.

This module only draws random numbers and stores them in the packed layouts the
kernels read; it contains none of the method's arithmetic (no decoding, no dot
products, no quantization of activations). Both the CUDA path and the CPU oracle
are fed from here, so nothing in the oracle's inputs comes from the kernels.

Layouts (all row-major, little-endian):
  Q4_0   [N][K/32] blocks of 18 B: fp16 scale d, then 16 bytes of nibbles.
  NVFP4  codes [N][K/2] (k even in the low nibble), E4M3 scales [N][K/16],
         one fp32 per-tensor scale.
  FP8    [N][K] E4M3 bytes, fp32 per-row scale [N].
  Activations fp32 [M][K] (Q4_0 path, quantized to Q8_1 per call) or fp16 [M][K].

Distributions (the workloads of the pages: Llama-2-7B Q4_0 decode in "Machine
Learning on NVIDIA CMP", section "llama.cpp results"; Qwen3.8-27B mixed NVFP4/FP8
in "v100-skinny README", sections "How QPN works" and "Native mixed-precision
checkpoint path"):
  Q4_0 nibbles uniform on 0..15; d = fp16(|N(0,1)| * 0.01).
  NVFP4 codes uniform over the 16 codes; scale = E4M3(|N(0,1)| * 0.5); g = 0.01.
  FP8 weights E4M3(N(0,1)); row scale 0.02.
  Activations N(0,1); optional fp16 outliers of magnitude 1e3..6e4.
The fp16 and E4M3 roundings of the drawn values are PyTorch's own conversions.
"""
from __future__ import annotations

import torch

Q4_0_BLOCK_BYTES = 18
Q8_1_BLOCK_BYTES = 36
NVFP4_GLOBAL_SCALE = 0.01
FP8_ROW_SCALE = 0.02


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def q4_0_weights(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """Q4_0 matrix as uint8 [N, K/32*18]."""
    assert K % 32 == 0
    nb = K // 32
    g = _gen(seed, device)
    nibbles = torch.randint(0, 256, (N, nb, 16), generator=g, dtype=torch.uint8, device=device)
    d = (torch.randn((N, nb), generator=g, device=device).abs_() * 0.01).to(torch.float16)
    out = torch.empty((N, nb, Q4_0_BLOCK_BYTES), dtype=torch.uint8, device=device)
    out[:, :, 0:2] = d.view(torch.uint8).view(N, nb, 2)
    out[:, :, 2:] = nibbles
    return out.view(N, nb * Q4_0_BLOCK_BYTES)


def q4_k_weights(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """Q4_K matrix as uint8 [N, K/256*144]: per 256-weight super-block fp16 d and
    dmin = |N(0,1)| * 0.001 and * 0.002, then 12 uniformly random bytes (the packed
    6-bit sub-block scales and minimums: every byte pattern is valid) and 128
    uniformly random bytes of nibbles."""
    assert K % 256 == 0
    ns = K // 256
    g = _gen(seed, device)
    body = torch.randint(0, 256, (N, ns, 140), generator=g, dtype=torch.uint8, device=device)
    d = (torch.randn((N, ns, 2), generator=g, device=device).abs_() *
         torch.tensor([0.001, 0.002], device=device)).to(torch.float16)
    out = torch.empty((N, ns, 144), dtype=torch.uint8, device=device)
    out[:, :, 0:4] = d.view(torch.uint8).view(N, ns, 4)
    out[:, :, 4:] = body
    return out.view(N, ns * 144)


def nvfp4_weights(N: int, K: int, seed: int, device="cpu"):
    """(codes uint8 [N, K/2], scales uint8 [N, K/16] E4M3, global scale float)."""
    assert K % 16 == 0
    g = _gen(seed, device)
    codes = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.uint8, device=device)
    s = torch.randn((N, K // 16), generator=g, device=device).abs_() * 0.5
    scales = s.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scales, NVFP4_GLOBAL_SCALE


def fp8_weights(N: int, K: int, seed: int, device="cpu"):
    """(w uint8 [N, K] E4M3, row_scale fp32 [N])."""
    g = _gen(seed, device)
    w = torch.randn((N, K), generator=g, device=device).to(torch.float8_e4m3fn).view(torch.uint8)
    rs = torch.full((N,), FP8_ROW_SCALE, dtype=torch.float32, device=device)
    return w, rs


def activations_f32(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn((M, K), generator=g, device=device, dtype=torch.float32)


def activations_f16(M: int, K: int, seed: int, device="cpu", outliers: int = 0) -> torch.Tensor:
    """fp16 [M, K] ~ N(0,1); ``outliers`` entries per row set to +-U(1e3, 6e4)."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outliers:
        idx = torch.randint(0, K, (M, outliers), generator=g, device=device)
        mag = torch.rand((M, outliers), generator=g, device=device) * (6.0e4 - 1.0e3) + 1.0e3
        sign = torch.randint(0, 2, (M, outliers), generator=g, device=device) * 2 - 1
        x.scatter_(1, idx, mag * sign)
    return x.to(torch.float16)


def sample_rows(N: int, count: int, seed: int) -> torch.Tensor:
    """Sorted distinct row indices: the first, the last and ``count - 2`` random rows."""
    count = min(count, N)
    g = _gen(seed, "cpu")
    picks = torch.randperm(N, generator=g)[: max(count - 2, 0)]
    rows = torch.cat([torch.tensor([0, N - 1]), picks]).unique()
    return rows[:count] if rows.numel() > count else rows
