"""Seeded synthetic inputs for the five cascaded-reduction workloads.

This module only draws random numbers and lays them out; it holds none of the
cascade's arithmetic.  Both the CUDA path and the CPU oracle consume what it
returns, so it is the one module they share.

Recipe (every tensor is drawn from ``torch.Generator(device).manual_seed(seed)``
in the order listed; fp32 draws are cast to bf16 where the workload is bf16):

* single-row decode (fp32, D=64, L=4096): q [64], K [L, 64], V [L, 64] ~ N(0,1),
  seed 1, scale 1/sqrt(64);
* split-KV decode (bf16, B=32, H=32, L=32768, D=128): q [B, H, D], K, V
  [B, H, L, D] ~ N(0,1), seed 2, scale 1/sqrt(128).  At full size (16 GiB)
  the draw runs on the GPU (``device='cuda'``) with a CUDA generator;
* MoE routing logits [16384, 256] ~ 2*N(0,1), seed 3 (top-8) and
  [65536, 64] ~ 2*N(0,1), seed 33 (top-2);
* FP8 quant->GEMM: X [M=4096, K=7168] ~ N(0,1) with a Bernoulli(0.001) mask
  of entries multiplied by 20 (outliers), then cast to bf16, seed 4; the
  weight W [K, N=4096] ~ N(0,1) is handed over pre-quantised: per output
  column scale sw_n = fp32(max_k |W_kn| / 448) and codes from torch's own
  float8_e4m3fn cast of W / sw, stored transposed as Wq [N, K] (K contiguous);
* causal prefill (bf16, B=4, H=32, N=8192, D=128): Q, K, V ~ N(0,1), seed 5,
  scale 1/sqrt(128);
* multi-latent attention decode (bf16, B=64 sequences, H=16 query heads,
  L=32768 keys, latent width Dk=576 = 512 + 64 rotary, value width Dv=512):
  q [B, H, Dk], C [B, L, Dk] ~ N(0,1), seed 6, scale 1/sqrt(192) (the
  128 + 64 query/key head width the latent form stands in for).

Smaller parity cases use the same recipe with smaller sizes.
"""

import math

import torch

SEEDS = {"decode_f32": 1, "decode_bf16": 2, "route_256": 3, "route_64": 33,
         "quant_gemm": 4, "prefill": 5, "mla": 6}

FULL = {
    "decode_f32": dict(R=1, L=4096, D=64),
    "decode_bf16": dict(B=32, H=32, L=32768, D=128),
    "route_256": dict(T=16384, E=256, k=8),
    "route_64": dict(T=65536, E=64, k=2),
    "quant_gemm": dict(M=4096, K=7168, N=4096),
    "prefill": dict(B=4, H=32, N=8192, D=128),
    "mla": dict(B=64, H=16, L=32768, Dk=576, Dv=512),
}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def decode_inputs(R, L, D, dtype=torch.float32, seed=1, device="cpu"):
    """q [R, D], K [R, L, D], V [R, L, D] ~ N(0,1) in ``dtype``."""
    g = _gen(seed, device)
    if device == "cpu":
        q = torch.randn(R, D, generator=g).to(dtype)
        K = torch.randn(R, L, D, generator=g).to(dtype)
        V = torch.randn(R, L, D, generator=g).to(dtype)
    else:
        q = torch.randn(R, D, generator=g, device=device, dtype=dtype)
        K = torch.randn(R, L, D, generator=g, device=device, dtype=dtype)
        V = torch.randn(R, L, D, generator=g, device=device, dtype=dtype)
    return q, K, V


def decode_scale(D):
    return 1.0 / math.sqrt(D)


def routing_logits(T, E, seed=3, device="cpu"):
    """logits [T, E] fp32 ~ 2 * N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn(T, E, generator=g, device=device) * 2.0


def quant_gemm_inputs(M, K, N, seed=4, outlier_p=0.001, outlier_mult=20.0):
    """X [M, K] bf16 with outliers; (Wq [N, K] uint8 e4m3 codes, sw [N] fp32)."""
    g = _gen(seed, "cpu")
    x = torch.randn(M, K, generator=g)
    mask = torch.rand(M, K, generator=g) < outlier_p
    x = torch.where(mask, x * outlier_mult, x).to(torch.bfloat16)
    w = torch.randn(K, N, generator=g)
    sw = w.abs().amax(dim=0) / 448.0
    wq = (w / sw).to(torch.float8_e4m3fn)          # library cast of the weight
    wq = wq.t().contiguous().view(torch.uint8)     # [N, K], K contiguous
    return x, wq, sw.to(torch.float32)


def prefill_inputs(B, H, N, D, seed=5, device="cpu"):
    """Q, K, V [B, H, N, D] bf16 ~ N(0,1)."""
    g = _gen(seed, device)
    if device == "cpu":
        return tuple(torch.randn(B, H, N, D, generator=g).to(torch.bfloat16) for _ in range(3))
    return tuple(torch.randn(B, H, N, D, generator=g, device=device, dtype=torch.bfloat16)
                 for _ in range(3))


def mla_inputs(B, H, L, Dk=576, seed=6, device="cpu"):
    """q [B, H, Dk], C [B, L, Dk] bf16 ~ N(0,1) (query heads, shared latent cache)."""
    g = _gen(seed, device)
    if device == "cpu":
        q = torch.randn(B, H, Dk, generator=g).to(torch.bfloat16)
        C = torch.randn(B, L, Dk, generator=g).to(torch.bfloat16)
    else:
        q = torch.randn(B, H, Dk, generator=g, device=device, dtype=torch.bfloat16)
        C = torch.randn(B, L, Dk, generator=g, device=device, dtype=torch.bfloat16)
    return q, C


def mla_scale():
    return 1.0 / math.sqrt(192)
