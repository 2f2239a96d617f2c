"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and
the benchmark.

This module holds no arithmetic of the compression method: only random draws
and the input recipe.  The random numbers the method itself draws (the
Rademacher sign vectors and the Gaussian QJL matrix S) are produced here, once,
and passed as inputs to both the oracle and the CUDA path.

Recipe (the configurations the decode and encode paths are measured on):

* K and V head vectors: Student-t with nu = 3 per coordinate,
  Z / sqrt(chi2_3 / 3) with chi2_3 a sum of three squared normals; four fixed
  outlier channels {7, 38, 71, 102} scaled by 20; keys get RoPE (interleaved
  pairs (2i, 2i+1), theta_i = 500000^(-2i/d)) at positions 0..T-1; clamped to
  +-6.0e4 and cast to fp16.  Per (layer, kind) sub-seed = 1000*base + 2*layer
  + (0 for K, 1 for V), base = 0.
* Query: fp16 N(0, 1), seed 1.
* Page table: a random permutation of the pool's pages, seed 2.
* Sign vectors: D_K from seed 42, D_V from seed 43; bit 0 of splitmix64
  output j is the sign of coordinate j (1 = negate).
* QJL matrix S [m, d], row-major: seed 44; splitmix64 -> 53-bit uniform
  doubles -> Box-Muller in fp64 -> fp32.

splitmix64 is Steele, Lea and Flood's generator (as popularised by Vigna's
xorshift notes): state += 0x9E3779B97F4A7C15, then two xor-shift-multiply
rounds.  Box-Muller (1958): z0 = r cos(2 pi u2), z1 = r sin(2 pi u2) with
r = sqrt(-2 ln u1).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

OUTLIER_CHANNELS = (7, 38, 71, 102)
OUTLIER_SCALE = 20.0
ROPE_BASE = 500000.0
FP16_CLAMP = 6.0e4
SEED_KV_BASE = 0
SEED_QUERY = 1
SEED_PAGES = 2
SEED_SIGNS_K = 42
SEED_SIGNS_V = 43
SEED_QJL = 44

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int) -> np.ndarray:
    """The first n outputs of splitmix64 started from ``seed`` (uint64)."""
    with np.errstate(over="ignore"):
        i = np.arange(1, n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def sign_bits(seed: int, d: int) -> np.ndarray:
    """uint8 [d]; 1 means coordinate j is negated."""
    return (splitmix64(seed, d) & np.uint64(1)).astype(np.uint8)


def gaussian_matrix(seed: int, m: int, d: int) -> np.ndarray:
    """fp32 [m, d] i.i.d. N(0, 1) via splitmix64 + Box-Muller (fp64)."""
    n = m * d
    npairs = (n + 1) // 2
    u = (splitmix64(seed, 2 * npairs) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    u1 = 1.0 - u[0::2]  # (0, 1]
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * npairs)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return z[:n].reshape(m, d).astype(np.float32)


def kv_subseed(layer: int, kind: int, base: int = SEED_KV_BASE) -> int:
    return 1000 * base + 2 * layer + kind


def heavy_tailed(shape, seed: int, device="cpu") -> torch.Tensor:
    """fp32 Student-t(3) draws with the outlier channels scaled (last dim = d)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(3):
        e = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(e, e)
    t = z / torch.sqrt(chi2 / 3.0)
    t[..., list(OUTLIER_CHANNELS)] *= OUTLIER_SCALE
    return t


def apply_rope(x: torch.Tensor, positions: torch.Tensor, base: float = ROPE_BASE) -> torch.Tensor:
    """RoPE on interleaved pairs (2i, 2i+1); x [..., T, H, d], positions [T]."""
    d = x.shape[-1]
    i = torch.arange(d // 2, device=x.device, dtype=torch.float64)
    theta = base ** (-2.0 * i / d)
    ang = positions.to(torch.float64)[:, None] * theta[None, :]  # [T, d/2]
    cos = torch.cos(ang).to(torch.float32)[:, None, :]  # [T, 1, d/2]
    sin = torch.sin(ang).to(torch.float32)[:, None, :]
    xe, xo = x[..., 0::2], x[..., 1::2]
    out = torch.empty_like(x)
    out[..., 0::2] = xe * cos - xo * sin
    out[..., 1::2] = xe * sin + xo * cos
    return out


def kv_history(B: int, T: int, H: int, d: int, layer: int, kind: int, device="cpu", base: int = SEED_KV_BASE) -> torch.Tensor:
    """fp16 [B, T, H, d] K (kind 0, with RoPE at positions 0..T-1) or V (kind 1)."""
    x = heavy_tailed((B, T, H, d), kv_subseed(layer, kind, base), device)
    if kind == 0:
        x = apply_rope(x, torch.arange(T, device=device))
    return x.clamp_(-FP16_CLAMP, FP16_CLAMP).to(torch.float16)


def query(B: int, Hq: int, d: int, device="cpu", seed: int = SEED_QUERY) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((B, Hq, d), generator=g, device=device, dtype=torch.float32).to(torch.float16)


def page_permutation(num_pages: int, seed: int = SEED_PAGES) -> torch.Tensor:
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randperm(num_pages, generator=g).to(torch.int32)


@dataclasses.dataclass(frozen=True)
class Format:
    """Cache format (plain numbers, mirrored by the C structs on both sides)."""

    head_dim: int = 128
    k_bits: int = 4
    v_bits: int = 4
    k_qjl: int = 0
    qjl_m: int = 128
    page_size: int = 64
    num_kv_heads: int = 8
    norm_correct: int = 0
    qjl_scale: float = 0.0
    k_mixed: int = 0


@dataclasses.dataclass(frozen=True)
class KiviFormat:
    """Format of the KIVI-style control arm (mirrored by tq_kivi_format)."""

    head_dim: int = 128
    k_bits: int = 2
    v_bits: int = 2
    page_size: int = 64
    num_kv_heads: int = 8


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    layers: int
    batch: int
    q_heads: int
    fmt: Format
    context: int
    window: int

    @property
    def kv_heads(self) -> int:
        return self.fmt.num_kv_heads

    @property
    def comp_tokens(self) -> int:
        return max(self.context - self.window, 0)

    @property
    def win_tokens(self) -> int:
        return min(self.context, self.window)

    @property
    def pages_per_seq(self) -> int:
        P = self.fmt.page_size
        return (self.comp_tokens + P - 1) // P


@dataclasses.dataclass(frozen=True)
class EncodeWorkload:
    name: str
    layers: int
    kv_heads: int
    tokens: int
    bits: tuple
    qjl_options: tuple
    qjl_m: int
    page_size: int


# The five synthetic workloads.
SINGLE_LAYER_T2K = DecodeWorkload("single_layer_b1_h32x8_t2048_k4v4", 1, 1, 32, Format(128, 4, 4, 0, 128, 64, 8), 2048, 0)
QWEN25_3B_T16K = DecodeWorkload("qwen2.5-3b_l36_b1_h16x2_t16384_k3qjl_v4_w128", 36, 1, 16, Format(128, 3, 4, 1, 128, 64, 2), 16384, 128)
LLAMA3_8B_T32K = DecodeWorkload("llama-3-8b_l32_b16_h32x8_t32768_k4v4_w128", 32, 16, 32, Format(128, 4, 4, 0, 128, 64, 8), 32768, 128)
BULK_ENCODE_64K = EncodeWorkload("bulk_encode_l32_h8_t65536", 32, 8, 65536, (2, 3, 4), (0, 1), 128, 64)
LONG_CTX_T128K = DecodeWorkload("long_ctx_l32_b4_h32x8_t131072_k2qjl_v2_w256", 32, 4, 32, Format(128, 2, 2, 1, 128, 128, 8), 131072, 256)

# The design study's recommended first product mode ('Packed format and
# complete bit accounting': keys 3.5 bits per channel, values 3.0, last 128
# tokens fp16) at the Llama-3-8B decode shape.
LLAMA3_8B_T32K_K35V3 = DecodeWorkload("llama-3-8b_l32_b16_h32x8_t32768_k35v3_w128", 32, 16, 32,
                                      Format(128, 3, 3, 0, 128, 64, 8, k_mixed=1), 32768, 128)

DECODE_WORKLOADS = (SINGLE_LAYER_T2K, QWEN25_3B_T16K, LLAMA3_8B_T32K, LONG_CTX_T128K, LLAMA3_8B_T32K_K35V3)

# The KIVI-style control arm ('Candidate key and value algorithms', Control
# baseline arm of the design study) at the Llama-3-8B decode shape: 2-bit
# keys and values (KIVI's own width) and 4-bit (the width of the TurboQuant
# workload it is compared with), the same 128-token fp16 window.
LLAMA3_8B_T32K_KIVI2 = DecodeWorkload("llama-3-8b_l32_b16_h32x8_t32768_kivi_k2v2_w128", 32, 16, 32, KiviFormat(128, 2, 2, 64, 8),
                                      32768, 128)
LLAMA3_8B_T32K_KIVI4 = DecodeWorkload("llama-3-8b_l32_b16_h32x8_t32768_kivi_k4v4_w128", 32, 16, 32, KiviFormat(128, 4, 4, 64, 8),
                                      32768, 128)
KIVI_WORKLOADS = (LLAMA3_8B_T32K_KIVI2, LLAMA3_8B_T32K_KIVI4)


def orthogonal_matrix(seed: int, m: int, d: int) -> np.ndarray:
    """fp32 [m, d] with orthonormal rows (m <= d): the Q factor of the QR
    decomposition of gaussian_matrix(seed, d, m), signs fixed so that R has a
    positive diagonal (a Haar-distributed draw)."""
    g = gaussian_matrix(seed, d, m).astype(np.float64)
    q, r = np.linalg.qr(g)
    q = q * np.sign(np.diag(r))[None, :]
    return np.ascontiguousarray(q.T).astype(np.float32)
