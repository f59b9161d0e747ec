"""Seeded synthetic inputs shared by the tests, the smoke run and the benchmark.

This module only draws numbers: Gaussian tensors from numpy's PCG64 stream (host) or
from torch's seeded CUDA generator (device, for workloads too large to draw on the
host), plus the round-to-nearest-even narrowing that turns them into bf16 values.
It holds none of the attention or retrieval arithmetic, and it imports neither the
kernels' binding nor the oracle, so both sides can take their inputs from it.

Host draws return float64 arrays whose values are exactly representable in the
storage dtype ("f32" or "bf16"), so a float64 consumer sees precisely the numbers the
device sees.
"""
from __future__ import annotations

import numpy as np

CHUNK = 64  # tokens per chunk (fixed at 64 by the method)


def _rng(seed: int, stream: int) -> np.random.Generator:
    # One independent PCG64 stream per (seed, tensor id).
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def bf16_bits_from_f32(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return u.astype(np.uint16)


def f64_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def quantize(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 draws to the storage dtype and return them widened back to float64."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return x32.astype(np.float64)
    if dtype == "bf16":
        return f64_from_bf16_bits(bf16_bits_from_f32(x32))
    raise ValueError(f"unknown dtype {dtype!r}")


def normal(seed: int, stream: int, shape, std: float = 1.0, dtype: str = "f32") -> np.ndarray:
    """N(0, std^2) draws, rounded to `dtype`, returned as float64."""
    x = _rng(seed, stream).standard_normal(size=tuple(shape)) * std
    return quantize(x, dtype)


def integers(seed: int, stream: int, low: int, high: int, shape) -> np.ndarray:
    return _rng(seed, stream).integers(low, high, size=tuple(shape))


# Stream ids, so that every tensor of a workload has its own reproducible draw.
S_Q, S_K, S_V, S_DO, S_QL, S_KL, S_Q2, S_KL2, S_DO2, S_PLANT, S_DSC = range(11)


def gca_inputs(seed, B, nQ, nC, H, dh, std, dtype, with_grad=True):
    """Q [B, nQ*64, H, dh], K/V [B, nC*64, H, dh], dO like Q (float64 values)."""
    out = {
        "q": normal(seed, S_Q, (B, nQ * CHUNK, H, dh), std, dtype),
        "k": normal(seed, S_K, (B, nC * CHUNK, H, dh), std, dtype),
        "v": normal(seed, S_V, (B, nC * CHUNK, H, dh), std, dtype),
    }
    if with_grad:
        out["do"] = normal(seed, S_DO, (B, nQ * CHUNK, H, dh), std, dtype)
    return out


def landmark_inputs(seed, B, nQ, nC, D, dtype, std=1.0):
    """Query landmarks [B, nQ, D] and key landmarks [B, nC, D] (float64 values)."""
    return {
        "q_lmk": normal(seed, S_QL, (B, nQ, D), std, dtype),
        "k_lmk": normal(seed, S_KL, (B, nC, D), std, dtype),
    }


def planted_landmarks(seed, B, nC, D, dtype):
    """Decode-time landmarks: one query landmark per sequence and nC past landmarks,
    all N(0,1), with one past chunk per sequence set equal to the query landmark."""
    lm = landmark_inputs(seed, B, 1, nC, D, dtype)
    jstar = integers(seed, S_PLANT, 0, nC, (B,))
    for b in range(B):
        lm["k_lmk"][b, jstar[b]] = lm["q_lmk"][b, 0]
    lm["jstar"] = jstar
    return lm


# ---------------------------------------------------------------------------
# Chunk encoder: input rows and synthetic weights.
# ---------------------------------------------------------------------------

S_ENC_X = 30  # stream ids 30.. belong to the encoder
ENC_MATRICES = {"w_qkv": (3, 1), "w_o": (1, 1), "w_1": (4, 1), "w_2": (1, 4), "w_kv": (2, 1)}  # (rows, cols) in units of d
ENC_VECTORS = {"ln1_g": 1, "ln1_b": 1, "b_qkv": 3, "b_o": 1, "ln2_g": 1, "ln2_b": 1, "b_1": 4, "b_2": 1}  # length in units of d


def encoder_inputs(seed, B, nC, d, dtype, std=1.0):
    """Encoder input x [B, nC * 65, d]: per chunk its 64 token rows, then its LMK row."""
    return normal(seed, S_ENC_X, (B, nC * (CHUNK + 1), d), std, dtype)


def encoder_params(seed, d, dtype, w_scale=1.0):
    """Synthetic encoder weights (float64 values).  Matrices are N(0, w_scale^2 / fan_in)
    rounded to `dtype`, so that every projection keeps its input's scale; biases are
    N(0, 0.02^2) and LayerNorm gains 1 + N(0, 0.1^2), shifts N(0, 0.1^2), all float32."""
    p = {}
    for n, (name, (r, c)) in enumerate(sorted(ENC_MATRICES.items())):
        p[name] = normal(seed, S_ENC_X + 1 + n, (r * d, c * d), w_scale / (c * d) ** 0.5, dtype)
    for n, (name, r) in enumerate(sorted(ENC_VECTORS.items())):
        std = 0.02 if name.startswith("b_") else 0.1
        v = normal(seed, S_ENC_X + 10 + n, (r * d,), std, "f32")
        p[name] = quantize(1.0 + v, "f32") if name.endswith("_g") else v
    return p


# ---------------------------------------------------------------------------
# Device-side draws for the full-size workloads (hundreds of MB to tens of GB).
# ---------------------------------------------------------------------------

def device_normal(seed: int, stream: int, shape, std, torch_dtype, device="cuda"):
    """Seeded N(0, std^2) tensor drawn directly on the device with torch's generator."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1000003 + int(stream)) & 0x7FFFFFFFFFFFFFFF)
    if torch_dtype == torch.float32:
        t = torch.empty(tuple(shape), dtype=torch.float32, device=device)
        t.normal_(0.0, float(std), generator=g)
        return t
    # Fill in slices so that a 50 GB bf16 tensor never needs a 100 GB float32 temporary.
    out = torch.empty(tuple(shape), dtype=torch_dtype, device=device)
    o = out.view(-1)
    step = 1 << 28
    tmp = torch.empty(min(step, max(o.numel(), 1)), dtype=torch.float32, device=device)
    for s in range(0, o.numel(), step):
        n = min(step, o.numel() - s)
        tmp[:n].normal_(0.0, float(std), generator=g)
        o[s:s + n].copy_(tmp[:n])
    return out
