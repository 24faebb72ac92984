"""Seeded, counter-based synthetic inputs shared by the CUDA path's tests and
bench and by the CPU oracle.

Nothing here computes any part of the method: it only draws numbers.

Values (Q, K, V, ConvKV weights) come from a counter hash, so any element of
any (layer, block, step, tensor) can be regenerated on its own, on the CPU
(NumPy) or on any torch device, with bit-identical results:

    key      = mix(seed, layer, block, step, tensor)
    u_i      = lowbias32(key ^ lowbias32(4*idx + i)) >> 8      (24-bit, i = 0..3)
    x (fp32) = ((u_0 + u_1 + u_2 + u_3) * 2^-24 - 2) * sqrt(3)

x is an Irwin-Hall(4) draw rescaled to mean 0 and variance 1; it stands in
for the N(0, 1) activations of the workloads.  `lowbias32` is Chris
Wellons' 32-bit integer finaliser (two multiply/xor-shift rounds,
constants 0x7feb352d and 0x846ca68b).  Every fp32 step above is a single
IEEE-754 round-to-nearest operation done in the same order on every backend.

Poses are host inputs drawn with NumPy's `default_rng(seed)`.
"""
from __future__ import annotations

import numpy as np

from .configs import StreamConfig

M32 = 0xFFFFFFFF
SQRT3_F32 = np.float32(1.7320508075688772)
TWO_POW_M24 = np.float32(2.0 ** -24)

# tensor ids used in the key
T_Q, T_K, T_V, T_CONVW = 1, 2, 3, 4


def _lowbias32_np(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint32, copy=True)
    x ^= x >> np.uint32(16)
    x *= np.uint32(0x7FEB352D)
    x ^= x >> np.uint32(15)
    x *= np.uint32(0x846CA68B)
    x ^= x >> np.uint32(16)
    return x


def _lowbias32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def stream_key(seed: int, layer: int, block: int, step: int, tensor: int) -> int:
    """32-bit key of one generated tensor."""
    k = _lowbias32_int(seed * 0x9E3779B9 + 0x632BE5AB)
    for part in (layer, block, step, tensor):
        k = _lowbias32_int(k ^ ((part + 0x68E31DA4) & M32))
    return k


def _u24_np(key: int, idx: np.ndarray, i: int) -> np.ndarray:
    c = (idx.astype(np.uint64) * 4 + i).astype(np.uint32)
    return _lowbias32_np(np.uint32(key) ^ _lowbias32_np(c)) >> np.uint32(8)


def normal_f32_np(key: int, idx: np.ndarray) -> np.ndarray:
    """fp32 draw for each flat element index in `idx` (NumPy backend)."""
    s = _u24_np(key, idx, 0).astype(np.float32) * TWO_POW_M24
    for i in (1, 2, 3):
        s = s + _u24_np(key, idx, i).astype(np.float32) * TWO_POW_M24
    return (s - np.float32(2.0)) * SQRT3_F32


def round_bf16_np(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest bf16 (ties to even); returned as fp32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32)


def tensor_np(key: int, shape, dtype: str, index_offset: int = 0,
              index_map=None) -> np.ndarray:
    """Whole tensor in row-major flat order, rounded to `dtype` ("f32"/"bf16"),
    returned as float32 values.  `index_map` optionally gives the flat indices
    to generate (for sampling a subset); otherwise all of prod(shape)."""
    if index_map is None:
        n = int(np.prod(shape))
        idx = np.arange(index_offset, index_offset + n, dtype=np.uint64)
    else:
        idx = np.asarray(index_map, dtype=np.uint64)
    x = normal_f32_np(key, idx)
    if dtype == "bf16":
        x = round_bf16_np(x)
    return x.reshape(shape) if index_map is None else x


# ---------------------------------------------------------------- torch backend
def _lowbias32_t(x):
    import torch
    m = torch.tensor(M32, dtype=torch.int64, device=x.device)
    x = x & m
    x = x ^ (x >> 16)
    x = (x * 0x7FEB352D) & m
    x = x ^ (x >> 15)
    x = (x * 0x846CA68B) & m
    x = x ^ (x >> 16)
    return x


def normal_f32_torch(key: int, idx):
    """Same draw as `normal_f32_np` on any torch device (idx: int64 tensor)."""
    import torch
    s = None
    for i in range(4):
        c = (idx * 4 + i) & M32
        u = _lowbias32_t(_lowbias32_t(c) ^ key) >> 8
        f = u.to(torch.float32) * float(TWO_POW_M24)
        s = f if s is None else s + f
    return (s - 2.0) * float(SQRT3_F32)


def tensor_torch(key: int, shape, dtype: str, device="cpu", chunk: int = 1 << 24):
    """Whole tensor of the given shape; dtype "f32" -> float32, "bf16" -> bfloat16."""
    import torch
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.float32 if dtype == "f32" else torch.bfloat16,
                      device=device)
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        idx = torch.arange(a, b, dtype=torch.int64, device=device)
        x = normal_f32_torch(key, idx)
        out[a:b] = x.to(out.dtype)
    return out.view(*shape)


# ------------------------------------------------------------------ workloads
def qkv_key(cfg: StreamConfig, layer: int, block: int, step: int, which: str) -> int:
    t = {"q": T_Q, "k": T_K, "v": T_V}[which]
    return stream_key(cfg.seed, layer, block, step, t)


def conv_weight_key(cfg: StreamConfig, layer: int, which: str) -> int:
    return stream_key(cfg.seed + 7919, layer, 0, 0, T_CONVW * 2 + (which == "v"))


def conv_weights_np(cfg: StreamConfig, layer: int) -> np.ndarray:
    """Depthwise Conv1d weights [2 (K,V)][H][D][kernel], sigma 0.2, bf16 values."""
    H, D, R = cfg.num_heads, cfg.head_dim, cfg.conv_kernel
    out = []
    for which in ("k", "v"):
        x = tensor_np(conv_weight_key(cfg, layer, which), (H, D, R), "f32")
        out.append(round_bf16_np(x * np.float32(0.2)))
    return np.stack(out)


def conv_weights_torch(cfg: StreamConfig, layer: int, device="cpu"):
    import torch
    H, D, R = cfg.num_heads, cfg.head_dim, cfg.conv_kernel
    out = []
    for which in ("k", "v"):
        x = tensor_torch(conv_weight_key(cfg, layer, which), (H, D, R), "f32", device)
        out.append((x * float(np.float32(0.2))).to(torch.bfloat16))
    return torch.stack(out)


def poses(cfg: StreamConfig, n_blocks: int | None = None) -> np.ndarray:
    """Per-block driving pose: [n_blocks, 17, 2] keypoints in [0, 1] (fp32)."""
    r = cfg.pose
    n = cfg.n_blocks if n_blocks is None else n_blocks
    rng = np.random.default_rng(r.seed)
    b = np.arange(n, dtype=np.float64)[:, None, None]
    if r.kind == "sinusoid":
        amp = rng.uniform(0.1, 0.3, size=(17, 2))
        phi = rng.uniform(0.0, 2 * np.pi, size=(17, 2))
        jumps = rng.uniform(size=n) < r.jump_prob
        new_phase = rng.uniform(0.0, 2 * np.pi, size=n)
        psi = np.zeros(n)
        cur = 0.0
        for i in range(n):
            if jumps[i]:
                cur = new_phase[i]
            psi[i] = cur
        noise = rng.normal(0.0, r.noise, size=(n, 17, 2))
        kp = 0.5 + amp * np.sin(2 * np.pi * b / r.period + phi + psi[:, None, None]) + noise
    elif r.kind == "clusters":
        centres = rng.uniform(0.2, 0.8, size=(r.n_clusters, 17, 2))
        perm = rng.permutation(r.n_clusters)
        noise = rng.normal(0.0, r.noise, size=(n, 17, 2))
        kp = centres[perm[np.arange(n) % r.n_clusters]] + noise
    else:
        raise ValueError(r.kind)
    return np.clip(kp, 0.0, 1.0).astype(np.float32)
