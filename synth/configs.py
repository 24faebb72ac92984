"""Workload shapes for the five synthetic streams.

This module holds sizes only: no step of the attention, retrieval or
compression arithmetic lives here.  Both the CUDA path (through its Python
binding) and the CPU oracle read these shapes, which is why they sit in a
module of their own.

Shapes follow the streams the pages describe:
  * LiveAnimate (ai-feeds.com, "方法"): PR-Sink = static sink (first block) +
    pose-retrieved dynamic sink + rolling window of the 3 most recent blocks.
  * SoulX-LiveAct (youleyou.com, "技术内核"): ConvKV memory, exact recent K/V,
    older K/V compressed about 5:1 by a 1D convolution into fixed memory with
    RoPE positions reset; FP8 KV cache ("上手实践指南").
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class PoseRecipe:
    """How the per-block driving pose (17 2D keypoints in [0, 1]) is drawn."""
    kind: str                 # "sinusoid" | "clusters"
    period: int = 8           # blocks per pose cycle (sinusoid)
    noise: float = 0.01       # std of the additive gaussian noise
    jump_prob: float = 0.0    # per-block probability of a random phase jump
    n_clusters: int = 0       # number of distinct pose clusters (clusters)
    seed: int = 0


@dataclass(frozen=True)
class StreamConfig:
    name: str
    num_layers: int
    num_heads: int
    head_dim: int
    frames_per_block: int     # latent frames per block (F)
    grid_h: int               # latent patch rows
    grid_w: int               # latent patch columns
    policy: str               # "prsink" | "convkv"
    static_sink: int          # 1: the first generated block is kept forever
    dyn_topk: int             # k of the pose-retrieved dynamic sink
    window: int               # rolling window of exact recent blocks
    n_blocks: int             # stream length
    n_steps: int              # denoising steps per block (attention calls per layer)
    qkv_dtype: str            # "f32" | "bf16"
    kv_dtype: str             # cache storage: "f32" | "bf16" | "e4m3"
    pose: PoseRecipe = field(default_factory=lambda: PoseRecipe("sinusoid"))
    conv_kernel: int = 5
    conv_stride: int = 5
    mem_slots: int = 4096
    rope_theta: float = 10000.0
    history_mode: str = "resident"   # "resident" | "external"
    seed: int = 0
    rope_dims: tuple | None = None   # explicit (t, h, w) split of the head dim

    @property
    def tokens_per_block(self) -> int:
        return self.frames_per_block * self.grid_h * self.grid_w

    @property
    def pose_dim(self) -> int:
        return 34

    @property
    def softmax_scale(self) -> float:
        return self.head_dim ** -0.5

    @property
    def rope_split(self) -> tuple[int, int, int]:
        """Head-dim split into (t, h, w) rotary parts: w = h = 2*floor(D/6)
        unless rope_dims gives one."""
        if self.rope_dims:
            return tuple(self.rope_dims)
        d = self.head_dim
        hw = 2 * (d // 6)
        return d - 2 * hw, hw, hw

    def with_(self, **kw) -> "StreamConfig":
        from dataclasses import replace
        return replace(self, **kw)


# Tiny CPU-checkable stream: 2 heads x 64, one 8x8 latent frame per block.
C1_TINY = StreamConfig(
    name="c1_tiny", num_layers=1, num_heads=2, head_dim=64,
    frames_per_block=1, grid_h=8, grid_w=8, policy="prsink",
    static_sink=1, dyn_topk=1, window=3, n_blocks=24, n_steps=1,
    qkv_dtype="f32", kv_dtype="f32",
    pose=PoseRecipe("sinusoid", period=8, noise=0.01, seed=0))

# Mid stream: 12 heads x 128, 2 frames of 26x30 patches.
C2_MID = StreamConfig(
    name="c2_mid", num_layers=1, num_heads=12, head_dim=128,
    frames_per_block=2, grid_h=26, grid_w=30, policy="prsink",
    static_sink=1, dyn_topk=1, window=3, n_blocks=64, n_steps=1,
    qkv_dtype="bf16", kv_dtype="bf16",
    pose=PoseRecipe("sinusoid", period=12, noise=0.01, seed=0))

# 14B-DiT-shaped chunk attention: 40 heads x 128, 3 frames of 30x52 patches
# (480x832 video, 8x VAE, 2x2 patches), 40 layers, 3 denoising steps.
C3_14B = StreamConfig(
    name="c3_14b", num_layers=40, num_heads=40, head_dim=128,
    frames_per_block=3, grid_h=30, grid_w=52, policy="prsink",
    static_sink=1, dyn_topk=2, window=3, n_blocks=3600, n_steps=3,
    qkv_dtype="bf16", kv_dtype="bf16",
    pose=PoseRecipe("sinusoid", period=30, noise=0.01, jump_prob=0.01, seed=0),
    history_mode="external")

# ConvKV at 14B shape: 720x416 video -> 26x45 patches x 3 frames.
C4_CONVKV = StreamConfig(
    name="c4_convkv", num_layers=40, num_heads=40, head_dim=128,
    frames_per_block=3, grid_h=26, grid_w=45, policy="convkv",
    static_sink=0, dyn_topk=0, window=3, n_blocks=1000, n_steps=3,
    qkv_dtype="bf16", kv_dtype="bf16",
    pose=PoseRecipe("sinusoid", period=30, noise=0.01, seed=0),
    conv_kernel=5, conv_stride=5, mem_slots=4096)

# Long-stream FP8 stress: c3 shapes, e4m3 K/V, top-4 over 10000 blocks of
# 50 repeating pose clusters.
C5_FP8 = StreamConfig(
    name="c5_fp8", num_layers=40, num_heads=40, head_dim=128,
    frames_per_block=3, grid_h=30, grid_w=52, policy="prsink",
    static_sink=1, dyn_topk=4, window=3, n_blocks=10000, n_steps=3,
    qkv_dtype="bf16", kv_dtype="e4m3",
    pose=PoseRecipe("clusters", noise=0.02, n_clusters=50, seed=0),
    history_mode="external")

CONFIGS = {c.name: c for c in (C1_TINY, C2_MID, C3_14B, C4_CONVKV, C5_FP8)}
