"""CPU oracle for block-causal chunk attention over a bounded KV cache.

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
CPU-baseline / reference legs of `bench.py` may import or run this package.
It shares no code with the CUDA path: plain NumPy, fp64 unless a step's
rounding is part of what is being checked (stored bf16 / e4m3 values), and
no blocking, fusion or reordering beyond the definitions it restates.

Sources (web pages on the subject):
  * "LiveAnimate: 实时稳定长时流式人体动画" (ai-feeds.com), sections 方法 and
    实验: PR-Sink = static sink (first generated block, kept forever) +
    dynamic sink (history blocks retrieved by pose similarity) + rolling
    window of the 3 most recent blocks; block-causal generation where each
    block depends only on the reference and earlier blocks; cache size and
    per-block latency do not grow with stream length.
  * "Soul App开源实时数字人生成框架SoulX-LiveAct详解" (youleyou.com), section
    技术内核: ConvKV memory keeps the most recent frames' K/V exact and
    compresses older K/V with a 1D convolution (about 5:1) into fixed-length
    memory whose RoPE positions are reset; FP8 KV cache (上手实践指南).

Where the pages leave a step open, the reading taken is written next to the
function that takes it.

Parity status of each function (what pins it in tests/test_oracle_*.py):
  pose.descriptor / pose.cosine_scores / pose.select_topk : pinned (scipy
                           cosine distance, identity / translation / scale,
                           brute-force top-k with ties, whole-stream brute force)
  rope.rotate            : pinned (complex multiplication for the default and
                           explicit (t, h, w) splits, norm, identity, shift,
                           closed form)
  rope.block_positions   : pinned (hand-written raster list)
  attention.softmax_attention : pinned (torch SDPA / scipy softmax, uniform V)
  stream.plan_*          : pinned (constant KV length, window/sink invariants)
  stream.context_kv / chunk_attention : pinned (positions typed out by hand
                           for PR-Sink slots and for the ConvKV memory at
                           (j, 0, 0); the e4m3 branch reduces to the bf16
                           branch on exactly representable blocks, and a key
                           turned twice fails that pin; zero query -> mean of
                           V; shift / slot-permutation invariance; library
                           attention without RoPE)
  stream.rotate_within_block_f32 / fp8_store : pinned (fp64 rotation within
                           fp32 rounding; per-head scales)
  convkv.*               : pinned (torch conv1d, closed-form weights, FIFO cap)
  e4m3.*                 : pinned (format table, torch float8 cast, RNE ties)
No function is left unpinned.
"""
