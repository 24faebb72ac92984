"""Worker side of the oracle process pool used by the full-shape GPU parity
tests: one head group of one chunk-attention call.  Imports only the oracle,
so a spawned worker starts without torch or the CUDA library."""
from oracle import stream as ostream


def attend(task):
    """task = (stream config, oracle Context, q [T, h, D], {block: (k, v)},
    memory (k, v) or None, query rows or None) -> O [rows, h, D] (fp64)."""
    sc, ctx, q, kv, mem, rows = task
    return ostream.chunk_attention(sc, ctx, q, lambda b: kv[b], mem=mem, rows=rows)
