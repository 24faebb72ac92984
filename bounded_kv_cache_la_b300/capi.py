"""ctypes binding of the C ABI in include/la_cache.h (same names, argument
marshalling only: every step of the path runs in the library's kernels).

The library must be built (bounded_kv_cache_la_b300.build); loading fails
loudly if it is missing -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblacache.so")

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_OOM, LA_ERR_CUDA, LA_ERR_STATE, LA_ERR_TIMEOUT, \
    LA_ERR_UNSUPPORTED, LA_ERR_DEVICE = range(8)
LA_POLICY_PR_SINK, LA_POLICY_CONVKV = 0, 1
LA_F32, LA_BF16, LA_E4M3 = 0, 1, 2
LA_HISTORY_RESIDENT, LA_HISTORY_EXTERNAL = 0, 1
LA_ATTN_AUTO, LA_ATTN_TENSOR, LA_ATTN_SIMT = 0, 1, 2
LA_MAX_SLOTS, LA_MAX_TOPK = 16, 8
LA_NOALLOC_MAX_ROWS = 65536

DTYPES = {"f32": LA_F32, "bf16": LA_BF16, "e4m3": LA_E4M3}

# Every symbol include/la_cache.h declares.
EXPORTS = (
    "la_cache_required_bytes", "la_cache_create", "la_cache_destroy", "la_select_context",
    "la_fill_block", "la_chunk_attention", "la_cache_append_block", "la_stream_step",
    "la_cache_load_history", "la_fill_window", "la_get_error", "la_context_plan",
    "la_debug_page", "la_debug_memory", "la_set_profile_events", "la_launch_count",
    "la_status_string", "la_pose_topk_noalloc", "la_refresh_sink", "la_prefetch_context",
    "la_debug_inject", "la_cache_state_bytes", "la_cache_save_state", "la_cache_restore",
    "la_attention_schedule",
)
LA_INJECT_ATTN_STALL = 1
LA_INJECT_BAD_FRAME = 2


class la_cache_config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("frames_per_block", ctypes.c_int32), ("grid_h", ctypes.c_int32), ("grid_w", ctypes.c_int32),
        ("rope_t", ctypes.c_int32), ("rope_h", ctypes.c_int32), ("rope_w", ctypes.c_int32),
        ("rope_theta", ctypes.c_float),
        ("policy", ctypes.c_int32), ("static_sink", ctypes.c_int32), ("dyn_topk", ctypes.c_int32),
        ("window", ctypes.c_int32), ("pose_dim", ctypes.c_int32), ("max_history", ctypes.c_int32),
        ("conv_kernel", ctypes.c_int32), ("conv_stride", ctypes.c_int32),
        ("mem_slots", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("history_mode", ctypes.c_int32), ("attn_impl", ctypes.c_int32),
    ]


class la_context(ctypes.Structure):
    _fields_ = [
        ("block", ctypes.c_int32), ("n_slots", ctypes.c_int32), ("kv_len", ctypes.c_int32),
        ("mem_tokens", ctypes.c_int32),
        ("block_id", ctypes.c_int32 * LA_MAX_SLOTS), ("t0", ctypes.c_int32 * LA_MAX_SLOTS),
        ("n_dyn", ctypes.c_int32), ("dyn_ids", ctypes.c_int32 * LA_MAX_TOPK),
        ("dyn_scores", ctypes.c_float * LA_MAX_TOPK), ("topk_gap", ctypes.c_float),
        ("need_fill", ctypes.c_int32 * LA_MAX_TOPK),
    ]

    def as_dict(self) -> dict:
        n = self.n_slots
        return {
            "block": self.block, "n_slots": n, "kv_len": self.kv_len,
            "mem_tokens": self.mem_tokens,
            "blocks": list(self.block_id[:n]), "t0": list(self.t0[:n]),
            "dyn_ids": list(self.dyn_ids[:self.n_dyn]),
            "dyn_scores": list(self.dyn_scores[:self.n_dyn]),
            "gap": self.topk_gap, "need_fill": list(self.need_fill[:self.n_dyn]),
        }


LA_FILL_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                              ctypes.c_void_p, ctypes.c_void_p)

_lib = None


class LaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: status {status} ({_status_text(status)}) {detail}".strip())


def _status_text(s: int) -> str:
    if _lib is None:
        return str(s)
    return _lib.la_status_string(s).decode()


def load() -> ctypes.CDLL:
    """Loads liblacache.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run `python -m bounded_kv_cache_la_b300.build`"
                           " (no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    cfgp = ctypes.POINTER(la_cache_config)
    ctxp = ctypes.POINTER(la_context)
    sig = {
        "la_cache_required_bytes": (sz, [cfgp]),
        "la_cache_create": (i32, [cfgp, vp, sz, vp, vp, ctypes.POINTER(vp)]),
        "la_cache_destroy": (i32, [vp]),
        "la_cache_state_bytes": (sz, [vp]),
        "la_cache_save_state": (i32, [vp, vp, sz]),
        "la_cache_restore": (i32, [cfgp, vp, sz, vp, vp, sz, vp, ctypes.POINTER(vp)]),
        "la_select_context": (i32, [vp, ctypes.POINTER(ctypes.c_float), ctxp, vp]),
        "la_fill_block": (i32, [vp, i32, i32, vp, vp, vp]),
        "la_chunk_attention": (i32, [vp, i32, vp, vp, vp, vp, vp]),
        "la_cache_append_block": (i32, [vp, i32, vp, vp, vp]),
        "la_stream_step": (i32, [vp, ctypes.POINTER(ctypes.c_float), i32, ctypes.POINTER(vp),
                                 ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                 LA_FILL_FN, vp, vp]),
        "la_cache_load_history": (i32, [vp, ctypes.POINTER(ctypes.c_float), i32, vp]),
        "la_fill_window": (i32, [vp, i32, i32, vp, vp, vp]),
        "la_refresh_sink": (i32, [vp, i32, vp, vp, vp]),
        "la_prefetch_context": (i32, [vp, ctypes.POINTER(ctypes.c_float), ctxp, vp]),
        "la_debug_inject": (i32, [vp, i32, i32]),
        "la_get_error": (i32, [vp, ctypes.c_char_p, sz]),
        "la_context_plan": (i32, [cfgp, i32, ctypes.POINTER(ctypes.c_int32), i32, ctxp]),
        "la_debug_page": (i32, [vp, i32, i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp)]),
        "la_debug_memory": (i32, [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                  ctypes.POINTER(vp), ctypes.POINTER(i32), ctypes.POINTER(i32)]),
        "la_set_profile_events": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), i32]),
        "la_launch_count": (ctypes.c_uint64, []),
        "la_status_string": (ctypes.c_char_p, [i32]),
        "la_pose_topk_noalloc": (i32, [vp, vp, i32, ctypes.POINTER(ctypes.c_float), i32, i32, i32,
                                       i32, vp, vp, vp, vp, vp]),
        "la_attention_schedule": (i32, [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32), i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def config_for(sc, *, attn_impl: int = LA_ATTN_AUTO, num_layers: int | None = None,
               max_history: int | None = None, history_mode: str | None = None) -> la_cache_config:
    """C config from a stream-shape description (duck-typed: the attributes
    of synth.StreamConfig)."""
    dt, dh, dw = sc.rope_split
    c = la_cache_config()
    c.num_layers = sc.num_layers if num_layers is None else num_layers
    c.num_heads = sc.num_heads
    c.head_dim = sc.head_dim
    c.frames_per_block = sc.frames_per_block
    c.grid_h = sc.grid_h
    c.grid_w = sc.grid_w
    c.rope_t, c.rope_h, c.rope_w = dt, dh, dw
    c.rope_theta = sc.rope_theta
    c.policy = LA_POLICY_PR_SINK if sc.policy == "prsink" else LA_POLICY_CONVKV
    c.static_sink = sc.static_sink
    c.dyn_topk = sc.dyn_topk
    c.window = sc.window
    c.pose_dim = 34
    c.max_history = (sc.n_blocks + 1) if max_history is None else max_history
    c.conv_kernel = sc.conv_kernel
    c.conv_stride = sc.conv_stride
    c.mem_slots = sc.mem_slots
    c.q_dtype = DTYPES[sc.qkv_dtype]
    c.kv_dtype = DTYPES[sc.kv_dtype]
    c.softmax_scale = sc.softmax_scale
    hm = sc.history_mode if history_mode is None else history_mode
    c.history_mode = LA_HISTORY_EXTERNAL if hm == "external" else LA_HISTORY_RESIDENT
    c.attn_impl = attn_impl
    return c


def _check(st: int, where: str, handle=None):
    if st != LA_OK:
        detail = ""
        if handle is not None and _lib is not None:
            buf = ctypes.create_string_buffer(256)
            _lib.la_get_error(handle, buf, 256)
            detail = buf.value.decode(errors="replace")
        raise LaError(st, where, detail)


def la_cache_required_bytes(cfg: la_cache_config) -> int:
    return load().la_cache_required_bytes(ctypes.byref(cfg))


def la_launch_count() -> int:
    return int(load().la_launch_count())


def la_context_plan(cfg: la_cache_config, block: int, dyn_ids=()) -> dict:
    lib = load()
    arr = (ctypes.c_int32 * max(1, len(dyn_ids)))(*dyn_ids)
    out = la_context()
    _check(lib.la_context_plan(ctypes.byref(cfg), block, arr, len(dyn_ids), ctypes.byref(out)),
           "la_context_plan")
    return out.as_dict()


def la_pose_topk_noalloc(table, inv_norm, query_kp, pose_row, c0, c1, k, ids_out, scores_out,
                         n_out, status_out, stream=None):
    """Pose top-k with the library's fixed scratch (no device allocation).

    table [max_rows, 36] and inv_norm [max_rows] are caller-owned float32
    device tensors; ids_out (int32), scores_out (float32) hold k + 1 entries,
    n_out and status_out (int32) one each, all on the device.  query_kp:
    host, 17 x 2."""
    import numpy as np
    kp = np.ascontiguousarray(np.asarray(query_kp, dtype=np.float32).reshape(34))
    _check(load().la_pose_topk_noalloc(
        _ptr(table), _ptr(inv_norm), int(table.shape[0]),
        kp.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), pose_row, c0, c1, k,
        _ptr(ids_out), _ptr(scores_out), _ptr(n_out), _ptr(status_out), _stream_handle(stream)),
        "la_pose_topk_noalloc")


def la_attention_schedule(T: int, H: int, n_slots: int, num_sms: int):
    """Host only: the tensor-core attention's work items per CTA, as a list
    of G lists of item numbers (full units, then pieces of a split tile)."""
    nt = (T + 127) // 128
    n_max = 2 * (H * (nt // 2) + (H * n_slots if nt & 1 else 0)) + 1
    buf = (ctypes.c_int32 * max(1, n_max))()
    G = load().la_attention_schedule(T, H, n_slots, num_sms, buf, n_max)
    if G < 0:
        raise LaError(LA_ERR_INVALID_ARG, "la_attention_schedule")
    off = list(buf[:G + 1])
    items = list(buf[G + 1:G + 1 + off[G]])
    return [items[off[c]:off[c + 1]] for c in range(G)]


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t if isinstance(t, int) else t.data_ptr())


class Cache:
    """A cache whose pool is a torch uint8 tensor on the current CUDA device.

    Methods map one-to-one onto the C calls; tensors are passed by address."""

    def __init__(self, cfg: la_cache_config, conv_w=None, stream=None, restore=None):
        """restore: (pool_bytes, state) from save_checkpoint() to resume a
        stream instead of starting one."""
        import torch
        self.lib = load()
        self.cfg = cfg
        nbytes = la_cache_required_bytes(cfg)
        if nbytes == 0:
            raise LaError(LA_ERR_INVALID_ARG, "la_cache_required_bytes")
        self.nbytes = nbytes
        self.pool = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
        base = self.pool.data_ptr()
        self.base = (base + 255) // 256 * 256
        self.conv_w = conv_w
        h = ctypes.c_void_p()
        cw = _ptr(conv_w) if conv_w is not None else None
        if restore is None:
            _check(self.lib.la_cache_create(ctypes.byref(cfg), ctypes.c_void_p(self.base), nbytes, cw,
                                            _stream_handle(stream), ctypes.byref(h)),
                   "la_cache_create")
        else:
            pool_bytes, state = restore
            self.pool_view().copy_(pool_bytes)
            buf = ctypes.create_string_buffer(bytes(state), len(state))
            _check(self.lib.la_cache_restore(ctypes.byref(cfg), ctypes.c_void_p(self.base), nbytes, cw,
                                             buf, len(state), _stream_handle(stream), ctypes.byref(h)),
                   "la_cache_restore")
        self.h = h

    def pool_view(self):
        """The pool's la_cache_required_bytes bytes as a uint8 tensor."""
        off = self.base - self.pool.data_ptr()
        return self.pool[off:off + self.nbytes]

    def save_checkpoint(self):
        """(pool bytes on the CPU, host-state blob) between blocks."""
        import torch
        n = self.lib.la_cache_state_bytes(self.h)
        buf = ctypes.create_string_buffer(n)
        _check(self.lib.la_cache_save_state(self.h, buf, n), "la_cache_save_state")
        torch.cuda.synchronize()
        return self.pool_view().cpu(), buf.raw

    def close(self):
        if getattr(self, "h", None):
            self.lib.la_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def la_select_context(self, query_pose, stream=None) -> dict:
        import numpy as np
        kp = None
        if query_pose is not None:
            arr = np.ascontiguousarray(np.asarray(query_pose, dtype=np.float32).reshape(34))
            kp = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
        out = la_context()
        _check(self.lib.la_select_context(self.h, kp, ctypes.byref(out), _stream_handle(stream)),
               "la_select_context", self.h)
        return out.as_dict()

    def la_prefetch_context(self, next_pose, stream=None) -> dict:
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(next_pose, dtype=np.float32).reshape(34))
        out = la_context()
        _check(self.lib.la_prefetch_context(self.h, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                            ctypes.byref(out), _stream_handle(stream)),
               "la_prefetch_context", self.h)
        return out.as_dict()

    def la_chunk_attention(self, layer, q, k, v, out, stream=None):
        _check(self.lib.la_chunk_attention(self.h, layer, _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                           _stream_handle(stream)), "la_chunk_attention", self.h)

    def la_cache_append_block(self, layer, k, v, stream=None):
        _check(self.lib.la_cache_append_block(self.h, layer, _ptr(k), _ptr(v),
                                              _stream_handle(stream)),
               "la_cache_append_block", self.h)

    def la_fill_block(self, layer, block_id, k, v, stream=None):
        _check(self.lib.la_fill_block(self.h, layer, block_id, _ptr(k), _ptr(v),
                                      _stream_handle(stream)), "la_fill_block", self.h)

    def la_fill_window(self, layer, block_id, k, v, stream=None):
        _check(self.lib.la_fill_window(self.h, layer, block_id, _ptr(k), _ptr(v),
                                       _stream_handle(stream)), "la_fill_window", self.h)

    def la_refresh_sink(self, layer, k, v, stream=None):
        _check(self.lib.la_refresh_sink(self.h, layer, _ptr(k), _ptr(v), _stream_handle(stream)),
               "la_refresh_sink", self.h)

    def la_cache_load_history(self, kps, stream=None):
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(kps, dtype=np.float32).reshape(-1, 34))
        _check(self.lib.la_cache_load_history(self.h, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                              arr.shape[0], _stream_handle(stream)),
               "la_cache_load_history", self.h)

    def la_stream_step(self, pose, n_steps, q, k, v, out, fill=None, stream=None):
        """q, k, v, out: sequences of n_steps * L tensors, entry [step * L + layer].
        fill(layer, block_id) -> (k, v) tensors supplies EXTERNAL history."""
        import numpy as np
        n = len(q)
        arrs = [(ctypes.c_void_p * n)(*[x.data_ptr() for x in seq]) for seq in (q, k, v, out)]
        kp = np.ascontiguousarray(np.asarray(pose, dtype=np.float32).reshape(34))
        keep = []

        def _fill(handle, layer, block_id, user, stream_):
            try:
                kk, vv = fill(layer, block_id)
                keep.append((kk, vv))
                return self.lib.la_fill_block(handle, layer, block_id, _ptr(kk), _ptr(vv), stream_)
            except Exception:
                return LA_ERR_STATE

        cb = LA_FILL_FN(_fill) if fill is not None else LA_FILL_FN()
        _check(self.lib.la_stream_step(self.h, kp.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                       n_steps, *arrs, cb, None, _stream_handle(stream)),
               "la_stream_step", self.h)

    def la_get_error(self) -> tuple[int, str]:
        buf = ctypes.create_string_buffer(256)
        st = self.lib.la_get_error(self.h, buf, 256)
        return st, buf.value.decode(errors="replace")

    def la_debug_page(self, layer, block_id, which):
        p, s = ctypes.c_void_p(), ctypes.c_void_p()
        _check(self.lib.la_debug_page(self.h, layer, block_id, which, ctypes.byref(p),
                                      ctypes.byref(s)), "la_debug_page")
        return p.value, s.value

    def la_debug_memory(self, layer):
        k, v, r = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        n, o = ctypes.c_int(), ctypes.c_int()
        _check(self.lib.la_debug_memory(self.h, layer, ctypes.byref(k), ctypes.byref(v),
                                        ctypes.byref(r), ctypes.byref(n), ctypes.byref(o)),
               "la_debug_memory")
        return k.value, v.value, r.value, n.value, o.value

    def la_debug_inject(self, what, count):
        _check(self.lib.la_debug_inject(self.h, what, count), "la_debug_inject")

    def la_set_profile_events(self, starts, stops):
        """starts/stops: sequences of raw cudaEvent_t handles (ints)."""
        n = len(starts)
        a = (ctypes.c_void_p * max(1, n))(*starts)
        b = (ctypes.c_void_p * max(1, n))(*stops)
        _check(self.lib.la_set_profile_events(self.h, a, b, n), "la_set_profile_events")

    def view(self, addr: int, nbytes: int):
        """uint8 view of `nbytes` of the pool starting at device address addr."""
        off = addr - self.pool.data_ptr()
        assert 0 <= off and off + nbytes <= self.pool.numel()
        return self.pool[off:off + nbytes]
