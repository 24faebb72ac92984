"""C-ABI library: loads, exports every declared symbol, and its host-only
planning logic agrees with the oracle (no GPU needed)."""
import os
import re
import subprocess

import numpy as np
import pytest

from bounded_kv_cache_la_b300 import capi
from oracle import stream
from synth import C1_TINY, C2_MID, C3_14B, C4_CONVKV, C5_FP8, gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "la_cache.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(l for l in text.splitlines() if "typedef" not in l)
    return set(re.findall(r"\b(la_[a-z_]+)\s*\(", text))


def test_header_and_binding_agree():
    assert _declared_functions() == set(capi.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = _declared_functions() - exported
    assert not missing, missing
    for name in _declared_functions():
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for s in range(8):
        assert lib.la_status_string(s)


@pytest.mark.parametrize("sc", [C1_TINY, C2_MID, C3_14B, C4_CONVKV, C5_FP8])
def test_required_bytes(sc):
    cfg = capi.config_for(sc)
    n = capi.la_cache_required_bytes(cfg)
    assert n > 0
    T, H, D = sc.tokens_per_block, sc.num_heads, sc.head_dim
    elt = {"f32": 4, "bf16": 2, "e4m3": 1}[sc.kv_dtype]
    page = T * H * D * elt
    # at least every attended block's K and V for every layer
    n_blocks = 1 + sc.dyn_topk + sc.window + 1 if sc.policy == "prsink" else sc.window + 1
    assert n >= 2 * page * n_blocks * sc.num_layers
    if sc is C3_14B:
        assert n < 60e9          # bounded: independent of the 3600-block stream


def test_invalid_configs_rejected():
    cfg = capi.config_for(C2_MID)
    cfg.rope_t += 2
    assert capi.la_cache_required_bytes(cfg) == 0
    cfg = capi.config_for(C2_MID)
    cfg.dyn_topk = 20
    assert capi.la_cache_required_bytes(cfg) == 0
    cfg = capi.config_for(C2_MID)
    cfg.head_dim = 96
    assert capi.la_cache_required_bytes(cfg) == 0
    cfg = capi.config_for(C2_MID)
    cfg.grid_h, cfg.grid_w = 1024, 1025           # 2 x 1024 x 1025 tokens per block
    assert capi.la_cache_required_bytes(cfg) == 0


@pytest.mark.parametrize("sc,n", [(C1_TINY, 24), (C2_MID, 64), (C3_14B, 400), (C5_FP8, 300)])
def test_plan_matches_oracle_prsink(sc, n):
    cfg = capi.config_for(sc)
    ctxs = stream.plan_stream(sc, gen.poses(sc, n_blocks=n), n)
    for ctx in ctxs:
        got = capi.la_context_plan(cfg, ctx.block, ctx.dyn_ids)
        assert got["blocks"] == ctx.blocks
        assert got["t0"] == ctx.t0
        assert got["kv_len"] == ctx.kv_len
        assert got["mem_tokens"] == 0


@pytest.mark.parametrize("sc", [
    C2_MID.with_(dyn_topk=8, window=6),                       # 16 slots
    C2_MID.with_(static_sink=0),
    C2_MID.with_(dyn_topk=0),
    C2_MID.with_(static_sink=0, dyn_topk=0, window=1),
    C5_FP8.with_(window=5, dyn_topk=6),
])
def test_plan_matches_oracle_other_policies(sc):
    """Slot order, RoPE bases and KV length for other sink / top-k / window
    settings, over a stream long enough to fill every slot."""
    n = 40
    cfg = capi.config_for(sc, max_history=n + 2)
    for ctx in stream.plan_stream(sc, gen.poses(sc, n_blocks=n), n):
        got = capi.la_context_plan(cfg, ctx.block, ctx.dyn_ids)
        assert got["blocks"] == ctx.blocks
        assert got["t0"] == ctx.t0
        assert got["kv_len"] == ctx.kv_len


@pytest.mark.parametrize("kernel,stride", [(5, 5), (3, 2), (4, 4), (7, 5)])
def test_plan_matches_oracle_convkv(kernel, stride):
    sc = C4_CONVKV.with_(conv_kernel=kernel, conv_stride=stride)
    cfg = capi.config_for(sc)
    for b in range(0, 1000, 7):
        ctx = stream.plan_convkv(sc, b)
        got = capi.la_context_plan(cfg, b, [])
        assert got["blocks"] == ctx.blocks
        assert got["t0"] == ctx.t0
        assert got["mem_tokens"] == ctx.mem_tokens
        assert got["kv_len"] == ctx.kv_len


def test_plan_rejects_bad_dynamic_ids():
    cfg = capi.config_for(C2_MID)
    for ids in ([0], [9], [3, 3], [50]):
        with pytest.raises(capi.LaError):
            capi.la_context_plan(cfg, 10, ids)


def test_restore_rejects_foreign_blobs(lib):
    """la_cache_restore checks the blob before it touches the device: a blob
    that is not a state blob, or that carries another config, is refused."""
    import ctypes
    cfg = capi.config_for(C2_MID)
    other = capi.config_for(C2_MID.with_(dyn_topk=2))
    out = ctypes.c_void_p()
    fake_pool = ctypes.c_void_p(0x10000)       # never dereferenced on these paths

    def restore(blob, c=cfg):
        buf = ctypes.create_string_buffer(blob, len(blob))
        return lib.la_cache_restore(ctypes.byref(c), fake_pool, 1 << 30, None, buf, len(blob), None,
                                    ctypes.byref(out))

    header = (0x5343414C).to_bytes(4, "little") + (1).to_bytes(4, "little")
    assert restore(b"not a cache state blob") == capi.LA_ERR_INVALID_ARG
    assert restore(header) == capi.LA_ERR_INVALID_ARG                       # truncated
    assert restore(header + bytes(other)) == capi.LA_ERR_INVALID_ARG        # another config
    wrong_version = (0x5343414C).to_bytes(4, "little") + (2).to_bytes(4, "little")
    assert restore(wrong_version + bytes(cfg)) == capi.LA_ERR_INVALID_ARG
    assert lib.la_cache_state_bytes(None) == 0


def test_struct_layouts_match_header(tmp_path):
    """The ctypes mirrors of la_cache_config and la_context have the size and
    field offsets the C compiler gives the header's structs, and the
    header's constants match the binding's."""
    import ctypes
    fields = {"la_cache_config": [f[0] for f in capi.la_cache_config._fields_],
              "la_context": [f[0] for f in capi.la_context._fields_]}
    lines = ['#include <stdio.h>', '#include "la_cache.h"', "int main(void) {"]
    for st, names in fields.items():
        lines.append(f'  printf("{st} %zu\\n", sizeof({st}));')
        for n in names:
            lines.append(f'  printf("{st}.{n} %zu\\n", offsetof({st}, {n}));')
    for c in ("LA_MAX_SLOTS", "LA_MAX_TOPK", "LA_INJECT_ATTN_STALL", "LA_INJECT_BAD_FRAME",
              "LA_ERR_DEVICE", "LA_ATTN_SIMT", "LA_HISTORY_EXTERNAL"):
        lines.append(f'  printf("{c} %d\\n", (int){c});')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for st, names in fields.items():
        cls = getattr(capi, st)
        assert int(got[st]) == ctypes.sizeof(cls), st
        for n in names:
            assert int(got[f"{st}.{n}"]) == getattr(cls, n).offset, (st, n)
    for c in ("LA_MAX_SLOTS", "LA_MAX_TOPK", "LA_INJECT_ATTN_STALL", "LA_INJECT_BAD_FRAME",
              "LA_ERR_DEVICE", "LA_ATTN_SIMT", "LA_HISTORY_EXTERNAL"):
        assert int(got[c]) == getattr(capi, c), c


def test_fast_division_magic(tmp_path):
    """The kernels divide token indices by run-time constants with a
    multiply-high, an add and a shift (FastDiv in csrc/la_internal.h).  The
    host-made multipliers, used the way the device uses them, give n / d
    exactly for every divisor up to 5000 on 4000 spread numerators each and
    on the edge numerators (0, d - 1, d, 2^31 - 1)."""
    src = tmp_path / "fastdiv.cpp"
    src.write_text(r'''
#include <cstdio>
#include "la_internal.h"
int main() {
  long long bad = 0, checked = 0;
  auto check = [&](const la::FastDiv& f, uint32_t n, uint32_t d) {
    const uint32_t q = (uint32_t)((((uint64_t)n * f.m >> 32) + n) >> f.l);   // umulhi + add + shift
    bad += q != n / d;
    ++checked;
  };
  for (uint32_t d = 1; d <= 5000; ++d) {
    const la::FastDiv f = la::make_fastdiv(d);
    for (uint32_t k = 0; k < 4000; ++k)
      check(f, (uint32_t)(((uint64_t)k * 2654435761u + d * 40503u) % (1u << 31)), d);
    for (uint32_t n : {0u, d - 1, d, 0x7fffffffu}) check(f, n, d);
  }
  std::printf("%lld %lld\n", checked, bad);
  return bad != 0;
}
''')
    exe = tmp_path / "fastdiv"
    subprocess.run(["g++", "-std=c++17", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "bounded_kv_cache_la_b300", "csrc"),
                    "-I", os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    checked, bad = map(int, out.stdout.split())
    assert out.returncode == 0 and bad == 0 and checked == 5000 * 4004


@pytest.mark.parametrize("T,H,S,sms", [(4680, 40, 7, 148), (4680, 40, 9, 148), (4680, 40, 5, 148),
                                       (3510, 40, 7, 148), (1560, 12, 6, 148), (48, 3, 4, 148),
                                       (4680, 64, 7, 148), (4680, 40, 7, 132), (390, 4, 6, 148),
                                       (4680, 1, 7, 148), (4608, 40, 7, 148)])
def test_attention_schedule_every_item_once_and_balanced(lib, T, H, S, sms):
    """The tensor-core attention's work table: every item exactly once, at
    most num_sms CTAs, the estimated time per CTA within one item of the
    mean (list scheduling), each piece of a split tile dealt after its
    head's full units, and at the 14B shape (37 query tiles per head) a
    slowest CTA under 5.3 full units (dealing the odd tile whole, two per
    CTA on 20 CTAs, gave 5.74)."""
    from bounded_kv_cache_la_b300 import capi
    lists = capi.la_attention_schedule(T, H, S, sms)
    nt = (T + 127) // 128
    n_full = nt // 2
    P = S if nt & 1 else 0
    n_items = H * n_full + H * P
    G = min(n_items, sms)
    assert len(lists) == G
    assert sorted(u for l in lists for u in l) == list(range(n_items))
    t_piece = 0.78 / P + 0.02 if P else 0.0
    cost = lambda u: 1.0 if u < H * n_full else t_piece
    load = [sum(cost(u) for u in l) for l in lists]
    assert max(load) <= sum(load) / G + 1.0 + 1e-9
    order = {}
    for c, l in enumerate(lists):
        for i, u in enumerate(l):
            order[u] = (c, i)
    if T == 4680 and H == 40 and sms == 148:
        assert max(load) < 5.3
    # the pieces of a head never run before one of its full units on the same CTA
    for c, l in enumerate(lists):
        seen_piece_heads = set()
        for u in l:
            if u >= H * n_full:
                seen_piece_heads.add((u - H * n_full) // P)
            else:
                assert u // n_full not in seen_piece_heads
    assert capi.la_attention_schedule.__doc__
    with pytest.raises(capi.LaError):
        capi.la_attention_schedule(0, H, S, sms)
