"""libtq on the host: load, exported symbols, host-side arithmetic, argument checks.

No test here launches a kernel; every call either runs host code only or
returns an error before reaching the GPU.
"""

import ctypes
import json
import os
import re

import numpy as np
import pytest

from oracle import codebook as ocb
from oracle import layout as olay

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tq():
    from turboquant_paged_kv_gb300 import build
    build.build()
    import turboquant_paged_kv_gb300 as tq
    return tq


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\**\s+\**(tq_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(tq):
    from turboquant_paged_kv_gb300 import _abi
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    lib = ctypes.CDLL(tq.lib_path())
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(_abi.EXPORTED) == declared
    # matches the header's TQ_ABI_VERSION
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    assert tq.tq_version() == int(re.search(r"#define TQ_ABI_VERSION (\d+)", text).group(1)) == 105


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_host_codebook_equals_oracle(tq, d, bits):
    cb = tq.tq_build_codebook(d, bits)
    n = 2 ** bits
    assert cb.num_levels == n and cb.bits == bits and cb.head_dim == d
    got = np.array(cb.centroids[:n], dtype=np.float32)
    ref = ocb.codebook(d, bits)
    assert np.array_equal(got, ref)
    assert np.array_equal(np.array(cb.midpoints[: n - 1], dtype=np.float32), ocb.midpoints_fp32(ref))


@pytest.mark.parametrize("preset", ["k8v4", "4bit_nc", "k3v4_nc", "3bit_nc"])
@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_layout_equals_oracle(tq, preset, bs):
    cfg = tq.make_config(preset, 32, 8, block_size=bs)
    got = tq.tq_layout_for(cfg)
    ref = olay.tile_layout(olay.PRESETS[preset], 128, bs, 8)
    key, value, slot, _ = olay.preset_slot_sizes(olay.PRESETS[preset], 128)
    assert (got.key_packed_bytes, got.value_packed_bytes, got.slot_bytes) == (key, value, slot)
    assert got.tile_bytes == ref.tile_bytes and got.block_bytes == ref.block_bytes
    assert (got.k_off, got.k_row_bytes, got.v_off, got.v_row_bytes) == (ref.k_off, ref.kb, ref.v_off, ref.vb)
    assert (got.knorm_off, got.vscale_off, got.vzero_off) == (ref.knorm_off, ref.vscale_off, ref.vzero_off)


def test_unsupported_shapes(tq):
    from turboquant_paged_kv_gb300 import _abi
    lay = _abi.tq_layout()
    lib = _abi.load()
    for cfg, want in [(tq.make_config("4bit_nc", 8, 8, head_dim=96), _abi.TQ_ERR_UNSUPPORTED),
                      (tq.make_config("4bit_nc", 8, 8, block_size=8), _abi.TQ_ERR_UNSUPPORTED),
                      (tq.make_config(17, 8, 8), _abi.TQ_ERR_INVALID_ARG),
                      (tq.make_config("3bit_nc", 8, 8), _abi.TQ_OK),
                      (tq.make_config("4bit_nc", 8, 8, flags=2), _abi.TQ_ERR_INVALID_ARG),
                      (tq.make_config("4bit_nc", 8, 8, flags=tq.TQ_FLAG_INDICES_READY), _abi.TQ_OK)]:
        assert lib.tq_layout_for(ctypes.byref(cfg), ctypes.byref(lay)) == want


def test_workspace_size_matches_pages_example(tq, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "memory.json")))["decode_workspace"]
    cfg = tq.make_config("4bit_nc", g["num_heads"], 8, partition_tokens=512)
    size = tq.tq_decode_workspace_size(cfg, g["max_num_reqs"], g["max_num_splits"] * 512)
    # one partial per (sequence, KV head, partition) -- (d + 1) fp32 for each of
    # the G query heads, the pages' mid_o -- plus one per warp of the largest
    # persistent grid (256 CTAs x 16 warps), where a warp's range splits a segment
    group = g["num_heads"] // 8
    rows = g["max_num_reqs"] * g["num_heads"] * g["max_num_splits"]
    extra = 256 * 16 * group * (g["head_size"] + 1) * 4
    assert size == rows * (g["head_size"] + 1) * 4 + extra
    assert abs((size - extra) - g["mid_o_bytes_approx"]) / g["mid_o_bytes_approx"] < 0.01
    assert tq.tq_decode_workspace_size(cfg, -1, 10) == 0


def test_host_argument_errors_return_before_launch(tq):
    from turboquant_paged_kv_gb300 import _abi
    lib = _abi.load()
    cfg = tq.make_config("4bit_nc", 32, 8)
    cb = tq.tq_build_codebook(128, 4)
    cb3 = tq.tq_build_codebook(128, 3)
    ok16 = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    st = lambda *a: lib.tq_store(ctypes.byref(cfg), *a)  # noqa: E731
    # zero tokens is a no-op even with null pointers
    assert st(ctypes.byref(cb), None, None, 1, 0, None, None, 0, None, None) == _abi.TQ_OK
    assert st(ctypes.byref(cb), None, ok16, 1, 5, ok16, ok16, 4, None, None) == _abi.TQ_ERR_INVALID_ARG
    assert st(ctypes.byref(cb), odd, ok16, 1, 5, ok16, ok16, 4, None, None) == _abi.TQ_ERR_MISALIGNED
    assert st(ctypes.byref(cb3), ok16, ok16, 1, 5, ok16, ok16, 4, None, None) == _abi.TQ_ERR_INVALID_ARG
    assert st(ctypes.byref(cb), ok16, ok16, 7, 5, ok16, ok16, 4, None, None) == _abi.TQ_ERR_INVALID_ARG
    dec = lambda cfg_, ws_bytes, out=ok16, q=ok16: lib.tq_decode(  # noqa: E731
        ctypes.byref(cfg_), ctypes.byref(cb), q, 1, ok16, 10, ok16, 4, ok16, 2, 64, 0.0, out, 2, ok16,
        ws_bytes, None, None)
    need = tq.tq_decode_workspace_size(cfg, 2, 64)
    assert dec(cfg, need - 1) == _abi.TQ_ERR_WORKSPACE_TOO_SMALL
    assert dec(cfg, need, out=odd) == _abi.TQ_ERR_MISALIGNED
    assert dec(cfg, need, q=odd) == _abi.TQ_ERR_MISALIGNED
    assert dec(cfg, need, q=None) == _abi.TQ_ERR_INVALID_ARG
    wide = tq.make_config("4bit_nc", 32, 2)          # 16 query heads per KV head
    assert dec(wide, 1 << 30) == _abi.TQ_ERR_UNSUPPORTED
    uneven = tq.make_config("4bit_nc", 30, 8)
    assert dec(uneven, 1 << 30) == _abi.TQ_ERR_INVALID_ARG
    badpart = tq.make_config("4bit_nc", 32, 8, partition_tokens=40)
    assert dec(badpart, 1 << 30) == _abi.TQ_ERR_INVALID_ARG


def test_decode_append_argument_errors_return_before_launch(tq):
    from turboquant_paged_kv_gb300 import _abi
    lib = _abi.load()
    cfg = tq.make_config("4bit_nc", 32, 8)
    cb = tq.tq_build_codebook(128, 4)
    ok16 = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    need = tq.tq_decode_workspace_size(cfg, 2, 64)

    def app(new_k=ok16, new_v=ok16, out=ok16, ws_bytes=need, batch=2, out_dtype=2):
        return lib.tq_decode_append(ctypes.byref(cfg), ctypes.byref(cb), ok16, 1, new_k, new_v, ok16, 10, ok16, 4,
                                    ok16, batch, 64, 0.0, out, out_dtype, ok16, ws_bytes, None, None)

    assert app(new_k=None) == _abi.TQ_ERR_INVALID_ARG
    assert app(new_v=None) == _abi.TQ_ERR_INVALID_ARG
    assert app(out=None) == _abi.TQ_ERR_INVALID_ARG
    assert app(new_k=odd) == _abi.TQ_ERR_MISALIGNED
    assert app(new_v=odd) == _abi.TQ_ERR_MISALIGNED
    assert app(out=odd) == _abi.TQ_ERR_MISALIGNED
    assert app(ws_bytes=need - 1) == _abi.TQ_ERR_WORKSPACE_TOO_SMALL
    assert app(out_dtype=9) == _abi.TQ_ERR_INVALID_ARG
    # an empty batch is a no-op even with null rows
    assert app(new_k=None, new_v=None, batch=0) == _abi.TQ_OK


def test_dequant_argument_errors_return_before_launch(tq):
    from turboquant_paged_kv_gb300 import _abi
    lib = _abi.load()
    cfg = tq.make_config("4bit_nc", 32, 8)
    cb = tq.tq_build_codebook(128, 4)
    cb3 = tq.tq_build_codebook(128, 3)
    ok16 = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    odd4 = ctypes.c_void_p(0x10002)

    def dq(cfg_=cfg, cb_=cb, cache=ok16, table=ok16, stride=4, lens=ok16, batch=2, max_len=64,
           kout=ok16, vout=ok16, dtype=1, status=None):
        return lib.tq_dequant(ctypes.byref(cfg_), None if cb_ is None else ctypes.byref(cb_), cache, 10, table,
                              stride, lens, batch, max_len, kout, vout, dtype, status, None)

    # empty requests are no-ops even with null pointers
    assert dq(cache=None, table=None, lens=None, kout=None, vout=None, batch=0) == _abi.TQ_OK
    assert dq(cache=None, table=None, lens=None, kout=None, vout=None, max_len=0) == _abi.TQ_OK
    assert dq(kout=None) == _abi.TQ_ERR_INVALID_ARG
    assert dq(lens=None) == _abi.TQ_ERR_INVALID_ARG
    assert dq(vout=odd) == _abi.TQ_ERR_MISALIGNED
    assert dq(cache=odd) == _abi.TQ_ERR_MISALIGNED
    assert dq(table=odd4) == _abi.TQ_ERR_MISALIGNED
    assert dq(status=odd4) == _abi.TQ_ERR_MISALIGNED
    assert dq(cb_=cb3) == _abi.TQ_ERR_INVALID_ARG        # codebook of the wrong width
    assert dq(cb_=None) == _abi.TQ_ERR_INVALID_ARG
    assert dq(dtype=7) == _abi.TQ_ERR_INVALID_ARG
    assert dq(stride=0) == _abi.TQ_ERR_INVALID_ARG
    assert dq(batch=-1) == _abi.TQ_ERR_INVALID_ARG
    assert dq(cfg_=tq.make_config("3bit_nc", 32, 8, head_dim=64), cb_=cb3) == _abi.TQ_ERR_UNSUPPORTED
    assert dq(cfg_=tq.make_config("4bit_nc", 32, 8, block_size=24)) == _abi.TQ_ERR_UNSUPPORTED
    # FP8 keys need no codebook; this call would launch, so only the argument
    # checks that come first are exercised
    assert dq(cfg_=tq.make_config("k8v4", 32, 8), cb_=None, kout=None) == _abi.TQ_ERR_INVALID_ARG


def test_dequant_binding_rejects_mixed_output_dtypes(tq):
    import torch
    cfg = tq.make_config("4bit_nc", 32, 8)
    cb = tq.tq_build_codebook(128, 4)
    k = torch.empty((1, 16, 8, 128), dtype=torch.bfloat16)
    v = torch.empty((1, 16, 8, 128), dtype=torch.float32)
    with pytest.raises(ValueError):
        tq.tq_dequant(cfg, cb, torch.empty(16), torch.zeros((1, 1), dtype=torch.int32),
                      torch.zeros(1, dtype=torch.int32), 16, k, v)


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_prod_layout_equals_oracle(tq, bs):
    from oracle import qjl
    lay = tq.tq_prod_layout_for(tq.make_config("prod3", 32, 8, block_size=bs))
    ref = qjl.prod_tile_layout(128, bs, 8, 2)
    assert (lay.mse_bits, lay.tile_bytes, lay.slot_bytes) == (2, ref.tile_bytes, ref.slot_bytes)
    assert (lay.k_off, lay.k_row_bytes, lay.sign_off, lay.sign_row_bytes) == (ref.k_off, ref.kb, ref.s_off, ref.sb)
    assert (lay.norm_off, lay.rnorm_off, lay.block_bytes) == (ref.norm_off, ref.rnorm_off, ref.block_bytes)


def test_prod_argument_errors_return_before_launch(tq):
    from turboquant_paged_kv_gb300 import _abi
    lib = _abi.load()
    cfg = tq.make_config("prod3", 32, 8)
    cb2 = tq.tq_build_codebook(128, 2)
    cb4 = tq.tq_build_codebook(128, 4)
    ok16 = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    lay = _abi.tq_layout()
    # the prod preset has no K/V layout, and the K/V presets no prod layout
    assert lib.tq_layout_for(ctypes.byref(cfg), ctypes.byref(lay)) == _abi.TQ_ERR_UNSUPPORTED
    play = _abi.tq_prod_layout()
    assert lib.tq_prod_layout_for(ctypes.byref(tq.make_config("4bit_nc", 32, 8)), ctypes.byref(play)) == \
        _abi.TQ_ERR_INVALID_ARG
    assert lib.tq_prod_layout_for(ctypes.byref(tq.make_config("prod3", 32, 8, head_dim=64)), ctypes.byref(play)) == \
        _abi.TQ_ERR_UNSUPPORTED

    def st(cb=cb2, S=ok16, key=ok16, dtype=1, n=5, slots=ok16, cache=ok16, status=None, cfg_=cfg):
        return lib.tq_prod_store(ctypes.byref(cfg_), None if cb is None else ctypes.byref(cb), S, key, dtype, n,
                                 slots, cache, 4, status, None)

    assert st(S=None, key=None, slots=None, cache=None, n=0) == _abi.TQ_OK
    assert st(cb=cb4) == _abi.TQ_ERR_INVALID_ARG
    assert st(cb=None) == _abi.TQ_ERR_INVALID_ARG
    assert st(S=None) == _abi.TQ_ERR_INVALID_ARG
    assert st(dtype=2) == _abi.TQ_ERR_INVALID_ARG
    assert st(S=odd) == _abi.TQ_ERR_MISALIGNED
    assert st(key=odd) == _abi.TQ_ERR_MISALIGNED
    assert st(slots=ctypes.c_void_p(0x10004)) == _abi.TQ_ERR_MISALIGNED
    assert st(n=-1) == _abi.TQ_ERR_INVALID_ARG

    def sc(cfg_=cfg, cb=cb2, S=ok16, q=ok16, cache=ok16, table=ok16, lens=ok16, batch=2, L=64, out=ok16,
           ws=ok16, ws_bytes=None):
        need = tq.tq_prod_scores_workspace_size(cfg_, batch)
        return lib.tq_prod_scores(ctypes.byref(cfg_), None if cb is None else ctypes.byref(cb), S, q, 1, cache, 4,
                                  table, 4, lens, batch, L, 0.0, out, ws, need if ws_bytes is None else ws_bytes,
                                  None, None)

    assert tq.tq_prod_scores_workspace_size(cfg, 2) == 2 * 8 * 32 * (32 + 12) * 4   # per KV head: 32 lanes x (32 operand words + 12 constants)
    assert sc(S=None, q=None, cache=None, table=None, lens=None, out=None, ws=None, batch=0) == _abi.TQ_OK
    assert sc(ws_bytes=100) == _abi.TQ_ERR_WORKSPACE_TOO_SMALL
    assert sc(cb=cb4) == _abi.TQ_ERR_INVALID_ARG
    assert sc(out=None) == _abi.TQ_ERR_INVALID_ARG
    assert sc(out=odd) == _abi.TQ_ERR_MISALIGNED
    assert sc(table=ctypes.c_void_p(0x10002)) == _abi.TQ_ERR_MISALIGNED
    assert sc(cfg_=tq.make_config("prod3", 32, 2)) == _abi.TQ_ERR_UNSUPPORTED     # 16 query heads per KV head
    assert sc(cfg_=tq.make_config("prod3", 30, 8)) == _abi.TQ_ERR_INVALID_ARG
    skew = tq.tq_build_codebook(128, 2)
    skew.centroids[0] *= 1.5                   # not of the form {-A, -B, B, A}
    assert sc(cb=skew) == _abi.TQ_ERR_INVALID_ARG


def test_continue_workspace_and_argument_errors(tq):
    from turboquant_paged_kv_gb300 import _abi
    lib = _abi.load()
    cfg = tq.make_config("4bit_nc", 32, 8)
    # one record (d floats + an LSE) per (query, query head, 512-position partition)
    assert tq.tq_continue_workspace_size(cfg, 128, 4224) == 128 * 32 * 9 * 129 * 4
    assert tq.tq_continue_workspace_size(tq.make_config("4bit_nc", 32, 8, partition_tokens=128), 3, 300) == \
        (3 * 32 * 3 * 129 * 4 + 15) // 16 * 16
    assert tq.tq_continue_workspace_size(tq.make_config("4bit_nc", 24, 8), 4, 64) == 0        # G = 3
    assert tq.tq_continue_workspace_size(tq.make_config("4bit_nc", 32, 8, partition_tokens=8192), 4, 64) == 0
    cb = tq.tq_build_codebook(128, 4)
    cb3 = tq.tq_build_codebook(128, 3)
    ok16 = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)

    def cont(cfg_=cfg, cb_=cb, q=ok16, qs=ok16, batch=2, total=10, mql=8, cache=ok16, table=ok16, lens=ok16,
             out=ok16, ws=ok16, ws_bytes=None, qd=1, od=2):
        need = tq.tq_continue_workspace_size(cfg_, total, 64)
        return lib.tq_continue(ctypes.byref(cfg_), None if cb_ is None else ctypes.byref(cb_), q, qd, qs, batch,
                               total, mql, cache, 10, table, 4, lens, 64, 0.0, out, od, ws,
                               need if ws_bytes is None else ws_bytes, None, None)

    assert cont(q=None, qs=None, cache=None, table=None, lens=None, out=None, ws=None, total=0) == _abi.TQ_OK
    assert cont(q=None, qs=None, cache=None, table=None, lens=None, out=None, ws=None, batch=0) == _abi.TQ_OK
    assert cont(ws_bytes=64) == _abi.TQ_ERR_WORKSPACE_TOO_SMALL
    assert cont(cb_=cb3) == _abi.TQ_ERR_INVALID_ARG
    assert cont(qd=2) == _abi.TQ_ERR_INVALID_ARG
    assert cont(od=7) == _abi.TQ_ERR_INVALID_ARG
    assert cont(qs=None) == _abi.TQ_ERR_INVALID_ARG
    assert cont(out=odd) == _abi.TQ_ERR_MISALIGNED
    assert cont(qs=ctypes.c_void_p(0x10002)) == _abi.TQ_ERR_MISALIGNED
    assert cont(cfg_=tq.make_config("4bit_nc", 24, 8)) == _abi.TQ_ERR_UNSUPPORTED
    assert cont(batch=-1) == _abi.TQ_ERR_INVALID_ARG
