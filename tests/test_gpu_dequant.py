"""GPU parity of tq_dequant and of the continuation-chunk decode against the
oracle (through the C ABI binding).

The GPU reads ORACLE-written caches, so both sides expand identical packed
bytes and no oracle input comes from the CUDA path.

The gates are those of ``parity.assert_dequant_close`` (derived there from
the kernel's arithmetic) and, for the continuation chunks, the decode gate.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import decode as od
from oracle import dequant as dq
from parity import OracleCache, assert_decode_close, assert_dequant_close, key_bits

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from turboquant_paged_kv_gb300 import build
    build.build()
    import turboquant_paged_kv_gb300 as tq
    return tq


_ORACLE = {}


def oracle_case(name, **over):
    key = (name, tuple(sorted(over.items())))
    if key not in _ORACLE:
        w = workloads.get(name, **over)
        inp = workloads.make_inputs(w)
        _ORACLE[key] = (w, inp, OracleCache(w, inp).fill())
    return _ORACLE[key]


def _config(tq, w):
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size)
    cb = None if w.preset == "k8v4" else tq.tq_build_codebook(w.d, key_bits(w.preset))
    return cfg, cb


def gpu_dequant(tq, w, inp, cache_np, out_dtype=torch.float32, seq_lens=None, block_table=None,
                max_seq_len=None, status=None):
    cfg, cb = _config(tq, w)
    lens = inp.seq_lens if seq_lens is None else seq_lens
    table = inp.block_table if block_table is None else block_table
    msl = inp.max_seq_len if max_seq_len is None else max_seq_len
    shape = (w.batch, msl, w.n_kv, w.d)
    kout = torch.full(shape, float("nan"), dtype=out_dtype, device="cuda")
    vout = torch.full(shape, float("nan"), dtype=out_dtype, device="cuda")
    tq.tq_dequant(cfg, cb, torch.from_numpy(cache_np).cuda(), table.cuda(), lens.cuda(), msl, kout, vout,
                  dev_status=status)
    torch.cuda.synchronize()
    return kout.float().cpu().numpy(), vout.float().cpu().numpy()


def oracle_dequant(oc, seq_lens, block_table, max_seq_len):
    return dq.dequantize(oc.cache, oc.lay, oc.preset, oc.cent, np.asarray(block_table), np.asarray(seq_lens),
                         max_seq_len)


@pytest.mark.parametrize("name", ["tiny", "gqa_small", "k3v4_small", "k8v4_small", "long_small", "3bit_small"])
def test_dequant_matches_oracle_f32(tq, name):
    w, inp, oc = oracle_case(name)
    gk, gv = gpu_dequant(tq, w, inp, oc.cache)
    rk, rv = oracle_dequant(oc, inp.seq_lens, inp.block_table, inp.max_seq_len)
    ek, ev = assert_dequant_close(gk, gv, rk, rv, torch.float32, w.preset == "k8v4")
    print(f"{name}: max key error {ek:.2e}, max value error {ev:.2e}")


@pytest.mark.parametrize("name", ["tiny", "gqa_small", "k8v4_small", "3bit_small"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_dequant_matches_oracle_16bit_out(tq, name, dtype):
    w, inp, oc = oracle_case(name)
    gk, gv = gpu_dequant(tq, w, inp, oc.cache, out_dtype=dtype)
    rk, rv = oracle_dequant(oc, inp.seq_lens, inp.block_table, inp.max_seq_len)
    assert_dequant_close(gk, gv, rk, rv, dtype, w.preset == "k8v4")


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_dequant_block_sizes(tq, bs):
    w, inp, oc = oracle_case("gqa_small", block_size=bs)
    gk, gv = gpu_dequant(tq, w, inp, oc.cache)
    rk, rv = oracle_dequant(oc, inp.seq_lens, inp.block_table, inp.max_seq_len)
    assert_dequant_close(gk, gv, rk, rv, torch.float32, False)


def test_dequant_empty_sequence_and_rows_past_the_length(tq):
    w, inp, oc = oracle_case("gqa_small")
    lens = inp.seq_lens.clone()
    lens[0] = 0
    lens[2] = 1
    msl = int(inp.seq_lens.max()) + 40          # rows beyond every length
    gk, gv = gpu_dequant(tq, w, inp, oc.cache, seq_lens=lens, max_seq_len=msl)
    rk, rv = oracle_dequant(oc, lens, inp.block_table, msl)
    assert_dequant_close(gk, gv, rk, rv, torch.float32, False)
    assert np.all(gk[0] == 0) and np.all(gv[0] == 0)
    assert np.all(gk[2, 1:] == 0) and np.any(gk[2, 0] != 0)


def test_dequant_bad_block_id_is_flagged(tq):
    w, inp, oc = oracle_case("gqa_small")
    table = inp.block_table.clone()
    table[1, 3] = inp.num_blocks + 7
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gk, gv = gpu_dequant(tq, w, inp, oc.cache, block_table=table, status=status)
    assert int(status.item()) & tq.TQ_DEV_BLOCK_OUT_OF_RANGE
    assert np.all(gk[1, 48:64] == 0) and np.all(gv[1, 48:64] == 0)
    rk, rv = oracle_dequant(oc, inp.seq_lens, inp.block_table, inp.max_seq_len)
    keep = np.ones(inp.max_seq_len, bool)
    keep[48:64] = False
    assert_dequant_close(gk[:, keep], gv[:, keep], rk[:, keep], rv[:, keep], torch.float32, False)


def test_dequant_too_long_sequence_is_flagged(tq):
    w, inp, oc = oracle_case("gqa_small")
    lens = inp.seq_lens.clone()
    lens[1] = 10_000_000
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    msl = int(inp.seq_lens.max())
    gk, gv = gpu_dequant(tq, w, inp, oc.cache, seq_lens=lens, max_seq_len=msl, status=status)
    assert int(status.item()) & tq.TQ_DEV_SEQ_TOO_LONG
    # the sequence is cut at max_seq_len (517 = its own length here)
    rk, rv = oracle_dequant(oc, inp.seq_lens, inp.block_table, msl)
    assert_dequant_close(gk, gv, rk, rv, torch.float32, False)


def test_gpu_store_then_dequant_keeps_key_length(tq):
    # GPU store -> GPU dequant, checked by properties the method fixes (no
    # oracle input from the GPU): with norm correction the key keeps its
    # length up to the fp16 rounding of the stored norm, and the mean relative
    # squared error sits near the 4-bit codebook distortion 0.0095
    w = workloads.get("gqa_small")
    inp = workloads.make_inputs(w)
    cfg, cb = _config(tq, w)
    lay = tq.tq_layout_for(cfg)
    cache = torch.zeros(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device="cuda")
    starts = dict(inp.fill_order)
    kv = [inp.kv_for_sequence(b, "cpu") for b in range(w.batch)]
    for b, (k, v) in enumerate(kv):
        s0 = starts[b]
        tq.tq_store(cfg, cb, k.cuda(), v.cuda(), inp.fill_slots[s0:s0 + k.shape[0]].cuda(), cache)
    shape = (w.batch, inp.max_seq_len, w.n_kv, w.d)
    kout = torch.empty(shape, dtype=torch.float32, device="cuda")
    vout = torch.empty(shape, dtype=torch.float32, device="cuda")
    tq.tq_dequant(cfg, cb, cache, inp.block_table.cuda(), inp.seq_lens.cuda(), inp.max_seq_len, kout, vout)
    torch.cuda.synchronize()
    errs = []
    for b, (k, v) in enumerate(kv):
        length = k.shape[0]
        kk = k.double().numpy()
        kh = kout[b, :length].double().cpu().numpy()
        ratio = np.linalg.norm(kh, axis=-1) / np.linalg.norm(kk, axis=-1)
        assert np.max(np.abs(ratio - 1)) <= 2.0 ** -11 + 1e-5
        errs.append((((kk - kh) ** 2).sum(-1) / (kk * kk).sum(-1)).ravel())
        vv = v.double().numpy()
        mn = vv.min(-1, keepdims=True)
        s = (vv.max(-1, keepdims=True) - mn) / 15
        # half a step, plus the fp16 rounding of scale (times the code) and zero
        tol = s * (0.5 + 16 * 2.0 ** -11) + np.abs(mn) * 2.0 ** -11 + 1e-6
        assert np.all(np.abs(vout[b, :length].double().cpu().numpy() - vv) <= tol)
    assert 0.90 * 0.0095010 <= np.concatenate(errs).mean() <= 1.05 * 0.0095010


@pytest.mark.parametrize("name,q_len", [("gqa_small", 23), ("k8v4_small", 128), ("k3v4_small", 1)])
def test_continuation_chunk_through_decode(tq, name, q_len):
    # each query of the chunk is a decode request of length cached_len + i + 1
    # over the sequence's block-table row
    w, inp, oc = oracle_case(name)
    b = int(np.argmax(inp.seq_lens.numpy()))
    length = int(inp.seq_lens[b])
    cached = length - q_len
    g = torch.Generator().manual_seed(11)
    qc = torch.randn((q_len, w.n_q, w.d), generator=g).to(torch.bfloat16)
    ref = od.continuation_decode(qc.double().numpy(), oc.cache, oc.lay, oc.preset, oc.cent,
                                 inp.block_table.numpy()[b], cached)
    cfg, cb = _config(tq, w)
    lens = torch.arange(cached + 1, length + 1, dtype=torch.int32)
    table = inp.block_table[b:b + 1].expand(q_len, -1).contiguous()
    out = torch.full((q_len, w.n_q, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(tq.tq_decode_workspace_size(cfg, q_len, length), dtype=torch.uint8, device="cuda")
    tq.tq_decode(cfg, cb, qc.cuda(), torch.from_numpy(oc.cache).cuda(), table.cuda(), lens.cuda(), length, out, ws)
    torch.cuda.synchronize()
    err = assert_decode_close(out.cpu().numpy(), ref, torch.float32)
    print(f"{name} continuation of {q_len} queries: max|gpu-oracle| = {err:.2e}")


def test_dequant_fullsize_gqa_sampled(tq):
    # the whole gqa batch (32 x 4096 tokens, 8 KV heads) dequantised in one
    # launch to bf16; two sequences carry the oracle's bytes and are compared
    # with the oracle's expansion
    from oracle import codebook as ocb
    from oracle import layout as olay
    from oracle import store as ost
    w = workloads.get("gqa")
    host = workloads.make_inputs(w, "cpu")
    dev = torch.device("cuda", 0)
    cfg, cb = _config(tq, w)
    bb = tq.tq_layout_for(cfg).block_bytes
    cache = torch.zeros(host.num_blocks * bb, dtype=torch.uint8, device=dev)
    starts = dict(host.fill_order)
    for b in range(w.batch):
        k, v = host.kv_for_sequence(b, dev)
        s0 = starts[b]
        tq.tq_store(cfg, cb, k, v, host.fill_slots[s0:s0 + k.shape[0]].to(dev), cache)
    preset = olay.PRESETS[w.preset]
    lay = olay.tile_layout(preset, w.d, w.block_size, w.n_kv)
    cent = ocb.codebook(w.d, 4)
    mid = ocb.midpoints_fp32(cent)
    blocks = cache.view(host.num_blocks, bb)
    refs = {}
    for b in (3, 30):
        k, v = (x.double().numpy() for x in host.kv_for_sequence(b, "cpu"))
        length = k.shape[0]
        nb = length // w.block_size
        ocache = np.zeros(nb * bb, dtype=np.uint8)
        ost.store(k, v, np.arange(length), ocache, lay, preset, cent, mid)
        ids = host.block_table[b, :nb].to(torch.int64).to(dev)
        blocks[ids] = torch.from_numpy(ocache.reshape(nb, bb)).to(dev)
        refs[b] = dq.dequantize(ocache, lay, preset, cent, np.arange(nb)[None, :], np.array([length]), length)
    shape = (w.batch, host.max_seq_len, w.n_kv, w.d)
    kout = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    vout = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tq.tq_dequant(cfg, cb, cache, host.block_table.to(dev), host.seq_lens.to(dev), host.max_seq_len, kout, vout,
                  dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b, (rk, rv) in refs.items():
        ek, ev = assert_dequant_close(kout[b:b + 1].float().cpu().numpy(), vout[b:b + 1].float().cpu().numpy(),
                                      rk, rv, torch.bfloat16, False)
        print(f"gqa seq {b}: max key error {ek:.2e}, max value error {ev:.2e}")
