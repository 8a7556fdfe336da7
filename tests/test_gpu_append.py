"""GPU parity of tq_decode_append (a decode step whose newest token per
sequence is stored by the decode's split kernel itself) against the two-call
step tq_store + tq_decode, and against the oracle (through the C ABI binding).

Both GPU paths start from the same ORACLE-written cache holding positions
0 .. L_b - 2 of every sequence; the newest position L_b - 1 comes in as raw
key and value rows. Gates:
  - cache bytes: bit-identical to tq_store's (the same quantisation code, one
    launch shape), and tq_store's bytes against the oracle's quantisation of
    the same rows (the store's own gate, ``parity.compare_store``);
  - outputs: bit-identical to tq_store + tq_decode (same bytes, same consumer
    count, same work split), and within the decode gate of the oracle's decode
    over its own fully written cache.
"""

import numpy as np
import pytest
import torch

import workloads
from parity import OracleCache, assert_decode_close, compare_store, key_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from turboquant_paged_kv_gb300 import build
    build.build()
    import turboquant_paged_kv_gb300 as tq
    return tq


_CASES = {}


def oracle_case(name, **over):
    """(workload, inputs, raw kv, cache of all but the newest positions, fully written cache)."""
    key = (name, tuple(sorted(over.items())))
    if key not in _CASES:
        w = workloads.get(name, **over)
        inp = workloads.make_inputs(w)
        kv = [inp.kv_for_sequence(b, "cpu") for b in range(w.batch)]
        base = OracleCache(w, inp, kv=[(k[:-1], v[:-1]) for k, v in kv]).fill()
        full = OracleCache(w, inp, kv=kv).fill()
        _CASES[key] = (w, inp, kv, base, full)
    return _CASES[key]


def newest_rows(w, inp, kv):
    """new_k, new_v [B, n_kv, d] (position L_b - 1; zeros for empty sequences) and their slots [B]."""
    new_k = torch.zeros((w.batch, w.n_kv, w.d), dtype=w.torch_dtype)
    new_v = torch.zeros_like(new_k)
    slots = torch.full((w.batch,), -1, dtype=torch.int64)
    starts = dict(inp.fill_order)
    for b, (k, v) in enumerate(kv):
        length = k.shape[0]
        if length > 0:
            new_k[b], new_v[b] = k[length - 1], v[length - 1]
            slots[b] = inp.fill_slots[starts[b] + length - 1]
    return new_k, new_v, slots


def run_both(tq, w, inp, kv, base, partition=0, seq_lens=None, table=None, max_len=None, out_dtype=torch.float32):
    """(append cache, append out, append status, two-call cache, two-call out, two-call status)."""
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size, partition_tokens=partition)
    cb = None if w.preset == "k8v4" else tq.tq_build_codebook(w.d, key_bits(w.preset))
    lens = (inp.seq_lens if seq_lens is None else seq_lens).cuda()
    tab = (inp.block_table if table is None else table).cuda()
    msl = inp.max_seq_len if max_len is None else max_len
    new_k, new_v, slots = newest_rows(w, inp, kv)
    q = inp.q.cuda()
    ws = torch.empty(max(tq.tq_decode_workspace_size(cfg, w.batch, msl), 16), dtype=torch.uint8, device="cuda")
    res = []
    for fused in (True, False):
        cache = torch.from_numpy(base.cache.copy()).cuda()
        out = torch.full((w.batch, w.n_q, w.d), float("nan"), dtype=out_dtype, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            tq.tq_decode_append(cfg, cb, q, new_k.cuda(), new_v.cuda(), cache, tab, lens, msl, out, ws,
                                dev_status=status)
        else:
            tq.tq_store(cfg, cb, new_k.cuda(), new_v.cuda(), slots.cuda(), cache, dev_status=status)
            tq.tq_decode(cfg, cb, q, cache, tab, lens, msl, out, ws, dev_status=status)
        torch.cuda.synchronize()
        res += [cache.cpu().numpy(), out.float().cpu().numpy(), int(status.item())]
    return res


@pytest.mark.parametrize("name,partition", [
    ("gqa_small", 0),       # G = 4, stream-K
    ("gqa_small", 16),      # one tile per partition
    ("gqa_small", 128),
    ("long_small", 0),      # G = 8
    ("k3v4_small", 0),      # 3-bit keys, 4-bit values
    ("3bit_small", 0),      # 3-bit keys and values (values straddle 16-bit words)
    ("k8v4_small", 0),      # e4m3 keys, no rotation
    ("tiny", 0),            # G = 1, fp16 inputs
])
def test_append_matches_store_then_decode_and_oracle(tq, name, partition):
    w, inp, kv, base, full = oracle_case(name)
    ca, oa, sa, cb_, ob, sb = run_both(tq, w, inp, kv, base, partition=partition)
    assert sa == 0 and sb == 0
    assert np.array_equal(ca, cb_), "append cache bytes differ from tq_store's"
    assert np.array_equal(oa, ob), "append outputs differ from tq_store + tq_decode"
    new_k, new_v, slots = newest_rows(w, inp, kv)
    live = slots.numpy() >= 0
    compare_store(ca, base, new_k.double().numpy()[live], new_v.double().numpy()[live], slots.numpy()[live])
    ref = full.decode(inp.q.double().numpy())
    err = assert_decode_close(oa, ref, torch.float32)
    print(f"{name} partition {partition}: max|append - oracle| = {err:.2e}")


def test_append_ragged_edges(tq):
    # lengths 1 (the newest token is the only one), 16 and 32 (newest at row 15
    # of a tile; 32 fills two blocks of 16), 0 (nothing stored, zeros out)
    w, inp, kv, base, full = oracle_case("gqa_small", batch=5, lens=(1, 16, 0, 32, 45))
    ca, oa, sa, cb_, ob, sb = run_both(tq, w, inp, kv, base)
    assert sa == 0 and sb == 0
    assert np.array_equal(ca, cb_)
    assert np.array_equal(oa, ob)
    assert np.all(oa[2] == 0)
    assert_decode_close(oa, full.decode(inp.q.double().numpy()), torch.float32)


def test_append_half_outputs(tq):
    w, inp, kv, base, full = oracle_case("gqa_small")
    for dt in (torch.bfloat16, torch.float16):
        ca, oa, _, cb_, ob, _ = run_both(tq, w, inp, kv, base, out_dtype=dt)
        assert np.array_equal(ca, cb_)
        assert np.array_equal(oa, ob)


def test_append_skips_cut_and_missing_sequences(tq):
    w, inp, kv, base, full = oracle_case("gqa_small")
    # sequence 1 (517 positions) is longer than max_seq_len: cut, flagged,
    # nothing stored for it; sequence 2's newest block id is out of range:
    # flagged, nothing stored for it
    table = inp.block_table.clone()
    l2 = int(inp.seq_lens[2])
    table[2, (l2 - 1) // w.block_size] = inp.num_blocks + 5
    ca, oa, sa, _, _, _ = run_both(tq, w, inp, kv, base, table=table, max_len=400)
    assert sa & 4 and sa & 2, f"status {sa}"    # TQ_DEV_SEQ_TOO_LONG, TQ_DEV_BLOCK_OUT_OF_RANGE
    new_k, new_v, slots = newest_rows(w, inp, kv)
    lay = base.lay
    # bytes of the cache blocks holding sequences 1 and 2's newest positions are untouched
    for b in (1, 2):
        blk = int(slots[b]) // w.block_size
        lo, hi = blk * lay.block_bytes, (blk + 1) * lay.block_bytes
        assert np.array_equal(ca[lo:hi], base.cache[lo:hi]), f"sequence {b}'s newest block was written"
    # sequence 0 was stored as the store would
    compare_store(ca, base, new_k.double().numpy()[:1], new_v.double().numpy()[:1], slots.numpy()[:1])
