"""GPU parity of tq_continue (multi-query continuation chunks) against the
oracle's continuation_decode and against the per-query tq_decode path
(through the C ABI binding).

The GPU reads ORACLE-written caches (the chunk's keys and values included,
as the method stores them before attending), so both sides expand identical
packed bytes. Gate: the decode gate of ``parity.assert_decode_close``; the
kernel's per-position arithmetic is the decode kernel's.
"""

import numpy as np
import pytest
import torch

import workloads
from oracle import decode as od
from parity import OracleCache, assert_decode_close, key_bits

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


def _config(tq, w, partition=0):
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size, partition_tokens=partition)
    cb = None if w.preset == "k8v4" else tq.tq_build_codebook(w.d, key_bits(w.preset))
    return cfg, cb


def run_continue(tq, w, inp, cache_np, q_lens, q, out_dtype=torch.float32, partition=0, status=None,
                 max_q_len=None):
    """tq_continue over all sequences of the workload, chunk b being the last
    q_lens[b] positions of sequence b."""
    cfg, cb = _config(tq, w, partition)
    qs = torch.zeros(w.batch + 1, dtype=torch.int32)
    qs[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
    total = int(qs[-1])
    msl = inp.max_seq_len
    out = torch.full((total, w.n_q, w.d), float("nan"), dtype=out_dtype, device="cuda")
    ws = torch.empty(max(tq.tq_continue_workspace_size(cfg, total, msl), 16), dtype=torch.uint8, device="cuda")
    tq.tq_continue(cfg, cb, q.cuda(), qs.cuda(), max(q_lens) if max_q_len is None else max_q_len,
                   torch.from_numpy(cache_np).cuda(), inp.block_table.cuda(), inp.seq_lens.cuda(), msl, out, ws,
                   dev_status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), qs.numpy()


def oracle_chunks(w, inp, oc, q_lens, q):
    """Oracle continuation_decode of each sequence's chunk, stacked [total_q, n_q, d]."""
    qs = np.concatenate([[0], np.cumsum(q_lens)])
    ref = np.zeros((int(qs[-1]), w.n_q, w.d))
    for b, ql in enumerate(q_lens):
        if ql == 0:
            continue
        length = int(inp.seq_lens[b])
        ref[qs[b]:qs[b + 1]] = od.continuation_decode(q[qs[b]:qs[b + 1]].double().numpy(), oc.cache, oc.lay,
                                                      oc.preset, oc.cent, inp.block_table.numpy()[b],
                                                      length - ql)
    return ref


def chunk_queries(w, total, seed=11):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((total, w.n_q, w.d), generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("q_len", [1, 23, 128])
def test_continue_single_chunk_matches_oracle_and_per_query_decode(tq, q_len):
    # one sequence of 517 positions whose last q_len are the chunk
    w, inp, oc = oracle_case("gqa_small", batch=1, lens=(517,))
    q = chunk_queries(w, q_len)
    got, _ = run_continue(tq, w, inp, oc.cache, [q_len], q)
    ref = oracle_chunks(w, inp, oc, [q_len], q)
    err = assert_decode_close(got, ref, torch.float32)
    # the per-query path: tq_decode with lengths cached + 1 .. cached + q_len
    cfg, cb = _config(tq, w)
    length = int(inp.seq_lens[0])
    lens = torch.arange(length - q_len + 1, length + 1, dtype=torch.int32)
    table = inp.block_table[0:1].expand(q_len, -1).contiguous()
    out = torch.empty((q_len, w.n_q, w.d), dtype=torch.float32, device="cuda")
    ws = torch.empty(tq.tq_decode_workspace_size(cfg, q_len, length), dtype=torch.uint8, device="cuda")
    tq.tq_decode(cfg, cb, q.cuda(), torch.from_numpy(oc.cache).cuda(), table.cuda(), lens.cuda(), length, out, ws)
    torch.cuda.synchronize()
    per_query = out.cpu().numpy()
    assert_decode_close(got, per_query.astype(np.float64), torch.float32)
    print(f"continuation of {q_len}: max|gpu-oracle| = {err:.2e}, "
          f"max|continue - per-query decode| = {np.abs(got - per_query).max():.2e}")


@pytest.mark.parametrize("name,over,q_lens,partition", [
    ("gqa_small", {}, [40, 0, 64], 0),             # ragged chunks, an empty one
    ("gqa_small", {}, [300, 3, 17], 128),          # a chunk longer than 128; 128-position partitions
    ("gqa_small", {}, [5, 9, 2], 16),              # one tile per partition
    ("long_small", {}, [33, 100], 0),              # G = 8: one query per warp
    ("k3v4_small", {}, [20, 7, 12], 0),            # 3-bit keys, 4-bit values
    ("3bit_small", {}, [30, 31, 1], 0),            # 3-bit keys and values
    ("k8v4_small", {}, [16, 1, 50], 0),            # e4m3 keys
    ("tiny", {}, [37, 100], 0),                    # G = 1: eight queries per warp; fp16 inputs
])
def test_continue_batched_matches_oracle(tq, name, over, q_lens, partition):
    w, inp, oc = oracle_case(name, **over)
    q = chunk_queries(w, sum(q_lens)).to(w.torch_dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got, _ = run_continue(tq, w, inp, oc.cache, q_lens, q, partition=partition, status=status)
    assert int(status.item()) == 0
    ref = oracle_chunks(w, inp, oc, q_lens, q)
    err = assert_decode_close(got, ref, torch.float32)
    print(f"{name} chunks {q_lens}: max|gpu-oracle| = {err:.2e}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_continue_half_outputs(tq, out_dtype):
    w, inp, oc = oracle_case("gqa_small")
    q_lens = [12, 64, 8]
    q = chunk_queries(w, sum(q_lens))
    got, _ = run_continue(tq, w, inp, oc.cache, q_lens, q, out_dtype=out_dtype)
    assert_decode_close(got, oracle_chunks(w, inp, oc, q_lens, q), out_dtype)


def test_continue_rows_past_max_q_len_are_flagged(tq):
    w, inp, oc = oracle_case("gqa_small")
    q_lens = [10, 4, 6]
    q = chunk_queries(w, sum(q_lens))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got, _ = run_continue(tq, w, inp, oc.cache, q_lens, q, status=status, max_q_len=8)
    assert int(status.item()) & 4
    ref = oracle_chunks(w, inp, oc, q_lens, q)
    # sequences 1 and 2 are whole; sequence 0's first 8 rows are served, its
    # last 2 come out 0
    assert_decode_close(got[10:], ref[10:], torch.float32)
    assert_decode_close(got[:8], ref[:8], torch.float32)
    assert np.all(got[8:10] == 0)
