"""GPU parity of tq_decode against the oracle (through the C ABI binding).

The GPU decodes an ORACLE-written cache, so both sides read identical packed
bytes and no oracle input comes from the CUDA path.
"""

import numpy as np
import pytest
import torch

import workloads
from parity import OracleCache, assert_decode_close, cosine, key_bits, unquantized_attention

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
        oc = OracleCache(w, inp).fill()
        q = inp.q.double().numpy()
        _ORACLE[key] = (w, inp, oc, q, oc.decode(q))
    return _ORACLE[key]


def gpu_decode(tq, w, inp, cache_np, out_dtype=torch.float32, partition_tokens=None, seq_lens=None,
               block_table=None, q=None, status=None, max_seq_len=None, flags=0):
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size,
                         partition_tokens=w.partition_tokens if partition_tokens is None else partition_tokens,
                         flags=flags)
    cb = None if w.preset == "k8v4" else tq.tq_build_codebook(w.d, key_bits(w.preset))
    cache = torch.from_numpy(cache_np).cuda()
    lens = (inp.seq_lens if seq_lens is None else seq_lens).cuda()
    table = (inp.block_table if block_table is None else block_table).cuda()
    qq = (inp.q if q is None else q).cuda()
    msl = int(lens.max().item()) if max_seq_len is None else max_seq_len
    out = torch.full((w.batch, w.n_q, w.d), float("nan"), dtype=out_dtype, device="cuda")
    ws = torch.empty(tq.tq_decode_workspace_size(cfg, w.batch, max(msl, 1)), dtype=torch.uint8, device="cuda")
    tq.tq_decode(cfg, cb, qq, cache, table, lens, max(msl, 1), out, ws, dev_status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


# partition_tokens None: the workload's own (fixed partitions, split + reduce
# kernels); 0: stream-K, where tq_decode merges in the split kernel itself
@pytest.mark.parametrize("pt", [None, 0])
@pytest.mark.parametrize("name", ["tiny", "gqa_small", "k3v4_small", "k8v4_small", "long_small", "3bit_small"])
def test_decode_matches_oracle_f32(tq, name, pt):
    w, inp, oc, q, ref = oracle_case(name)
    got = gpu_decode(tq, w, inp, oc.cache, partition_tokens=pt)
    err = assert_decode_close(got, ref, torch.float32)
    assert err < 1e-3
    # reported, not gated: agreement with unquantised attention
    cos = cosine(ref, unquantized_attention(q, oc.kv, w.n_kv))
    print(f"{name}: max|gpu-oracle| = {err:.2e}, cos(oracle, unquantised) = {cos:.5f}")


@pytest.mark.parametrize("pt", [None, 0])
@pytest.mark.parametrize("name", ["tiny", "gqa_small", "long_small", "3bit_small"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_matches_oracle_16bit_out(tq, name, dtype, pt):
    w, inp, oc, q, ref = oracle_case(name)
    got = gpu_decode(tq, w, inp, oc.cache, out_dtype=dtype, partition_tokens=pt)
    assert_decode_close(got, ref, dtype)


def test_decode_fp16_query(tq):
    w, inp, oc, q, ref = oracle_case("gqa_small")
    qh = inp.q.to(torch.float16)
    ref16 = oc.decode(qh.double().numpy())
    got = gpu_decode(tq, w, inp, oc.cache, q=qh)
    assert_decode_close(got, ref16, torch.float32)


@pytest.mark.parametrize("pt", [0, 16, 48, 128, 512, 4096])
def test_decode_partition_invariance(tq, pt):
    w, inp, oc, q, ref = oracle_case("gqa_small")
    got = gpu_decode(tq, w, inp, oc.cache, partition_tokens=pt)
    assert_decode_close(got, ref, torch.float32)


# TQ_FLAG_INDICES_READY only moves the reads of lengths and block ids before
# the split kernel's dependency wait: the same arithmetic, bit-identical output.
@pytest.mark.parametrize("name", ["gqa_small", "k3v4_small", "long_small"])
def test_decode_indices_ready_flag(tq, name):
    w, inp, oc, q, ref = oracle_case(name)
    plain = gpu_decode(tq, w, inp, oc.cache, partition_tokens=0)
    early = gpu_decode(tq, w, inp, oc.cache, partition_tokens=0, flags=tq.TQ_FLAG_INDICES_READY)
    assert np.array_equal(plain, early)
    assert_decode_close(early, ref, torch.float32)


# The reduce has two launch shapes: a CTA per query head when there are few
# (sequence, KV head) pairs (every small workload above), a CTA per pair when
# they outnumber half the SMs (40 x 8 = 320 pairs here).
@pytest.mark.parametrize("pt", [None, 0])
def test_decode_many_pairs(tq, pt):
    w, inp, oc, q, ref = oracle_case("k3v4_small", batch=40)
    got = gpu_decode(tq, w, inp, oc.cache, partition_tokens=pt)
    assert_decode_close(got, ref, torch.float32)


# Many pairs and no fixed partitions, with empty and 1-token sequences: the
# per-pair reduce shape writes the zero rows and merges one-record segments.
def test_decode_many_pairs_empty_and_single_token(tq):
    w, inp, oc, q, _ = oracle_case("k3v4_small", batch=40)
    lens = inp.seq_lens.clone()
    lens[0] = 0
    lens[7] = 1
    lens[39] = 0
    ref = oc.decode(q, seq_lens=lens.numpy())
    got = gpu_decode(tq, w, inp, oc.cache, seq_lens=lens, max_seq_len=int(inp.seq_lens.max()), partition_tokens=0)
    assert np.all(got[0] == 0.0) and np.all(got[39] == 0.0)
    assert_decode_close(got, ref, torch.float32)


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_decode_block_sizes(tq, bs):
    w, inp, oc, q, ref = oracle_case("gqa_small", block_size=bs)
    got = gpu_decode(tq, w, inp, oc.cache)
    assert_decode_close(got, ref, torch.float32)


@pytest.mark.parametrize("pt", [None, 0])
def test_decode_empty_and_single_token_sequences(tq, pt):
    w, inp, oc, q, _ = oracle_case("gqa_small")
    lens = inp.seq_lens.clone()
    lens[0] = 0
    lens[2] = 1
    ref = oc.decode(q, seq_lens=lens.numpy())
    got = gpu_decode(tq, w, inp, oc.cache, seq_lens=lens, max_seq_len=int(inp.seq_lens.max()), partition_tokens=pt)
    assert np.all(got[0] == 0.0)
    assert_decode_close(got, ref, torch.float32)


def test_decode_bad_block_id_is_flagged(tq):
    w, inp, oc, q, ref = oracle_case("gqa_small")
    table = inp.block_table.clone()
    table[1, 3] = inp.num_blocks + 7
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = gpu_decode(tq, w, inp, oc.cache, block_table=table, status=status)
    assert int(status.item()) & tq.TQ_DEV_BLOCK_OUT_OF_RANGE
    # sequences that do not touch the bad entry are unaffected
    assert_decode_close(got[[0, 2]], ref[[0, 2]], torch.float32)
    assert np.all(np.isfinite(got))


def test_decode_too_long_sequence_is_flagged(tq):
    w, inp, oc, q, ref = oracle_case("gqa_small")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = inp.seq_lens.clone()
    lens[1] = 10_000_000
    got = gpu_decode(tq, w, inp, oc.cache, seq_lens=lens, status=status,
                     max_seq_len=int(inp.seq_lens.max()))
    assert int(status.item()) & tq.TQ_DEV_SEQ_TOO_LONG
    assert np.all(np.isfinite(got))
    assert_decode_close(got[[0, 2]], ref[[0, 2]], torch.float32)


def test_decode_gqa_head_mapping_with_constant_values(tq):
    # KV head j holds constant value vectors (j + 1) / 4: query head h must
    # return (h // group + 1) / 4 whatever the keys are.
    w = workloads.get("gqa_small", lens=(20, 33, 16))
    inp = workloads.make_inputs(w)
    kv = []
    for b in range(w.batch):
        k, _ = inp.kv_for_sequence(b, "cpu")
        v = ((torch.arange(w.n_kv, dtype=torch.float32) + 1) / 4).view(1, -1, 1).expand(k.shape[0], -1, w.d)
        kv.append((k, v.to(k.dtype).contiguous()))
    oc = OracleCache(w, inp, kv).fill()
    got = gpu_decode(tq, w, inp, oc.cache)
    for h in range(w.n_q):
        np.testing.assert_allclose(got[:, h], (h // (w.n_q // w.n_kv) + 1) / 4, atol=1e-5)


def test_gpu_store_then_decode_end_to_end(tq):
    # GPU store + GPU decode compared with the oracle's own store + decode:
    # differences come only from boundary flips, which are rare.
    w, inp, oc, q, ref = oracle_case("long_small")
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, partition_tokens=w.partition_tokens)
    cb = tq.tq_build_codebook(128, 4)
    lay = tq.tq_layout_for(cfg)
    cache = torch.zeros(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device="cuda")
    k = torch.cat([x[0] for x in oc.kv]).cuda()
    v = torch.cat([x[1] for x in oc.kv]).cuda()
    tq.tq_store(cfg, cb, k, v, inp.fill_slots.cuda(), cache)
    got = gpu_decode(tq, w, inp, cache.cpu().numpy())
    assert_decode_close(got, ref, torch.float32)


@pytest.mark.parametrize("pt", [None, 0])
def test_decode_all_sequences_empty(tq, pt):
    w, inp, oc, q, _ = oracle_case("gqa_small")
    lens = torch.zeros_like(inp.seq_lens)
    got = gpu_decode(tq, w, inp, oc.cache, seq_lens=lens, max_seq_len=16, partition_tokens=pt)
    assert np.all(got == 0.0)


@pytest.mark.parametrize("pt", [None, 0])
def test_store_decode_dequant_capture_in_cuda_graph(tq, pt):
    # the calls only enqueue kernels (no allocation, no synchronisation), so a
    # serving step can be captured once and replayed: the replay must give
    # the eager results bit for bit, and the oracle's within the gates
    w, inp, oc, q, ref = oracle_case("gqa_small")
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size,
                         partition_tokens=w.partition_tokens if pt is None else pt)
    cb = tq.tq_build_codebook(w.d, 4)
    dev = torch.device("cuda", 0)
    base = torch.from_numpy(oc.cache).to(dev)
    cache = base.clone()
    table = inp.block_table.to(dev)
    lens = inp.seq_lens.to(dev)
    msl = inp.max_seq_len
    qd = inp.q.to(dev)
    # one new token per sequence, written over its last cached position
    g = torch.Generator().manual_seed(3)
    new_k = torch.randn((w.batch, w.n_kv, w.d), generator=g).to(torch.bfloat16).to(dev)
    new_v = torch.randn((w.batch, w.n_kv, w.d), generator=g).to(torch.bfloat16).to(dev)
    last = inp.seq_lens.to(torch.int64) - 1
    slots = (inp.block_table[torch.arange(w.batch), last // w.block_size].to(torch.int64) * w.block_size
             + last % w.block_size).to(dev)
    out = torch.empty((w.batch, w.n_q, w.d), dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_decode_workspace_size(cfg, w.batch, msl), dtype=torch.uint8, device=dev)
    kout = torch.empty((w.batch, msl, w.n_kv, w.d), dtype=torch.bfloat16, device=dev)
    vout = torch.empty_like(kout)

    def step():
        tq.tq_store(cfg, cb, new_k, new_v, slots, cache)
        tq.tq_decode(cfg, cb, qd, cache, table, lens, msl, out, ws)
        tq.tq_dequant(cfg, cb, cache, table, lens, msl, kout, vout)

    step()
    torch.cuda.synchronize()
    eager = (cache.clone(), out.clone(), kout.clone(), vout.clone())
    cache.copy_(base)
    out.zero_()
    kout.zero_()
    vout.zero_()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    cache.copy_(base)                  # capture ran nothing; start from the same cache
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (cache, out, kout, vout)):
        assert torch.equal(a, b)
    # the oracle: the same new tokens stored by the oracle, then its decode
    oc2 = OracleCache(w, inp).fill()
    from oracle import store as ost
    ost.store(new_k.double().cpu().numpy(), new_v.double().cpu().numpy(), slots.cpu().numpy(), oc2.cache, oc2.lay,
              oc2.preset, oc2.cent, oc2.mid)
    ref2 = oc2.decode(q)
    assert_decode_close(out.cpu().numpy(), ref2, torch.float32)
