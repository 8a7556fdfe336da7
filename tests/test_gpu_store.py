"""GPU parity of tq_store against the oracle (through the C ABI binding)."""

import numpy as np
import pytest
import torch

import workloads
from parity import OracleCache, compare_store, key_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from turboquant_paged_kv_gb300 import build
    build.build()
    import turboquant_paged_kv_gb300 as tq
    return tq


def _gpu_fill(tq, w, inp, kv_cpu, status=None):
    lay = tq.tq_layout_for(tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size))
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size)
    cb = None if w.preset == "k8v4" else tq.tq_build_codebook(w.d, key_bits(w.preset))
    cache = torch.full((inp.num_blocks * lay.block_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    k = torch.cat([kv[0] for kv in kv_cpu]).cuda()
    v = torch.cat([kv[1] for kv in kv_cpu]).cuda()
    slots = inp.fill_slots.cuda()
    tq.tq_store(cfg, cb, k, v, slots, cache, dev_status=status)
    torch.cuda.synchronize()
    return cache, cfg, cb


@pytest.mark.parametrize("name,bs", [("tiny", 16), ("gqa_small", 16), ("gqa_small", 32), ("gqa_small", 64),
                                     ("gqa_small", 128), ("k3v4_small", 16), ("k8v4_small", 16),
                                     ("long_small", 16), ("3bit_small", 16), ("3bit_small", 64)])
def test_store_matches_oracle(tq, name, bs):
    w = workloads.get(name, block_size=bs)
    inp = workloads.make_inputs(w)
    kv = [inp.kv_for_sequence(b, "cpu") for b in range(w.batch)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache, _, _ = _gpu_fill(tq, w, inp, kv, status)
    assert int(status.item()) == 0
    oc = OracleCache(w, inp, kv)
    k = torch.cat([x[0] for x in kv]).double().numpy()
    v = torch.cat([x[1] for x in kv]).double().numpy()
    stats = compare_store(cache.cpu().numpy(), oc, k, v, inp.fill_slots.numpy())
    assert stats["key_coords"] > 0


def test_store_negative_slots_write_nothing(tq):
    w = workloads.get("gqa_small")
    inp = workloads.make_inputs(w)
    kv = [inp.kv_for_sequence(b, "cpu") for b in range(w.batch)]
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv)
    cb = tq.tq_build_codebook(128, 4)
    lay = tq.tq_layout_for(cfg)
    cache = torch.full((inp.num_blocks * lay.block_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    k = torch.cat([x[0] for x in kv]).cuda()
    v = torch.cat([x[1] for x in kv]).cuda()
    slots = inp.fill_slots.clone()
    drop = torch.arange(slots.numel()) % 3 == 1
    slots[drop] = -1
    tq.tq_store(cfg, cb, k, v, slots.cuda(), cache)
    host = cache.cpu().numpy()
    oc = OracleCache(w, inp, kv)
    compare_store(host, oc, k.cpu().double().numpy(), v.cpu().double().numpy(), slots.numpy())
    # every byte of a dropped token's slot (every head) is still the sentinel
    from oracle import decode as od
    s = inp.fill_slots[drop].numpy()
    for h in range(w.n_kv):
        kb, vb, kn, vs, vz = od.read_positions(host, oc.lay, s // 16, s % 16, h)
        assert np.all(kb == 0xA5) and np.all(vb == 0xA5)
        assert np.all(kn == 0xA5A5) and np.all(vs == 0xA5A5) and np.all(vz == 0xA5A5)


def test_store_out_of_range_slot_is_flagged_and_skipped(tq):
    cfg = tq.make_config("4bit_nc", 8, 2)
    cb = tq.tq_build_codebook(128, 4)
    lay = tq.tq_layout_for(cfg)
    nb = 3
    cache = torch.zeros(nb * lay.block_bytes, dtype=torch.uint8, device="cuda")
    k = torch.randn(3, 2, 128, device="cuda").to(torch.bfloat16)
    slots = torch.tensor([5, nb * 16 + 1, -4], dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_store(cfg, cb, k, k, slots, cache, dev_status=status)
    assert int(status.item()) & tq.TQ_DEV_SLOT_OUT_OF_RANGE
    ref = torch.zeros_like(cache)
    tq.tq_store(cfg, cb, k[:1], k[:1], slots[:1], ref)
    assert torch.equal(cache, ref)


def test_store_empty_is_noop(tq):
    cfg = tq.make_config("4bit_nc", 8, 2)
    cb = tq.tq_build_codebook(128, 4)
    cache = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    e = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    tq.tq_store(cfg, cb, e, e, torch.empty(0, dtype=torch.int64, device="cuda"), cache)
    assert int(cache.sum()) == 0
