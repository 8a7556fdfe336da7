"""tq_decode_noalloc: tq_decode with the library's fixed device scratch array.

Collected last on purpose: the GPU tests also hold when the entry point's
first call (its per-device set-up) happens after every other test has run, and
they pass alone in a fresh process because the fixture builds and loads the
library itself.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads


@pytest.fixture(scope="module")
def tq():
    import os
    import shutil
    from turboquant_paged_kv_gb300 import build
    # the host-side test below needs the library but no GPU: build it where a
    # CUDA toolkit is present, else use an existing build, else skip
    nvcc = os.path.exists(build.NVCC) or shutil.which("nvcc")
    if nvcc:
        build.build()
    elif not os.path.exists(build.LIB_PATH):
        pytest.skip("libtq.so is not built and no nvcc is available to build it")
    import turboquant_paged_kv_gb300 as tq
    return tq


def _largest_batch_that_fits(tq, cfg, max_seq_len):
    lo, hi = 0, 1 << 20
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if tq.tq_decode_workspace_size(cfg, mid, max_seq_len) <= tq.TQ_DECODE_NOALLOC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_oversized_problem_is_rejected_before_any_cuda_call(tq):
    from turboquant_paged_kv_gb300 import _abi
    lib = _abi.load()
    cfg = tq.make_config("4bit_nc", 32, 8, partition_tokens=512)
    cb = tq.tq_build_codebook(128, 4)
    msl = 4096
    fit = _largest_batch_that_fits(tq, cfg, msl)
    assert 0 < fit < (1 << 20)
    assert tq.tq_decode_workspace_size(cfg, fit + 1, msl) > tq.TQ_DECODE_NOALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p(0x10000)
    call = lambda cfg_, batch: lib.tq_decode_noalloc(  # noqa: E731
        ctypes.byref(cfg_), ctypes.byref(cb), p, 1, p, 10, p, 4, p, batch, msl, 0.0, p, 2, None, None)
    # no GPU is needed for either answer: both return before the set-up
    assert call(cfg, fit + 1) == _abi.TQ_ERR_WORKSPACE_TOO_SMALL
    assert call(tq.make_config("4bit_nc", 30, 8), 2) == _abi.TQ_ERR_INVALID_ARG
    with pytest.raises(tq.TQError, match="workspace"):
        _abi.check("tq_decode_noalloc", call(cfg, fit + 1))


def _gpu_case(tq, name, **over):
    w = workloads.get(name, **over)
    dev = torch.device("cuda", 0)
    inp = workloads.make_inputs(w, device=dev)
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size,
                         partition_tokens=w.partition_tokens)
    bits = {"4bit_nc": 4, "k3v4_nc": 3}.get(w.preset)
    cb = tq.tq_build_codebook(w.d, bits) if bits else None
    lay = tq.tq_layout_for(cfg)
    cache = torch.zeros(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device=dev)
    for b in range(w.batch):
        k, v = inp.kv_for_sequence(b, dev)
        s0 = dict(inp.fill_order)[b]
        tq.tq_store(cfg, cb, k, v, inp.fill_slots[s0:s0 + k.shape[0]], cache)
    return w, inp, cfg, cb, cache


def _with_workspace(tq, cfg, cb, q, cache, table, lens, msl, out_dtype):
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=q.device)
    ws = torch.empty(tq.tq_decode_workspace_size(cfg, q.shape[0], msl), dtype=torch.uint8, device=q.device)
    tq.tq_decode(cfg, cb, q, cache, table, lens, msl, out, ws)
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("name,out_dtype", [("gqa_small", torch.float32), ("k8v4_small", torch.bfloat16)])
def test_two_calls_in_a_row_match_tq_decode(tq, name, out_dtype):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    w, inp, cfg, cb, cache = _gpu_case(tq, name)
    msl = int(inp.seq_lens.max())
    # call 1: the workload as given; call 2: another query and shorter
    # sequences, so stale partials of call 1 are left in the scratch array
    q2 = torch.randn(inp.q.shape, generator=torch.Generator().manual_seed(99)).to(inp.q.dtype).cuda()
    lens2 = (inp.seq_lens * 2 // 3).clamp(min=1).to(torch.int32)
    calls = [(inp.q, inp.seq_lens), (q2, lens2)]
    refs = [_with_workspace(tq, cfg, cb, q, cache, inp.block_table, lens, msl, out_dtype) for q, lens in calls]
    outs = [torch.full(inp.q.shape, float("nan"), dtype=out_dtype, device="cuda") for _ in calls]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_decode_noalloc(cfg, cb, calls[0][0], cache, inp.block_table, calls[0][1], msl, outs[0],
                         dev_status=status)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    tq.tq_decode_noalloc(cfg, cb, calls[1][0], cache, inp.block_table, calls[1][1], msl, outs[1],
                         dev_status=status)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, "the second call changed free device memory"
    assert int(status.item()) == 0
    for got, ref in zip(outs, refs):
        g = got.float().cpu().numpy()
        r = ref.float().cpu().numpy()
        assert np.all(np.isfinite(g))
        # the same kernels on the same inputs with the same launch shape: the
        # results must agree bit for bit (a stale partial left in the shared
        # array by the first call would show here)
        assert np.array_equal(g, r), f"{name}: max|noalloc - tq_decode| = {np.abs(g - r).max():.2e}"
