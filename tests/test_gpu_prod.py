"""GPU parity of the TurboQuant_prod key path (tq_prod_store, tq_prod_scores)
against the oracle (oracle.qjl), through the C ABI binding.

Gates (derived from the arithmetic; the oracle computes in float64):
  * Lloyd-Max indices bit-exact except coordinates whose rotated value is
    within 1e-5 of a midpoint (as for the MSE presets), mismatch fraction
    <= 1e-4;
  * sign bits: the oracle's signs of S r for the GPU's own indices, exact
    except where |(S r)_i| <= 1e-5 * ||S_i|| * ||r|| (the kernel's fp32 sum of
    128 products errs by at most 128 * 2^-24 * ||S_i|| ||r|| ~ 7.6e-6 of it,
    plus the fp32 rotation's error in r); mismatch fraction <= 1e-4;
  * fp16 key norm and residual norm within 1 ulp (the residual norm that of
    the GPU's indices);
  * scores within 3e-4 * M of the oracle's estimate from the same cache, with
    M = scale * ||k|| * (sum_j |q_r,j c[idx_j]| + sqrt(pi/2) / d * ||r|| *
    sum_j |(S q_r)_j|), the sum of the absolute terms of the estimate: the
    kernel's products take q_r and S q_r rounded to fp16 (at most 2^-12
    relative each; the bit operands are exact and the sums are of the same
    rounded values) and accumulate in fp32 (128-term sums, ~1e-5 of M), so
    its error stays below (2^-12 + 3e-5) * M.
"""

import math

import numpy as np
import pytest
import torch

import workloads
from oracle import codebook as ocb
from oracle import qjl
from oracle import rotation

pytestmark = pytest.mark.gpu

IDX_BAND = 1e-5
SIGN_BAND = 1e-5
MAX_MISMATCH_FRACTION = 1e-4
SCORE_RTOL = 3e-4


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need CUDA")
    from turboquant_paged_kv_gb300 import build
    build.build()
    import turboquant_paged_kv_gb300 as tq
    return tq


class Case:
    def __init__(self, tq, w):
        self.w = w
        self.inp = workloads.make_inputs(w)
        self.cfg = tq.make_config("prod3", w.n_q, w.n_kv, block_size=w.block_size)
        self.lay = tq.tq_prod_layout_for(self.cfg)
        self.olay = qjl.prod_tile_layout(w.d, w.block_size, w.n_kv, 2)
        self.cb = tq.tq_build_codebook(w.d, 2)
        self.cent = ocb.codebook(w.d, 2)
        self.mid = ocb.midpoints_fp32(self.cent)
        self.S = workloads.projection(w)
        self.keys = [self.inp.kv_for_sequence(b, "cpu")[0] for b in range(w.batch)]

    def fill(self, tq, status=None):
        cache = torch.full((self.inp.num_blocks * self.lay.block_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
        k = torch.cat(self.keys).cuda() if self.keys else torch.zeros(0, self.w.n_kv, self.w.d, dtype=self.w.torch_dtype, device="cuda")
        tq.tq_prod_store(self.cfg, self.cb, self.S.cuda(), k, self.inp.fill_slots.cuda(), cache, dev_status=status)
        torch.cuda.synchronize()
        return cache

    def scores(self, tq, cache, q=None, max_seq_len=None, seq_lens=None, block_table=None, scale=0.0, status=None):
        q = self.inp.q if q is None else q
        lens = self.inp.seq_lens if seq_lens is None else seq_lens
        table = self.inp.block_table if block_table is None else block_table
        L = self.inp.max_seq_len if max_seq_len is None else max_seq_len
        out = torch.full((self.w.batch, self.w.n_q, L), float("nan"), dtype=torch.float32, device="cuda")
        ws = torch.empty(tq.tq_prod_scores_workspace_size(self.cfg, self.w.batch), dtype=torch.uint8, device="cuda")
        tq.tq_prod_scores(self.cfg, self.cb, self.S.cuda(), q.cuda(), cache, table.cuda(), lens.cuda(), L, out, ws,
                          scale=scale, dev_status=status)
        torch.cuda.synchronize()
        return out.cpu().numpy()


def compare_prod_store(c: Case, gpu_cache: np.ndarray):
    w, lay = c.w, c.olay
    k = torch.cat(c.keys).double().numpy()
    slots = c.inp.fill_slots.numpy()
    rows_k = k.reshape(-1, w.d)
    S = c.S.double().numpy()
    info = qjl.prod_quantize(rows_k, S, c.cent, c.mid, 2)
    blocks, offs = slots // w.block_size, slots % w.block_size
    stats = {"coords": 0, "idx_mismatch": 0, "sign_mismatch": 0}
    s_norm = np.linalg.norm(S, axis=1)
    for h in range(w.n_kv):
        rows = np.arange(len(slots)) * w.n_kv + h
        gidx, gsigns, gnorm, grnorm = qjl.prod_read(gpu_cache, lay, blocks, offs, h)
        oidx, y = info["idx"][rows], info["y"][rows]
        near = np.min(np.abs(y[:, :, None] - c.mid.astype(np.float64)[None, None, :]), axis=-1) < IDX_BAND
        mism = gidx != oidx
        assert not np.any(mism & ~near), f"index mismatch away from a midpoint (head {h})"
        mine = qjl.prod_quantize(rows_k[rows], S, c.cent, c.mid, 2, idx=gidx)
        osigns = 2.0 * mine["sign_bits"] - 1.0
        band = SIGN_BAND * s_norm[None, :] * mine["rnorm"][:, None]
        smism = gsigns != osigns
        assert not np.any(smism & (np.abs(mine["proj"]) > band)), f"sign mismatch away from zero (head {h})"
        assert np.all(np.abs(_bits(gnorm) - info["norm_bits"][rows].astype(np.int64)) <= 1), "key norm off by > 1 ulp"
        assert np.all(np.abs(_bits(grnorm) - mine["rnorm_bits"].astype(np.int64)) <= 1), "residual norm off by > 1 ulp"
        stats["coords"] += gidx.size
        stats["idx_mismatch"] += int(mism.sum())
        stats["sign_mismatch"] += int(smism.sum())
    assert stats["idx_mismatch"] <= MAX_MISMATCH_FRACTION * stats["coords"]
    assert stats["sign_mismatch"] <= MAX_MISMATCH_FRACTION * stats["coords"]
    return stats


def _bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16).astype(np.int64)


def assert_scores_close(c: Case, gpu: np.ndarray, host_cache: np.ndarray, q: np.ndarray, lens, table, L, scale):
    S = c.S.double().numpy()
    ref = qjl.prod_scores(q, S, host_cache, c.olay, c.cent, table, lens, L, scale)
    sc = 1.0 / math.sqrt(c.w.d) if scale <= 0 else scale
    group = c.w.n_q // c.w.n_kv
    cent = c.cent.astype(np.float32).astype(np.float64)
    bound = np.zeros_like(ref)
    for b in range(c.w.batch):
        n = int(lens[b])
        if n == 0:
            continue
        pos = np.arange(n)
        blocks = np.asarray(table[b])[pos // c.w.block_size]
        for h in range(c.w.n_kv):
            idx, _, norm, rnorm = qjl.prod_read(host_cache, c.olay, blocks, pos % c.w.block_size, h)
            heads = list(range(h * group, (h + 1) * group))
            qr = rotation.rotate(q[b, heads])                     # [G, d]
            mse_abs = np.abs(qr) @ np.abs(cent[idx]).T            # [G, n]
            qjl_abs = np.abs(qr @ S.T).sum(-1)                    # [G]
            bound[b, heads, :n] = sc * norm * (mse_abs + math.sqrt(math.pi / 2) / c.w.d * rnorm * qjl_abs[:, None])
    assert np.all(np.isfinite(gpu)), "a score was not written"
    err = np.abs(gpu - ref)
    bad = err > SCORE_RTOL * bound + 1e-30
    assert not np.any(bad), f"score error {err.max():.3e} (worst at {np.unravel_index(err.argmax(), err.shape)})"
    return float((err / np.maximum(bound, 1e-30)).max())


@pytest.mark.parametrize("name,bs,overrides", [("prod_small", 16, {}), ("prod_small", 64, {}),
                                                ("prod_small", 32, {"dtype": "fp16"}),
                                                ("prod_small", 128, {"n_q": 64})])
def test_prod_store_and_scores_match_oracle(tq, name, bs, overrides):
    c = Case(tq, workloads.get(name, block_size=bs, **overrides))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache = c.fill(tq, status)
    assert int(status.item()) == 0
    host = cache.cpu().numpy()
    stats = compare_prod_store(c, host)
    assert stats["coords"] > 0
    gpu = c.scores(tq, cache, status=status)
    assert int(status.item()) == 0
    assert_scores_close(c, gpu, host, c.inp.q.double().numpy(), c.inp.seq_lens.numpy(),
                        c.inp.block_table.numpy(), c.inp.max_seq_len, 0.0)


def test_prod_scores_ragged_and_padded(tq):
    """An empty sequence, max_seq_len past every length (rows zero-padded) and
    an explicit scale."""
    w = workloads.get("prod_small", lens=(0, 45, 16), n_q=8, n_kv=8)
    c = Case(tq, w)
    cache = c.fill(tq)
    L = 77
    gpu = c.scores(tq, cache, max_seq_len=L, scale=0.25)
    assert np.all(gpu[0] == 0) and np.all(gpu[1, :, 45:] == 0) and np.all(gpu[2, :, 16:] == 0)
    assert_scores_close(c, gpu, cache.cpu().numpy(), c.inp.q.double().numpy(), c.inp.seq_lens.numpy(),
                        c.inp.block_table.numpy(), L, 0.25)


def test_prod_store_negative_and_out_of_range_slots(tq):
    w = workloads.get("prod_small", lens=(40,), batch=1)
    c = Case(tq, w)
    cache = torch.full((c.inp.num_blocks * c.lay.block_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    k = c.keys[0].cuda()
    slots = torch.full((40,), -1, dtype=torch.int64)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.tq_prod_store(c.cfg, c.cb, c.S.cuda(), k, slots.cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and bool((cache == 0xA5).all())
    slots[3] = c.inp.num_blocks * w.block_size + 5      # past the cache
    tq.tq_prod_store(c.cfg, c.cb, c.S.cuda(), k, slots.cuda(), cache, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1 and bool((cache == 0xA5).all())


def test_prod_scores_bad_block_is_flagged(tq):
    w = workloads.get("prod_small", lens=(40, 20), batch=2)
    c = Case(tq, w)
    cache = c.fill(tq)
    table = c.inp.block_table.clone()
    table[1, 0] = c.inp.num_blocks + 3
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu = c.scores(tq, cache, block_table=table, status=status)
    assert int(status.item()) & 2
    assert np.all(gpu[1, :, :16] == 0) and np.all(np.isfinite(gpu))   # the tile of the bad block reads as 0


@pytest.mark.parametrize("n_tok", [1, 127, 129, 1000])
def test_prod_store_group_tails(tq, n_tok):
    """Token counts around the store's 128-vector groups (n_kv = 1: vectors =
    tokens), each slot compared with the oracle."""
    w = workloads.get("prod_small", lens=(n_tok,), batch=1, n_q=2, n_kv=1)
    c = Case(tq, w)
    compare_prod_store(c, c.fill(tq).cpu().numpy())
