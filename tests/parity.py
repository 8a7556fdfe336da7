"""Helpers shared by the GPU parity tests: oracle-side cache fills and the
element-by-element comparisons with their tolerances.

Tolerances (from the method's stated gates):
  * packed key indices bit-exact, except coordinates whose rotated value lies
    within 1e-5 of a decision midpoint; the mismatch fraction must stay <= 1e-4;
  * value codes bit-exact, except where (v - min) / s + 1/2 is within 1e-5 of
    an integer;
  * fp16 norm, scale and zero within 1 ulp (the norm compared against the
    oracle's norm for the GPU's own indices, so a boundary flip elsewhere in
    the vector does not count twice);
  * decode output: max |gpu - oracle| <= 2e-3 on fp32 output; for bf16/fp16
    output 2e-3 plus half an output ulp of the oracle value;
  * full dequant (derived from its arithmetic): index-coded keys within
    1e-6 * ||k|| per vector on fp32 output (stored_norm * c[idx] is one
    rounding, the 7 butterfly stages one each and the 1 / sqrt(d) scale one,
    so the error is at most 9 * 2^-24 * sum |stored_norm * c[idx_i]| / sqrt(d)
    <= 9 * 2^-24 * ||k||); FP8 keys exact (every e4m3 value is an f16, bf16
    and f32 value); values exactly the fp32 rounding of the oracle's value (one
    fused multiply-add of fp16 scale, integer code and fp16 zero); 16-bit
    outputs that plus half an output ulp (at least half the type's smallest
    subnormal step).
"""

from __future__ import annotations

import math

import numpy as np
import torch

import workloads
from oracle import codebook as ocb
from oracle import decode as od
from oracle import layout as olay
from oracle import numerics
from oracle import store as ost

def key_bits(preset: str):
    """Codebook bits of a preset's keys (None for e4m3 keys)."""
    return {"4bit_nc": 4, "k3v4_nc": 3, "3bit_nc": 3}.get(preset)


BOUNDARY_BAND = 1e-5
MAX_MISMATCH_FRACTION = 1e-4
DECODE_ATOL = 2e-3


class OracleCache:
    """Oracle-written cache for a workload (host uint8), with codebook and layout."""

    def __init__(self, w: workloads.Workload, inp: workloads.Inputs, kv=None):
        self.w = w
        self.inp = inp
        self.preset = olay.PRESETS[w.preset]
        self.lay = olay.tile_layout(self.preset, w.d, w.block_size, w.n_kv)
        if self.preset.key_fp8:
            self.cent = self.mid = None
        else:
            self.cent = ocb.codebook(w.d, self.preset.key_bits)
            self.mid = ocb.midpoints_fp32(self.cent)
        self.cache = np.zeros(inp.num_blocks * self.lay.block_bytes, dtype=np.uint8)
        self.kv = kv if kv is not None else [inp.kv_for_sequence(b, "cpu") for b in range(w.batch)]

    def fill(self, seqs=None, chunk=16384):
        """Oracle-store every token of the given sequences (all by default)."""
        seqs = range(self.w.batch) if seqs is None else seqs
        starts = dict(self.inp.fill_order)
        slots = self.inp.fill_slots.cpu().numpy()
        for b in seqs:
            k, v = self.kv[b]
            length = k.shape[0]
            s0 = starts[b]
            for c0 in range(0, length, chunk):
                c1 = min(length, c0 + chunk)
                ost.store(k[c0:c1].double().numpy(), v[c0:c1].double().numpy(), slots[s0 + c0: s0 + c1],
                          self.cache, self.lay, self.preset, self.cent, self.mid)
        return self

    def decode(self, q: np.ndarray, heads=None, seq_lens=None):
        lens = self.inp.seq_lens.cpu().numpy() if seq_lens is None else seq_lens
        return od.decode(q, self.cache, self.lay, self.preset, self.cent,
                         self.inp.block_table.cpu().numpy(), lens, heads=heads)


def compare_store(gpu_cache: np.ndarray, oc: OracleCache, k: np.ndarray, v: np.ndarray, slots: np.ndarray):
    """Compare GPU-written slots with the oracle's quantisation of the same
    inputs (k, v [N, n_kv, d] float64; slots [N]). Returns a stats dict and
    raises AssertionError on a gate violation."""
    lay, preset = oc.lay, oc.preset
    d = oc.w.d
    n_tok, n_kv, _ = k.shape
    ok = slots >= 0
    k, v, slots = k[ok], v[ok], slots[ok]
    rows_k = k.reshape(-1, d)
    rows_v = v.reshape(-1, d)
    if preset.key_fp8:
        kinfo = {"packed": numerics.e4m3_encode(rows_k)}
    else:
        kinfo = ost.quantize_keys(rows_k, oc.cent, oc.mid, preset.key_bits, preset.norm_correction)
    vinfo = ost.quantize_values(rows_v, preset.value_bits)
    blocks = slots // lay.block_size
    offs = slots % lay.block_size
    stats = {"key_coords": 0, "key_mismatch": 0, "value_coords": 0, "value_mismatch": 0}
    for h in range(n_kv):
        kb, vb, kn, vs, vz = od.read_positions(gpu_cache, lay, blocks, offs, h)
        rows = np.arange(len(slots)) * n_kv + h
        # ---- keys
        if preset.key_fp8:
            assert np.array_equal(kb, kinfo["packed"][rows]), "e4m3 key bytes differ"
            stats["key_coords"] += kb.size
        else:
            gidx = ost.unpack_bits(kb, preset.key_bits, d)
            oidx = kinfo["idx"][rows]
            y = kinfo["y"][rows]
            near = np.min(np.abs(y[:, :, None] - oc.mid.astype(np.float64)[None, None, :]), axis=-1) < BOUNDARY_BAND
            mism = gidx != oidx
            assert not np.any(mism & ~near), f"key index mismatch away from a boundary (head {h})"
            assert np.all(np.abs(gidx - oidx) <= 1)
            stats["key_coords"] += gidx.size
            stats["key_mismatch"] += int(mism.sum())
            # stored norm vs the oracle's norm correction for the GPU's own indices
            c = oc.cent.astype(np.float64)
            n = kinfo["norm"][rows]
            expect = numerics.fp16_bits(n / np.sqrt((c[gidx] ** 2).sum(-1) + 1e-16)).astype(np.int64)
            assert np.all(np.abs(kn.astype(np.int64) - expect) <= 1), "key norm off by more than 1 ulp"
        # ---- values
        gq = ost.unpack_bits(vb, preset.value_bits, d)
        oq = vinfo["codes"][rows]
        t = (rows_v[rows].astype(np.float32) - vinfo["min32"][rows][:, None]) / vinfo["scale32"][rows][:, None] + 0.5
        near_v = np.abs(t - np.round(t)) < BOUNDARY_BAND
        vm = gq != oq
        assert not np.any(vm & ~near_v), f"value code mismatch away from a rounding boundary (head {h})"
        stats["value_coords"] += gq.size
        stats["value_mismatch"] += int(vm.sum())
        assert np.all(np.abs(vs.astype(np.int64) - vinfo["scale_bits"][rows].astype(np.int64)) <= 1)
        assert np.all(np.abs(vz.astype(np.int64) - vinfo["zero_bits"][rows].astype(np.int64)) <= 1)
    if stats["key_coords"]:
        assert stats["key_mismatch"] / stats["key_coords"] <= MAX_MISMATCH_FRACTION
    assert stats["value_mismatch"] / max(1, stats["value_coords"]) <= MAX_MISMATCH_FRACTION
    return stats


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    mant = {torch.bfloat16: 8, torch.float16: 11, torch.float32: 24}[dtype]
    ax = np.maximum(np.abs(x), 1e-30)
    return 0.5 * np.exp2(np.floor(np.log2(ax)) - (mant - 1))


def assert_decode_close(gpu: np.ndarray, ref: np.ndarray, dtype: torch.dtype):
    err = np.abs(gpu.astype(np.float64) - ref)
    tol = DECODE_ATOL + (0 if dtype == torch.float32 else half_ulp(ref, dtype))
    bad = err > tol
    assert not np.any(bad), f"decode error {err.max():.3e} exceeds tolerance (worst at {np.unravel_index(err.argmax(), err.shape)})"
    return float(err.max())


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = a.reshape(-1).astype(np.float64)
    b = b.reshape(-1).astype(np.float64)
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def unquantized_attention(q: np.ndarray, kv, n_kv: int, scale=None):
    """Plain softmax attention on the unquantised inputs (for the reported cosine)."""
    bsz, n_q, d = q.shape
    group = n_q // n_kv
    scale = 1 / math.sqrt(d) if scale is None else scale
    out = np.zeros_like(q)
    for b in range(bsz):
        k, v = kv[b]
        k = k.double().numpy()
        v = v.double().numpy()
        if k.shape[0] == 0:
            continue
        for h in range(n_q):
            s = k[:, h // group] @ q[b, h] * scale
            e = np.exp(s - s.max())
            out[b, h] = (e / e.sum()) @ v[:, h // group]
    return out


_MANT = {torch.bfloat16: 8, torch.float16: 11, torch.float32: 24}
_MIN_HALF_STEP = {torch.bfloat16: 2.0 ** -134, torch.float16: 2.0 ** -25, torch.float32: 2.0 ** -150}


def _half_ulp_floor(x, dtype):
    ax = np.maximum(np.abs(x), 1e-300)
    return np.maximum(0.5 * np.exp2(np.floor(np.log2(ax)) - (_MANT[dtype] - 1)), _MIN_HALF_STEP[dtype])


def assert_dequant_close(gk, gv, rk, rv, dtype, fp8_keys):
    """Element-by-element gate of the module docstring; returns the max errors."""
    assert np.all(np.isfinite(gk)) and np.all(np.isfinite(gv)), "an output element was not written"
    ek = np.abs(gk - rk)
    if fp8_keys:
        assert np.all(ek == 0), f"FP8 key mismatch {ek.max():.3e}"
    else:
        tol32 = 1e-6 * np.linalg.norm(rk, axis=-1, keepdims=True)
        tol = tol32 if dtype == torch.float32 else tol32 + _half_ulp_floor(np.abs(rk) + tol32, dtype)
        assert np.all(ek <= tol), f"key error {ek.max():.3e} over tolerance"
    ev = np.abs(gv - rv)
    if dtype == torch.float32:
        assert np.array_equal(gv, rv.astype(np.float32).astype(np.float64)), f"value mismatch {ev.max():.3e}"
    else:
        tol = 2.0 ** -24 * np.abs(rv) + _half_ulp_floor(np.abs(rv) * (1 + 2.0 ** -23), dtype)
        assert np.all(ev <= tol), f"value error {ev.max():.3e} over tolerance"
    return float(ek.max()), float(ev.max())
