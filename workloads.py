"""Seeded synthetic workloads for the TurboQuant paged-KV store and decode.

This module only draws inputs (queries, keys, values, sequence lengths, block
tables, slot mappings); it holds none of the quantisation or attention
arithmetic, so the tests, the benchmark and the reference oracle can all
consume the same tensors without sharing any of the method's code.

Every tensor comes from a ``torch.Generator`` seeded from (workload seed,
tensor kind, sequence index), so any one sequence can be regenerated on its
own, on the CPU or on a GPU (the two devices give different but equally
seeded streams; a test always hands the very same tensors to both sides).
Values are drawn in float32 and cast round-to-nearest-even to the workload's
input dtype (fp16 or bf16); the oracle reads the exact cast values.

Workloads (shapes follow the TurboQuant paged-cache setting: d = 128,
block_size = 16):

  tiny      4bit_nc, n_q = n_kv = 1, 2 sequences of 37 and 128 tokens; K, V
            fp16 N(0,1) with channels 3 and 77 scaled x10; q fp16 N(0,1).
  gqa       4bit_nc, batch 32 x 4096 tokens, n_q 32 / n_kv 8; q, K, V bf16
            N(0,1) with one outlier channel (1% of d, rounded up to one) per
            tensor and head scaled x8; block table a random permutation.
  k3v4      k3v4_nc, batch 64, lengths uniform in [512, 16384]; bf16 N(0,1);
            512-token split-K partitions.
  k8v4      k8v4, batch 128 x 8192; plus a store of an 8192-token bf16 prefill
            chunk through a random slot mapping into 512 fresh blocks.
  long      4bit_nc, batch 4 x 131072, n_q 64 / n_kv 8; bf16 N(0,1) K, V with
            one channel per head drawn Student-t (nu = 3); 256 partitions of 512.
  3bit      3bit_nc (3-bit keys and values) on the gqa shape and distributions.
  prod      prod3 keys (2-bit Lloyd-Max code + 1-bit QJL residual signs) on the
            gqa shape and distributions; the QJL projection S is d x d
            float32 N(0, 1) (``projection``).

``*_small`` variants keep the head structure and distributions with a few
hundred tokens per sequence so the CPU oracle finishes in seconds.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

__all__ = ["Workload", "WORKLOADS", "get", "Inputs", "make_inputs", "projection"]

_KIND = {"q": 1, "k": 2, "v": 3, "lens": 4, "perm": 5, "slots": 6, "ch": 7,
         "sk": 8, "sv": 9, "proj": 10}


@dataclass(frozen=True)
class Workload:
    name: str
    preset: str
    batch: int
    n_q: int
    n_kv: int
    lens: tuple = ()                 # fixed lengths, or () with len_range
    len_range: tuple = ()            # (lo, hi) inclusive uniform draw
    fixed_len: int = 0               # every sequence this long
    d: int = 128
    block_size: int = 16
    dtype: str = "bf16"
    partition_tokens: int = 512
    outlier: str = "none"            # none | fixed10 | one_x8 | student_t
    store_tokens: int = 0            # extra prefill chunk stored via random slots
    store_extra_blocks: int = 0
    seed: int = 0
    note: str = ""

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16


WORKLOADS = {
    "tiny": Workload("tiny", "4bit_nc", 2, 1, 1, lens=(37, 128), dtype="fp16",
                     outlier="fixed10", note="2 seqs of 37 and 128 tokens"),
    "gqa": Workload("gqa", "4bit_nc", 32, 32, 8, fixed_len=4096, outlier="one_x8",
                    note="batch 32 x ctx 4096, n_q 32, n_kv 8"),
    "k3v4": Workload("k3v4", "k3v4_nc", 64, 32, 8, len_range=(512, 16384),
                     note="batch 64, ctx U[512,16384]"),
    "k8v4": Workload("k8v4", "k8v4", 128, 32, 8, fixed_len=8192, store_tokens=8192,
                     store_extra_blocks=512, note="batch 128 x ctx 8192 + 8192-token store"),
    "long": Workload("long", "4bit_nc", 4, 64, 8, fixed_len=131072, outlier="student_t",
                     note="batch 4 x ctx 131072, n_q 64, n_kv 8"),
    # oracle-sized variants: same heads and distributions, ragged short lengths
    "gqa_small": Workload("gqa_small", "4bit_nc", 3, 32, 8, lens=(300, 517, 64),
                          outlier="one_x8", partition_tokens=128),
    "k3v4_small": Workload("k3v4_small", "k3v4_nc", 3, 32, 8, len_range=(40, 700),
                           partition_tokens=128),
    "k8v4_small": Workload("k8v4_small", "k8v4", 3, 32, 8, lens=(257, 16, 400),
                           store_tokens=300, store_extra_blocks=24, partition_tokens=128),
    "long_small": Workload("long_small", "4bit_nc", 2, 64, 8, lens=(1500, 333),
                           outlier="student_t", partition_tokens=256),
    # 3bit_nc (3-bit keys and 3-bit values) on the gqa shape
    "3bit": Workload("3bit", "3bit_nc", 32, 32, 8, fixed_len=4096, outlier="one_x8",
                     note="batch 32 x ctx 4096, n_q 32, n_kv 8, 3-bit K and V"),
    "3bit_small": Workload("3bit_small", "3bit_nc", 3, 32, 8, lens=(300, 517, 64),
                           outlier="one_x8", partition_tokens=128),
    # TurboQuant_prod keys (key-only cache) on the gqa shape
    "prod": Workload("prod", "prod3", 32, 32, 8, fixed_len=4096, outlier="one_x8",
                     note="batch 32 x ctx 4096, n_q 32, n_kv 8, 2-bit code + QJL signs"),
    "prod_small": Workload("prod_small", "prod3", 3, 32, 8, lens=(300, 517, 64), outlier="one_x8"),
}


def get(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def _gen(w: Workload, kind: str, index: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(((w.seed * 1000003 + _KIND[kind]) * 1000033 + index) & 0x7FFFFFFFFFFF)
    return g


def _outlier_channels(w: Workload, kind: str, heads: int) -> torch.Tensor:
    """One seeded channel per head (CPU generator, so it is device independent)."""
    g = _gen(w, "ch", _KIND[kind], "cpu")
    return torch.randint(0, w.d, (heads,), generator=g)


def _draw(w: Workload, kind: str, index: int, shape, device) -> torch.Tensor:
    """float32 N(0,1) draws [..., heads, d] with the workload's outlier recipe."""
    g = _gen(w, kind, index, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    heads = shape[-2]
    if w.outlier == "fixed10" and kind in ("k", "v", "sk", "sv"):
        x[..., 3] *= 10.0
        x[..., 77] *= 10.0
    elif w.outlier == "one_x8":
        ch = _outlier_channels(w, kind, heads).to(device)
        x[..., torch.arange(heads, device=device), ch] *= 8.0
    elif w.outlier == "student_t" and kind in ("k", "v", "sk", "sv"):
        ch = _outlier_channels(w, kind, heads).to(device)
        lead = shape[:-2]
        z = torch.randn(lead + (heads, 4), generator=g, device=device, dtype=torch.float32)
        chi2 = (z[..., 1:] ** 2).sum(-1) / 3.0
        t = z[..., 0] / torch.sqrt(chi2)
        x[..., torch.arange(heads, device=device), ch] = t
    return x.to(w.torch_dtype)


@dataclass
class Inputs:
    """All host-side structure of one workload (tensors on ``device``)."""
    w: Workload
    seq_lens: torch.Tensor           # [B] int32
    block_table: torch.Tensor        # [B, max_blocks] int32, padded with -1
    num_blocks: int                  # physical blocks in the cache
    q: torch.Tensor                  # [B, n_q, d]
    fill_slots: torch.Tensor         # [sum(L)] int64, slot of every cached token
    fill_order: list = field(default_factory=list)   # (b, start) per sequence

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.seq_lens.numel() else 0

    def kv_for_sequence(self, b: int, device=None):
        """K, V [L_b, n_kv, d] of sequence b (regenerated from its own seeds)."""
        device = device or self.q.device
        length = int(self.seq_lens[b])
        shape = (length, self.w.n_kv, self.w.d)
        return _draw(self.w, "k", b, shape, device), _draw(self.w, "v", b, shape, device)

    def store_chunk(self, device=None):
        """The extra prefill chunk (k, v [N, n_kv, d], slot_mapping [N] int64)."""
        device = device or self.q.device
        n = self.w.store_tokens
        shape = (n, self.w.n_kv, self.w.d)
        k = _draw(self.w, "sk", 0, shape, device)
        v = _draw(self.w, "sv", 0, shape, device)
        g = _gen(self.w, "slots", 0, "cpu")
        first = self.num_blocks - self.w.store_extra_blocks
        slots = torch.randperm(self.w.store_extra_blocks * self.w.block_size, generator=g)[:n]
        slots = (slots + first * self.w.block_size).to(torch.int64).to(device)
        return k, v, slots


def projection(w: Workload, device="cpu") -> torch.Tensor:
    """The QJL projection S [d, d] float32, i.i.d. N(0, 1) (row i = projection i)."""
    g = _gen(w, "proj", 0, "cpu")
    return torch.randn((w.d, w.d), generator=g, dtype=torch.float32).to(device)


def make_inputs(w: Workload, device="cpu") -> Inputs:
    g = _gen(w, "lens", 0, "cpu")
    if w.lens:
        lens = torch.tensor(w.lens, dtype=torch.int32)
    elif w.fixed_len:
        lens = torch.full((w.batch,), w.fixed_len, dtype=torch.int32)
    else:
        lo, hi = w.len_range
        lens = torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int32)
    bs = w.block_size
    nblk = [(int(x) + bs - 1) // bs for x in lens]
    used = sum(nblk)
    num_blocks = used + w.store_extra_blocks
    perm = torch.randperm(used, generator=_gen(w, "perm", 0, "cpu")).to(torch.int32)
    max_blocks = max(nblk) if nblk else 0
    table = torch.full((w.batch, max(max_blocks, 1)), -1, dtype=torch.int32)
    slots = []
    order = []
    at = 0
    start = 0
    for b, nb in enumerate(nblk):
        table[b, :nb] = perm[at: at + nb]
        at += nb
        length = int(lens[b])
        pos = torch.arange(length)
        slots.append(table[b, pos // bs].to(torch.int64) * bs + pos % bs)
        order.append((b, start))
        start += length
    fill = torch.cat(slots) if slots else torch.zeros(0, dtype=torch.int64)
    q = _draw(w, "q", 0, (w.batch, w.n_q, w.d), device)
    return Inputs(w, lens.to(device), table.to(device), num_blocks, q, fill.to(device), order)
