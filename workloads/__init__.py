"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module only draws random numbers and builds input structure (shapes, valid lengths,
the tile-sparsity pattern).  It holds none of the attention arithmetic, so the CPU oracle
and the CUDA path can both take their inputs from here without sharing any of the method.

The workloads stand in for the ones the FlashAttention pages measure on (BERT-large at
sequence 512, GPT-2 small at 1024, long-range 16K, block-sparse Path-256 at 64K; "FlashAttention
paper story", results table; "FlashAttention: Exact Attention with Less GPU Memory", "What it
measured").  No dataset is used: values are i.i.d.
normal, drawn in float32 from a CPU ``torch.Generator`` and rounded to the working dtype.
Draw order inside one workload: Q, K, V, dO, then the valid key lengths.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

TILE = 128  # granularity of the block-sparsity mask (rows and columns of score tiles)


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "bf16", "fp16" or "fp32"
    causal: bool = False
    value_scale: float = 1.0          # Q/K/V are N(0,1) times this
    pad_lengths: Optional[tuple] = None  # (lo, hi): per-sequence valid key length ~ U{lo..hi}
    block_sparse: bool = False        # local band of 4 tiles + 2 global tiles (rows and cols)
    backward: bool = True
    Nk: Optional[int] = None          # key length when it differs from N (decode shapes)
    Hkv: Optional[int] = None         # key/value heads when fewer than H (grouped-query attention)
    seq_lens: Optional[tuple] = None  # packed sequences: their lengths (B = 1, N = their sum)

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5


def packed_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    """n sequence lengths ~ U{lo..hi} from a seeded CPU generator (input structure only)."""
    g = torch.Generator().manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g))


_VARLEN = packed_lengths(24, 256, 4096, seed=7)

WORKLOADS = {
    # fp32 correctness case: B1 H1 N128 d64, non-causal, forward only
    "fp32_n128_d64": Workload("fp32_n128_d64", 1, 1, 128, 64, "fp32", backward=False),
    # BERT-large-shaped encoder attention with key padding, lengths U{256..512}
    "bert_large_pad_n512": Workload("bert_large_pad_n512", 8, 16, 512, 64, "bf16",
                                    pad_lengths=(256, 512)),
    # GPT-2-small-shaped decoder attention, causal, inputs scaled by 1.5 (wide logits)
    "gpt2_small_causal_n1024": Workload("gpt2_small_causal_n1024", 8, 12, 1024, 64, "bf16",
                                        causal=True, value_scale=1.5),
    # long-context attention B1 H16 N16384 d128, both mask settings
    "long_n16k_d128": Workload("long_n16k_d128", 1, 16, 16384, 128, "bf16"),
    "long_n16k_d128_causal": Workload("long_n16k_d128_causal", 1, 16, 16384, 128, "bf16",
                                      causal=True),
    # a smaller long-context case for profiler captures (inputs still larger than L2)
    "long_n8k_d128": Workload("long_n8k_d128", 1, 16, 8192, 128, "bf16"),
    # decode-shaped: 16 new queries per sequence against a 32K-key cache (forward only)
    "decode_q16_k32k_d128": Workload("decode_q16_k32k_d128", 8, 16, 16, 128, "bf16",
                                     backward=False, Nk=32768),
    # grouped-query attention: 32 query heads on 8 key/value heads, B2 N8192 d128, causal
    "gqa_causal_n8k_h32_kv8_d128": Workload("gqa_causal_n8k_h32_kv8_d128", 2, 32, 8192, 128,
                                            "bf16", causal=True, Hkv=8),
    # packed sequences: 24 sequences of U{256..4096} tokens back to back, H16 d128, causal
    "varlen_causal_h16_d128": Workload("varlen_causal_h16_d128", 1, 16, sum(_VARLEN), 128, "bf16",
                                       causal=True, seq_lens=_VARLEN),
    # grouped-query decode: 32 query heads on 8 key/value heads, 16 new queries per sequence
    # against a 32K-key cache (forward only)
    "decode_gqa_q16_k32k_h32_kv8_d128": Workload("decode_gqa_q16_k32k_h32_kv8_d128", 8, 32, 16, 128,
                                                 "bf16", backward=False, Nk=32768, Hkv=8),
    # block-sparse attention B1 H8 N65536 d64, local band + global tiles
    "block_sparse_n64k_d64": Workload("block_sparse_n64k_d64", 1, 8, 65536, 64, "bf16",
                                      block_sparse=True),
}


def local_global_tile_mask(n_tiles: int, band: int = 4, n_global: int = 2) -> torch.Tensor:
    """uint8 [n_tiles, n_tiles]: tile (I, J) kept iff |I-J| <= band or I < n_global or J < n_global.

    This is the sparsity *pattern* of the block-sparse workload ("FlashAttention paper story", block-sparse
    paragraph: local windows plus global tokens); it is input structure, not arithmetic.
    """
    idx = torch.arange(n_tiles)
    keep = ((idx[:, None] - idx[None, :]).abs() <= band) | (idx[:, None] < n_global) | (idx[None, :] < n_global)
    return keep.to(torch.uint8)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[name]


def make_inputs(w: Workload, seed: int = 0, heads: Optional[int] = None, N: Optional[int] = None,
                B: Optional[int] = None, kv_heads: Optional[int] = None) -> dict:
    """Draw one workload's inputs on the CPU.

    Returns a dict with q, k, v, do ([B,H,N,d] in the workload dtype), kv_lens (int32 [B] or
    None), block_mask (uint8 [T,T] or None), plus the scalar settings.  ``heads``/``N``/``B``
    override the sizes for reduced test cases (same recipe, smaller tensors).  ``kv_heads``
    gives k and v fewer heads than q (grouped-query attention); the default is the workload's
    own key/value head count, or one key/value head per query head when ``heads`` overrides H.
    """
    B = w.B if B is None else B
    H = w.H if heads is None else heads
    N = w.N if N is None else N
    Nk = N if w.Nk is None else w.Nk
    g = torch.Generator().manual_seed(seed)
    dt = torch_dtype(w.dtype)
    shape = (B, H, N, w.d)
    if kv_heads is None:
        kv_heads = w.Hkv if (w.Hkv is not None and heads is None) else H
    kshape = (B, kv_heads, Nk, w.d)
    q = (torch.randn(shape, generator=g) * w.value_scale).to(dt)
    k = (torch.randn(kshape, generator=g) * w.value_scale).to(dt)
    v = (torch.randn(kshape, generator=g) * w.value_scale).to(dt)
    do = torch.randn(shape, generator=g).to(dt)
    kv_lens = None
    if w.pad_lengths is not None:
        lo, hi = w.pad_lengths
        lo = min(lo, Nk)
        hi = min(hi, Nk)
        kv_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    block_mask = None
    if w.block_sparse:
        block_mask = local_global_tile_mask((N + TILE - 1) // TILE)
    return dict(q=q, k=k, v=v, do=do, kv_lens=kv_lens, block_mask=block_mask,
                causal=w.causal, scale=w.scale, dtype=w.dtype)


def random_tile_mask(n_tiles: int, density: float, seed: int) -> torch.Tensor:
    """uint8 [n_tiles, n_tiles] Bernoulli(density) tile mask, for edge-case tests."""
    g = torch.Generator().manual_seed(seed)
    return (torch.rand((n_tiles, n_tiles), generator=g) < density).to(torch.uint8)


def as_f64(t: torch.Tensor):
    """The exact values of a (possibly bf16) tensor as a float64 numpy array."""
    return t.to(torch.float64).numpy()


def make_packed_inputs(w: Workload, seed: int = 0) -> dict:
    """Inputs of a packed-sequence workload: q, k, v, dO as [heads, total, d] (same recipe and
    draw order as ``make_inputs``), the int32 offsets [n_seqs + 1] and the longest length."""
    x = make_inputs(w, seed=seed)
    offs = [0]
    for n in w.seq_lens:
        offs.append(offs[-1] + n)
    out = {n: x[n][0] for n in ("q", "k", "v", "do")}
    out.update(cu_seqlens=torch.tensor(offs, dtype=torch.int32), max_seqlen=max(w.seq_lens),
               causal=w.causal, scale=w.scale, dtype=w.dtype)
    return out
