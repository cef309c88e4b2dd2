"""Seeded synthetic inputs for deterministic context attention.

This module draws the random inputs that both the CUDA path and the CPU
oracle consume.  It holds none of the attention arithmetic: it makes
BF16-exact normal tensors, varlen batch offsets, rotary position embedding
applied to q/k *before* attention (the post-RoPE contract of "WS2 Attention
PR5 Drift Benchmark", Scope: CP attention consumes post-RoPE Q/K), and paged
KV pools with a randomly permuted page layout.

Every array is numpy; float tensors hold exact BF16 values in float32 so the
oracle can widen them exactly, and ``bf16_bits`` gives the raw 16-bit words a
device buffer holds.  Each tensor has its own stream: seed and a tensor id
feed numpy's PCG64 through a SeedSequence.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# tensor ids for independent streams
T_Q, T_K, T_V, T_DOUT, T_LENS, T_PAGES = 1, 2, 3, 4, 5, 6


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(tensor_id)])))


def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest BF16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(x) -> np.ndarray:
    """uint16 words of BF16-exact float32 values (no rounding: exact input)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("values are not BF16-exact")
    return (u >> 16).astype(np.uint16)


def bits_to_f32(bits) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, tensor_id: int, shape) -> np.ndarray:
    """N(0,1) draws rounded to BF16, as float32."""
    return bf16_round(rng(seed, tensor_id).standard_normal(size=shape, dtype=np.float32))


def cu_seqlens(lens) -> np.ndarray:
    out = np.zeros(len(lens) + 1, np.int32)
    out[1:] = np.cumsum(np.asarray(lens, np.int64))
    return out


def rope_rotate_half(x, cu, theta=1.0e6):
    """Rotary embedding, rotate-half (NeoX) pairing of dims (i, i + D/2),
    inverse frequency theta^(-2i/D), position = token index within its
    sequence; evaluated in float64, rounded once to BF16."""
    x = np.asarray(x, np.float32)
    t, h, d = x.shape
    half = d // 2
    pos = np.empty(t, np.float64)
    for s in range(len(cu) - 1):
        pos[cu[s]:cu[s + 1]] = np.arange(cu[s + 1] - cu[s], dtype=np.float64)
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = pos[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s_ = np.sin(ang)[:, None, :]
    x1 = x[..., :half].astype(np.float64)
    x2 = x[..., half:].astype(np.float64)
    y = np.concatenate([x1 * c - x2 * s_, x2 * c + x1 * s_], axis=-1)
    return bf16_round(y.astype(np.float32))


@dataclass
class Prefill:
    """Packed varlen ("THD") prefill problem."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    cu_q: np.ndarray
    cu_k: np.ndarray
    hq: int
    hkv: int
    d: int
    scale: float
    block: int
    meta: dict = field(default_factory=dict)


def prefill_problem(lens, hq=32, hkv=8, d=128, block=128, seed=0, rope=False,
                    theta=1.0e6, kv_lens=None) -> Prefill:
    """q/k/v ~ N(0,1) in BF16 for sequences of ``lens`` query tokens.  With
    ``kv_lens`` the KV side is longer (chunked replay: the queries are the
    last q_len tokens of each sequence's cache)."""
    kv_lens = list(lens) if kv_lens is None else list(kv_lens)
    cu_q = cu_seqlens(lens)
    cu_k = cu_seqlens(kv_lens)
    q = normal_bf16(seed, T_Q, (int(cu_q[-1]), hq, d))
    k = normal_bf16(seed, T_K, (int(cu_k[-1]), hkv, d))
    v = normal_bf16(seed, T_V, (int(cu_k[-1]), hkv, d))
    if rope:
        q = rope_rotate_half(q, cu_q, theta)
        k = rope_rotate_half(k, cu_k, theta)
    return Prefill(q, k, v, cu_q, cu_k, hq, hkv, d, 1.0 / np.sqrt(d), block,
                   {"lens": list(lens), "kv_lens": kv_lens, "seed": seed, "rope": rope})


def permute_batch(p: Prefill, order) -> Prefill:
    """Same sequences, packed in another order."""
    lq = np.diff(p.cu_q)
    lk = np.diff(p.cu_k)
    qs = [p.q[p.cu_q[s]:p.cu_q[s + 1]] for s in range(len(lq))]
    ks = [p.k[p.cu_k[s]:p.cu_k[s + 1]] for s in range(len(lk))]
    vs = [p.v[p.cu_k[s]:p.cu_k[s + 1]] for s in range(len(lk))]
    order = list(order)
    return Prefill(np.concatenate([qs[s] for s in order]), np.concatenate([ks[s] for s in order]),
                   np.concatenate([vs[s] for s in order]), cu_seqlens([lq[s] for s in order]),
                   cu_seqlens([lk[s] for s in order]), p.hq, p.hkv, p.d, p.scale, p.block,
                   dict(p.meta, order=order))


@dataclass
class PagedDecode:
    q: np.ndarray            # [n, hq, d] float32 (BF16-exact)
    k_bits: np.ndarray       # [n_pages, page_size, hkv, d] uint16 BF16 words
    v_bits: np.ndarray
    page_table: np.ndarray   # [n, max_pages] int32 (-1 past a sequence's last page)
    seqlens: np.ndarray      # [n] int32
    page_size: int
    hq: int
    hkv: int
    d: int
    scale: float
    seed: int

    def seq_kv(self, s):
        """Contiguous K, V of sequence s ([ctx, hkv, d] float32), regenerated
        from the seed (the pool holds the same values)."""
        return decode_seq_kv(self.seed, s, int(self.seqlens[s]), self.hkv, self.d)

    @property
    def k_pool(self):
        return bits_to_f32(self.k_bits)

    @property
    def v_pool(self):
        return bits_to_f32(self.v_bits)


def decode_seq_kv(seed, s, ctx, hkv, d):
    k = normal_bf16(seed * 1000 + s + 1, T_K, (ctx, hkv, d))
    v = normal_bf16(seed * 1000 + s + 1, T_V, (ctx, hkv, d))
    return k, v


def paged_decode_problem(n=64, ctx_lo=512, ctx_hi=32768, hq=32, hkv=8, d=128, page_size=16,
                         seed=3, ctx=None, spare_pages=0, garbage_tail=True) -> PagedDecode:
    """Context lengths ~ U[ctx_lo, ctx_hi] (integers, from the seed) unless
    ``ctx`` is given; every sequence's KV lives in pages of ``page_size``
    tokens scattered over the pool by a seeded random permutation.  Unused
    tail slots of a sequence's last page (and spare pages) hold NaN when
    ``garbage_tail``, so a kernel that let them into its arithmetic would show
    it."""
    if ctx is None:
        ctx = rng(seed, T_LENS).integers(ctx_lo, ctx_hi + 1, size=n)
    ctx = np.asarray(ctx, np.int64)
    n = len(ctx)
    pages_per = (ctx + page_size - 1) // page_size
    n_pages = int(pages_per.sum()) + int(spare_pages)
    max_pages = int(pages_per.max())
    perm = rng(seed, T_PAGES).permutation(n_pages).astype(np.int32)
    q = normal_bf16(seed, T_Q, (n, hq, d))
    fill = 0x7FC0 if garbage_tail else 0
    k_bits = np.full((n_pages, page_size, hkv, d), fill, np.uint16)
    v_bits = np.full((n_pages, page_size, hkv, d), fill, np.uint16)
    page_table = np.full((n, max_pages), -1, np.int32)
    nxt = 0
    for s in range(n):
        c, npg = int(ctx[s]), int(pages_per[s])
        ks, vs = decode_seq_kv(seed, s, c, hkv, d)
        pad_k = np.full((npg * page_size, hkv, d), fill, np.uint16)
        pad_v = np.full((npg * page_size, hkv, d), fill, np.uint16)
        pad_k[:c] = bf16_bits(ks)
        pad_v[:c] = bf16_bits(vs)
        phys = perm[nxt:nxt + npg]
        nxt += npg
        page_table[s, :npg] = phys
        k_bits[phys] = pad_k.reshape(npg, page_size, hkv, d)
        v_bits[phys] = pad_v.reshape(npg, page_size, hkv, d)
    return PagedDecode(q, k_bits, v_bits, page_table, ctx.astype(np.int32), page_size, hq, hkv,
                       d, 1.0 / np.sqrt(d), seed)


# The five synthetic workloads (sizes, shapes and value distributions of the
# Qwen3-8B attention target).
CFG_TINY = dict(lens=[256], hq=32, hkv=8, d=128, block=64, seed=0)
CFG_PREFILL = dict(lens=[4096, 3000, 1024, 777], hq=32, hkv=8, d=128, block=128, seed=1,
                   rope=True)
CFG_CHUNKED = dict(lens=[8192, 8192], hq=16, hkv=4, d=128, block=128, seed=2)
CFG_DECODE = dict(n=64, ctx_lo=512, ctx_hi=32768, hq=32, hkv=8, d=128, page_size=16, seed=3)
CFG_BACKWARD = dict(lens=[4096, 4096], hq=32, hkv=8, d=128, block=128, seed=4)


def lm_head(width: int, rows: int, vocab: int = 512, seed: int = 7):
    """The seeded synthetic lm_head of the dlogp drift class: FP32 weights
    W [width, vocab] ~ N(0, 1/width) and one selected token per row (uniform
    over the vocabulary).  Only the draw lives here; the projection and the
    log-softmax are computed by whoever checks the outputs."""
    g = np.random.default_rng([seed, width, vocab])
    w = (g.standard_normal((width, vocab)) / np.sqrt(width)).astype(np.float32)
    tok = g.integers(0, vocab, size=rows)
    return w, tok


def prefill_flops(cu_q, cu_k, hq, d) -> float:
    """Algorithmic causal flops: 4 * D * Hq * (visible (row, key) pairs)."""
    pairs = 0
    for s in range(len(cu_q) - 1):
        ql = int(cu_q[s + 1] - cu_q[s])
        kl = int(cu_k[s + 1] - cu_k[s])
        # row i sees kl - ql + i + 1 keys
        pairs += ql * (kl - ql) + ql * (ql + 1) // 2
    return 4.0 * d * hq * pairs
