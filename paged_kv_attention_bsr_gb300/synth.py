"""Seeded synthetic BSR workloads shared by the tests, the smoke check and the benchmark.

This module only *constructs inputs*: request lengths, page tables drawn from
a shuffled physical pool, and N(0, 1) values cast to the storage dtype. It
holds none of the attention arithmetic, so both the CUDA path and the CPU
oracle can consume what it makes without sharing any computation.

Workload shapes follow the pages' workloads: Llama-3.1 8B / 70B attention
shapes (FlashInfer digest, "性能提升"), skewed length distributions
("动态工作负载处理"), n = 4 parallel generations over a shared prefix
("用于前缀共享的可组合格式"), and the quick-start snippet's single-request
decode q[32,128], k/v[2048,32,128] (gittoolsai.com page, "基本用法"). The
ShareGPT traces used on the pages are not available here; the uniform and
lognormal length draws below stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

HEAD_DIM = 128
SEED_BASE = 20260000


@dataclass
class BSRCache:
    """One paged pool plus the page table of a batch (all host-side)."""
    page_size: int
    num_kv_heads: int
    head_dim: int
    k_pool: torch.Tensor          # [num_pages, Hk, P, D] (HND) storage dtype, CPU
    v_pool: torch.Tensor
    kv_indptr: np.ndarray         # int32 [B+1]
    kv_indices: np.ndarray        # int32 [nnz]
    last_page_len: np.ndarray     # int32 [B]
    kv_lens: np.ndarray           # int64 [B] (the lengths the table was built from)
    k_scale: Optional[torch.Tensor] = None  # FP8 pools: float32 [Hk] per-head scales
    v_scale: Optional[torch.Tensor] = None

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])


@dataclass
class Workload:
    name: str
    kind: str                     # "decode" | "append" | "composable"
    dtype: torch.dtype
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    sm_scale: float
    q: torch.Tensor               # decode [B, Hq, D]; append [sum qo, Hq, D]
    cache: BSRCache
    qo_indptr: Optional[np.ndarray] = None
    causal: bool = False
    extra: Dict[str, object] = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.cache.kv_indptr) - 1


def normal_values(shape, dtype: torch.dtype, seed: int) -> torch.Tensor:
    """i.i.d. N(0,1) drawn in fp32 and rounded (RNE) to the storage dtype."""
    g = torch.Generator().manual_seed(int(seed))
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    chunk = 1 << 24
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        flat[s:e] = torch.randn(e - s, generator=g, dtype=torch.float32).to(dtype)
    return out


def page_table(kv_lens, page_size: int, pool_pages: int, rng: np.random.Generator,
               shuffle_pool: bool = True):
    """Pages drawn without replacement from a shuffled physical pool."""
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    n_pages = (kv_lens + page_size - 1) // page_size
    total = int(n_pages.sum())
    if total > pool_pages:
        raise ValueError(f"pool of {pool_pages} pages cannot hold {total} pages")
    pool_order = rng.permutation(pool_pages) if shuffle_pool else np.arange(pool_pages)
    kv_indices = pool_order[:total].astype(np.int32)
    kv_indptr = np.zeros(len(kv_lens) + 1, np.int32)
    kv_indptr[1:] = np.cumsum(n_pages)
    last = np.where(n_pages > 0, kv_lens - page_size * (n_pages - 1), 0).astype(np.int32)
    return kv_indptr, kv_indices, last


def make_cache(kv_lens, page_size: int, pool_pages: int, num_kv_heads: int,
               dtype: torch.dtype, seed: int, head_dim: int = HEAD_DIM,
               shuffle_pool: bool = True) -> BSRCache:
    rng = np.random.default_rng(seed)
    kv_indptr, kv_indices, last = page_table(kv_lens, page_size, pool_pages, rng,
                                             shuffle_pool)
    shape = (pool_pages, num_kv_heads, page_size, head_dim)
    k_pool = normal_values(shape, dtype, seed * 4 + 1)
    v_pool = normal_values(shape, dtype, seed * 4 + 2)
    return BSRCache(page_size, num_kv_heads, head_dim, k_pool, v_pool, kv_indptr,
                    kv_indices, last, np.asarray(kv_lens, np.int64))


def make_fp8_cache(kv_lens, page_size: int, pool_pages: int, num_kv_heads: int, seed: int,
                   head_dim: int = HEAD_DIM, shuffle_pool: bool = True) -> BSRCache:
    """A pool stored as FP8 E4M3 bytes with one scale per kv head (for K and
    for V): values drawn N(0, 1) in fp32, scale = the head's largest |value|
    / 448 (the largest E4M3 magnitude), stored = value / scale rounded to E4M3
    by torch's conversion. k_pool / v_pool are uint8 tensors of the bytes;
    the scales (float32 [Hk]) are the cache's ``k_scale`` / ``v_scale``
    attributes."""
    rng = np.random.default_rng(seed)
    kv_indptr, kv_indices, last = page_table(kv_lens, page_size, pool_pages, rng, shuffle_pool)
    shape = (pool_pages, num_kv_heads, page_size, head_dim)
    pools, scales = [], []
    for k in (1, 2):
        x = normal_values(shape, torch.float32, seed * 4 + k)
        amax = x.abs().amax(dim=(0, 2, 3)).clamp_min(1e-30)
        scale = (amax / 448.0).float()
        q8 = (x / scale[None, :, None, None]).to(torch.float8_e4m3fn)
        pools.append(q8.view(torch.uint8))
        scales.append(scale)
    return BSRCache(page_size, num_kv_heads, head_dim, pools[0], pools[1], kv_indptr,
                    kv_indices, last, np.asarray(kv_lens, np.int64), scales[0], scales[1])


def fp8_decode_workload(name, kv_lens, page_size, pool_pages, num_qo_heads, num_kv_heads,
                        dtype, seed, head_dim=HEAD_DIM) -> Workload:
    """Decode over an FP8 E4M3 KV cache (make_fp8_cache); q is 16-bit."""
    cache = make_fp8_cache(kv_lens, page_size, pool_pages, num_kv_heads, seed, head_dim)
    q = normal_values((len(kv_lens), num_qo_heads, head_dim), dtype, seed * 4 + 3)
    return Workload(name, "decode_fp8kv", dtype, num_qo_heads, num_kv_heads, head_dim,
                    1.0 / math.sqrt(head_dim), q, cache)


def decode_workload(name, kv_lens, page_size, pool_pages, num_qo_heads, num_kv_heads,
                    dtype, seed, head_dim=HEAD_DIM, sm_scale=None) -> Workload:
    cache = make_cache(kv_lens, page_size, pool_pages, num_kv_heads, dtype, seed,
                       head_dim)
    q = normal_values((len(kv_lens), num_qo_heads, head_dim), dtype, seed * 4 + 3)
    return Workload(name, "decode", dtype, num_qo_heads, num_kv_heads, head_dim,
                    sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim),
                    q, cache)


def append_workload(name, qo_lens, kv_lens, page_size, pool_pages, num_qo_heads,
                    num_kv_heads, dtype, seed, causal=True, head_dim=HEAD_DIM,
                    sm_scale=None) -> Workload:
    cache = make_cache(kv_lens, page_size, pool_pages, num_kv_heads, dtype, seed,
                       head_dim)
    qo_indptr = np.zeros(len(qo_lens) + 1, np.int32)
    qo_indptr[1:] = np.cumsum(np.asarray(qo_lens, np.int64))
    q = normal_values((int(qo_indptr[-1]), num_qo_heads, head_dim), dtype, seed * 4 + 3)
    return Workload(name, "append", dtype, num_qo_heads, num_kv_heads, head_dim,
                    sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim),
                    q, cache, qo_indptr=qo_indptr, causal=causal)


def rope_tables(max_pos: int, head_dim: int = HEAD_DIM, theta: float = 500000.0,
                llama31: bool = True, factor: float = 8.0, low_freq_factor: float = 1.0,
                high_freq_factor: float = 4.0, original_max_pos: int = 8192):
    """cos / sin tables float32 [max_pos, head_dim / 2] of LLaMA-style rotary
    position embedding, the LLaMA 3.1 variant included (README copy on
    gittoolsai.com, feature list). Pair i turns by pos * f_i with
    f_i = theta^(-2 i / head_dim); with llama31, the LLaMA 3.1 frequency
    rescaling for long contexts: wavelengths 2 pi / f_i shorter than
    original_max_pos / high_freq_factor keep f_i, those longer than
    original_max_pos / low_freq_factor use f_i / factor, and the band between
    blends the two linearly in original_max_pos / wavelength. Angles and
    their cosines / sines are evaluated in float64, then rounded once."""
    half = head_dim // 2
    f = theta ** (-2.0 * np.arange(half, dtype=np.float64) / head_dim)
    if llama31:
        wavelen = 2.0 * math.pi / f
        lo_wl = original_max_pos / low_freq_factor
        hi_wl = original_max_pos / high_freq_factor
        smooth = (original_max_pos / wavelen - low_freq_factor) / (high_freq_factor - low_freq_factor)
        blended = (1.0 - smooth) * f / factor + smooth * f
        f = np.where(wavelen < hi_wl, f, np.where(wavelen > lo_wl, f / factor, blended))
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * f[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# --------------------------------------------------------------------------
# The five benchmark workloads (seed = 20260000 + workload number).
# --------------------------------------------------------------------------

def single_request_decode(seed: int = SEED_BASE + 1) -> Workload:
    """1 request, Hq = Hk = 32, fp16, kv_len 2048 at P = 16: 128 pages placed in
    a random order inside a 256-page pool (the quick-start snippet's shapes)."""
    rng = np.random.default_rng(seed)
    pool = 256
    kv_indices = rng.permutation(pool)[:128].astype(np.int32)
    shape = (pool, 32, 16, HEAD_DIM)
    cache = BSRCache(16, 32, HEAD_DIM, normal_values(shape, torch.float16, seed * 4 + 1),
                     normal_values(shape, torch.float16, seed * 4 + 2),
                     np.array([0, 128], np.int32), kv_indices,
                     np.array([16], np.int32), np.array([2048], np.int64))
    q = normal_values((1, 32, HEAD_DIM), torch.float16, seed * 4 + 3)
    return Workload("single_decode_h32_kv2048_fp16", "decode", torch.float16, 32, 32,
                    HEAD_DIM, 1.0 / math.sqrt(HEAD_DIM), q, cache)


def uniform_gqa_decode(seed: int = SEED_BASE + 2, batch: int = 64,
                       pool_pages: int = 20000) -> Workload:
    """Llama-3.1-8B shape: B = 64, Hq = 32, Hk = 8, bf16, P = 16, kv_len ~ U[1024, 4096]."""
    rng = np.random.default_rng(seed)
    kv_lens = rng.integers(1024, 4096, size=batch, endpoint=True)
    w = decode_workload("uniform_gqa_decode_b64_h32kv8_p16_bf16", kv_lens, 16,
                        pool_pages, 32, 8, torch.bfloat16, seed)
    return w


def fp8_uniform_gqa_decode(seed: int = SEED_BASE + 8, batch: int = 64,
                           pool_pages: int = 20000) -> Workload:
    """The uniform GQA decode shape (B = 64, Hq = 32, Hk = 8, kv_len
    U[1024, 4096], P = 16, shuffled 20000-page pool) over an FP8 E4M3 KV
    cache with per-head scales; q and the output are bf16."""
    rng = np.random.default_rng(seed)
    kv_lens = rng.integers(1024, 4096, size=batch, endpoint=True)
    return fp8_decode_workload("fp8kv_uniform_gqa_decode_b64_h32kv8_p16", kv_lens, 16,
                               pool_pages, 32, 8, torch.bfloat16, seed)


def vector_sparse_decode(seed: int = SEED_BASE + 6, batch: int = 64,
                         pool_pages: int = 200000) -> Workload:
    """The uniform GQA decode batch (B = 64, Hq = 32, Hk = 8, bf16,
    kv_len ~ U[1024, 4096]) stored at page_size 1: every token is its own
    page, drawn without replacement from a shuffled pool of 200000 one-token
    pages (vector-level sparsity, the BSR format at block size 1)."""
    rng = np.random.default_rng(seed)
    kv_lens = rng.integers(1024, 4096, size=batch, endpoint=True)
    return decode_workload("vector_sparse_decode_b64_h32kv8_p1_bf16", kv_lens, 1, pool_pages,
                           32, 8, torch.bfloat16, seed)


def skewed_lengths(rng: np.random.Generator, n_long=4, n_short=124):
    short = np.floor(np.exp(rng.normal(math.log(512.0), 0.75, size=n_short)))
    short = np.clip(short, 16, 4096).astype(np.int64)
    lens = np.concatenate([np.full(n_long, 32768, np.int64), short])
    return lens[rng.permutation(len(lens))]


def skewed_gqa_decode(seed: int = SEED_BASE + 3, pool_pages: int = 20000) -> Workload:
    """Llama-3.1-70B per-layer shape: B = 128, Hq = 64, Hk = 8, bf16, P = 16;
    4 requests of 32768 tokens, 124 lognormal(ln 512, 0.75) clipped to [16, 4096]."""
    rng = np.random.default_rng(seed)
    kv_lens = skewed_lengths(rng)
    return decode_workload("skewed_gqa_decode_b128_h64kv8_p16_bf16", kv_lens, 16,
                           pool_pages, 64, 8, torch.bfloat16, seed)


def shared_prefix_decode(seed: int = SEED_BASE + 4, prompts: int = 16, n: int = 4,
                         prefix_len: int = 8192, prefix_page: int = 128,
                         suffix_page: int = 16) -> Workload:
    """Composable formats: each prompt's prefix is stored once at P = 128 and
    read by its n generations; each generation's own suffix (U[256, 1024]
    tokens) lives in a second pool at P = 16. Hq = 32, Hk = 8, bf16.

    The returned workload's ``cache`` is the suffix pool (decode); the prefix
    pool and its per-prompt table are in ``extra``; ``q`` holds one row per
    generation, which is also the prefix pass's query (qo_len = n per prompt).
    """
    rng = np.random.default_rng(seed)
    Hq, Hk = 32, 8
    suffix_lens = rng.integers(256, 1024, size=prompts * n, endpoint=True)
    suffix_pool = int(((suffix_lens + suffix_page - 1) // suffix_page).sum()) + 256
    suffix = make_cache(suffix_lens, suffix_page, suffix_pool, Hk, torch.bfloat16, seed)
    prefix_pages_each = prefix_len // prefix_page
    prefix_pool = prompts * prefix_pages_each + 64
    prefix = make_cache(np.full(prompts, prefix_len), prefix_page, prefix_pool, Hk,
                        torch.bfloat16, seed + 1000)
    q = normal_values((prompts * n, Hq, HEAD_DIM), torch.bfloat16, seed * 4 + 3)
    qo_indptr = (np.arange(prompts + 1) * n).astype(np.int32)
    return Workload("shared_prefix_decode_16x4_prefix8192p128_suffixp16_bf16",
                    "composable", torch.bfloat16, Hq, Hk, HEAD_DIM,
                    1.0 / math.sqrt(HEAD_DIM), q, suffix,
                    extra={"prefix": prefix, "prefix_qo_indptr": qo_indptr, "n": n,
                           "prompts": prompts})


def causal_append(seed: int = SEED_BASE + 5, batch: int = 16,
                  pool_pages: int = 10000) -> Workload:
    """B = 16 new-token chunks U[128, 1024] on top of U[0, 8192] existing tokens,
    end-aligned causal mask, Hq = 32, Hk = 8, bf16, P = 16."""
    rng = np.random.default_rng(seed)
    qo_lens = rng.integers(128, 1024, size=batch, endpoint=True)
    existing = rng.integers(0, 8192, size=batch, endpoint=True)
    kv_lens = existing + qo_lens
    return append_workload("causal_append_b16_h32kv8_p16_bf16", qo_lens, kv_lens, 16,
                           pool_pages, 32, 8, torch.bfloat16, seed, causal=True)


def pod_mixed_batch(seed: int = SEED_BASE + 7, n_prefill: int = 16, n_decode: int = 64,
                    pool_pages: int = 30000) -> Workload:
    """One serving batch with both kinds of request (POD-style prefill +
    decode): the causal-append shape (16 chunks of U[128, 1024] new tokens on
    U[0, 8192] existing ones) and the uniform GQA decode shape (64 requests,
    kv_len U[1024, 4096], one new token), Hq = 32, Hk = 8, bf16, P = 16, in
    one shuffled pool and one request order (shuffled). ``extra`` lists which
    requests are prefill and which decode, so that the same batch can also
    be run as two separate launches."""
    rng = np.random.default_rng(seed)
    qo_p = rng.integers(128, 1024, size=n_prefill, endpoint=True)
    kv_p = rng.integers(0, 8192, size=n_prefill, endpoint=True) + qo_p
    kv_d = rng.integers(1024, 4096, size=n_decode, endpoint=True)
    qo_lens = np.concatenate([qo_p, np.ones(n_decode, np.int64)])
    kv_lens = np.concatenate([kv_p, kv_d])
    perm = rng.permutation(len(qo_lens))
    w = append_workload("pod_mixed_prefill16_decode64_h32kv8_p16_bf16", qo_lens[perm],
                        kv_lens[perm], 16, pool_pages, 32, 8, torch.bfloat16, seed, causal=True)
    w.extra["prefill"] = np.nonzero(qo_lens[perm] > 1)[0]
    w.extra["decode"] = np.nonzero(qo_lens[perm] == 1)[0]
    return w


def sub_batch(w: Workload, rows, as_decode: bool = False) -> Workload:
    """The requests `rows` of an append workload as a batch of their own, on
    the same pool (page table and queries gathered; values shared). With
    as_decode, every request must have one query row and the result is a
    decode workload."""
    c = w.cache
    rows = np.asarray(rows, np.int64)
    n = np.diff(c.kv_indptr)[rows]
    indptr = np.zeros(len(rows) + 1, np.int32)
    indptr[1:] = np.cumsum(n)
    indices = np.concatenate([c.kv_indices[c.kv_indptr[r]:c.kv_indptr[r + 1]] for r in rows]
                             ) if len(rows) else np.zeros(0, np.int32)
    cache = BSRCache(c.page_size, c.num_kv_heads, c.head_dim, c.k_pool, c.v_pool, indptr,
                     indices.astype(np.int32), c.last_page_len[rows].copy(),
                     c.kv_lens[rows].copy())
    qo = np.diff(w.qo_indptr)[rows]
    q_rows = np.concatenate([np.arange(w.qo_indptr[r], w.qo_indptr[r + 1]) for r in rows])
    q = w.q[torch.from_numpy(q_rows)]
    if as_decode:
        if np.any(qo != 1):
            raise ValueError("a decode sub-batch needs one query row per request")
        return Workload(w.name + "_decode", "decode", w.dtype, w.num_qo_heads, w.num_kv_heads,
                        w.head_dim, w.sm_scale, q, cache)
    qo_indptr = np.zeros(len(rows) + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo)
    return Workload(w.name + "_sub", "append", w.dtype, w.num_qo_heads, w.num_kv_heads,
                    w.head_dim, w.sm_scale, q, cache, qo_indptr=qo_indptr, causal=w.causal)


def cascade_workload(name: str, gens, prefix_lens, suffix_lens, prefix_page: int,
                     suffix_page: int, num_qo_heads: int, num_kv_heads: int,
                     dtype: torch.dtype, seed: int, slack_pages: int = 7) -> Workload:
    """A composable-format batch with ragged shapes: prompt p has gens[p]
    generations (0 allowed), a prefix of prefix_lens[p] tokens (pool at
    prefix_page) and generation b a suffix of suffix_lens[b] tokens (pool at
    suffix_page); both pools shuffled, with slack_pages unused pages each.
    Same field layout as shared_prefix_decode."""
    gens = np.asarray(gens, np.int64)
    prompts, B = len(gens), int(gens.sum())
    prefix_lens = np.asarray(prefix_lens, np.int64)
    suffix_lens = np.asarray(suffix_lens, np.int64)
    pages0 = int(((prefix_lens + prefix_page - 1) // prefix_page).sum()) + slack_pages
    pages1 = int(((suffix_lens + suffix_page - 1) // suffix_page).sum()) + slack_pages
    prefix = make_cache(prefix_lens, prefix_page, pages0, num_kv_heads, dtype, seed + 1000)
    suffix = make_cache(suffix_lens, suffix_page, pages1, num_kv_heads, dtype, seed)
    q = normal_values((B, num_qo_heads, HEAD_DIM), dtype, seed * 4 + 3)
    qo_indptr = np.concatenate([[0], np.cumsum(gens)]).astype(np.int32)
    return Workload(name, "composable", dtype, num_qo_heads, num_kv_heads, HEAD_DIM,
                    1.0 / math.sqrt(HEAD_DIM), q, suffix,
                    extra={"prefix": prefix, "prefix_qo_indptr": qo_indptr, "n": None,
                           "prompts": prompts})


def flat_layout_of_composable(w: Workload, page_size: int = 16) -> BSRCache:
    """The same logical KV as a shared-prefix workload, in one pool with one page
    size: each generation's table lists its prompt's prefix pages (shared by
    its generations) followed by its own suffix pages. A prefix followed by a
    non-empty suffix must fill whole small pages (its length a multiple of
    page_size)."""
    prefix: BSRCache = w.extra["prefix"]
    suffix = w.cache
    qo_indptr = w.extra["prefix_qo_indptr"]
    prompts = w.extra["prompts"]
    Hk, D = suffix.num_kv_heads, suffix.head_dim
    if suffix.page_size != page_size or prefix.page_size % page_size:
        raise ValueError("flat layout needs the suffix page size to divide the prefix's")
    ratio = prefix.page_size // page_size
    # Re-page the prefix pool: each big page becomes `ratio` consecutive small pages.
    pk = prefix.k_pool.view(prefix.num_pages, Hk, ratio, page_size, D).permute(0, 2, 1, 3, 4)
    pv = prefix.v_pool.view(prefix.num_pages, Hk, ratio, page_size, D).permute(0, 2, 1, 3, 4)
    pk = pk.reshape(prefix.num_pages * ratio, Hk, page_size, D)
    pv = pv.reshape(prefix.num_pages * ratio, Hk, page_size, D)
    base = prefix.num_pages * ratio
    k_pool = torch.cat([pk, suffix.k_pool], 0).contiguous()
    v_pool = torch.cat([pv, suffix.v_pool], 0).contiguous()
    indptr = [0]
    indices: List[int] = []
    last = []
    lens = []
    for p in range(prompts):
        big = prefix.kv_indices[prefix.kv_indptr[p]:prefix.kv_indptr[p + 1]]
        len0 = int(prefix.kv_lens[p])
        small = (big[:, None].astype(np.int64) * ratio + np.arange(ratio)[None, :]).reshape(-1)
        small = small[:(len0 + page_size - 1) // page_size]
        for r in range(int(qo_indptr[p]), int(qo_indptr[p + 1])):
            own = suffix.kv_indices[suffix.kv_indptr[r]:suffix.kv_indptr[r + 1]] + base
            if len(own) and len0 % page_size:
                raise ValueError("a prefix followed by a suffix must fill whole small pages")
            indices.extend(small.tolist())
            indices.extend(own.tolist())
            indptr.append(len(indices))
            if len(own):
                last.append(int(suffix.last_page_len[r]))
            elif len(small):
                last.append(len0 - page_size * (len(small) - 1))
            else:
                last.append(0)
            lens.append(len0 + int(suffix.kv_lens[r]))
    return BSRCache(page_size, Hk, D, k_pool, v_pool, np.array(indptr, np.int32),
                    np.array(indices, np.int32), np.array(last, np.int32),
                    np.array(lens, np.int64))


WORKLOADS = {
    "single_decode": single_request_decode,
    "uniform_decode": uniform_gqa_decode,
    "skewed_decode": skewed_gqa_decode,
    "shared_prefix": shared_prefix_decode,
    "causal_append": causal_append,
    "sparse_decode": vector_sparse_decode,
    "pod_mixed": pod_mixed_batch,
    "fp8_decode": fp8_uniform_gqa_decode,
}
