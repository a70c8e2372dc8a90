"""Seeded synthetic decode batches.

This module only draws inputs - context lengths, page tables and values - and
holds none of the attention arithmetic, so both the CUDA path and the
float64 oracle can be fed from it.

The five named configurations are the decode workloads this library is
measured on:

``tiny``         B=4, 8 qo / 8 kv heads, head_dim 64, fp32, lengths
                 {17, 64, 100, 255}; the 29 pages are drawn without replacement
                 from a 64-page pool in seeded random order.
``gqa_uniform``  B=64, 32 qo / 8 kv heads (group 4), head_dim 128, bf16,
                 every length 2048; page ids a seeded permutation of the pool.
``ragged``       B=450, 32/8 heads, head_dim 128, bf16, lengths log-uniform in
                 [256, 64000] - the heterogeneous mix (256 to 64,000 tokens)
                 of the incident on the page "FlashInfer vs FlashAttention-3".
``long_split``   B=1, 32/32 heads (MHA), head_dim 128, bf16, length 65536: one
                 sequence that has to be split across the whole GPU.
``fp8_kv``       B=128, 64/8 heads (group 8), head_dim 128, bf16 q, K and V
                 stored as FP8 E4M3 with one fp32 scale each (amax / 448),
                 lengths uniform in [1024, 8192].

``fp8_kv_token_scales``  the fp8_kv shapes and lengths, with K and V
                 magnitudes that vary per token and kv head (N(0,1) times
                 2^u, u uniform in [-3, 3]) stored as E4M3 with one fp32
                 scale per (page, kv head, slot) = amax over head_dim / 448
                 - the spread that underflows under a single static scale.

``spec_decode``  the gqa_uniform batch with two query tokens per request
                 (speculative verification of one draft token): q is
                 [B, 2, Hq, D] and each request's last two cache positions are
                 the two query tokens' own K/V.

``cascade``      B=64, 32/8 heads, head_dim 128, bf16: every request starts
                 with the same 32768-token prefix (2048 shared pages, 134 MB
                 of KV - more than the 129 MB L2, e.g. a shared retrieved
                 document) followed by U{1..512} tokens of its own.  The
                 batch's page table lists each request's full sequence (prefix
                 pages first); extra["prefix_pages"] says how many are shared.

``spec_decode_ragged``  the fp8_kv shapes (B=128, 64/8 heads, group 8,
                 E4M3 KV, lengths U{1024..8192}) verifying U{1..4} draft
                 tokens per request (speculative decoding with a draft length
                 of its own per request): q is ragged [sum of drafts, 64, 128]
                 with extra["qo_indptr"]; up to 32 columns per (request, kv
                 head).

``gqa_unified_max``  the gqa_uniform batch (same seed, same values), decoded
                 with the unified-max softmax against cauchy_schwarz_bound.

``cauchy_schwarz_bound`` turns a batch's values into the static logit bound
that the unified-max softmax takes as an input (norms only, no scores).

All use page_size 16 and the combined [num_pages, 2, 16, Hkv, D] layout.
Lengths and page tables come from a CPU ``torch.Generator``; values from a
generator on the target device, both seeded with the config's seed
(1000 + its position).  last_page_len = len - 16 * (pages - 1), i.e.
len mod 16, or 16 when that is 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE_SIZE = 16
E4M3_MAX = 448.0


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    q_dtype: torch.dtype
    kv_dtype: torch.dtype
    seed: int
    page_size: int = PAGE_SIZE
    q_len: int = 1

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads


CONFIGS: dict[str, DecodeConfig] = {
    "tiny": DecodeConfig("tiny", 4, 8, 8, 64, torch.float32, torch.float32, 1001),
    "gqa_uniform": DecodeConfig("gqa_uniform", 64, 32, 8, 128, torch.bfloat16, torch.bfloat16, 1002),
    "ragged": DecodeConfig("ragged", 450, 32, 8, 128, torch.bfloat16, torch.bfloat16, 1003),
    "long_split": DecodeConfig("long_split", 1, 32, 32, 128, torch.bfloat16, torch.bfloat16, 1004),
    "fp8_kv": DecodeConfig("fp8_kv", 128, 64, 8, 128, torch.bfloat16, torch.float8_e4m3fn, 1005),
    "fp8_kv_token_scales": DecodeConfig("fp8_kv_token_scales", 128, 64, 8, 128, torch.bfloat16,
                                        torch.float8_e4m3fn, 1006),
    "spec_decode": DecodeConfig("spec_decode", 64, 32, 8, 128, torch.bfloat16, torch.bfloat16,
                                1007, q_len=2),
    "cascade": DecodeConfig("cascade", 64, 32, 8, 128, torch.bfloat16, torch.bfloat16, 1008),
    "spec_decode_ragged": DecodeConfig("spec_decode_ragged", 128, 64, 8, 128, torch.bfloat16,
                                       torch.float8_e4m3fn, 1009, q_len=4),
    # the gqa_uniform batch itself (same seed), run with the unified-max softmax
    "gqa_unified_max": DecodeConfig("gqa_unified_max", 64, 32, 8, 128, torch.bfloat16,
                                    torch.bfloat16, 1002),
}
CASCADE_PREFIX_PAGES = 2048


def draw_lengths(cfg: DecodeConfig, gen: torch.Generator) -> np.ndarray:
    """Context length of every request of a named configuration."""
    if cfg.name == "tiny":
        return np.array([17, 64, 100, 255], dtype=np.int64)
    if cfg.name in ("gqa_uniform", "spec_decode", "gqa_unified_max"):
        return np.full(cfg.batch, 2048, dtype=np.int64)
    if cfg.name == "ragged":
        u = torch.rand(cfg.batch, generator=gen, dtype=torch.float64).numpy()
        lo, hi = math.log(256.0), math.log(64000.0)
        return np.rint(np.exp(lo + u * (hi - lo))).astype(np.int64)
    if cfg.name == "long_split":
        return np.full(cfg.batch, 65536, dtype=np.int64)
    if cfg.name == "cascade":   # the request's own tokens after the shared prefix
        return torch.randint(1, 513, (cfg.batch,), generator=gen).numpy().astype(np.int64)
    if cfg.name in ("fp8_kv", "fp8_kv_token_scales", "spec_decode_ragged"):
        return torch.randint(1024, 8193, (cfg.batch,), generator=gen).numpy().astype(np.int64)
    raise KeyError(cfg.name)


@dataclass
class DecodeBatch:
    """One decode batch: device tensors plus host copies of the page table."""
    q: torch.Tensor                 # [B, Hq, D], or [B, q_len, Hq, D]
    paged_kv: torch.Tensor          # [num_pages, 2, P, Hkv, D]
    indptr: torch.Tensor            # [B+1] int32, host
    indices: torch.Tensor           # [nnz] int32, on the device of paged_kv
    last_page_len: torch.Tensor     # [B] int32, host
    lengths: np.ndarray             # [B] int64
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    k_scale: float = 1.0
    v_scale: float = 1.0
    name: str = "custom"
    extra: dict = field(default_factory=dict)
    q_len: int = 1

    @property
    def batch(self) -> int:
        return int(self.indptr.shape[0] - 1)

    @property
    def num_pages(self) -> int:
        return int(self.paged_kv.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.lengths.sum())


def page_table(lengths, page_size: int, pool_pages: int | None, gen: torch.Generator,
               shuffle: bool = True):
    """indptr, indices, last_page_len for the given lengths.

    Page ids are the first sum(pages) entries of a seeded permutation of
    range(pool_pages) (or range(sum(pages)) when pool_pages is None), in the
    permutation's order; shuffle=False hands them out in order instead.
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    pages = (lengths + page_size - 1) // page_size
    last = np.where(pages > 0, lengths - (pages - 1) * page_size, 0)
    # requests with no pages: last_page_len is ignored, keep it valid
    last = np.where(pages > 0, last, page_size)
    indptr = np.zeros(len(lengths) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(pages)
    nnz = int(indptr[-1])
    pool = nnz if pool_pages is None else int(pool_pages)
    if pool < nnz:
        raise ValueError("page pool smaller than the pages requested")
    if shuffle:
        ids = torch.randperm(pool, generator=gen)[:nnz].numpy()
    else:
        ids = np.arange(nnz)
    return (torch.from_numpy(indptr.astype(np.int32)), torch.from_numpy(ids.astype(np.int32)),
            torch.from_numpy(last.astype(np.int32)), pool)


def _fp8_quantise(x: torch.Tensor) -> tuple[torch.Tensor, float]:
    """Per-tensor E4M3 quantisation of the input recipe: scale = amax / 448,
    codes = round-to-nearest-even cast of x / scale."""
    amax = float(x.abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    return (x / scale).to(torch.float8_e4m3fn), scale


def make_batch(*, batch_lengths, num_qo_heads: int, num_kv_heads: int, head_dim: int,
               q_dtype: torch.dtype, kv_dtype: torch.dtype, seed: int, device="cuda",
               page_size: int = PAGE_SIZE, pool_pages: int | None = None, shuffle: bool = True,
               name: str = "custom", token_scales: bool = False, q_len: int = 1,
               token_spread: float = 3.0) -> DecodeBatch:
    """A seeded batch with explicit lengths (any shape the library supports).
    token_scales=True (E4M3 only) draws per-token magnitudes 2^u, u uniform
    in [-token_spread, token_spread] (0: plain N(0,1) values), and stores one
    scale per (page, kv head, slot) in extra["k_scales"] / extra["v_scales"]."""
    gen = torch.Generator().manual_seed(seed)
    return _fill(batch_lengths, gen, num_qo_heads, num_kv_heads, head_dim, q_dtype, kv_dtype,
                 seed, device, page_size, pool_pages, shuffle, name, token_scales, q_len,
                 token_spread)


def make_cascade_batch(*, prefix_pages: int, suffix_lengths, num_qo_heads: int,
                       num_kv_heads: int, head_dim: int, dtype: torch.dtype, seed: int,
                       device="cuda", page_size: int = PAGE_SIZE, name="cascade",
                       kv_dtype: torch.dtype | None = None) -> DecodeBatch:
    """Requests sharing `prefix_pages` full pages, each followed by its own
    suffix of the given length.  The page table lists every full sequence
    (shared page ids first); extra["prefix_pages"] is the shared count.
    kv_dtype (default: dtype) may be E4M3, quantised with one scale per half
    as make_batch does."""
    gen = torch.Generator().manual_seed(seed)
    suffix_lengths = np.asarray(suffix_lengths, dtype=np.int64)
    sfx_pages = (suffix_lengths + page_size - 1) // page_size
    pool = prefix_pages + int(sfx_pages.sum())
    perm = torch.randperm(pool, generator=gen).numpy().astype(np.int32)
    prefix_ids, own = perm[:prefix_pages], perm[prefix_pages:]
    ids, indptr, last = [], [0], []
    off = 0
    for n, npg in zip(suffix_lengths, sfx_pages):
        ids.append(prefix_ids)
        ids.append(own[off:off + npg])
        off += npg
        indptr.append(indptr[-1] + prefix_pages + int(npg))
        last.append(int(n - (npg - 1) * page_size) if npg else page_size)
    lengths = prefix_pages * page_size + suffix_lengths
    dev = torch.device(device)
    vgen = torch.Generator(device=dev).manual_seed(seed)
    B = len(suffix_lengths)
    q = torch.randn((B, num_qo_heads, head_dim), generator=vgen, device=dev).to(dtype)
    kv_dtype = dtype if kv_dtype is None else kv_dtype
    k_scale = v_scale = 1.0
    if kv_dtype == torch.float8_e4m3fn:
        kv = torch.empty((pool, 2, page_size, num_kv_heads, head_dim), dtype=kv_dtype, device=dev)
        scales = []
        for half in range(2):
            x = torch.randn((pool, page_size, num_kv_heads, head_dim), generator=vgen,
                            device=dev, dtype=torch.float32)
            codes, s = _fp8_quantise(x)
            kv[:, half] = codes
            scales.append(s)
        k_scale, v_scale = scales
    else:
        kv = torch.randn((pool, 2, page_size, num_kv_heads, head_dim), generator=vgen,
                         device=dev, dtype=kv_dtype)
    return DecodeBatch(q=q, paged_kv=kv, indptr=torch.tensor(indptr, dtype=torch.int32),
                       indices=torch.from_numpy(np.concatenate(ids).astype(np.int32)).to(dev),
                       last_page_len=torch.tensor(last, dtype=torch.int32), lengths=lengths,
                       num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                       page_size=page_size, k_scale=k_scale, v_scale=v_scale, name=name,
                       extra={"prefix_pages": prefix_pages})


def cascade_parts(b: DecodeBatch):
    """(prefix page ids, suffix indptr, suffix indices, suffix last_page_len)
    of a cascade batch - the shared pages and each request's own pages."""
    npre = b.extra["prefix_pages"]
    indptr = b.indptr.numpy().astype(np.int64)
    ids = b.indices.cpu().numpy()
    prefix = ids[:npre]
    own, sfx_indptr = [], [0]
    for i in range(b.batch):
        seg = ids[indptr[i] + npre:indptr[i + 1]]
        own.append(seg)
        sfx_indptr.append(sfx_indptr[-1] + len(seg))
    dev = b.indices.device
    own_ids = np.concatenate(own) if own else np.zeros(0, np.int32)
    return (torch.from_numpy(prefix.astype(np.int32)).to(dev),
            torch.tensor(sfx_indptr, dtype=torch.int32),
            torch.from_numpy(own_ids.astype(np.int32)).to(dev), b.last_page_len.clone())


def make_config_batch(name: str, device="cuda", max_requests: int | None = None) -> DecodeBatch:
    """The named configuration, drawn from its seed.  max_requests keeps only
    the first requests of its length draw (a smaller batch of the same length
    distribution, e.g. for a profiler capture that must fit a few GB)."""
    cfg = CONFIGS[name]
    if name == "cascade":
        gen = torch.Generator().manual_seed(cfg.seed)
        return make_cascade_batch(prefix_pages=CASCADE_PREFIX_PAGES,
                                  suffix_lengths=draw_lengths(cfg, gen),
                                  num_qo_heads=cfg.num_qo_heads, num_kv_heads=cfg.num_kv_heads,
                                  head_dim=cfg.head_dim, dtype=cfg.q_dtype, seed=cfg.seed,
                                  device=device)
    gen = torch.Generator().manual_seed(cfg.seed)
    lengths = draw_lengths(cfg, gen)
    if max_requests is not None:
        lengths = lengths[:max_requests]
    pool = 64 if name == "tiny" else None
    if name == "spec_decode_ragged":   # U{1..4} draft tokens per request
        drafts = torch.randint(1, cfg.q_len + 1, (len(lengths),), generator=gen).numpy()
        return make_ragged_q_batch(batch_lengths=lengths, q_counts=drafts,
                                   num_qo_heads=cfg.num_qo_heads, num_kv_heads=cfg.num_kv_heads,
                                   head_dim=cfg.head_dim, q_dtype=cfg.q_dtype,
                                   kv_dtype=cfg.kv_dtype, seed=cfg.seed, device=device,
                                   name=name, gen=gen)
    return _fill(lengths, gen, cfg.num_qo_heads, cfg.num_kv_heads, cfg.head_dim, cfg.q_dtype,
                 cfg.kv_dtype, cfg.seed, device, cfg.page_size, pool, True, name,
                 name == "fp8_kv_token_scales", cfg.q_len)


def make_ragged_q_batch(*, batch_lengths, q_counts, num_qo_heads: int, num_kv_heads: int,
                        head_dim: int, q_dtype: torch.dtype, kv_dtype: torch.dtype, seed: int,
                        device="cuda", page_size: int = PAGE_SIZE, name: str = "custom",
                        gen: torch.Generator | None = None) -> DecodeBatch:
    """A seeded batch whose request i carries q_counts[i] query tokens (the
    last positions of its cache): q is [sum(q_counts), Hq, D] and
    extra["qo_indptr"] the request boundaries of its rows."""
    gen = gen if gen is not None else torch.Generator().manual_seed(seed)
    counts = np.asarray(q_counts, dtype=np.int64)
    b = _fill(batch_lengths, gen, num_qo_heads, num_kv_heads, head_dim, q_dtype, kv_dtype, seed,
              device, page_size, None, True, name, False, 1)
    qo = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    vgen = torch.Generator(device=b.q.device).manual_seed(seed + 7919)
    b.q = torch.randn((int(qo[-1]), num_qo_heads, head_dim), generator=vgen, device=b.q.device,
                      dtype=torch.float32).to(q_dtype)
    b.extra["qo_indptr"] = qo
    return b


def _fp8_token_quantise(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Per-token E4M3 quantisation of x [pages, P, Hkv, D]: one scale per
    (page, slot, kv head) = amax over D / 448.  Returns the codes and the
    scales laid out [pages, Hkv, P]."""
    amax = x.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = (x / scale).to(torch.float8_e4m3fn)
    return codes, scale.squeeze(-1).permute(0, 2, 1).contiguous()


def _fill(lengths, gen, Hq, Hkv, D, q_dtype, kv_dtype, seed, device, P, pool_pages, shuffle,
          name, token_scales=False, q_len=1, token_spread=3.0) -> DecodeBatch:
    lengths = np.asarray(lengths, dtype=np.int64)
    indptr, ids, last, pool = page_table(lengths, P, pool_pages, gen, shuffle)
    B = len(lengths)
    dev = torch.device(device)
    vgen = torch.Generator(device=dev).manual_seed(seed)
    q_shape = (B, Hq, D) if q_len == 1 else (B, q_len, Hq, D)
    q = torch.randn(q_shape, generator=vgen, device=dev, dtype=torch.float32).to(q_dtype)
    k_scale = v_scale = 1.0
    extra = {}
    if token_scales:
        if kv_dtype != torch.float8_e4m3fn:
            raise ValueError("per-token scales are for E4M3 KV")
        kv = torch.empty((pool, 2, P, Hkv, D), dtype=kv_dtype, device=dev)
        for half, key in ((0, "k_scales"), (1, "v_scales")):
            u = torch.rand((pool, P, Hkv, 1), generator=vgen, device=dev)
            mag = torch.exp2((u * 2 - 1) * token_spread)
            x = torch.randn((pool, P, Hkv, D), generator=vgen, device=dev) * mag
            codes, scales = _fp8_token_quantise(x)
            kv[:, half] = codes
            extra[key] = scales
            del x, codes, mag
    elif kv_dtype == torch.float8_e4m3fn:
        kv = torch.empty((pool, 2, P, Hkv, D), dtype=kv_dtype, device=dev)
        scales = []
        for half in range(2):
            x = torch.randn((pool, P, Hkv, D), generator=vgen, device=dev, dtype=torch.float32)
            codes, s = _fp8_quantise(x)
            kv[:, half] = codes
            scales.append(s)
            del x, codes
        k_scale, v_scale = scales
    else:
        kv = torch.randn((pool, 2, P, Hkv, D), generator=vgen, device=dev, dtype=kv_dtype)
    return DecodeBatch(q=q, paged_kv=kv, indptr=indptr, indices=ids.to(dev),
                       last_page_len=last, lengths=lengths, num_qo_heads=Hq,
                       num_kv_heads=Hkv, head_dim=D, page_size=P, k_scale=k_scale,
                       v_scale=v_scale, name=name, extra=extra, q_len=q_len)


def cauchy_schwarz_bound(b: DecodeBatch, sm_scale: float | None = None) -> float:
    """A bound on every logit sm_scale * k_scale * (q . k) of the batch that
    looks at no score: |q . k| <= |q| |k| (Cauchy-Schwarz), with the largest
    query norm of the batch and the largest key norm of the whole cache (a
    statistic a cache can keep as it is written).  The static bound a
    unified-max softmax starts from."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(b.head_dim)
    qn = b.q.float().norm(dim=-1).max().item()
    kn = 0.0
    for lo in range(0, b.num_pages, 4096):   # chunked: fp32 copies of a large cache
        k = b.paged_kv[lo:lo + 4096, 0].float()
        kn = max(kn, k.norm(dim=-1).max().item())
    return float(sm_scale * b.k_scale * qn * kn)
