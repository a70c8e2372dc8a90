"""Test-side marshalling between torch tensors and the float64 oracle.

Nothing here computes attention: it converts stored tensors to the raw bit
arrays the oracle reads, and cuts sub-batches out of a large batch so that
sampled requests can be checked one by one.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_decode_fa_gb300.workloads import DecodeBatch


def as_bits(t: torch.Tensor):
    """(numpy array of the stored bits, oracle element-type code)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.float32:
        return t.numpy(), oracle.F32
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), oracle.BF16
    if t.dtype == torch.float16:
        return t.view(torch.int16).numpy().view(np.uint16), oracle.F16
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy(), oracle.E4M3
    raise TypeError(t.dtype)


def oracle_decode(b: DecodeBatch, orc=None, sm_scale=None, num_threads=0):
    """Run the oracle on a whole batch; returns float64 (o, lse).  A batch
    with per-token scales (extra["k_scales"]) uses the per-token oracle."""
    orc = orc or oracle._default()
    q, qc = as_bits(b.q)
    kv, kc = as_bits(b.paged_kv)
    if "qo_indptr" in b.extra:
        return orc.batch_decode_ragged_q(
            q, qc, kv, kc, b.indptr.numpy(), b.indices.cpu().numpy(), b.last_page_len.numpy(),
            np.asarray(b.extra["qo_indptr"]), b.num_qo_heads, b.num_kv_heads, b.head_dim,
            b.page_size, sm_scale=sm_scale, k_scale=b.k_scale, v_scale=b.v_scale,
            num_threads=num_threads)
    if b.q_len > 1:
        return orc.batch_decode_multi(
            q, qc, kv, kc, b.indptr.numpy(), b.indices.cpu().numpy(), b.last_page_len.numpy(),
            b.q_len, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, sm_scale=sm_scale,
            k_scale=b.k_scale, v_scale=b.v_scale, num_threads=num_threads)
    if "k_scales" in b.extra:
        return orc.batch_decode_token_scales(
            q, qc, kv, kc, b.indptr.numpy(), b.indices.cpu().numpy(), b.last_page_len.numpy(),
            b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size,
            b.extra["k_scales"].cpu().numpy(), b.extra["v_scales"].cpu().numpy(),
            sm_scale=sm_scale, num_threads=num_threads)
    return orc.batch_decode(q, qc, kv, kc, b.indptr.numpy(), b.indices.cpu().numpy(),
                            b.last_page_len.numpy(), b.num_qo_heads, b.num_kv_heads,
                            b.head_dim, b.page_size, sm_scale=sm_scale, k_scale=b.k_scale,
                            v_scale=b.v_scale, num_threads=num_threads)


def sub_batch(b: DecodeBatch, requests) -> DecodeBatch:
    """The given requests of b as a compact host batch (their pages copied)."""
    requests = [int(r) for r in requests]
    indptr = b.indptr.numpy().astype(np.int64)
    ids = b.indices.cpu().numpy()
    pages, counts = [], []
    for r in requests:
        pages.append(ids[indptr[r]:indptr[r + 1]])
        counts.append(indptr[r + 1] - indptr[r])
    page_ids = np.concatenate(pages) if pages else np.zeros(0, np.int64)
    sel = torch.from_numpy(page_ids.astype(np.int64)).to(b.paged_kv.device)
    kv = b.paged_kv.index_select(0, sel).to("cpu") if len(page_ids) else b.paged_kv[:1].to("cpu")
    new_indptr = np.zeros(len(requests) + 1, np.int64)
    new_indptr[1:] = np.cumsum(counts)
    rq = torch.tensor(requests, dtype=torch.int64, device=b.q.device)
    extra = {}
    q_sel = b.q.index_select(0, rq).to("cpu") if "qo_indptr" not in b.extra else None
    if "qo_indptr" in b.extra:   # ragged query rows: the requests' own rows, re-indexed
        qo = np.asarray(b.extra["qo_indptr"], np.int64)
        rows = np.concatenate([np.arange(qo[r], qo[r + 1]) for r in requests] + [np.zeros(0, np.int64)])
        q_sel = b.q.index_select(0, torch.from_numpy(rows).to(b.q.device)).to("cpu")
        counts = [int(qo[r + 1] - qo[r]) for r in requests]
        extra["qo_indptr"] = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    for key in ("k_scales", "v_scales"):
        if key in b.extra:
            t = b.extra[key]
            extra[key] = (t.index_select(0, sel).to("cpu") if len(page_ids) else t[:1].to("cpu"))
    return DecodeBatch(
        q=q_sel, paged_kv=kv,
        indptr=torch.from_numpy(new_indptr.astype(np.int32)),
        indices=torch.arange(len(page_ids), dtype=torch.int32),
        last_page_len=b.last_page_len[requests].clone(),
        lengths=b.lengths[requests], num_qo_heads=b.num_qo_heads,
        num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size,
        k_scale=b.k_scale, v_scale=b.v_scale, name=b.name + "-sub", extra=extra, q_len=b.q_len)


def dense_pages(K, V, page_size, perm_seed=0, pool_extra=0, pad_value=np.nan):
    """Lay per-request dense K/V ([len, Hkv, D] float32 arrays) into a shuffled
    page pool.  Slots past each request's length are filled with pad_value.
    Returns (paged_kv float32 [pages, 2, P, Hkv, D], indptr, indices, last)."""
    rng = np.random.default_rng(perm_seed)
    Hkv, D = K[0].shape[1], K[0].shape[2]
    npg = [(k.shape[0] + page_size - 1) // page_size for k in K]
    nnz = sum(npg)
    pool = nnz + pool_extra
    perm = rng.permutation(pool)[:nnz]
    kv = np.full((pool, 2, page_size, Hkv, D), pad_value, dtype=np.float32)
    indptr = np.zeros(len(K) + 1, np.int32)
    indptr[1:] = np.cumsum(npg)
    last = np.zeros(len(K), np.int32)
    for i, (k, v) in enumerate(zip(K, V)):
        n = k.shape[0]
        last[i] = n - (npg[i] - 1) * page_size if npg[i] else page_size
        for t in range(n):
            page = perm[indptr[i] + t // page_size]
            kv[page, 0, t % page_size] = k[t]
            kv[page, 1, t % page_size] = v[t]
    return kv, indptr, perm.astype(np.int32), last
