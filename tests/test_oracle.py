"""Pins of the float64 oracle against things other than itself: worked closed
forms, the special cases the method reduces to, brute force, library
routines, and invariants that a dropped term, a wrong sign, index or operand
would break.  CPU only.

The pin functions take the oracle instance as an argument so that
test_oracle_mutations.py can run them on copies of the oracle with a planted
mistake and show that each mistake is caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import dense_pages

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _decode_dense(orc, q, K, V, page_size=4, sm_scale=None, perm_seed=0, pool_extra=3):
    """Oracle over per-request dense fp32 K/V laid into shuffled pages."""
    kv, indptr, indices, last = dense_pages(K, V, page_size, perm_seed, pool_extra)
    Hq = q.shape[1]
    Hkv, D = K[0].shape[1], K[0].shape[2]
    return orc.batch_decode(np.ascontiguousarray(q, np.float32), oracle.F32, kv, oracle.F32,
                            indptr, indices, last, Hq, Hkv, D, page_size, sm_scale=sm_scale)


# ---------------------------------------------------------------- element decoding

def pin_e4m3_all_codes(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.decode_e4m3(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1.0, got[0x80]) == -1.0


def pin_e4m3_spec_points(orc):
    # OCP FP8 E4M3: bias 7, 3 mantissa bits, no infinities.
    assert orc.decode_e4m3(0x7E) == 448.0            # largest finite
    assert orc.decode_e4m3(0x08) == 2.0 ** -6        # smallest normal
    assert orc.decode_e4m3(0x01) == 2.0 ** -9        # smallest subnormal
    assert orc.decode_e4m3(0x07) == 7 * 2.0 ** -9    # largest subnormal
    assert orc.decode_e4m3(0x38) == 1.0
    assert orc.decode_e4m3(0xB8) == -1.0
    assert orc.decode_e4m3(0x3C) == 1.5
    assert math.isnan(orc.decode_e4m3(0x7F)) and math.isnan(orc.decode_e4m3(0xFF))


def pin_bf16_codes(orc):
    bits = torch.arange(65536, dtype=torch.int32)
    ref = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    sample = list(range(0, 65536, 7)) + [0x3F80, 0xC000, 0x7F80, 0xFF80, 0x0001, 0x8000]
    got = np.array([orc.decode_bf16(b) for b in sample])
    r = ref[sample]
    nan = np.isnan(r)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], r[~nan])
    assert orc.decode_bf16(0x3F80) == 1.0 and orc.decode_bf16(0xC000) == -2.0


def pin_f16_codes(orc):
    ref = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([orc.decode_f16(b) for b in range(0, 65536, 3)])
    r = ref[::3]
    nan = np.isnan(r)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], r[~nan])


def test_e4m3_all_codes(orc):
    pin_e4m3_all_codes(orc)


def test_e4m3_spec_points(orc):
    pin_e4m3_spec_points(orc)


def test_bf16_codes(orc):
    pin_bf16_codes(orc)


def test_f16_codes(orc):
    pin_f16_codes(orc)


# ---------------------------------------------------------------- closed forms

def pin_single_key(orc):
    """len = 1: softmax of one logit is 1, so o = v0 and lse = the logit."""
    rng = np.random.default_rng(1)
    D, Hkv, g = 8, 2, 2
    K = [rng.standard_normal((1, Hkv, D)).astype(np.float32)]
    V = [rng.standard_normal((1, Hkv, D)).astype(np.float32)]
    q = rng.standard_normal((1, Hkv * g, D)).astype(np.float32)
    o, lse = _decode_dense(orc, q, K, V, sm_scale=0.37)
    for h in range(Hkv * g):
        kvh = h // g
        np.testing.assert_allclose(o[0, h], V[0][0, kvh].astype(np.float64), rtol=0, atol=1e-15)
        s = 0.37 * float(np.dot(q[0, h].astype(np.float64), K[0][0, kvh].astype(np.float64)))
        assert abs(lse[0, h] - s) < 1e-12


def pin_identical_keys(orc):
    """n equal keys: equal weights, o = mean(V), lse = s + ln n."""
    rng = np.random.default_rng(2)
    D, n = 16, 37
    k = rng.standard_normal(D).astype(np.float32)
    K = [np.tile(k, (n, 1, 1))]
    V = [rng.standard_normal((n, 1, D)).astype(np.float32)]
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    o, lse = _decode_dense(orc, q, K, V, page_size=8)
    np.testing.assert_allclose(o[0, 0], V[0][:, 0].astype(np.float64).mean(0), rtol=0, atol=1e-13)
    s = float(np.dot(q[0, 0].astype(np.float64), k.astype(np.float64))) / math.sqrt(D)
    assert abs(lse[0, 0] - (s + math.log(n))) < 1e-12


def pin_zero_query(orc):
    """q = 0: uniform weights, lse = ln n."""
    rng = np.random.default_rng(3)
    D, n = 8, 21
    K = [rng.standard_normal((n, 1, D)).astype(np.float32)]
    V = [rng.standard_normal((n, 1, D)).astype(np.float32)]
    q = np.zeros((1, 1, D), np.float32)
    o, lse = _decode_dense(orc, q, K, V, page_size=4)
    np.testing.assert_allclose(o[0, 0], V[0][:, 0].astype(np.float64).mean(0), rtol=0, atol=1e-13)
    assert abs(lse[0, 0] - math.log(n)) < 1e-12


def pin_convexity(orc):
    """Constant V gives o = c; in general o lies inside the range of V."""
    rng = np.random.default_rng(4)
    D, n = 8, 50
    K = [rng.standard_normal((n, 1, D)).astype(np.float32) * 3]
    c = rng.standard_normal(D).astype(np.float32)
    Vc = [np.tile(c, (n, 1, 1))]
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    o, _ = _decode_dense(orc, q, K, Vc)
    np.testing.assert_allclose(o[0, 0], c.astype(np.float64), rtol=0, atol=1e-12)
    V = [rng.standard_normal((n, 1, D)).astype(np.float32)]
    o, _ = _decode_dense(orc, q, K, V)
    assert np.all(o[0, 0] <= V[0][:, 0].max(0) + 1e-12)
    assert np.all(o[0, 0] >= V[0][:, 0].min(0) - 1e-12)


def pin_split_merge(orc):
    """Split the KV axis at a page boundary, decode both halves, merge with the
    rule: equals the unsplit result (same recurrence applied hierarchically)."""
    rng = np.random.default_rng(5)
    D, P, Hkv, g = 16, 4, 2, 2
    n = 4 * P + 3
    K = rng.standard_normal((n, Hkv, D)).astype(np.float32)
    V = rng.standard_normal((n, Hkv, D)).astype(np.float32)
    q = rng.standard_normal((1, Hkv * g, D)).astype(np.float32)
    o_full, lse_full = _decode_dense(orc, q, [K], [V], page_size=P)
    parts = []
    for lo, hi in ((0, 2 * P), (2 * P, n)):
        parts.append(_decode_dense(orc, q, [K[lo:hi]], [V[lo:hi]], page_size=P))
    o_m, lse_m = orc.merge_states(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    np.testing.assert_allclose(o_m, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_m, lse_full, rtol=0, atol=1e-12)
    # three-way split, folded in order
    cuts = (0, P, 3 * P, n)
    pieces = [_decode_dense(orc, q, [K[a:b]], [V[a:b]], page_size=P) for a, b in zip(cuts, cuts[1:])]
    o3, l3 = orc.merge_many([p[0] for p in pieces], [p[1] for p in pieces])
    np.testing.assert_allclose(o3, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l3, lse_full, rtol=0, atol=1e-12)


def pin_gqa_equals_repeated_mha(orc):
    """Query head h reads kv head h // g: GQA equals MHA over kv heads repeated g times."""
    rng = np.random.default_rng(6)
    D, Hkv, g, n = 8, 3, 4, 23
    K = [rng.standard_normal((n, Hkv, D)).astype(np.float32)]
    V = [rng.standard_normal((n, Hkv, D)).astype(np.float32)]
    q = rng.standard_normal((1, Hkv * g, D)).astype(np.float32)
    o_g, l_g = _decode_dense(orc, q, K, V)
    K_r = [np.repeat(K[0], g, axis=1)]
    V_r = [np.repeat(V[0], g, axis=1)]
    o_m, l_m = _decode_dense(orc, q, K_r, V_r)
    np.testing.assert_array_equal(o_g, o_m)
    np.testing.assert_array_equal(l_g, l_m)


def pin_page_permutation(orc):
    """Physical page placement does not matter once indices follow it."""
    rng = np.random.default_rng(7)
    K = [rng.standard_normal((n, 2, 8)).astype(np.float32) for n in (5, 17, 9)]
    V = [rng.standard_normal((n, 2, 8)).astype(np.float32) for n in (5, 17, 9)]
    q = rng.standard_normal((3, 4, 8)).astype(np.float32)
    a = _decode_dense(orc, q, K, V, perm_seed=1)
    b = _decode_dense(orc, q, K, V, perm_seed=2, pool_extra=11)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def _brute(q, K, V, scale):
    """Pure-Python loops, independent of the oracle: softmax(q.K^T * scale) V."""
    Hq = len(q)
    Hkv = len(K[0])
    g = Hq // Hkv
    outs, lses = [], []
    for h in range(Hq):
        kvh = h // g
        s = [scale * sum(a * b for a, b in zip(q[h], K[t][kvh])) for t in range(len(K))]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        tot = sum(w)
        outs.append([sum(w[t] * V[t][kvh][d] for t in range(len(K))) / tot for d in range(len(q[h]))])
        lses.append(mx + math.log(tot))
    return outs, lses


def pin_brute_force(orc):
    rng = np.random.default_rng(8)
    for trial in range(6):
        D = int(rng.integers(1, 6))
        Hkv = int(rng.integers(1, 3))
        g = int(rng.integers(1, 3))
        P = int(rng.integers(1, 5))
        lens = [int(x) for x in rng.integers(1, 12, size=int(rng.integers(1, 4)))]
        K = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in lens]
        V = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in lens]
        q = rng.standard_normal((len(lens), Hkv * g, D)).astype(np.float32)
        scale = float(rng.uniform(0.1, 2.0))
        o, lse = _decode_dense(orc, q, K, V, page_size=P, sm_scale=scale, perm_seed=trial)
        for i in range(len(lens)):
            bo, bl = _brute(q[i].astype(np.float64).tolist(), K[i].astype(np.float64).tolist(),
                            V[i].astype(np.float64).tolist(), scale)
            np.testing.assert_allclose(o[i], np.array(bo), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[i], np.array(bl), rtol=0, atol=1e-12)


def pin_torch_dense(orc):
    """Against torch's float64 softmax and matmul on the gathered, dequantised
    tensors, for fp32, bf16 and fp8-with-scales storage."""
    gen = torch.Generator().manual_seed(9)
    for kv_dtype, q_dtype in ((torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                              (torch.float8_e4m3fn, torch.bfloat16), (torch.float16, torch.float16)):
        B, Hq, Hkv, D, P = 3, 4, 2, 16, 4
        lens = [1, 9, 14]
        npg = [(n + P - 1) // P for n in lens]
        num_pages = sum(npg) + 2
        kv32 = torch.randn((num_pages, 2, P, Hkv, D), generator=gen)
        kv = kv32.to(kv_dtype)
        q = torch.randn((B, Hq, D), generator=gen).to(q_dtype)
        ks, vs = (0.75, 1.5) if kv_dtype == torch.float8_e4m3fn else (1.0, 1.0)
        perm = torch.randperm(num_pages, generator=gen)[: sum(npg)].to(torch.int32)
        indptr = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
        last = np.array([n - (p - 1) * P for n, p in zip(lens, npg)], np.int32)
        from tests.helpers import as_bits
        qb, qc = as_bits(q)
        kb, kc = as_bits(kv)
        o, lse = orc.batch_decode(qb, qc, kb, kc, indptr, perm.numpy(), last, Hq, Hkv, D, P,
                                  k_scale=ks, v_scale=vs)
        kvd = kv.to(torch.float64)
        for i, n in enumerate(lens):
            ids = perm[indptr[i]:indptr[i + 1]].long()
            Kd = (kvd[ids, 0].reshape(-1, Hkv, D)[:n] * ks)
            Vd = (kvd[ids, 1].reshape(-1, Hkv, D)[:n] * vs)
            qd = q[i].to(torch.float64)
            g = Hq // Hkv
            Kr = Kd.repeat_interleave(g, dim=1)  # [n, Hq, D]
            Vr = Vd.repeat_interleave(g, dim=1)
            s = torch.einsum("hd,nhd->hn", qd, Kr) / math.sqrt(D)
            w = torch.softmax(s, dim=-1)
            ref_o = torch.einsum("hn,nhd->hd", w, Vr).numpy()
            ref_lse = torch.logsumexp(s, dim=-1).numpy()
            np.testing.assert_allclose(o[i], ref_o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[i], ref_lse, rtol=0, atol=1e-12)


def _fp8_batch(seed, lens=(1, 9, 14, 33), Hq=4, Hkv=2, D=16, P=4):
    gen = torch.Generator().manual_seed(seed)
    npg = [(n + P - 1) // P for n in lens]
    num_pages = sum(npg) + 2
    kv = (torch.randn((num_pages, 2, P, Hkv, D), generator=gen) * 40).to(torch.float8_e4m3fn)
    q = torch.randn((len(lens), Hq, D), generator=gen).to(torch.bfloat16)
    perm = torch.randperm(num_pages, generator=gen)[: sum(npg)].to(torch.int32)
    indptr = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    last = np.array([n - (p - 1) * P for n, p in zip(lens, npg)], np.int32)
    ks = (torch.rand((num_pages, Hkv, P), generator=gen) * 0.05 + 0.001).to(torch.float32)
    vs = (torch.rand((num_pages, Hkv, P), generator=gen) * 0.05 + 0.001).to(torch.float32)
    return kv, q, perm, indptr, last, ks, vs, lens, (Hq, Hkv, D, P)


def pin_token_scales_dense(orc):
    """Per-token, per-kv-head scales against torch float64 on the tensors
    dequantised element by element with their own scale."""
    from tests.helpers import as_bits
    kv, q, perm, indptr, last, ks, vs, lens, (Hq, Hkv, D, P) = _fp8_batch(13)
    qb, qc = as_bits(q)
    kb, kc = as_bits(kv)
    o, lse = orc.batch_decode_token_scales(qb, qc, kb, kc, indptr, perm.numpy(), last, Hq, Hkv,
                                           D, P, ks.numpy(), vs.numpy())
    kvd = kv.to(torch.float64)
    # [pages, Hkv, P] -> [pages, P, Hkv, 1] to match [pages, 2, P, Hkv, D]
    ksd = ks.to(torch.float64).permute(0, 2, 1).unsqueeze(-1)
    vsd = vs.to(torch.float64).permute(0, 2, 1).unsqueeze(-1)
    g = Hq // Hkv
    for i, n in enumerate(lens):
        ids = perm[indptr[i]:indptr[i + 1]].long()
        Kd = (kvd[ids, 0] * ksd[ids]).reshape(-1, Hkv, D)[:n]
        Vd = (kvd[ids, 1] * vsd[ids]).reshape(-1, Hkv, D)[:n]
        s = torch.einsum("hd,nhd->hn", q[i].to(torch.float64), Kd.repeat_interleave(g, 1))
        s = s / math.sqrt(D)
        ref_o = torch.einsum("hn,nhd->hd", torch.softmax(s, -1), Vd.repeat_interleave(g, 1))
        np.testing.assert_allclose(o[i], ref_o.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[i], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def pin_token_scales_uniform(orc):
    """Every per-token scale equal to c is the per-tensor scale c."""
    from tests.helpers import as_bits
    kv, q, perm, indptr, last, ks, vs, lens, (Hq, Hkv, D, P) = _fp8_batch(14)
    qb, qc = as_bits(q)
    kb, kc = as_bits(kv)
    ks[:] = 0.015625  # exactly representable in float32
    vs[:] = 0.5
    a = orc.batch_decode_token_scales(qb, qc, kb, kc, indptr, perm.numpy(), last, Hq, Hkv, D, P,
                                      ks.numpy(), vs.numpy())
    b = orc.batch_decode(qb, qc, kb, kc, indptr, perm.numpy(), last, Hq, Hkv, D, P,
                         k_scale=0.015625, v_scale=0.5)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def _head_scale_case(seed=15):
    from tests.helpers import as_bits
    kv, q, perm, indptr, last, _, _, lens, (Hq, Hkv, D, P) = _fp8_batch(seed, Hq=6, Hkv=3)
    rng = np.random.default_rng(seed)
    kh = (rng.random(Hkv) * 0.05 + 0.002).astype(np.float32)
    vh = (rng.random(Hkv) * 0.05 + 0.002).astype(np.float32)
    qb, qc = as_bits(q)
    kb, kc = as_bits(kv)
    return (qb, qc, kb, kc, indptr, perm.numpy(), last, Hq, Hkv, D, P), kh, vh, kv, q, lens


def head_scales_match_per_tensor_per_head(orc, o, lse, args, kh, vh):
    """Rows of kv head h's query heads equal the per-tensor oracle run with
    k_scale = kh[h], v_scale = vh[h] (the heads do not interact)."""
    qb, qc, kb, kc, indptr, ids, last, Hq, Hkv, D, P = args
    g = Hq // Hkv
    for h in range(Hkv):
        ro, rl = orc.batch_decode(qb, qc, kb, kc, indptr, ids, last, Hq, Hkv, D, P,
                                  k_scale=float(kh[h]), v_scale=float(vh[h]))
        rows = slice(h * g, (h + 1) * g)
        np.testing.assert_allclose(o[:, rows], ro[:, rows], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, rows], rl[:, rows], rtol=0, atol=1e-12)


def pin_head_scales_per_head(orc):
    """One scale per kv head: each head's rows are the per-tensor result
    with that head's two scales."""
    args, kh, vh, *_ = _head_scale_case()
    o, lse = orc.batch_decode_head_scales(*args, kh, vh)
    head_scales_match_per_tensor_per_head(orc, o, lse, args, kh, vh)


def pin_head_scales_dense(orc):
    """One scale per kv head against torch float64 on K and V dequantised
    with their head's scale."""
    args, kh, vh, kv, q, lens = _head_scale_case(16)
    qb, qc, kb, kc, indptr, ids, last, Hq, Hkv, D, P = args
    o, lse = orc.batch_decode_head_scales(*args, kh, vh)
    kvd = kv.to(torch.float64)
    khd = torch.tensor(kh, dtype=torch.float64)[:, None]
    vhd = torch.tensor(vh, dtype=torch.float64)[:, None]
    g = Hq // Hkv
    for i, n in enumerate(lens):
        pid = torch.from_numpy(ids[indptr[i]:indptr[i + 1]]).long()
        Kd = kvd[pid, 0].reshape(-1, Hkv, D)[:n] * khd
        Vd = kvd[pid, 1].reshape(-1, Hkv, D)[:n] * vhd
        s = torch.einsum("hd,nhd->hn", q[i].to(torch.float64), Kd.repeat_interleave(g, 1))
        s = s / math.sqrt(D)
        ref_o = torch.einsum("hn,nhd->hd", torch.softmax(s, -1), Vd.repeat_interleave(g, 1))
        np.testing.assert_allclose(o[i], ref_o.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[i], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def _multi_batch(seed, lens=(5, 16, 17, 40), q_len=3, Hq=4, Hkv=2, D=8, P=4):
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in lens]
    kv, indptr, indices, last = dense_pages(K, V, P, perm_seed=seed, pool_extra=2)
    q = rng.standard_normal((len(lens), q_len, Hq, D)).astype(np.float32)
    return q, K, V, kv, indptr, indices, last, lens, (q_len, Hq, Hkv, D, P)


def pin_multi_token_truncation(orc):
    """Query token i of a request equals single-token decode over the request
    cut after position len - q_len + i (same pages, shorter last page)."""
    q, K, V, kv, indptr, indices, last, lens, (ql, Hq, Hkv, D, P) = _multi_batch(15)
    o, lse = orc.batch_decode_multi(q, oracle.F32, kv, oracle.F32, indptr, indices, last, ql, Hq,
                                    Hkv, D, P)
    for r, n in enumerate(lens):
        for i in range(ql):
            vis = n - ql + i + 1
            npg = (vis + P - 1) // P
            ip = np.array([0, npg], np.int32)
            ids = indices[indptr[r]:indptr[r] + npg]
            lp = np.array([vis - (npg - 1) * P], np.int32)
            o1, l1 = orc.batch_decode(np.ascontiguousarray(q[r, i][None]), oracle.F32, kv,
                                      oracle.F32, ip, ids, lp, Hq, Hkv, D, P)
            np.testing.assert_array_equal(o[r, i], o1[0])
            np.testing.assert_array_equal(lse[r, i], l1[0])


def pin_multi_token_causal_dense(orc):
    """Against torch float64 attention with an explicit causal mask over the
    draft tokens."""
    q, K, V, kv, indptr, indices, last, lens, (ql, Hq, Hkv, D, P) = _multi_batch(16, q_len=4)
    o, lse = orc.batch_decode_multi(q, oracle.F32, kv, oracle.F32, indptr, indices, last, ql, Hq,
                                    Hkv, D, P)
    g = Hq // Hkv
    for r, n in enumerate(lens):
        Kr = torch.from_numpy(K[r]).double().repeat_interleave(g, 1)   # [n, Hq, D]
        Vr = torch.from_numpy(V[r]).double().repeat_interleave(g, 1)
        qd = torch.from_numpy(q[r]).double()                             # [ql, Hq, D]
        s = torch.einsum("ihd,nhd->ihn", qd, Kr) / math.sqrt(D)
        pos = torch.arange(n)
        limit = n - ql + torch.arange(ql)
        s = s.masked_fill(pos[None, None, :] > limit[:, None, None], -math.inf)
        np.testing.assert_allclose(o[r], torch.einsum("ihn,nhd->ihd", torch.softmax(s, -1), Vr).numpy(),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


def pin_multi_token_one_is_decode(orc):
    q, K, V, kv, indptr, indices, last, lens, (ql, Hq, Hkv, D, P) = _multi_batch(17, q_len=1)
    a = orc.batch_decode_multi(q, oracle.F32, kv, oracle.F32, indptr, indices, last, 1, Hq, Hkv,
                               D, P)
    b = orc.batch_decode(q[:, 0], oracle.F32, kv, oracle.F32, indptr, indices, last, Hq, Hkv, D, P)
    np.testing.assert_array_equal(a[0][:, 0], b[0])
    np.testing.assert_array_equal(a[1][:, 0], b[1])
    with pytest.raises(ValueError):   # a request shorter than q_len
        orc.batch_decode_multi(np.zeros((4, 6, Hq, D), np.float32), oracle.F32, kv, oracle.F32,
                               indptr, indices, last, 6, Hq, Hkv, D, P)


def _ragged_q_batch(seed, lens=(5, 0, 16, 17, 40, 3), nq=(3, 0, 1, 4, 2, 3), Hq=4, Hkv=2, D=8,
                    P=4):
    rng = np.random.default_rng(seed)
    K = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((n, Hkv, D)).astype(np.float32) for n in lens]
    kv, indptr, indices, last = dense_pages(K, V, P, perm_seed=seed, pool_extra=2)
    qo_indptr = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = rng.standard_normal((int(qo_indptr[-1]), Hq, D)).astype(np.float32)
    return q, K, V, kv, indptr, indices, last, qo_indptr, lens, nq, (Hq, Hkv, D, P)


def pin_ragged_q_truncation(orc):
    """Query token j of request i (n_i tokens) equals single-token decode over
    the request cut after position len_i - n_i + j."""
    q, K, V, kv, indptr, indices, last, qo, lens, nq, (Hq, Hkv, D, P) = _ragged_q_batch(18)
    o, lse = orc.batch_decode_ragged_q(q, oracle.F32, kv, oracle.F32, indptr, indices, last, qo,
                                       Hq, Hkv, D, P)
    assert o.shape[0] == sum(nq)
    for r, (n, k) in enumerate(zip(lens, nq)):
        for j in range(k):
            vis = n - k + j + 1
            npg = (vis + P - 1) // P
            ip = np.array([0, npg], np.int32)
            ids = indices[indptr[r]:indptr[r] + npg]
            lp = np.array([vis - (npg - 1) * P], np.int32)
            row = qo[r] + j
            o1, l1 = orc.batch_decode(np.ascontiguousarray(q[row][None]), oracle.F32, kv,
                                      oracle.F32, ip, ids, lp, Hq, Hkv, D, P)
            np.testing.assert_array_equal(o[row], o1[0])
            np.testing.assert_array_equal(lse[row], l1[0])


def pin_ragged_q_sdpa(orc):
    """Against torch's float64 scaled_dot_product_attention (a library
    routine) with a boolean mask of the positions each query token sees."""
    import torch.nn.functional as F
    q, K, V, kv, indptr, indices, last, qo, lens, nq, (Hq, Hkv, D, P) = _ragged_q_batch(19)
    o, lse = orc.batch_decode_ragged_q(q, oracle.F32, kv, oracle.F32, indptr, indices, last, qo,
                                       Hq, Hkv, D, P)
    g = Hq // Hkv
    for r, (n, k) in enumerate(zip(lens, nq)):
        if k == 0:
            continue
        Kr = torch.from_numpy(K[r]).double().repeat_interleave(g, 1).transpose(0, 1)  # [Hq, n, D]
        Vr = torch.from_numpy(V[r]).double().repeat_interleave(g, 1).transpose(0, 1)
        qr = torch.from_numpy(q[qo[r]:qo[r + 1]]).double().transpose(0, 1)            # [Hq, k, D]
        mask = torch.arange(n)[None, :] <= (n - k + torch.arange(k))[:, None]          # [k, n]
        ref = F.scaled_dot_product_attention(qr, Kr, Vr, attn_mask=mask)              # [Hq, k, D]
        np.testing.assert_allclose(o[qo[r]:qo[r + 1]], ref.transpose(0, 1).numpy(), rtol=0,
                                   atol=1e-12)


def pin_ragged_q_one_token_is_decode(orc):
    """n_i = 1 for every request is plain decode; n_i = q_len for every
    request is the uniform multi-token decode; a request shorter than its
    draft count is refused."""
    q, K, V, kv, indptr, indices, last, qo, lens, nq, (Hq, Hkv, D, P) = _ragged_q_batch(
        20, lens=(5, 16, 17, 40), nq=(1, 1, 1, 1))
    a = orc.batch_decode_ragged_q(q, oracle.F32, kv, oracle.F32, indptr, indices, last, qo, Hq,
                                  Hkv, D, P)
    b = orc.batch_decode(q, oracle.F32, kv, oracle.F32, indptr, indices, last, Hq, Hkv, D, P)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    q, K, V, kv, indptr, indices, last, qo, lens, nq, (Hq, Hkv, D, P) = _ragged_q_batch(
        21, lens=(5, 16, 17, 40), nq=(3, 3, 3, 3))
    a = orc.batch_decode_ragged_q(q, oracle.F32, kv, oracle.F32, indptr, indices, last, qo, Hq,
                                  Hkv, D, P)
    m = orc.batch_decode_multi(q.reshape(4, 3, Hq, D), oracle.F32, kv, oracle.F32, indptr,
                               indices, last, 3, Hq, Hkv, D, P)
    np.testing.assert_array_equal(a[0], m[0].reshape(12, Hq, D))
    with pytest.raises(ValueError):
        orc.batch_decode_ragged_q(np.zeros((6, Hq, D), np.float32), oracle.F32, kv, oracle.F32,
                                  indptr, indices, last, [0, 6, 6, 6, 6], Hq, Hkv, D, P)


def pin_empty_request(orc):
    rng = np.random.default_rng(10)
    K = [rng.standard_normal((5, 1, 4)).astype(np.float32)]
    V = [rng.standard_normal((5, 1, 4)).astype(np.float32)]
    kv, indptr, indices, last = dense_pages(K, V, 4, 0, 2)
    indptr = np.array([0, 0, indptr[1]], np.int32)  # request 0 empty, request 1 = K/V
    last = np.array([3, last[0]], np.int32)
    q = rng.standard_normal((2, 1, 4)).astype(np.float32)
    o, lse = orc.batch_decode(q, oracle.F32, kv, oracle.F32, indptr, indices, last, 1, 1, 4, 4)
    assert np.all(o[0] == 0.0) and lse[0, 0] == -math.inf
    assert np.all(np.isfinite(o[1])) and np.isfinite(lse[1, 0])


def pin_padding_never_read(orc):
    """Slots past last_page_len (NaN in dense_pages) and unused pool pages
    must not reach the result."""
    rng = np.random.default_rng(11)
    lens = (7, 13, 1, 16)
    K = [rng.standard_normal((n, 1, 8)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((n, 1, 8)).astype(np.float32) for n in lens]
    q = rng.standard_normal((4, 1, 8)).astype(np.float32)
    o, lse = _decode_dense(orc, q, K, V, page_size=4)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def pin_golden_decode(orc):
    with open(os.path.join(GOLDEN, "decode_worked_examples.json")) as f:
        spec = json.load(f)
    for case in spec["cases"]:
        P, Hq, Hkv, D = case["page_size"], case["num_qo_heads"], case["num_kv_heads"], case["head_dim"]
        kv = np.full((case["num_pages"], 2, P, Hkv, D), np.nan, np.float32)
        indptr, indices, last = [0], [], []
        for r, (Kt, Vt, ids) in enumerate(zip(case["tokens_K"], case["tokens_V"], case["page_ids"])):
            for t, (k, v) in enumerate(zip(Kt, Vt)):
                kv[ids[t // P], 0, t % P] = k
                kv[ids[t // P], 1, t % P] = v
            indices += ids
            indptr.append(indptr[-1] + len(ids))
            last.append(len(Kt) - (len(ids) - 1) * P)
        o, lse = orc.batch_decode(np.array(case["q"], np.float32), oracle.F32, kv, oracle.F32,
                                  np.array(indptr), np.array(indices), np.array(last),
                                  Hq, Hkv, D, P, sm_scale=case["sm_scale"])
        np.testing.assert_allclose(o, np.array(case["expected_o"]), rtol=0, atol=1e-6)
        np.testing.assert_allclose(lse, np.array(case["expected_lse"]), rtol=0, atol=1e-6)


def pin_rejects_bad_args(orc):
    kv = np.zeros((2, 2, 4, 1, 4), np.float32)
    q = np.zeros((1, 1, 4), np.float32)
    with pytest.raises(ValueError):   # last_page_len 0
        orc.batch_decode(q, oracle.F32, kv, oracle.F32, [0, 1], [0], [0], 1, 1, 4, 4)
    with pytest.raises(ValueError):   # page id out of the pool
        orc.batch_decode(q, oracle.F32, kv, oracle.F32, [0, 1], [2], [1], 1, 1, 4, 4)
    with pytest.raises(ValueError):   # decreasing indptr
        orc.batch_decode(np.zeros((2, 1, 4), np.float32), oracle.F32, kv, oracle.F32,
                         [0, 1, 0], [0], [1, 1], 1, 1, 4, 4)


@pytest.mark.parametrize("pin", [
    pin_single_key, pin_identical_keys, pin_zero_query, pin_convexity, pin_split_merge,
    pin_gqa_equals_repeated_mha, pin_page_permutation, pin_brute_force, pin_torch_dense,
    pin_empty_request, pin_padding_never_read, pin_golden_decode, pin_rejects_bad_args,
    pin_token_scales_dense, pin_token_scales_uniform, pin_head_scales_per_head,
    pin_head_scales_dense, pin_multi_token_truncation,
    pin_multi_token_causal_dense, pin_multi_token_one_is_decode, pin_ragged_q_truncation,
    pin_ragged_q_sdpa, pin_ragged_q_one_token_is_decode])
def test_decode_pins(orc, pin):
    pin(orc)


# ---------------------------------------------------------------- merge rule

def pin_golden_merge(orc):
    with open(os.path.join(GOLDEN, "merge_worked_examples.json")) as f:
        spec = json.load(f)
    for case in spec["cases"]:
        lb = -math.inf if case["lse_b"] == "-inf" else case["lse_b"]
        o, lse = orc.merge_states(np.array([case["o_a"]]), np.array([case["lse_a"]]),
                                  np.array([case["o_b"]]), np.array([lb]))
        np.testing.assert_allclose(o[0], case["expected_o"], rtol=0, atol=1e-14)
        assert abs(lse[0] - case["expected_lse"]) < 1e-14


def pin_merge_algebra(orc):
    rng = np.random.default_rng(12)
    n, D = 64, 8
    st = [(rng.standard_normal((n, D)), rng.standard_normal(n) * 5) for _ in range(3)]
    (a, la), (b, lb), (c, lc) = st
    ab = orc.merge_states(a, la, b, lb)
    ba = orc.merge_states(b, lb, a, la)
    np.testing.assert_allclose(ab[0], ba[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ab[1], ba[1], rtol=0, atol=1e-13)
    left = orc.merge_states(ab[0], ab[1], c, lc)
    bc = orc.merge_states(b, lb, c, lc)
    right = orc.merge_states(a, la, bc[0], bc[1])
    np.testing.assert_allclose(left[0], right[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(left[1], right[1], rtol=0, atol=1e-12)
    # lse of the merge is the log of the summed weights
    np.testing.assert_allclose(ab[1], np.logaddexp(la, lb), rtol=0, atol=1e-13)
    # empty state is the identity; two empties stay empty without NaN
    e = orc.merge_states(a, la, np.zeros_like(a), np.full(n, -np.inf))
    np.testing.assert_array_equal(e[0], a)
    np.testing.assert_array_equal(e[1], la)
    z = orc.merge_states(np.zeros((2, D)), np.full(2, -np.inf), np.zeros((2, D)), np.full(2, -np.inf))
    assert np.all(z[0] == 0) and np.all(z[1] == -np.inf)


@pytest.mark.parametrize("pin", [pin_golden_merge, pin_merge_algebra])
def test_merge_pins(orc, pin):
    pin(orc)


# ---------------------------------------------------------------- plan coverage definition

def test_golden_coverage():
    with open(os.path.join(GOLDEN, "coverage_worked_example.json")) as f:
        spec = json.load(f)
    got = oracle.expected_coverage(spec["indptr"], spec["num_kv_heads"])
    np.testing.assert_array_equal(got, np.array(spec["expected"]))


def test_golden_token_coverage():
    """Token-level coverage on the hand-worked example: lengths from the
    page counts and last_page_len, each kv head covering tokens 0 .. len-1."""
    with open(os.path.join(GOLDEN, "token_coverage_worked_example.json")) as f:
        spec = json.load(f)
    args = (spec["indptr"], spec["last_page_len"], spec["num_kv_heads"], spec["page_size"])
    np.testing.assert_array_equal(
        oracle.request_lengths(spec["indptr"], spec["last_page_len"], spec["page_size"]),
        spec["lengths"])
    runs = np.array(spec["expected_runs"])
    np.testing.assert_array_equal(oracle.expected_token_intervals(*args), runs)
    want = np.array([(r, h, t) for r, h, a, b in runs for t in range(a, b)])
    np.testing.assert_array_equal(oracle.expected_token_coverage(*args), want)


def test_token_coverage_refines_page_coverage():
    """Independent route on random batches: every covered page position p of
    request i contributes slots 0..15 (last page: 0..last-1) as tokens
    (p - indptr[i]) * 16 + slot; the union equals the token coverage."""
    rng = np.random.default_rng(3)
    for _ in range(20):
        B = int(rng.integers(1, 12))
        pages = rng.integers(0, 6, size=B)
        indptr = np.concatenate([[0], np.cumsum(pages)])
        last = rng.integers(1, 17, size=B)
        Hkv = int(rng.integers(1, 4))
        got = set(map(tuple, oracle.expected_token_coverage(indptr, last, Hkv, 16).tolist()))
        want = set()
        for r, h, p in oracle.expected_coverage(indptr, Hkv).tolist():
            n = last[r] if p == indptr[r + 1] - 1 else 16
            want |= {(r, h, (p - indptr[r]) * 16 + s) for s in range(n)}
        assert got == want


def test_threads_reported(orc):
    assert orc.max_threads() >= 1
