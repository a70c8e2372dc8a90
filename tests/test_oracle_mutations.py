"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that the pins of test_oracle.py catch every one.  This is what makes the
pins worth trusting: each mistake below is the kind a careless restatement
of the method would make."""
import os

import numpy as np
import pytest

import oracle
from tests import test_oracle as T

# (name, text in oracle.c, replacement, pins expected to fail on it)
MUTATIONS = [
    ("gqa head mapping", "const int kvh = h / g;", "const int kvh = h % Hkv;",
     [T.pin_gqa_equals_repeated_mha, T.pin_torch_dense]),
    ("dropped logit scale", "s[t] = sm_scale * acc;", "s[t] = acc;",
     [T.pin_single_key, T.pin_torch_dense, T.pin_brute_force]),
    ("lse without the max", "lse[u] = m + log(den);", "lse[u] = log(den);",
     [T.pin_single_key, T.pin_identical_keys]),
    ("K and V swapped", "kv_offset(page, 0, slot, kvh, d, P, Hkv, D));",
     "kv_offset(page, 1, slot, kvh, d, P, Hkv, D));",
     [T.pin_torch_dense, T.pin_brute_force, T.pin_golden_decode]),
    ("last page read in full", "(int64_t)(np - 1) * P + last_page_len[i]", "(int64_t)np * P",
     [T.pin_padding_never_read, T.pin_golden_decode]),
    ("no max subtraction in the weights", "den += exp(s[t] - m);", "den += exp(s[t]);",
     [T.pin_identical_keys, T.pin_brute_force]),
    ("e4m3 exponent bias 8", "pow(2.0, e - 7)", "pow(2.0, e - 8)",
     [T.pin_e4m3_all_codes, T.pin_e4m3_spec_points]),
    ("e4m3 subnormal scale", "((double)m / 8.0) * pow(2.0, 1 - 7)", "((double)m / 8.0) * pow(2.0, -7)",
     [T.pin_e4m3_all_codes, T.pin_e4m3_spec_points]),
    ("k_scale ignored", "double kd = ks * load_elem", "double kd = load_elem",
     [T.pin_torch_dense, T.pin_token_scales_dense]),
    ("per-token K scale ignored",
     "k_scales ? (double)k_scales[(page * Hkv + kvh) * P + slot] : k_scale;",
     "k_scale;", [T.pin_token_scales_dense]),
    ("per-token scale index transposed",
     "v_scales ? (double)v_scales[(page * Hkv + kvh) * P + slot] : v_scale;",
     "v_scales ? (double)v_scales[(page * P + slot) * Hkv + kvh] : v_scale;",
     [T.pin_token_scales_dense]),
    ("draft token sees the whole draft", "const int64_t visible = len - q_len + qi + 1;",
     "const int64_t visible = len;",
     [T.pin_multi_token_truncation, T.pin_multi_token_causal_dense]),
    ("draft mask off by one", "const int64_t visible = len - q_len + qi + 1;",
     "const int64_t visible = len - q_len + qi;",
     [T.pin_multi_token_truncation, T.pin_multi_token_causal_dense]),
    ("ragged draft mask off by one", "const int64_t visible = len - nq + j + 1;",
     "const int64_t visible = len - nq + j;",
     [T.pin_ragged_q_truncation, T.pin_ragged_q_sdpa]),
    ("ragged drafts all stop at the first", "const int64_t visible = len - nq + j + 1;",
     "const int64_t visible = len - nq + 1;",
     [T.pin_ragged_q_truncation, T.pin_ragged_q_sdpa]),
    ("merge weight of b uses a", "d_b * w_b;", "d_b * w_a;",
     [T.pin_golden_merge, T.pin_merge_algebra, T.pin_split_merge]),
    ("merge sign flipped", "exp(m_b - m_new);", "exp(m_new - m_b);",
     [T.pin_golden_merge, T.pin_merge_algebra]),
]


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, pins):
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
    # the same slip made everywhere the statement occurs
    so = oracle.compile_variant(src.replace(old, new), os.path.join(tmp_path, "mut.so"))
    bad = oracle.Oracle(so)
    for pin in pins:
        with pytest.raises((AssertionError, ValueError)):
            pin(bad)


@pytest.mark.parametrize("axis", ["slot", "page"])
def test_head_scale_broadcast_mistake_is_caught(axis):
    """The per-head oracle broadcasts [num_kv_heads] scales over
    [num_pages, num_kv_heads, page_size]; a broadcast along the wrong axis
    (the scales taken by slot or by page instead of by head) breaks the
    per-head pin."""
    orc = oracle._default()
    args, kh, vh, *_ = T._head_scale_case()
    qb, qc, kb, kc, indptr, ids, last, Hq, Hkv, D, P = args
    num_pages = kb.size // (2 * P * Hkv * D)
    shape = (num_pages, Hkv, P)
    k_by = np.resize(kh, P if axis == "slot" else num_pages).astype(np.float32)
    v_by = np.resize(vh, P if axis == "slot" else num_pages).astype(np.float32)
    if axis == "slot":
        ks = np.broadcast_to(k_by[None, None, :], shape)
        vs = np.broadcast_to(v_by[None, None, :], shape)
    else:
        ks = np.broadcast_to(k_by[:, None, None], shape)
        vs = np.broadcast_to(v_by[:, None, None], shape)
    o, lse = orc.batch_decode_token_scales(*args, ks, vs)
    with pytest.raises(AssertionError):
        T.head_scales_match_per_tensor_per_head(orc, o, lse, args, kh, vh)
