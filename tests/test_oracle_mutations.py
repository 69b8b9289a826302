"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in an oracle function (a wrong RoPE pairing or
sign, sum instead of mean, a missing gain, a wrong softmax scale, a wrong GQA
head map, an off-by-one causal limit, an unweighted combine, a split
partition that drops the remainder, truncating bf16 rounding) and re-runs
the pins that should notice it; every one must fail.  The mistakes live only
in this test, on the CPU.
"""


import numpy as np

import oracle.reference as ref
from tests import test_oracle_attention as ta
from tests import test_oracle_bf16 as tb
from tests import test_oracle_norm_rope as tn


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


# ------------------------------------------------------------- mutations

def rope_interleaved(x, pos, theta):
    # GPT-J pairing (2i, 2i+1) instead of neox (i, i + D/2)
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    i = np.arange(D // 2, dtype=np.float64)
    ang = np.asarray(pos, np.float64)[..., None] * np.float64(theta) ** (-2.0 * i / D)
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return out


def rope_wrong_sign(x, pos, theta):
    return ref.rope_neox(x, -np.asarray(pos, np.float64), theta)


def rope_wrong_freq(x, pos, theta):
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    i = np.arange(D // 2, dtype=np.float64)
    ang = np.asarray(pos, np.float64)[..., None] * np.float64(theta) ** (-i / D)   # 2 dropped
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rms_sum(x, gamma, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * gamma


def rms_no_gain(x, gamma, eps):
    return ref.rms_norm(x, np.ones_like(np.asarray(gamma, np.float64)), eps)


def bf16_truncate(x):
    x32 = np.asarray(x, np.float64).astype(np.float32)
    return (x32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def combine_unweighted(o, lse):
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    fin = np.isfinite(lse)
    n = np.maximum(fin.sum(axis=-1, keepdims=True), 1)
    out = (np.where(fin[..., None], o, 0.0)).sum(axis=-2) / n
    return out, lse.max(axis=-1)


def ranges_drop_remainder(num_pages, num_splits, chunk_pages):
    out = []
    for j in range(num_splits):
        p0 = min(j * chunk_pages, num_pages)
        p1 = min((j + 1) * chunk_pages, num_pages)
        out.append((p0, max(p0, p1)))
    return out


# --------------------------------------------------------------- the cases

def test_rope_mistakes_are_caught(monkeypatch):
    for bad in (rope_interleaved, rope_wrong_sign, rope_wrong_freq):
        monkeypatch.setattr(tn, "rope_neox", bad)
        caught = [_fails(tn.test_rope_hand_example_pairs_and_frequencies),
                  _fails(tn.test_rope_golden),
                  _fails(tn.test_rope_equals_complex_rotation)]
        assert any(caught), bad.__name__


def test_rmsnorm_mistakes_are_caught(monkeypatch):
    for bad in (rms_sum, rms_no_gain):
        monkeypatch.setattr(tn, "rms_norm", bad)
        caught = [_fails(tn.test_rmsnorm_hand_example), _fails(tn.test_rmsnorm_golden)]
        assert any(caught), bad.__name__


def test_bf16_truncation_is_caught(monkeypatch):
    monkeypatch.setattr(tb, "f64_to_bf16_bits", bf16_truncate)
    assert _fails(tb.test_ties_go_to_even) or _fails(tb.test_matches_torch_cast_on_float32_inputs)


def test_wrong_softmax_scale_is_caught(monkeypatch):
    orig = ref._softmax_attend
    monkeypatch.setattr(ref, "_softmax_attend", lambda q, K, V, scale: orig(q, K, V, scale * 2.0))
    assert _fails(ta.test_matches_scalar_loop_brute_force)
    assert _fails(ta.test_matches_torch_sdpa_on_contiguous_cache, 1)


def test_wrong_gqa_head_map_is_caught(monkeypatch):
    # q head h reading kv head h % Hkv instead of h // G
    def attention_bad_map(q, k_cache, v_cache, block_tables, seq_lens, block_size, q_len=1,
                          scale=None, seqs=None):
        Hq, Hkv = q.shape[2], k_cache.shape[2]
        perm = np.array([h % Hkv for h in range(Hq)])
        G = Hq // Hkv
        # present the same result layout: regroup q so that group g holds heads h % Hkv == g
        order = np.argsort(perm, kind="stable")
        out, lse = ref.paged_attention(q[:, :, order], k_cache, v_cache, block_tables, seq_lens,
                                       block_size, q_len, scale, seqs)
        inv = np.argsort(order)
        return out[:, :, inv], lse[:, :, inv]
    monkeypatch.setattr(ta, "paged_attention", attention_bad_map)
    assert _fails(ta.test_matches_torch_sdpa_on_contiguous_cache, 1)


def test_causal_off_by_one_is_caught(monkeypatch):
    # verify query t seeing one key fewer than it should
    def attention_short(q, k_cache, v_cache, block_tables, seq_lens, block_size, q_len=1,
                        scale=None, seqs=None):
        if q_len == 1:
            return ref.paged_attention(q, k_cache, v_cache, block_tables, seq_lens, block_size,
                                       q_len, scale, seqs)
        return ref.paged_attention(q, k_cache, v_cache, block_tables,
                                   np.asarray(seq_lens) - 1, block_size, q_len, scale, seqs)
    monkeypatch.setattr(ta, "paged_attention", attention_short)
    assert _fails(ta.test_matches_torch_sdpa_on_contiguous_cache, 3)


def test_unweighted_combine_is_caught(monkeypatch):
    monkeypatch.setattr(ta, "lse_combine", combine_unweighted)
    assert _fails(ta.test_lse_combine_closed_forms)
    assert _fails(ta.test_split_equals_unsplit, 4, 3, 1)


def test_partition_dropping_the_remainder_is_caught(monkeypatch):
    monkeypatch.setattr(ta, "split_page_ranges", ranges_drop_remainder)
    assert _fails(ta.test_split_ranges_cover_every_page_once)
    monkeypatch.setattr(ref, "split_page_ranges", ranges_drop_remainder)
    assert _fails(ta.test_split_equals_unsplit, 2, 2, 1)


def test_append_to_wrong_slot_is_caught(monkeypatch):
    orig = ref.norm_rope_append

    def append_shifted(q, k, v, positions, slot_mapping, *rest):
        return orig(q, k, v, positions, np.asarray(slot_mapping) + 1, *rest)
    monkeypatch.setattr(tn, "norm_rope_append", append_shifted)
    assert _fails(tn.test_append_places_exactly_the_mapped_slots)
