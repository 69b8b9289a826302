"""Pins for the oracle's paged attention, split-KV partials and LSE combine.

Operation: InfiniLM PR #585, section "概述 / Summary", item 1 (pure decode
through a paged split-KV kernel over the BSHD cache) and item 4 (verify of
k+1 tokens in one forward, causal among the draft tokens).  The pages print no
numbers for it, so every pin is mathematical: brute force against a library
routine and an independent scalar loop on tiny contiguous caches, invariance
to the physical block order, split = unsplit, and closed forms.
"""

import math

import numpy as np
import pytest
import torch

from oracle import (bf16_bits_to_f64, f64_to_bf16_bits, lse_combine,
                    paged_attention, paged_attention_splits, split_page_ranges)


def _bits(x):
    return f64_to_bf16_bits(np.asarray(x, np.float64))


def _case(seed, B=3, q_len=1, Hq=4, Hkv=2, D=16, bs=4, lens=(1, 7, 13), perm=True, extra_blocks=2):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int64)
    pages = [-(-int(n) // bs) for n in lens]
    NB = sum(pages) + extra_blocks
    ids = rng.permutation(NB) if perm else np.arange(NB)
    bt = np.full((B, max(pages)), -1, np.int64)
    c = 0
    for b, p in enumerate(pages):
        bt[b, :p] = ids[c:c + p]
        c += p
    q = _bits(rng.standard_normal((B, q_len, Hq, D)))
    kc = _bits(rng.standard_normal((NB, bs, Hkv, D)))
    vc = _bits(rng.standard_normal((NB, bs, Hkv, D)))
    return q, kc, vc, bt, lens, bs


def _contiguous_kv(kc, vc, bt_row, n, bs):
    """Keys 0..n-1 of one sequence as a dense [n, Hkv, D] array (plain loop)."""
    K = np.stack([kc[bt_row[i // bs], i % bs] for i in range(n)]) if n else np.zeros((0,) + kc.shape[2:], kc.dtype)
    V = np.stack([vc[bt_row[i // bs], i % bs] for i in range(n)]) if n else np.zeros((0,) + vc.shape[2:], vc.dtype)
    return bf16_bits_to_f64(K), bf16_bits_to_f64(V)


@pytest.mark.parametrize("q_len", [1, 3])
def test_matches_torch_sdpa_on_contiguous_cache(q_len):
    # identity block table: the paged cache is a plain contiguous KV array
    q, kc, vc, bt, lens, bs = _case(10, q_len=q_len, lens=(5, 9, 16), perm=False, extra_blocks=0)
    out, lse = paged_attention(q, kc, vc, bt, lens, bs, q_len=q_len)
    B, T, Hq, D = q.shape
    Hkv = kc.shape[2]
    for b in range(B):
        n = int(lens[b])
        K, V = _contiguous_kv(kc, vc, bt[b], n, bs)            # [n, Hkv, D]
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)   # [Hq, n, D]
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        Q = torch.from_numpy(bf16_bits_to_f64(q[b])).permute(1, 0, 2)              # [Hq, T, D]
        # query t may see keys j <= n - T + t
        mask = torch.arange(n)[None, :] <= (n - T + torch.arange(T))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, Kt, Vt, attn_mask=mask)
        assert np.allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_matches_scalar_loop_brute_force():
    q, kc, vc, bt, lens, bs = _case(11, B=2, lens=(3, 6), Hq=2, Hkv=1, D=4)
    out, lse = paged_attention(q, kc, vc, bt, lens, bs)
    for b in range(2):
        n = int(lens[b])
        for h in range(2):
            qv = bf16_bits_to_f64(q[b, 0, h])
            scores = []
            for j in range(n):
                kk = bf16_bits_to_f64(kc[bt[b, j // bs], j % bs, 0])
                scores.append(sum(qv[d] * kk[d] for d in range(4)) / 2.0)   # D^-1/2 = 1/2
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            acc = [0.0] * 4
            for j in range(n):
                vv = bf16_bits_to_f64(vc[bt[b, j // bs], j % bs, 0])
                for d in range(4):
                    acc[d] += w[j] * vv[d]
            Z = sum(w)
            assert np.allclose(out[b, 0, h], [a / Z for a in acc], rtol=1e-13, atol=1e-14)
            assert math.isclose(lse[b, 0, h], m + math.log(Z), rel_tol=1e-13)


def test_block_permutation_invariance_bit_identical():
    q, kc, vc, bt, lens, bs = _case(12, lens=(4, 11, 17))
    out, lse = paged_attention(q, kc, vc, bt, lens, bs)
    rng = np.random.default_rng(99)
    NB = kc.shape[0]
    perm = rng.permutation(NB)             # new physical id of old block i is perm[i]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    out2, lse2 = paged_attention(q, kc2, vc2, bt2, lens, bs)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("S,C", [(1, 100), (2, 2), (3, 1), (4, 3), (8, 1), (5, 5)])
@pytest.mark.parametrize("q_len", [1, 4])
def test_split_equals_unsplit(S, C, q_len):
    q, kc, vc, bt, lens, bs = _case(13, q_len=q_len, lens=(4, 11, 30))
    out, lse = paged_attention(q, kc, vc, bt, lens, bs, q_len=q_len)
    o, l = paged_attention_splits(q, kc, vc, bt, lens, bs, S, C, q_len=q_len)
    out2, lse2 = lse_combine(o, l)
    assert np.allclose(out2, out, rtol=0, atol=1e-12)
    assert np.allclose(lse2, lse, rtol=0, atol=1e-12)


def test_split_ranges_cover_every_page_once():
    for P in [0, 1, 5, 16, 33]:
        for S in [1, 2, 3, 7]:
            for C in [1, 2, 5, 40]:
                seen = []
                for p0, p1 in split_page_ranges(P, S, C):
                    assert 0 <= p0 <= p1 <= P
                    seen.extend(range(p0, p1))
                assert seen == list(range(P))


def test_equal_keys_closed_form():
    # every key equal -> uniform weights: out = mean(V), lse = s + ln(n)
    q, kc, vc, bt, lens, bs = _case(14, B=1, lens=(10,))
    kc[:] = kc[0, 0]
    out, lse = paged_attention(q, kc, vc, bt, lens, bs)
    K, V = _contiguous_kv(kc, vc, bt[0], 10, bs)
    D = q.shape[-1]
    for h in range(q.shape[2]):
        g = h // (q.shape[2] // kc.shape[2])
        s = bf16_bits_to_f64(q[0, 0, h]) @ K[0, g] / math.sqrt(D)
        assert np.allclose(out[0, 0, h], V[:, g].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert math.isclose(lse[0, 0, h], s + math.log(10), rel_tol=1e-13, abs_tol=1e-13)


def test_single_key_returns_v0_exactly():
    q, kc, vc, bt, lens, bs = _case(15, B=1, lens=(1,))
    out, lse = paged_attention(q, kc, vc, bt, lens, bs)
    V0 = bf16_bits_to_f64(vc[bt[0, 0], 0])
    G = q.shape[2] // kc.shape[2]
    for h in range(q.shape[2]):
        assert np.array_equal(out[0, 0, h], V0[h // G])


def test_empty_sequence_gives_zero_and_minus_inf():
    q, kc, vc, bt, lens, bs = _case(16, B=2, lens=(0, 5))
    out, lse = paged_attention(q, kc, vc, bt, lens, bs)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1]))


def test_verify_qlen1_equals_decode_and_token_t_equals_shorter_decode():
    q, kc, vc, bt, lens, bs = _case(17, q_len=5, lens=(9, 14, 22))
    out, lse = paged_attention(q, kc, vc, bt, lens, bs, q_len=5)
    for t in range(5):
        lens_t = lens - 5 + t + 1
        o1, l1 = paged_attention(q[:, t:t + 1], kc, vc, bt, lens_t, bs, q_len=1)
        assert np.array_equal(o1[:, 0], out[:, t]) and np.array_equal(l1[:, 0], lse[:, t])


def test_gqa_with_duplicated_kv_heads_equals_mha():
    q, kc, vc, bt, lens, bs = _case(18, B=2, Hq=4, Hkv=2, lens=(6, 13))
    out, lse = paged_attention(q, kc, vc, bt, lens, bs)
    kc4 = np.repeat(kc, 2, axis=2)       # head h of the MHA cache = kv head h // 2
    vc4 = np.repeat(vc, 2, axis=2)
    out4, lse4 = paged_attention(q, kc4, vc4, bt, lens, bs)
    # equal up to BLAS summation order (grouped rows vs one row per head)
    assert np.allclose(out, out4, rtol=0, atol=1e-13) and np.allclose(lse, lse4, rtol=0, atol=1e-13)


def test_lse_combine_closed_forms():
    o = np.array([[1.0, 2.0], [3.0, 6.0]])[None]          # [1, S=2, D=2]
    out, l = lse_combine(o, np.array([[0.0, 0.0]]))
    assert np.allclose(out, [[2.0, 4.0]]) and np.isclose(l[0], math.log(2.0))
    out, l = lse_combine(o, np.array([[0.0, -np.inf]]))
    assert np.array_equal(out, [[1.0, 2.0]]) and l[0] == 0.0
    out, l = lse_combine(o, np.array([[-np.inf, -np.inf]]))
    assert np.array_equal(out, [[0.0, 0.0]]) and np.isneginf(l[0])
    # weights exp(lse): lse = (ln 1, ln 3) -> out = (1*o0 + 3*o1)/4
    out, l = lse_combine(o, np.array([[0.0, math.log(3.0)]]))
    assert np.allclose(out, [[2.5, 5.0]]) and np.isclose(l[0], math.log(4.0))
