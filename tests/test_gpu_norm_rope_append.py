"""GPU parity of pkvqk_norm_rope_append against the fp64 oracle.

Operation: InfiniLM PR #585, section "概述 / Summary", item 2 (fused per-head
RMSNorm + full-rotary RoPE) and item 1 (append into the BSHD paged cache).
Bar: q_hat / k_hat within 1 bf16 ulp of the oracle's correctly rounded value,
v rows and every untouched cache byte bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_qk_gb300 import workloads
from tests._parity import ULP_TOL, bf16_ulp_distance, bits

pytestmark = pytest.mark.gpu


def _run_and_check(lib, p, q=None, k=None, v=None, k_cache=None, v_cache=None, slots=None):
    """Run the GPU op on (views of) the problem's tensors and compare with the oracle."""
    q = p.q.clone() if q is None else q
    k = p.k if k is None else k
    v = p.v if v is None else v
    k_cache = p.k_cache.clone() if k_cache is None else k_cache
    v_cache = p.v_cache.clone() if v_cache is None else v_cache
    slots = p.slot_mapping if slots is None else slots
    q_in, k_in, v_in = bits(q), bits(k), bits(v)
    kc_in, vc_in = bits(k_cache), bits(v_cache)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.norm_rope_append(q, k, v, p.positions, slots, p.gamma_q, p.gamma_k, p.theta, p.eps,
                         k_cache, v_cache, status_flags=flags)
    torch.cuda.synchronize()
    qh, kc, vc, _, _ = oracle.norm_rope_append(
        q_in, k_in, v_in, p.positions.cpu().numpy(), slots.cpu().numpy(),
        bits(p.gamma_q), bits(p.gamma_k), p.theta, p.eps, kc_in, vc_in, p.block_size)
    dq = bf16_ulp_distance(bits(q), qh)
    assert dq.max() <= ULP_TOL, f"q_hat off by {dq.max()} ulp"
    dk = bf16_ulp_distance(bits(k_cache), kc)
    assert dk.max() <= ULP_TOL, f"k cache off by {dk.max()} ulp"
    # only the appended slots may differ from the input cache
    assert np.array_equal(bits(v_cache), vc), "v cache not bit-exact"
    changed = np.any(bits(k_cache) != kc_in, axis=(2, 3))
    touched = np.any(kc != kc_in, axis=(2, 3))
    assert not np.any(changed & ~touched), "k cache written outside the mapped slots"
    return flags.item(), dq, dk


def test_decode_tiny(lib):
    p = workloads.decode_tiny(device="cuda")
    f, dq, dk = _run_and_check(lib, p)
    assert f == 0
    # most values are bit-exact; 1-ulp differences only at near-ties
    assert (dq == 0).mean() > 0.99


def test_verify_tokens_and_long_positions(lib):
    # 32 sequences x 5 tokens at positions up to ~8200, plus long positions
    p = workloads.verify_causal(device="cuda")
    _run_and_check(lib, p)
    big = p.positions.clone()
    big[:] = torch.arange(32767 - big.numel() + 1, 32768, device="cuda")
    p.positions = big
    _run_and_check(lib, p)


def test_gqa8_heads(lib):
    p = workloads.make_problem("gqa8_small", 32, 4, 128, 16, [17, 40, 1, 300], 1, 64, 901, "cuda")
    _run_and_check(lib, p)


def test_strided_qkv_views_and_interleaved_cache(lib):
    """q/k/v as views of one fused qkv buffer; K/V as views of an interleaved
    (num_blocks, 2, block_size, Hkv, D) allocation (no copy)."""
    p = workloads.make_problem("strided", 16, 8, 128, 16, [5, 33, 100], 1, 24, 902, "cuda")
    T, Hq, Hkv, D = p.T, p.Hq, p.Hkv, p.D
    qkv = torch.empty(T, Hq + 2 * Hkv, D, dtype=torch.bfloat16, device="cuda")
    qkv[:, :Hq] = p.q
    qkv[:, Hq:Hq + Hkv] = p.k
    qkv[:, Hq + Hkv:] = p.v
    q, k, v = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv], qkv[:, Hq + Hkv:]
    both = torch.stack([p.k_cache, p.v_cache], dim=1).contiguous()   # [NB, 2, bs, Hkv, D]
    kc, vc = both[:, 0], both[:, 1]
    _run_and_check(lib, p, q=q, k=k, v=v, k_cache=kc, v_cache=vc)
    # v part of qkv unchanged, k part unchanged (only q is written in place)
    assert torch.equal(qkv[:, Hq:Hq + Hkv], p.k) and torch.equal(qkv[:, Hq + Hkv:], p.v)


def test_padding_and_bad_slots(lib):
    p = workloads.make_problem("slots", 16, 8, 128, 16, [3, 20, 47, 9], 1, 12, 903, "cuda")
    slots = p.slot_mapping.clone()
    slots[1] = -1                                   # padding token: nothing written
    slots[2] = p.num_blocks * p.block_size + 5      # out of range: skipped + flagged
    f, _, _ = _run_and_check(lib, p, slots=slots)
    assert f & lib.FLAG_BAD_SLOT


def test_block_size_256(lib):
    p = workloads.make_problem("bs256", 16, 8, 128, 256, [1, 255, 256, 700], 1, 8, 904, "cuda")
    _run_and_check(lib, p)


def test_cancellation_many_tokens_long_positions(lib):
    """4096 tokens x 24 heads at positions up to 65535: the rotation
    a_i cos - a_{i+D/2} sin lands near zero for some elements, where a plain
    fp32 rotation is many ulps off; the bar stays 1 ulp."""
    T, Hq, Hkv, D, bs, NB = 4096, 16, 8, 128, 16, 8
    g = torch.Generator(device="cuda").manual_seed(912)
    p = workloads.make_problem("cancel", Hq, Hkv, D, bs, [1], 1, NB, 912, "cuda")
    p.q = torch.randn(T, Hq, D, generator=g, device="cuda").to(torch.bfloat16)
    p.k = torch.randn(T, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    p.v = torch.randn(T, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    p.positions = torch.randint(0, 65536, (T,), generator=g, device="cuda")
    slots = torch.full((T,), -1, dtype=torch.int64, device="cuda")
    slots[:NB * bs] = torch.randperm(NB * bs, generator=g, device="cuda")
    _, dq, dk = _run_and_check(lib, p, slots=slots)
    assert dq.max() <= 1


def test_zero_tokens_is_noop(lib):
    p = workloads.decode_tiny(device="cuda")
    kc = p.k_cache.clone()
    lib.norm_rope_append(p.q[:0], p.k[:0], p.v[:0], p.positions[:0], p.slot_mapping[:0],
                         p.gamma_q, p.gamma_k, p.theta, p.eps, kc, p.v_cache)
    torch.cuda.synchronize()
    assert torch.equal(kc, p.k_cache)


def _append_both(lib, p, positions, table_positions, slots=None):
    """The same inputs through pkvqk_norm_rope_append and, with a rotary table
    of table_positions positions, pkvqk_norm_rope_append_cached."""
    slots = p.slot_mapping if slots is None else slots
    table = torch.empty(max(lib.rope_table_bytes(table_positions), 16), dtype=torch.uint8,
                        device="cuda")
    lib.rope_table_build(table, table_positions, p.theta)
    outs = []
    for cached in (False, True):
        q, kc, vc = p.q.clone(), p.k_cache.clone(), p.v_cache.clone()
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        if cached:
            lib.norm_rope_append_cached(q, p.k, p.v, positions, slots, p.gamma_q, p.gamma_k,
                                        p.theta, p.eps, kc, vc, table, table_positions,
                                        status_flags=flags)
        else:
            lib.norm_rope_append(q, p.k, p.v, positions, slots, p.gamma_q, p.gamma_k, p.theta,
                                 p.eps, kc, vc, status_flags=flags)
        torch.cuda.synchronize()
        outs.append((q, kc, vc, flags.item()))
    return outs


@pytest.mark.parametrize("T", [5, 2048])
def test_rope_table_gives_the_same_bits(lib, T):
    """Angles from the table are the ones the kernel computes per token: q, the
    cache and the flags are bit-identical, for positions inside the table, past
    its end (computed per token) and at its edges; few tokens (one half-warp per
    vector) and many (the narrow-CTA form)."""
    Hq, Hkv, D, bs, NB = 16, 8, 128, 16, 160
    g = torch.Generator(device="cuda").manual_seed(931 + T)
    p = workloads.make_problem("table", Hq, Hkv, D, bs, [1], 1, NB, 931, "cuda")
    p.q = torch.randn(T, Hq, D, generator=g, device="cuda").to(torch.bfloat16)
    p.k = torch.randn(T, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    p.v = torch.randn(T, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    P = 40960
    pos = torch.randint(0, 65536, (T,), generator=g, device="cuda")
    edges = torch.tensor([0, 1, P - 1, P, P + 1, 65535, 32767], device="cuda")
    pos[:min(T, edges.numel())] = edges[:min(T, edges.numel())]
    slots = torch.full((T,), -1, dtype=torch.int64, device="cuda")
    n = min(T, NB * bs)
    slots[:n] = torch.randperm(NB * bs, generator=g, device="cuda")[:n]
    (q0, k0, v0, f0), (q1, k1, v1, f1) = _append_both(lib, p, pos, P, slots)
    assert torch.equal(bits_t(q0), bits_t(q1))
    assert torch.equal(bits_t(k0), bits_t(k1)) and torch.equal(bits_t(v0), bits_t(v1))
    assert f0 == f1 == 0


def test_rope_table_path_matches_oracle(lib):
    # the cached path against the fp64 oracle at the 1-ulp bar (verify tokens at
    # positions up to ~8200, all inside a 16384-position table)
    p = workloads.verify_causal(device="cuda")
    (_, _, _, _), (q1, kc1, vc1, f1) = _append_both(lib, p, p.positions, 16384)
    qh, kc, vc, _, _ = oracle.norm_rope_append(
        bits(p.q), bits(p.k), bits(p.v), p.positions.cpu().numpy(),
        p.slot_mapping.cpu().numpy(), bits(p.gamma_q), bits(p.gamma_k), p.theta, p.eps,
        bits(p.k_cache), bits(p.v_cache), p.block_size)
    assert bf16_ulp_distance(bits(q1), qh).max() <= ULP_TOL
    assert bf16_ulp_distance(bits(kc1), kc).max() <= ULP_TOL
    assert np.array_equal(bits(vc1), vc)
    assert f1 == 0


def bits_t(t):
    return t.view(torch.int16)
