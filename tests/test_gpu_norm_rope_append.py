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
