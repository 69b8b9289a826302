"""The seeded input generators (CPU): the same seed gives the same inputs,
and every problem is a valid paged-cache state -- each sequence's pages are
distinct physical blocks, unused table entries are -1, and every new token's
slot is where the block table places its position.  All parity tests and the
benchmark read their inputs from these generators."""

import numpy as np
import torch

from paged_kv_cache_qk_gb300 import workloads

SMALL = {
    "decode_tiny": lambda: workloads.decode_tiny(),
    "decode_uniform": lambda: workloads.decode_uniform(3, 100),
    "verify_like": lambda: workloads.make_problem("v", 16, 8, 128, 16, [40, 77, 5], 5, 12, 99),
    "gqa8_like": lambda: workloads.make_problem("g", 32, 4, 128, 16, [1, 300, 17], 1, 40, 98),
    "bs256": lambda: workloads.make_problem("b", 16, 8, 128, 256, [700, 3], 1, 9, 97),
    "chunked": lambda: workloads.chunked_prefill(batch=2, chunk=64, lo=0, hi=200),
    "varlen": lambda: workloads.varlen_prefill(batch=3, lo=5, hi=90),
}


def _tensors(p):
    names = ("q", "k", "v", "gamma_q", "gamma_k", "positions", "slot_mapping", "k_cache",
             "v_cache", "block_tables", "seq_lens")
    return {n: getattr(p, n) for n in names}


def test_same_seed_same_inputs():
    for name, mk in SMALL.items():
        a, b = _tensors(mk()), _tensors(mk())
        for n in a:
            assert torch.equal(a[n], b[n]), (name, n)


def test_problems_are_valid_paged_cache_states():
    for name, mk in SMALL.items():
        p = mk()
        bs = p.block_size
        bt = p.block_tables.numpy()
        lens = p.seq_lens.numpy().astype(np.int64)
        assert np.array_equal(lens, p.seq_lens_host)
        used = []
        for b in range(p.B):
            n_pages = -(-int(lens[b]) // bs)
            row = bt[b]
            assert np.all((row[:n_pages] >= 0) & (row[:n_pages] < p.num_blocks)), name
            assert np.all(row[n_pages:] == -1), name
            used.extend(row[:n_pages].tolist())
        assert len(used) == len(set(used)), f"{name}: a physical block is shared"
        # new tokens: positions seq_len - q_len_b + t, slots in the sequence's own pages
        q_lens = (p.q_lens_host if p.q_lens_host is not None
                  else np.full(p.B, p.q_len, np.int64))
        pos = p.positions.numpy()
        slots = p.slot_mapping.numpy()
        t0 = 0
        for b in range(p.B):
            for t in range(int(q_lens[b])):
                n = int(lens[b] - q_lens[b] + t)
                assert pos[t0 + t] == n, name
                assert slots[t0 + t] == int(bt[b][n // bs]) * bs + n % bs, name
            t0 += int(q_lens[b])
        assert t0 == p.T == p.q.shape[0] == p.k.shape[0] == p.v.shape[0]
        if p.cu_seqlens is not None:
            assert np.array_equal(p.cu_seqlens.numpy(), np.concatenate([[0], np.cumsum(q_lens)]))
        # bf16 everywhere the kernels read bf16; gains near 1
        for n in ("q", "k", "v", "k_cache", "v_cache", "gamma_q", "gamma_k"):
            assert getattr(p, n).dtype == torch.bfloat16, (name, n)
        g = p.gamma_q.float()
        assert (g - 1).abs().max() < 1.0 and g.std() > 0.01


def test_configuration_seeds_follow_the_base_seed():
    # the tiny configuration draws from BASE_SEED (the benchmark seed 714); the
    # uniform sweep from BASE_SEED + 1; another seed gives other values
    a = workloads.decode_tiny()
    again = workloads.make_problem("decode_tiny", 16, 8, 128, 16, a.seq_lens_host, 1, 64,
                                   workloads.BASE_SEED, table_width=16)
    assert workloads.BASE_SEED == 714
    for n in ("q", "k", "v", "k_cache", "block_tables", "slot_mapping"):
        assert torch.equal(getattr(a, n), getattr(again, n)), n
    other = workloads.make_problem("decode_tiny", 16, 8, 128, 16, a.seq_lens_host, 1, 64,
                                   workloads.BASE_SEED + 1, table_width=16)
    assert not torch.equal(a.q, other.q)
    u = workloads.decode_uniform(2, 64)
    u_again = workloads.make_problem(u.name, 16, 8, 128, 16, u.seq_lens_host, 1, u.num_blocks,
                                     workloads.BASE_SEED + 1)
    assert torch.equal(u.q, u_again.q) and torch.equal(u.block_tables, u_again.block_tables)
