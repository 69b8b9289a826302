"""Helpers shared by the GPU parity tests: moving seeded inputs to the oracle
and comparing the CUDA path's outputs with the oracle's.

Tolerances (written here once, used by every parity test):
  * slot / index placement and v rows: bit-exact;
  * q_hat and k_hat: within 1 bf16 ulp of the oracle's correctly rounded
    value (the kernel computes in fp32 and rounds once);
  * attention output: max |gpu - oracle| <= 2e-2 and mean <= 2e-3 against
    the float64 oracle (the bf16 output itself carries up to 2^-9 relative
    rounding);
  * lse: |gpu - oracle| <= 1e-3 (fp32 scores of bf16 products, fp32 sums).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
ULP_TOL = 1


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def widen(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits(t))


def compact_cache(problem, seqs, k_cache=None, v_cache=None):
    """Gather the blocks of the sequences in `seqs` (torch indexing on the
    device), returning (k_bits, v_bits, block_table_rows, seq_lens) for the
    oracle with block ids remapped to the compact cache.  The oracle's result
    does not depend on physical block ids (pinned by the permutation test)."""
    k_cache = problem.k_cache if k_cache is None else k_cache
    v_cache = problem.v_cache if v_cache is None else v_cache
    bt = problem.block_tables_host
    bs = problem.block_size
    rows, ids = [], []
    for b in seqs:
        P = -(-int(problem.seq_lens_host[b]) // bs)
        rows.append(list(range(len(ids), len(ids) + P)))
        ids.extend(int(x) for x in bt[b, :P])
    width = max(1, max((len(r) for r in rows), default=1))
    table = np.full((len(seqs), width), -1, np.int64)
    for i, r in enumerate(rows):
        table[i, :len(r)] = r
    if not ids:
        ids = [0]
    idx = torch.tensor(ids, dtype=torch.long, device=k_cache.device)
    kb = bits(k_cache.index_select(0, idx))
    vb = bits(v_cache.index_select(0, idx))
    return kb, vb, table, problem.seq_lens_host[list(seqs)]


def oracle_attention(problem, q_bits, seqs=None, k_cache=None, v_cache=None, scale=None):
    """Oracle output/lse for the sequences in `seqs` (all if None).

    q_bits: uint16 [B*q_len, Hq, D].  Returns (out [n, q_len, Hq, D], lse [n, q_len, Hq]).
    """
    B, T = problem.B, problem.q_len
    if seqs is None:
        seqs = list(range(B))
    kb, vb, table, lens = compact_cache(problem, seqs, k_cache, v_cache)
    q = q_bits.reshape(B, T, problem.Hq, problem.D)[list(seqs)]
    return oracle.paged_attention(q, kb, vb, table, lens, problem.block_size, q_len=T, scale=scale)


def assert_attention_close(gpu_out_bits, ref_out, gpu_lse=None, ref_lse=None, what=""):
    got = oracle.bf16_bits_to_f64(gpu_out_bits)
    assert got.shape == ref_out.shape, (got.shape, ref_out.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref_out)
    assert err.max() <= OUT_MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    if gpu_lse is not None:
        g = np.asarray(gpu_lse, np.float64)
        r = np.asarray(ref_lse, np.float64)
        both_inf = np.isneginf(g) & np.isneginf(r)
        assert np.array_equal(np.isneginf(g), np.isneginf(r)), f"{what}: -inf lse pattern differs"
        d = np.abs(np.where(both_inf, 0.0, g - r))
        assert d.max() <= LSE_ABS, f"{what}: lse err {d.max():.3e}"
    return err.max(), err.mean()
