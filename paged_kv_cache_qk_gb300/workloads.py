"""Seeded synthetic inputs for the paged decode-attention step.

This module only draws inputs; it holds none of the method's arithmetic (no
norm, rotation, attention or combine).  Both the CUDA path's tests/bench and
the CPU oracle consume what it returns.

Shapes follow the Qwen3 attention layouts used by the serving pages (InfiniLM
PR #585, Qwen3-0.6B / 1.7B; InfiniLM issue #498, Qwen3-30B-A3B with
``--block-size`` and ``--num-blocks``):

* ``decode_tiny``       16q/8kv, D=128, batch 4, seq_len ~ U[1, 256], a random
                        permutation of 64 physical blocks of 16 slots.
* ``decode_uniform``    16q/8kv, D=128, batch B, every context = ctx,
                        num_blocks = B * ctx / 16, shuffled block ids.
* ``decode_long``       16q/8kv, D=128, batch 8, context 32768.
* ``decode_gqa8``       32q/4kv (group 8), D=128, batch 64, contexts
                        log-uniform in [256, 16384], cache = 120% of the
                        pages needed, shuffled block ids.
* ``verify_causal``     16q/8kv, D=128, batch 32, 5 query tokens per sequence
                        (k = 4 draft tokens + 1), prior context U[2048, 8192].
* ``varlen_prefill``    16q/8kv, D=128, batch 16 fresh prompts of U[128, 2048]
                        tokens each, packed back to back (varlen).
* ``chunked_prefill``   16q/8kv, D=128, batch 8, a chunk of 512 new tokens per
                        sequence after a prior context U[0, 6144] (the chunks
                        of a ~6.5k-token prompt, the size the pages inject in
                        their decode-stall workload).

Every tensor is drawn from a generator seeded per problem.  Host-side values
that a scheduler knows without touching the device (sequence lengths, block
assignment, max length) are drawn with numpy on the host; bulk values (q, k, v,
the cache contents) are drawn with a torch generator on the target device so
multi-GB caches are produced in place.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

BASE_SEED = 714


@dataclasses.dataclass
class Problem:
    name: str
    Hq: int
    Hkv: int
    D: int
    block_size: int
    q_len: int
    seq_lens_host: np.ndarray          # int64 [B], counting the q_len new tokens
    block_tables_host: np.ndarray      # int32 [B, maxP]
    num_blocks: int
    theta: float
    eps: float
    # device (or CPU) tensors
    q: torch.Tensor                    # bf16 [B*q_len, Hq, D]
    k: torch.Tensor                    # bf16 [B*q_len, Hkv, D]
    v: torch.Tensor                    # bf16 [B*q_len, Hkv, D]
    gamma_q: torch.Tensor              # bf16 [D]
    gamma_k: torch.Tensor              # bf16 [D]
    positions: torch.Tensor            # int64 [B*q_len]
    slot_mapping: torch.Tensor         # int64 [B*q_len]
    k_cache: torch.Tensor              # bf16 [NB, bs, Hkv, D]
    v_cache: torch.Tensor              # bf16 [NB, bs, Hkv, D]
    block_tables: torch.Tensor         # int32 [B, maxP]
    seq_lens: torch.Tensor             # int32 [B]
    # varlen problems only: new tokens per sequence, and their row offsets
    q_lens_host: np.ndarray | None = None      # int64 [B]
    cu_seqlens: torch.Tensor | None = None     # int32 [B + 1]

    @property
    def B(self) -> int:
        return int(self.seq_lens_host.shape[0])

    @property
    def T(self) -> int:
        if self.q_lens_host is not None:
            return int(self.q_lens_host.sum())
        return self.B * self.q_len

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens_host.max()) if self.B else 0

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens_host.sum())


def _pages(n: int, bs: int) -> int:
    return -(-int(n) // bs)


def make_problem(name, Hq, Hkv, D, block_size, seq_lens, q_len, num_blocks,
                 seed, device="cpu", block_perm=True, table_width=None,
                 theta=1.0e6, eps=1.0e-6):
    """Build a Problem for the given per-sequence lengths.

    seq_lens counts the q_len new tokens; the new tokens of sequence b sit at
    positions seq_len - q_len .. seq_len - 1 and are given slots in the
    sequence's own pages.  q_len is one count for every sequence or (varlen)
    one per sequence; varlen problems pack the new tokens back to back and
    carry their row offsets (cu_seqlens).  Physical blocks are a seeded random
    permutation of [0, num_blocks); unused table entries are -1.
    """
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, np.int64)
    B = seq_lens.shape[0]
    varlen = not np.isscalar(q_len)
    q_lens = np.asarray(q_len, np.int64) if varlen else np.full(B, int(q_len), np.int64)
    assert q_lens.shape == (B,) and np.all(q_lens >= 0) and np.all(q_lens <= seq_lens)
    pages = [_pages(n, block_size) for n in seq_lens]
    need = int(sum(pages))
    assert need <= num_blocks, (need, num_blocks)
    ids = rng.permutation(num_blocks) if block_perm else np.arange(num_blocks)
    width = max(pages) if table_width is None else table_width
    width = max(width, 1)
    bt = np.full((B, width), -1, np.int32)
    cur = 0
    for b, p in enumerate(pages):
        bt[b, :p] = ids[cur:cur + p]
        cur += p
    positions = np.concatenate(
        [np.arange(n - ql, n, dtype=np.int64) for n, ql in zip(seq_lens, q_lens)]
    ) if B else np.zeros(0, np.int64)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int64)
    slots = np.empty_like(positions)
    for b in range(B):
        for t in range(int(q_lens[b])):
            n = int(positions[cu[b] + t])
            slots[cu[b] + t] = int(bt[b, n // block_size]) * block_size + n % block_size

    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    T = int(cu[-1])

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)

    q = randn(T, Hq, D)
    k = randn(T, Hkv, D)
    v = randn(T, Hkv, D)
    gamma_q = (1.0 + 0.1 * torch.randn(D, generator=g, device=dev)).to(torch.bfloat16)
    gamma_k = (1.0 + 0.1 * torch.randn(D, generator=g, device=dev)).to(torch.bfloat16)
    k_cache = torch.empty(num_blocks, block_size, Hkv, D, dtype=torch.bfloat16, device=dev)
    v_cache = torch.empty_like(k_cache)
    # fill in slabs to bound the fp32 temporary
    step = max(1, (1 << 26) // max(1, block_size * Hkv * D))
    for s in range(0, num_blocks, step):
        e = min(num_blocks, s + step)
        k_cache[s:e] = torch.randn(e - s, block_size, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
        v_cache[s:e] = torch.randn(e - s, block_size, Hkv, D, generator=g, device=dev).to(torch.bfloat16)
    return Problem(
        name=name, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
        q_len=int(q_lens.max()) if (varlen and B) else int(q_len) if not varlen else 0,
        seq_lens_host=seq_lens, block_tables_host=bt, num_blocks=num_blocks,
        theta=theta, eps=eps, q=q, k=k, v=v, gamma_q=gamma_q, gamma_k=gamma_k,
        positions=torch.from_numpy(positions).to(dev),
        slot_mapping=torch.from_numpy(slots).to(dev),
        k_cache=k_cache, v_cache=v_cache,
        block_tables=torch.from_numpy(bt).to(dev),
        seq_lens=torch.from_numpy(seq_lens.astype(np.int32)).to(dev),
        q_lens_host=q_lens if varlen else None,
        cu_seqlens=torch.from_numpy(cu.astype(np.int32)).to(dev) if varlen else None,
    )


# ---------------------------------------------------------------- workloads

def decode_tiny(device="cpu", seed=BASE_SEED):
    """16q/8kv, D=128, batch 4, seq_len ~ U[1,256], 64 permuted blocks of 16."""
    rng = np.random.default_rng(seed)
    seq_lens = rng.integers(1, 257, size=4)
    return make_problem("decode_tiny", 16, 8, 128, 16, seq_lens, 1, 64, seed,
                        device, table_width=16)


def decode_uniform(batch, ctx, device="cpu", seed=BASE_SEED + 1):
    """16q/8kv, D=128; every sequence has context ctx; cache = exactly the pages."""
    seq_lens = np.full(batch, ctx, np.int64)
    nb = batch * _pages(ctx, 16)
    return make_problem(f"decode_uniform_b{batch}_ctx{ctx}", 16, 8, 128, 16,
                        seq_lens, 1, nb, seed, device)


def decode_long(device="cpu", seed=BASE_SEED + 2, batch=8, ctx=32768):
    """16q/8kv, D=128, batch 8, context 32768 (Qwen3-1.7B long context)."""
    seq_lens = np.full(batch, ctx, np.int64)
    nb = batch * _pages(ctx, 16)
    return make_problem(f"decode_long_b{batch}_ctx{ctx}", 16, 8, 128, 16,
                        seq_lens, 1, nb, seed, device)


def decode_gqa8(device="cpu", seed=BASE_SEED + 3, batch=64, lo=256, hi=16384):
    """32q/4kv, D=128, batch 64, contexts log-uniform in [lo, hi], 120% cache."""
    rng = np.random.default_rng(seed)
    ctx = np.exp(rng.uniform(math.log(lo), math.log(hi), size=batch))
    seq_lens = np.clip(np.rint(ctx).astype(np.int64), lo, hi)
    need = sum(_pages(n, 16) for n in seq_lens)
    nb = int(math.ceil(1.2 * need))
    return make_problem(f"decode_gqa8_b{batch}", 32, 4, 128, 16, seq_lens, 1,
                        nb, seed, device)


def verify_causal(device="cpu", seed=BASE_SEED + 4, batch=32, q_len=5,
                  lo=2048, hi=8192):
    """16q/8kv, D=128, batch 32, q_len = k+1 = 5, prior context U[lo, hi]."""
    rng = np.random.default_rng(seed)
    prior = rng.integers(lo, hi + 1, size=batch)
    seq_lens = prior + q_len
    nb = int(sum(_pages(n, 16) for n in seq_lens))
    return make_problem(f"verify_causal_b{batch}_k{q_len - 1}", 16, 8, 128, 16,
                        seq_lens, q_len, nb, seed, device)


def chunked_prefill(device="cpu", seed=BASE_SEED + 5, batch=8, chunk=512, lo=0, hi=6144,
                    Hq=16, Hkv=8, block_size=16, extra_blocks=0):
    """16q/8kv, D=128: `chunk` new tokens per sequence after a prior context
    U[lo, hi] (0 = the prompt's first chunk); cache = the pages needed plus
    `extra_blocks`, shuffled block ids."""
    rng = np.random.default_rng(seed)
    prior = rng.integers(lo, hi + 1, size=batch)
    seq_lens = prior + chunk
    nb = int(sum(_pages(n, block_size) for n in seq_lens)) + extra_blocks
    return make_problem(f"chunked_prefill_b{batch}_c{chunk}", Hq, Hkv, 128, block_size,
                        seq_lens, chunk, nb, seed, device)


def varlen_prefill(device="cpu", seed=BASE_SEED + 6, batch=16, lo=128, hi=2048, prior_lo=0,
                   prior_hi=0, Hq=16, Hkv=8, block_size=16):
    """16q/8kv, D=128: `batch` prompts of U[lo, hi] new tokens each (varlen,
    packed), after a prior context U[prior_lo, prior_hi] (0: fresh prompts);
    cache = the pages needed, shuffled block ids."""
    rng = np.random.default_rng(seed)
    q_lens = rng.integers(lo, hi + 1, size=batch)
    prior = rng.integers(prior_lo, prior_hi + 1, size=batch)
    seq_lens = prior + q_lens
    nb = max(1, int(sum(_pages(n, block_size) for n in seq_lens)))
    return make_problem(f"varlen_prefill_b{batch}", Hq, Hkv, 128, block_size, seq_lens, q_lens,
                        nb, seed, device)
