"""GPU parity of pkvqk_paged_prefill (tcgen05 multi-query attention) against
the fp64 oracle.

Operation: InfiniLM PR #585, section "概述 / Summary", item 4 (chunked
prefill; the verify step's fixed b x (k+1) shape) over the paged cache of
item 1: new token t of a sequence attends causally to every key up to its own
position.  Small cases compare every row; the benchmark-sized chunked-prefill
workload compares sampled tokens, each against the oracle's decode of that
token (query t of a q_len chunk sees exactly the keys a single query at
seq_len - q_len + t + 1 sees, a property the oracle's own pins check).
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_qk_gb300 import workloads
from tests._parity import (assert_attention_close, bits, compact_cache, oracle_attention)

pytestmark = pytest.mark.gpu


def _prefill(lib, p, num_splits=1, hint=None, q=None, k_cache=None, v_cache=None, flags=None,
             scale=0.0):
    q = p.q if q is None else q
    k_cache = p.k_cache if k_cache is None else k_cache
    v_cache = p.v_cache if v_cache is None else v_cache
    out = torch.full((p.B, p.q_len, p.Hq, p.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.B, p.q_len, p.Hq), float("nan"), device="cuda")
    hint = p.max_seq_len if hint is None else hint
    nbytes = lib.prefill_workspace_bytes(p.B, p.q_len, p.Hq, p.D, num_splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    lib.paged_prefill(q, k_cache, v_cache, p.block_tables, p.seq_lens, out, q_len=p.q_len,
                      num_splits=num_splits, max_seq_len_hint=hint, scale=scale, lse_out=lse,
                      workspace=ws, status_flags=flags)
    torch.cuda.synchronize()
    return out, lse


def _problem(Hq, Hkv, q_len, bs, priors, seed, extra_blocks=0):
    seq_lens = np.asarray(priors, np.int64) + q_len
    nb = int(sum(-(-int(n) // bs) for n in seq_lens)) + extra_blocks
    return workloads.make_problem(f"prefill_{Hq}_{Hkv}_{q_len}_{bs}", Hq, Hkv, 128, bs, seq_lens,
                                  q_len, max(nb, 1), seed, "cuda")


def _check_all(p, out, lse, what, scale=None):
    ref, ref_lse = oracle_attention(p, bits(p.q), scale=scale)
    return assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse, what)


# (Hq, Hkv, q_len, block_size, priors): row tiles of 128 packed (token, head)
# rows -- exact, ragged, several per kv head; fresh prompts (prior 0), short
# and long priors; GQA groups 1, 2, 3, 4, 8, 16; page sizes 16 .. 256 and a
# non-power-of-two 48
CASES = [
    (16, 8, 64, 16, [0, 100, 300]),
    (16, 8, 200, 16, [37, 0, 513]),
    (32, 4, 40, 32, [250, 1]),
    (16, 16, 130, 64, [0, 700]),
    (16, 8, 33, 256, [300, 5]),
    (16, 8, 50, 48, [61, 190]),
    (16, 8, 5, 16, [2000, 17, 0]),
    (16, 8, 1, 16, [900, 0, 31]),
    # several CTAs per kv head with a ragged last one: without tile B (600 rows,
    # pages of 256; 580 rows, pages of 48), GQA 8 (800 rows, a 32-row tile B),
    # GQA 1 with a fresh 700-token prompt
    (16, 8, 300, 256, [300, 5]),
    (16, 8, 290, 48, [61, 190]),
    (32, 4, 100, 32, [250, 1]),
    (16, 16, 700, 64, [0, 700]),
    # a group of 3: tiles start mid-token, so Q comes in and the output rows go
    # out by thread loads and stores instead of the row-tile TMA boxes
    (12, 4, 90, 16, [100, 0]),
    (12, 4, 200, 32, [0, 333]),
    # the TMA row-tile boxes for groups 4 and 16 (64 dims x G heads x 128/G
    # tokens): whole and ragged tiles
    (32, 8, 70, 32, [0, 200]),
    (16, 1, 40, 16, [70, 3]),
    # pages whose size is not a power of two: V boxes of 32 slots (pages of 96
    # and 160) and 64 (pages of 192), both dim halves per box, key tiles that
    # start inside a page
    (16, 8, 150, 96, [200, 33]),
    (16, 8, 70, 160, [500, 0]),
    (16, 8, 130, 192, [90, 401]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"Hq{c[0]}-Hkv{c[1]}-T{c[2]}-bs{c[3]}")
def test_prefill_all_rows_match_oracle(lib, case):
    Hq, Hkv, q_len, bs, priors = case
    p = _problem(Hq, Hkv, q_len, bs, priors, seed=900 + q_len + bs)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _prefill(lib, p, flags=flags)
    assert flags.item() == 0
    _check_all(p, out, lse, f"prefill {case}")


@pytest.mark.parametrize("S", [2, 3, 7])
def test_prefill_splits_match_oracle(lib, S):
    p = _problem(16, 8, 96, 16, [1500, 40, 0, 777], seed=31 + S)
    out, lse = _prefill(lib, p, num_splits=S)
    _check_all(p, out, lse, f"prefill S={S}")


@pytest.mark.parametrize("S", [2, 5])
def test_prefill_many_row_tiles_splits_match_oracle(lib, S):
    # 600 rows per kv head (three CTAs, the last one ragged) over split key ranges
    p = _problem(16, 8, 300, 16, [1500, 40, 0, 777], seed=41 + S)
    out, lse = _prefill(lib, p, num_splits=S)
    _check_all(p, out, lse, f"prefill pair S={S}")


def test_prefill_short_hint_last_split_takes_the_rest(lib):
    # a hint below the longest sequence: the last split covers every key past
    # (S-1) * C pages, so nothing is dropped
    p = _problem(16, 8, 20, 16, [1000, 300], seed=5)
    out, lse = _prefill(lib, p, num_splits=4, hint=200)
    _check_all(p, out, lse, "short hint")


def test_prefill_custom_scale(lib):
    p = _problem(16, 8, 24, 16, [300, 10], seed=8)
    out, lse = _prefill(lib, p, scale=0.05)
    _check_all(p, out, lse, "scale 0.05", scale=0.05)


def test_prefill_equals_verify_decode_kernel(lib):
    """q_len 5 (the verify shape): the tensor-core kernel and the decode
    kernel's verify path both match the oracle and each other closely."""
    p = workloads.verify_causal(device="cuda", batch=6)
    out_p, lse_p = _prefill(lib, p)
    out_d = torch.empty_like(out_p)
    lse_d = torch.empty_like(lse_p)
    lib.paged_decode(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, out_d, q_len=p.q_len,
                     num_splits=1, max_seq_len_hint=p.max_seq_len, lse_out=lse_d)
    torch.cuda.synchronize()
    _check_all(p, out_p, lse_p, "verify via prefill")
    diff = (out_p.float() - out_d.float()).abs()
    assert diff.max().item() <= 2e-2
    assert (lse_p - lse_d).abs().max().item() <= 1e-3


def test_chained_append_then_prefill(lib):
    """The benchmarked prefill step: the chunk's q/k normalised and rotated
    (angles from the per-position table), k/v appended, then the tensor-core
    prefill over the cache.  The oracle runs the same chain on the same
    inputs: its norm/RoPE/append, then its paged causal attention."""
    p = _problem(16, 8, 200, 16, [37, 0, 513], seed=83)
    q = p.q.clone()
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    q_in, kc_in, vc_in = bits(q), bits(kc), bits(vc)
    P = int(p.positions.max().item()) + 1
    table = torch.empty(lib.rope_table_bytes(P), dtype=torch.uint8, device="cuda")
    lib.rope_table_build(table, P, p.theta)
    lib.norm_rope_append_cached(q, p.k, p.v, p.positions, p.slot_mapping, p.gamma_q, p.gamma_k,
                                p.theta, p.eps, kc, vc, table, P)
    out, lse = _prefill(lib, p, q=q, k_cache=kc, v_cache=vc)
    qh, kco, vco, _, _ = oracle.norm_rope_append(
        q_in, bits(p.k), bits(p.v), p.positions.cpu().numpy(), p.slot_mapping.cpu().numpy(),
        bits(p.gamma_q), bits(p.gamma_k), p.theta, p.eps, kc_in, vc_in, p.block_size)
    ref, ref_lse = oracle.paged_attention(qh.reshape(p.B, p.q_len, p.Hq, p.D), kco, vco,
                                          p.block_tables_host, p.seq_lens_host, p.block_size,
                                          q_len=p.q_len)
    assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse, "chained prefill")


def test_prefill_without_lse_output(lib):
    """lse_out = NULL: the outputs are the same bits as with it, through both
    output paths (whole row tiles leave by TMA boxes, the ragged last tile by
    thread stores; 300 tokens x group 2 = two whole tiles and a partial one)."""
    p = _problem(16, 8, 300, 16, [37, 0, 513], seed=81)
    out_l, lse = _prefill(lib, p)
    out = torch.full_like(out_l, float("nan"))
    lib.paged_prefill(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, out, q_len=p.q_len,
                      max_seq_len_hint=p.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(out, out_l)
    assert torch.isfinite(lse).all()


def test_prefill_rows_without_keys(lib):
    # seq_len below q_len (tokens whose position would be negative) and an
    # empty sequence: their rows see no key -> 0 output and lse = -inf
    p = _problem(16, 8, 8, 16, [0, 0], seed=12)
    p.seq_lens = torch.tensor([3, 0], dtype=torch.int32, device="cuda")
    p.seq_lens_host = np.array([3, 0], np.int64)
    out, lse = _prefill(lib, p, hint=8)
    ref, ref_lse = oracle_attention(p, bits(p.q))
    got = oracle.bf16_bits_to_f64(bits(out))
    empty = np.isneginf(ref_lse)
    assert empty.sum() == (5 + 8) * 16
    assert np.array_equal(np.isneginf(lse.cpu().numpy()), empty)
    assert np.all(got[empty] == 0.0)
    assert np.abs(got[~empty] - ref[~empty]).max() <= 2e-2


@pytest.mark.parametrize("bs,priors", [(16, [100, 7]), (96, [150, 7]), (192, [300, 41])],
                         ids=["bs16", "bs96", "bs192"])
def test_prefill_ignores_non_finite_slots_past_the_end(lib, bs, priors):
    """Cache slots past a sequence's last key (the rest of its last page) may
    hold anything, NaN included; they must not reach the output.  Page sizes
    16, 96 and 192 put the zeroed V rows in boxes of 16, 32 and 64 slots."""
    p = _problem(16, 8, 40, bs, priors, seed=21)
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    for b in range(p.B):
        L = int(p.seq_lens_host[b])
        last = int(p.block_tables_host[b, (L - 1) // bs])
        kc[last, L % bs or bs:] = float("nan")
        vc[last, L % bs or bs:] = float("nan")
    out, lse = _prefill(lib, p, k_cache=kc, v_cache=vc)
    ref, ref_lse = oracle_attention(p, bits(p.q), k_cache=kc, v_cache=vc)
    assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse, "nan tail")


@pytest.mark.parametrize("prior,page,bad", [(64, 1, "past"), (600, 20, "past"), (600, 20, "neg")],
                         ids=["tile0", "tile2", "tile2-negative"])
def test_prefill_bad_block_id_is_flagged_and_reads_zeros(lib, prior, page, bad):
    # a page of key tile 0 (fetched before the loop) or of key tile 2 (its id
    # fetched one tile ahead, during tile 1); ids past the extent or negative
    p = _problem(16, 8, 16, 16, [prior], seed=3, extra_blocks=4)
    bt = p.block_tables.clone()
    bt[0, page] = p.num_blocks + 10 if bad == "past" else -5   # 16 keys -> zeros
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(p.B, p.q_len, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    lib.paged_prefill(p.q, p.k_cache, p.v_cache, bt, p.seq_lens, out, q_len=p.q_len,
                      max_seq_len_hint=p.max_seq_len, status_flags=flags)
    torch.cuda.synchronize()
    assert flags.item() & lib.FLAG_BAD_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    # the oracle on a cache whose block 1 of the sequence is zero gives the same
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    blk = int(p.block_tables_host[0, page])
    kc[blk] = 0
    vc[blk] = 0
    ref, _ = oracle_attention(p, bits(p.q), k_cache=kc, v_cache=vc)
    assert_attention_close(bits(out), ref, what="bad block")


def test_prefill_chunked_workload_sampled(lib):
    """The benchmark workload (8 sequences x 512-token chunks after prior
    context U[0, 6144]) in the benchmark's launch configuration; sampled
    tokens of every sequence against the oracle's decode of that token."""
    p = workloads.chunked_prefill(device="cuda")
    S = lib.choose_prefill_splits(p.B, p.Hkv, p.q_len, p.Hq // p.Hkv, p.max_seq_len)
    out, lse = _prefill(lib, p, num_splits=S)
    rng = np.random.default_rng(44)
    qb = bits(p.q).reshape(p.B, p.q_len, p.Hq, p.D)
    kb, vb, table, lens = compact_cache(p, list(range(p.B)))
    for b in range(p.B):
        for t in sorted(set([0, p.q_len - 1] + list(rng.integers(0, p.q_len, 2)))):
            ctx = int(lens[b]) - p.q_len + t + 1
            ref, ref_lse = oracle.paged_attention(qb[b:b + 1, t:t + 1], kb, vb, table[b:b + 1],
                                                  np.array([ctx]), p.block_size)
            assert_attention_close(bits(out[b:b + 1, t:t + 1]), ref,
                                   lse[b:b + 1, t:t + 1].cpu().numpy(), ref_lse,
                                   f"chunked b={b} t={t}")


def test_prefill_rejects_bad_arguments(lib):
    p = _problem(16, 8, 8, 16, [10], seed=1)
    out = torch.empty(p.B, p.q_len, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.PkvqkError) as e:
        lib.paged_prefill(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, out,
                          q_len=p.q_len, num_splits=0)
    assert e.value.status == lib.PKVQK_ERR_INVALID_ARG
    with pytest.raises(lib.PkvqkError) as e:
        lib.paged_prefill(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, out,
                          q_len=p.q_len, num_splits=3)       # no workspace
    assert e.value.status == lib.PKVQK_ERR_WORKSPACE_TOO_SMALL


# ------------------------------------------------------------------ varlen

def _varlen(lib, p, num_splits=1, hint=None, total_q=None):
    total_q = p.T if total_q is None else total_q
    out = torch.full((max(total_q, 1), p.Hq, p.D), float("nan"), dtype=torch.bfloat16,
                     device="cuda")[:total_q]
    lse = torch.full((max(total_q, 1), p.Hq), float("nan"), device="cuda")[:total_q]
    hint = p.max_seq_len if hint is None else hint
    nbytes = lib.prefill_workspace_bytes(1, total_q, p.Hq, p.D, num_splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.paged_prefill_varlen(p.q, p.cu_seqlens, max(p.q_len, 1), p.k_cache, p.v_cache,
                             p.block_tables, p.seq_lens, out, num_splits=num_splits,
                             max_seq_len_hint=hint, lse_out=lse, workspace=ws,
                             status_flags=flags)
    torch.cuda.synchronize()
    assert flags.item() == 0
    return out, lse


def _check_varlen(p, out, lse, what):
    """Each sequence against the oracle run on that sequence alone."""
    qb = bits(p.q)
    cu = p.cu_seqlens.cpu().numpy()
    for b in range(p.B):
        ql = int(p.q_lens_host[b])
        if ql == 0:
            continue
        kb, vb, table, lens = compact_cache(p, [b])
        ref, ref_lse = oracle.paged_attention(qb[cu[b]:cu[b + 1]].reshape(1, ql, p.Hq, p.D), kb,
                                              vb, table, lens, p.block_size, q_len=ql)
        assert_attention_close(bits(out[cu[b]:cu[b + 1]]).reshape(1, ql, p.Hq, p.D), ref,
                               lse[cu[b]:cu[b + 1]].cpu().numpy().reshape(1, ql, p.Hq), ref_lse,
                               f"{what} seq {b} (q_len {ql}, keys {int(lens[0])})")


@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (32, 4)])
def test_varlen_prefill_matches_oracle(lib, Hq, Hkv):
    # fresh prompts and later chunks mixed; lengths across row-tile edges
    # (1, 64, 127/128/129 rows per kv head at group 2 and 8, 300, 700)
    q_lens = [1, 64, 65, 128, 300, 7, 700, 33]
    prior = [0, 0, 400, 0, 1000, 5, 0, 2500]
    seq_lens = np.asarray(prior) + np.asarray(q_lens)
    nb = int(sum(-(-int(n) // 16) for n in seq_lens))
    p = workloads.make_problem("varlen", Hq, Hkv, 128, 16, seq_lens, q_lens, nb, 77, "cuda")
    out, lse = _varlen(lib, p)
    _check_varlen(p, out, lse, f"varlen Hq{Hq}/Hkv{Hkv}")


@pytest.mark.parametrize("S", [1, 4])
def test_varlen_prefill_workload(lib, S):
    p = workloads.varlen_prefill(device="cuda", batch=6, lo=100, hi=900, prior_hi=600)
    out, lse = _varlen(lib, p, num_splits=S)
    _check_varlen(p, out, lse, f"varlen workload S={S}")


def test_varlen_equals_fixed_when_lengths_agree(lib):
    # the same kernel arithmetic: varlen with equal lengths is bit-identical
    # to the fixed-q_len entry point
    p = _problem(16, 8, 150, 16, [0, 300, 77], seed=19)
    p.q_lens_host = np.full(p.B, p.q_len, np.int64)
    p.cu_seqlens = torch.arange(0, (p.B + 1) * p.q_len, p.q_len, dtype=torch.int32,
                                device="cuda")
    out_f, lse_f = _prefill(lib, p)
    out_v, lse_v = _varlen(lib, p)
    assert torch.equal(out_v, out_f.reshape(p.T, p.Hq, p.D))
    assert torch.equal(lse_v, lse_f.reshape(p.T, p.Hq))


def test_varlen_empty_sequences_and_short_grid(lib):
    # zero-token sequences write nothing; max_q_len covers the longest
    q_lens = [0, 5, 0, 260]
    seq_lens = np.asarray([10, 5, 0, 300])
    p = workloads.make_problem("varlen0", 16, 8, 128, 16, seq_lens, q_lens,
                               int(sum(-(-int(n) // 16) for n in seq_lens)), 5, "cuda")
    out, lse = _varlen(lib, p)
    _check_varlen(p, out, lse, "varlen with empty sequences")
    assert torch.isfinite(out.float()).all()


def _sampled_tokens(lib, p, out, lse, rng, per_seq=3):
    """Sampled tokens of every sequence against the oracle's decode of that
    token (query t of a q_len chunk sees the keys a single query at
    seq_len - q_len + t + 1 sees)."""
    qb = bits(p.q)
    cu = (p.cu_seqlens.cpu().numpy() if p.cu_seqlens is not None
          else np.arange(p.B + 1) * p.q_len)
    q_lens = p.q_lens_host if p.q_lens_host is not None else np.full(p.B, p.q_len)
    kb, vb, table, lens = compact_cache(p, list(range(p.B)))
    for b in range(p.B):
        ql = int(q_lens[b])
        if ql == 0:
            continue
        for t in sorted(set([0, ql - 1] + list(rng.integers(0, ql, per_seq)))):
            row = int(cu[b]) + t
            ctx = int(lens[b]) - ql + t + 1
            ref, ref_lse = oracle.paged_attention(qb[row:row + 1].reshape(1, 1, p.Hq, p.D), kb, vb,
                                                  table[b:b + 1], np.array([ctx]), p.block_size)
            assert_attention_close(bits(out[row:row + 1]).reshape(1, 1, p.Hq, p.D), ref,
                                   lse[row:row + 1].cpu().numpy().reshape(1, 1, p.Hq), ref_lse,
                                   f"b={b} t={t}")


def test_prefill_4x2048_workload_sampled(lib):
    """The 4 x 2048-token chunk workload in the benchmark's configuration."""
    p = workloads.chunked_prefill(device="cuda", batch=4, chunk=2048, lo=0, hi=8192)
    S = lib.choose_prefill_splits(p.B, p.Hkv, p.q_len, p.Hq // p.Hkv, p.max_seq_len)
    out, lse = _prefill(lib, p, num_splits=S)
    _sampled_tokens(lib, p, out.reshape(p.T, p.Hq, p.D), lse.reshape(p.T, p.Hq),
                    np.random.default_rng(45))


def test_prefill_19x512_ctx16k_workload_sampled(lib):
    """The long-context chunk workload (19 x 512-token chunks after 16384
    prior tokens, four full waves of CTAs) in the benchmark's configuration."""
    p = workloads.chunked_prefill(device="cuda", batch=19, chunk=512, lo=16384, hi=16384)
    S = lib.choose_prefill_splits(p.B, p.Hkv, p.q_len, p.Hq // p.Hkv, p.max_seq_len)
    out, lse = _prefill(lib, p, num_splits=S)
    _sampled_tokens(lib, p, out.reshape(p.T, p.Hq, p.D), lse.reshape(p.T, p.Hq),
                    np.random.default_rng(47), per_seq=1)


def test_varlen_prefill_16_workload_sampled(lib):
    """The varlen benchmark workload: 16 fresh prompts of U[128, 2048] tokens."""
    p = workloads.varlen_prefill(device="cuda")
    out, lse = _varlen(lib, p)
    _sampled_tokens(lib, p, out, lse, np.random.default_rng(46), per_seq=2)


@pytest.mark.parametrize("S", [1, 3])
def test_prefill_step_captures_and_replays(lib, S):
    """Append + prefill record into a CUDA graph and replay bit-identically
    (every call is host-decided and allocation-free)."""
    p = workloads.chunked_prefill(device="cuda", batch=2, chunk=300, lo=100, hi=900)
    nbytes = lib.prefill_workspace_bytes(p.B, p.q_len, p.Hq, p.D, S)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    q0, kc0, vc0 = p.q.clone(), p.k_cache.clone(), p.v_cache.clone()

    def step(q, kc, vc, out, lse, stream):
        lib.norm_rope_append(q, p.k, p.v, p.positions, p.slot_mapping, p.gamma_q, p.gamma_k,
                             p.theta, p.eps, kc, vc, stream=stream)
        lib.paged_prefill(q, kc, vc, p.block_tables, p.seq_lens, out, q_len=p.q_len,
                          num_splits=S, max_seq_len_hint=p.max_seq_len, lse_out=lse,
                          workspace=ws, stream=stream)

    q_e, kc_e, vc_e = q0.clone(), kc0.clone(), vc0.clone()
    out_e = torch.empty(p.B, p.q_len, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    lse_e = torch.empty(p.B, p.q_len, p.Hq, device="cuda")
    step(q_e, kc_e, vc_e, out_e, lse_e, torch.cuda.current_stream())
    torch.cuda.synchronize()

    q_g, kc_g, vc_g = q0.clone(), kc0.clone(), vc0.clone()
    out_g, lse_g = torch.zeros_like(out_e), torch.zeros_like(lse_e)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(q_g, kc_g, vc_g, out_g, lse_g, s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        q_g.copy_(q0)
        kc_g.copy_(kc0)
        vc_g.copy_(vc0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out_g, out_e) and torch.equal(lse_g, lse_e)
        assert torch.equal(kc_g, kc_e) and torch.equal(q_g, q_e)


def test_prefill_stacked_cache_and_strided_q(lib):
    """K/V as strided views of one (num_blocks, 2, block_size, Hkv, D)
    allocation, and q as the q part of a fused [tokens, Hq + 2 Hkv, D]
    projection output: no copy of either is made."""
    p = _problem(16, 8, 70, 16, [200, 0, 33], seed=61)
    both = torch.stack([p.k_cache, p.v_cache], dim=1).contiguous()
    qkv = torch.empty(p.T, p.Hq + 2 * p.Hkv, p.D, dtype=torch.bfloat16, device="cuda")
    qkv[:, :p.Hq] = p.q
    qkv[:, p.Hq:] = 7.0                           # k/v parts: must not be read as q
    q_view = qkv[:, :p.Hq]
    for S in (1, 2):
        out, lse = _prefill(lib, p, num_splits=S, q=q_view, k_cache=both[:, 0],
                            v_cache=both[:, 1])
        _check_all(p, out, lse, f"stacked cache, strided q, S={S}")
