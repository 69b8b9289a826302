"""GPU parity of pkvqk_paged_decode / pkvqk_lse_combine against the fp64 oracle.

Operation: InfiniLM PR #585, section "概述 / Summary", item 1 (pure-decode
paged split-KV attention over the BSHD cache) and item 4 (verify of k+1 draft
tokens, causal among them).  Every row of every sequence is compared at the
small sizes; at the full workload sizes a seeded sample of sequences is
compared (every head and query token of each sampled sequence), in the same
launch configuration as the benchmark.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_qk_gb300 import workloads
from tests._parity import assert_attention_close, bits, oracle_attention

pytestmark = pytest.mark.gpu


def _decode(lib, p, q=None, num_splits=1, hint=None, lse=True, k_cache=None, v_cache=None,
            flags=None, scale=0.0):
    """Run pkvqk_paged_decode; num_splits=0 is the balanced schedule, -1 uses
    the library's split heuristic (pkvqk_choose_num_splits) explicitly."""
    q = p.q if q is None else q
    k_cache = p.k_cache if k_cache is None else k_cache
    v_cache = p.v_cache if v_cache is None else v_cache
    out = torch.full((p.B, p.q_len, p.Hq, p.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_out = torch.full((p.B, p.q_len, p.Hq), float("nan"), device="cuda") if lse else None
    hint = p.max_seq_len if hint is None else hint
    S = num_splits
    if S < 0:
        S = lib.choose_num_splits(p.B, p.Hkv, p.q_len * p.Hq // p.Hkv, max(hint, 1),
                                  p.total_tokens, p.block_size)
    nbytes = lib.decode_workspace_bytes(p.B, p.q_len, p.Hq, p.D, S)
    ws = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    lib.paged_decode(q, k_cache, v_cache, p.block_tables, p.seq_lens, out, q_len=p.q_len,
                     num_splits=S, max_seq_len_hint=hint, scale=scale, lse_out=lse_out,
                     workspace=ws, status_flags=flags)
    torch.cuda.synchronize()
    return out, lse_out, S


def _check(p, out, lse_out, seqs=None, what=""):
    ref, ref_lse = oracle_attention(p, bits(p.q), seqs=seqs)
    sel = list(range(p.B)) if seqs is None else list(seqs)
    return assert_attention_close(bits(out[sel]), ref, lse_out[sel].cpu().numpy(), ref_lse, what)


@pytest.mark.parametrize("S", [0, 1, 4, -1])
def test_decode_tiny_all_rows(lib, S):
    p = workloads.decode_tiny(device="cuda")
    out, lse, _ = _decode(lib, p, num_splits=S)
    _check(p, out, lse, what=f"tiny S={S}")


def test_decode_tiny_splits_beyond_pages(lib):
    # more splits than a short sequence has pages: empty splits must weigh 0
    p = workloads.decode_tiny(device="cuda")
    for S in (7, 16, 64):
        out, lse, _ = _decode(lib, p, num_splits=S, hint=256)
        _check(p, out, lse, what=f"tiny S={S}")


def test_chained_norm_rope_append_then_decode(lib):
    """The whole step: q/k normalised and rotated, k/v appended, then decode.
    The oracle runs the same chain on the same inputs."""
    p = workloads.decode_tiny(device="cuda", seed=777)
    q = p.q.clone()
    kc, vc = p.k_cache.clone(), p.v_cache.clone()
    q_in, kc_in, vc_in = bits(q), bits(kc), bits(vc)
    lib.norm_rope_append(q, p.k, p.v, p.positions, p.slot_mapping, p.gamma_q, p.gamma_k,
                         p.theta, p.eps, kc, vc)
    out, lse, _ = _decode(lib, p, q=q, num_splits=2, k_cache=kc, v_cache=vc)
    qh, kco, vco, _, _ = oracle.norm_rope_append(
        q_in, bits(p.k), bits(p.v), p.positions.cpu().numpy(), p.slot_mapping.cpu().numpy(),
        bits(p.gamma_q), bits(p.gamma_k), p.theta, p.eps, kc_in, vc_in, p.block_size)
    ref, ref_lse = oracle.paged_attention(qh.reshape(p.B, 1, p.Hq, p.D), kco, vco,
                                          p.block_tables_host, p.seq_lens_host, p.block_size)
    assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse, "chained")


@pytest.mark.parametrize("batch,ctx", [(1, 512), (8, 512), (8, 2048), (4, 8192)])
def test_decode_uniform_small_points_all_rows(lib, batch, ctx):
    p = workloads.decode_uniform(batch, ctx, device="cuda")
    for S in (1, 0, -1):
        out, lse, S_used = _decode(lib, p, num_splits=S)
        _check(p, out, lse, what=f"b{batch} ctx{ctx} S={S_used}")


def test_decode_uniform_64x8192_sampled(lib):
    """The benchmark workload (64 x 8192) on the balanced schedule, 6 sampled
    sequences compared in full (the split schedule the benchmark times is
    covered by the sweep test below)."""
    p = workloads.decode_uniform(64, 8192, device="cuda")
    out, lse, S = _decode(lib, p, num_splits=0)
    seqs = sorted(np.random.default_rng(5).choice(64, 6, replace=False).tolist())
    _check(p, out, lse, seqs=seqs, what=f"64x8192 S={S}")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("batch,ctx", [(b, c) for b in (1, 8, 32, 64) for c in (512, 2048, 8192)])
def test_decode_sweep_point_in_bench_configuration(lib, batch, ctx):
    """Every point of the batch x context sweep in the launch configuration
    the benchmark times (the split heuristic's count): the first, the last
    and one seeded sequence compared in full."""
    p = workloads.decode_uniform(batch, ctx, device="cuda")
    out, lse, S = _decode(lib, p, num_splits=-1)
    pick = int(np.random.default_rng(batch * 131 + ctx).integers(batch))
    seqs = sorted({0, batch - 1, pick})
    _check(p, out, lse, seqs=seqs, what=f"{batch}x{ctx} S={S}")


@pytest.mark.parametrize("name,Hq,Hkv,B,ctx,seed", [
    ("gqa8_uniform", 32, 4, 64, 4096, 3), ("gqa4_uniform", 32, 8, 32, 8192, 7)])
def test_uniform_gqa_workloads_in_bench_configuration(lib, name, Hq, Hkv, B, ctx, seed):
    """The two uniform GQA workloads the benchmark times (GQA-8 64 x 4096,
    and GQA-4 32 x 8192 on the mma tiles), with its inputs and split count."""
    p = workloads.make_problem(name, Hq, Hkv, 128, 16, np.full(B, ctx), 1, B * ctx // 16,
                               workloads.BASE_SEED + seed, device="cuda")
    out, lse, S = _decode(lib, p, num_splits=-1)
    _check(p, out, lse, seqs=[0, B // 2, B - 1], what=f"{name} S={S}")


@pytest.mark.parametrize("S", [0, -1, 1, 8, 32, 128])
def test_decode_long_32k_sampled(lib, S):
    p = workloads.decode_long(device="cuda")
    out, lse, S_used = _decode(lib, p, num_splits=S)
    _check(p, out, lse, seqs=[0, 5], what=f"32k S={S_used}")


def test_gqa8_tensor_core_path_sampled(lib):
    p = workloads.decode_gqa8(device="cuda")
    out, lse, S = _decode(lib, p, num_splits=0)
    _check(p, out, lse, seqs=[3, 40], what="gqa8 balanced")
    out, lse, S = _decode(lib, p, num_splits=-1)
    order = np.argsort(p.seq_lens_host)
    seqs = sorted({int(order[0]), int(order[1]), int(order[32]), int(order[-1]), 7})
    _check(p, out, lse, seqs=seqs, what=f"gqa8 S={S}")
    assert torch.isfinite(out.float()).all()


def test_gqa8_small_all_rows(lib):
    p = workloads.make_problem("gqa8_small", 32, 4, 128, 16, [1, 17, 40, 300, 16, 33], 1, 64,
                               905, "cuda")
    for S in (0, 1, 3):
        out, lse, _ = _decode(lib, p, num_splits=S)
        _check(p, out, lse, what=f"gqa8 small S={S}")


def test_verify_causal_sampled(lib):
    p = workloads.verify_causal(device="cuda")
    for S in (0, -1):
        out, lse, S_used = _decode(lib, p, num_splits=S)
        _check(p, out, lse, seqs=[0, 9, 31], what=f"verify S={S_used}")


@pytest.mark.parametrize("q_len,Hq,Hkv", [(5, 16, 8), (2, 16, 8), (3, 8, 8), (4, 32, 8), (2, 32, 4),
                                           (1, 8, 8), (1, 24, 8)])
def test_multi_query_small_all_rows(lib, q_len, Hq, Hkv):
    # rows per kv head = q_len * group covers both kernel families (1..2:
    # CUDA cores; 3..16: mma tiles), including one row (MHA) and 3 rows
    lens = [q_len, q_len + 1, 16 + q_len, 100, 37]
    p = workloads.make_problem("mq", Hq, Hkv, 128, 16, lens, q_len, 40, 906 + q_len, "cuda")
    for S in (0, 1, 2):
        out, lse, _ = _decode(lib, p, num_splits=S)
        _check(p, out, lse, what=f"q_len={q_len} Hq={Hq} Hkv={Hkv} S={S}")


@pytest.mark.parametrize("q_len,Hq,Hkv", [(5, 64, 8), (3, 48, 8), (16, 32, 8), (9, 16, 8)])
def test_multi_query_beyond_16_rows_all_rows(lib, q_len, Hq, Hkv):
    # more than 16 rows per kv head (18 .. 128): the call runs on the
    # tensor-core multi-query kernel; every schedule argument stays valid
    lens = [q_len, q_len + 1, 16 + q_len, 300, 37, 129 + q_len]
    p = workloads.make_problem("mq16", Hq, Hkv, 128, 16, lens, q_len, 40, 930 + q_len, "cuda")
    rows = q_len * Hq // Hkv
    assert rows > 16
    for S in (0, 1, 3, -1):
        out, lse, S_used = _decode(lib, p, num_splits=S)
        assert S_used >= 1 or S == 0
        _check(p, out, lse, what=f"q_len={q_len} Hq={Hq} Hkv={Hkv} S={S_used}")


def test_partials_beyond_16_rows_equal_decode(lib):
    # the tensor-core route writes the decode kernel's partial layout, so
    # partials + pkvqk_lse_combine reproduce the merged call bit for bit
    q_len, Hq, Hkv, S = 5, 64, 8, 3
    p = workloads.make_problem("mq16p", Hq, Hkv, 128, 16, [5, 300, 77, 1000], q_len, 100, 941,
                               "cuda")
    out, lse, _ = _decode(lib, p, num_splits=S)
    nbytes = lib.decode_workspace_bytes(p.B, q_len, p.Hq, p.D, S)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    lib.paged_decode_partials(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, ws,
                              q_len=q_len, num_splits=S, max_seq_len_hint=p.max_seq_len)
    rows = p.B * q_len * p.Hq
    ws_f = ws.view(torch.float32)
    ws_o = ws_f[: rows * S * 128]
    ws_lse = ws_f[rows * S * 128: rows * S * 129]
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    lib.lse_combine(ws_o, ws_lse, rows, S, out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    _check(p, out2, lse2, what="partials + combine, 40 rows per kv head")


def test_edge_lengths_and_empty_sequence(lib):
    # seq_len 0 -> zeros and -inf; lengths at tile / page boundaries
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 255, 256]
    p = workloads.make_problem("edges", 16, 8, 128, 16, [max(n, 1) for n in lens], 1, 64, 907, "cuda")
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    p.seq_lens = sl
    p.seq_lens_host = np.asarray(lens, np.int64)
    for S in (0, 1, 3):
        out, lse, _ = _decode(lib, p, num_splits=S)
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
        _check(p, out, lse, seqs=list(range(1, len(lens))), what=f"edges S={S}")


@pytest.mark.parametrize("bs", [32, 64, 256])
def test_larger_block_sizes(lib, bs):
    lens = [1, bs - 1, bs, bs + 1, 3 * bs + 7]
    nb = sum(-(-n // bs) for n in lens) + 3
    p = workloads.make_problem(f"bs{bs}", 16, 8, 128, bs, lens, 1, nb, 908, "cuda")
    for S in (0, 1, 2):
        out, lse, _ = _decode(lib, p, num_splits=S)
        _check(p, out, lse, what=f"bs={bs} S={S}")


def test_balanced_schedule_mixed_lengths_all_rows(lib):
    """One long sequence cut across many CTAs next to short ones, empties, and
    more CTAs than pages elsewhere in the list."""
    lens = [0, 3, 16, 17, 6000, 1, 0, 95, 2048, 33]
    p = workloads.make_problem("mixed", 16, 8, 128, 16, [max(n, 1) for n in lens], 1,
                               sum(-(-max(n, 1) // 16) for n in lens) + 4, 915, "cuda")
    p.seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    p.seq_lens_host = np.asarray(lens, np.int64)
    out, lse, _ = _decode(lib, p, num_splits=0)
    for b in (0, 6):
        assert torch.all(out[b] == 0) and torch.all(torch.isneginf(lse[b]))
    _check(p, out, lse, seqs=[1, 2, 3, 4, 5, 7, 8, 9], what="balanced mixed")


def test_balanced_schedule_tiny_batch_fewer_pages_than_ctas(lib):
    p = workloads.make_problem("tiny1", 16, 8, 128, 16, [40], 1, 3, 916, "cuda")
    out, lse, _ = _decode(lib, p, num_splits=0)
    _check(p, out, lse, what="balanced 1 seq, 3 pages")


def test_interleaved_cache_view_no_copy(lib):
    # K/V as strided views of a (num_blocks, 2, block_size, Hkv, D) allocation
    p = workloads.make_problem("kvstack", 16, 8, 128, 16, [40, 3, 77], 1, 16, 909, "cuda")
    both = torch.stack([p.k_cache, p.v_cache], dim=1).contiguous()
    for S in (0, 2):
        out, lse, _ = _decode(lib, p, num_splits=S, k_cache=both[:, 0], v_cache=both[:, 1])
        _check(p, out, lse, what=f"interleaved cache S={S}")


def test_partials_plus_combine_equals_decode(lib):
    p = workloads.decode_uniform(8, 2048, device="cuda")
    S = 5
    out, lse, _ = _decode(lib, p, num_splits=S)
    nbytes = lib.decode_workspace_bytes(p.B, 1, p.Hq, p.D, S)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    lib.paged_decode_partials(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, ws,
                              num_splits=S, max_seq_len_hint=p.max_seq_len)
    rows = p.B * p.Hq
    ws_f = ws.view(torch.float32)
    ws_o = ws_f[: rows * S * 128]
    ws_lse = ws_f[rows * S * 128: rows * S * 129]
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    lib.lse_combine(ws_o, ws_lse, rows, S, out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # partials against the oracle's own split partials (same partition)
    seqs = [0, 3]
    pages = -(-p.max_seq_len // p.block_size)
    chunk = -(-pages // S)
    ref_o, ref_l = oracle.paged_attention_splits(
        bits(p.q).reshape(p.B, 1, p.Hq, p.D)[seqs], *_compact(p, seqs), p.block_size, S, chunk)
    got_o = ws_o.view(p.B, p.Hq, S, 128)[seqs].cpu().numpy()
    got_l = ws_lse.view(p.B, p.Hq, S)[seqs].cpu().numpy()
    assert np.abs(got_o - ref_o[:, 0]).max() < 2e-3
    fin = np.isfinite(ref_l[:, 0])
    assert np.array_equal(np.isfinite(got_l), fin)
    assert np.abs(got_l[fin] - ref_l[:, 0][fin]).max() < 1e-3


def test_workspace_reuse_across_split_counts(lib):
    """One workspace reused by calls with different split counts, without
    clearing in between."""
    p = workloads.decode_uniform(8, 2048, device="cuda")
    nbytes = max(lib.decode_workspace_bytes(p.B, 1, p.Hq, p.D, S) for S in (3, 5, 8))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ref, ref_lse = oracle_attention(p, bits(p.q), seqs=[2, 7])
    for S in (3, 5, 3, 8, 5, 3):
        out = torch.full((p.B, 1, p.Hq, p.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((p.B, 1, p.Hq), float("nan"), device="cuda")
        lib.paged_decode(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, out,
                         num_splits=S, max_seq_len_hint=p.max_seq_len, lse_out=lse, workspace=ws)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert_attention_close(bits(out[[2, 7]]), ref, lse[[2, 7]].cpu().numpy(), ref_lse,
                               f"reused workspace S={S}")


def _compact(p, seqs):
    from tests._parity import compact_cache
    kb, vb, table, lens = compact_cache(p, seqs)
    return kb, vb, table, lens


def test_combine_standalone_against_oracle(lib):
    rng = np.random.default_rng(11)
    rows, S = 37, 9
    o = rng.standard_normal((rows, S, 128)).astype(np.float32)
    lse = (rng.standard_normal((rows, S)) * 3).astype(np.float32)
    lse[rng.random((rows, S)) < 0.3] = -np.inf
    lse[5, :] = -np.inf                                    # an all-empty row
    out = torch.empty(rows, 128, dtype=torch.bfloat16, device="cuda")
    lse_out = torch.empty(rows, device="cuda")
    lib.lse_combine(torch.from_numpy(o).cuda(), torch.from_numpy(lse).cuda(), rows, S, out, lse_out)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.lse_combine(o.astype(np.float64), lse.astype(np.float64))
    got = oracle.bf16_bits_to_f64(bits(out))
    assert np.abs(got - ref).max() <= 2 ** -8 * np.abs(ref).max() + 1e-6
    g = lse_out.cpu().numpy()
    assert np.isneginf(g[5]) and np.all(got[5] == 0)
    fin = np.isfinite(ref_lse)
    assert np.abs(g[fin] - ref_lse[fin]).max() < 1e-5


@pytest.mark.parametrize("S", [0, 3])
def test_block_permutation_invariance_and_determinism(lib, S):
    p = workloads.decode_uniform(4, 2048, device="cuda")
    out1, lse1, _ = _decode(lib, p, num_splits=S)
    out1b, lse1b, _ = _decode(lib, p, num_splits=S)
    assert torch.equal(out1, out1b) and torch.equal(lse1, lse1b)     # bit-identical reruns
    perm = torch.randperm(p.num_blocks, generator=torch.Generator().manual_seed(3)).cuda()
    kc2 = torch.empty_like(p.k_cache)
    vc2 = torch.empty_like(p.v_cache)
    kc2[perm] = p.k_cache
    vc2[perm] = p.v_cache
    bt2 = perm[p.block_tables.long()].to(torch.int32)
    p2 = workloads.Problem(**{**p.__dict__, "block_tables": bt2})
    out2, lse2, _ = _decode(lib, p2, num_splits=S, k_cache=kc2, v_cache=vc2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_bad_block_id_is_flagged_not_faulted(lib):
    p = workloads.make_problem("badblk", 16, 8, 128, 16, [40, 20], 1, 8, 910, "cuda")
    bt = p.block_tables.clone()
    bt[0, 1] = p.num_blocks + 100        # out of range: TMA fills zeros, flag raised
    p2 = workloads.Problem(**{**p.__dict__, "block_tables": bt})
    for S in (1, 0):
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse, _ = _decode(lib, p2, num_splits=S, flags=flags)
        assert flags.item() & lib.FLAG_BAD_BLOCK_ID
        # the untouched sequence is still right
        _check(p, out, lse, seqs=[1], what=f"bad block, other seq S={S}")


def test_custom_scale(lib):
    p = workloads.decode_tiny(device="cuda")
    out, lse, _ = _decode(lib, p, num_splits=0, scale=0.05)
    ref, ref_lse = oracle_attention(p, bits(p.q), scale=0.05)
    assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse, "scale 0.05")


def test_workspace_shared_by_balanced_and_split_calls(lib):
    """One workspace, zeroed once, across balanced and split calls of
    different shapes: nothing in it carries from one call to the next."""
    probs = [workloads.decode_uniform(8, 2048, device="cuda"),
             workloads.make_problem("bal-mixed", 32, 4, 128, 16, [3000, 17, 900, 4100, 1], 1,
                                    600, 818, "cuda"),
             workloads.verify_causal(device="cuda", batch=6)]
    nbytes = max(lib.decode_workspace_bytes(p.B, p.q_len, p.Hq, p.D, S)
                 for p in probs for S in (0, 3))
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    # balanced calls of every shape, then again interleaved with split calls
    calls = [(p, 0) for p in probs] + [(p, S) for p in probs for S in (3, 0)]
    for i, (p, S) in enumerate(calls):
        out = torch.full((p.B, p.q_len, p.Hq, p.D), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        lse = torch.full((p.B, p.q_len, p.Hq), float("nan"), device="cuda")
        lib.paged_decode(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, out,
                         q_len=p.q_len, num_splits=S, max_seq_len_hint=p.max_seq_len,
                         lse_out=lse, workspace=ws)
        torch.cuda.synchronize()
        ref, ref_lse = oracle_attention(p, bits(p.q))
        assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse,
                               f"workspace reuse call {i} ({p.name}, S={S})")


def test_host_pointer_rejected_after_device_calls(lib):
    """The residency check (pageable host memory where device memory is
    expected) fires on every call, also right after successful device calls,
    and a rejected call launches nothing."""
    p = workloads.decode_tiny(device="cuda")
    out, lse, _ = _decode(lib, p, num_splits=1)
    _check(p, out, lse, what="before the host-pointer call")
    for host_arg in ("q", "seq_lens"):
        kw = {"q": p.q, "seq_lens": p.seq_lens}
        kw[host_arg] = kw[host_arg].cpu()
        out2 = torch.full_like(out, float("nan"))
        with pytest.raises(lib.PkvqkError) as ei:
            lib.paged_decode(kw["q"], p.k_cache, p.v_cache, p.block_tables, kw["seq_lens"], out2,
                             q_len=p.q_len, num_splits=1, max_seq_len_hint=p.max_seq_len)
        assert ei.value.status == lib.PKVQK_ERR_POINTER_RESIDENCY
        torch.cuda.synchronize()
        assert torch.isnan(out2.float()).all()
    # the same device pointers still pass afterwards
    out3, lse3, _ = _decode(lib, p, num_splits=1)
    assert torch.equal(out3, out)


def test_balanced_schedule_any_workspace_contents(lib):
    """Whatever the workspace holds before a balanced-schedule call (all
    ones, random bytes, a previous call's partials and unit table), the
    result is the same and matches the oracle."""
    lens = list(np.random.default_rng(951).integers(1, 3000, size=24))
    p = workloads.make_problem("bal_ws", 32, 4, 128, 16, lens, 1, 24 * 190, 951, "cuda")
    nbytes = lib.decode_workspace_bytes(p.B, 1, p.Hq, p.D, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ref, ref_lse = oracle_attention(p, bits(p.q))
    gen = torch.Generator(device="cuda").manual_seed(7)
    fills = ["ones", "random", "reuse", "reuse"]
    prev = None
    for fill in fills:
        if fill == "ones":
            ws.fill_(0xFF)
        elif fill == "random":
            ws.copy_(torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda",
                                   generator=gen))
        out = torch.full((p.B, 1, p.Hq, p.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((p.B, 1, p.Hq), float("nan"), device="cuda")
        lib.paged_decode(p.q, p.k_cache, p.v_cache, p.block_tables, p.seq_lens, out,
                         num_splits=0, max_seq_len_hint=p.max_seq_len, lse_out=lse, workspace=ws)
        torch.cuda.synchronize()
        assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse, f"balanced ws {fill}")
        if prev is not None:
            assert torch.equal(out, prev)        # the page partition fixes every bit
        prev = out
