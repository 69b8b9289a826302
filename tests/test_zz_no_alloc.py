"""GPU test of pkvqk_paged_decode_static_ws, the decode entry point for
callers that cannot allocate device memory (a plugin given only input and
output pointers, code running while its allocator refuses allocations).

It keeps the split partials in a fixed array inside the library instead of a
caller workspace.  Its results must match pkvqk_paged_decode (with a caller
workspace) within the attention tolerances used by every parity test, on two
calls in a row with different shapes (the shared array keeps the previous
call's contents), and with num_splits == 0, where the call picks its own split
count with pkvqk_choose_num_splits.  This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import oracle
from paged_kv_cache_qk_gb300 import workloads
from tests._parity import assert_attention_close, bits, oracle_attention

pytestmark = pytest.mark.gpu


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _run_both(lib, p, S, S_static=None):
    """(out, lse) from the caller-workspace entry point with split count S and
    from the static one with S_static (default: S)."""
    S_static = S if S_static is None else S_static
    lay = lib.cache_layout(p.k_cache)
    stream = torch.cuda.current_stream().cuda_stream
    shape = (p.B, p.q_len, p.Hq, p.D)
    out_ref = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    lse_ref = torch.empty(shape[:3], device="cuda")
    ws_bytes = lib.decode_workspace_bytes(p.B, p.q_len, p.Hq, p.D, S)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    lib.check(lib.pkvqk_paged_decode(
        _ptr(p.q), p.q.stride(0), p.q.stride(1), _ptr(p.k_cache), _ptr(p.v_cache),
        ctypes.byref(lay), _ptr(p.block_tables), p.block_tables.shape[1], _ptr(p.seq_lens),
        p.B, p.q_len, p.Hq, S, p.max_seq_len, 0.0, _ptr(out_ref), _ptr(lse_ref),
        _ptr(ws), ws_bytes, None, stream))
    out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(shape[:3], float("nan"), device="cuda")
    lib.check(lib.pkvqk_paged_decode_static_ws(
        _ptr(p.q), p.q.stride(0), p.q.stride(1), _ptr(p.k_cache), _ptr(p.v_cache),
        ctypes.byref(lay), _ptr(p.block_tables), p.block_tables.shape[1], _ptr(p.seq_lens),
        p.B, p.q_len, p.Hq, S_static, p.max_seq_len, 0.0, _ptr(out), _ptr(lse), None, stream))
    torch.cuda.synchronize()
    return out_ref, lse_ref, out, lse


def test_static_workspace_matches_caller_workspace_two_calls(lib):
    cases = [
        (workloads.decode_uniform(8, 2048, device="cuda"), 5),
        (workloads.make_problem("verify_small", 16, 8, 128, 16, [9, 300, 77, 1030], 5, 100,
                                931, "cuda"), 3),
    ]
    for p, S in cases:
        out_ref, lse_ref, out, lse = _run_both(lib, p, S)
        # within the parity tolerances of the existing entry point's output ...
        assert_attention_close(bits(out), oracle.bf16_bits_to_f64(bits(out_ref)),
                               lse.cpu().numpy(), lse_ref.cpu().numpy(), f"static ws S={S}")
        # ... and both against the fp64 oracle on one sequence
        ref, ref_lse = oracle_attention(p, bits(p.q), seqs=[1])
        assert_attention_close(bits(out[1:2]), ref, lse[1:2].cpu().numpy(), ref_lse, "oracle")


def test_static_workspace_chooses_its_split_count(lib):
    """num_splits == 0: the call takes the split count pkvqk_choose_num_splits
    gives for the hint (a uniform batch of hint-long sequences), never the
    balanced schedule, whose workspace it does not hold."""
    cases = [
        workloads.decode_uniform(8, 2048, device="cuda"),
        workloads.make_problem("static_mixed", 16, 8, 128, 16, [3, 900, 41, 2500, 17, 1200], 1,
                               400, 937, "cuda"),
    ]
    for p in cases:
        rows = p.q_len * p.Hq // p.Hkv
        S = lib.choose_num_splits(p.B, p.Hkv, rows, p.max_seq_len, p.max_seq_len * p.B,
                                  p.block_size)
        assert S >= 1
        out_ref, lse_ref, out, lse = _run_both(lib, p, S, S_static=0)
        # the same split count, so the same partials and merge
        assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16)), f"S={S}"
        assert torch.equal(lse, lse_ref)
        ref, ref_lse = oracle_attention(p, bits(p.q))
        assert_attention_close(bits(out), ref, lse.cpu().numpy(), ref_lse, f"static ws S=0->{S}")


def test_static_workspace_rejects_oversized_calls(lib):
    cap = lib.pkvqk_static_workspace_capacity()
    assert cap == 16 << 20
    p = workloads.decode_uniform(8, 2048, device="cuda")
    lay = lib.cache_layout(p.k_cache)
    S = 256                                  # 8 x 16 heads x 256 splits x 129 x 4 B > 16 MiB
    need = lib.decode_workspace_bytes(p.B, 1, p.Hq, p.D, S)
    assert need > cap
    out = torch.zeros(p.B, 1, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    st = lib.pkvqk_paged_decode_static_ws(
        _ptr(p.q), p.q.stride(0), p.q.stride(1), _ptr(p.k_cache), _ptr(p.v_cache),
        ctypes.byref(lay), _ptr(p.block_tables), p.block_tables.shape[1], _ptr(p.seq_lens),
        p.B, 1, p.Hq, S, p.max_seq_len, 0.0, _ptr(out), None, None,
        torch.cuda.current_stream().cuda_stream)
    assert st == lib.PKVQK_ERR_WORKSPACE_TOO_SMALL
    assert "static workspace" in lib.pkvqk_last_error().decode()
    torch.cuda.synchronize()
    assert torch.all(out == 0)               # nothing launched
