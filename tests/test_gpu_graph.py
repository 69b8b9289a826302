"""The decode step records into a CUDA graph and replays bit-identically.

InfiniLM PR #585 runs decode as a captured paged CUDA graph (section
"概述 / Summary", item 3: graph hardening; the issue #498 page captures
decode graphs per batch bucket).  Every pkvqk call is host-decided and
allocation-free, so append + decode (+ combine) capture as kernel nodes with
programmatic-launch edges; replaying the graph must give the same bits as
running the calls eagerly, for the split and the balanced schedules, and with
the append's rotary sin/cos read from a per-position table built before the
capture (the form the benchmark's steps use).
"""

import pytest
import torch

from paged_kv_cache_qk_gb300 import workloads
from tests._parity import assert_attention_close, bits, oracle_attention

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S,table", [(1, False), (3, False), (0, False), (3, True)])
def test_step_captures_and_replays_bit_identically(lib, S, table):
    p = workloads.decode_uniform(8, 2048, device="cuda")
    P = int(p.positions.max().item()) + 1
    rope = torch.empty(lib.rope_table_bytes(P), dtype=torch.uint8, device="cuda")
    lib.rope_table_build(rope, P, p.theta)
    torch.cuda.synchronize()
    nbytes = lib.decode_workspace_bytes(p.B, 1, p.Hq, p.D, S)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda") if nbytes else None
    q0 = p.q.clone()
    kc0, vc0 = p.k_cache.clone(), p.v_cache.clone()

    def step(q, kc, vc, out, lse, stream):
        if table:
            lib.norm_rope_append_cached(q, p.k, p.v, p.positions, p.slot_mapping, p.gamma_q,
                                        p.gamma_k, p.theta, p.eps, kc, vc, rope, P,
                                        stream=stream)
        else:
            lib.norm_rope_append(q, p.k, p.v, p.positions, p.slot_mapping, p.gamma_q,
                                 p.gamma_k, p.theta, p.eps, kc, vc, stream=stream)
        lib.paged_decode(q, kc, vc, p.block_tables, p.seq_lens, out, num_splits=S,
                         max_seq_len_hint=p.max_seq_len, lse_out=lse, workspace=ws,
                         stream=stream)

    # eager reference
    q_e, kc_e, vc_e = q0.clone(), kc0.clone(), vc0.clone()
    out_e = torch.empty(p.B, 1, p.Hq, p.D, dtype=torch.bfloat16, device="cuda")
    lse_e = torch.empty(p.B, 1, p.Hq, device="cuda")
    step(q_e, kc_e, vc_e, out_e, lse_e, torch.cuda.current_stream())
    torch.cuda.synchronize()

    # capture on a side stream, then replay twice from fresh inputs
    q_g, kc_g, vc_g = q0.clone(), kc0.clone(), vc0.clone()
    out_g = torch.zeros_like(out_e)
    lse_g = torch.zeros_like(lse_e)
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
        assert torch.equal(kc_g, kc_e) and torch.equal(vc_g, vc_e) and torch.equal(q_g, q_e)
    # and the replayed result is the attention of the appended cache
    ref, ref_lse = oracle_attention(p, bits(q_g), seqs=[0, 5], k_cache=kc_g, v_cache=vc_g)
    assert_attention_close(bits(out_g[[0, 5]]), ref, lse_g[[0, 5]].cpu().numpy(), ref_lse,
                           f"graph S={S} table={table}")
