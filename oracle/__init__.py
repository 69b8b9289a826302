"""fp64 CPU oracle for the paged decode-attention hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
package; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may call it.  It shares no code with the CUDA
path: it is a plain restatement, in numpy float64, of what the operations are
defined to compute.

Sources (web pages; cited by title and section):

* InfiniLM PR #585 "perf: Qwen3 offline inference — hybrid attention backend,
  fused rms_norm_rope, chunked prefill + prompt-lookup spec decoding",
  section "概述 / Summary":
    - item 1: pure decode runs a paged split-KV kernel that reads the
      FlashAttention BSHD paged cache through strided views;
    - item 2: a fused per-head RMSNorm + full-rotary RoPE ("rms_norm_rope");
    - item 4: speculative verify runs one fused forward of fixed b x (k+1)
      shape; section "测量结果" fixes k = 4.
* The same page, section "依赖与 CI": the fused op is "per-head RMSNorm +
  RoPE".

Where the pages leave a step open the plain reading is taken; every such
reading is listed in the module docstring of ``oracle.reference``.

Pinning status: every public function is pinned by tests in
``tests/test_oracle_*.py`` against closed forms, invariants and independent
brute-force restatements; no function is "parity unpinned".
"""

from .reference import (  # noqa: F401
    bf16_bits_to_f64,
    f64_to_bf16_bits,
    rms_norm,
    rope_neox,
    norm_rope_append,
    paged_attention,
    paged_attention_splits,
    split_page_ranges,
    lse_combine,
)
