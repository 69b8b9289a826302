"""Host-side tests of the C ABI (no GPU needed).

* libpkvqk.so loads and exports every function include/pkvqk.h declares;
* argument validation returns the documented status before any launch;
* the host-only helpers (split heuristic, workspace size) follow their
  documented formulas.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkvqk.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_qk_gb300 import build
    build.build()
    from paged_kv_cache_qk_gb300 import binding
    return binding


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"PKVQK_API\s+[\w\s\*]+?\b(pkvqk_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["pkvqk_norm_rope_append", "pkvqk_paged_decode", "pkvqk_lse_combine",
              "pkvqk_choose_num_splits", "pkvqk_decode_workspace_bytes"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for n in declared_functions():
        assert hasattr(so, n), f"{n} not exported"
    assert set(declared_functions()) <= set(lib.EXPORTED)
    assert lib.pkvqk_abi_version() == 1


def _layout(lib, nb=64, bs=16, hkv=8, d=128, strides=None):
    if strides is None:
        strides = (bs * hkv * d, hkv * d, d)
    return lib.CacheLayout(nb, bs, hkv, d, 0, *strides)


FAKE = 0x10000  # never dereferenced: every case below fails before pointer checks


def _decode(lib, lay, B=4, q_len=1, Hq=16, S=1, hint=256, ws=0, maxp=16, qs=(2048, 128)):
    return lib.pkvqk_paged_decode(FAKE, qs[0], qs[1], FAKE, FAKE, ctypes.byref(lay), FAKE, maxp,
                                  FAKE, B, q_len, Hq, S, hint, 0.0, FAKE, None, FAKE, ws, None,
                                  None)


def test_decode_validation_errors(lib):
    lay = _layout(lib)
    assert _decode(lib, _layout(lib, d=64)) == lib.PKVQK_ERR_UNSUPPORTED
    assert "head_dim" in lib.pkvqk_last_error().decode()
    assert _decode(lib, _layout(lib, bs=8)) == lib.PKVQK_ERR_UNSUPPORTED
    assert _decode(lib, _layout(lib, bs=24)) == lib.PKVQK_ERR_UNSUPPORTED
    assert _decode(lib, lay, q_len=0) == lib.PKVQK_ERR_INVALID_ARG
    assert _decode(lib, lay, q_len=17) == lib.PKVQK_ERR_INVALID_ARG
    assert _decode(lib, lay, Hq=12) == lib.PKVQK_ERR_INVALID_ARG            # 12 % 8 != 0
    # 24 rows per kv head take the tensor-core route, which checks its own
    # workspace need (rows x splits x 129 x 4 bytes) before any pointer
    assert _decode(lib, lay, Hq=64, q_len=3, S=4, ws=100) == lib.PKVQK_ERR_WORKSPACE_TOO_SMALL
    # the balanced schedule there becomes a split count (> 1 for 32 CTAs
    # over 8192 keys), whose partials need a workspace too
    assert _decode(lib, lay, Hq=64, q_len=3, S=0, ws=100, hint=8192,
                   maxp=512) == lib.PKVQK_ERR_WORKSPACE_TOO_SMALL
    assert _decode(lib, lay, S=257) == lib.PKVQK_ERR_INVALID_ARG
    assert _decode(lib, lay, S=-1) == lib.PKVQK_ERR_INVALID_ARG
    assert _decode(lib, lay, S=0, ws=100) == lib.PKVQK_ERR_WORKSPACE_TOO_SMALL
    assert _decode(lib, lay, S=4, ws=100) == lib.PKVQK_ERR_WORKSPACE_TOO_SMALL
    assert _decode(lib, lay, maxp=0) == lib.PKVQK_ERR_INVALID_ARG
    assert _decode(lib, lay, qs=(2048, 100)) == lib.PKVQK_ERR_INVALID_ARG   # q head stride % 8
    assert _decode(lib, _layout(lib, strides=(16384, 1020, 128))) == lib.PKVQK_ERR_INVALID_ARG
    assert _decode(lib, _layout(lib, nb=0)) == lib.PKVQK_ERR_INVALID_ARG
    # batch 0 is a valid no-op
    assert _decode(lib, lay, B=0) == lib.PKVQK_OK
    assert lib.pkvqk_last_error().decode() == ""


def test_partials_need_explicit_splits(lib):
    lay = _layout(lib)
    r = lib.pkvqk_paged_decode_partials(FAKE, 2048, 128, FAKE, FAKE, ctypes.byref(lay), FAKE, 16,
                                        FAKE, 4, 1, 16, 1, 256, 0.0, FAKE, 1 << 20, None, None)
    assert r == lib.PKVQK_ERR_INVALID_ARG


def test_append_validation_errors(lib):
    lay = _layout(lib)

    def call(theta=1e6, eps=1e-6, T=4, Hq=16, lay=lay, qst=2048):
        return lib.pkvqk_norm_rope_append(FAKE, qst, 128, FAKE, 1024, 128, FAKE, 1024, 128,
                                          FAKE, FAKE, FAKE, FAKE, theta, eps, T, Hq, FAKE, FAKE,
                                          ctypes.byref(lay), None, None)
    assert call(theta=0.0) == lib.PKVQK_ERR_INVALID_ARG
    assert call(theta=float("nan")) == lib.PKVQK_ERR_INVALID_ARG
    assert call(eps=-1.0) == lib.PKVQK_ERR_INVALID_ARG
    assert call(T=-1) == lib.PKVQK_ERR_INVALID_ARG
    assert call(Hq=0) == lib.PKVQK_ERR_INVALID_ARG
    assert call(qst=2047) == lib.PKVQK_ERR_INVALID_ARG
    assert call(lay=_layout(lib, d=256)) == lib.PKVQK_ERR_UNSUPPORTED
    assert call(T=0) == lib.PKVQK_OK


def test_combine_validation_errors(lib):
    c = lib.pkvqk_lse_combine
    assert c(FAKE, FAKE, 4, 64, 2, FAKE, None, None) == lib.PKVQK_ERR_UNSUPPORTED
    assert c(FAKE, FAKE, -1, 128, 2, FAKE, None, None) == lib.PKVQK_ERR_INVALID_ARG
    assert c(FAKE, FAKE, 4, 128, 0, FAKE, None, None) == lib.PKVQK_ERR_INVALID_ARG
    assert c(FAKE, FAKE, 0, 128, 2, FAKE, None, None) == lib.PKVQK_OK


def test_workspace_bytes_formula(lib):
    assert lib.decode_workspace_bytes(4, 1, 16, 128, 1) == 0
    assert lib.decode_workspace_bytes(4, 1, 16, 128, 0) > 0       # balanced schedule bound
    for B, T, Hq, S in [(4, 1, 16, 4), (64, 1, 16, 19), (32, 5, 16, 8), (1, 1, 8, 2)]:
        # partials [rows][S][128] + lse [rows][S]
        raw = B * T * Hq * S * 129 * 4
        assert lib.decode_workspace_bytes(B, T, Hq, 128, S) == (raw + 255) // 256 * 256
    assert lib.decode_workspace_bytes(4, 1, 16, 64, 4) == 0
    # balanced bound: ((SMs + batch) q_len Hq (D + 1) 4 + batch Hq 8), the first
    # part 16-byte aligned, rounded up to 256; without a GPU the library assumes
    # 148 SMs
    for B, T, Hq in [(4, 1, 16), (64, 1, 32), (32, 5, 16), (1, 1, 8)]:
        doc = (148 + B) * T * Hq * 129 * 4 + B * Hq * 8
        got = lib.decode_workspace_bytes(B, T, Hq, 128, 0)
        assert doc <= got <= doc + 16 + 255 and got % 256 == 0


def test_split_heuristic_is_host_only_and_bounded(lib):
    for B, hkv, rows, L, sms in [(1, 8, 2, 512, 148), (64, 8, 2, 8192, 152), (8, 8, 2, 32768, 152),
                                 (64, 4, 8, 16384, 152), (32, 8, 10, 8197, 152), (4, 8, 2, 1, 152)]:
        S = lib.choose_num_splits(B, hkv, rows, L, B * L, 16, sms)
        assert 1 <= S <= 256                      # uniform lengths: a split count
        assert S <= max(1, -(-L // 16))           # never more splits than pages
    # a single long sequence is spread over many splits; a full batch is not split much
    assert lib.choose_num_splits(8, 8, 2, 32768, 8 * 32768, 16, 152) >= 8
    assert lib.choose_num_splits(1, 8, 2, 512, 512, 16, 152) >= 2
    assert lib.choose_num_splits(0, 8, 2, 512, 0, 16, 152) == 1
    # large batch of strongly mixed lengths (under half of batch x max keys):
    # the balanced schedule
    assert lib.choose_num_splits(64, 4, 8, 16384, 230000, 16, 152) == 0
    # a milder mix (the speculative-verify batch, ~0.65 of batch x max keys):
    # the split count, rounded to the nearest
    assert lib.choose_num_splits(32, 8, 10, 8197, 172000, 16, 152) == 6
    # small mixed batch: still a split count
    assert lib.choose_num_splits(4, 8, 2, 256, 600, 16, 152) >= 1


def test_split_heuristic_above_16_rows_is_the_tensor_core_choice(lib):
    # above 16 rows per kv head pkvqk_paged_decode runs the multi-query
    # tensor-core kernel, so the chooser gives that kernel's split count
    # (never the balanced schedule, which that kernel does not have)
    for B, hkv, rows, L in [(4, 8, 40, 8192), (1, 8, 24, 512), (64, 8, 40, 16384),
                            (32, 4, 128, 8197)]:
        S = lib.choose_num_splits(B, hkv, rows, L, B * L // 2, 16, 152)
        assert S == lib.choose_prefill_splits(B, hkv, rows, 1, L, 152)
        assert S >= 1


def test_static_ws_reports_argument_errors_before_its_capacity(lib):
    # arguments pkvqk_paged_decode rejects come back as argument errors from
    # the static-workspace entry point too, even where their partials would
    # also overflow its fixed array (16 MiB)
    lay = _layout(lib)

    def call(B=4, q_len=1, Hq=16, S=1, lay=lay):
        return lib.pkvqk_paged_decode_static_ws(FAKE, 2048, 128, FAKE, FAKE, ctypes.byref(lay),
                                                FAKE, 16, FAKE, B, q_len, Hq, S, 256, 0.0, FAKE,
                                                None, None, None)
    assert call(B=4096, S=300) == lib.PKVQK_ERR_INVALID_ARG            # num_splits > 256
    assert "num_splits" in lib.pkvqk_last_error().decode()
    assert call(B=4096, q_len=17, S=200) == lib.PKVQK_ERR_INVALID_ARG  # q_len > 16
    assert call(B=4096, Hq=12, S=200) == lib.PKVQK_ERR_INVALID_ARG     # Hq % Hkv != 0
    assert call(lay=_layout(lib, d=64)) == lib.PKVQK_ERR_UNSUPPORTED
    # a valid call whose partials do not fit is refused before any launch
    assert call(B=4096, S=200) == lib.PKVQK_ERR_WORKSPACE_TOO_SMALL
    assert call(B=0, S=4) == lib.PKVQK_OK


def test_rope_table_size_and_argument_errors(lib):
    # 1 KiB per position (16 lanes x 4 float4s), nothing outside 1 .. 2^21
    assert lib.rope_table_bytes(1) == 1024
    assert lib.rope_table_bytes(40960) == 40960 * 1024
    assert lib.rope_table_bytes(0) == 0 and lib.rope_table_bytes(-3) == 0
    assert lib.rope_table_bytes((1 << 21) + 1) == 0
    b = lib.pkvqk_rope_table_build
    assert b(FAKE, -1, 1e6, None) == lib.PKVQK_ERR_INVALID_ARG
    assert b(FAKE, (1 << 21) + 1, 1e6, None) == lib.PKVQK_ERR_INVALID_ARG
    assert b(FAKE, 16, 0.0, None) == lib.PKVQK_ERR_INVALID_ARG
    assert b(FAKE, 16, float("nan"), None) == lib.PKVQK_ERR_INVALID_ARG
    assert b(FAKE, 0, 1e6, None) == lib.PKVQK_OK           # nothing to build
    lay = _layout(lib)

    def cached(table_positions, theta=1e6, T=4):
        return lib.pkvqk_norm_rope_append_cached(FAKE, 2048, 128, FAKE, 1024, 128, FAKE, 1024,
                                                 128, FAKE, FAKE, FAKE, FAKE, theta, 1e-6, T, 16,
                                                 FAKE, FAKE, ctypes.byref(lay), FAKE,
                                                 table_positions, None, None)
    assert cached(-1) == lib.PKVQK_ERR_INVALID_ARG
    assert cached((1 << 21) + 1) == lib.PKVQK_ERR_INVALID_ARG
    assert cached(16, theta=0.0) == lib.PKVQK_ERR_INVALID_ARG  # the append's own checks follow
    assert cached(16, T=0) == lib.PKVQK_OK
