"""Plain fp64 definitions of the paged decode-attention hot path.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Slow on purpose: no
blocking, fusion or reordering beyond what each definition states.  bf16 data
travels as raw uint16 bit patterns; every computation is float64.

Operations, with the page passage each follows (InfiniLM PR #585, "perf: Qwen3
offline inference — hybrid attention backend, fused rms_norm_rope, chunked
prefill + prompt-lookup spec decoding", section "概述 / Summary"):

* ``rms_norm``        — Summary item 2, "per-head RMSNorm" (section "依赖与 CI").
* ``rope_neox``       — Summary item 2, "full-rotary" RoPE.
* ``norm_rope_append``— Summary items 1+2: norm + RoPE on q and k, then k and v
                        written into the BSHD paged cache.
* ``paged_attention`` — Summary item 1, the pure-decode attention over the
                        paged cache; item 4 for the k+1-token verify shape.
* ``split_page_ranges``, ``paged_attention_splits``, ``lse_combine``
                      — Summary item 1, "splitkv": the KV range of a sequence
                        is cut into splits whose partial softmax results merge
                        by log-sum-exp.

Readings taken where the pages are silent (each is stated again where used):

R1  RMSNorm gain is multiplicative: y = x / sqrt(mean(x^2) + eps) * gamma
    (Qwen3 convention; the (1 + w) Gemma gain on the Ascend page belongs to a
    different model).
R2  Norm first, then RoPE ("rms_norm_rope"); no rounding between them; q and
    k are rounded once to bf16 (round-to-nearest-even) after RoPE.
R3  neox rotate-half pairing (i, i + D/2), inv_freq_i = theta^(-2i/D),
    i in [0, D/2), rotary over the whole head (full rotary).
R4  Decode position of the new token is seq_len - 1; verify token t of a
    q_len-token step sits at seq_len - q_len + t.
R5  Softmax scale defaults to D^-1/2.
R6  GQA: q head h reads kv head h // (Hq / Hkv).
R7  A slot outside [0, num_blocks * block_size) (negative = padding) writes
    nothing.
R8  v is appended unchanged (only q and k are normalised and rotated).
R9  Verify is causal: query t sees keys n < seq_len - q_len + t + 1.
R10 A split (or a sequence) with no visible key contributes o = 0 and
    lse = -inf; a row with no key at all outputs 0 and lse = -inf.
R11 Split partition: with chunk C pages, split j covers pages
    [j*C, (j+1)*C) for j < S-1 and [(S-1)*C, P) for j = S-1, clipped to the
    sequence's P = ceil(seq_len / block_size) pages.  The combined result
    does not depend on the partition (up to rounding).
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "rms_norm",
    "rope_neox",
    "norm_rope_append",
    "paged_attention",
    "split_page_ranges",
    "paged_attention_splits",
    "lse_combine",
]


# --------------------------------------------------------------------------
# bf16 <-> float64
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly.

    A bf16 value is the top half of an IEEE binary32 with the low 16 bits zero.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):          # NaN patterns widen to NaN
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 to bf16 once, round-to-nearest-even (IEEE 754).

    bf16 keeps 8 significant bits and binary32's exponent range.  For finite
    |x| = m * 2^e with m in [0.5, 1), the spacing of bf16 values around |x| is
    2^(e-8), floored at the subnormal spacing 2^-133.  Dividing by a power of
    two is exact in float64, so np.rint (ties to even) applied to |x| / q gives
    the correctly rounded multiple of q in a single rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    finite = np.isfinite(x)
    _, e = np.frexp(np.where(finite & (ax > 0), ax, 1.0))
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    r = np.rint(ax / q) * q
    r = np.where(finite, r, ax)
    r = np.where(r >= 2.0 ** 128, np.inf, r)          # overflow rounds to inf
    r = np.copysign(r, x)
    r32 = r.astype(np.float32)                        # exact: r is a bf16 value
    bits = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits


# --------------------------------------------------------------------------
# per-head RMSNorm and neox RoPE
# --------------------------------------------------------------------------

def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """Per-head RMSNorm over the last axis (reading R1).

    y = x / sqrt(mean(x^2) + eps) * gamma, gamma broadcast over heads.
    """
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, np.float64)


def rope_neox(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """neox rotate-half RoPE over the last axis (reading R3).

    x has shape [..., D]; pos broadcasts against x's leading axes (one position
    per vector).  Pair (i, i + D/2) is rotated by angle pos * theta^(-2i/D).
    """
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = np.float64(theta) ** (-2.0 * i / D)
    ang = np.asarray(pos, np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def norm_rope_append(q, k, v, positions, slot_mapping, gamma_q, gamma_k,
                     theta, eps, k_cache, v_cache, block_size):
    """Fused per-head RMSNorm + RoPE on q and k, then k/v written to the cache.

    q: uint16 [T, Hq, D]; k, v: uint16 [T, Hkv, D]; positions, slot_mapping:
    int [T]; gamma_q, gamma_k: uint16 [D]; caches: uint16 [NB, bs, Hkv, D].

    Returns (q_hat_bits [T, Hq, D], k_cache_new, v_cache_new, k_hat_f64,
    q_hat_f64).  The caches are copies; inputs are not modified.  q_hat_f64 /
    k_hat_f64 are the unrounded float64 results (for error analysis).

    Steps (readings R1-R3, R7, R8): widen to float64; RMSNorm with the head's
    gamma; RoPE at positions[t]; round once to bf16; for each t with a valid
    slot s, k_cache[s // bs, s % bs, :, :] = k_hat[t], v_cache[...] = v[t].
    """
    eps64 = np.float64(np.float32(eps))
    theta64 = np.float64(np.float32(theta))
    pos = np.asarray(positions, np.int64)
    qf = bf16_bits_to_f64(q)
    kf = bf16_bits_to_f64(k)
    gq = bf16_bits_to_f64(gamma_q)
    gk = bf16_bits_to_f64(gamma_k)
    q_hat = rope_neox(rms_norm(qf, gq, eps64), pos[:, None], theta64)
    k_hat = rope_neox(rms_norm(kf, gk, eps64), pos[:, None], theta64)
    q_bits = f64_to_bf16_bits(q_hat)
    k_bits = f64_to_bf16_bits(k_hat)

    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    nslots = kc.shape[0] * block_size
    v = np.asarray(v, np.uint16)
    for t, s in enumerate(np.asarray(slot_mapping, np.int64).tolist()):
        if s < 0 or s >= nslots:
            continue
        blk, off = s // block_size, s % block_size
        kc[blk, off] = k_bits[t]
        vc[blk, off] = v[t]
    return q_bits, kc, vc, k_hat, q_hat


# --------------------------------------------------------------------------
# paged attention
# --------------------------------------------------------------------------

def _gather_rows(cache_bits, block_table_row, key_idx, block_size, kv_head):
    """Explicit page gather: key n lives at cache[block_table[n // bs], n % bs]."""
    blocks = np.asarray(block_table_row, np.int64)[key_idx // block_size]
    offs = key_idx % block_size
    return bf16_bits_to_f64(cache_bits[blocks, offs, kv_head, :])


def _softmax_attend(qvec, K, V, scale):
    """Dense softmax attention of rows qvec [R, D] over keys K, V [n, D].

    Returns (out [R, D], lse [R]); no key -> out 0, lse -inf (reading R10).
    """
    R, D = qvec.shape
    if K.shape[0] == 0:
        return np.zeros((R, D)), np.full(R, -np.inf)
    s = scale * (qvec @ K.T)                       # [R, n]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ V) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, block_size,
                    q_len=1, scale=None, seqs=None):
    """Softmax attention of each query over its sequence's paged keys.

    q: uint16 [B, q_len, Hq, D]; caches uint16 [NB, bs, Hkv, D];
    block_tables int [B, maxP]; seq_lens int [B] (counting the q_len new
    tokens).  Query t of sequence b sees keys n = 0 .. seq_len - q_len + t
    (reading R9; q_len = 1 is plain decode) of kv head h // G (R6), gathered
    page by page through the block table.  No split.

    ``seqs`` optionally restricts the work to a subset of sequence indices
    (rows of other sequences are left as NaN).

    Returns (out float64 [B, q_len, Hq, D], lse float64 [B, q_len, Hq]).
    """
    q = np.asarray(q, np.uint16)
    B, T, Hq, D = q.shape
    assert T == q_len
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = D ** -0.5
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    qf = bf16_bits_to_f64(q)
    bt = np.asarray(block_tables, np.int64)
    sl = np.asarray(seq_lens, np.int64)
    for b in (range(B) if seqs is None else seqs):
        for t in range(T):
            ctx = int(sl[b]) - T + t + 1
            keys = np.arange(max(ctx, 0), dtype=np.int64)
            for g in range(Hkv):
                K = _gather_rows(k_cache, bt[b], keys, block_size, g)
                V = _gather_rows(v_cache, bt[b], keys, block_size, g)
                rows = qf[b, t, g * G:(g + 1) * G, :]
                o, ls = _softmax_attend(rows, K, V, scale)
                out[b, t, g * G:(g + 1) * G] = o
                lse[b, t, g * G:(g + 1) * G] = ls
    return out, lse


def split_page_ranges(num_pages: int, num_splits: int, chunk_pages: int):
    """Page range [p0, p1) of every split of a sequence with num_pages pages.

    Reading R11: split j < S-1 covers [j*C, (j+1)*C); split S-1 covers
    [(S-1)*C, num_pages); each range is clipped to [0, num_pages).
    """
    out = []
    for j in range(num_splits):
        p0 = j * chunk_pages
        p1 = num_pages if j == num_splits - 1 else (j + 1) * chunk_pages
        p0, p1 = min(p0, num_pages), min(p1, num_pages)
        out.append((p0, max(p0, p1)))
    return out


def paged_attention_splits(q, k_cache, v_cache, block_tables, seq_lens,
                           block_size, num_splits, chunk_pages, q_len=1,
                           scale=None):
    """Per-split partial attention (split-KV), each split over its page range.

    Returns (o float64 [B, q_len, Hq, S, D], lse float64 [B, q_len, Hq, S]):
    o is the split's normalised partial output and lse its log-sum-exp; empty
    splits give o = 0, lse = -inf (reading R10).
    """
    q = np.asarray(q, np.uint16)
    B, T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = D ** -0.5
    S = num_splits
    o = np.zeros((B, T, Hq, S, D))
    lse = np.full((B, T, Hq, S), -np.inf)
    qf = bf16_bits_to_f64(q)
    bt = np.asarray(block_tables, np.int64)
    for b in range(B):
        L = int(seq_lens[b])
        P = -(-L // block_size)
        for j, (p0, p1) in enumerate(split_page_ranges(P, S, chunk_pages)):
            for t in range(T):
                ctx = L - T + t + 1
                lo, hi = p0 * block_size, min(p1 * block_size, max(ctx, 0))
                keys = np.arange(lo, max(lo, hi), dtype=np.int64)
                for g in range(Hkv):
                    K = _gather_rows(k_cache, bt[b], keys, block_size, g)
                    V = _gather_rows(v_cache, bt[b], keys, block_size, g)
                    rows = qf[b, t, g * G:(g + 1) * G, :]
                    oo, ll = _softmax_attend(rows, K, V, scale)
                    o[b, t, g * G:(g + 1) * G, j] = oo
                    lse[b, t, g * G:(g + 1) * G, j] = ll
    return o, lse


def lse_combine(o, lse):
    """Merge split partials by log-sum-exp over the split axis.

    o: [..., S, D], lse: [..., S].  M = max_j lse_j; w_j = exp(lse_j - M);
    out = sum_j w_j o_j / sum_j w_j; lse = M + log(sum_j w_j).  Splits with
    lse = -inf carry weight 0; if every split is empty the row outputs 0 and
    lse = -inf (reading R10).
    """
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    M = lse.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(M)
    Ms = np.where(empty, 0.0, M)
    w = np.where(np.isfinite(lse), np.exp(lse - Ms), 0.0)
    wsum = w.sum(axis=-1, keepdims=True)
    safe = np.where(wsum > 0, wsum, 1.0)
    out = (w[..., None] * o).sum(axis=-2) / safe
    out = np.where(empty, 0.0, out)
    lse_out = np.where(empty[..., 0], -np.inf, (Ms + np.log(safe))[..., 0])
    return out, lse_out
