"""Plain fp64 CPU oracle for sparse MLA decode over fp8_ds_mla records.

TEST INFRASTRUCTURE ONLY.  This module is the independent checker of the CUDA
path.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may import it.  It shares
no code, table or constant generator with ``sparse_mla_decode_csr_gb300``; the
CUDA path never imports it and never falls back to it.

Every function is written from the definitions on the pages, in numpy float64,
with no blocking, fusion or reordering beyond what the definition states:

* [P1] "vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla_gfx950" (FlyDSL sparse
  MLA forward over fp8_ds_mla records, gfx950): module docstring (record
  layout, tiles/masking, preconditions, writer scale rule) and the epilogue of
  ``build_sparse_mla_fp8ds_module`` (normalisation, LSE definition).
* [P2] "vllm.models.deepseek_v41.amd.mono.attention.back" (K2 back):
  ``stage_split`` (per-chunk partial, max and sum) and ``stage_combine``
  (chunk merge with the per-head sink).
* E4M3 follows the OCP 8-bit floating point specification (E4M3, "fn"
  variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
  subnormals at exponent 0, no infinities, S.1111.111 is NaN, max 448.  The
  448 and 57344 constants of the [P1] writer rule are this format's.

Readings where the pages are silent (c-numbers as in the design notes):

* c1  positions >= len and entries < 0 are masked, with or without has_invalid.
* c2  an entry >= n_kv_rows is masked like -1 (the pages leave it undefined).
* c2b a position whose offset into ``indices`` falls outside [0, n_indices) is
      masked (the [P1] bounded index view makes such reads harmless).
* c3  a row with no valid key gives out = 0 and lse = -inf, sink or not.
* c4  duplicates inside a row count once per position.
* c5  the LSE excludes the sink; the sink only enlarges the denominator.
* c6  the sink is in the natural-log units of sm_scale * q.k.
* c9  the writer rounds x / scale to E4M3 round-to-nearest-even, saturating.
* c11 a zero scale gives a zero latent; the key still attends through rope.
* lens: effective length = min(slice length, max(lens[q], 0)).

Parity is pinned for every function here (tests/test_oracle_pins.py); no
function is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

# --- record layout, [P1] module docstring ("Record (656 B): 512 e4m3 latent |
# 4 f32 per-128 pow2 scales | 64 bf16 rope").
RECORD_BYTES = 656
LATENT_DIM = 512
ROPE_DIM = 64
QK_DIM = LATENT_DIM + ROPE_DIM
SCALE_BLOCK = 128
N_SCALES = LATENT_DIM // SCALE_BLOCK
SCALE_OFFSET = LATENT_DIM  # bytes [512, 528): 4 little-endian f32
ROPE_OFFSET = SCALE_OFFSET + 4 * N_SCALES  # bytes [528, 656): 64 bf16

# --- writer constants, [P1] module docstring, "Preconditions": scale =
# pow2ceil(max(amax, 1e-4) / 448).
E4M3_MAX = 448.0
WRITER_AMAX_FLOOR = 1e-4


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Value of one OCP E4M3 code (the 'fn' variant, bias 7, no infinities)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:  # subnormal: (man / 8) * 2^(1 - 7)
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def e4m3_table() -> np.ndarray:
    """All 256 E4M3 code values as float64 (NaN for the two NaN codes)."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


_E4M3 = e4m3_table()
# Finite non-negative codes 0x00..0x7E, whose values increase with the code.
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = _E4M3[:0x7F]


def e4m3_encode_rne(x: np.ndarray) -> np.ndarray:
    """Round float64 values to E4M3 codes: nearest, ties to even, saturating.

    Reading c9: the pages fix the writer's scale but not its rounding; this
    takes round-to-nearest-even and saturates magnitudes above 448 (which the
    writer's scale never produces).
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")  # first value >= a
    hi = np.clip(hi, 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_hi = d_hi < d_lo
    tie = d_hi == d_lo
    even_hi = (_POS_CODES[hi] & 1) == 0
    pick_hi = np.where(tie, even_hi, pick_hi)
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(np.isnan(x), 0x7F, code)
    code = code | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64: bf16 is the top half of f32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits_exact(x: np.ndarray) -> np.ndarray:
    """float64 values that are exactly bf16 to their bit patterns (asserts)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32)
    if np.any(bits & np.uint32(0xFFFF)):
        raise ValueError("value is not representable in bf16")
    return (bits >> np.uint32(16)).astype(np.uint16)


def pow2ceil(y: np.ndarray) -> np.ndarray:
    """Smallest power of two >= y, for y > 0 (exact: powers of two map to themselves)."""
    y = np.asarray(y, dtype=np.float64)
    m, e = np.frexp(y)  # y = m * 2^e, m in [0.5, 1)
    return np.where(m == 0.5, y, np.ldexp(1.0, e))


# ---------------------------------------------------------------------------
# Record writer and reader, [P1] module docstring ("Record", "Preconditions")
# ---------------------------------------------------------------------------

def writer_scales(latent: np.ndarray) -> np.ndarray:
    """Per-128 scale = pow2ceil(max(amax, 1e-4) / 448) for latent [N, 512]."""
    blocks = np.abs(np.asarray(latent, dtype=np.float64)).reshape(-1, N_SCALES, SCALE_BLOCK)
    amax = blocks.max(axis=2)
    return pow2ceil(np.maximum(amax, WRITER_AMAX_FLOOR) / E4M3_MAX)


def pack_records(latent_bf16: np.ndarray, rope_bf16: np.ndarray) -> np.ndarray:
    """Writer: bf16 latent [N, 512] and bf16 rope [N, 64] (uint16 bits) -> uint8 [N, 656].

    Bytes [0, 512) = E4M3(latent / scale_b) with b = d // 128; bytes [512, 528)
    = the 4 scales as little-endian f32; bytes [528, 656) = the rope bf16 bits
    verbatim.
    """
    latent_bits = np.asarray(latent_bf16, dtype=np.uint16)
    rope_bits = np.asarray(rope_bf16, dtype=np.uint16)
    n = latent_bits.shape[0]
    assert latent_bits.shape == (n, LATENT_DIM) and rope_bits.shape == (n, ROPE_DIM)
    x = bf16_to_f64(latent_bits)
    scales = writer_scales(x)  # [N, 4]
    per_dim = np.repeat(scales, SCALE_BLOCK, axis=1)  # [N, 512]
    codes = e4m3_encode_rne(x / per_dim)
    rec = np.zeros((n, RECORD_BYTES), dtype=np.uint8)
    rec[:, :LATENT_DIM] = codes
    rec[:, SCALE_OFFSET:ROPE_OFFSET] = scales.astype("<f4").view(np.uint8).reshape(n, 16)
    rec[:, ROPE_OFFSET:] = rope_bits.astype("<u2").view(np.uint8).reshape(n, 2 * ROPE_DIM)
    return rec


def unpack_records(rec: np.ndarray):
    """Reader: uint8 [N, 656] -> (latent [N, 512], rope [N, 64], scales [N, 4]) in float64.

    latent_d = e4m3(byte_d) * scale_{d // 128}; rope = bf16 (exact in float64).
    """
    rec = np.asarray(rec, dtype=np.uint8)
    n = rec.shape[0]
    scales = np.ascontiguousarray(rec[:, SCALE_OFFSET:ROPE_OFFSET]).view("<f4").astype(np.float64)
    scales = scales.reshape(n, N_SCALES)
    codes = rec[:, :LATENT_DIM]
    latent = _E4M3[codes] * np.repeat(scales, SCALE_BLOCK, axis=1)
    rope_bits = np.ascontiguousarray(rec[:, ROPE_OFFSET:]).view("<u2").reshape(n, ROPE_DIM)
    rope = bf16_to_f64(rope_bits)
    return latent, rope, scales


# ---------------------------------------------------------------------------
# Decode: the plain definition of masked sparse softmax attention
# ---------------------------------------------------------------------------

def row_positions(r: int, indices, indptr, lens, n_kv_rows: int):
    """Row r's valid keys as (positions, kv row ids), [P1] "Tiles" paragraph.

    Slice = indices[indptr[r] : indptr[r + 1]], length clamped at 0; lens (if
    given) caps it (reading for lens).  Position p is valid when its offset
    lies inside the index buffer (c2b) and 0 <= indices[offset] < n_kv_rows
    (c1, c2).
    """
    beg = int(indptr[r])
    end = int(indptr[r + 1])
    length = max(end - beg, 0)
    if lens is not None:
        length = min(length, max(int(lens[r]), 0))
    pos, ids = [], []
    n_idx = len(indices)
    for p in range(length):
        off = beg + p
        if off < 0 or off >= n_idx:
            continue
        idx = int(indices[off])
        if 0 <= idx < n_kv_rows:
            pos.append(p)
            ids.append(idx)
    return np.array(pos, dtype=np.int64), np.array(ids, dtype=np.int64)


def row_keys(kv: np.ndarray, ids: np.ndarray):
    """K [n, 576] (dequantised latent then rope) and V [n, 512] (latent) of the ids."""
    latent, rope, _ = unpack_records(kv[ids])
    return np.concatenate([latent, rope], axis=1), latent


def row_scores(q_row: np.ndarray, keys: np.ndarray, sm_scale: float) -> np.ndarray:
    """s[h, t] = sm_scale * sum_{d < 576} q[h, d] * k[t, d]  ([P1] QK over 576 dims)."""
    return float(sm_scale) * (q_row @ keys.T)


def softmax_out(scores: np.ndarray, values: np.ndarray, sink):
    """Masked softmax attention of one row over its valid keys.

    m = max_t s; l = sum_t exp(s - m); lse = m + ln l ([P1] epilogue: natural-log
    LSE over unmasked keys, sink excluded (c5)).  The sink enters the output
    denominator the way [P2] stage_combine folds it:
    m_f = max(m, sink), den = exp(sink - m_f) + l * exp(m - m_f),
    out = sum_t exp(s - m) v_t * exp(m - m_f) / den.
    No key: out = 0, lse = -inf (c3).
    """
    h = scores.shape[0]
    if scores.shape[1] == 0:
        return np.zeros((h, LATENT_DIM)), np.full(h, -np.inf)
    m = scores.max(axis=1)
    e = np.exp(scores - m[:, None])
    l = e.sum(axis=1)
    lse = m + np.log(l)
    acc = e @ values  # [H, 512]
    if sink is None:
        return acc / l[:, None], lse
    sink = np.asarray(sink, dtype=np.float64)
    m_f = np.maximum(m, sink)
    den = np.exp(sink - m_f) + l * np.exp(m - m_f)
    return acc * (np.exp(m - m_f) / den)[:, None], lse


def sparse_mla_decode(q, kv, indices, indptr, lens=None, sm_scale=1.0 / 24.0,
                      sink=None, n_kv_rows=None, rows=None):
    """The whole decode: out [n_q, H, 512], lse [n_q, H], n_valid [n_q] (float64/int64).

    q: float64 [n_q, H, 576] (exact bf16 values); kv: uint8 [n_kv_rows, 656];
    indices/indptr/lens: int arrays; sink: float [H] or None.  ``rows``
    restricts the computation to a subset of rows (the others stay 0 / -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, n_heads, _ = q.shape
    if n_kv_rows is None:
        n_kv_rows = kv.shape[0]
    out = np.zeros((n_q, n_heads, LATENT_DIM))
    lse = np.full((n_q, n_heads), -np.inf)
    n_valid = np.zeros(n_q, dtype=np.int64)
    for r in (range(n_q) if rows is None else rows):
        _, ids = row_positions(r, indices, indptr, lens, n_kv_rows)
        n_valid[r] = len(ids)
        keys, values = row_keys(kv, ids)
        s = row_scores(q[r], keys, sm_scale)
        out[r], lse[r] = softmax_out(s, values, sink)
    return out, lse, n_valid


# ---------------------------------------------------------------------------
# Split-KV flash decoding: per-chunk partials and their combine, [P2]
# ---------------------------------------------------------------------------

def split_partials(q, kv, indices, indptr, lens=None, sm_scale=1.0 / 24.0,
                   chunk_len=128, n_chunks=None, n_kv_rows=None, rows=None):
    """Per (row, chunk) partials, [P2] stage_split.

    Chunk c of a row covers slice positions [c * chunk_len, (c + 1) * chunk_len).
    For each head: m_c = max of the chunk's valid scores, l_c = sum exp(s - m_c),
    O_c = sum exp(s - m_c) * v (unnormalised).  A chunk with no valid key has
    m_c = -inf, l_c = 0, O_c = 0.  Returns O [n_q, C, H, 512], m [n_q, C, H],
    l [n_q, C, H], n_valid [n_q, C].
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, n_heads, _ = q.shape
    if n_kv_rows is None:
        n_kv_rows = kv.shape[0]
    if n_chunks is None:
        longest = max([max(int(indptr[r + 1]) - int(indptr[r]), 0) for r in range(n_q)] + [0])
        n_chunks = max(1, -(-longest // chunk_len))
    o_part = np.zeros((n_q, n_chunks, n_heads, LATENT_DIM))
    m_part = np.full((n_q, n_chunks, n_heads), -np.inf)
    l_part = np.zeros((n_q, n_chunks, n_heads))
    n_valid = np.zeros((n_q, n_chunks), dtype=np.int64)
    for r in (range(n_q) if rows is None else rows):
        pos, ids = row_positions(r, indices, indptr, lens, n_kv_rows)
        for c in range(n_chunks):
            sel = (pos >= c * chunk_len) & (pos < (c + 1) * chunk_len)
            n_valid[r, c] = int(sel.sum())
            if not sel.any():
                continue
            keys, values = row_keys(kv, ids[sel])
            s = row_scores(q[r], keys, sm_scale)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            m_part[r, c] = m
            l_part[r, c] = e.sum(axis=1)
            o_part[r, c] = e @ values
    return o_part, m_part, l_part, n_valid


def combine(o_part, m_part, l_part, sink=None):
    """Merge chunk partials into (out, lse), [P2] stage_combine.

    m* = max_c m_c; w_c = exp(m_c - m*); l = sum_c l_c w_c; lse = m* + ln l
    (sink excluded, c5).  m_f = max(m*, sink); den = exp(sink - m_f) +
    l exp(m* - m_f); out = sum_c O_c w_c exp(m* - m_f) / den.  Rows whose
    chunks are all empty give 0 / -inf.
    """
    n_q, _, n_heads, _ = o_part.shape
    out = np.zeros((n_q, n_heads, LATENT_DIM))
    lse = np.full((n_q, n_heads), -np.inf)
    for r in range(n_q):
        for h in range(n_heads):
            mc = m_part[r, :, h]
            live = np.isfinite(mc)
            if not live.any():
                continue
            m_star = mc[live].max()
            w = np.exp(mc[live] - m_star)
            l = float((l_part[r, live, h] * w).sum())
            acc = (o_part[r, live, h, :] * w[:, None]).sum(axis=0)
            lse[r, h] = m_star + math.log(l)
            if sink is None:
                out[r, h] = acc / l
            else:
                s = float(sink[h])
                m_f = max(m_star, s)
                den = math.exp(s - m_f) + l * math.exp(m_star - m_f)
                out[r, h] = acc * (math.exp(m_star - m_f) / den)
    return out, lse
