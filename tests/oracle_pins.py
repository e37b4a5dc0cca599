"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each ``pin_*`` takes the oracle module and raises AssertionError on a
mismatch.  None of them re-types the oracle's formulas: they compare against
library routines (torch's float8_e4m3fn / bfloat16 views, torch.softmax),
hand-worked values (tests/golden), closed forms and invariants.  The
mutation tests plant plausible mistakes in the oracle and check that at least
one pin fails for each.
"""

from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# independent helpers (torch dtype views; no oracle code)
# ---------------------------------------------------------------------------

def torch_decode_records(rec: np.ndarray):
    """K [N, 576] and V [N, 512] of records decoded with torch's own dtype views."""
    t = torch.from_numpy(np.ascontiguousarray(rec))
    lat = t[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    sc = t[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
    lat = lat * sc.repeat_interleave(128, dim=1)
    rope = t[:, 528:656].contiguous().view(torch.bfloat16).to(torch.float64)
    return torch.cat([lat, rope], dim=1).numpy(), lat.numpy()


def random_records(n: int, seed: int, scale_exp=(-10, -5)) -> np.ndarray:
    """Records with random non-NaN E4M3 codes, random power-of-two scales and
    random bf16 rope (a direct draw of the byte format, no writer involved)."""
    rng = np.random.default_rng(seed)
    rec = np.zeros((n, 656), dtype=np.uint8)
    codes = rng.integers(0, 256, size=(n, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3F
    rec[:, :512] = codes
    exps = rng.integers(scale_exp[0], scale_exp[1] + 1, size=(n, 4))
    scales = np.ldexp(np.ones((n, 4), dtype=np.float32), exps).astype("<f4")
    rec[:, 512:528] = scales.view(np.uint8).reshape(n, 16)
    rope = torch.randn(n, 64, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    rec[:, 528:] = rope.view(torch.uint8).numpy().reshape(n, 128)
    return rec


def random_q(n_q: int, heads: int, seed: int, std=0.05) -> np.ndarray:
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(n_q, heads, 576, generator=g) * std).to(torch.bfloat16)
    return q.to(torch.float64).numpy()


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def pin_e4m3_table(orc):
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    got = orc.e4m3_table()
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "E4M3 NaN codes differ"
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "E4M3 code values differ from torch.float8_e4m3fn"


def pin_e4m3_encode(orc):
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = vals.to(torch.float64).numpy()
    finite = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (finite[1:] + finite[:-1]) / 2.0  # exact ties (float64)
    rng = np.random.default_rng(7)
    rand = rng.uniform(-448, 448, 20000) * np.exp2(-rng.integers(0, 14, 20000))
    x = np.concatenate([finite, mids, -mids, rand])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode_rne(x)
    assert np.array_equal(got, ref), "E4M3 rounding differs from torch (RNE)"


def pin_bf16(orc):
    bits = np.arange(0, 1 << 16, 97, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = orc.bf16_to_f64(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~ok) and np.array_equal(got[ok], ref[ok])


def pin_pow2ceil(orc):
    k = np.arange(-30, 20)
    p = np.ldexp(1.0, k)
    assert np.array_equal(orc.pow2ceil(p), p), "powers of two must map to themselves"
    assert np.array_equal(orc.pow2ceil(p * (1 + 2 ** -40)), 2 * p)
    assert np.array_equal(orc.pow2ceil(p * 0.75), p)
    assert float(orc.pow2ceil(np.array([3.0 / 448]))[0]) == 2.0 ** -7


# ---------------------------------------------------------------------------
# writer / reader
# ---------------------------------------------------------------------------

def load_golden_writer():
    lat = np.zeros(512)
    rope = np.zeros(64)
    want = np.zeros(656, dtype=np.uint8)
    deq = np.zeros(512)
    with open(os.path.join(GOLDEN, "writer_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, a, b = line.split()
            if kind == "latent":
                lat[int(a)] = float(b)
            elif kind == "rope":
                rope[int(a)] = float(b)
            elif kind == "byte":
                want[int(a)] = int(b, 16)
            elif kind == "dequant":
                deq[int(a)] = float(b)
    return lat, rope, want, deq


def pin_writer_golden(orc):
    lat, rope, want, deq = load_golden_writer()
    lat_b = bf16_bits(torch.from_numpy(lat))[None]
    rope_b = bf16_bits(torch.from_numpy(rope))[None]
    rec = orc.pack_records(lat_b, rope_b)
    assert rec.shape == (1, 656)
    bad = np.nonzero(rec[0] != want)[0]
    assert bad.size == 0, f"writer bytes differ at offsets {bad[:8].tolist()}"
    got_lat, got_rope, _ = orc.unpack_records(want[None])
    assert np.array_equal(got_lat[0], deq), "reader values differ from the worked example"
    assert np.array_equal(got_rope[0], rope)


def pin_roundtrip(orc):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(64, 512, generator=g) * torch.exp2(torch.randint(-10, 10, (64, 1), generator=g).float())
    x[3, 128:256] = 0.0  # an all-zero block
    xb = x.to(torch.bfloat16)
    rope = torch.randn(64, 64, generator=g).to(torch.bfloat16)
    rec = orc.pack_records(bf16_bits(xb), bf16_bits(rope))
    # the reader agrees with torch's own decode of the same bytes
    k_ref, v_ref = torch_decode_records(rec)
    lat, rp, sc = orc.unpack_records(rec)
    assert np.array_equal(lat, v_ref) and np.array_equal(rp, k_ref[:, 512:])
    # scales are powers of two
    m, _ = np.frexp(sc)
    assert np.all(m == 0.5), "writer scales must be powers of two"
    # E4M3 keeps 3 mantissa bits: |x - deq| <= 2^-4 |x| for normals, <= 2^-10 scale below
    xf = xb.to(torch.float64).numpy()
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, np.repeat(sc, 128, axis=1) * 2.0 ** -10)
    assert np.all(np.abs(lat - xf) <= bound * (1 + 1e-12)), "quantisation error above E4M3 bound"
    # the dequantised values are a fixed point of writer then reader
    rec2 = orc.pack_records(bf16_bits(torch.from_numpy(lat)), bf16_bits(rope))
    lat2, _, _ = orc.unpack_records(rec2)
    assert np.array_equal(lat2, lat)


def pin_scale_bound(orc):
    # |latent| <= 57344 iff every scale <= 2^7 (gfx950 page, writer precondition)
    for amax, ok in ((57344.0, True), (57600.0, False), (1.0, True), (65536.0, False)):
        x = np.zeros((1, 512))
        x[0, 200] = amax
        rec = orc.pack_records(bf16_bits(torch.from_numpy(x)), np.zeros((1, 64), dtype=np.uint16))
        _, _, sc = orc.unpack_records(rec)
        assert (sc.max() <= 2.0 ** 7) == ok, (amax, sc)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def _scores_by_loops(qrow, kvec, sm_scale):
    return [sm_scale * math.fsum(float(qrow[h, d]) * float(kvec[d]) for d in range(576))
            for h in range(qrow.shape[0])]


def pin_single_key(orc):
    rec = random_records(50, seed=3)
    q = random_q(1, 4, seed=4)
    indices = np.array([-1, 17, -1, 99999], dtype=np.int32)
    indptr = np.array([0, 4], dtype=np.int32)
    out, lse, nv = orc.sparse_mla_decode(q, rec, indices, indptr, sm_scale=0.125)
    k_ref, v_ref = torch_decode_records(rec[17:18])
    assert nv[0] == 1
    assert np.array_equal(out[0], np.broadcast_to(v_ref[0], (4, 512))), "one key: out must equal its latent"
    s0 = _scores_by_loops(q[0], k_ref[0], 0.125)
    assert np.allclose(lse[0], s0, rtol=1e-13, atol=1e-13), "one key: lse must equal its score"


def pin_two_key_closed_form(orc):
    # q = 2 e_0, k_A = e_0 (latent), k_B = 0, sm_scale 1/2 -> s = (1, 0)
    rec = np.zeros((2, 656), dtype=np.uint8)
    one = np.array([1.0], dtype="<f4").view(np.uint8)
    for r in range(2):
        for b in range(4):
            rec[r, 512 + 4 * b: 516 + 4 * b] = one
    rec[0, 0] = 0x38  # E4M3 1.0
    rec[0, 5] = 0x40  # E4M3 2.0 at latent dim 5
    rec[1, 5] = 0x30  # E4M3 0.5 at latent dim 5
    q = np.zeros((1, 1, 576))
    q[0, 0, 0] = 2.0
    e = math.e
    pa, pb = e / (e + 1), 1 / (e + 1)
    for sink in (None, 0.5):
        out, lse, _ = orc.sparse_mla_decode(q, rec, np.array([0, 1], np.int32),
                                            np.array([0, 2], np.int32), sm_scale=0.5,
                                            sink=None if sink is None else np.array([sink]))
        den = (e + 1) if sink is None else (e + 1 + math.exp(sink))
        assert math.isclose(lse[0, 0], math.log(e + 1), rel_tol=1e-14)
        assert math.isclose(out[0, 0, 0], e / den, rel_tol=1e-14)
        assert math.isclose(out[0, 0, 5], (2.0 * e + 0.5) / den, rel_tol=1e-14)
        if sink is None:
            assert math.isclose(out[0, 0, 5], 2.0 * pa + 0.5 * pb, rel_tol=1e-14)


def pin_mask_invariance(orc):
    rec = random_records(40, seed=5)
    q = random_q(2, 3, seed=6)
    base_idx = np.array([3, 7, 11, 30, 2, 9, 1, 0], dtype=np.int32)
    out0, lse0, nv0 = orc.sparse_mla_decode(q, rec, base_idx, np.array([0, 4, 8], np.int32), sm_scale=0.1)
    # -1 entries, indices >= n_kv_rows, and trailing positions past lens change nothing
    noisy = np.array([3, -1, 7, 40, 11, -5, 30, -1, 2, -1, 9, 1, 12345, 0, 5], dtype=np.int32)
    indptr = np.array([0, 8, 15], dtype=np.int32)
    lens = np.array([8, 6], dtype=np.int32)  # row 1 keeps positions 0..5 = 2,-1,9,1,12345,0
    out1, lse1, nv1 = orc.sparse_mla_decode(q, rec, noisy, indptr, lens=None, sm_scale=0.1)
    assert np.array_equal(nv1, [4, 5])
    out2, lse2, nv2 = orc.sparse_mla_decode(q, rec, noisy, indptr, lens=lens, sm_scale=0.1)
    assert np.array_equal(nv2, nv0)
    np.testing.assert_allclose(out2, out0, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse2, lse0, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out1[0], out0[0], rtol=1e-13, atol=1e-15)


def pin_permutation(orc):
    rec = random_records(300, seed=8)
    q = random_q(1, 5, seed=9)
    rng = np.random.default_rng(10)
    idx = rng.choice(300, 200, replace=False).astype(np.int32)
    indptr = np.array([0, 200], np.int32)
    out0, lse0, _ = orc.sparse_mla_decode(q, rec, idx, indptr, sm_scale=0.2)
    out1, lse1, _ = orc.sparse_mla_decode(q, rec, idx[rng.permutation(200)], indptr, sm_scale=0.2)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13)


def pin_dense_bruteforce(orc):
    n, heads = 48, 4
    rec = random_records(n, seed=12)
    q = random_q(3, heads, seed=13, std=0.02)
    sink = np.array([0.3, -1.0, 2.0, -30.0])
    k, v = torch_decode_records(rec)
    k_t, v_t = torch.from_numpy(k), torch.from_numpy(v)
    for r in range(3):
        idx = np.arange(n, dtype=np.int32)
        out, lse, _ = orc.sparse_mla_decode(q[r:r + 1], rec, idx, np.array([0, n], np.int32),
                                            sm_scale=0.0625, sink=sink)
        s = 0.0625 * (torch.from_numpy(q[r]) @ k_t.T)  # [H, n]
        s_ext = torch.cat([s, torch.from_numpy(sink)[:, None]], dim=1)  # sink as a value-less key
        p = torch.softmax(s_ext, dim=1)[:, :n]
        ref_out = p @ v_t
        ref_lse = torch.logsumexp(s, dim=1)
        np.testing.assert_allclose(out[0], ref_out.numpy(), rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(lse[0], ref_lse.numpy(), rtol=1e-13)


def pin_empty_rows(orc):
    rec = random_records(10, seed=14)
    q = random_q(4, 2, seed=15)
    indices = np.array([-1, -1, 10, 3], dtype=np.int32)
    indptr = np.array([0, 2, 2, 3, 4], dtype=np.int32)  # all-invalid, empty, >= n, valid
    lens = np.array([2, 0, 1, 0], dtype=np.int32)  # row 3 truncated to nothing
    for sink in (None, np.array([1.0, -2.0])):
        out, lse, nv = orc.sparse_mla_decode(q, rec, indices, indptr, lens=lens, sink=sink)
        assert np.array_equal(nv, [0, 0, 0, 0])
        assert np.all(out == 0.0) and np.all(np.isneginf(lse))


def pin_sink_closed_form(orc):
    rec = random_records(120, seed=16)
    q = random_q(2, 6, seed=17)
    idx = np.random.default_rng(18).integers(0, 120, 150).astype(np.int32)
    indptr = np.array([0, 70, 150], np.int32)
    sink = np.array([-3.0, 0.0, 0.7, 2.5, 8.0, -np.inf])
    out0, lse0, _ = orc.sparse_mla_decode(q, rec, idx, indptr, sm_scale=0.3)
    out1, lse1, _ = orc.sparse_mla_decode(q, rec, idx, indptr, sm_scale=0.3, sink=sink)
    np.testing.assert_array_equal(lse1, lse0)  # the sink never enters the LSE
    factor = 1.0 / (1.0 + np.exp(sink[None, :] - lse0))  # sum e^s / (sum e^s + e^sink)
    np.testing.assert_allclose(out1, out0 * factor[:, :, None], rtol=1e-12, atol=1e-15)


def pin_split_combine(orc):
    rec = random_records(500, seed=19)
    q = random_q(3, 4, seed=20)
    rng = np.random.default_rng(21)
    idx = rng.integers(-50, 520, 900).astype(np.int32)  # with -ve and >= n entries
    indptr = np.array([0, 300, 301, 900], np.int32)
    sink = np.array([0.5, -0.5, 1.5, 3.0])
    out0, lse0, nv0 = orc.sparse_mla_decode(q, rec, idx, indptr, sm_scale=0.15, sink=sink)
    for ck in (1, 7, 64, 599, 600):
        o, m, l, nv = orc.split_partials(q, rec, idx, indptr, sm_scale=0.15, chunk_len=ck)
        assert np.array_equal(nv.sum(axis=1), nv0)
        out1, lse1 = orc.combine(o, m, l, sink=sink)
        np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse1, lse0, rtol=1e-12)


def pin_lse_direct(orc):
    rec = random_records(30, seed=22)
    q = random_q(1, 2, seed=23)
    idx = np.array([4, 9, 29, 0, 13], np.int32)
    _, lse, _ = orc.sparse_mla_decode(q, rec, idx, np.array([0, 5], np.int32), sm_scale=0.4)
    k, _ = torch_decode_records(rec[idx])
    for h in range(2):
        s = [_scores_by_loops(q[0][h:h + 1], k[t], 0.4)[0] for t in range(5)]
        m = max(s)
        ref = m + math.log(math.fsum(math.exp(x - m) for x in s))
        assert math.isclose(lse[0, h], ref, rel_tol=1e-13, abs_tol=1e-13)


def pin_duplicates(orc):
    rec = random_records(20, seed=24)
    q = random_q(1, 3, seed=25)
    out1, lse1, _ = orc.sparse_mla_decode(q, rec, np.array([6], np.int32), np.array([0, 1], np.int32))
    out2, lse2, nv = orc.sparse_mla_decode(q, rec, np.array([6, 6], np.int32), np.array([0, 2], np.int32))
    assert nv[0] == 2
    np.testing.assert_allclose(lse2, lse1 + math.log(2.0), rtol=1e-14)
    np.testing.assert_allclose(out2, out1, rtol=1e-14)


def pin_index_buffer_bounds(orc):
    # positions whose offset lies outside the index buffer are masked
    rec = random_records(20, seed=26)
    q = random_q(2, 2, seed=27)
    idx = np.array([1, 2, 3], np.int32)
    indptr = np.array([1, 6, 3], np.int32)  # row 0 runs past the buffer; row 1 is negative
    _, _, nv = orc.sparse_mla_decode(q, rec, idx, indptr)
    assert np.array_equal(nv, [2, 0])



def pin_foreign_scales(orc):
    # reading c10: a block scale the writer never writes (not a power of two,
    # negative, zero, large, f32 subnormal) is taken as stored.  One key per
    # row, so out is that key's latent; hand values: E4M3 0x38 = 1, 0xB8 = -1,
    # 0x01 = 2^-9 (smallest subnormal), 0x7E = 448.
    scales = np.array([3.0, -0.5, 0.0, 1000.0], dtype="<f4")
    codes = np.array([0x38, 0xB8, 0x01, 0x7E], dtype=np.uint8)
    hand = np.array([1.0, -1.0, 2.0 ** -9, 448.0])
    rec = np.zeros((2, 656), dtype=np.uint8)
    for b in range(4):
        rec[0, 128 * b:128 * (b + 1)] = np.roll(codes, b)[np.arange(128) % 4]
    rec[0, 512:528] = scales.view(np.uint8)
    rec[1] = rec[0]
    rec[1, 512:528] = np.full(4, 1e-40, dtype="<f4").view(np.uint8)  # f32 subnormal
    q = random_q(2, 2, seed=31)
    out, _, nv = orc.sparse_mla_decode(q, rec, np.array([0, 1], np.int32), np.array([0, 1, 2], np.int32))
    assert np.array_equal(nv, [1, 1])
    want = np.zeros((2, 512))
    for b in range(4):
        vals = np.roll(hand, b)[np.arange(128) % 4]
        want[0, 128 * b:128 * (b + 1)] = vals * float(scales[b])
        want[1, 128 * b:128 * (b + 1)] = vals * float(np.float32(1e-40))
    assert np.array_equal(out[:, 0], want) and np.array_equal(out[:, 1], want), "foreign scales: latent as stored"
    _, v_ref = torch_decode_records(rec)
    assert np.array_equal(out[:, 0], v_ref), "foreign scales: torch's dtype views agree"

ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
