"""The oracle against its pins (CPU only), and planted mistakes against the pins."""

import numpy as np
import pytest

import oracle.smla_oracle as orc
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin):
    pin(orc)


# --- planted mistakes: every one must make at least one pin fail -------------

def _mut_rope_dropped(mp):
    real = orc.row_keys

    def row_keys(kv, ids):
        k, v = real(kv, ids)
        k = k.copy()
        k[:, 512:] = 0.0
        return k, v
    mp.setattr(orc, "row_keys", row_keys)


def _mut_scales_reversed(mp):
    real = orc.unpack_records

    def unpack_records(rec):
        lat, rope, sc = real(rec)
        blocks = lat.reshape(lat.shape[0], 4, 128) / np.maximum(sc[:, :, None], 1e-300)
        lat = (blocks * sc[:, ::-1, None]).reshape(lat.shape[0], 512)
        return lat, rope, sc
    mp.setattr(orc, "unpack_records", unpack_records)


def _mut_sink_in_lse(mp):
    real = orc.softmax_out

    def softmax_out(scores, values, sink):
        out, lse = real(scores, values, sink)
        if sink is not None and scores.shape[1]:
            lse = np.logaddexp(lse, np.asarray(sink, dtype=np.float64))
        return out, lse
    mp.setattr(orc, "softmax_out", softmax_out)


def _mut_negative_wraps(mp):
    def row_positions(r, indices, indptr, lens, n_kv_rows):
        beg, end = int(indptr[r]), int(indptr[r + 1])
        length = max(end - beg, 0)
        if lens is not None:
            length = min(length, max(int(lens[r]), 0))
        pos, ids = [], []
        for p in range(length):
            off = beg + p
            if 0 <= off < len(indices):
                idx = int(indices[off])
                if idx < n_kv_rows:  # negative entries wrap around instead of masking
                    pos.append(p)
                    ids.append(idx % n_kv_rows)
        return np.array(pos, dtype=np.int64), np.array(ids, dtype=np.int64)
    mp.setattr(orc, "row_positions", row_positions)


def _mut_lens_ignored(mp):
    real = orc.row_positions
    mp.setattr(orc, "row_positions", lambda r, i, p, lens, n: real(r, i, p, None, n))


def _mut_e4m3_bias8(mp):
    mp.setattr(orc, "_E4M3", orc.e4m3_table() / 2.0)
    mp.setattr(orc, "e4m3_table", lambda: np.array([orc.e4m3_value(c) / 2.0 for c in range(256)]))


def _mut_ties_away(mp):
    real = orc.e4m3_encode_rne

    def enc(x):
        x = np.asarray(x, dtype=np.float64)
        c = real(x)
        up = real(np.nextafter(np.abs(x), np.inf)) & 0x7F
        return np.where(np.abs(x) < 448, (c & 0x80) | up, c).astype(np.uint8)
    mp.setattr(orc, "e4m3_encode_rne", enc)


def _mut_no_amax_floor(mp):
    def writer_scales(latent):
        blocks = np.abs(np.asarray(latent, dtype=np.float64)).reshape(-1, 4, 128)
        amax = np.maximum(blocks.max(axis=2), 1e-30)
        return orc.pow2ceil(amax / 448.0)
    mp.setattr(orc, "writer_scales", writer_scales)


def _mut_combine_no_rescale(mp):
    def combine(o_part, m_part, l_part, sink=None):
        n_q, _, n_heads, _ = o_part.shape
        out = np.zeros((n_q, n_heads, 512))
        lse = np.full((n_q, n_heads), -np.inf)
        for r in range(n_q):
            for h in range(n_heads):
                live = np.isfinite(m_part[r, :, h])
                if not live.any():
                    continue
                l = l_part[r, live, h].sum()  # chunk maxima ignored
                lse[r, h] = m_part[r, live, h].max() + np.log(l)
                out[r, h] = o_part[r, live, h].sum(axis=0) / l
        return out, lse
    mp.setattr(orc, "combine", combine)


def _mut_sink_numerator(mp):
    real = orc.softmax_out

    def softmax_out(scores, values, sink):
        return real(scores, values, None)  # the sink is ignored
    mp.setattr(orc, "softmax_out", softmax_out)


def _mut_scale_squared(mp):
    real = orc.row_scores
    mp.setattr(orc, "row_scores", lambda q, k, s: real(q, k, s * s))



def _mut_scale_exponent_only(mp):
    real = orc.unpack_records

    def unpack_records(rec):  # a reader that keeps only each scale's power of two
        lat, rope, sc = real(rec)
        p2 = np.where(sc > 0, np.exp2(np.floor(np.log2(np.where(sc > 0, sc, 1.0)))), 0.0)
        blocks = lat.reshape(lat.shape[0], 4, 128) / np.where(sc != 0, sc, 1.0)[:, :, None]
        return (blocks * p2[:, :, None]).reshape(lat.shape[0], 512), rope, p2
    mp.setattr(orc, "unpack_records", unpack_records)

MUTATIONS = [v for k, v in sorted(globals().items()) if k.startswith("_mut_")]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=[m.__name__[5:] for m in MUTATIONS])
def test_planted_mistake_is_caught(mutate, monkeypatch):
    mutate(monkeypatch)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutate.__name__}"
