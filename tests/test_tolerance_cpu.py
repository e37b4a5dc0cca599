"""The GPU tests' rounding allowance is itself checked on the CPU: it is small
on well-conditioned N(0,1) data, and it bounds an f32 evaluation of the method
(scores and weights in float32) on heavy-tailed keys."""

import numpy as np
import torch

import oracle
from smla_testlib import ATOL, RTOL, allowance, bits


def _case(seed, heavy):
    g = torch.Generator().manual_seed(seed)
    n_kv, n_q, heads = 600, 3, 16
    lat = torch.randn(n_kv, 512, generator=g)
    if heavy:
        z = torch.randn(n_kv, 512, 3, generator=g).square().sum(-1)
        lat = lat * torch.sqrt(3.0 / z) * torch.exp2(torch.randint(-8, 13, (n_kv, 4), generator=g).float()
                                                      ).repeat_interleave(128, 1)
    lat = lat.to(torch.bfloat16).clamp(-57344, 57344)
    rope = torch.randn(n_kv, 64, generator=g).to(torch.bfloat16)
    rec = oracle.pack_records(bits(lat), bits(rope))
    q = torch.randn(n_q, heads, 576, generator=g).to(torch.bfloat16).double().numpy()
    idx = torch.randint(0, n_kv, (n_q * 500,), generator=g).int().numpy()
    ptr = (np.arange(n_q + 1) * 500).astype(np.int32)
    sink = torch.randn(heads, generator=g).double().numpy()
    return q, rec, idx, ptr, sink


def _f32_method(q, rec, idx, ptr, sink, sm_scale):
    """Scores, softmax and PV evaluated in float32 (the rounding the allowance models)."""
    n_q, heads, _ = q.shape
    out = np.zeros((n_q, heads, 512))
    for r in range(n_q):
        _, ids = oracle.row_positions(r, idx, ptr, None, rec.shape[0])
        k, v = oracle.row_keys(rec, ids)
        s = (q[r].astype(np.float32) @ k.astype(np.float32).T) * np.float32(sm_scale)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True) + np.exp(sink.astype(np.float32)[:, None] - m)
        p = (e / den).astype(np.float32)
        out[r] = p @ v.astype(np.float32)
    return out


def test_allowance_is_small_on_normal_data():
    q, rec, idx, ptr, sink = _case(1, heavy=False)
    a_out, a_lse = allowance(q, rec, idx, ptr, None, 1 / 24, sink)
    assert a_out.max() < 1e-2 and a_lse.max() < 5e-3  # well below atol 2e-2


def test_allowance_bounds_an_f32_evaluation_on_heavy_tails():
    q, rec, idx, ptr, sink = _case(2, heavy=True)
    ref, _, _ = oracle.sparse_mla_decode(q, rec, idx, ptr, None, 1 / 24, sink)
    got = _f32_method(q, rec, idx, ptr, sink, 1 / 24)
    a_out, _ = allowance(q, rec, idx, ptr, None, 1 / 24, sink)
    err = np.abs(got - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref) + a_out)
    assert a_out.max() > 1e-2  # heavy tails do need it
