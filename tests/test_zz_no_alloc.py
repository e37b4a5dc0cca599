"""smla_decode_noalloc (workspace in the library's fixed device scratch)
against smla_decode (caller workspace) on the same inputs, through the C ABI.

Two different problems run back to back through the no-alloc call, so the
second one starts from the scratch contents the first left behind.  Rows are
long enough that the tensor-core schedule shares them between CTAs (partials
and the merge kernel use the scratch); the CUDA-core kernel runs with forced
splits (ticket counters and partials in the scratch).
"""

import numpy as np
import pytest
import torch

import sparse_mla_decode_csr_gb300 as smla

pytestmark = pytest.mark.gpu
DEV = "cuda"


def problem(seed, n_q, heads, row_len, n_kv, sink):
    g = torch.Generator().manual_seed(seed)
    lat = torch.randn(n_kv, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(n_kv, 64, generator=g).to(torch.bfloat16)
    kv = torch.empty(n_kv, 656, dtype=torch.uint8, device=DEV)
    smla.smla_pack_records(lat.to(DEV), rope.to(DEV), kv)
    lens = [row_len - 37 * r for r in range(n_q)]
    indices = torch.randint(-1, n_kv, (sum(lens),), generator=g, dtype=torch.int32)
    indptr = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    return dict(q=torch.randn(n_q, heads, 576, generator=g).to(torch.bfloat16).to(DEV), kv=kv, n_kv=n_kv,
                indices=indices.to(DEV), indptr=indptr.to(DEV), max_row_len=max(lens),
                sink=torch.randn(heads, generator=g).to(DEV) if sink else None)


def run(fn, c, kernel, num_splits):
    n_q, heads = c["q"].shape[0], c["q"].shape[1]
    out = torch.full((n_q, heads, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((n_q, heads), float("nan"), dtype=torch.float32, device=DEV)
    nv = torch.full((n_q,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = dict(max_row_len=c["max_row_len"], has_invalid=True, n_valid=nv, status=st,
              num_splits=num_splits, kernel=kernel)
    fn(c["q"], c["kv"], c["n_kv"], c["indices"], c["indptr"], None, 0.0417, c["sink"], out, lse, **kw)
    torch.cuda.synchronize()
    return out.float().cpu(), lse.cpu(), nv.cpu(), int(st.item())


@pytest.mark.parametrize("kernel,num_splits", [(smla.KERNEL_TENSOR_CORE, 0), (smla.KERNEL_CUDA_CORE, 3)])
def test_noalloc_matches_decode_on_two_calls_in_a_row(kernel, num_splits):
    cases = [problem(1, 9, 16, 3000, 20000, sink=True), problem(2, 5, 64, 2100, 7000, sink=False)]
    for i, c in enumerate(cases):
        ref = run(smla.smla_decode, c, kernel, num_splits)
        got = run(smla.smla_decode_noalloc, c, kernel, num_splits)
        assert torch.isfinite(got[0]).all(), f"call {i}: non-finite output"
        # the same kernels with the same plan on the same inputs: bit for bit,
        # so that a stale-scratch bug of any size shows up
        assert torch.equal(got[0], ref[0]), f"call {i}: out differs by {(got[0] - ref[0]).abs().max():.3g}"
        assert torch.equal(got[1], ref[1]), f"call {i}: lse differs"
        assert torch.equal(got[2], ref[2]), f"call {i}: contributing-key counts differ"
        assert got[3] == ref[3]


def test_noalloc_rejects_a_call_beyond_the_scratch():
    # 8 rows x 64 forced chunks -> 512 CTAs, 1024 partial slots x 64 heads x 2 KiB > 64 MiB
    c = problem(3, 8, 64, 600, 1000, sink=False)
    need = smla.smla_decode_workspace_size(8, 64, c["max_row_len"], int(c["indices"].numel()), 64)
    assert need > smla.NOALLOC_SCRATCH_BYTES
    out = torch.zeros(8, 64, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(8, 64, dtype=torch.float32, device=DEV)
    with pytest.raises(smla.SmlaError) as e:
        smla.smla_decode_noalloc(c["q"], c["kv"], c["n_kv"], c["indices"], c["indptr"], None, 0.0417,
                                 None, out, lse, max_row_len=c["max_row_len"], num_splits=64)
    assert e.value.code == smla.SMLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0 and torch.count_nonzero(lse) == 0  # nothing launched
