"""libsmla.so on the host: it loads, exports every symbol include/smla.h
declares, plans splits sanely, and rejects bad arguments before any CUDA call."""

import ctypes
import os
import re

import pytest

import sparse_mla_decode_csr_gb300 as smla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "smla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(smla_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 6, names
    lib = ctypes.CDLL(smla.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in smla.h but not exported"
    assert set(smla.EXPORTED_SYMBOLS) <= set(names)


def test_status_bits_are_distinct():
    bits = [smla.STATUS_INDEX_OOB, smla.STATUS_TIMEOUT, smla.STATUS_SMEM_LAYOUT, smla.STATUS_FOREIGN_SCALE]
    assert len(set(bits)) == len(bits) and all(b & (b - 1) == 0 for b in bits)
    text = open(os.path.join(ROOT, "include", "smla.h")).read()
    for name, v in [("INDEX_OOB", 1), ("TIMEOUT", 2), ("SMEM_LAYOUT", 4), ("FOREIGN_SCALE", 8)]:
        assert re.search(rf"#define SMLA_STATUS_{name} 0x{v:x}\b", text), name


def test_strerror_names_every_code():
    for code in range(0, -9, -1):
        assert smla.strerror(code) != "unknown status"
    assert smla.strerror(-99) == "unknown status"


@pytest.mark.parametrize("n_q,heads,row_len", [
    (4, 16, 128), (64, 16, 2048), (256, 16, 2048), (128, 64, 2048), (4, 64, 16384),
    (1, 1, 1), (1000, 64, 100), (7, 33, 5000), (3, 16, 0)])
def test_plan_properties_cuda_core(n_q, heads, row_len):
    p = smla.smla_plan(n_q, heads, row_len, n_q * row_len, 0, 152, kernel=smla.KERNEL_CUDA_CORE)
    assert p.kernel == smla.KERNEL_CUDA_CORE
    assert 1 <= p.num_splits <= smla.MAX_SPLITS
    assert p.tile_len == 64 and p.chunk_len % p.tile_len == 0 and p.chunk_len > 0
    assert p.num_splits * p.chunk_len >= row_len
    assert (p.num_splits - 1) * p.chunk_len < max(row_len, 1)  # no chunk wholly past the row
    assert p.grid == n_q * p.num_splits
    assert p.partial_slots == (n_q * p.num_splits if p.num_splits > 1 else 0)
    assert (p.workspace_bytes == 0) == (p.num_splits == 1)
    if p.num_splits > 1:
        need = n_q * 4 + p.partial_slots * heads * (512 + 2) * 4 + p.partial_slots * 4
        assert p.workspace_bytes >= need


@pytest.mark.parametrize("n_q,heads,row_len", [
    (4, 16, 128), (32, 16, 2048), (64, 16, 2048), (256, 16, 2048), (128, 64, 2048), (4, 64, 16384), (1, 1, 1)])
def test_plan_properties_tensor_core(n_q, heads, row_len):
    p = smla.smla_plan(n_q, heads, row_len, n_q * row_len, 0, 152)
    # the default resolves to the native-fp8 kernel (up to 64 heads)
    assert p.kernel == smla.KERNEL_TENSOR_CORE_FP8 and p.tile_len == 128
    hg = 2 if heads > 32 else 1  # two CTAs (head groups of up to 32) share a schedule range above 32 heads
    assert p.head_groups == hg and p.grid == 152 // hg  # persistent: one CTA per SM
    assert p.partial_slots == 2 * p.grid
    # rows of at most 4 parts are merged inside the kernel; the merge kernel
    # runs only when top-k rows would span more CTAs
    assert p.merge_kernel == (-(-p.grid // n_q) + 1 > 4)
    need = 8 * n_q + (n_q + 1) * 8 + p.partial_slots * heads * (512 + 2) * 4 + p.partial_slots * 4
    assert p.workspace_bytes >= need
    for k in (1, 3, 64):
        f = smla.smla_plan(n_q, heads, row_len, n_q * row_len, k, 152)
        assert f.grid == min(n_q * k, 65535 // hg)
    b = smla.smla_plan(n_q, heads, row_len, n_q * row_len, 0, 152, kernel=smla.KERNEL_TENSOR_CORE_BF16)
    assert b.kernel == smla.KERNEL_TENSOR_CORE_BF16 and b.tile_len == 64 and b.grid == 152
    assert b.head_groups == 1 and b.merge_kernel == 1 and b.partial_slots == 2 * b.grid


def test_plan_splits_short_batches_and_respects_forcing():
    cc = smla.KERNEL_CUDA_CORE
    assert smla.smla_plan(4, 64, 16384, 4 * 16384, 0, 152, kernel=cc).num_splits > 16  # long rows split
    assert smla.smla_plan(2048, 16, 2048, 2048 * 2048, 0, 152, kernel=cc).num_splits == 1
    for k in (1, 2, 5, 64):
        assert smla.smla_plan(3, 16, 700, 2100, k, 152, kernel=cc).num_splits == k
    with pytest.raises(smla.SmlaError):
        smla.smla_plan(3, 16, 700, 2100, 65, 152)
    with pytest.raises(smla.SmlaError):
        smla.smla_plan(3, 65, 700, 2100, 0, 152)
    with pytest.raises(smla.SmlaError):
        smla.smla_plan(-1, 16, 700, 2100, 0, 152)
    with pytest.raises(smla.SmlaError):
        smla.smla_plan(3, 16, 700, 2100, 0, 152, kernel=7)
    with pytest.raises(smla.SmlaError):  # more than 64 heads
        smla.smla_plan(3, 65, 700, 2100, 0, 152, kernel=smla.KERNEL_TENSOR_CORE_FP8)
    for k in (smla.KERNEL_TENSOR_CORE_BF16, smla.KERNEL_TENSOR_CORE_FP8):
        assert smla.smla_plan(3, 16, 700, 2100, 0, 152, kernel=k).kernel == k


def _params(**kw):
    p = smla.DecodeParams()
    p.n_q, p.num_heads = 2, 16
    p.q, p.q_stride_row, p.q_stride_head = 0x1000, 16 * 576, 576
    p.kv_cache, p.n_kv_rows = 0x2000, 100
    p.indices, p.n_indices, p.indptr = 0x3000, 10, 0x4000
    p.out, p.out_stride_row, p.out_stride_head = 0x5000, 16 * 512, 512
    p.sm_scale = 0.05
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(out=None), -1), (dict(indptr=None), -1), (dict(kv_cache=None), -1),
    (dict(num_heads=0), -2), (dict(num_heads=65), -2), (dict(n_q=-1), -2),
    (dict(n_kv_rows=(1 << 31) + 1), -2), (dict(sm_scale=float("nan")), -2),
    (dict(q_stride_head=100), -3), (dict(out_stride_row=512), -3),
    (dict(q=0x1008), -4), (dict(out_stride_head=516, out_stride_row=16 * 516), -4), (dict(kv_cache=0x2004), -4),
    (dict(num_splits=65), -6), (dict(num_splits=-1), -6), (dict(kernel=4), -2),
    (dict(kernel=3, num_heads=65), -2),
])
def test_decode_rejects_bad_arguments_on_host(kw, code):
    p = _params(**kw)
    rc = smla.lib.smla_decode(ctypes.byref(p), None, 0, None)
    assert rc == code, (kw, rc, smla.strerror(rc))


@pytest.mark.parametrize("kw,code", [
    (dict(q=None, kernel=1, num_splits=3), -1), (dict(indptr=None, kernel=1, num_splits=3), -1),
    (dict(q=0x1008, kernel=1, num_splits=3), -4), (dict(q_stride_head=100), -3), (dict(num_heads=65), -2)])
def test_noalloc_rejects_bad_arguments_before_enqueueing(kw, code):
    # the checks run before the call touches the device (no CUDA device here):
    # the CUDA-core split plan's ticket clear is never enqueued for a bad call
    p = _params(**kw)
    rc = smla.lib.smla_decode_noalloc(ctypes.byref(p), None)
    assert rc == code, (kw, rc, smla.strerror(rc))


def test_decode_with_empty_batch_is_a_noop():
    p = _params(n_q=0, q=None, out=None, indptr=None)
    assert smla.lib.smla_decode(ctypes.byref(p), None, 0, None) == 0


def test_pack_rejects_bad_arguments_on_host():
    f = smla.lib.smla_pack_records
    assert f(None, 512, 0x1000, 64, 4, 0x2000, None) == -1
    assert f(0x1000, 500, 0x1000, 64, 4, 0x2000, None) == -3
    assert f(0x1004, 512, 0x1000, 64, 4, 0x2000, None) == -4
    assert f(0x1000, 512, 0x1000, 64, -1, 0x2000, None) == -2
    assert f(0x1000, 512, 0x1000, 64, 0, 0x2000, None) == 0


def test_plan_trims_rows_only_for_the_tensor_core_kernel_with_has_invalid():
    base = smla.smla_plan(256, 16, 2048, 256 * 2048, 0, 152)
    trim = smla.smla_plan(256, 16, 2048, 256 * 2048, 0, 152, has_invalid=True)
    cc = smla.smla_plan(256, 16, 2048, 256 * 2048, 0, 152, kernel=smla.KERNEL_CUDA_CORE, has_invalid=True)
    assert base.trim_kernel == 0 and trim.trim_kernel == 1 and cc.trim_kernel == 0
    # the trimmed lengths take one more int32 per row at the end of the workspace
    assert trim.workspace_bytes >= base.workspace_bytes + 4 * 256
    assert trim.grid == base.grid and trim.partial_slots == base.partial_slots
