"""Python binding of libsmla.so: sparse MLA decode over fp8_ds_mla records.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of libsmla.so; there is no CPU or PyTorch fallback, and importing
fails loudly when the library has not been built (``python -c "import
__graft_entry__ as g; g.build()"``).  PyTorch supplies device memory and
streams.  The entry points keep the names of the C ABI in include/smla.h.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsmla.so")

RECORD_BYTES = 656
LATENT_DIM = 512
ROPE_DIM = 64
QK_DIM = 576
MAX_HEADS = 64
MAX_SPLITS = 64
STATUS_INDEX_OOB = 0x1
STATUS_TIMEOUT = 0x2
STATUS_SMEM_LAYOUT = 0x4
STATUS_FOREIGN_SCALE = 0x8
KERNEL_TENSOR_CORE = 0       # default: native fp8 where supported, else bf16 tensor cores
KERNEL_CUDA_CORE = 1
KERNEL_TENSOR_CORE_BF16 = 2
KERNEL_TENSOR_CORE_FP8 = 3
NOALLOC_SCRATCH_BYTES = 64 << 20  # SMLA_NOALLOC_SCRATCH_BYTES
SMLA_ERR_WORKSPACE = -5


class SmlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} (status {code})")
        self.code = code


class DecodeParams(ctypes.Structure):
    _fields_ = [
        ("n_q", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("q", ctypes.c_void_p),
        ("q_stride_row", ctypes.c_int64),
        ("q_stride_head", ctypes.c_int64),
        ("kv_cache", ctypes.c_void_p),
        ("n_kv_rows", ctypes.c_int64),
        ("indices", ctypes.c_void_p),
        ("n_indices", ctypes.c_int64),
        ("indptr", ctypes.c_void_p),
        ("lens", ctypes.c_void_p),
        ("max_row_len", ctypes.c_int32),
        ("has_invalid", ctypes.c_int32),
        ("sm_scale", ctypes.c_float),
        ("sink", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("out_stride_row", ctypes.c_int64),
        ("out_stride_head", ctypes.c_int64),
        ("lse", ctypes.c_void_p),
        ("n_valid", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
        ("num_splits", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int32),
        ("grid", ctypes.c_int32),
        ("tile_len", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
        ("chunk_len", ctypes.c_int32),
        ("partial_slots", ctypes.c_int32),
        ("merge_kernel", ctypes.c_int32),
        ("trim_kernel", ctypes.c_int32),
        ("head_groups", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built: run `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(LIB_PATH)
    lib.smla_plan.argtypes = [ctypes.POINTER(DecodeParams), ctypes.c_int32, ctypes.POINTER(PlanInfo)]
    lib.smla_plan.restype = ctypes.c_int
    lib.smla_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeParams)]
    lib.smla_decode_workspace_size.restype = ctypes.c_size_t
    lib.smla_decode.argtypes = [ctypes.POINTER(DecodeParams), ctypes.c_void_p, ctypes.c_size_t,
                                ctypes.c_void_p]
    lib.smla_decode.restype = ctypes.c_int
    lib.smla_decode_noalloc.argtypes = [ctypes.POINTER(DecodeParams), ctypes.c_void_p]
    lib.smla_decode_noalloc.restype = ctypes.c_int
    lib.smla_pack_records.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                      ctypes.c_void_p]
    lib.smla_pack_records.restype = ctypes.c_int
    lib.smla_strerror.argtypes = [ctypes.c_int]
    lib.smla_strerror.restype = ctypes.c_char_p
    lib.smla_device_check.argtypes = []
    lib.smla_device_check.restype = ctypes.c_int
    lib.smla_set_wait_limit.argtypes = [ctypes.c_uint64, ctypes.c_int]
    lib.smla_set_wait_limit.restype = ctypes.c_int
    return lib


lib = _load()

EXPORTED_SYMBOLS = ("smla_plan", "smla_decode_workspace_size", "smla_decode", "smla_decode_noalloc",
                    "smla_pack_records", "smla_strerror", "smla_device_check", "smla_set_wait_limit")


def strerror(code: int) -> str:
    return lib.smla_strerror(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _plan_params(n_q, num_heads, max_row_len=0, n_indices=0, num_splits=0,
                 kernel=KERNEL_TENSOR_CORE, has_invalid=False) -> DecodeParams:
    p = DecodeParams()
    p.n_q, p.num_heads, p.max_row_len, p.n_indices = int(n_q), int(num_heads), int(max_row_len), int(n_indices)
    p.num_splits, p.kernel, p.has_invalid = int(num_splits), int(kernel), int(bool(has_invalid))
    return p


def smla_plan(n_q: int, num_heads: int, max_row_len: int = 0, n_indices: int = 0,
              num_splits: int = 0, num_sms: int = 0, kernel: int = KERNEL_TENSOR_CORE,
              has_invalid: bool = False) -> PlanInfo:
    """The launch plan of a decode call (pure host arithmetic when num_sms > 0)."""
    info = PlanInfo()
    p = _plan_params(n_q, num_heads, max_row_len, n_indices, num_splits, kernel, has_invalid)
    rc = lib.smla_plan(ctypes.byref(p), int(num_sms), ctypes.byref(info))
    if rc != 0:
        raise SmlaError(rc, "smla_plan")
    return info


def smla_decode_workspace_size(n_q: int, num_heads: int, max_row_len: int = 0,
                               n_indices: int = 0, num_splits: int = 0,
                               kernel: int = KERNEL_TENSOR_CORE, has_invalid: bool = False) -> int:
    p = _plan_params(n_q, num_heads, max_row_len, n_indices, num_splits, kernel, has_invalid)
    return int(lib.smla_decode_workspace_size(ctypes.byref(p)))


_WS: dict = {}


def workspace(nbytes: int, device, layout=None) -> Optional[torch.Tensor]:
    """A cached workspace of at least nbytes on device, ready for a call with
    the given layout key (n_q, heads, plan).

    smla_decode needs the per-row ticket counters at the start of the
    workspace to be zero, and leaves them zero; a call with another layout may
    have written partials over that region, so the counters are re-zeroed
    (on the current stream) whenever the layout changes.
    """
    if nbytes == 0:
        return None
    dev = torch.device(device)
    key = (dev.type, dev.index)
    ws, last = _WS.get(key, (None, None))
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=dev)
    elif layout != last:
        n_q = layout[0] if layout else ws.numel() // 4
        ws[: min(ws.numel(), 8 * n_q + 256)].zero_()
    _WS[key] = (ws, layout)
    return ws


def smla_decode(q: torch.Tensor, kv_cache: torch.Tensor, n_kv_rows: int, indices: torch.Tensor,
                indptr: torch.Tensor, lens: Optional[torch.Tensor], sm_scale: float,
                sink: Optional[torch.Tensor], out: torch.Tensor, lse: Optional[torch.Tensor],
                stream=None, *, max_row_len: int = 0, has_invalid: bool = False,
                n_valid: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                num_splits: int = 0, workspace_tensor: Optional[torch.Tensor] = None,
                kernel: int = KERNEL_TENSOR_CORE) -> None:
    """Sparse MLA decode into ``out`` (bf16 [n_q, H, 512]) and ``lse`` (f32 [n_q, H]).

    q: bf16 [n_q, H, 576]; kv_cache: uint8 [n_kv_rows, 656]; indices/indptr/lens:
    int32; sink: f32 [H] or None; n_valid: int32 [n_q] or None; status: int32 [1]
    or None.  All tensors on the current CUDA device.  See include/smla.h.
    """
    assert q.dtype == torch.bfloat16 and q.dim() == 3 and q.stride(2) == 1
    assert out.dtype == torch.bfloat16 and out.dim() == 3 and out.stride(2) == 1
    assert kv_cache.dtype == torch.uint8
    for t in (indices, indptr, lens, n_valid, status):
        assert t is None or t.dtype == torch.int32
    assert sink is None or sink.dtype == torch.float32
    assert lse is None or (lse.dtype == torch.float32 and lse.is_contiguous())
    n_q, heads = int(q.shape[0]), int(q.shape[1])
    p = DecodeParams()
    p.n_q, p.num_heads = n_q, heads
    p.q, p.q_stride_row, p.q_stride_head = q.data_ptr(), q.stride(0), q.stride(1)
    p.kv_cache, p.n_kv_rows = kv_cache.data_ptr(), int(n_kv_rows)
    p.indices, p.n_indices = _ptr(indices), int(indices.numel())
    p.indptr, p.lens = _ptr(indptr), _ptr(lens)
    p.max_row_len, p.has_invalid = int(max_row_len), int(bool(has_invalid))
    p.sm_scale = float(sm_scale)
    p.sink = _ptr(sink)
    p.out, p.out_stride_row, p.out_stride_head = out.data_ptr(), out.stride(0), out.stride(1)
    p.lse, p.n_valid, p.status = _ptr(lse), _ptr(n_valid), _ptr(status)
    p.num_splits = int(num_splits)
    p.kernel = int(kernel)
    ws = workspace_tensor
    if ws is None:
        plan = PlanInfo()
        rc = lib.smla_plan(ctypes.byref(p), 0, ctypes.byref(plan))
        if rc != 0:
            raise SmlaError(rc, "smla_plan")
        ws = workspace(int(plan.workspace_bytes), q.device,
                       (n_q, heads, plan.kernel, plan.grid, plan.num_splits, plan.chunk_len, plan.trim_kernel))
    rc = lib.smla_decode(ctypes.byref(p), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream))
    if rc != 0:
        raise SmlaError(rc, "smla_decode")


def smla_decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, n_kv_rows: int,
                        indices: torch.Tensor, indptr: torch.Tensor, lens: Optional[torch.Tensor],
                        sm_scale: float, sink: Optional[torch.Tensor], out: torch.Tensor,
                        lse: Optional[torch.Tensor], stream=None, *, max_row_len: int = 0,
                        has_invalid: bool = False, n_valid: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None, num_splits: int = 0,
                        kernel: int = KERNEL_TENSOR_CORE) -> None:
    """smla_decode with the library's fixed device scratch as workspace (no
    allocation on the call path; for callers that cannot allocate device
    memory at call time).  Arguments as smla_decode.  Calls on one device
    share that scratch: calls that may overlap on the GPU must be ordered.
    The first call on a device sets up the scratch address; make it before
    any stream capture.  See include/smla.h."""
    assert q.dtype == torch.bfloat16 and q.dim() == 3 and q.stride(2) == 1
    assert out.dtype == torch.bfloat16 and out.dim() == 3 and out.stride(2) == 1
    assert kv_cache.dtype == torch.uint8
    for t in (indices, indptr, lens, n_valid, status):
        assert t is None or t.dtype == torch.int32
    assert sink is None or sink.dtype == torch.float32
    assert lse is None or (lse.dtype == torch.float32 and lse.is_contiguous())
    p = DecodeParams()
    p.n_q, p.num_heads = int(q.shape[0]), int(q.shape[1])
    p.q, p.q_stride_row, p.q_stride_head = q.data_ptr(), q.stride(0), q.stride(1)
    p.kv_cache, p.n_kv_rows = kv_cache.data_ptr(), int(n_kv_rows)
    p.indices, p.n_indices = _ptr(indices), int(indices.numel())
    p.indptr, p.lens = _ptr(indptr), _ptr(lens)
    p.max_row_len, p.has_invalid = int(max_row_len), int(bool(has_invalid))
    p.sm_scale = float(sm_scale)
    p.sink = _ptr(sink)
    p.out, p.out_stride_row, p.out_stride_head = out.data_ptr(), out.stride(0), out.stride(1)
    p.lse, p.n_valid, p.status = _ptr(lse), _ptr(n_valid), _ptr(status)
    p.num_splits, p.kernel = int(num_splits), int(kernel)
    rc = lib.smla_decode_noalloc(ctypes.byref(p), _stream(stream))
    if rc == SMLA_ERR_WORKSPACE:
        raise SmlaError(rc, f"smla_decode_noalloc: the call needs more than the "
                            f"{NOALLOC_SCRATCH_BYTES}-byte fixed scratch")
    if rc != 0:
        raise SmlaError(rc, "smla_decode_noalloc")


def smla_pack_records(latent: torch.Tensor, rope: torch.Tensor, kv_out: torch.Tensor,
                      stream=None) -> None:
    """Record writer: bf16 latent [n, 512] + bf16 rope [n, 64] -> uint8 kv_out [n, 656]."""
    assert latent.dtype == torch.bfloat16 and rope.dtype == torch.bfloat16
    assert kv_out.dtype == torch.uint8 and kv_out.is_contiguous()
    assert latent.stride(1) == 1 and rope.stride(1) == 1
    n = int(latent.shape[0])
    assert rope.shape[0] == n and kv_out.numel() >= n * RECORD_BYTES
    rc = lib.smla_pack_records(latent.data_ptr(), latent.stride(0), rope.data_ptr(), rope.stride(0),
                               n, kv_out.data_ptr(), _stream(stream))
    if rc != 0:
        raise SmlaError(rc, "smla_pack_records")


def smla_device_check() -> int:
    return int(lib.smla_device_check())


def smla_set_wait_limit(limit_ns: int, stall_first_wait: bool = False) -> None:
    """Limit of every in-kernel pipeline wait (0: the 2 s default), and the
    timeout-path test switch; see smla.h."""
    rc = lib.smla_set_wait_limit(int(limit_ns), int(bool(stall_first_wait)))
    if rc != 0:
        raise SmlaError(rc, "smla_set_wait_limit")
