"""Shared helpers of the GPU parity tests: build a case on both sides, run the
CUDA path through the C ABI, run the oracle on the same inputs, compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import smla_workloads as W
import sparse_mla_decode_csr_gb300 as smla

ATOL = 2e-2
RTOL = 1e-2
NORM_RTOL = 1e-2


def bits(x: torch.Tensor) -> np.ndarray:
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def pack_gpu(lat: torch.Tensor, rope: torch.Tensor, dev) -> torch.Tensor:
    kv = torch.empty(lat.shape[0], 656, dtype=torch.uint8, device=dev)
    smla.smla_pack_records(lat.to(dev), rope.to(dev), kv)
    return kv


def build_cache(w: W.Workload, dev, gen_device="cuda") -> torch.Tensor:
    kv = torch.empty(w.n_kv_rows, 656, dtype=torch.uint8, device=dev)
    for s in range(W.n_slabs(w)):
        lat, rope = W.latent_slab(w, s, gen_device)
        start = s * W.SLAB_ROWS
        smla.smla_pack_records(lat.to(dev), rope.to(dev), kv[start:start + lat.shape[0]])
        del lat, rope
    return kv


KERNELS = {"tc": smla.KERNEL_TENSOR_CORE, "simt": smla.KERNEL_CUDA_CORE,
           "bf16": smla.KERNEL_TENSOR_CORE_BF16, "fp8": smla.KERNEL_TENSOR_CORE_FP8}
FP8_MAX_HEADS = 64


def run_gpu(q, kv, n_kv_rows, indices, indptr, lens, sm_scale, sink, *, max_row_len=0,
            has_invalid=False, num_splits=0, out=None, q_view=None, kernel="tc"):
    dev = kv.device
    n_q, heads = q.shape[0], q.shape[1]
    if out is None:
        out = torch.full((n_q, heads, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((n_q, heads), float("nan"), dtype=torch.float32, device=dev)
    n_valid = torch.full((n_q,), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    smla.smla_decode(q if q_view is None else q_view, kv, n_kv_rows, indices, indptr, lens, sm_scale,
                     sink, out, lse, max_row_len=max_row_len, has_invalid=has_invalid,
                     n_valid=n_valid, status=status, num_splits=num_splits, kernel=KERNELS[kernel])
    torch.cuda.synchronize()
    return out, lse, n_valid, int(status.item())


U32 = 2.0 ** -24  # unit roundoff of f32


def allowance(q, rec, indices, indptr, lens, sm_scale, sink, n_kv_rows=None, operand_rel=0.0):
    """Rounding allowance of an f32 evaluation of the method, per output element.

    Scores: an f32 dot product of 576 terms is within ds_t = 576 u sum_d |q_d k_td|
    of the exact one (standard forward bound; doubled here for slack).  To
    first order a score error moves out_d by sum_t w_t ds_t |v_td - out_d| and
    the LSE by max_t ds_t (w_t the softmax weights incl. the sink).  Weights
    rounded to bf16 add 2^-8 sum_t w_t |v_td|.  For N(0,1) data this is ~1e-3;
    it only matters where the problem is ill-conditioned (heavy-tailed keys,
    near-tied scores).  Uses the oracle's own row slicing and record reader.

    operand_rel: relative rounding of k and v on their way into the products
    (0 where they enter exactly); it adds operand_rel sum_d |q_d k_td| to each
    score's error and operand_rel sum_t w_t |v_td| to each output.
    """
    q = np.asarray(q, dtype=np.float64)
    n_q, heads, _ = q.shape
    if n_kv_rows is None:
        n_kv_rows = rec.shape[0]
    out_allow = np.zeros((n_q, heads, 512))
    lse_allow = np.zeros((n_q, heads))
    for r in range(n_q):
        _, ids = oracle.row_positions(r, indices, indptr, lens, n_kv_rows)
        if len(ids) == 0:
            continue
        keys, values = oracle.row_keys(rec, ids)
        s = oracle.row_scores(q[r], keys, sm_scale)
        ds = (2.0 * 576 * U32 + operand_rel) * abs(sm_scale) * (np.abs(q[r]) @ np.abs(keys).T)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True)
        if sink is not None:
            den = den + np.exp(np.asarray(sink, dtype=np.float64)[:, None] - m)
        w = e / den
        av = np.abs(values)
        out = w @ values
        wd = w * ds
        out_allow[r] = wd @ av + wd.sum(axis=1, keepdims=True) * np.abs(out) + (2.0 ** -8 + operand_rel) * (w @ av)
        lse_allow[r] = ds.max(axis=1)
    return out_allow, lse_allow


def compare(out_gpu, lse_gpu, ref_out, ref_lse, what="", allow=None, stats=None):
    """Element-wise |gpu - ref| <= 2e-2 + 1e-2 |ref| (+ the f32 rounding
    allowance of ill-conditioned elements) for out and finite lse; the
    norm-relative error of each (row, head) output <= 1e-2 (+ the norm of the
    allowance); -inf lse exactly where the oracle has it.

    stats (a dict, optional) receives how many out elements pass only through
    the allowance ("allowance_only") and the largest allowance ("max_allowance")."""
    a_out, a_lse = (0.0, 0.0) if allow is None else allow
    g = out_gpu.float().cpu().double().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref_out)
    bare = ATOL + RTOL * np.abs(ref_out)
    excess = err - (bare + a_out)
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: out off by {err[worst]:.4g} at {worst} "
                               f"(ref {ref_out[worst]:.4g}, gpu {g[worst]:.4g})")
    if stats is not None:
        stats["allowance_only"] = int((err > bare).sum())
        stats["max_allowance"] = float(np.max(a_out)) if np.size(a_out) else 0.0
    num = np.linalg.norm(g - ref_out, axis=-1)
    den = np.linalg.norm(ref_out, axis=-1)
    slack = np.linalg.norm(np.broadcast_to(a_out, ref_out.shape), axis=-1)
    rel = np.where(den > 0, np.maximum(num - slack, 0) / np.maximum(den, 1e-300), num)
    assert rel.max() <= NORM_RTOL, f"{what}: norm-relative out error {rel.max():.3g}"
    lg = lse_gpu.cpu().double().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(ref_lse)), f"{what}: -inf lse pattern differs"
    fin = np.isfinite(ref_lse)
    assert np.isfinite(lg[fin]).all()
    al = np.broadcast_to(a_lse, ref_lse.shape)[fin]
    lex = np.abs(lg[fin] - ref_lse[fin]) - (ATOL + RTOL * np.abs(ref_lse[fin]) + al)
    assert lex.size == 0 or lex.max() <= 0, f"{what}: lse off by {lex.max():.3g} over tolerance"
    return float(rel.max())


def oracle_subproblem(w: W.Workload, indices: torch.Tensor, indptr: torch.Tensor, rows,
                      kv_gpu: torch.Tensor, gen_device="cuda", lens=None):
    """Records and remapped CSR of a sample of rows, for the oracle.

    The oracle packs the sampled rows' records itself from the generator's
    bf16 values; the bytes are compared with the GPU writer's (bit-exact).
    Returns (rec, idx_sub, indptr_sub, lens_sub) where indices point into rec
    (masked entries keep a masked value).
    """
    ind = indices.cpu().numpy()
    ptr = indptr.cpu().numpy()
    slices = [ind[max(ptr[r], 0):max(ptr[r + 1], ptr[r], 0)] for r in rows]
    cat = np.concatenate(slices) if slices else np.zeros(0, np.int32)
    valid = (cat >= 0) & (cat < w.n_kv_rows)
    ids = np.unique(cat[valid])
    lat, rope = W.latent_rows(w, torch.from_numpy(ids), gen_device)
    rec = oracle.pack_records(bits(lat), bits(rope))
    gpu_rec = kv_gpu[torch.from_numpy(ids).to(kv_gpu.device).long()].cpu().numpy()
    assert np.array_equal(gpu_rec, rec), "GPU record writer differs from the oracle's"
    remap = np.searchsorted(ids, np.where(valid, cat, 0))
    sub = np.where(valid, remap, np.where(cat < 0, -1, len(ids))).astype(np.int32)
    lens_sub = None
    if lens is not None:
        lens_sub = lens.cpu().numpy()[list(rows)]
    ptr_sub = np.concatenate([[0], np.cumsum([len(s) for s in slices])]).astype(np.int32)
    return rec, sub, ptr_sub, lens_sub


def tc_schedule(lens, G, tile=64, start_slots=2, tile_slots=1):
    """The tensor-core kernels' row parts, restated from smla.h: rows cut into
    tile-key tiles; row r takes start_slots schedule slots and then tile_slots
    slots per tile, in row order; CTA c takes slots [c W / G, (c+1) W / G) and
    the tiles whose first slot lies there; a part of a shared row lands in
    slot 2 c + (R_r < b_c ? 0 : 1), R_r the first slot of the row's first
    tile.  Returns {row: [(cta, slot, first position, end position), ...]}."""
    tiles = [max(1, -(-L // tile)) for L in lens]
    starts = np.concatenate([[0], np.cumsum([start_slots + tile_slots * n for n in tiles])]).astype(np.int64)
    W = int(starts[-1])
    b = [c * W // G for c in range(G + 1)]
    parts = {}
    for r, L in enumerate(lens):
        R, nt = int(starts[r]) + start_slots, tiles[r]
        for c in range(G):
            # the tiles t with R + tile_slots t in [b_c, b_c+1)
            lo_t = min(nt, max(0, -(-(b[c] - R) // tile_slots)))
            hi_t = min(nt, max(0, -(-(b[c + 1] - R) // tile_slots)))
            if lo_t < hi_t:
                slot = 2 * c + (0 if R < b[c] else 1)
                parts.setdefault(r, []).append((c, slot, lo_t * tile, min(hi_t * tile, L)))
    return parts
