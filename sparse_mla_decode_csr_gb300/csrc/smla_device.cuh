// Device helpers shared by the decode kernels: row slicing and masking, the
// epilogue of an unsplit row, and the split-KV combine.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "smla_internal.h"

namespace smla {

// Device-side copy of what a decode kernel reads (plain pointers, no structs
// with host-only members).
struct DecodeArgs {
  const uint16_t* q;
  int64_t q_stride_row, q_stride_head;
  const uint8_t* kv;
  int64_t n_kv_rows;
  const int32_t* indices;
  int64_t n_indices;
  const int32_t* indptr;
  const int32_t* lens;
  const float* sink;
  uint16_t* out;
  int64_t out_stride_row, out_stride_head;
  float* lse;
  int32_t* n_valid;
  int32_t* status;
  float sm_scale_log2;  // sm_scale * log2(e): scores are kept in log2 units
  int32_t n_q, heads, splits, chunk_len, has_invalid;
  int32_t grid, merge_kernel;  // tensor-core schedule
  int32_t merge_min_parts;     // the merge kernel leaves rows of fewer parts alone
  int32_t head_groups;         // native-fp8 kernel: CTAs per schedule range (heads split)
  int32_t row_start_slots;     // tensor-core schedule: slots charged for starting a row
  int32_t tile_slots;          //   and slots per tile (a tile belongs to the CTA holding its first slot)
  // split workspace
  int32_t* ticket;
  int64_t* row_tile;  // tensor-core schedule: first tile of each row, then T
  float* o_part;
  float* ml_part;
  int32_t* nv_part;
};

// Schedule slots charged for starting a row (its epilogue and q staging cost
// about two tiles of pipeline time): row r occupies kRowStartSlots virtual
// slots and then its T_r tiles in the slot space the CTAs split evenly.
constexpr int kRowStartSlots = 2;  // (the bf16 kernel's charge; see DecodeArgs::row_start_slots)

inline DecodeArgs make_decode_args(const DecodeLaunch& L) {
  DecodeArgs a{};
  const smla_decode_params& p = L.p;
  a.q = static_cast<const uint16_t*>(p.q);
  a.q_stride_row = p.q_stride_row;
  a.q_stride_head = p.q_stride_head;
  a.kv = static_cast<const uint8_t*>(p.kv_cache);
  a.n_kv_rows = p.n_kv_rows;
  a.indices = p.indices;
  a.n_indices = p.n_indices;
  a.indptr = p.indptr;
  a.lens = p.lens;
  a.sink = p.sink;
  a.out = static_cast<uint16_t*>(p.out);
  a.out_stride_row = p.out_stride_row;
  a.out_stride_head = p.out_stride_head;
  a.lse = p.lse;
  a.n_valid = p.n_valid;
  a.status = p.status;
  a.sm_scale_log2 = p.sm_scale * kLog2e;
  a.n_q = p.n_q;
  a.heads = p.num_heads;
  a.splits = L.plan.num_splits;
  a.chunk_len = L.plan.chunk_len;
  a.has_invalid = p.has_invalid;
  a.grid = L.plan.grid;
  a.merge_kernel = L.plan.merge_kernel;
  // the native-fp8 kernel merges rows of up to kMaxInKernelParts parts itself
  a.merge_min_parts = L.plan.kernel == SMLA_KERNEL_TENSOR_CORE_FP8 ? kMaxInKernelParts + 1 : 2;
  a.head_groups = L.plan.head_groups > 0 ? L.plan.head_groups : 1;
  a.row_start_slots = kRowStartSlots;  // (the native-fp8 launcher sets its own)
  a.tile_slots = 1;
  if (L.ws.total > 0) {
    char* ws = static_cast<char*>(L.workspace);
    a.ticket = reinterpret_cast<int32_t*>(ws + L.ws.ticket_off);
    a.row_tile = reinterpret_cast<int64_t*>(ws + L.ws.rowtile_off);
    a.o_part = reinterpret_cast<float*>(ws + L.ws.o_off);
    a.ml_part = reinterpret_cast<float*>(ws + L.ws.ml_off);
    a.nv_part = reinterpret_cast<int32_t*>(ws + L.ws.nv_off);
  }
  return a;
}

// The (row, chunk) unit of a CTA and the slice positions it covers.  Rows are
// taken in reverse order, so that under a causal index pattern the long tail
// rows start first (the gfx950 page issues its rows the same way).
struct Unit {
  int32_t row, chunk;
  int64_t beg;   // offset of the row's slice in indices[]
  int32_t p0, p1;  // positions [p0, p1) of the slice handled here
};

__device__ __forceinline__ Unit unit_of(const DecodeArgs& a, int32_t unit_id) {
  Unit u;
  u.row = a.n_q - 1 - unit_id / a.splits;
  u.chunk = unit_id % a.splits;
  const int64_t beg = a.indptr[u.row];
  const int64_t end = a.indptr[u.row + 1];
  int64_t len = end - beg;
  if (len < 0) len = 0;
  if (a.lens) {
    const int64_t cap = a.lens[u.row];
    len = cap < len ? (cap < 0 ? 0 : cap) : len;
  }
  if (len > INT32_MAX) len = INT32_MAX;
  const int64_t c0 = int64_t(u.chunk) * a.chunk_len;
  int64_t c1 = (u.chunk == a.splits - 1) ? len : c0 + a.chunk_len;
  if (c1 > len) c1 = len;
  u.beg = beg;
  u.p0 = int32_t(c0 < len ? c0 : len);
  u.p1 = int32_t(c1 > u.p0 ? c1 : u.p0);
  return u;
}

// Record row of slice position p, or -1 when the position is masked: offset
// outside the index buffer, entry < 0, or entry >= n_kv_rows (flagged).
__device__ __forceinline__ int32_t key_of(const DecodeArgs& a, int64_t beg, int32_t p) {
  const int64_t off = beg + p;
  if (off < 0 || off >= a.n_indices) return -1;
  const int32_t idx = __ldg(a.indices + off);
  if (idx >= a.n_kv_rows) {
    if (a.status) atomicOr(a.status, SMLA_STATUS_INDEX_OOB);
    return -1;
  }
  return idx < 0 ? -1 : idx;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Output factor and LSE of one head from its final (m, l) in log2 units:
//   out = acc * factor, factor = 2^(m - m_f) / (2^(s - m_f) + l 2^(m - m_f)),
//   m_f = max(m, s), s = sink * log2(e)        (the K2-back combine's fold)
//   lse = (m + log2 l) * ln 2                  (the gfx950 epilogue's LSE)
// and factor = 0, lse = -inf when l == 0 (no key); a NaN l (a NaN score)
// gives NaN for both.  finish_head_v takes the head's sink value already
// loaded (has_sink: a sink is given).
__device__ __forceinline__ void finish_head_v(float m, float l, bool has_sink, float sink_h, float* factor,
                                              float* lse) {
  if (l == 0.f) {
    *factor = 0.f;
    *lse = -INFINITY;
    return;
  }
  // (hardware approximations, relative error ~2^-21: out is bf16 and the
  // LSE is compared at 1e-2; the accurate library forms are long code paths
  // run once per row at a kernel's end)
  *lse = (m + __log2f(l)) * kLn2;
  if (!has_sink) {
    *factor = __fdividef(1.f, l);
    return;
  }
  const float s = sink_h * kLog2e;
  const float mf = fmaxf(m, s);
  const float wm = exp2f(m - mf);
  *factor = __fdividef(wm, exp2f(s - mf) + l * wm);
}

__device__ __forceinline__ void finish_head(float m, float l, const float* sink, int h,
                                            float* factor, float* lse) {
  finish_head_v(m, l, sink != nullptr, sink != nullptr ? sink[h] : 0.f, factor, lse);
}

}  // namespace smla

namespace smla {

// ---- the tensor-core kernel's balanced schedule (see smla_plan in smla.h) ----

constexpr int kSchedTile = 64;
// Slice length of row r: max(indptr[r+1] - indptr[r], 0), capped by lens.
__device__ __forceinline__ int32_t row_len(const DecodeArgs& a, int32_t r) {
  int64_t len = int64_t(__ldg(a.indptr + r + 1)) - __ldg(a.indptr + r);
  if (len < 0) len = 0;
  if (a.lens) {
    const int64_t cap = __ldg(a.lens + r);
    len = cap < len ? (cap < 0 ? 0 : cap) : len;
  }
  return int32_t(len > INT32_MAX ? INT32_MAX : len);
}

// Tiles of a row: every row has at least one (an empty row's tile has no keys
// and yields out = 0, lse = -inf).
__device__ __forceinline__ int32_t tiles_of_len(int32_t len) {
  return len > 0 ? (len + kSchedTile - 1) / kSchedTile : 1;
}

// First tile of CTA c: floor(c T / G).
__device__ __forceinline__ int64_t cta_begin(int64_t c, int64_t T, int64_t G) { return (c * T) / G; }

// The CTA whose range holds tile t: the largest c with floor(c T / G) <= t.
__device__ __forceinline__ int64_t cta_of_tile(int64_t t, int64_t T, int64_t G) {
  return ((t + 1) * G - 1) / T;
}

// Whether CTA c holds a tile of a row whose nt tiles start at slots
// F + S t (S a power of two): a tile belongs to the CTA whose range holds
// its first slot.
__device__ __forceinline__ bool cta_holds_tile(int64_t c, int64_t F, int32_t nt, int64_t S, int64_t T, int64_t G) {
  const int64_t b = cta_begin(c, T, G), e = cta_begin(c + 1, T, G);
  const int sh = __ffsll(S) - 1;  // (a shift, not a 64-bit division)
  const int64_t lo = b > F ? (b - F + S - 1) >> sh : 0;
  const int64_t hi = e > F ? (e - F + S - 1) >> sh : 0;
  return (hi < nt ? hi : nt) > (lo < nt ? lo : nt);
}

// Partial slot of row part (CTA c, row starting at tile P).
__device__ __forceinline__ int64_t part_slot(int64_t c, int64_t P, int64_t T, int64_t G) {
  return 2 * c + (P < cta_begin(c, T, G) ? 0 : 1);
}

}  // namespace smla
