// Sparse MLA decode with native-fp8 products on the 5th-generation tensor
// cores (tcgen05.mma kind::mxf8f6f4, block-scaled), persistent and balanced.
//
// The fp8_ds_mla records are gathered straight into the shared-memory operand
// layout of the MMAs (16-byte cp.async per lane, 128-byte swizzled rows): the
// 512 E4M3 latent bytes of a key are used as they are, with no conversion.
//
//   QK   S[128 keys, 2 HP] = K_lat[128 x 512] . [q_hi | q_lo]^T  (E4M3 x E4M3,
//        block-scaled: the record's power-of-two scale of each 128-dim block is
//        the E8M0 scale factor of the key rows, a per-(head, 32-dim block)
//        power of two normalises q) + K_rope[128 x 64] . q_rope^T (bf16).
//        q (bf16, 8 significant bits) is split into q_hi + q_lo, two E4M3
//        values with 4 significant bits each, in the N columns of the same MMA:
//        s = S[:, h] + S[:, HP + h] is q.k with every product exact.
//   softmax on S in log2 units with a lazily moved per-head reference max.
//   PV   O^T[128 dims, 2 HP] += V^T[128 dims x 32 keys] . [P'_hi | P'_lo]
//        (E4M3 x E4M3, block-scaled), four 128-dim blocks b.  V^T is the same
//        landed latent tile read MN-major.  The key's scale of block b is
//        folded into P'_b = p * scale_b, split hi + lo like q, with an E8M0
//        scale factor per (head, block) taken from the tile's maxima, so that
//        P' carries ~8 significant bits (as a bf16 P would) down to 2^-18 of
//        the tile's largest term.  O = O_hi + O_lo.
//
// Warp roles (16 warps, 512 threads, one CTA per SM):
//   0-3   softmax (warp q owns the keys of TMEM lane quarter q of S)
//   4-7   aux: E8M0 scale factors of each landed tile into TMEM, q staging
//         (hi/lo split and its scale factors) per row part, and each row
//         part's epilogue (out / lse or a partial of a shared row)
//   8     QK issuer (16 block-scaled K-steps and 4 bf16 rope K-steps, one
//         accumulator), 9 PV issuer (dim blocks one after another: a thread
//         issues one MMA every ~130 cycles into one accumulator and slower
//         when consecutive MMAs alternate accumulators)
//   10-15 loaders: keys lw, lw + 6, ... of every 128-key tile (64-bit record
//         addressing, masked keys zero-filled, out-of-range entries flagged)
//
// The schedule is that of the bf16 tensor-core kernel with 128-key tiles: rows
// cut into tiles, two start slots per row, CTA c takes the slots
// [floor(c W / G), floor((c+1) W / G)); rows shared between CTAs leave
// partials merged by the merge kernel.
//
// The maths is the sparse softmax attention of the gfx950 FlyDSL page (module
// docstring: record layout, CSR tiles, masking; its latent QK runs as a scaled
// fp8 MFMA with the record scale and q split hi + lo, which this kernel
// restates for tcgen05) with the sink folded as the DeepSeek-V4.1 "K2 back"
// page's stage_combine does.  The SM100 Mojo page's FP8 tcgen05 design is
// prior art; its TMA gather4 front end measured slower here than LSU gathers.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kTK = 128;        // keys per tile (M of QK)
constexpr int kHP = 16;         // padded heads
constexpr int kN = 2 * kHP;     // N of QK and PV: hi columns, then lo columns
constexpr int kStages = 2;
constexpr int kSoftmaxWarps = 4;
constexpr int kAuxWarp0 = 4;
constexpr int kQkWarp0 = 8;
constexpr int kPvWarp0 = 9;
constexpr int kLoadWarp0 = 10;
constexpr int kLoadWarps = 6;
constexpr int kKeysPerLoader = (kTK + kLoadWarps - 1) / kLoadWarps;  // 22 (keys lw, lw + 6, ...)
constexpr int kRowStart = 2;                      // schedule slots charged for starting a row
constexpr float kLazy = 16.f;                     // reference max moves when passed by > 2^16
constexpr float kInitMax = -1.0e30f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait

// ---- shared memory (bytes from a 1024-aligned base) ----
constexpr int kChunk = kTK * 128;                       // one 128-byte column block of a tile (16 KB)
constexpr int kOffRope = 4 * kChunk;
constexpr int kOffSc = 5 * kChunk;                      // scales: kTK x 16 B
constexpr int kOffIds = kOffSc + kTK * 16;              // record ids (or -1): kTK x 4 B
constexpr int kStageBytes = (kOffIds + kTK * 4 + 1023) / 1024 * 1024;
constexpr int kQLatChunk = kN * 128;                    // one K-chunk of [q_hi | q_lo] (4 KB)
constexpr int kQOffRope = 4 * kQLatChunk;
constexpr int kQBytes = (kQOffRope + kHP * 128 + 1023) / 1024 * 1024;
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kPBlock = 32 * kN;                        // P' of one 32-key chunk and dim block (1 KB)
constexpr int kOffP = kOffQ + 2 * kQBytes;
constexpr int kOffBar = kOffP + 16 * kPBlock;
constexpr int kNumBars = 32;
constexpr int kOffMisc = kOffBar + kNumBars * 8;

// ---- TMEM columns ----
constexpr uint32_t kColS = 0;      // S: [buffer] x kN
constexpr uint32_t kColO = 128;    // O: [buffer][block] x kN
constexpr uint32_t kColSfa = 384;  // record scale factors: [stage] x 16
constexpr uint32_t kColSfq = 416;  // q scale factors: [q buffer] x 16
constexpr uint32_t kColSfv = 448;  // V^T scale factors (all 1; 16 columns written, 4 read)
constexpr uint32_t kColSfp = 464;  // P' scale factors (byte b: dim block b)
constexpr uint32_t kTmemCols = 512;

__host__ __device__ constexpr uint32_t s_col(int sb) { return kColS + uint32_t(sb) * kN; }
__host__ __device__ constexpr uint32_t o_col(int ob, int b) { return kColO + uint32_t(4 * ob + b) * kN; }

struct Misc {
  uint32_t tmem_base;
  int32_t abort;
  int32_t first_row;
  int32_t n_tiles;
  int64_t first_tile;
  int64_t total_tiles;
  int64_t scan[64];
  int32_t red_max_t[2][kHP][kSoftmaxWarps];  // tile maxima per head and warp (order-preserving ints)
  int32_t red_sc[2][kSoftmaxWarps][4];     // largest biased exponent of each block's scale per warp
  float red_l[kSoftmaxWarps][kHP];
  int32_t red_nv[kSoftmaxWarps];
  float part_m[2][kHP];                 // per O buffer: a finished row part's (m, l, count)
  float part_l[2][kHP];
  int32_t part_nv[2];
  uint8_t sfq[kN][16];                  // q scale-factor bytes of the part being staged
};
constexpr int kSmemUsed = kOffMisc + int(sizeof(Misc));
constexpr int kSmemTotal = kSmemUsed + 1024;  // slack to align the base
static_assert(kSmemTotal <= 232448, "shared memory over the per-block limit");

enum Bar {
  kKvFull = 0,    // [2] loaders -> aux (tile landed)
  kKvEmpty = 2,   // [2] PV issuers -> loaders (tile consumed)
  kSfReady = 4,   // [2] aux -> QK issuers (scale factors in TMEM)
  kSFull = 6,     // [2] QK issuers -> softmax
  kSEmpty = 8,    // [2] softmax -> QK issuers
  kPFull = 10,    // softmax -> PV issuers (P' and its scale factors written)
  kPvDone = 11,   // PV issuers -> softmax (P' buffer free, O quiescent)
  kQFull = 12,    // [2] aux -> QK issuers
  kQEmpty = 14,   // [2] QK issuers -> aux
  kOFull = 16,    // [2] PV issuers -> aux (a part's O complete)
  kOEmpty = 18,   // [2] aux -> PV issuers and softmax (O buffer read out)
  kEpiReady = 20  // [2] softmax -> aux (a part's m, l, count posted)
};

__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t chunk16) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + (((chunk16 ^ r) & 7u) << 4);
}

// order-preserving int of a float (for integer max reductions)
__device__ __forceinline__ int32_t ord(float x) {
  const int32_t b = __float_as_int(x);
  return b >= 0 ? b : b ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float unord(int32_t o) { return __int_as_float(o >= 0 ? o : o ^ 0x7FFFFFFF); }

__device__ __forceinline__ float pow2f(int e) {  // 2^e for -126 <= e <= 127
  return __int_as_float((e + 127) << 23);
}

// hi = E4M3(x), lo = E4M3(x - hi) for a pair (round to nearest even, saturating)
__device__ __forceinline__ void split_pair(float x0, float x1, uint16_t& hi, uint16_t& lo) {
  hi = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  lo = __nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
}

struct Cursor {
  int32_t row, len, ntiles, ta, tb, t;
  int64_t P, beg, e;
  bool live;
  __device__ __forceinline__ static int32_t tiles_of(int32_t len) { return len > 0 ? (len + kTK - 1) / kTK : 1; }
  __device__ __forceinline__ void load_row(const DecodeArgs& a) {
    len = row_len(a, row);
    ntiles = tiles_of(len);
    beg = __ldg(a.indptr + row);
    const int64_t n = e - P;
    tb = int32_t(n < 0 ? 0 : (n < int64_t(ntiles) ? n : int64_t(ntiles)));
    if (tb <= 0) live = false;
  }
  __device__ __forceinline__ void init(const DecodeArgs& a, int32_t r0, int64_t P0, int64_t b, int64_t e_) {
    row = r0;
    P = P0 + kRowStart;
    e = e_;
    live = b < e_ && r0 < a.n_q;
    ta = tb = t = 0;
    if (!live) return;
    load_row(a);
    ta = int32_t(b > P ? b - P : 0);
    t = ta;
  }
  __device__ __forceinline__ void advance(const DecodeArgs& a) {
    if (!live) return;
    if (++t < tb) return;
    P += ntiles + kRowStart;
    ++row;
    if (P - kRowStart >= e || row >= a.n_q) {
      live = false;
      return;
    }
    load_row(a);
    ta = 0;
    t = 0;
  }
  __device__ __forceinline__ bool first() const { return t == ta; }
  __device__ __forceinline__ bool last() const { return t == tb - 1; }
  __device__ __forceinline__ bool whole() const { return ta == 0 && tb == ntiles; }
  __device__ __forceinline__ int32_t p0() const { return t * kTK; }
  __device__ __forceinline__ int32_t p1() const { return min(t * kTK + kTK, len); }
};

__device__ __forceinline__ void set_abort(Misc* ms, const DecodeArgs& a) {
  if (atomicExch(&ms->abort, 1) == 0 && a.status) atomicOr(a.status, SMLA_STATUS_TIMEOUT);
}

// A bounded pipeline wait; after any timeout every later wait returns false
// at once so that all roles reach the teardown.  Loops holding named barriers
// keep iterating after a failed wait (same barrier sequence in every thread).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Misc* ms, const DecodeArgs& a) {
  if (*reinterpret_cast<volatile int32_t*>(&ms->abort)) return false;
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  set_abort(ms, a);
  return false;
}
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, Misc* ms, const DecodeArgs& a) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, ms, a));
}

// Slot of a shared row part (the partial layout of the merge kernel).
__device__ __forceinline__ int64_t slot_of(int64_t c, int64_t P, int64_t T, int64_t G) {
  return 2 * c + (P < cta_begin(c, T, G) ? 0 : 1);
}

__global__ void __launch_bounds__(kThreads, 1) decode_fp8_kernel(DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  Misc* ms = reinterpret_cast<Misc*>(smem + kOffMisc);
  const int H = a.heads;
  const int64_t G = gridDim.x, c_id = blockIdx.x;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars + kKvFull + s, kLoadWarps);
      mbar_init(bars + kKvEmpty + s, 1);
      mbar_init(bars + kSfReady + s, 4);
      mbar_init(bars + kSFull + s, 1);
      mbar_init(bars + kSEmpty + s, kSoftmaxWarps);
      mbar_init(bars + kQFull + s, 4);
      mbar_init(bars + kQEmpty + s, 1);
      mbar_init(bars + kOFull + s, 1);
      mbar_init(bars + kOEmpty + s, 4);
      mbar_init(bars + kEpiReady + s, kSoftmaxWarps);
    }
    mbar_init(bars + kPFull, kSoftmaxWarps);
    mbar_init(bars + kPvDone, 1);
    ms->abort = 0;
    ms->first_row = a.n_q;
    ms->first_tile = 0;
    ms->n_tiles = 0;
    fence_mbar_init();
  }
  if (warp == kQkWarp0) {
    tmem_alloc(&ms->tmem_base, kTmemCols);
    tmem_relinquish();
  }

  // ---- schedule: slot counts of all rows, their prefix, this CTA's first row
  {
    const int n = a.n_q;
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min(tid * per, n), hi = min(lo + per, n);
    int64_t local = 0;
#pragma unroll 1
    for (int r = lo; r < hi; ++r) local += kRowStart + Cursor::tiles_of(row_len(a, r));
    int64_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) ms->scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int64_t v = lane < kThreads / 32 ? ms->scan[lane] : 0;
      int64_t t = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      if (lane < kThreads / 32) ms->scan[32 + lane] = t - v;
      if (lane == 31) ms->total_tiles = t;
    }
    __syncthreads();
    const int64_t Tt = ms->total_tiles;
    const int64_t b = cta_begin(c_id, Tt, G), e = cta_begin(c_id + 1, Tt, G);
    int64_t P = ms->scan[32 + warp] + x - local;
    int32_t mine = 0;
#pragma unroll 1
    for (int r = lo; r < hi; ++r) {
      const int32_t nt_r = Cursor::tiles_of(row_len(a, r));
      const int64_t w = kRowStart + nt_r;
      if (P <= b && b < P + w) {
        ms->first_row = r;
        ms->first_tile = P;
      }
      const int64_t t0 = P + kRowStart;
      const int64_t lo_t = b > t0 ? b : t0, hi_t = e < t0 + nt_r ? e : t0 + nt_r;
      if (hi_t > lo_t) mine += int32_t(hi_t - lo_t);
      if (c_id == 0 && a.row_tile) a.row_tile[r] = P;
      P += w;
    }
    if (c_id == 0 && tid == 0 && a.row_tile) a.row_tile[n] = Tt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (lane == 0 && mine != 0) atomicAdd(&ms->n_tiles, mine);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int64_t T = ms->total_tiles;
  const int64_t cb = cta_begin(c_id, T, G), ce = cta_begin(c_id + 1, T, G);
  const int32_t n_tiles = ms->n_tiles;
  const int32_t row0 = ms->first_row;
  const int64_t P0 = ms->first_tile;
  const uint32_t tmem = ms->tmem_base;
  const uint32_t smem_base = smem_u32(smem);

  if (warp < kSoftmaxWarps) {
    // =================== softmax ===================
    const int q = warp;
    const int t = 32 * q + lane;  // this thread's key row of the tile
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    float mref[kHP], lpart[kHP];
    int nv = 0;
#pragma unroll
    for (int h = 0; h < kHP; ++h) {
      mref[h] = kInitMax;
      lpart[h] = 0.f;
    }
    Cursor c;
    c.init(a, row0, P0, cb, ce);
    int pi = 0;  // row part index within this CTA
    for (int i = 0; i < n_tiles; ++i, c.advance(a)) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const bool first = c.first(), last = c.last();
      const int ob = pi & 1;
      const uint8_t* st = smem + s * kStageBytes;
      if (first) {
#pragma unroll
        for (int h = 0; h < kHP; ++h) lpart[h] = 0.f;
        nv = 0;
      }
      wait_warp(bars + kSFull + s, ph, ms, a);
      tc_fence_after();
      float x[kHP];
      {
        uint32_t r0[16], r1[16];
        tmem_ld16(tmem + lane_base + s_col(s), r0);       // q_hi columns (+ rope)
        tmem_ld16(tmem + lane_base + s_col(s) + 16, r1);  // q_lo columns
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kHP; ++h) x[h] = __uint_as_float(r0[h]) + __uint_as_float(r1[h]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + kSEmpty + s);
      wait_warp(bars + kKvFull + s, ph, ms, a);  // (already complete) orders the loaders' ids and scales
      const int32_t id = *reinterpret_cast<const int32_t*>(st + kOffIds + 4 * t);
      const bool valid = id >= 0;
      nv += valid;
#pragma unroll
      for (int h = 0; h < kHP; ++h) x[h] = valid ? x[h] * a.sm_scale_log2 : -INFINITY;
      // tile maxima per head and the largest exponent of each block's scale
      const int rb = i & 1;  // reduction buffer (a warp may run one tile ahead)
#pragma unroll
      for (int h = 0; h < kHP; ++h) {
        const int32_t m = __reduce_max_sync(0xffffffffu, ord(x[h]));
        if (lane == h) ms->red_max_t[rb][h][q] = m;
      }
      {
        const uint4 scw = *reinterpret_cast<const uint4*>(st + kOffSc + 16 * t);
        const uint32_t sw[4] = {scw.x, scw.y, scw.z, scw.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int32_t e = __reduce_max_sync(0xffffffffu, valid ? int32_t((sw[b] >> 23) & 0xFF) : 0);
          if (lane == b) ms->red_sc[rb][q][b] = e;
        }
      }
      named_barrier(1, 32 * kSoftmaxWarps);
      float tmax[kHP];  // the tile's maximum of each head (over all four warps)
#pragma unroll
      for (int h = 0; h < kHP; ++h) {
        const int4 m4 = *reinterpret_cast<const int4*>(&ms->red_max_t[rb][h][0]);
        tmax[h] = unord(max(max(m4.x, m4.y), max(m4.z, m4.w)));
      }
      bool pv_waited = false;
      if (first) {
#pragma unroll
        for (int h = 0; h < kHP; ++h) {
          const float tm = tmax[h];
          mref[h] = (tm > kInitMax || tm != tm) ? tm : kInitMax;  // a NaN score keeps the row NaN
        }
      } else {
        bool need = false;
#pragma unroll
        for (int h = 0; h < kHP; ++h) need |= tmax[h] > mref[h] + kLazy;
        if (need) {  // uniform: every thread sees the same maxima
          // O holds PV of this part's earlier tiles: wait until they completed
          wait_warp(bars + kPvDone, (i - 1) & 1, ms, a);
          pv_waited = true;
          tc_fence_after();
          float alpha[kHP];
#pragma unroll
          for (int h = 0; h < kHP; ++h) {
            const float tm = tmax[h];
            const float mn = tm > mref[h] + kLazy ? tm : mref[h];
            alpha[h] = exp2f(mref[h] - mn);
            mref[h] = mn;
            lpart[h] *= alpha[h];
          }
#pragma unroll 1
          for (int k = 0; k < 8; ++k) {  // 4 blocks x (hi, lo) column groups of 16
            uint32_t v[16];
            const uint32_t ta = tmem + lane_base + o_col(ob, k >> 1) + 16 * (k & 1);
            tmem_ld16(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < kHP; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * alpha[h]);
            tmem_st16(ta, v);
          }
          tmem_wait_st();
        }
      }
      // p = 2^(x - mref); P'_b = p * scale_b in units of the E8M0 factor
      // 2^E(h, b), E = e_h + es_b - 8, where pmax_h = 2^(tmax_h - mref_h) < 2^e_h
      // and the tile's largest block-b scale < 2^es_b: P' / 2^E < 2^8 <= 448.
      // e_h is kept >= -20 (a head whose tile terms all lie 2^20 below its
      // reference keeps 2^-10 relative precision on them).  x becomes p 2^-e_h.
      int e_mine = 0;  // e_h of this lane's head (lane mod kHP), for the scale factors
#pragma unroll
      for (int h = 0; h < kHP; ++h) {
        const float p = exp2f(x[h] - mref[h]);  // x = -inf (masked) gives 0
        lpart[h] += p;
        const float pmax = exp2f(tmax[h] - mref[h]);
        int e = int((__float_as_uint(pmax) >> 23) & 0xFF) - 126;
        e = max(min(e, 17), -20);
        x[h] = p * pow2f(-e);
        if ((lane & (kHP - 1)) == h) e_mine = e;
      }
      if (i > 0 && !pv_waited) wait_warp(bars + kPvDone, (i - 1) & 1, ms, a);  // P' buffer free
      uint32_t sf_word = 0;
      {
        const int chunk = q;  // this warp's 32 keys
        uint32_t off0 = uint32_t(lane) * kN, off1 = off0 + 16;
        off0 ^= ((off0 >> 7) & 1u) << 4;
        off1 ^= ((off1 >> 7) & 1u) << 4;
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
          int32_t esb = ms->red_sc[rb][0][b];
#pragma unroll
          for (int w = 1; w < kSoftmaxWarps; ++w) esb = max(esb, ms->red_sc[rb][w][b]);
          const int es = max(esb, 1) - 126;  // the tile's block-b scales < 2^es
          sf_word |= uint32_t(min(max(e_mine + es - 8 + 127, 1), 254)) << (8 * b);
          const uint32_t scale_b = *reinterpret_cast<const uint32_t*>(st + kOffSc + 16 * t + 4 * b);
          const float sn = __uint_as_float(scale_b) * pow2f(min(max(8 - es, -126), 127));  // scale_b 2^(8 - es)
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int k = 0; k < kHP / 2; ++k) {
            uint16_t h2, l2;
            split_pair(x[2 * k] * sn, x[2 * k + 1] * sn, h2, l2);
            if (k & 1) {
              hw[k >> 1] |= uint32_t(h2) << 16;
              lw[k >> 1] |= uint32_t(l2) << 16;
            } else {
              hw[k >> 1] = h2;
              lw[k >> 1] = l2;
            }
          }
          uint8_t* blk = smem + kOffP + (4 * chunk + b) * kPBlock;
          *reinterpret_cast<uint4*>(blk + off0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(blk + off1) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      // P' scale factors: B row n (hi head n, lo head n - HP) of every dim block
      // b in byte b, the same in every TMEM lane quarter
      tmem_st1(tmem + lane_base + kColSfp, sf_word);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + kPFull);
      if (last) {
        // the part's l and count over its keys, for the aux warps' epilogue
#pragma unroll
        for (int h = 0; h < kHP; ++h) {
          float v = lpart[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == h) ms->red_l[q][h] = v;
        }
        const int32_t nvw = __reduce_add_sync(0xffffffffu, nv);
        if (lane == 0) ms->red_nv[q] = nvw;
        // the slot (m, l) of this O buffer was read by the epilogue two parts ago
        wait_warp(bars + kOEmpty + ob, ((pi >> 1) & 1) ^ 1, ms, a);
        named_barrier(1, 32 * kSoftmaxWarps);
        if (q == 0) {
          if (lane < kHP) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < kSoftmaxWarps; ++w) l += ms->red_l[w][lane];
            float m = mref[0];
#pragma unroll
            for (int k = 1; k < kHP; ++k) m = (k == lane) ? mref[k] : m;
            ms->part_m[ob][lane] = m;
            ms->part_l[ob][lane] = l;
          }
          if (lane == 0) {
            int32_t n = 0;
#pragma unroll
            for (int w = 0; w < kSoftmaxWarps; ++w) n += ms->red_nv[w];
            ms->part_nv[ob] = n;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + kEpiReady + ob);
        ++pi;
      }
    }
  } else if (warp < kQkWarp0) {
    // =================== aux: scale factors, q staging, epilogues ===================
    const int q = warp - kAuxWarp0;  // TMEM lane quarter
    const int ta = 32 * q + lane;    // 0..127
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    // V^T scale factors: 1 (E8M0 127) for every dim row and key block
    {
      uint32_t v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = 0x7F7F7F7Fu;
      tmem_st16(tmem + lane_base + kColSfv, v);
      tmem_wait_st();
    }
    // q of a row -> [q_hi | q_lo] E4M3 (K-major, 128-byte swizzled) with an
    // E8M0 factor per (head, 32 dims) that brings the block's largest |q| to
    // [2^7, 2^8); q_rope (bf16) copied as it is; then the factors into TMEM.
    auto stage_q = [&](int row, int qb) {
      uint8_t* qs = smem + kOffQ + qb * kQBytes;
#pragma unroll 1
      for (int blk = ta; blk < kHP * 16; blk += 128) {
        const int h = blk >> 4, kb = blk & 15;
        uint32_t hw[8], lw[8];
        int sfb = 127;
        if (h < H) {
          const uint4* src = reinterpret_cast<const uint4*>(a.q + row * a.q_stride_row + h * a.q_stride_head + 32 * kb);
          uint4 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) v[k] = __ldg(src + k);
          float f[32];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              f[8 * k + 2 * j] = __uint_as_float(w[j] << 16);
              f[8 * k + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
          }
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(f[k]));
          int e = amax > 0.f ? int((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 7 : 0;
          e = max(min(e, 120), -120);
          sfb = e + 127;
          const float inv = pow2f(-e);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            uint16_t h2, l2;
            split_pair(f[2 * k] * inv, f[2 * k + 1] * inv, h2, l2);
            if (k & 1) {
              hw[k >> 1] |= uint32_t(h2) << 16;
              lw[k >> 1] |= uint32_t(l2) << 16;
            } else {
              hw[k >> 1] = h2;
              lw[k >> 1] = l2;
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) hw[k] = lw[k] = 0u;
        }
        const int kc = kb >> 2, c0 = 2 * (kb & 3);
        uint8_t* base = qs + kc * kQLatChunk;
        *reinterpret_cast<uint4*>(base + sw128(h, c0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(base + sw128(h, c0 + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        *reinterpret_cast<uint4*>(base + sw128(kHP + h, c0)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        *reinterpret_cast<uint4*>(base + sw128(kHP + h, c0 + 1)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        ms->sfq[h][kb] = uint8_t(sfb);
        ms->sfq[kHP + h][kb] = uint8_t(sfb);
      }
      {  // rope: kHP rows x 128 bytes, one 16-byte chunk per thread
        const int h = ta >> 3, c16 = ta & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (h < H)
          v = __ldg(reinterpret_cast<const uint4*>(a.q + row * a.q_stride_row + h * a.q_stride_head + kLatent + 8 * c16));
        *reinterpret_cast<uint4*>(qs + kQOffRope + sw128(h, c16)) = v;
      }
      named_barrier(2, 128);
      {
        // q factors: row n = lane (row group 0), K-block group g in column 4 g,
        // byte k = K-block 4 g + k; the other columns of each group unused
        uint32_t v[16];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          v[4 * g] = *reinterpret_cast<const uint32_t*>(&ms->sfq[lane][4 * g]);
          v[4 * g + 1] = v[4 * g + 2] = v[4 * g + 3] = 0x7F7F7F7Fu;
        }
        tmem_st16(tmem + lane_base + kColSfq + 16 * qb, v);
        tmem_wait_st();
      }
      named_barrier(2, 128);  // sfq is reused by the next staging
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + kQFull + qb);
    };
    auto epilogue = [&](const Cursor& pc, int pi) {
      const int ob = pi & 1;
      const uint32_t ph = (pi >> 1) & 1;
      wait_warp(bars + kEpiReady + ob, ph, ms, a);
      wait_warp(bars + kOFull + ob, ph, ms, a);
      tc_fence_after();
      const int row = pc.row;
      const bool whole = pc.whole();
      int64_t slot = 0;
      if (!whole) slot = slot_of(c_id, pc.P, T, G);
      float fac[kHP];
#pragma unroll
      for (int h = 0; h < kHP; ++h) {
        float lse_h;
        if (whole) finish_head(ms->part_m[ob][h], ms->part_l[ob][h], a.sink, h < H ? h : 0, &fac[h], &lse_h);
        else fac[h] = 1.f;
      }
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        uint32_t v0[16], v1[16];
        tmem_ld16(tmem + lane_base + o_col(ob, b), v0);
        tmem_ld16(tmem + lane_base + o_col(ob, b) + 16, v1);
        tmem_wait_ld();
        const int d = 128 * b + ta;
        if (whole) {
          uint16_t* dst = a.out + int64_t(row) * a.out_stride_row + d;
#pragma unroll
          for (int h = 0; h < kHP; ++h) {
            if (h < H) {
              const float o = (__uint_as_float(v0[h]) + __uint_as_float(v1[h])) * fac[h];
              dst[int64_t(h) * a.out_stride_head] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
            }
          }
        } else {
          float* dst = a.o_part + (slot * H) * kLatent + d;
#pragma unroll
          for (int h = 0; h < kHP; ++h)
            if (h < H) dst[int64_t(h) * kLatent] = __uint_as_float(v0[h]) + __uint_as_float(v1[h]);
        }
      }
      if (ta < H) {
        const float m = ms->part_m[ob][ta], l = ms->part_l[ob][ta];
        if (whole) {
          float f, lse_h;
          finish_head(m, l, a.sink, ta, &f, &lse_h);
          if (a.lse) a.lse[int64_t(row) * H + ta] = lse_h;
        } else {
          reinterpret_cast<float2*>(a.ml_part)[slot * H + ta] = make_float2(m, l);
        }
      }
      if (ta == 0) {
        if (whole) {
          if (a.n_valid) a.n_valid[row] = ms->part_nv[ob];
        } else {
          a.nv_part[slot] = ms->part_nv[ob];
        }
      }
      tc_fence_before();
      named_barrier(2, 128);  // every aux thread read the part's (m, l) and O
      if (lane == 0) mbar_arrive(bars + kOEmpty + ob);
    };
    Cursor c;
    c.init(a, row0, P0, cb, ce);
    if (n_tiles > 0) stage_q(c.row, 0);
    Cursor prev = c;
    int pi = 0;  // part of tile i
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const uint8_t* st = smem + s * kStageBytes;
      // (1) the tile's record scale factors: row t = key, column 4 g + j holds
      // rows 32 j + lane, every byte the E8M0 of scale block g
      wait_warp(bars + kKvFull + s, ph, ms, a);
      {
        uint32_t v[16];
        bool foreign = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(st + kOffSc + 16 * (32 * j + lane));
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t e = (w[g] >> 23) & 0xFFu;
            // a positive normal power of two (any the writer makes) or zero
            foreign |= !(w[g] == 0u || ((w[g] & 0x807FFFFFu) == 0u && e != 0u && e != 0xFFu));
            v[4 * g + j] = e * 0x01010101u;
          }
        }
        tmem_st16(tmem + lane_base + kColSfa + 16 * s, v);
        tmem_wait_st();
        if (__any_sync(0xffffffffu, foreign) && lane == 0 && a.status) atomicOr(a.status, SMLA_STATUS_FOREIGN_SCALE);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + kSfReady + s);
      // (2) the previous part's epilogue, once this part has started
      if (i > 0 && c.first()) {
        epilogue(prev, pi - 1);
      }
      // (3) the next part's q, as soon as its buffer is free
      if (c.last() && i + 1 < n_tiles) {
        const int qb = (pi + 1) & 1;
        wait_warp(bars + kQEmpty + qb, (((pi + 1) >> 1) & 1) ^ 1, ms, a);
        stage_q(c.row + 1, qb);
      }
      if (c.last()) {
        prev = c;
        ++pi;
      }
      c.advance(a);
    }
    if (pi > 0) epilogue(prev, pi - 1);
  } else if (warp < kPvWarp0) {
    // =================== QK issuer ===================
    Cursor c;
    c.init(a, row0, P0, cb, ce);
    int pi = 0;
    for (int i = 0; i < n_tiles; ++i, c.advance(a)) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const int qb = pi & 1;
      const bool first = c.first(), last = c.last();
      wait_warp(bars + kSfReady + s, ph, ms, a);
      wait_warp(bars + kSEmpty + s, ph ^ 1, ms, a);
      if (first) wait_warp(bars + kQFull + qb, (pi >> 1) & 1, ms, a);
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = smem_base + s * kStageBytes;
        const uint32_t qs = smem_base + kOffQ + qb * kQBytes;
        const uint32_t d = tmem + s_col(s);
        // latent: 16 K-steps of 32 E4M3 (K-chunk kc = 128 dims = scale block kc)
#pragma unroll 1
        for (int ks = 0; ks < 16; ++ks) {
          const int kc = ks >> 2, sub = ks & 3;
          const uint64_t ad = smem_desc(st + kc * kChunk + 32 * sub, 16, 1024, kSw128);
          const uint64_t bd = smem_desc(qs + kc * kQLatChunk + 32 * sub, 16, 1024, kSw128);
          mma_mxf8_ss(d, ad, bd, idesc_mxf8(128, kN, 0, 0, sub, sub), tmem + kColSfa + 16 * s + 4 * kc,
                      tmem + kColSfq + 16 * qb + 4 * kc, ks > 0 ? 1u : 0u);
        }
        // rope: 4 K-steps of 16 bf16 into the q_hi columns
#pragma unroll 1
        for (int r = 0; r < 4; ++r) {
          const uint64_t ad = smem_desc(st + kOffRope + 32 * r, 16, 1024, kSw128);
          const uint64_t bd = smem_desc(qs + kQOffRope + 32 * r, 16, 1024, kSw128);
          mma_f16_ss(d, ad, bd, idesc_bf16(128, kHP, 0, 0), 1u);
        }
        mma_commit(bars + kSFull + s);
        if (last) mma_commit(bars + kQEmpty + qb);
      }
      __syncwarp();
      if (last) ++pi;
    }
  } else if (warp < kLoadWarp0) {
    // =================== PV issuer ===================
    Cursor c;
    c.init(a, row0, P0, cb, ce);
    int pi = 0;
    for (int i = 0; i < n_tiles; ++i, c.advance(a)) {
      const int s = i & 1;
      const int ob = pi & 1;
      const bool first = c.first(), last = c.last();
      wait_warp(bars + kPFull, i & 1, ms, a);
      if (first) wait_warp(bars + kOEmpty + ob, ((pi >> 1) & 1) ^ 1, ms, a);
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = smem_base + s * kStageBytes;
        // block-major: consecutive MMAs accumulate into the same O block
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            // V^T: dims of block b (M, contiguous) x keys 32 ch .. (K, rows)
            const uint64_t ad = smem_desc(st + b * kChunk + ch * 4096, 16384, 1024, kSw128);
            const uint64_t bd = smem_desc(smem_base + kOffP + (4 * ch + b) * kPBlock, 256, 256, kSw32);
            mma_mxf8_ss(tmem + o_col(ob, b), ad, bd, idesc_mxf8(128, kN, 1, 1, 0, b), tmem + kColSfv, tmem + kColSfp,
                        (first && ch == 0) ? 0u : 1u);
          }
        }
        mma_commit(bars + kPvDone);
        mma_commit(bars + kKvEmpty + s);
        if (last) mma_commit(bars + kOFull + ob);
      }
      __syncwarp();
      if (last) ++pi;
    }
  } else {
    // =================== loaders ===================
    const int lw = warp - kLoadWarp0;
    const int kc = lane >> 3, c16 = lane & 7;
    Cursor c;
    c.init(a, row0, P0, cb, ce);
    // raw entry of key (16 lw + lane) of the current tile, loaded a tile ahead
    auto raw_of = [&](const Cursor& cu) -> int32_t {
      const int32_t tk = lw + kLoadWarps * lane;  // key of this lane within the tile
      if (!cu.live || lane >= kKeysPerLoader || tk >= kTK) return -1;
      const int32_t p = cu.p0() + tk;
      const int64_t off = cu.beg + p;
      if (p >= cu.p1() || off < 0 || off >= a.n_indices) return -1;
      return __ldg(a.indices + off);
    };
    int32_t raw = raw_of(c);
    bool oob = false;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      Cursor nx = c;
      nx.advance(a);
      const int32_t raw_next = raw_of(nx);
      if (!wait_warp(bars + kKvEmpty + s, ph ^ 1, ms, a)) {
        c = nx;
        raw = raw_next;
        continue;
      }
      int32_t id = raw;
      if (id >= a.n_kv_rows) {
        oob = true;
        id = -1;
      }
      if (id < 0) id = -1;
      uint8_t* st = smem + s * kStageBytes;
      const uint32_t st32 = smem_base + s * kStageBytes;
#pragma unroll 2
      for (int j = 0; j < kKeysPerLoader; ++j) {
        const int t = lw + kLoadWarps * j;
        if (t >= kTK) break;
        const int32_t idj = __shfl_sync(0xffffffffu, id, j);
        if (idj >= 0) {
          const uint8_t* rec = a.kv + int64_t(idj) * kRecordBytes;
          cp_async16(st32 + kc * kChunk + sw128(t, c16), rec + 16 * lane);
          if (lane < 8)
            cp_async16(st32 + kOffRope + sw128(t, lane), rec + kRopeOffset + 16 * lane);
          else if (lane == 8)
            cp_async16(st32 + kOffSc + 16 * t, rec + kScaleOffset);
        } else {
          *reinterpret_cast<uint4*>(st + kc * kChunk + sw128(t, c16)) = make_uint4(0, 0, 0, 0);
          if (lane < 8)
            *reinterpret_cast<uint4*>(st + kOffRope + sw128(t, lane)) = make_uint4(0, 0, 0, 0);
          else if (lane == 8)
            *reinterpret_cast<uint4*>(st + kOffSc + 16 * t) =
                make_uint4(0x3F800000u, 0x3F800000u, 0x3F800000u, 0x3F800000u);
        }
      }
      if (lane < kKeysPerLoader && lw + kLoadWarps * lane < kTK)
        *reinterpret_cast<int32_t*>(st + kOffIds + 4 * (lw + kLoadWarps * lane)) = id;
      fence_proxy_async_smem();
      cp_async_mbar_arrive(bars + kKvFull + s);
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + kKvFull + s);
      c = nx;
      raw = raw_next;
    }
    if (__any_sync(0xffffffffu, oob) && lane == 0 && a.status) atomicOr(a.status, SMLA_STATUS_INDEX_OOB);
    cp_async_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool fp8_kernel_supports(int num_heads) { return num_heads >= 1 && num_heads <= kHP; }

int fp8_tile_len() { return kTK; }

cudaError_t launch_decode_fp8(const DecodeLaunch& L) {
  if (L.plan.grid <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
  if (e != cudaSuccess) return e;
  DecodeArgs args = make_decode_args(L);
  e = launch_trim(L, args);
  if (e != cudaSuccess) return e;
  decode_fp8_kernel<<<L.plan.grid, kThreads, kSmemTotal, L.stream>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess || !L.plan.merge_kernel) return e;
  return launch_merge(L, args);
}

}  // namespace smla
