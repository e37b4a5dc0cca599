// Sparse MLA decode on the 5th-generation tensor cores (tcgen05, TMEM).
//
// One CTA per (row, chunk) unit; 64-key tiles, double-buffered.  Warp roles:
//   warps 0-3 (and 4-7 at 64 heads)  softmax: warpgroup g owns head columns
//               [g*HH, (g+1)*HH), HH = all heads up to 32, 32 at 64 heads;
//               they also stage q, rescale O when a running max moves, and run
//               the epilogue with everyone else
//   every other warp but 12  converters: gather the tile's 656-byte records (64-bit
//               addressing), dequantise E4M3 * pow2 scale -> bf16 exactly, and
//               write the 64 x 576 bf16 key tile in the 128-byte-swizzled
//               K-major layout
//   warp 12     TMEM allocator and MMA issuer (one thread)
//
// Per tile i (stage s = i % 2):
//   QK  S^T[64 keys, HP heads] = K_tile[64 x 576] . Q^T       (M=64, N=HP, K=576)
//   softmax on S^T in log2 units with a lazily moved per-head reference max:
//       p = 2^(x - m_ref) with x = s * sm_scale * log2 e, m_ref raised (and O
//       rescaled in TMEM) only when a score exceeds m_ref + 8; p (<= 256) is
//       written as bf16 P^T
//   PV  O^T[128 d, HP] += V^T[128 d, 64 keys] . P^T[64 keys, HP], four 128-dim
//       M tiles; V^T is the same shared-memory key tile read MN-major.
// The split rows' partials and the last-arriver combine follow the CUDA-core
// kernel (same workspace layout).
//
// The maths is the sparse softmax attention of the gfx950 FlyDSL page (module
// docstring: record layout, CSR tiles, masking; epilogue: out and LSE) with
// the sink folded as the DeepSeek-V4.1 "K2 back" page's stage_combine does.
// That page's design (scaled fp8 MFMA, LDS DMA) is prior art for other
// hardware; this kernel dequantises to bf16 and uses tcgen05 instead.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kThreadsTC = 512;
constexpr int kTileK = 64;                       // keys per tile
constexpr int kDChunks = 9;                      // 576 dims = 9 x 64 (128-byte rows)
constexpr int kChunkBytes = kTileK * 128;        // one 64-dim column block of a tile
constexpr int kTileBytes = kDChunks * kChunkBytes;
constexpr int kStages = 2;
constexpr int kMmaWarp = 12;
constexpr float kRescaleMargin = 8.f;            // p <= 2^8 before a max update
constexpr float kInitMax = -1.0e30f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait

struct Misc {
  uint32_t tmem_base;
  int32_t abort;
  int32_t last_valid;
  int32_t nvalid;
  int32_t is_last;
  int32_t pad[3];
  int32_t flag[2][2][4];         // [warpgroup][stage][quarter] rescale votes
  uint8_t valid[kStages][kTileK];
  float mref[64];                // per-head reference maxima (log2 units)
  float alpha[2][32];
  float red[2][4][32];           // tile maxima, then (after the last tile) key sums
  float fac[64];
};

template <int HP>
struct TcLayout {
  // softmax warpgroups: one holds all head columns up to 32 heads, two at 64;
  // every other warp but the MMA issuer converts records
  static constexpr int SWG = HP == 64 ? 2 : 1;
  static constexpr int kSoftmaxWarps = 4 * SWG;
  static constexpr int kConvWarps = 15 - kSoftmaxWarps;
  static constexpr int kPerConv = (kTileK + kConvWarps - 1) / kConvWarps;  // records per converter warp and tile
  static constexpr int kBatch = kPerConv <= 6 ? kPerConv : (kPerConv + 1) / 2;  // records in flight
  static constexpr int HH = HP / SWG;             // head columns per softmax warpgroup
  static constexpr int q_bytes = kDChunks * HP * 128;
  static constexpr int p_row = 2 * HP;            // bytes of one key's P^T row
  static constexpr int p_bytes = kTileK * p_row;
  // 64 heads: q takes 72 KB, so P^T is single-buffered to stay within 227 KB
  static constexpr int p_stages = HP == 64 ? 1 : 2;
  static constexpr int off_q = kStages * kTileBytes;
  static constexpr int off_p = off_q + q_bytes;
  static constexpr int off_bar = off_p + p_stages * p_bytes;
  static constexpr int off_misc = off_bar + 16 * 8;
  static constexpr int used = off_misc + int(sizeof(Misc));
  // slack to align the dynamic shared memory base to 1024 bytes, when it fits
  static constexpr int slack = used + 1024 <= 232448 ? 1024 : 0;
  static constexpr int total = used + slack;
  static constexpr int tmem_cols = (6 * HP <= 128) ? 128 : (6 * HP <= 256 ? 256 : 512);
  static constexpr Swizzle p_swz = HP == 64 ? kSw128 : (HP == 32 ? kSw64 : kSw32);
  static constexpr uint32_t p_swmask = HP == 64 ? 7 : (HP == 32 ? 3 : 1);
  static constexpr uint32_t idesc_qk = idesc_bf16(64, HP, 0, 0);
  static constexpr uint32_t idesc_pv = idesc_bf16(128, HP, 1, 1);
};

// Offset of byte `b` (16-byte aligned) of row `r` inside a 128-byte-row
// swizzled block whose rows are 128 bytes apart (1024-byte atoms).
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t b) {
  return r * 128u + ((((b >> 4) ^ (r & 7u)) << 4) | (b & 15u));
}

// TMEM row of S^T for key r of the tile, for an M=64 MMA: rows 16 w .. 16 w + 15
// sit in lanes 32 w .. 32 w + 15 of warp quarter w.
__device__ __forceinline__ bool s_lane_active(int lane) { return lane < 16; }

__device__ __forceinline__ void set_abort(Misc* ms, const DecodeArgs& a) {
  if (atomicExch(&ms->abort, 1) == 0 && a.status) atomicOr(a.status, SMLA_STATUS_TIMEOUT);
}

// A pipeline wait.  Once any wait of the CTA has timed out, every later wait
// returns false at once, so that all roles run to the final barrier quickly;
// loops that contain named barriers keep iterating (never break) so that every
// thread executes the same barrier sequence.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Misc* ms, const DecodeArgs& a) {
  if (*reinterpret_cast<volatile int32_t*>(&ms->abort)) return false;
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  set_abort(ms, a);
  return false;
}

// The same, for a whole warp: the result is the same in every lane.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, Misc* ms, const DecodeArgs& a) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, ms, a));
}

// 16 E4M3 bytes times a power-of-two scale -> 16 bf16 (exact), as 2 x uint4.
__device__ __forceinline__ void dequant16_bf16(uint4 v, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(w[i] >> (16 * j)), __NV_E4M3);
      float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
      o[2 * i + j] = pack_bf16x2(f.x * scale, f.y * scale);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <int HP>
__global__ void __launch_bounds__(kThreadsTC, 1) decode_tc_kernel(DecodeArgs a) {
  using Lay = TcLayout<HP>;
  constexpr int HH = Lay::HH;
  constexpr int kSoftmaxWarps = Lay::kSoftmaxWarps;
  constexpr int kConvWarps = Lay::kConvWarps;
  constexpr int kPerConv = Lay::kPerConv;
  constexpr int kBatch = Lay::kBatch;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint8_t* q_s = smem + Lay::off_q;
  uint8_t* p_s = smem + Lay::off_p;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::off_bar);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 2;
  uint64_t* s_full = bars + 4;
  uint64_t* s_empty = bars + 6;
  uint64_t* p_full = bars + 8;
  uint64_t* pv_done = bars + 10;
  uint64_t* q_full = bars + 12;
  uint64_t* mma_drain = bars + 13;
  Misc* ms = reinterpret_cast<Misc*>(smem + Lay::off_misc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (Lay::slack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
    // no room to realign: refuse (uniformly, before any barrier or TMEM use)
    if (tid == 0 && a.status) atomicOr(a.status, SMLA_STATUS_TIMEOUT);
    return;
  }
  const Unit u = unit_of(a, blockIdx.x);
  const int H = a.heads;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full + s, kConvWarps);
      mbar_init(kv_empty + s, 1);
      mbar_init(s_full + s, 1);
      mbar_init(s_empty + s, kSoftmaxWarps);
      mbar_init(p_full + s, kSoftmaxWarps);
      mbar_init(pv_done + s, 1);
    }
    mbar_init(q_full, kSoftmaxWarps);
    mbar_init(mma_drain, 1);
    ms->abort = 0;
    for (int h = 0; h < 64; ++h) ms->mref[h] = kInitMax;
    ms->last_valid = u.p0 - 1;
    ms->nvalid = 0;
    ms->is_last = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ms->tmem_base, Lay::tmem_cols);
    tmem_relinquish();
  }
  // Rows padded with -1 (has_invalid): stop after the last entry >= 0.
  int p1 = u.p1;
  if (a.has_invalid && u.p1 > u.p0) {
    __syncthreads();
    int last = u.p0 - 1;
    for (int p = u.p0 + tid; p < u.p1; p += kThreadsTC) {
      const int64_t off = u.beg + p;
      if (off >= 0 && off < a.n_indices && __ldg(a.indices + off) >= 0) last = p;
    }
    if (last >= u.p0) atomicMax(&ms->last_valid, last);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (a.has_invalid) p1 = ms->last_valid + 1 > u.p0 ? ms->last_valid + 1 : u.p0;
  const int nt = (p1 - u.p0 + kTileK - 1) / kTileK;
  const uint32_t tmem = ms->tmem_base;
  const uint32_t tiles_u32 = smem_u32(tiles);
  const uint32_t q_u32 = smem_u32(q_s);
  const uint32_t p_u32 = smem_u32(p_s);

  float lpart[HH];
#pragma unroll
  for (int h = 0; h < HH; ++h) lpart[h] = 0.f;

  if (warp < kSoftmaxWarps) {
    // ---------------- softmax warpgroups ----------------
    const int wg = warp >> 2, qd = warp & 3;
    for (int i = tid; i < HP * (kQK / 8); i += 32 * kSoftmaxWarps) {
      const int h = i / (kQK / 8), c16 = i % (kQK / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (h < H)
        v = __ldg(reinterpret_cast<const uint4*>(a.q + u.row * a.q_stride_row + h * a.q_stride_head + c16 * 8));
      const uint32_t off = uint32_t(c16 >> 3) * (HP * 128) + uint32_t(h >> 3) * 1024u + sw128_off(h & 7, (c16 & 7) * 16);
      *reinterpret_cast<uint4*>(q_s + off) = v;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);

    const bool active = s_lane_active(lane);
    const int r = 16 * qd + lane;  // key of this thread within the tile (active lanes)
    const float* mr = ms->mref + wg * HH;  // this warpgroup's reference maxima (uniform)
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      wait_bar_warp(kv_full + s, ph, ms, a);
      wait_bar_warp(s_full + s, ph, ms, a);
      tc_fence_after();
      float x[HH];
      {
        const uint32_t taddr = tmem + (uint32_t(32 * qd) << 16) + uint32_t(s * HP + wg * HH);
#pragma unroll
        for (int c = 0; c < HH / 8; ++c) {
          uint32_t v[8];
          tmem_ld8(taddr + 8 * c, v);
#pragma unroll
          for (int k = 0; k < 8; ++k) x[8 * c + k] = __uint_as_float(v[k]);
        }
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + s);
      const bool valid = active && (r < kTileK) && ms->valid[s][active ? r : 0];
      bool need = false;
#pragma unroll
      for (int h = 0; h < HH; ++h) {
        x[h] = valid ? x[h] * a.sm_scale_log2 : -INFINITY;
        need |= x[h] > mr[h] + kRescaleMargin;
      }
      need = __any_sync(0xffffffffu, need);
      if (lane == 0) ms->flag[wg][s][qd] = need;
      named_barrier(1 + wg, 128);
      need = ms->flag[wg][s][0] | ms->flag[wg][s][1] | ms->flag[wg][s][2] | ms->flag[wg][s][3];
      if (need) {
        // exact tile max of this warpgroup's heads, then move the references
#pragma unroll
        for (int h = 0; h < HH; ++h) {
          float t = x[h];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
          if (lane == 0) ms->red[wg][qd][h] = t;
        }
        named_barrier(1 + wg, 128);
#pragma unroll
        for (int h = 0; h < HH; ++h) {
          const float tm = fmaxf(fmaxf(ms->red[wg][0][h], ms->red[wg][1][h]),
                                 fmaxf(ms->red[wg][2][h], ms->red[wg][3][h]));
          const float al = ex2(mr[h] - fmaxf(mr[h], tm));
          lpart[h] *= al;
          if (tid == wg * 128) ms->alpha[wg][h] = al;
        }
        named_barrier(1 + wg, 128);  // everyone has read the old references
        if (tid == wg * 128) {
          for (int h = 0; h < HH; ++h) {
            const float tm = fmaxf(fmaxf(ms->red[wg][0][h], ms->red[wg][1][h]),
                                   fmaxf(ms->red[wg][2][h], ms->red[wg][3][h]));
            ms->mref[wg * HH + h] = fmaxf(mr[h], tm);
          }
        }
        named_barrier(1 + wg, 128);  // the new references are visible
        if (j > 0) {
          // O^T columns of this warpgroup's heads, all four 128-dim tiles:
          // wait for PV(j-1), then scale in place.
          wait_bar_warp(pv_done + ((j - 1) & 1), ((j - 1) >> 1) & 1, ms, a);
          tc_fence_after();
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
            const uint32_t taddr = tmem + (uint32_t(32 * qd) << 16) + uint32_t(2 * HP + mt * HP + wg * HH);
#pragma unroll
            for (int c = 0; c < HH / 8; ++c) {
              uint32_t v[8];
              tmem_ld8(taddr + 8 * c, v);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 8; ++k)
                v[k] = __float_as_uint(__uint_as_float(v[k]) * ms->alpha[wg][8 * c + k]);
              tmem_st8(taddr + 8 * c, v);
            }
          }
          tmem_wait_st();
        }
      }
      // p = 2^(x - m_ref) as bf16 into P^T (key rows, head columns contiguous)
      uint32_t pk[HH / 2];
#pragma unroll
      for (int h = 0; h < HH; h += 2) {
        const float p0 = ex2(x[h] - mr[h]);
        const float p1v = ex2(x[h + 1] - mr[h + 1]);
        lpart[h] += p0;
        lpart[h + 1] += p1v;
        pk[h / 2] = pack_bf16x2(p0, p1v);
      }
      // the P stage is free once the PV that last read it has completed
      if (Lay::p_stages == 2)
        wait_bar_warp(pv_done + s, ph ^ 1, ms, a);  // PV(j-2)
      else if (j > 0)
        wait_bar_warp(pv_done + ((j - 1) & 1), ((j - 1) >> 1) & 1, ms, a);  // PV(j-1)
      const int ps = Lay::p_stages == 2 ? s : 0;
      if (active) {
        uint8_t* prow = p_s + ps * Lay::p_bytes;
#pragma unroll
        for (int c = 0; c < HH / 8; ++c) {
          uint32_t off = uint32_t(r) * Lay::p_row + uint32_t(wg * (HH / 8) + c) * 16u;
          off ^= ((off >> 7) & Lay::p_swmask) << 4;
          *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + s);
    }
    // per-head sums of this warpgroup over its 64 keys, and the final maxima
#pragma unroll
    for (int h = 0; h < HH; ++h) {
      float t = active ? lpart[h] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if (lane == 0) ms->red[wg][qd][h] = t;
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = wait_bar(q_full, 0, ms, a);
      auto issue_pv = [&](int j) -> bool {
        const int s = j & 1;
        if (!wait_bar(p_full + s, (j >> 1) & 1, ms, a)) return false;
        tc_fence_after();
        const uint32_t tile = tiles_u32 + s * kTileBytes;
        const uint32_t pst = p_u32 + (Lay::p_stages == 2 ? s : 0) * Lay::p_bytes;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const uint32_t d = tmem + uint32_t(2 * HP + mt * HP);
#pragma unroll
          for (int k = 0; k < kTileK / 16; ++k) {
            const uint64_t ad = smem_desc(tile + (2 * mt) * kChunkBytes + k * 2048, kChunkBytes, 1024, kSw128);
            const uint64_t bd = smem_desc(pst + k * 16 * Lay::p_row, 8 * Lay::p_row, 8 * Lay::p_row, Lay::p_swz);
            mma_f16_ss(d, ad, bd, Lay::idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          }
        }
        mma_commit(kv_empty + s);
        mma_commit(pv_done + s);
        return true;
      };
      for (int i = 0; ok && i < nt; ++i) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!wait_bar(kv_full + s, ph, ms, a) || !wait_bar(s_empty + s, ph ^ 1, ms, a)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tile = tiles_u32 + s * kTileBytes;
        const uint32_t d = tmem + uint32_t(s * HP);
#pragma unroll
        for (int k = 0; k < kQK / 16; ++k) {
          const int c = k >> 2, kk = k & 3;
          const uint64_t ad = smem_desc(tile + c * kChunkBytes + kk * 32, 16, 1024, kSw128);
          const uint64_t bd = smem_desc(q_u32 + c * (HP * 128) + kk * 32, 16, 1024, kSw128);
          mma_f16_ss(d, ad, bd, Lay::idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(s_full + s);
        if (i > 0 && !issue_pv(i - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && nt > 0) issue_pv(nt - 1);
      // every issued MMA has completed before anyone reads O or frees TMEM
      mma_commit(mma_drain);
      if (!mbar_wait(mma_drain, 0, kWaitLimitNs)) set_abort(ms, a);
    }
    __syncwarp();
  } else {
    // ---------------- converters ----------------
    // Warp cw takes records cw, cw + 7, ... of each tile (kPerConv at most).
    // Lane k holds the record row of the warp's k-th record; the records of
    // tile i + 2 are prefetched into L2 while tile i is converted.
    const int cw = warp < kMmaWarp ? warp - kSoftmaxWarps : warp - kSoftmaxWarps - 1;  // 0..6
    int nvalid = 0;
    const int ck = lane >> 2;                 // 64-dim column block of this lane's 16 dims
    const int b0 = (lane & 3) * 32;           // byte offset of those dims within the 128-byte row
    const bool hi_first = (lane >> 2) & 1;    // alternate store order: conflict-free phases
    auto tile_keys = [&](int i) -> int32_t {  // this lane's record row in tile i, or -1
      const int r = cw + kConvWarps * lane;
      const int p = u.p0 + i * kTileK + r;
      return (i < nt && lane < kPerConv && r < kTileK && p < p1) ? key_of(a, u.beg, p) : -1;
    };
    auto prefetch = [&](int32_t id) {
      if (id >= 0) prefetch_l2(a.kv + int64_t(id) * kRecordBytes, kRecordBytes);
    };
    int32_t key_cur = tile_keys(0);
    int32_t key_nxt = tile_keys(1);
    prefetch(key_cur);
    prefetch(key_nxt);
    for (int i = 0; i < nt; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      uint8_t* tile = tiles + s * kTileBytes;
      const int32_t key_nn = tile_keys(i + 2);
      prefetch(key_nn);
      bool waited = false;
      bool ok = true;
      for (int k0 = 0; k0 < kPerConv; k0 += kBatch) {
        int32_t idx[kBatch];
        uint4 lat[kBatch], rp[kBatch];
        float sc[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int32_t id = __shfl_sync(0xffffffffu, key_cur, (k0 + b) & 31);
          idx[b] = (k0 + b < kPerConv) ? id : -1;
          lat[b] = make_uint4(0, 0, 0, 0);
          rp[b] = make_uint4(0, 0, 0, 0);
          sc[b] = 0.f;
          if (idx[b] >= 0) {
            const uint8_t* rec = a.kv + int64_t(idx[b]) * kRecordBytes;
            lat[b] = __ldg(reinterpret_cast<const uint4*>(rec) + lane);
            sc[b] = __ldg(reinterpret_cast<const float*>(rec + kScaleOffset) + (lane >> 3));
            if (lane < 8) rp[b] = __ldg(reinterpret_cast<const uint4*>(rec + kRopeOffset) + lane);
          }
        }
        if (!waited) {
          waited = true;
          if (!wait_bar_warp(kv_empty + s, ph ^ 1, ms, a)) {
            ok = false;
            break;
          }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int r = cw + kConvWarps * (k0 + b);
          if (k0 + b >= kPerConv || r >= kTileK) break;
          uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
          if (idx[b] >= 0) dequant16_bf16(lat[b], sc[b], lo, hi);
          uint8_t* rowbase = tile + ck * kChunkBytes + (r >> 3) * 1024;
          const uint4 first = hi_first ? hi : lo, second = hi_first ? lo : hi;
          *reinterpret_cast<uint4*>(rowbase + sw128_off(r & 7, b0 + (hi_first ? 16 : 0))) = first;
          *reinterpret_cast<uint4*>(rowbase + sw128_off(r & 7, b0 + (hi_first ? 0 : 16))) = second;
          if (lane < 8)
            *reinterpret_cast<uint4*>(tile + 8 * kChunkBytes + (r >> 3) * 1024 + sw128_off(r & 7, lane * 16)) = rp[b];
          if (lane == 0) {
            ms->valid[s][r] = idx[b] >= 0;
            nvalid += idx[b] >= 0;
          }
        }
      }
      if (!ok) break;
      if (!waited && !wait_bar_warp(kv_empty + s, ph ^ 1, ms, a)) break;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(kv_full + s);
      key_cur = key_nxt;
      key_nxt = key_nn;
    }
    if (lane == 0 && nvalid) atomicAdd(&ms->nvalid, nvalid);
  }

  // ---------------- epilogue (all warps) ----------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool aborted = ms->abort != 0;
  static_assert(TcLayout<HP>::total <= 232448, "shared memory over the per-block limit");
  if (tid < H) {
    const int g = tid / HH, hh = tid % HH;
    const float l = ms->red[g][0][hh] + ms->red[g][1][hh] + ms->red[g][2][hh] + ms->red[g][3][hh];
    const float m = ms->mref[tid];
    if (a.splits == 1) {
      float fac, lse;
      finish_head(m, nt > 0 ? l : 0.f, a.sink, tid, &fac, &lse);
      ms->fac[tid] = fac;
      if (a.lse && !aborted) a.lse[int64_t(u.row) * H + tid] = lse;
    } else {
      const int64_t rc = int64_t(u.row) * a.splits + u.chunk;
      const bool live = nt > 0 && l > 0.f;
      if (!aborted) {
        a.ml_part[(rc * H + tid) * 2] = live ? m : -INFINITY;
        a.ml_part[(rc * H + tid) * 2 + 1] = live ? l : 0.f;
      }
    }
  }
  __syncthreads();
  {
    // O^T readout: warp w takes 128-dim tile w / 4, lanes of quarter w % 4.
    const int mt = warp >> 2, qd = warp & 3;
    const int dg = mt * 128 + qd * 32 + lane;
    const int64_t rc = int64_t(u.row) * a.splits + u.chunk;
#pragma unroll 1
    for (int c = 0; c < HP / 8; ++c) {
      uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (nt > 0) {
        tmem_ld8(tmem + (uint32_t(32 * qd) << 16) + uint32_t(2 * HP + mt * HP + 8 * c), v);
        tmem_wait_ld();
      }
      if (aborted) continue;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int h = 8 * c + k;
        if (h >= H) break;
        const float o = nt > 0 ? __uint_as_float(v[k]) : 0.f;
        if (a.splits == 1) {
          const __nv_bfloat16 bv = __float2bfloat16_rn(o * ms->fac[h]);
          *reinterpret_cast<__nv_bfloat16*>(a.out + u.row * a.out_stride_row + h * a.out_stride_head + dg) = bv;
        } else {
          a.o_part[(rc * H + h) * kLatent + dg] = o;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::tmem_cols);
  }
  if (aborted) return;
  if (a.splits == 1) {
    if (tid == 0 && a.n_valid) a.n_valid[u.row] = ms->nvalid;
    return;
  }
  // ---- split row: the last chunk to finish merges the partials.
  const int C = a.splits;
  if (tid == 0) a.nv_part[int64_t(u.row) * C + u.chunk] = ms->nvalid;
  __threadfence();
  __syncthreads();
  if (tid == 0) ms->is_last = (atomicAdd(a.ticket + u.row, 1) == C - 1);
  __syncthreads();
  if (!ms->is_last) return;
  __threadfence();
  float* w_s = reinterpret_cast<float*>(tiles);  // [H][C] merge weights (tiles are free now)
  if (tid < H) {
    const int h = tid;
    float mstar = -INFINITY;
    for (int c = 0; c < C; ++c) {
      const int64_t o = ((int64_t(u.row) * C + c) * H + h) * 2;
      if (__ldcg(a.ml_part + o + 1) > 0.f) mstar = fmaxf(mstar, __ldcg(a.ml_part + o));
    }
    float L = 0.f;
    for (int c = 0; c < C; ++c) {
      const int64_t o = ((int64_t(u.row) * C + c) * H + h) * 2;
      const float lc = __ldcg(a.ml_part + o + 1);
      const float w = lc > 0.f ? exp2f(__ldcg(a.ml_part + o) - mstar) : 0.f;
      w_s[h * C + c] = w;
      L += lc * w;
    }
    float fac, lse;
    finish_head(mstar, L, a.sink, h, &fac, &lse);
    ms->fac[h] = fac;
    if (a.lse) a.lse[int64_t(u.row) * H + h] = lse;
  }
  if (tid == 0) {
    int tot = 0;
    for (int c = 0; c < C; ++c) tot += __ldcg(a.nv_part + int64_t(u.row) * C + c);
    if (a.n_valid) a.n_valid[u.row] = tot;
    a.ticket[u.row] = 0;  // leave the counter zero for the next call
  }
  __syncthreads();
  const int d = tid;  // 512 threads, one latent dim each
  for (int h = 0; h < H; ++h) {
    float o = 0.f;
    for (int c = 0; c < C; ++c) {
      const float w = w_s[h * C + c];
      if (w != 0.f) o = fmaf(w, __ldcg(a.o_part + ((int64_t(u.row) * C + c) * H + h) * kLatent + d), o);
    }
    a.out[u.row * a.out_stride_row + h * a.out_stride_head + d] =
        __bfloat16_as_ushort(__float2bfloat16_rn(o * ms->fac[h]));
  }
}

template <int HP>
cudaError_t launch_tc_hp(const DecodeLaunch& L) {
  const int smem = TcLayout<HP>::total;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<HP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<HP><<<L.plan.grid, kThreadsTC, smem, L.stream>>>(make_decode_args(L));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeLaunch& L) {
  if (L.plan.grid <= 0) return cudaSuccess;
  const int H = L.p.num_heads;
  if (H <= 16) return launch_tc_hp<16>(L);
  if (H <= 32) return launch_tc_hp<32>(L);
  return launch_tc_hp<64>(L);
}

}  // namespace smla
