// Sparse MLA decode on CUDA cores (fp32 FMA): one CTA per (row, chunk) unit,
// 32-key tiles.  It is the plain GPU formulation of the method, kept as the
// cross-check of the tensor-core kernel and for head counts it does not take.
//
// Per tile: the 32 slice positions are resolved to record rows (masking as in
// the gfx950 page's "Tiles" paragraph), each record's 512 E4M3 latent values
// are dequantised with their per-128 power-of-two scale and stored with the
// 64 bf16 rope dims as fp32 rows; QK over 576 dims, the online softmax in
// log2 units and PV over the 512 latent dims follow.  A split row's chunks
// write (O, m, l) partials; the last chunk to finish merges them (K2 back,
// stage_combine) -- it takes a ticket with one atomicAdd and never waits.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kThreads = 256;
constexpr int kT = 32;         // keys per tile
constexpr int kKP = kQK + 1;   // padded fp32 row of a key (odd: conflict-free column reads)

template <int HP>
struct SimtSmem {
  static constexpr size_t q_bytes = size_t(HP) * kQK * 2;
  static constexpr size_t k_bytes = size_t(kT) * kKP * 4;
  static constexpr size_t p_bytes = size_t(HP) * kT * 4;
  static constexpr size_t head_bytes = size_t(HP) * 4 * 4 + size_t(HP) * SMLA_MAX_SPLITS * 4;
  static constexpr size_t total = q_bytes + k_bytes + p_bytes + head_bytes + kT * 4 + 16;
};

__device__ __forceinline__ void dequant16(uint4 v, float scale, float* dst) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(w[i] >> (16 * j)), __NV_E4M3);
      float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
      dst[4 * i + 2 * j] = f.x * scale;
      dst[4 * i + 2 * j + 1] = f.y * scale;
    }
  }
}

template <int HP>
__global__ void __launch_bounds__(kThreads, 1) decode_simt_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  using S = SimtSmem<HP>;
  uint16_t* q_s = reinterpret_cast<uint16_t*>(smem);
  float* k_s = reinterpret_cast<float*>(smem + S::q_bytes);
  float* p_s = reinterpret_cast<float*>(smem + S::q_bytes + S::k_bytes);
  float* m_s = reinterpret_cast<float*>(smem + S::q_bytes + S::k_bytes + S::p_bytes);
  float* l_s = m_s + HP;
  float* alpha_s = l_s + HP;
  float* fac_s = alpha_s + HP;
  float* w_s = fac_s + HP;  // [HP][splits] combine weights
  int32_t* idx_s = reinterpret_cast<int32_t*>(w_s + HP * SMLA_MAX_SPLITS);
  int32_t* flag_s = idx_s + kT;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Unit u = unit_of(a, blockIdx.x);
  const int H = a.heads;

  // q row -> shared (bf16), padded heads zero.
  for (int i = tid; i < HP * (kQK / 8); i += kThreads) {
    const int h = i / (kQK / 8), part = i % (kQK / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h < H)
      v = *reinterpret_cast<const uint4*>(a.q + u.row * a.q_stride_row + h * a.q_stride_head + part * 8);
    *reinterpret_cast<uint4*>(q_s + h * kQK + part * 8) = v;
  }
  if (tid < HP) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  float acc[HP][2];
#pragma unroll
  for (int h = 0; h < HP; ++h) acc[h][0] = acc[h][1] = 0.f;
  int nvalid = 0;  // counted by thread 0
  __syncthreads();

  for (int t0 = u.p0; t0 < u.p1; t0 += kT) {
    if (tid < kT) {
      const int p = t0 + tid;
      idx_s[tid] = p < u.p1 ? key_of(a, u.beg, p) : -1;
    }
    __syncthreads();
    if (tid == 0)
      for (int t = 0; t < kT; ++t) nvalid += idx_s[t] >= 0;
    // gather + dequantise: warp w takes keys w, w + 8, ...
    for (int t = warp; t < kT; t += kThreads / 32) {
      const int32_t idx = idx_s[t];
      float* row = k_s + t * kKP;
      float vals[16];
      if (idx >= 0) {
        const uint8_t* rec = a.kv + int64_t(idx) * kRecordBytes;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(rec + lane * 16));
        const float sc = __ldg(reinterpret_cast<const float*>(rec + kScaleOffset) + (lane >> 3));
        dequant16(v, sc, vals);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) vals[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) row[lane * 16 + i] = vals[i];
      if (lane < 8) {
        uint4 r = make_uint4(0, 0, 0, 0);
        if (idx >= 0)
          r = __ldg(reinterpret_cast<const uint4*>(a.kv + int64_t(idx) * kRecordBytes + kRopeOffset) + lane);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          row[kLatent + lane * 8 + 2 * i] = __uint_as_float(w[i] << 16);
          row[kLatent + lane * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
      }
    }
    __syncthreads();
    // QK: score of (h, t) in log2 units; masked keys -inf.
    for (int pr = tid; pr < HP * kT; pr += kThreads) {
      const int h = pr / kT, t = pr % kT;
      const uint16_t* qh = q_s + h * kQK;
      const float* kt = k_s + t * kKP;
      float s = 0.f;
#pragma unroll 8
      for (int d = 0; d < kQK; d += 2) {
        const uint32_t qq = *reinterpret_cast<const uint32_t*>(qh + d);
        s = fmaf(__uint_as_float(qq << 16), kt[d], s);
        s = fmaf(__uint_as_float(qq & 0xFFFF0000u), kt[d + 1], s);
      }
      p_s[h * kT + t] = idx_s[t] >= 0 ? s * a.sm_scale_log2 : -INFINITY;
    }
    __syncthreads();
    // online softmax: one thread per head.
    if (tid < HP) {
      const int h = tid;
      float mx = -INFINITY;
      for (int t = 0; t < kT; ++t) mx = fmaxf(mx, p_s[h * kT + t]);
      const float m_old = m_s[h];
      const float m_new = fmaxf(m_old, mx);
      const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_old - m_new);
      float sum = 0.f;
      for (int t = 0; t < kT; ++t) {
        const float s = p_s[h * kT + t];
        const float pv = (s == -INFINITY) ? 0.f : exp2f(s - m_new);
        p_s[h * kT + t] = pv;
        sum += pv;
      }
      l_s[h] = l_s[h] * alpha + sum;
      m_s[h] = m_new;
      alpha_s[h] = alpha;
    }
    __syncthreads();
    // PV: thread owns latent dims 2 tid, 2 tid + 1.
    {
      const int d = 2 * tid;
#pragma unroll
      for (int h = 0; h < HP; ++h) {
        const float al = alpha_s[h];
        float o0 = acc[h][0] * al, o1 = acc[h][1] * al;
        for (int t = 0; t < kT; ++t) {
          // rows are kKP (odd) floats apart: scalar reads, no 8-byte vector
          const float pv = p_s[h * kT + t];
          o0 = fmaf(pv, k_s[t * kKP + d], o0);
          o1 = fmaf(pv, k_s[t * kKP + d + 1], o1);
        }
        acc[h][0] = o0;
        acc[h][1] = o1;
      }
    }
    __syncthreads();
  }

  const int d = 2 * tid;
  if (a.splits == 1) {
    if (tid < H) {
      float fac, lse;
      finish_head(m_s[tid], l_s[tid], a.sink, tid, &fac, &lse);
      fac_s[tid] = fac;
      if (a.lse) a.lse[int64_t(u.row) * H + tid] = lse;
    }
    if (tid == 0 && a.n_valid) a.n_valid[u.row] = nvalid;
    __syncthreads();
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      if (h < H) {
        const float f = fac_s[h];
        *reinterpret_cast<uint32_t*>(a.out + u.row * a.out_stride_row + h * a.out_stride_head + d) =
            pack_bf16x2(acc[h][0] * f, acc[h][1] * f);
      }
    }
    return;
  }

  // ---- split row: publish this chunk's partial, then maybe combine.
  const int C = a.splits;
  const int64_t rc = int64_t(u.row) * C + u.chunk;
#pragma unroll
  for (int h = 0; h < HP; ++h) {
    if (h < H)
      *reinterpret_cast<float2*>(a.o_part + (rc * H + h) * kLatent + d) = make_float2(acc[h][0], acc[h][1]);
  }
  if (tid < H) {
    a.ml_part[(rc * H + tid) * 2] = m_s[tid];
    a.ml_part[(rc * H + tid) * 2 + 1] = l_s[tid];
  }
  if (tid == 0) a.nv_part[rc] = nvalid;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(a.ticket + u.row, 1);
    flag_s[0] = (prev == C - 1);
  }
  __syncthreads();
  if (!flag_s[0]) return;
  __threadfence();
  // Last arriver: merge the C chunks of this row.
  if (tid < H) {
    const int h = tid;
    float mstar = -INFINITY;
    for (int c = 0; c < C; ++c) {
      const int64_t o = ((int64_t(u.row) * C + c) * H + h) * 2;
      const float lc = __ldcg(a.ml_part + o + 1);
      if (lc > 0.f) mstar = fmaxf(mstar, __ldcg(a.ml_part + o));
    }
    float L = 0.f;
    for (int c = 0; c < C; ++c) {
      const int64_t o = ((int64_t(u.row) * C + c) * H + h) * 2;
      const float lc = __ldcg(a.ml_part + o + 1);
      const float w = lc > 0.f ? exp2f(__ldcg(a.ml_part + o) - mstar) : 0.f;
      w_s[h * SMLA_MAX_SPLITS + c] = w;
      L += lc * w;
    }
    float fac, lse;
    finish_head(mstar, L, a.sink, h, &fac, &lse);
    fac_s[h] = fac;
    if (a.lse) a.lse[int64_t(u.row) * H + h] = lse;
  }
  if (tid == 0) {
    int tot = 0;
    for (int c = 0; c < C; ++c) tot += __ldcg(a.nv_part + int64_t(u.row) * C + c);
    if (a.n_valid) a.n_valid[u.row] = tot;
    a.ticket[u.row] = 0;  // leave the counter zero for the next call
  }
  __syncthreads();
  for (int h = 0; h < H; ++h) {
    float o0 = 0.f, o1 = 0.f;
    for (int c = 0; c < C; ++c) {
      const float w = w_s[h * SMLA_MAX_SPLITS + c];
      if (w != 0.f) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(
            a.o_part + ((int64_t(u.row) * C + c) * H + h) * kLatent + d));
        o0 = fmaf(w, v.x, o0);
        o1 = fmaf(w, v.y, o1);
      }
    }
    const float f = fac_s[h];
    *reinterpret_cast<uint32_t*>(a.out + u.row * a.out_stride_row + h * a.out_stride_head + d) =
        pack_bf16x2(o0 * f, o1 * f);
  }
}

template <int HP>
cudaError_t launch_hp(const DecodeLaunch& L) {
  const size_t smem = SimtSmem<HP>::total;
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<HP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  decode_simt_kernel<HP><<<L.plan.grid, kThreads, smem, L.stream>>>(make_decode_args(L));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeLaunch& L) {
  if (L.plan.grid <= 0) return cudaSuccess;
  const int H = L.p.num_heads;
  if (H <= 16) return launch_hp<16>(L);
  if (H <= 32) return launch_hp<32>(L);
  return launch_hp<64>(L);
}

}  // namespace smla
