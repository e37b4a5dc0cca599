// Sparse MLA decode on the 5th-generation tensor cores (tcgen05, TMEM),
// persistent and balanced.
//
// Schedule (documented with smla_plan in smla.h): every row is cut into 64-key
// tiles and takes two slots for the cost of starting it followed by its tiles;
// the rows' slots form one space of W slots, and CTA c of the grid takes the
// slots [floor(c W / G), floor((c+1) W / G)), streaming through the tiles in
// its range across row boundaries.  A row wholly inside one CTA's range is
// finished there; a shared row gets one (O, m, l) partial per CTA and is
// merged by the merge kernel below.  With has_invalid, trim_rows_kernel first
// cuts each row at its last entry >= 0.
//
// Warp roles (16 warps):
//   warps 0-3 (and 4-7 at 64 heads)  softmax: warpgroup g owns head columns
//               [g*HH, (g+1)*HH) (HH = all heads up to 32, 32 at 64 heads); they
//               also stage q, move the reference maxima (rescaling O in TMEM),
//               and run each row part's epilogue (partials of shared rows)
//   warps 12-14 MMA issuers, one thread each on three different SM
//               sub-partitions (a single thread issues a tcgen05.mma only every
//               ~50 cycles; QK on one thread instead of two makes a decode step
//               ~10% slower): 12 and 13 issue the two halves of QK's K = 576
//               into two S accumulators, 14 issues PV; warp 12 owns TMEM
//   warps 4-11 (8-11 at 64 heads)  latent converters: gather the 512 E4M3
//               bytes and the four scales of each tile's records (64-bit
//               addressing), dequantise E4M3 * pow2 scale -> bf16 exactly
//               (a tile or batch holding any other scale is converted again
//               by a general pass: e4m3 * scale in f32, rounded to bf16), and
//               write the 64 x 512 bf16 latent of the key tile in the
//               128-byte-swizzled K-major layout.  Up to 32 heads the latent
//               bytes travel by cp.async into a per-warp shared-memory ring
//               about a tile ahead of the conversion; at 64 heads (no
//               shared memory left) into registers one batch ahead
//   warp 15     rope copier: the records' 128-byte bf16 rope goes straight into
//               the key tile by cp.async (completion tracked by the tile's
//               mbarrier), zeros for masked keys; it also writes the keys'
//               validity flags and flags out-of-range indices
//
// Per tile i (stage s = i % 2), within the row part it belongs to:
//   QK  S^T[64 keys, HP heads] = K_tile[64 x 576] . Q^T       (M=64, N=HP, K=576)
//   softmax on S^T in log2 units with a lazily moved per-head reference max:
//       p = 2^(x - m_ref), x = s * sm_scale * log2 e; m_ref is raised (and O
//       rescaled in TMEM) only when a score exceeds m_ref + 24, so p <= 2^24
//       (exact in bf16's range; f32 sums stay far from overflow);
//       p is written as bf16 P^T
//   PV  O^T[128 d, HP] += V^T[128 d, 64 keys] . P^T[64 keys, HP], four 128-dim
//       M tiles; V^T is the same shared-memory key tile read MN-major.
// O has two TMEM buffers (alternating between row parts) where they fit.
// Shared rows are merged by merge_rows_kernel, launched right after.
// The latent dims are stored permuted within each 4-dim group (see
// latent_dim_of); q is staged in the same order and the epilogue undoes it.
//
// The maths is the sparse softmax attention of the gfx950 FlyDSL page (module
// docstring: record layout, CSR tiles, masking; epilogue: out and LSE) with
// the sink folded as the DeepSeek-V4.1 "K2 back" page's stage_combine does,
// and its split/combine for rows shared between CTAs.  The pages' kernels
// (scaled fp8 MFMA on gfx950, FP8 tcgen05 with a TMA gather4 front end on
// SM100) are prior art; this kernel dequantises to bf16 (exact) instead.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_ptx.cuh"

#ifdef SMLA_TRACE
// Optional stage trace (compile with -DSMLA_TRACE): lane 0 of each warp writes
// (%globaltimer ns | tag << 48 | tile << 56) into
// g_smla_trace[(cta * 16 + warp) * kTraceEvents + k].  Off in normal builds.
__device__ unsigned long long* g_smla_trace;
extern "C" int smla_trace_set(void* buf) {
  unsigned long long* p = static_cast<unsigned long long*>(buf);
  return int(cudaMemcpyToSymbol(g_smla_trace, &p, sizeof(p)));
}
#endif

namespace smla {

// Limit of every pipeline wait in ns (0: kWaitLimitNs), and whether the first
// softmax wait of each CTA waits on a barrier nothing signals (so that it runs
// out: a test of the timeout path); read at kernel start.
__device__ uint64_t g_tc_wait_ns;
__device__ int32_t g_tc_stall;

namespace {

using namespace ptx;

#ifdef SMLA_TRACE
constexpr int kTraceEvents = 256;
// tr_buf (the buffer, read once per thread) and tr_k (this warp's event
// count, kept equal in all lanes) are locals of the kernel.
#define SMLA_TR(tag, tile)                                                                              \
  do {                                                                                                  \
    if (tr_buf != nullptr && (threadIdx.x & 31) == 0 && tr_k < kTraceEvents)                            \
      tr_buf[(size_t(blockIdx.x) * 16 + (threadIdx.x >> 5)) * kTraceEvents + tr_k] =                    \
          (globaltimer() & 0xFFFFFFFFFFFFull) | (uint64_t((tag) & 0xFF) << 48) | (uint64_t((tile) & 0xFF) << 56); \
    ++tr_k;                                                                                             \
  } while (0)
#else
#define SMLA_TR(tag, tile) ((void)0)
#endif

constexpr int kThreadsTC = 512;
constexpr int kTileK = 64;                       // keys per tile
constexpr int kDChunks = 9;                      // 576 dims = 9 x 64 (128-byte rows)
constexpr int kChunkBytes = kTileK * 128;        // one 64-dim column block of a tile
constexpr int kTileBytes = kDChunks * kChunkBytes;
constexpr int kStages = 2;
constexpr int kQkWarpA = 12;   // QK K-steps [0, 18) -> S accumulator 0; owns TMEM
constexpr int kQkWarpB = 13;   // QK K-steps [18, 36) -> S accumulator 1
constexpr int kPvWarp = 14;    // PV
constexpr int kRopeWarp = 15;  // rope copier
constexpr int kQkSteps = kQK / 16;
constexpr float kRescaleMargin = 24.f;           // p <= 2^24 before a max update
constexpr float kInitMax = -1.0e30f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait (default) and per MMA drain

static_assert(kSchedTile == kTileK, "schedule and pipeline tiles must agree");

struct Misc {
  uint32_t tmem_base;
  int32_t abort;
  uint64_t wait_ns;       // limit of a pipeline wait
  int32_t stall;          // first softmax wait on a barrier never signalled
  int32_t is_last;
  int32_t first_row;      // schedule: first row of this CTA's range
  int64_t first_tile;     // schedule: that row's first slot
  int64_t total_tiles;    // schedule: W, the slot total
  int32_t n_tiles;        // schedule: this CTA's (real) tiles
  uint8_t valid[kStages][kTileK];
  float mref[64];         // per-head reference maxima (log2 units)
  float alpha[2][32];
  float red[2][4][32];    // tile maxima; key sums at a part's end
  float fac[64];
  int32_t nvr[4];         // key counts of a part, per quarter
};

template <int HP>
struct TcLayout {
  // softmax warpgroups: one holds all head columns up to 32 heads, two at 64;
  // the warps between them and the MMA issuers convert latents
  static constexpr int SWG = HP == 64 ? 2 : 1;
  static constexpr int kSoftmaxWarps = 4 * SWG;
  static constexpr int kConvWarps = 12 - kSoftmaxWarps;            // warps [4 SWG, 12)
  static constexpr int kPerConv = kTileK / kConvWarps;              // records per converter warp and tile
  static constexpr int kBatch = 8;                                   // records per load batch
  static constexpr int kSub = kPerConv / kBatch;                     // batches per tile
  static_assert(kPerConv * kConvWarps == kTileK && kSub * kBatch == kPerConv, "converter split");
  static constexpr int HH = HP / SWG;             // head columns per softmax warpgroup
  static constexpr int q_bytes = kDChunks * HP * 128;
  static constexpr int p_row = 2 * HP;            // bytes of one key's P^T row
  static constexpr int p_bytes = kTileK * p_row;
  // 64 heads: q takes 72 KB, so P^T is single-buffered to stay within 227 KB
  static constexpr int p_stages = HP == 64 ? 1 : 2;
  static constexpr int off_q = kStages * kTileBytes;
  static constexpr int off_p = off_q + q_bytes;
  static constexpr int off_bar = off_p + p_stages * p_bytes;
  static constexpr int off_misc = off_bar + 32 * 8;  // 17 barriers used
  // Up to 32 heads each converter warp also owns a ring of kRing raw-latent
  // slots (512 B) in shared memory, filled by cp.async kRing - 1 records ahead
  // of the conversion; at 64 heads there is no room and latents are gathered
  // into registers one batch ahead instead (kRing = 0).
  static constexpr int off_ring = (off_misc + int(sizeof(Misc)) + 127) / 128 * 128;
  static constexpr int ring_fit = (232448 - 1024 - off_ring) / (kConvWarps * kLatent);
  static constexpr int kRing = HP == 64 ? 0 : (ring_fit > 16 ? 16 : ring_fit);
  static_assert(HP == 64 || kRing >= 4, "ring too small");
  static constexpr int used = off_ring + kConvWarps * kRing * kLatent;
  // slack to align the dynamic shared memory base to 1024 bytes, when it fits
  static constexpr int slack = used + 1024 <= 232448 ? 1024 : 0;
  static constexpr int total = used + slack;
  // TMEM: S (2 stages x 2 accumulators) in [0, 4 HP), then n_ob O buffers of 4 HP columns
  static constexpr int n_ob = (4 * HP + 8 * HP <= 512) ? 2 : 1;
  static constexpr int tmem_need = 4 * HP + n_ob * 4 * HP;
  static constexpr int tmem_cols = tmem_need <= 128 ? 128 : (tmem_need <= 256 ? 256 : 512);
  static constexpr Swizzle p_swz = HP == 64 ? kSw128 : (HP == 32 ? kSw64 : kSw32);
  static constexpr uint32_t p_swmask = HP == 64 ? 7 : (HP == 32 ? 3 : 1);
  static constexpr uint32_t idesc_qk = idesc_bf16(64, HP, 0, 0);
  static constexpr uint32_t idesc_pv = idesc_bf16(128, HP, 1, 1);
  __host__ __device__ static constexpr uint32_t s_col(int stage, int acc) { return (2 * stage + acc) * HP; }
  __host__ __device__ static constexpr uint32_t o_col(int ob, int mt) { return 4 * HP + (ob * 4 + mt) * HP; }
};

// Offset of byte `b` (16-byte aligned) of row `r` inside a 128-byte-row
// swizzled block whose rows are 128 bytes apart (1024-byte atoms).
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t b) {
  return r * 128u + ((((b >> 4) ^ (r & 7u)) << 4) | (b & 15u));
}

// For an M=64 MMA, rows 16 w .. 16 w + 15 of S^T sit in lanes 32 w .. 32 w + 15
// of TMEM lane quarter w: lanes 0-15 of each warp hold keys.
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
  if (mbar_wait(bar, parity, ms->wait_ns)) return true;
  set_abort(ms, a);
  return false;
}

// The same, for a whole warp: the result is the same in every lane.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, Misc* ms, const DecodeArgs& a) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, ms, a));
}

// 16 E4M3 bytes (one lane's uint4) times a power-of-two scale -> 16 bf16,
// exactly, with integer bit placement and packed-bf16 multiplies (no
// float-format conversions, which run at a fraction of the ALU rate).  A byte
// s.eeee.mmm put into bf16 bits as s | eeee.mmm << 4 is the bf16 of value
// e4m3 * 2^-120 (E4M3 subnormals land on bf16 subnormals).  One exact multiply
// by scale * 2^120 finishes it when the scale is a normal power of two up to
// 2^7 (the record writer's scales for |latent| <= 57344: plain_scale);
// other scales go through dequant16_any.  Codes 0x7F / 0xFF (E4M3 NaN, never
// written by the writer) decode as finite values.
//
// Each 32-bit word [b0 b1 b2 b3] yields the pairs (b0, b2) and (b1, b3): five
// integer operations per four values.  So the lane's dims come out in the
// order 0 2 1 3 4 6 5 7 | 8 10 9 11 12 14 13 15; see latent_dim_of.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void dequant16(uint4 v, uint32_t m1, uint32_t (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t e = ((w[j] << 4) & 0x07F007F0u) | ((w[j] << 8) & 0x80008000u);  // b0, b2
    const uint32_t d = ((w[j] >> 4) & 0x07F007F0u) | (w[j] & 0x80008000u);         // b1, b3
    o[2 * j] = bf16x2_mul(e, m1);
    o[2 * j + 1] = bf16x2_mul(d, m1);
  }
}

// A scale word that dequant16 turns into an exact one-multiply factor: a
// positive normal power of two no larger than 2^7.
__device__ __forceinline__ bool plain_scale(uint32_t scw) {
  return (scw & 0x807FFFFFu) == 0u && scw - 0x00800000u <= 0x43000000u - 0x00800000u;
}

// The general path, for any f32 scale (zero, above 2^7, not a power of two,
// negative): each value e4m3 * scale is formed in f32 and rounded to bf16, so
// it is exact whenever that product is a bf16 (zero and power-of-two scales in
// range) and otherwise within one bf16 rounding (plus an f32 one).  The bytes
// go to f32 by the same bit placement as in dequant16 (value e4m3 * 2^-120,
// subnormals included), and the output pairs are ordered as there.
__device__ __forceinline__ float e4m3_scaled(uint32_t b, float sc) {  // b: the code in bits 0-7
  return __uint_as_float(((b & 0x7Fu) << 20) | ((b & 0x80u) << 24)) * 0x1p120f * sc;
}

__device__ __forceinline__ void dequant16_any(uint4 v, uint32_t scw, uint32_t (&o)[8]) {
  const float sc = __uint_as_float(scw);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    o[2 * j] = pack_bf16x2(e4m3_scaled(w[j], sc), e4m3_scaled(w[j] >> 16, sc));           // b0, b2
    o[2 * j + 1] = pack_bf16x2(e4m3_scaled(w[j] >> 8, sc), e4m3_scaled(w[j] >> 24, sc));  // b1, b3
  }
}

// Latent position p (0..511) of the shared-memory key tile, and of the staged
// q, holds latent dim latent_dim_of(p): bits 0 and 1 of p swapped (the pair
// order above) and, in odd 64-dim column blocks, bit 3 flipped (there the two
// 8-dim halves of a lane's 16 dims are stored in the opposite order, which
// keeps the converters' shared-memory stores free of bank conflicts).  The map
// is its own inverse.  QK contracts over positions, so it only has to be the
// same for K and q; the epilogue writes O^T lane p to dim latent_dim_of(p).
__device__ __forceinline__ int latent_dim_of(int p) {
  const int t = p ^ (((p >> 6) & 1) << 3);
  return (t & ~3) | ((t & 1) << 1) | ((t >> 1) & 1);
}

// Walks this CTA's tiles: row, slice positions, and where the row part starts
// and ends.  Every role keeps its own copy and advances it tile by tile.
struct Cursor {
  int32_t row;      // current row
  int32_t len;      // its slice length
  int32_t ntiles;   // its tile count T_row
  int32_t ta, tb;   // this CTA's tiles of the row: [ta, tb)
  int32_t t;        // current tile of the row
  int64_t P;        // the slot of the row's first tile (after its start slots)
  int64_t beg;      // offset of the row's slice in indices[]
  int64_t e;        // end of this CTA's slot range
  bool live;

  __device__ __forceinline__ void load_row(const DecodeArgs& a) {
    len = row_len(a, row);
    ntiles = tiles_of_len(len);
    beg = __ldg(a.indptr + row);
    const int64_t n = e - P;
    tb = int32_t(n < 0 ? 0 : (n < int64_t(ntiles) ? n : int64_t(ntiles)));
    if (tb <= 0) live = false;  // the range ends before this row's first tile
  }
  // r0: the row whose slots hold b; P0: its first slot.
  __device__ __forceinline__ void init(const DecodeArgs& a, int32_t r0, int64_t P0, int64_t b, int64_t e_) {
    row = r0;
    P = P0 + kRowStartSlots;
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
    P += ntiles + kRowStartSlots;
    ++row;
    if (P - kRowStartSlots >= e || row >= a.n_q) {
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
  __device__ __forceinline__ int32_t p0() const { return t * kTileK; }
  __device__ __forceinline__ int32_t p1() const {
    const int32_t x = t * kTileK + kTileK;
    return x < len ? x : len;
  }
};

template <int HP>
__global__ void __launch_bounds__(kThreadsTC, 1) decode_tc_kernel(DecodeArgs a) {
  using Lay = TcLayout<HP>;
  constexpr int HH = Lay::HH;
  constexpr int kSoftmaxWarps = Lay::kSoftmaxWarps;
  constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
  constexpr int kConvWarps = Lay::kConvWarps;
  constexpr int kPerConv = Lay::kPerConv;
  constexpr int kBatch = Lay::kBatch;
  constexpr int kSub = Lay::kSub;
  static_assert(Lay::total <= 232448, "shared memory over the per-block limit");
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#ifdef SMLA_TRACE
  unsigned long long* const tr_buf = g_smla_trace;
  int tr_k = 0;
#endif
  if (Lay::slack == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
    // no room to realign: refuse (uniformly, before any barrier or TMEM use)
    if (tid == 0 && a.status) atomicOr(a.status, SMLA_STATUS_SMEM_LAYOUT);
    return;
  }
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
  uint64_t* o_free = bars + 12;
  uint64_t* q_full = bars + 14;
  uint64_t* mma_drain = bars + 15;
  uint64_t* stall_bar = bars + 16;  // never signalled (timeout-path test)
  Misc* ms = reinterpret_cast<Misc*>(smem + Lay::off_misc);
  const int H = a.heads;
  const int64_t G = gridDim.x;
  const int64_t c_id = blockIdx.x;

  SMLA_TR(3, 0);  // kernel entry
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full + s, kConvWarps + 1);  // latent converters and the rope copier
      mbar_init(kv_empty + s, 1);
      mbar_init(s_full + s, 2);  // both QK halves
      mbar_init(s_empty + s, kSoftmaxWarps);
      mbar_init(p_full + s, kSoftmaxWarps);
      mbar_init(pv_done + s, 1);
      mbar_init(o_free + s, kSoftmaxWarps);
    }
    mbar_init(q_full, kSoftmaxWarps);
    mbar_init(mma_drain, 3);  // the three issuers
    mbar_init(stall_bar, 1);
    ms->abort = 0;
    const uint64_t w = g_tc_wait_ns;
    ms->wait_ns = w != 0 ? w : kWaitLimitNs;
    ms->stall = g_tc_stall;
    ms->is_last = 0;
    ms->first_row = a.n_q;
    ms->first_tile = 0;
    ms->n_tiles = 0;
    fence_mbar_init();
  }
  if (warp == kQkWarpA) {
    tmem_alloc(&ms->tmem_base, Lay::tmem_cols);
    tmem_relinquish();
  }

  // ---- schedule: tile counts of all rows, their prefix, and this CTA's first row.
  {
    int64_t* scan = reinterpret_cast<int64_t*>(tiles);  // tiles are free until the pipeline starts
    const int n = a.n_q;
    const int per = (n + kThreadsTC - 1) / kThreadsTC;
    const int lo = min(tid * per, n), hi = min(lo + per, n);
    int64_t local = 0;
#pragma unroll 1  // rolled (run once; small code)
    for (int r = lo; r < hi; ++r) local += kRowStartSlots + tiles_of_len(row_len(a, r));
    // exclusive scan of the 512 partial sums: within each warp, then over the
    // 16 warp totals
    int64_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int64_t v = lane < kThreadsTC / 32 ? scan[lane] : 0;
      int64_t t = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      if (lane < kThreadsTC / 32) scan[32 + lane] = t - v;  // warp offsets
      if (lane == 31) ms->total_tiles = t;
    }
    __syncthreads();
    const int64_t Tt = ms->total_tiles;
    const int64_t b = cta_begin(c_id, Tt, G), e = cta_begin(c_id + 1, Tt, G);
    int64_t P = scan[32 + warp] + x - local;  // slots before this thread's rows
    int32_t mine = 0;                         // tiles of these rows in [b, e)
#pragma unroll 1
    for (int r = lo; r < hi; ++r) {
      const int32_t nt_r = tiles_of_len(row_len(a, r));
      const int64_t w = kRowStartSlots + nt_r;
      if (P <= b && b < P + w) {
        ms->first_row = r;
        ms->first_tile = P;
      }
      const int64_t t0 = P + kRowStartSlots;
      const int64_t lo_t = b > t0 ? b : t0, hi_t = e < t0 + nt_r ? e : t0 + nt_r;
      if (hi_t > lo_t) mine += int32_t(hi_t - lo_t);
      if (c_id == 0 && a.row_tile) a.row_tile[r] = P;  // for the merge kernel
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
  SMLA_TR(1, 0);  // schedule known
  const int64_t T = ms->total_tiles;
  const int64_t cb = cta_begin(c_id, T, G), ce = cta_begin(c_id + 1, T, G);
  const int32_t n_tiles = ms->n_tiles;  // this CTA's tiles
  const int32_t row0 = ms->first_row;
  const int64_t P0 = ms->first_tile;
  const uint32_t tmem = ms->tmem_base;
  const uint32_t tiles_u32 = smem_u32(tiles);
  const uint32_t q_u32 = smem_u32(q_s);
  const uint32_t p_u32 = smem_u32(p_s);

  if (warp < kSoftmaxWarps) {
    // =================== softmax warpgroups ===================
    const int wg = warp >> 2, qd = warp & 3;
    const bool active = s_lane_active(lane);
    const int r = 16 * qd + lane;  // key of this thread within the tile (active lanes)
    float* mr = ms->mref + wg * HH;  // this warpgroup's reference maxima (uniform)
    float lpart[HH];
#pragma unroll
    for (int h = 0; h < HH; ++h) lpart[h] = 0.f;
    int nv = 0;
    // Stage row `row`'s q (bf16, 128-byte swizzled K-major [9][HP][128],
    // latent dims in latent_dim_of order) and signal the QK issuers.  Called
    // when every QK that read the previous q has completed.
    auto stage_q = [&](int row) {
      SMLA_TR(25, row);
      for (int k = tid; k < HP * (kQK / 8); k += kSoftmaxThreads) {
        const int h = k / (kQK / 8), c16 = k % (kQK / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (h < H)
          v = __ldg(reinterpret_cast<const uint4*>(a.q + row * a.q_stride_row + h * a.q_stride_head + c16 * 8));
        int pc = c16;  // position chunk of these 8 dims (latent_dim_of, applied per chunk)
        if (c16 < kLatent / 8) {
          pc = c16 ^ ((c16 >> 3) & 1);
          v = make_uint4(__byte_perm(v.x, v.y, 0x5410), __byte_perm(v.x, v.y, 0x7632),
                         __byte_perm(v.z, v.w, 0x5410), __byte_perm(v.z, v.w, 0x7632));
        }
        const uint32_t off =
            uint32_t(pc >> 3) * (HP * 128) + uint32_t(h >> 3) * 1024u + sw128_off(h & 7, (pc & 7) * 16);
        *reinterpret_cast<uint4*>(q_s + off) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    };
    Cursor c;
    c.init(a, row0, P0, cb, ce);
    int seg = 0;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const bool first = c.first(), last = c.last();
      const int ob = Lay::n_ob == 2 ? (seg & 1) : 0;
      if (i == 0) stage_q(c.row);  // later rows' q is staged once the previous part's P is out
      if (last && i + 1 < n_tiles) {
        // the next row's q is staged after this tile's P: bring it into L2 now
        const char* qn = reinterpret_cast<const char*>(a.q + int64_t(c.row + 1) * a.q_stride_row);
        for (int k = tid; k < H * (kQK * 2 / 128); k += kSoftmaxThreads) {
          const int h = k / (kQK * 2 / 128), line = k % (kQK * 2 / 128);
          prefetch_l2_line(qn + int64_t(h) * a.q_stride_head * 2 + line * 128);
        }
      }
      if (first) {
#pragma unroll
        for (int h = 0; h < HH; ++h) lpart[h] = 0.f;
        nv = 0;
      }
      SMLA_TR(10, i);
      if (i == 0 && ms->stall) wait_bar_warp(stall_bar, 0, ms, a);
      wait_bar_warp(kv_full + s, ph, ms, a);
      wait_bar_warp(s_full + s, ph, ms, a);
      SMLA_TR(11, i);
      tc_fence_after();
      float x[HH];
      {
        // S = the two QK halves' accumulators
        const uint32_t ta = tmem + (uint32_t(32 * qd) << 16) + Lay::s_col(s, 0) + uint32_t(wg * HH);
        const uint32_t tb = tmem + (uint32_t(32 * qd) << 16) + Lay::s_col(s, 1) + uint32_t(wg * HH);
#pragma unroll
        for (int cc = 0; cc < HH / 8; ++cc) {
          uint32_t v[8], w8[8];
          tmem_ld8(ta + 8 * cc, v);
          tmem_ld8(tb + 8 * cc, w8);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k) x[8 * cc + k] = __uint_as_float(v[k]) + __uint_as_float(w8[k]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + s);
      SMLA_TR(14, i);
      const bool valid = active && ms->valid[s][r];
      nv += valid;
      bool need = first;
#pragma unroll
      for (int h = 0; h < HH; ++h) {
        x[h] = valid ? x[h] * a.sm_scale_log2 : -INFINITY;
        need |= x[h] > mr[h] + kRescaleMargin;
      }
      need = named_barrier_or(1 + wg, 128, need);  // any thread of the warpgroup
      SMLA_TR(15, i);
      if (need) {
        // exact tile max of this warpgroup's heads (a butterfly reduce-scatter:
        // lane L ends with head L's max over the warp's keys), then lane h of the
        // warpgroup's first warp moves head h's reference and publishes its
        // factor; a row part starts from scratch (its old reference is -inf)
        {
          float v[HH];
#pragma unroll
          for (int h = 0; h < HH; ++h) v[h] = x[h];
#pragma unroll
          for (int hs = HH / 2; hs >= 1; hs >>= 1) {
            const bool up = (lane & hs) != 0;
#pragma unroll
            for (int j = 0; j < hs; ++j) {
              const float send = up ? v[j] : v[j + hs];
              const float keep = up ? v[j + hs] : v[j];
              v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, hs));
            }
          }
          float t = v[0];
          if (HH < 32) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, HH));
          if (lane < HH) ms->red[wg][qd][lane] = t;
        }
        named_barrier(1 + wg, 128);
        SMLA_TR(26, i);
        if (qd == 0 && lane < HH) {
          const int h = lane;
          const float tm = fmaxf(fmaxf(ms->red[wg][0][h], ms->red[wg][1][h]),
                                 fmaxf(ms->red[wg][2][h], ms->red[wg][3][h]));
          const float old = first ? kInitMax : mr[h];
          const float nm = fmaxf(old, tm);
          ms->alpha[wg][h] = ex2(old - nm);
          mr[h] = nm;
        }
        named_barrier(1 + wg, 128);  // the new references and factors are visible
#pragma unroll
        for (int h = 0; h < HH; ++h) lpart[h] *= ms->alpha[wg][h];
        SMLA_TR(27, i);
        if (!first) {
          // O^T columns of this warpgroup's heads, all four 128-dim tiles:
          // wait for PV(i-1), then scale in place.
          wait_bar_warp(pv_done + ((i - 1) & 1), ((i - 1) >> 1) & 1, ms, a);
          tc_fence_after();
          SMLA_TR(28, i);
          // 8-head chunks whose factors are all 1 keep their columns as they are
          uint32_t todo = 0;
#pragma unroll
          for (int cc = 0; cc < HH / 8; ++cc) {
            bool one = true;
#pragma unroll
            for (int k = 0; k < 8; ++k) one &= ms->alpha[wg][8 * cc + k] == 1.f;
            todo |= one ? 0u : (1u << cc);
          }
          constexpr int kCb = HH / 8 < 2 ? HH / 8 : 2;  // 8-column chunks per load batch
#pragma unroll 1
          for (int mt = 0; mt < 4 && todo != 0; ++mt) {
            const uint32_t taddr = tmem + (uint32_t(32 * qd) << 16) + Lay::o_col(ob, mt) + uint32_t(wg * HH);
#pragma unroll
            for (int c0 = 0; c0 < HH / 8; c0 += kCb) {
              if (!(todo & (((1u << kCb) - 1) << c0))) continue;
              // kCb chunks: all loads, one wait, scale, all stores
              uint32_t v[8 * kCb];
#pragma unroll
              for (int u = 0; u < kCb; ++u) tmem_ld8(taddr + 8 * (c0 + u), *reinterpret_cast<uint32_t(*)[8]>(&v[8 * u]));
              tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < kCb; ++u) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  v[8 * u + k] = __float_as_uint(__uint_as_float(v[8 * u + k]) * ms->alpha[wg][8 * (c0 + u) + k]);
                tmem_st8(taddr + 8 * (c0 + u), *reinterpret_cast<const uint32_t(*)[8]>(&v[8 * u]));
              }
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
        const float p1 = ex2(x[h + 1] - mr[h + 1]);
        lpart[h] += p0;
        lpart[h + 1] += p1;
        pk[h / 2] = pack_bf16x2(p0, p1);
      }
      SMLA_TR(16, i);
      // the P stage is free once the PV that last read it has completed
      if (Lay::p_stages == 2)
        wait_bar_warp(pv_done + s, ph ^ 1, ms, a);  // PV(i-2)
      else if (i > 0)
        wait_bar_warp(pv_done + ((i - 1) & 1), ((i - 1) >> 1) & 1, ms, a);  // PV(i-1)
      SMLA_TR(17, i);
      const int ps = Lay::p_stages == 2 ? s : 0;
      if (active) {
        uint8_t* prow = p_s + ps * Lay::p_bytes;
#pragma unroll
        for (int cc = 0; cc < HH / 8; ++cc) {
          uint32_t off = uint32_t(r) * Lay::p_row + uint32_t(wg * (HH / 8) + cc) * 16u;
          off ^= ((off >> 7) & Lay::p_swmask) << 4;
          *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + s);
      SMLA_TR(12, i);
      // The next row's q, before this part's epilogue, so that its QKs can
      // start meanwhile: every QK that read this row's q completed before S
      // was read above.
      if (last && i + 1 < n_tiles) stage_q(c.row + 1);

      if (last) {
        // ---------- epilogue of this row part ----------
        {
          // per-head key sums of this warp by a butterfly reduce-scatter: at
          // the step of half width hs a lane keeps the upper half of its heads
          // when its lane bit hs is set; after the steps lane L (< HH) holds
          // head L's sum over its 16-lane half, then the halves are added.
          float v[HH];
#pragma unroll
          for (int h = 0; h < HH; ++h) v[h] = active ? lpart[h] : 0.f;
#pragma unroll
          for (int hs = HH / 2; hs >= 1; hs >>= 1) {
            const bool up = (lane & hs) != 0;
#pragma unroll
            for (int j = 0; j < hs; ++j) {
              const float send = up ? v[j] : v[j + hs];
              const float keep = up ? v[j + hs] : v[j];
              v[j] = keep + __shfl_xor_sync(0xffffffffu, send, hs);
            }
          }
          float t = v[0];
          if (HH < 32) t += __shfl_xor_sync(0xffffffffu, t, HH);
          if (lane < HH) ms->red[wg][qd][lane] = t;
        }
        if (wg == 0) {
          int t = nv;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
          if (lane == 0) ms->nvr[qd] = t;
        }
        named_barrier(3, kSoftmaxThreads);
        SMLA_TR(24, i);
        const bool whole = c.whole();
        const int64_t slot = whole ? -1 : part_slot(c_id, c.P, T, G);
        const int row = c.row;
        if (tid < H) {
          const int g = tid / HH, hh = tid % HH;
          const float l = ms->red[g][0][hh] + ms->red[g][1][hh] + ms->red[g][2][hh] + ms->red[g][3][hh];
          const float m = ms->mref[tid];
          if (whole) {
            float fac, lse;
            finish_head(m, l, a.sink, tid, &fac, &lse);
            ms->fac[tid] = fac;
            if (a.lse) a.lse[int64_t(row) * H + tid] = lse;
          } else {
            a.ml_part[(slot * H + tid) * 2] = l > 0.f ? m : -INFINITY;
            a.ml_part[(slot * H + tid) * 2 + 1] = l > 0.f ? l : 0.f;
          }
        }
        if (tid == 0) {
          const int tot = ms->nvr[0] + ms->nvr[1] + ms->nvr[2] + ms->nvr[3];
          if (whole) {
            if (a.n_valid) a.n_valid[row] = tot;
          } else {
            a.nv_part[slot] = tot;
          }
        }
        named_barrier(3, kSoftmaxThreads);
        SMLA_TR(18, i);
        // O^T of the part: wait for its last PV, then read it out.
        wait_bar_warp(pv_done + s, ph, ms, a);
        tc_fence_after();
        SMLA_TR(19, i);
#pragma unroll 1
        for (int mt = wg; mt < 4; mt += Lay::SWG) {
          const int dg = latent_dim_of(mt * 128 + qd * 32 + lane);
          constexpr int kOc = HP / 8 < 2 ? HP / 8 : 2;  // 8-column chunks per TMEM wait
#pragma unroll 1
          for (int cc = 0; cc < HP / 8; cc += kOc) {
            uint32_t v[8 * kOc];
#pragma unroll
            for (int u = 0; u < kOc; ++u)
              tmem_ld8(tmem + (uint32_t(32 * qd) << 16) + Lay::o_col(ob, mt) + uint32_t(8 * (cc + u)),
                       *reinterpret_cast<uint32_t(*)[8]>(&v[8 * u]));
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 8 * kOc; ++k) {
              const int h = 8 * cc + k;
              if (h >= H) break;
              const float o = __uint_as_float(v[k]);
              if (whole)
                a.out[row * a.out_stride_row + h * a.out_stride_head + dg] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(o * ms->fac[h]));
              else
                a.o_part[(slot * H + h) * kLatent + dg] = o;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free + ob);
        SMLA_TR(13, i);
        ++seg;
      }
      c.advance(a);
    }
  } else if (warp == kQkWarpA || warp == kQkWarpB) {
    // =================== QK issuers (one K half each) ===================
    if (lane == 0) {
      const int half = warp == kQkWarpA ? 0 : 1;
      const int k0 = half * (kQkSteps / 2), k1 = k0 + kQkSteps / 2;
      Cursor c;
      c.init(a, row0, P0, cb, ce);
      int q_uses = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (c.first() && !wait_bar(q_full, (q_uses++) & 1, ms, a)) break;
        SMLA_TR(20, i);
        if (!wait_bar(kv_full + s, ph, ms, a) || !wait_bar(s_empty + s, ph ^ 1, ms, a)) break;
        SMLA_TR(21, i);
        tc_fence_after();
        const uint32_t tile = tiles_u32 + s * kTileBytes;
        const uint32_t d = tmem + Lay::s_col(s, half);
        // K step k reads bytes [32 (k % 4), +32) of every 128-byte row of
        // 64-dim chunk k / 4: the descriptors' start addresses (16-byte units)
        // step by 2, and to the next chunk after every fourth step.  Rolled:
        // the issue rate bounds this loop, and small code keeps the
        // instruction caches free for the other roles.
        const uint64_t a0 = smem_desc(tile, 16, 1024, kSw128), b0 = smem_desc(q_u32, 16, 1024, kSw128);
        uint32_t alo = uint32_t(a0) + uint32_t((k0 >> 2) * (kChunkBytes >> 4) + (k0 & 3) * 2);
        uint32_t blo = uint32_t(b0) + uint32_t((k0 >> 2) * (HP * 128 >> 4) + (k0 & 3) * 2);
        const uint32_t ahi = uint32_t(a0 >> 32), bhi = uint32_t(b0 >> 32);
#pragma unroll 1
        for (int k = k0; k < k1; ++k) {
          mma_f16_ss_w(d, alo, ahi, blo, bhi, Lay::idesc_qk, k > k0 ? 1u : 0u);
          const bool next_chunk = (k & 3) == 3;
          alo += next_chunk ? uint32_t((kChunkBytes >> 4) - 6) : 2u;
          blo += next_chunk ? uint32_t((HP * 128 >> 4) - 6) : 2u;
        }
        mma_commit(s_full + s);
        SMLA_TR(22, i);
        c.advance(a);
      }
      // every issued MMA has completed before TMEM is freed
      mma_commit(mma_drain);
      if (!mbar_wait(mma_drain, 0, kWaitLimitNs)) set_abort(ms, a);
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // =================== PV issuer ===================
    if (lane == 0) {
      Cursor c;
      c.init(a, row0, P0, cb, ce);
      int seg = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i & 1;
        const bool first = c.first();
        const int ob = Lay::n_ob == 2 ? (seg & 1) : 0;
        // a row part's first PV overwrites its O buffer: the epilogue of the
        // part that used it before must have read it out
        if (first && !wait_bar(o_free + ob, ((seg / Lay::n_ob) & 1) ^ 1, ms, a)) break;
        SMLA_TR(40, i);
        if (!wait_bar(p_full + s, (i >> 1) & 1, ms, a)) break;
        SMLA_TR(41, i);
        tc_fence_after();
        const uint32_t tile = tiles_u32 + s * kTileBytes;
        const uint32_t pst = p_u32 + (Lay::p_stages == 2 ? s : 0) * Lay::p_bytes;
        // k-major order: consecutive MMAs go to different O tiles.  O tile mt
        // reads 64-dim chunks 2 mt and 2 mt + 1; K step k (16 keys) starts
        // 2048 bytes into them and 16 P^T rows down (k rolled, as in the QK
        // issue).
        const uint64_t a0 = smem_desc(tile, kChunkBytes, 1024, kSw128);
        const uint64_t b0 = smem_desc(pst, 8 * Lay::p_row, 8 * Lay::p_row, Lay::p_swz);
        uint32_t alo = uint32_t(a0), blo = uint32_t(b0);
        const uint32_t ahi = uint32_t(a0 >> 32), bhi = uint32_t(b0 >> 32);
#pragma unroll 1
        for (int k = 0; k < kTileK / 16; ++k) {
          const uint32_t acc = (first && k == 0) ? 0u : 1u;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt)
            mma_f16_ss_w(tmem + Lay::o_col(ob, mt), alo + uint32_t(mt * (2 * kChunkBytes >> 4)), ahi, blo, bhi,
                         Lay::idesc_pv, acc);
          alo += 2048 >> 4;
          blo += 16 * Lay::p_row >> 4;
        }
        mma_commit(kv_empty + s);
        mma_commit(pv_done + s);
        SMLA_TR(42, i);
        if (c.last()) ++seg;
        c.advance(a);
      }
      mma_commit(mma_drain);
      if (!mbar_wait(mma_drain, 0, kWaitLimitNs)) set_abort(ms, a);
    }
    __syncwarp();
  } else if (warp == kRopeWarp) {
    // =================== rope copier ===================
    // Lane L holds the raw index entries of keys L and L + 32 of a tile, loaded
    // three tiles ahead and validated when their tile's copies are issued.
    auto raw_pair = [&](const Cursor& cu, int j) -> int32_t {
      const int kk = lane + 32 * j;
      if (!cu.live) return INT32_MIN;
      const int p = cu.p0() + kk;
      const int64_t off = cu.beg + p;
      if (p >= cu.p1() || off < 0 || off >= a.n_indices) return INT32_MIN;
      return __ldg(a.indices + off);
    };
    auto valid_key = [&](int32_t raw) -> int32_t {  // record row, or -1 when masked
      if (raw >= a.n_kv_rows) {
        if (a.status) atomicOr(a.status, SMLA_STATUS_INDEX_OOB);
        return -1;
      }
      return raw < 0 ? -1 : raw;
    };
    Cursor c3;
    c3.init(a, row0, P0, cb, ce);
    int32_t ra0 = raw_pair(c3, 0), rb0 = raw_pair(c3, 1);
    c3.advance(a);
    int32_t ra1 = raw_pair(c3, 0), rb1 = raw_pair(c3, 1);
    c3.advance(a);
    int32_t ra2 = raw_pair(c3, 0), rb2 = raw_pair(c3, 1);
    const uint8_t* kv_rope = a.kv + kScaleOffset + 16 + 16 * (lane & 7);  // rope chunk lane % 8
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      c3.advance(a);
      const int32_t ra3 = raw_pair(c3, 0), rb3 = raw_pair(c3, 1);
      SMLA_TR(50, i);
      if (!wait_bar_warp(kv_empty + s, ph ^ 1, ms, a)) break;
      SMLA_TR(51, i);
      const int32_t ka = valid_key(ra0), kb = valid_key(rb0);
      ms->valid[s][lane] = ka >= 0;
      ms->valid[s][lane + 32] = kb >= 0;
      uint8_t* rope_blk = tiles + s * kTileBytes + 8 * kChunkBytes;
#pragma unroll 1
      for (int m = 0; m < kTileK / 4; ++m) {
        const int key = 4 * m + (lane >> 3);
        const int32_t id = __shfl_sync(0xffffffffu, m < 8 ? ka : kb, key & 31);
        const uint32_t off = uint32_t(key) * 128u + ((uint32_t(lane & 7) ^ uint32_t(key & 7)) << 4);
        if (id >= 0)
          cp_async16(smem_u32(rope_blk + off), kv_rope + int64_t(id) * kRecordBytes);
        else
          *reinterpret_cast<uint4*>(rope_blk + off) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();        // the zero rows, for the tensor core
      cp_async_mbar_arrive(kv_full + s);  // the copies land before the tile is full
      __syncwarp();
      if (lane == 0) mbar_arrive(kv_full + s);
      SMLA_TR(52, i);
      ra0 = ra1; rb0 = rb1;
      ra1 = ra2; rb1 = rb2;
      ra2 = ra3; rb2 = rb3;
    }
    cp_async_wait_all();
  } else {
    // =================== latent converters ===================
    // Converter cw takes records cw, cw + kConvWarps, ... of each tile
    // (kPerConv of them), in kSub batches of kBatch; lane k of a key word holds
    // the record row of the warp's k-th record of a tile (-1 when masked).
    // Raw index entries are loaded three tiles ahead and validated when their
    // tile's first batch is loaded; each batch's loads are in flight while
    // the previous batch is converted.  Lane L converts latent bytes
    // [16 L, 16 L + 16) of every record (scale L / 8).
    const int cw = warp - kSoftmaxWarps;
    if constexpr (Lay::kRing > 0) {
      // Ring pipeline.  Record j of this warp's sequence (tile j / kPerConv,
      // record j % kPerConv) is copied into ring slot j % R by cp.async when
      // record j - R + 1 is converted; every lane copies and later reads only
      // its own 16 bytes of a slot, so a lane's cp.async.wait_group is all the
      // synchronisation the ring needs.  Keys of tiles t .. t+2 are held
      // validated, raw entries of tiles t+3 and t+4 are in flight; each tile's
      // scales (lane L: word L % 4 of record L / 4) are loaded a tile ahead.
      constexpr int R = Lay::kRing;
      static_assert(kPerConv * 4 == 32 && R <= 2 * kPerConv, "ring pipeline shape");
      const uint32_t ring_lane = smem_u32(smem + Lay::off_ring) + uint32_t(cw * R * kLatent) + 16u * lane;
      const uint8_t* kv_lat = a.kv + 16 * lane;
      const uint8_t* kv_sc = a.kv + kScaleOffset + 4 * (lane & 3);
      const uint32_t c_off = uint32_t(lane >> 2) * kChunkBytes;
      const uint32_t hf = (lane >> 2) & 1;
      const uint32_t slot_lo = ((uint32_t(lane & 3) * 2 + hf) << 4);
      const uint32_t slot_hi = ((uint32_t(lane & 3) * 2 + (hf ^ 1)) << 4);
      auto raw_key = [&](const Cursor& cu) -> int32_t {
        const int rr = cw + kConvWarps * lane;
        if (!cu.live || lane >= kPerConv) return INT32_MIN;
        const int p = cu.p0() + rr;
        const int64_t off = cu.beg + p;
        if (p >= cu.p1() || off < 0 || off >= a.n_indices) return INT32_MIN;
        return __ldg(a.indices + off);
      };
      auto key_id = [&](int32_t raw) -> int32_t { return (raw < 0 || raw >= a.n_kv_rows) ? -1 : raw; };
      auto load_scales = [&](int32_t keys) -> uint32_t {
        const int32_t id = __shfl_sync(0xffffffffu, keys, lane >> 2);
        return id >= 0 ? ldg_u32_now(kv_sc + int64_t(id) * kRecordBytes) : 0x3F800000u;  // masked: scale 1
      };
      Cursor cr;  // tile of the newest raw entries
      cr.init(a, row0, P0, cb, ce);
      const int32_t r0 = raw_key(cr);  // all five loads in flight before any is used
      cr.advance(a);
      const int32_t r1 = raw_key(cr);
      cr.advance(a);
      const int32_t r2 = raw_key(cr);
      cr.advance(a);
      int32_t r3 = raw_key(cr);
      cr.advance(a);
      int32_t r4 = raw_key(cr);
      int32_t k0 = key_id(r0), k1 = key_id(r1), k2 = key_id(r2);
      uint32_t sc_cur = load_scales(k0), sc_next = load_scales(k1);
      const int n_total = n_tiles * kPerConv;
      // Records go in groups of G (one cp.async group each), converted
      // together so that their dependency chains overlap.
      constexpr int G = R >= 12 ? 4 : 2;
      constexpr int RG = R / G;  // ring slots in groups
      static_assert(kPerConv % G == 0, "groups within a tile");
      static_assert(RG >= 3, "at least two groups in flight");
      int t = 0;       // tile being converted (keys k0)
      bool fast = false;   // this tile takes the fast path
      bool plain = false;  // every scale of this tile is plain (masked records count as plain);
                           // otherwise the tile is converted again at its end
      // the warp's rows cw + kConvWarps kk all have r % 8 == cw % 8 (kConvWarps is 8)
      static_assert(kConvWarps == 8, "row swizzle constant per warp");
      const uint32_t x_row = uint32_t(cw & 7) << 4;
      int gslot = 0;   // ring group slot of the group being converted
      int igslot = 0;  // ring group slot of the group being issued
      auto issue = [&](int jj0) {  // copy records jj0 .. jj0+G-1 (tiles t .. t+2) into group slot igslot
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int jj = jj0 + g;
          const int d = jj / kPerConv - t;
          const int32_t id =
              jj < n_total ? __shfl_sync(0xffffffffu, d == 0 ? k0 : (d == 1 ? k1 : k2), jj % kPerConv) : -1;
          if (id >= 0)
            cp_async16(ring_lane + uint32_t((igslot * G + g) * kLatent), kv_lat + int64_t(id) * kRecordBytes);
        }
        cp_async_commit();
        igslot = igslot + 1 == RG ? 0 : igslot + 1;
      };
#pragma unroll 1
      for (int jj = 0; jj < (RG - 1) * G; jj += G) issue(jj);
#pragma unroll 1
      for (int j = 0; j < n_total; j += G) {
        const int k = j % kPerConv;
        if (k == 0) {
          if (j > 0) {  // next tile: move the key and scale pipelines on
            ++t;
            k0 = k1;
            k1 = k2;
            k2 = key_id(r3);
            r3 = r4;
            cr.advance(a);
            r4 = raw_key(cr);
            sc_cur = sc_next;
            sc_next = load_scales(k1);
          }
          SMLA_TR(30, t);
          if (!wait_bar_warp(kv_empty + (t & 1), ((t >> 1) & 1) ^ 1, ms, a)) break;
          SMLA_TR(31, t);
        }
        const int s = t & 1;
        if (k == 0) {
          // per tile: every scale plain, and every key valid too -> the fast path
          const bool pl = plain_scale(sc_cur);
          plain = __all_sync(0xffffffffu, pl);
          fast = __all_sync(0xffffffffu, pl && (lane >= kPerConv || k0 >= 0));
        }
        cp_async_wait_group<RG - 2>();  // this lane's 16 bytes of records j .. j+G-1 have landed
        uint8_t* tile_base = tiles + s * kTileBytes + c_off + uint32_t(cw) * 128u;  // row r = cw + kConvWarps kk
        if (fast) {
          uint4 v[G];
          uint32_t m1[G];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            v[g] = ld_shared_v4(ring_lane + uint32_t((gslot * G + g) * kLatent));
            const uint32_t scw = __shfl_sync(0xffffffffu, sc_cur, 4 * (k + g) + (lane >> 3));
            m1[g] = __byte_perm(scw, 0u, 0x3232) + 0x3C003C00u;  // bf16 scale * 2^120, twice
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            uint32_t o[8];
            dequant16(v[g], m1[g], o);
            uint8_t* rb = tile_base + uint32_t(kConvWarps * (k + g)) * 128u;
            *reinterpret_cast<uint4*>(rb + (slot_lo ^ x_row)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(rb + (slot_hi ^ x_row)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        } else {
#pragma unroll 1
          for (int g = 0; g < G; ++g) {
            const int32_t id = __shfl_sync(0xffffffffu, k0, k + g);
            uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (id >= 0) {  // uniform over the warp
              const uint4 v = ld_shared_v4(ring_lane + uint32_t((gslot * G + g) * kLatent));
              const uint32_t scw = __shfl_sync(0xffffffffu, sc_cur, 4 * (k + g) + (lane >> 3));
              dequant16(v, __byte_perm(scw, 0u, 0x3232) + 0x3C003C00u /* scale 2^120, twice */, o);
            }
            uint8_t* rb = tile_base + uint32_t(kConvWarps * (k + g)) * 128u;
            *reinterpret_cast<uint4*>(rb + (slot_lo ^ x_row)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(rb + (slot_hi ^ x_row)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        issue(j + (RG - 1) * G);  // into the group slot read one step ago
        gslot = gslot + 1 == RG ? 0 : gslot + 1;
        if (k + G == kPerConv) {
          if (!plain) {
            // a scale that is not plain (never written by the record writer):
            // the tile's valid records again, from global memory, by the
            // general path, over the rows stored above (same lanes, same bytes)
#pragma unroll 1
            for (int kk = 0; kk < kPerConv; ++kk) {
              const int32_t id = __shfl_sync(0xffffffffu, k0, kk);
              if (id < 0) continue;  // uniform over the warp
              uint32_t o[8];
              dequant16_any(ldg_v4_now(kv_lat + int64_t(id) * kRecordBytes),
                            __shfl_sync(0xffffffffu, sc_cur, 4 * kk + (lane >> 3)), o);
              uint8_t* rb = tile_base + uint32_t(kConvWarps * kk) * 128u;
              *reinterpret_cast<uint4*>(rb + (slot_lo ^ x_row)) = make_uint4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<uint4*>(rb + (slot_hi ^ x_row)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(kv_full + s);
          SMLA_TR(32, t);
        }
      }
      cp_async_wait_all();
    } else {
    const uint8_t* kv_lat = a.kv + 16 * lane;
    const uint8_t* kv_sc = a.kv + kScaleOffset + 4 * (lane & 3);  // scale word lane % 4 of a record
    const uint32_t c_off = uint32_t(lane >> 2) * kChunkBytes;  // 64-dim column block of the lane's dims
    const uint32_t hf = (lane >> 2) & 1;                      // odd block: halves stored swapped
    const uint32_t slot_lo = ((uint32_t(lane & 3) * 2 + hf) << 4);
    const uint32_t slot_hi = ((uint32_t(lane & 3) * 2 + (hf ^ 1)) << 4);
    auto raw_key = [&](const Cursor& cu) -> int32_t {
      const int rr = cw + kConvWarps * lane;
      if (!cu.live || lane >= kPerConv) return INT32_MIN;
      const int p = cu.p0() + rr;
      const int64_t off = cu.beg + p;
      if (p >= cu.p1() || off < 0 || off >= a.n_indices) return INT32_MIN;
      return __ldg(a.indices + off);
    };
    auto key_id = [&](int32_t raw) -> int32_t { return (raw < 0 || raw >= a.n_kv_rows) ? -1 : raw; };
    // A batch: kBatch records' latent bytes (lane L: bytes [16 L, 16 L + 16)),
    // their scales (lane L: word L % 4 of record L / 4) and the key word.
    struct Batch {
      uint4 lat[kBatch];
      uint32_t sc;
      int32_t keys;
    };
    static_assert(kBatch * 4 == 32, "one scale word per lane");
    auto load_rec = [&](Batch& B, int k, int sub) {
      const int32_t id = __shfl_sync(0xffffffffu, B.keys, (sub * kBatch + k) & 31);
      B.lat[k] = make_uint4(0, 0, 0, 0);  // a masked record converts to zeros
      if (id >= 0) B.lat[k] = ldg_v4_now(kv_lat + int64_t(id) * kRecordBytes);
    };
    auto load_scales = [&](Batch& B, int32_t keys, int sub) {
      B.keys = keys;
      const int32_t id = __shfl_sync(0xffffffffu, keys, (sub * kBatch + (lane >> 2)) & 31);
      B.sc = 0x3F800000u;  // a masked record (zero latent) takes scale 1: the plain path
      if (id >= 0) B.sc = ldg_u32_now(kv_sc + int64_t(id) * kRecordBytes);
    };
    // Record k of a batch: dequantise and store row r = cw + kConvWarps kk of
    // the tile (16-byte slots swizzled with r % 8).  The one-multiply path,
    // exact for plain scales; a batch holding any other scale is redone by
    // convert_general after it.
    auto store_rec = [&](uint8_t* tile, int k, int sub, const uint32_t (&o)[8]) {
      const int r = cw + kConvWarps * (sub * kBatch + k);
      uint8_t* rb = tile + c_off + uint32_t(r) * 128u;
      const uint32_t x = uint32_t(r & 7) << 4;
      *reinterpret_cast<uint4*>(rb + (slot_lo ^ x)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(rb + (slot_hi ^ x)) = make_uint4(o[4], o[5], o[6], o[7]);
    };
    auto convert_rec = [&](const Batch& B, int k, uint8_t* tile, int sub) {
      const uint32_t scw = __shfl_sync(0xffffffffu, B.sc, 4 * k + (lane >> 3));  // scale of lane's block
      uint32_t o[8];
      dequant16(B.lat[k], __byte_perm(scw, 0u, 0x3232) + 0x3C003C00u /* scale 2^120, twice */, o);
      store_rec(tile, k, sub, o);
    };
    // A batch with a scale that is not plain (never written by the record
    // writer): every valid record again, by the general path, over the rows
    // convert_rec stored (the same lanes store the same bytes, in order).
    auto convert_general = [&](const Batch& B, uint8_t* tile, int sub) {
#pragma unroll 1
      for (int k = 0; k < kBatch; ++k) {
        const int32_t id = __shfl_sync(0xffffffffu, B.keys, (sub * kBatch + k) & 31);
        if (id < 0) continue;  // uniform over the warp: a masked record stays zero
        uint32_t o[8];
        dequant16_any(ldg_v4_now(kv_lat + int64_t(id) * kRecordBytes),
                      __shfl_sync(0xffffffffu, B.sc, 4 * k + (lane >> 3)), o);
        store_rec(tile, k, sub, o);
      }
    };
    Cursor c3;  // the tile whose raw entries are loaded next
    c3.init(a, row0, P0, cb, ce);
    int32_t rk0 = raw_key(c3);
    c3.advance(a);
    int32_t rk1 = raw_key(c3);
    c3.advance(a);
    int32_t rk2 = raw_key(c3);
    int sub_l = 0;            // batch of the loading tile
    int32_t keys_l = key_id(rk0);
    auto next_load = [&]() {  // move the loading point one batch on
      if (++sub_l == kSub) {
        sub_l = 0;
        c3.advance(a);
        const int32_t rk3 = raw_key(c3);
        keys_l = key_id(rk1);
        rk1 = rk2;
        rk2 = rk3;
      }
    };
    const int n_batches = n_tiles * kSub;
    // One batch step: convert `cur` record by record, issuing the loads of
    // `nxt` (the next batch) in between, so that the gathers' L1 work and the
    // conversion overlap.
    auto step = [&](int q, const Batch& cur, Batch& nxt) -> bool {
      const int i = q / kSub, sub = q % kSub;
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const bool more = q + 1 < n_batches;
      const int nsub = sub_l;
      if (more) load_scales(nxt, keys_l, nsub);
      SMLA_TR(30, i);
      if (sub == 0 && !wait_bar_warp(kv_empty + s, ph ^ 1, ms, a)) return false;
      SMLA_TR(31, i);
      uint8_t* tile = tiles + s * kTileBytes;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        convert_rec(cur, k, tile, sub);
        if (more) load_rec(nxt, k, nsub);
      }
      if (!__all_sync(0xffffffffu, plain_scale(cur.sc))) convert_general(cur, tile, sub);
      if (more) next_load();
      if (sub == kSub - 1) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(kv_full + s);
        SMLA_TR(32, i);
      }
      return true;
    };
    Batch A, B;
    if (n_batches > 0) {
      load_scales(A, keys_l, 0);
#pragma unroll
      for (int k = 0; k < kBatch; ++k) load_rec(A, k, 0);
      next_load();
    }
    for (int q = 0; q < n_batches; q += 2) {
      if (!step(q, A, B)) break;
      if (q + 1 < n_batches && !step(q + 1, B, A)) break;
    }
    }
  }

  SMLA_TR(2, 0);
  // ---------------- teardown ----------------
  tc_fence_before();
  __syncthreads();
  if (warp == kQkWarpA) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::tmem_cols);
  }
}

// Merge kernel: merges each head's partials of a row that was shared between
// CTAs of the decode launch ([P2] stage_combine: max of the parts' maxima,
// rescaled sums, sink in the denominator); rows finished whole there are
// skipped.  The decode launch's CTA 0 left every row's first slot and the
// slot total in the workspace.  kSplit = 1: a warp per (row, head), four per
// CTA.  kSplit = 8 (rows shared by many CTAs): a CTA of eight warps per
// (row, head), warp w taking parts ca + w, ca + w + 8, ..., the warps'
// results meeting in shared memory.  One pass: a part's slot comes from the
// schedule, so its (m, l) and its O rows (lane L: latent dims [16 L, 16 L +
// 16)) are loaded together, two parts at a time with kSplit = 1 (fewer
// registers, more CTAs per SM: rows of a few parts are latency bound) and four
// with kSplit = 8, and the warp keeps a running maximum, rescaling its sums
// when it moves.
constexpr int kMergeWarps = 4;   // warps per CTA with kSplit = 1
constexpr int kMergeSplit = 8;   // warps per (row, head) for rows with many parts

template <int kSplit>
__global__ void __launch_bounds__(32 * (kSplit == 1 ? kMergeWarps : kSplit)) merge_rows_kernel(DecodeArgs a) {
  constexpr int kMergeBatch = kSplit == 1 ? 2 : 4;  // parts' loads in flight per warp
  __shared__ float red_m[kSplit], red_l[kSplit];
  __shared__ int32_t red_nv[kSplit];
  __shared__ float red_acc[kSplit][16][33];  // [warp][value][lane], padded
  const int lane = threadIdx.x & 31;
  const int w = kSplit == 1 ? 0 : int(threadIdx.x >> 5);  // this warp's place among the pair's warps
  const int H = a.heads;
  const int64_t pair = kSplit == 1 ? int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5) : int64_t(blockIdx.x);
  if (pair >= int64_t(a.n_q) * H) return;
  const int row = int(pair / H), h = int(pair % H);
  const int64_t P = __ldcg(a.row_tile + row) + a.row_start_slots;  // the row's first tile slot
  const int64_t T = __ldcg(a.row_tile + a.n_q), G = a.grid;
  const int64_t S = a.tile_slots;  // tile t of the row: first slot P + S t
  const int32_t nt = int32_t((__ldcg(a.row_tile + row + 1) - P) >> (__ffsll(S) - 1));
  const int64_t ca = cta_of_tile(P, T, G), cb = cta_of_tile(P + S * (nt - 1), T, G);
  if (ca == cb) return;  // finished whole by one CTA
  if (a.merge_min_parts > 2) {  // rows of fewer parts were merged by the decode kernel
    int64_t parts = 0;
    for (int64_t c = ca; c <= cb && parts < a.merge_min_parts; ++c) parts += cta_holds_tile(c, P, nt, S, T, G);
    if (parts < a.merge_min_parts) return;
  }
  // this warp's parts: c = ca + w + kSplit i
  const int64_t first = ca + w;
  const int64_t n_mine = first <= cb ? (cb - first) / kSplit + 1 : 0;
  float mrun = -INFINITY, lsum = 0.f;  // running maximum and the sum against it
  int nvsum = 0;
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.f;
#pragma unroll 1
  for (int64_t i0 = 0; i0 < n_mine; i0 += 32) {
    // lane j: part i0 + j's slot (from the schedule) and its (m, l)
    const int64_t c = first + kSplit * (i0 + lane);
    int64_t sl = -1;
    float2 ml = make_float2(-INFINITY, 0.f);
    if (c <= cb && cta_holds_tile(c, P, nt, S, T, G)) {  // a CTA with tiles of the row
      sl = part_slot(c, P, T, G);
      ml = __ldcg(reinterpret_cast<const float2*>(a.ml_part + (sl * H + h) * 2));
    }
    if (h == 0 && sl >= 0) nvsum += __ldcg(a.nv_part + sl);
    const int n = int(n_mine - i0 < 32 ? n_mine - i0 : 32);
#pragma unroll 1
    for (int j = 0; j < n; j += kMergeBatch) {
      float4 v[kMergeBatch][4];
      int64_t slj[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {  // O rows first: their addresses need only the slot
        slj[u] = __shfl_sync(0xffffffffu, sl, (j + u) & 31);
        if (j + u >= n) slj[u] = -1;
        const float4* src = reinterpret_cast<const float4*>(a.o_part + (slj[u] * H + h) * kLatent + 16 * lane);
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = slj[u] >= 0 ? __ldcg(src + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const float m = __shfl_sync(0xffffffffu, ml.x, (j + u) & 31);
        const float l = __shfl_sync(0xffffffffu, ml.y, (j + u) & 31);
        if (slj[u] < 0 || !(l > 0.f)) continue;  // uniform over the warp
        if (m > mrun) {  // the running maximum moves: rescale what was summed
          const float f = exp2f(mrun - m);
          lsum *= f;
#pragma unroll
          for (int q = 0; q < 16; ++q) acc[q] *= f;
          mrun = m;
        }
        const float wt = exp2f(m - mrun);
        lsum = fmaf(l, wt, lsum);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[4 * q] = fmaf(wt, v[u][q].x, acc[4 * q]);
          acc[4 * q + 1] = fmaf(wt, v[u][q].y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(wt, v[u][q].z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(wt, v[u][q].w, acc[4 * q + 3]);
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) nvsum += __shfl_xor_sync(0xffffffffu, nvsum, o);
  float mstar = mrun;
  if (kSplit > 1) {
    if (lane == 0) {
      red_m[w] = mrun;
      red_l[w] = lsum;
      red_nv[w] = nvsum;
    }
#pragma unroll
    for (int q = 0; q < 16; ++q) red_acc[w][q][lane] = acc[q];
    __syncthreads();
    if (w != 0) return;
    mstar = red_m[0];
#pragma unroll
    for (int k = 1; k < kSplit; ++k) mstar = fmaxf(mstar, red_m[k]);
    lsum = 0.f;
    nvsum = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) acc[q] = 0.f;
#pragma unroll 1
    for (int k = 0; k < kSplit; ++k) {
      const float f = red_l[k] > 0.f ? exp2f(red_m[k] - mstar) : 0.f;
      lsum = fmaf(red_l[k], f, lsum);
      nvsum += red_nv[k];
#pragma unroll
      for (int q = 0; q < 16; ++q) acc[q] = fmaf(f, red_acc[k][q][lane], acc[q]);
    }
  }
  float fac = 0.f, lse = 0.f;
  finish_head(mstar, lsum, a.sink, h, &fac, &lse);
  if (lane == 0) {
    if (a.lse) a.lse[int64_t(row) * H + h] = lse;
    if (h == 0 && a.n_valid) a.n_valid[row] = nvsum;
  }
  uint4 lo, hi;
  lo.x = pack_bf16x2(acc[0] * fac, acc[1] * fac);
  lo.y = pack_bf16x2(acc[2] * fac, acc[3] * fac);
  lo.z = pack_bf16x2(acc[4] * fac, acc[5] * fac);
  lo.w = pack_bf16x2(acc[6] * fac, acc[7] * fac);
  hi.x = pack_bf16x2(acc[8] * fac, acc[9] * fac);
  hi.y = pack_bf16x2(acc[10] * fac, acc[11] * fac);
  hi.z = pack_bf16x2(acc[12] * fac, acc[13] * fac);
  hi.w = pack_bf16x2(acc[14] * fac, acc[15] * fac);
  uint4* dst = reinterpret_cast<uint4*>(a.out + row * a.out_stride_row + h * a.out_stride_head + 16 * lane);
  dst[0] = lo;
  dst[1] = hi;
}

// Row trimming ([P1] "Tiles", has_invalid: rows may end in -1 padding): a CTA
// of kTrimWarps warps per row finds the last slice position holding an entry
// >= 0 and writes that position + 1 as the row's length for the decode
// launch.  The slice is cut into chunks of 512 positions; warp w takes chunks
// last - w, last - w - kTrimWarps, ... (16 loads per lane in flight per chunk)
// and stops at its first chunk with such an entry; the row's answer is the
// largest over the warps.  Every position cut off is masked, so the results
// are unchanged; the decode only skips tiles that hold no key.
constexpr int kTrimWarps = 4;
constexpr int kTrimUnroll = 16;
constexpr int kTrimChunk = 32 * kTrimUnroll;

__global__ void __launch_bounds__(32 * kTrimWarps) trim_rows_kernel(DecodeArgs a, int32_t* lens_out) {
  __shared__ int32_t best_w[kTrimWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = int(blockIdx.x);
  const int32_t len = row_len(a, row);
  const int64_t beg = __ldg(a.indptr + row);
  const int32_t n_chunks = (len + kTrimChunk - 1) / kTrimChunk;
  int32_t found = 0;
#pragma unroll 1
  for (int32_t ch = n_chunks - 1 - warp; ch >= 0; ch -= kTrimWarps) {
    int32_t best = 0;
#pragma unroll
    for (int u = 0; u < kTrimUnroll; ++u) {
      const int32_t pos = ch * kTrimChunk + 32 * u + lane;
      const int64_t off = beg + pos;
      const int32_t v = (pos < len && off >= 0 && off < a.n_indices) ? __ldg(a.indices + off) : -1;
      if (v >= 0) best = pos + 1;  // positions grow with u
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (best > 0) {
      found = best;
      break;
    }
  }
  if (lane == 0) best_w[warp] = found;
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t keep = 0;
#pragma unroll
    for (int w = 0; w < kTrimWarps; ++w) keep = max(keep, best_w[w]);
    lens_out[row] = keep;
  }
}

template <int HP>
cudaError_t launch_tc_hp(const DecodeLaunch& L) {
  const int smem = TcLayout<HP>::total;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<HP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  DecodeArgs args = make_decode_args(L);
  e = launch_trim(L, args);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<HP><<<L.plan.grid, kThreadsTC, smem, L.stream>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess || !L.plan.merge_kernel) return e;
  return launch_merge(L, args);
}

}  // namespace

cudaError_t launch_trim(const DecodeLaunch& L, DecodeArgs& args) {
  if (!(L.plan.trim_kernel && L.ws.lens_off >= 0)) return cudaSuccess;
  int32_t* lens_trim = reinterpret_cast<int32_t*>(static_cast<char*>(L.workspace) + L.ws.lens_off);
  trim_rows_kernel<<<unsigned(L.p.n_q), 32 * kTrimWarps, 0, L.stream>>>(args, lens_trim);
  args.lens = lens_trim;  // the caller's lens already capped these
  return cudaGetLastError();
}

cudaError_t launch_merge(const DecodeLaunch& L, const DecodeArgs& args) {
  const int64_t pairs = int64_t(L.p.n_q) * L.p.num_heads;
  // rows shared by many CTAs (few rows over the grid) split each head's parts
  // over a CTA's eight warps
  if (int64_t(L.plan.grid) > 8 * int64_t(L.p.n_q))
    merge_rows_kernel<kMergeSplit><<<unsigned(pairs), 32 * kMergeSplit, 0, L.stream>>>(args);
  else
    merge_rows_kernel<1><<<unsigned((pairs + kMergeWarps - 1) / kMergeWarps), 32 * kMergeWarps, 0, L.stream>>>(args);
  return cudaGetLastError();
}

cudaError_t tc_set_wait_limit(uint64_t ns, int stall) {
  const int32_t st = stall ? 1 : 0;
  const cudaError_t e = cudaMemcpyToSymbol(g_tc_wait_ns, &ns, sizeof(ns));
  return e != cudaSuccess ? e : cudaMemcpyToSymbol(g_tc_stall, &st, sizeof(st));
}

cudaError_t launch_decode_tc(const DecodeLaunch& L) {
  if (L.plan.grid <= 0) return cudaSuccess;
  const int H = L.p.num_heads;
  if (H <= 16) return launch_tc_hp<16>(L);
  if (H <= 32) return launch_tc_hp<32>(L);
  return launch_tc_hp<64>(L);
}

}  // namespace smla
