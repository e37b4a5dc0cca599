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
//   0-3   softmax (warp q owns the keys of TMEM lane quarter q of S; heads
//         16 at a time, per-head values one per lane; at 32 heads only heads
//         0..15); each then issues the tile's PV of one 128-dim block
//   4-7   aux: E8M0 scale factors of each landed tile into TMEM, then the
//         tile's QK (16 heads: all four warps issue part of the K-steps into
//         their own accumulator; 32 heads: warps 4 and 5; a thread issues one
//         MMA every ~120 cycles); at 32 heads also the softmax of heads
//         16..31; each row part's epilogue (out / lse, or a partial of a
//         shared row) and, at 16 heads, the next part's q staging
//   8-15  loaders: keys lw, lw + 8, ... of every 128-key tile (64-bit record
//         addressing, masked keys zero-filled, out-of-range entries flagged);
//         at 32 heads also a new part's q staging
//
// The schedule is that of the bf16 tensor-core kernel counted in half-tile
// slots: a row takes one slot for its start and two per 128-key tile, CTA c
// takes the slots [floor(c W / G), floor((c+1) W / G)) and the tiles whose
// first slot lies there.  A row shared by up to four CTAs is merged inside
// the launch by the CTA whose part arrives last (per-row tickets); longer
// rows are left to the merge kernel.
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

#include <cstddef>
#include <cstdint>

#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_ptx.cuh"

#ifdef SMLA_TRACE
// Optional stage trace (compile with -DSMLA_TRACE): lane 0 of each warp writes
// (%globaltimer ns | tag << 48 | tile << 56) into
// g_smla_trace_fp8[(cta * 20 + warp) * 256 + k].  Off in normal builds.
__device__ unsigned long long* g_smla_trace_fp8;
extern "C" int smla_trace_fp8_set(void* buf) {
  unsigned long long* p = static_cast<unsigned long long*>(buf);
  return int(cudaMemcpyToSymbol(g_smla_trace_fp8, &p, sizeof(p)));
}
#define F8_TR(tag, tile)                                                                                  \
  do {                                                                                                    \
    if (tr_buf != nullptr && (threadIdx.x & 31) == 0 && tr_k < 256)                                       \
      tr_buf[(size_t(blockIdx.x) * 20 + (threadIdx.x >> 5)) * 256 + tr_k] =                               \
          (smla::ptx::globaltimer() & 0xFFFFFFFFFFFFull) | (uint64_t((tag) & 0xFF) << 48) |                \
          (uint64_t((tile) & 0xFF) << 56);                                                                 \
    ++tr_k;                                                                                               \
  } while (0)
#else
#define F8_TR(tag, tile) ((void)0)
#endif

namespace smla {

// Limit of every pipeline wait in ns (0: kWaitLimitNs), and whether the first
// softmax wait of each CTA waits on a barrier nothing signals (so that it runs
// out: a test of the timeout path); read at kernel start.
__device__ uint64_t g_fp8_wait_ns;
__device__ int32_t g_fp8_stall;

namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kTK = 128;        // keys per tile (M of QK)
constexpr int kStages = 2;
constexpr int kSoftmaxWarps = 4;   // one per TMEM lane quarter
constexpr int kAuxWarp0 = 4;        // aux warps; the first kQkSplit of them issue QK
constexpr int kLoadWarp0 = 8;
constexpr int kLoadWarps = 8;
constexpr int kKeysPerLoader = kTK / kLoadWarps;  // 16 (keys lw, lw + 8, ...)
constexpr float kLazy = 16.f;                     // reference max moves when passed by > 2^16
constexpr float kInitMax = -1.0e30f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait (default) and per MMA drain
constexpr int kMaxHP = 32;
// schedule slots per 128-key tile: a tile belongs to the CTA whose slot range
// holds its first slot, so that the CTAs' tile counts differ by at most one
// even where row starts cost fractions of a tile
constexpr int kTileSlots = 2;  // (a power of two: the merge kernel shifts by its log)

// ---- shared memory of a stage (bytes from a 1024-aligned base) ----
constexpr int kChunk = kTK * 128;                       // one 128-byte column block of a tile (16 KB)
constexpr int kOffRope = 4 * kChunk;                    // rope rows; P' of the tile once QK is done
constexpr int kOffSc = 5 * kChunk;                      // scales: kTK x 16 B
constexpr int kOffIds = kOffSc + kTK * 16;              // record ids (or -1): kTK x 4 B
constexpr int kStageBytes = (kOffIds + kTK * 4 + 1023) / 1024 * 1024;

// Layout of the kernel for HP padded heads per CTA (16 or 32).
//   S columns  [hi heads 0..HP-1 | lo heads 0..HP-1] (QK's N order: q rows the same)
//   O columns  per 128-dim block: [hi g0 | lo g0 | hi g1 | lo g1], g = 16-head group
//              (PV's N order: the P' rows the same), so that a 32-row group of
//              P' scale factors holds one head group
template <int HP>
struct Cfg {
  static constexpr int kN = 2 * HP;                     // N of QK and of PV
  static constexpr int kPass = HP / 16;                 // 16-head groups
  // QK: kQkSplit accumulators, one issuer each (16 heads: four issuers of 4
  // latent K-steps and one rope K-step each; 32 heads: two issuers of 8 and
  // 2); S single-buffered so that the TMEM columns fit
  static constexpr int kQkSplit = HP == 16 ? 4 : 2;
  // schedule slots charged for starting a row (its q staging and epilogue):
  // half a tile (kTileSlots = 2), measured best on decode (48.0 us against
  // 49.9 at two tiles) with ragged, wide and long unchanged within noise
  static constexpr int kRowStart = 1;
  // 32 heads: the aux warps take the softmax of heads 16..31 (the second
  // 16-head pass) of every tile, the softmax warps heads 0..15
  static constexpr bool kSplitPass = HP == 32;
  static constexpr int kPassA = kSplitPass ? 1 : kPass;           // passes of the softmax warps
  static constexpr int kSReaders = kSplitPass ? 8 : 4;            // warps reading a tile's S
  static constexpr int kSBuf = 1;
  static constexpr int kLatSteps = 16 / kQkSplit;       // latent K-steps of an issuer
  static constexpr int kNQ = HP == 16 ? 2 : 1;          // q buffers
  static constexpr int kNO = HP == 16 ? 2 : 1;          // O buffers in TMEM
  static constexpr int kQLatChunk = kN * 128;           // one K-chunk of [q_hi | q_lo]
  static constexpr int kQOffRope = 4 * kQLatChunk;
  static constexpr int kQBytes = (kQOffRope + HP * 128 + 1023) / 1024 * 1024;
  static constexpr int kPBlock = 32 * kN;               // P' of one 32-key chunk and dim block
  // P' of a tile: 16 blocks [chunk][dim block]; the first 16 KB sit in the
  // stage's rope rows (free once the tile's QK is done), the rest (32 heads)
  // in one extra buffer shared by both stages
  static constexpr int kPInRope = kChunk / kPBlock;     // blocks in the rope rows (16 or 8)
  static constexpr int kPExtra = 16 * kPBlock - kChunk; // 0 or 16 KB
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffPx = kOffQ + kNQ * kQBytes;
  static constexpr int kOffBar = kOffPx + kPExtra;
  static constexpr int kOffMisc = kOffBar + 32 * 8;
  static constexpr Swizzle kPSw = kN == 32 ? kSw32 : kSw64;
  static constexpr uint32_t kPSwMask = kN / 16 - 1;
  // TMEM columns
  static constexpr uint32_t kColS = 0;                            // [buffer][accumulator] x kN
  static constexpr uint32_t kColO = kSBuf * kQkSplit * kN;        // [buffer][block] x kN
  static constexpr uint32_t kColSfa = kColO + kNO * 4 * kN;       // record scale factors [stage] x 16
  static constexpr uint32_t kColSfq = kColSfa + 32;               // q scale factors [q buffer] x 16
  static constexpr uint32_t kColSfv = kColSfq + 16 * kNQ;         // V^T scale factors (all 1)
  static constexpr uint32_t kColSfp = kColSfv + 16;               // P' scale factors [stage] x 4: head group
  // scale-factor addresses of an MMA start on a multiple of 4 columns (the
  // 32x128b layout of a 128-row block spans 4 columns)
  __host__ __device__ static constexpr uint32_t sfp_col(int s) { return kColSfp + 4u * uint32_t(s); }
  static_assert(kColSfa % 16 == 0 && kColSfq % 16 == 0 && kColSfv % 16 == 0 && kColSfp % 4 == 0, "SF columns");
  static_assert(kColSfp + 8 <= 512, "TMEM columns");
  __host__ __device__ static constexpr uint32_t s_col(int sb, int acc = 0) {
    return kColS + uint32_t(sb * kQkSplit + acc) * kN;
  }
  __host__ __device__ static constexpr uint32_t o_col(int ob, int b) { return kColO + uint32_t(4 * ob + b) * kN; }
};

struct Misc {
  uint32_t tmem_base;
  int32_t abort;
  uint64_t wait_ns;  // limit of a pipeline wait
  int32_t stall;     // first softmax wait on kStall (never signalled)
  int32_t first_row;
  int32_t n_tiles;
  int64_t first_tile;
  int64_t total_tiles;
  int64_t scan[64];
  alignas(16) int32_t red_max_t[2][kMaxHP][4];  // tile maxima per head and lane quarter (order-preserving ints; read as one 16-byte word)
  int32_t red_sc[2][2][4][4];       // [group][buffer][lane quarter][block]: largest biased scale exponent
  float red_l[4][kMaxHP];
  int32_t red_nv[4];
  float part_m[2][kMaxHP];                      // per O buffer: a finished row part's (m, l, count)
  float part_l[2][kMaxHP];
  int32_t part_nv[2];
  uint8_t sfq[2 * kMaxHP][16];                  // q scale-factor bytes of the part being staged
  float fac[kMaxHP];                            // epilogue: output factors of a whole row's heads
  int32_t fast;                                 // the final part completes its row (decided at its last tile)
  int32_t fast_s_own;                           //   the stage that takes this part's O
  int32_t late;                                 // the same, decided in the final part's epilogue
  int32_t fnv[kMaxInKernelParts];               // final-part merge: the other parts' key counts
  // parts staged in shared memory for a combine: part j's O rows of heads
  // [cb_h, cb_h + cb_nh) at byte offset cb_row[j] (rows of 512 f32), its
  // (m, l) per head at cb_ml[j]
  uint32_t cb_row[kMaxInKernelParts];
  float2 cb_ml[kMaxInKernelParts][kMaxHP];
  int32_t last_row;                             // schedule: the row of this CTA's last slot
  int64_t last_tile;                            //   and that row's first slot
  // the CTAs sharing this CTA's first (x = 0) and last (x = 1) row: their
  // number, the range [ca, cz] they lie in, and the slots of the first
  // kMaxInKernelParts of them (found after the prologue, used by the merge)
  int32_t mparts[2];
  int64_t mP[2];                                // the row's first tile slot
  int64_t mca[2];
  int64_t mcz[2];
  int32_t mnt[2];                               // the row's tiles
  int64_t mslot[2][kMaxInKernelParts];
  int32_t n_merge;                              // rows this CTA completes and merges at its end
  int32_t merge_row[2];
  int32_t merge_x[2];                           // which of the two rows above
  int32_t merge_kind[2];                        // 1, 2: staged by the final part (see aux_stage_final)
  int32_t merge_own_nv;                         //   and that part's key count and slot
  int64_t merge_own_slot;
#ifdef SMLA_TRACE
  uint64_t merge_t[8];
#endif
};
// (the 16-byte reads of red_max_t rows and 4-byte reads of sfq rows need these)
static_assert(offsetof(Misc, red_max_t) % 16 == 0 && offsetof(Misc, sfq) % 4 == 0, "Misc layout");
static_assert(Cfg<16>::kOffMisc % 16 == 0 && Cfg<32>::kOffMisc % 16 == 0, "Misc alignment");
template <int HP>
constexpr int smem_total() { return Cfg<HP>::kOffMisc + int(sizeof(Misc)) + 1024; }  // + slack to align the base
static_assert(smem_total<16>() <= 232448 && smem_total<32>() <= 232448, "shared memory over the per-block limit");

enum Bar {
  kKvFull = 0,    // [2] loaders -> aux (tile landed)
  kKvEmpty = 2,   // [2] PV issuers -> loaders (tile consumed)
  kSFull = 6,     // [2] QK issuers -> softmax
  kSEmpty = 8,    // [2] softmax -> QK issuers
  kPvDone = 11,   // PV issuers -> softmax (P' buffer free, O quiescent)
  kQEmpty = 14,   // [2] QK issuers -> aux (a q buffer's last QK completed)
  kOFull = 16,    // [2] PV issuers -> aux (a part's O complete)
  kOEmpty = 18,   // [2] aux -> PV issuers and softmax (O buffer read out)
  kEpiReady = 20, // [2] softmax -> aux (a part's m, l, count posted)
  kDrain = 22,    // MMA issuers: every MMA they issued has completed
  kStall = 23,    // never signalled (timeout-path test)
  kMerge = 24,    // the end merge's bulk copies
  kPReady = 25,   // [2] 32 heads: aux warps -> PV issuers (heads 16..31 of a tile's P' written)
  kQReady = 27    // 32 heads: loader warps -> QK issuers (a new part's q staged)
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

// hi = E4M3(y), lo = E4M3(y - hi) for an f16 pair (round to nearest even,
// saturating); y - hi is exact in f16 (hi is within a factor 2 of y)
__device__ __forceinline__ void split_h2(uint32_t y, uint16_t& hi, uint16_t& lo) {
  __half2_raw yr;
  yr.x = uint16_t(y & 0xFFFFu);
  yr.y = uint16_t(y >> 16);
  hi = __nv_cvt_halfraw2_to_fp8x2(yr, __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&yr), *reinterpret_cast<const __half2*>(&hr));
  lo = __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&r), __NV_SATFINITE, __NV_E4M3);
}

// Four E4M3 codes of non-negative values (bytes < 0x80) -> the codes of the
// values times 2^-m (0 <= m <= 16): exponent fields lowered by m, and 0 for a
// value whose exponent field is <= m (it would leave the normal range).
__device__ __forceinline__ uint32_t lower_codes(uint32_t x, int m) {
  if (m == 0) return x;
  if (m >= 15) return 0u;                                     // exponent fields are at most 15
  const uint32_t t = uint32_t(8 * (m + 1)) * 0x01010101u;     // byte >= 8 (m + 1) <=> exponent field > m
  const uint32_t d = (x | 0x80808080u) - t;                   // bit 7 of a byte: byte >= t (no borrow)
  const uint32_t keep = ((d & 0x80808080u) >> 7) * 0xFFu;
  return (x & keep) - ((uint32_t(8 * m) * 0x01010101u) & keep);
}

// The same for an f32 pair (q staging: full f32 precision into the split)
__device__ __forceinline__ void split_pair(float x0, float x1, uint16_t& hi, uint16_t& lo) {
  hi = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  lo = __nv_cvt_float2_to_fp8x2(make_float2(x0 - hf.x, x1 - hf.y), __NV_SATFINITE, __NV_E4M3);
}

// Sum over the 32 lanes of v[h] for 16 heads at once: each halving step keeps
// half of the heads and adds the partner's copy of them, so that lane L ends
// with the total of head (L >> 1) & 15 (16 shuffles instead of 80).
__device__ __forceinline__ float sum16(const float (&v)[16], int lane) {
  float w8[8], w4[4], w2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float keep = b4 ? v[8 + j] : v[j], give = b4 ? v[j] : v[8 + j];
    w8[j] = keep + __shfl_xor_sync(0xffffffffu, give, 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float keep = b3 ? w8[4 + j] : w8[j], give = b3 ? w8[j] : w8[4 + j];
    w4[j] = keep + __shfl_xor_sync(0xffffffffu, give, 8);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = b2 ? w4[2 + j] : w4[j], give = b2 ? w4[j] : w4[2 + j];
    w2[j] = keep + __shfl_xor_sync(0xffffffffu, give, 4);
  }
  float w = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
  return w + __shfl_xor_sync(0xffffffffu, w, 1);
}

template <int kRowStart>
struct Cursor {
  int32_t row, len, ntiles, ta, tb, t;
  int64_t P, beg, e;
  bool live;
  __device__ __forceinline__ static int32_t tiles_of(int32_t len) { return len > 0 ? (len + kTK - 1) / kTK : 1; }
  __device__ __forceinline__ void load_row(const DecodeArgs& a) {
    len = row_len(a, row);
    ntiles = tiles_of(len);
    beg = __ldg(a.indptr + row);
    // the tiles whose first slot P + kTileSlots t lies before the range end
    const int64_t n = e > P ? (e - P + kTileSlots - 1) / kTileSlots : 0;
    tb = int32_t(n < int64_t(ntiles) ? n : int64_t(ntiles));
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
    ta = int32_t(b > P ? (b - P + kTileSlots - 1) / kTileSlots : 0);  // the first tile whose first slot is >= b
    t = ta;
  }
  __device__ __forceinline__ void advance(const DecodeArgs& a) {
    if (!live) return;
    if (++t < tb) return;
    P += int64_t(kTileSlots) * ntiles + kRowStart;
    ++row;
    if (P >= e || row >= a.n_q) {
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

__device__ __forceinline__ void set_abort(Misc* ms, int32_t* status) {
  if (atomicExch(&ms->abort, 1) == 0 && status) atomicOr(status, SMLA_STATUS_TIMEOUT);
}

// A bounded pipeline wait; after any timeout every later wait returns false
// at once so that all roles reach the teardown.  Loops holding named barriers
// keep iterating after a failed wait (same barrier sequence in every thread).
// The polling loop is out of line: one copy of it in the kernel's code.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, Misc* ms, int32_t* status) {
  if (*reinterpret_cast<volatile int32_t*>(&ms->abort)) return false;
  if (mbar_wait(bar, parity, ms->wait_ns)) return true;
  set_abort(ms, status);
  return false;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, Misc* ms, const DecodeArgs& a) {
  if (mbar_try_wait(bar, parity) && !*reinterpret_cast<volatile int32_t*>(&ms->abort)) return true;
  return wait_bar_slow(bar, parity, ms, a.status);
}
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, Misc* ms, const DecodeArgs& a) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, ms, a));
}

// The schedule's CTA boundaries (cta_begin / cta_of_tile of the shared
// schedule) through one out-of-line 64-bit division: a copy of the division
// routine at every call site would cost ~1 KB of instructions each.
__device__ __noinline__ int64_t div64(int64_t n, int64_t d) { return n / d; }
__device__ __forceinline__ int64_t cbeg(int64_t c, int64_t T, int64_t G) { return div64(c * T, G); }
__device__ __forceinline__ int64_t cof(int64_t t, int64_t T, int64_t G) { return div64((t + 1) * G - 1, T); }

// The tiles [lo, hi) of a row (first tile slot F, nt tiles, tile t at slot
// F + kTileSlots t) whose first slot lies in [b, e).
__device__ __forceinline__ void tiles_in(int64_t F, int32_t nt, int64_t b, int64_t e, int32_t& lo, int32_t& hi) {
  const int64_t l = b > F ? (b - F + kTileSlots - 1) / kTileSlots : 0;
  const int64_t h = e > F ? (e - F + kTileSlots - 1) / kTileSlots : 0;
  lo = int32_t(l < nt ? l : nt);
  hi = int32_t(h < nt ? h : nt);
}
// Whether CTA c holds a tile of that row.
__device__ __forceinline__ bool holds(int64_t c, int64_t F, int32_t nt, int64_t T, int64_t G) {
  int32_t lo, hi;
  tiles_in(F, nt, cbeg(c, T, G), cbeg(c + 1, T, G), lo, hi);
  return hi > lo;
}

// Slot of a shared row part (the partial layout of the merge kernel).
__device__ __forceinline__ int64_t slot_of(int64_t c, int64_t P, int64_t T, int64_t G) {
  return 2 * c + (P < cbeg(c, T, G) ? 0 : 1);
}

// What the aux warps' out-of-line steps need from the kernel.
struct AuxCtx {
  const DecodeArgs* a;
  uint8_t* smem;
  Misc* ms;
  uint64_t* bars;
  uint32_t tmem, lane_base;
  int H, h0, Hl, hg, g, lane, ta;
  int64_t c_id, G, T;
};

// q of a row -> [q_hi | q_lo] E4M3 (K-major, 128-byte swizzled) with an E8M0
// factor per (head, 32 dims) that brings the block's largest |q| to
// [2^7, 2^8); q_rope (bf16) copied as it is; then the factors into TMEM.
// Run by one warp group of nthreads threads (x.ta < nthreads; the aux warps,
// or at 32 heads the loader warps at a row boundary) with its named barrier
// bar_id; sf_writer: this warp writes the factors of its TMEM lane quarter.
// Out of line: one copy of its code.
template <int HP>
__device__ __noinline__ void aux_stage_q(const AuxCtx& x, int row, int qb, int nthreads, uint32_t bar_id,
                                         bool sf_writer) {
  const DecodeArgs& a = *x.a;
  using C = Cfg<HP>;
  constexpr int kN = C::kN;
  Misc* ms = x.ms;
  const uint32_t tmem = x.tmem, lane_base = x.lane_base;
  const int h0 = x.h0, Hl = x.Hl, lane = x.lane, ta = x.ta;
  uint8_t* qs = x.smem + C::kOffQ + qb * C::kQBytes;
  // (the arguments' fields in registers, not reloaded after every store)
  const uint16_t* const q_rows = a.q + row * a.q_stride_row + h0 * a.q_stride_head;
  const int64_t qsh = a.q_stride_head;
  // The q loads of the thread's next unit are issued before the current one
  // is converted, and the rope loads first of all: one global round trip
  // instead of one per unit (the staging sits between two QKs at 32 heads).
  constexpr int kRopeUnits = (HP * 8 + 127) / 128;
  uint4 rv[kRopeUnits];
#pragma unroll
  for (int r = 0; r < kRopeUnits; ++r) {
    const int k = ta + nthreads * r, h = k >> 3, c16 = k & 7;
    rv[r] = make_uint4(0, 0, 0, 0);
    if (k < HP * 8 && h < Hl) rv[r] = __ldg(reinterpret_cast<const uint4*>(q_rows + h * qsh + kLatent + 8 * c16));
  }
  auto load_unit = [&](int blk, uint4 (&v)[4]) {
    const int h = blk >> 4, kb = blk & 15;
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = make_uint4(0, 0, 0, 0);
    if (blk < HP * 16 && h < Hl) {
      const uint4* src = reinterpret_cast<const uint4*>(q_rows + h * qsh + 32 * kb);
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldg(src + k);
    }
  };
  uint4 vn[4];
  load_unit(ta, vn);
#pragma unroll 1
  for (int blk = ta; blk < HP * 16; blk += nthreads) {
    const int h = blk >> 4, kb = blk & 15;
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = vn[k];
    load_unit(blk + nthreads, vn);
    uint32_t hw[8], lw[8];
    int sfb = 127;
    if (h < Hl) {
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
    uint8_t* base = qs + kc * C::kQLatChunk;
    *reinterpret_cast<uint4*>(base + sw128(h, c0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(base + sw128(h, c0 + 1)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    *reinterpret_cast<uint4*>(base + sw128(HP + h, c0)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    *reinterpret_cast<uint4*>(base + sw128(HP + h, c0 + 1)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
    ms->sfq[h][kb] = uint8_t(sfb);
    ms->sfq[HP + h][kb] = uint8_t(sfb);
  }
#pragma unroll
  for (int r = 0; r < kRopeUnits; ++r) {  // rope: HP rows x 128 bytes, 16-byte chunks
    const int k = ta + nthreads * r, h = k >> 3, c16 = k & 7;
    if (k < HP * 8) *reinterpret_cast<uint4*>(qs + C::kQOffRope + sw128(h, c16)) = rv[r];
  }
    named_barrier(bar_id, nthreads);
    if (sf_writer) {
      // q factors: B row n = 32 j + lane in column 4 g + j of K-block group
      // g, byte k = K-block 4 g + k; unused columns hold 1
      uint32_t v[16];
#pragma unroll
      for (int gk = 0; gk < 4; ++gk)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          v[4 * gk + j] = j < kN / 32 ? *reinterpret_cast<const uint32_t*>(&ms->sfq[32 * j + lane][4 * gk])
                                      : 0x7F7F7F7Fu;
      tmem_st16(tmem + lane_base + C::kColSfq + 16 * qb, v);
      tmem_wait_st();
    }
    // (sfq is reused by the next staging.  The QKs that read this q are
    // issued after a barrier that follows these writes: the aux warps' named
    // barrier after the next tile's scale factors, or at 32 heads the
    // mbarrier the loader warps arrive on; this fence orders the q writes
    // before them)
    fence_proxy_async_smem();
    tc_fence_before();
  }

// [P2] stage_combine, with the sink, of `parts` parts staged in shared memory
// (cb_row, cb_ml): out and lse of heads [hb, hb + nh) of `row`.  Unit u: head
// u / 32, dims 4 c + 128 e (c = u % 32, e = 0..3), so that a warp reads
// consecutive 16-byte words; threads t, t + nthreads, ...
__device__ __noinline__ void combine_staged(const DecodeArgs& a, const uint8_t* smem, const Misc* ms, int parts,
                                            int row, int hb, int nh, int t, int nthreads, bool dry = false) {
  // (the arguments' fields in registers: read through the reference they would
  // be reloaded from the parameter buffer after every store)
  uint16_t* const out_row = a.out + int64_t(row) * a.out_stride_row;
  const int64_t osh = a.out_stride_head;
  float* const lse_row = a.lse ? a.lse + int64_t(row) * a.heads : nullptr;
  const float* const sink = a.sink;
#pragma unroll 1
  for (int u = t; u < nh * 32; u += nthreads) {
    const int hh = u / 32, c = u % 32;
    // every part's (m, l) and 16 values first (independent loads), then the sums
    float2 ml[kMaxInKernelParts];
    uint4 v[kMaxInKernelParts][4];
#pragma unroll
    for (int j = 0; j < kMaxInKernelParts; ++j) {
      ml[j] = make_float2(-INFINITY, 0.f);
      if (j < parts) {
        ml[j] = ms->cb_ml[j][hh];
        const uint4* src = reinterpret_cast<const uint4*>(smem + ms->cb_row[j]) + (hh * kLatent + 4 * c) / 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) v[j][e] = src[32 * e];  // dims 128 e + 4 c ..
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[j][e] = make_uint4(0, 0, 0, 0);
      }
    }
    float mrun = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxInKernelParts; ++j)
      if (ml[j].y != 0.f) mrun = fmaxf(mrun, ml[j].x);  // parts without keys (l = 0) take no part
    float acc[16];
#pragma unroll
    for (int d = 0; d < 16; ++d) acc[d] = 0.f;
    float lsum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxInKernelParts; ++j) {
      const float wt = ml[j].y != 0.f ? ex2(ml[j].x - mrun) : 0.f;  // a NaN m or l stays NaN
      lsum = fmaf(ml[j].y, wt, lsum);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[4 * e] = fmaf(wt, __uint_as_float(v[j][e].x), acc[4 * e]);
        acc[4 * e + 1] = fmaf(wt, __uint_as_float(v[j][e].y), acc[4 * e + 1]);
        acc[4 * e + 2] = fmaf(wt, __uint_as_float(v[j][e].z), acc[4 * e + 2]);
        acc[4 * e + 3] = fmaf(wt, __uint_as_float(v[j][e].w), acc[4 * e + 3]);
      }
    }
    const int h = hb + hh;
    float fac, lse_h;
    finish_head(mrun, lsum, sink, h, &fac, &lse_h);
    if (dry) continue;  // (a run that only brings this code into the instruction caches)
    uint16_t* dst = out_row + int64_t(h) * osh + 4 * c;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint2*>(dst + 128 * e) = make_uint2(pack_bf16x2(acc[4 * e] * fac, acc[4 * e + 1] * fac),
                                                            pack_bf16x2(acc[4 * e + 2] * fac, acc[4 * e + 3] * fac));
    if (c == 0 && lse_row) lse_row[h] = lse_h;
  }
}

// The same for a row of more than kMaxInKernelParts parts (only a plan
// without the merge kernel leaves one here): part by part from global
// memory with a running maximum.
__device__ __noinline__ void combine_global(const DecodeArgs& a, int row, int hb, int nh, int64_t P, int32_t nt,
                                            int64_t ca, int64_t cz, int64_t T, int64_t G, int t, int nthreads) {
  const int H = a.heads;
  const float* const o_part = a.o_part;
  const float2* const ml_part = reinterpret_cast<const float2*>(a.ml_part);
  uint16_t* const out_row = a.out + int64_t(row) * a.out_stride_row;
  const int64_t osh = a.out_stride_head;
  float* const lse_row = a.lse ? a.lse + int64_t(row) * H : nullptr;
  const float* const sink = a.sink;
#pragma unroll 1
  for (int u = t; u < nh * 32; u += nthreads) {
    const int hh = u / 32, c = u % 32, h = hb + hh;
    float mrun = -INFINITY, lsum = 0.f;
    float acc[16];
#pragma unroll
    for (int d = 0; d < 16; ++d) acc[d] = 0.f;
#pragma unroll 1
    for (int64_t cc = ca; cc <= cz; ++cc) {
      if (!holds(cc, P, nt, T, G)) continue;
      const int64_t sl = slot_of(cc, P, T, G);
      const float2 mj = __ldcg(ml_part + sl * H + h);
      if (mj.y == 0.f) continue;
      if (mj.x > mrun) {  // the running maximum moves: rescale what was summed
        const float r = ex2(mrun - mj.x);
        lsum *= r;
#pragma unroll
        for (int d = 0; d < 16; ++d) acc[d] *= r;
        mrun = mj.x;
      }
      const float wt = ex2(mj.x - mrun);
      lsum = fmaf(mj.y, wt, lsum);
      const float* src = o_part + (sl * H + h) * kLatent + 4 * c;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + 128 * e));
        acc[4 * e] = fmaf(wt, v.x, acc[4 * e]);
        acc[4 * e + 1] = fmaf(wt, v.y, acc[4 * e + 1]);
        acc[4 * e + 2] = fmaf(wt, v.z, acc[4 * e + 2]);
        acc[4 * e + 3] = fmaf(wt, v.w, acc[4 * e + 3]);
      }
    }
    float fac, lse_h;
    finish_head(mrun, lsum, sink, h, &fac, &lse_h);
    uint16_t* dst = out_row + int64_t(h) * osh + 4 * c;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint2*>(dst + 128 * e) = make_uint2(pack_bf16x2(acc[4 * e] * fac, acc[4 * e + 1] * fac),
                                                            pack_bf16x2(acc[4 * e + 2] * fac, acc[4 * e + 3] * fac));
    if (c == 0 && lse_row) lse_row[h] = lse_h;
  }
}

// The CTA's final part completes a shared row whose other parts had all
// arrived when its last tile began: their O rows were then bulk-copied into
// the stage freed by the previous tile and their (m, l) and counts loaded
// (staging descriptors 1 .. parts - 1, see the aux loop).  Here (aux warps)
// this part's O goes from TMEM to the other stage (descriptor 0) with its
// (m, l), no partial of this part is written, and the row is queued for the
// CTA's end, where all threads combine it.
template <int HP>
__device__ __noinline__ void aux_stage_final(const AuxCtx& x, const Cursor<Cfg<HP>::kRowStart>& pc, int ob, int xi,
                                             int s_own, int kind) {
  using C = Cfg<HP>;
  Misc* ms = x.ms;
  uint64_t* bars = x.bars;
  const uint32_t tmem = x.tmem, lane_base = x.lane_base;
  const int Hl = x.Hl, lane = x.lane, ta = x.ta;
  float* ow = reinterpret_cast<float*>(x.smem + s_own * kStageBytes);  // this part's O [Hl][512]
  // this part's O^T rows: dim 128 b + ta of every block b
#pragma unroll 1
  for (int k = 0; k < 4 * C::kPass; ++k) {
    const int b = k / C::kPass, pass = k % C::kPass;
    uint32_t v0[16], v1[16];
    tmem_ld16(tmem + lane_base + C::o_col(ob, b) + 32 * pass, v0);       // hi
    tmem_ld16(tmem + lane_base + C::o_col(ob, b) + 32 * pass + 16, v1);  // lo
    tmem_wait_ld();
    const int hn = min(16, Hl - 16 * pass);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < hn) ow[(16 * pass + j) * kLatent + 128 * b + ta] = __uint_as_float(v0[j]) + __uint_as_float(v1[j]);
  }
  if (ta < Hl) ms->cb_ml[0][ta] = make_float2(ms->part_m[ob][ta], ms->part_l[ob][ta]);
  if (ta == 0) {
    ms->cb_row[0] = uint32_t(s_own * kStageBytes);
    const int k = ms->n_merge++;
    ms->merge_row[k] = pc.row;
    ms->merge_x[k] = xi;
    ms->merge_kind[k] = kind;
    ms->merge_own_nv = ms->part_nv[ob];
    ms->merge_own_slot = slot_of(x.c_id, pc.P, x.T, x.G);
  }
  tc_fence_before();
  named_barrier(2, 128);  // every aux thread read its O and (m, l)
  if (lane == 0) mbar_arrive(bars + kOEmpty + ob);
#ifdef SMLA_TRACE
  if (ta == 0) ms->merge_t[5] = globaltimer();
#endif
}

// A row part's epilogue (aux warps): out and lse of a whole row, or the
// part's partial (O, m, l, count) of a shared row and its ticket; the part
// that completes a row queues the row for the merge at the CTA's end.  The
// CTA's final part of a shared row whose other parts have all finished
// (their tickets are in, read before the waits) merges the row right here.
template <int HP>
__device__ __noinline__ void aux_epilogue(const AuxCtx& x, const Cursor<Cfg<HP>::kRowStart>& pc, int pi, bool final_part) {
  using C = Cfg<HP>;
  const DecodeArgs& a = *x.a;
  Misc* ms = x.ms;
  uint64_t* bars = x.bars;
  const uint32_t tmem = x.tmem, lane_base = x.lane_base;
  const int H = x.H, h0 = x.h0, Hl = x.Hl, lane = x.lane, ta = x.ta;
  const int64_t T = x.T, G = x.G;
  const int ob = pi % C::kNO;
  const uint32_t ph = (pi / C::kNO) & 1;
  const int row = pc.row;
  const bool whole = pc.whole();
  const int xi = pi == 0 ? 0 : 1;  // a shared row is this CTA's first or last one
  const int32_t parts = whole ? 1 : ms->mparts[xi];
  const int rows_bytes = Hl * kLatent * 4;
  // The final part of a shared row whose other parts have arrived by now
  // (tickets read before the waits) completes the row without a partial:
  // the stages are free once its last PV has completed, so the other parts'
  // O rows are bulk-copied into stage 0 and this part's O goes to stage 1.
  const bool may_late = final_part && !whole && !ms->fast && parts >= 2 && parts <= kMaxInKernelParts &&
                        (parts - 1) * rows_bytes <= kStageBytes;
  int32_t tk = -1;
  if (may_late && ta == 0) tk = ld_acquire_gpu(a.ticket + int64_t(row) * x.hg + x.g);
  wait_warp(bars + kEpiReady + ob, ph, ms, a);
  wait_warp(bars + kOFull + ob, ph, ms, a);
  tc_fence_after();
#ifdef SMLA_TRACE
  if (final_part && ta == 0) ms->merge_t[4] = globaltimer();
#endif
  if (final_part && ms->fast) {  // (decided when the part's last tile began)
    aux_stage_final<HP>(x, pc, ob, xi, ms->fast_s_own, 1);
    return;
  }
  if (may_late) {
    // (a field of its own: the aux warps leave their waits at different times,
    // and ms->fast is read after them above)
    if (ta == 0) {
      ms->late = tk == parts - 1;
      if (ms->late) {
        fence_proxy_async_global();  // (the other parts' partials are read by the async proxy)
        mbar_arrive_expect_tx(bars + kMerge, uint32_t((parts - 1) * rows_bytes));
        const int64_t own = slot_of(x.c_id, pc.P, T, G);
        int jj = 0;
        for (int j = 0; j < parts; ++j) {
          const int64_t sl = ms->mslot[xi][j];
          if (sl == own || jj >= parts - 1) continue;
          ms->cb_row[1 + jj] = uint32_t(jj * rows_bytes);
          bulk_g2s(smem_u32(x.smem + jj * rows_bytes), a.o_part + (sl * H + h0) * kLatent, uint32_t(rows_bytes),
                   bars + kMerge);
          ++jj;
        }
      }
    }
    named_barrier(2, 128);
    if (ms->late) {  // (the other parts' (m, l) and counts are loaded at the end merge)
      aux_stage_final<HP>(x, pc, ob, xi, 1, 2);
      return;
    }
  }
  const int64_t slot = whole ? 0 : slot_of(x.c_id, pc.P, T, G);
  // head ta's output factor and LSE (whole rows), or its partial (m, l)
  if (ta < Hl) {
    const float m = ms->part_m[ob][ta], l = ms->part_l[ob][ta];
    if (whole) {
      float f, lse_h;
      finish_head(m, l, a.sink, h0 + ta, &f, &lse_h);
      ms->fac[ta] = f;
      if (a.lse) a.lse[int64_t(row) * H + h0 + ta] = lse_h;
    } else {
      reinterpret_cast<float2*>(a.ml_part)[slot * H + h0 + ta] = make_float2(m, l);
    }
  }
  if (ta == 0) {
    if (whole) {
      if (a.n_valid && x.g == 0) a.n_valid[row] = ms->part_nv[ob];
    } else {
      a.nv_part[slot] = ms->part_nv[ob];  // the same count from either head group
    }
  }
  named_barrier(2, 128);  // the factors
  // (the arguments' fields in registers: read through the reference they would
  // be reloaded from the parameter buffer after every store)
  uint16_t* const out_rows = a.out + int64_t(row) * a.out_stride_row + int64_t(h0) * a.out_stride_head;
  const int64_t osh = a.out_stride_head;
  float* const o_rows = a.o_part + (slot * H + h0) * kLatent;
  // O^T rows of this thread: dim 128 b + ta of every block b; columns
  // [hi g | lo g] per 16-head group g
#pragma unroll 1
  for (int k = 0; k < 4 * C::kPass; ++k) {
    const int b = k / C::kPass, pass = k % C::kPass;
    const int d = 128 * b + ta;
    uint32_t v0[16], v1[16];
    tmem_ld16(tmem + lane_base + C::o_col(ob, b) + 32 * pass, v0);       // hi
    tmem_ld16(tmem + lane_base + C::o_col(ob, b) + 32 * pass + 16, v1);  // lo
    tmem_wait_ld();
    const int hn = min(16, Hl - 16 * pass);
    if (whole) {
      uint16_t* dst = out_rows + int64_t(16 * pass) * osh + d;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < hn)
          dst[int64_t(j) * osh] = __bfloat16_as_ushort(
              __float2bfloat16_rn((__uint_as_float(v0[j]) + __uint_as_float(v1[j])) * ms->fac[16 * pass + j]));
    } else {
      float* dst = o_rows + (16 * pass) * kLatent + d;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < hn) dst[int64_t(j) * kLatent] = __uint_as_float(v0[j]) + __uint_as_float(v1[j]);
    }
  }
  tc_fence_before();
  named_barrier(2, 128);  // every aux thread read the part's (m, l) and O
  // the O buffer is free for the next part's PV now, before the partial's fence
  if (lane == 0) mbar_arrive(bars + kOEmpty + ob);
  if (!whole) {
    __threadfence();        // the partial is visible device-wide before the ticket below
    named_barrier(2, 128);  // (every aux thread's part of it)
  }
  if (!whole && ta == 0) {
    // the CTAs holding this row's tiles ([P2] stage_split parts); the one whose
    // part arrives last merges the row (this head group) after its own work
    if (parts <= kMaxInKernelParts || !a.merge_kernel) {
      if (atomicAdd(a.ticket + int64_t(row) * x.hg + x.g, 1) == parts - 1) {
        __threadfence();  // (acquire: the other parts' partials are read after this)
        const int k = ms->n_merge++;
        ms->merge_row[k] = row;
        ms->merge_x[k] = xi;
        ms->merge_kind[k] = 0;
      }
    }
  }
}

// [P2] stage_combine, with the sink, of the rows this CTA completed through
// its tickets: every part's (m, l) and O, out and lse of heads [h0, h0 + Hl),
// the key count, and the row's ticket back to zero.  All threads of the CTA,
// after its own work (the stages' shared memory is free then).  The parts'
// slots were found after the prologue.  For rows of up to kMaxInKernelParts
// parts, one thread bulk-copies each part's O rows of 16 heads (32 KB) into
// shared memory (a plain-load gather of the same bytes is limited by the
// SM's load throughput) while the threads load the (m, l); then the staged
// combine.  Warp k loads row k's key counts first and sums them last.
static_assert(kMaxInKernelParts * 16 * kLatent * 4 <= kStages * kStageBytes, "merge staging fits the stages");
__device__ __noinline__ void end_merge(const DecodeArgs& a, uint8_t* smem, uint64_t* bar, Misc* ms, int tid,
                                       int h0, int Hl, int hg, int g, int64_t T, int64_t G) {
  const int H = a.heads;
  const int n_merge = ms->n_merge;
  const int warp = tid >> 5, lane = tid & 31;
  int32_t nv = 0;  // warp k < n_merge: key counts of row k's parts of this lane
  if (warp < n_merge) {
    const int xi = ms->merge_x[warp];
    const int parts = ms->mparts[xi];
    if (ms->merge_kind[warp] == 1) {  // counts loaded when the row was staged
      if (lane == 0) nv = ms->merge_own_nv;
      if (lane >= 1 && lane < parts) nv = ms->fnv[lane - 1];
    } else if (ms->merge_kind[warp] == 2) {  // this part's count, the others' from their slots
      if (lane == 0) nv = ms->merge_own_nv;
      if (lane < parts && ms->mslot[xi][lane] != ms->merge_own_slot) nv += __ldcg(a.nv_part + ms->mslot[xi][lane]);
    } else if (parts <= kMaxInKernelParts) {
      if (lane < parts) nv = __ldcg(a.nv_part + ms->mslot[xi][lane]);
    } else {
      const int64_t ca = ms->mca[xi], cz = ms->mcz[xi], P = ms->mP[xi];
      const int32_t nt = ms->mnt[xi];
      for (int64_t cc = ca + lane; cc <= cz; cc += 32)
        if (holds(cc, P, nt, T, G)) nv += __ldcg(a.nv_part + slot_of(cc, P, T, G));
    }
  }
#ifdef SMLA_TRACE
  if (tid == 0) ms->merge_t[0] = globaltimer();
#endif
  uint32_t uses = 0;  // completed phases of `bar`
  // the row staged by the final part first (its bulk copies are the barrier's
  // first phase, and the other merges reuse its shared memory)
#pragma unroll 1
  for (int k = 0; k < n_merge; ++k) {
    if (ms->merge_kind[k] == 0) continue;
    if (ms->merge_kind[k] == 2) {
      // the other parts' (m, l), in the order of their bulk copies
      const int xi = ms->merge_x[k], parts = ms->mparts[xi];
      if (tid < Hl) {
        int jj = 0;
        for (int j = 0; j < parts; ++j) {
          const int64_t sl = ms->mslot[xi][j];
          if (sl == ms->merge_own_slot || jj >= parts - 1) continue;
          ms->cb_ml[1 + jj][tid] = __ldcg(reinterpret_cast<const float2*>(a.ml_part) + sl * H + h0 + tid);
          ++jj;
        }
      }
      __syncthreads();
    }
    if (!mbar_wait(bar, 0, kWaitLimitNs)) set_abort(ms, a.status);
    uses = 1;
#ifdef SMLA_TRACE
    if (tid == 0) ms->merge_t[1] = globaltimer();
#endif
    combine_staged(a, smem, ms, ms->mparts[ms->merge_x[k]], ms->merge_row[k], h0, Hl, tid, kThreads);
#ifdef SMLA_TRACE
    if (tid == 0) ms->merge_t[2] = globaltimer();
#endif
  }
#pragma unroll 1
  for (int k = 0; k < n_merge; ++k) {
    if (ms->merge_kind[k] != 0) continue;
    const int row = ms->merge_row[k];
    const int xi = ms->merge_x[k];
    const int parts = ms->mparts[xi];
    if (parts > kMaxInKernelParts) {
      combine_global(a, row, h0, Hl, ms->mP[xi], ms->mnt[xi], ms->mca[xi], ms->mcz[xi], T, G, tid, kThreads);
      continue;
    }
#pragma unroll 1
    for (int hc = 0; hc < Hl; hc += 16) {  // 16 heads at a time
      const int nh = min(16, Hl - hc);
      __syncthreads();  // the staging buffer and descriptors are free
      if (tid == 0) {
        fence_proxy_async_global();  // (partials are read by the async proxy)
        mbar_arrive_expect_tx(bar, uint32_t(parts * nh * kLatent * 4));
        for (int j = 0; j < parts; ++j) {
          ms->cb_row[j] = uint32_t(j * (16 * kLatent * 4));
          bulk_g2s(smem_u32(smem + j * (16 * kLatent * 4)), a.o_part + (ms->mslot[xi][j] * H + h0 + hc) * kLatent,
                   uint32_t(nh * kLatent * 4), bar);
        }
      }
      if (tid < parts * nh) {
        const int j = tid / nh, hh = tid % nh;
        ms->cb_ml[j][hh] = __ldcg(reinterpret_cast<const float2*>(a.ml_part) + ms->mslot[xi][j] * H + h0 + hc + hh);
      }
      __syncthreads();
      if (!mbar_wait(bar, uses & 1, kWaitLimitNs)) set_abort(ms, a.status);
      ++uses;
      combine_staged(a, smem, ms, parts, row, h0 + hc, nh, tid, kThreads);
    }
  }
#ifdef SMLA_TRACE
  if (tid == 0) ms->merge_t[3] = globaltimer();
#endif
  // key counts and tickets (warp k: row k)
  if (warp < n_merge) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
    if (lane == 0) {
      const int row = ms->merge_row[warp];
      if (g == 0 && a.n_valid) a.n_valid[row] = nv;
      a.ticket[int64_t(row) * hg + g] = 0;  // ready for the next call
    }
  }
}

// Shared-memory offset of the P' block (32-key chunk ch, dim block b) of the
// tile in stage s: the first kPInRope blocks sit in the stage's rope rows,
// the rest (32 heads) in the extra buffer both stages share.
template <int HP>
__device__ __forceinline__ uint32_t p_block_off(int s, int ch, int b) {
  using C = Cfg<HP>;
  const int k = 4 * ch + b;
  return k < C::kPInRope ? uint32_t(s * kStageBytes + kOffRope + k * C::kPBlock)
                         : uint32_t(C::kOffPx + (k - C::kPInRope) * C::kPBlock);
}

// This thread's key of the tile in stage st: whether it is valid, its four
// block scales, and (into grp's buffer rb) the largest biased exponent of
// each block's scale over the warp's valid keys.
__device__ __forceinline__ bool tile_key(const uint8_t* st, int t, int lane, int q, int grp, int rb, Misc* ms,
                                         uint32_t (&sw)[4]) {
  const int32_t id = *reinterpret_cast<const int32_t*>(st + kOffIds + 4 * t);
  const bool valid = id >= 0;
  const uint4 scw = *reinterpret_cast<const uint4*>(st + kOffSc + 16 * t);
  sw[0] = scw.x;
  sw[1] = scw.y;
  sw[2] = scw.z;
  sw[3] = scw.w;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int32_t e = __reduce_max_sync(0xffffffffu, valid ? int32_t((sw[b] >> 23) & 0xFF) : 0);
    if (lane == b) ms->red_sc[grp][rb][q][b] = e;
  }
  return valid;
}

// What one softmax pass of a tile needs (per thread; in registers).
struct PassCtx {
  const DecodeArgs* a;
  uint8_t* smem;
  Misc* ms;
  uint64_t* bars;
  uint32_t tmem, lane_base;
  int q, lane, i, s, sb, rb, ob;
  bool first, valid, p_shared;
  uint32_t sw[4];             // the key's four block scales (f32 bits)
  int grp;                    // 0: softmax warps, 1: aux warps (own scale-exponent buffer)
  uint32_t bar_id;            // the group's named barrier (its four warps)
  int first_pass, last_pass;  // the group's passes
#ifdef SMLA_TRACE
  unsigned long long* tr_buf;
  int* tr_k;
#endif
};

// One 16-head pass (heads 16 pass .. 16 pass + 15) of a tile's softmax for this
// thread's key row: scores from S, the heads' tile maxima across the group's
// four lane quarters, the lazy reference update (rescaling O in TMEM), p and
// its sum, and the P' blocks and their scale factors for the PV.  Run by the
// softmax warps (every pass at 16 heads, pass 0 at 32) and at 32 heads by the
// aux warps (pass 1).
template <int HP>
__device__ __forceinline__ void softmax_pass(const PassCtx& z, const int pass, float& mref, float& lsum,
                                             bool& pv_waited, int (&es)[4]) {
  using C = Cfg<HP>;
  constexpr int kN = C::kN;
  const DecodeArgs& a = *z.a;
  uint8_t* const smem = z.smem;
  Misc* const ms = z.ms;
  uint64_t* const bars = z.bars;
  const uint32_t tmem = z.tmem, lane_base = z.lane_base;
  const int q = z.q, lane = z.lane, i = z.i, s = z.s, sb = z.sb, rb = z.rb, ob = z.ob;
  const bool first = z.first, valid = z.valid, p_shared = z.p_shared;
  const int hl = lane & 15;         // per-head values: lane hl (and hl + 16) holds head 16 pass + hl
  const int hs = (lane >> 1) & 15;  // head (of the pass) of this lane's sum of p (see sum16)
  const uint32_t sw[4] = {z.sw[0], z.sw[1], z.sw[2], z.sw[3]};
#ifdef SMLA_TRACE
  unsigned long long* const tr_buf = z.tr_buf;
  int& tr_k = *z.tr_k;
#endif
  // scores x = (S_hi + S_lo) sm_scale log2(e) of heads 16 pass .. + 15, -inf when masked
  float x[16];
  {
    const float xs = a.sm_scale_log2;
#pragma unroll
    for (int h = 0; h < 16; ++h) x[h] = 0.f;
#pragma unroll 1
    for (int acc = 0; acc < C::kQkSplit; ++acc) {
      // accumulator acc: q_hi columns (+ rope) and q_lo columns, one wait
      uint32_t r0[16], r1[16];
      tmem_ld16(tmem + lane_base + C::s_col(sb, acc) + 16 * pass, r0);
      tmem_ld16(tmem + lane_base + C::s_col(sb, acc) + HP + 16 * pass, r1);
      tmem_wait_ld();
#pragma unroll
      for (int h = 0; h < 16; ++h) x[h] += __uint_as_float(r0[h]) + __uint_as_float(r1[h]);
    }
#pragma unroll
    for (int h = 0; h < 16; ++h) x[h] = valid ? x[h] * xs : -INFINITY;
  }
  if (pass == z.last_pass) {  // the group's last S columns of the tile
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kSEmpty + sb);  // S read
  }
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    const int32_t m = __reduce_max_sync(0xffffffffu, ord(x[h]));
    if (lane == h) ms->red_max_t[rb][16 * pass + h][q] = m;
  }
  named_barrier(z.bar_id, 128);
  if (pass == z.first_pass) F8_TR(11, i);
  // the tile's maximum of head 16 pass + hl over the four lane quarters
  float tm;
  {
    const uint4 m4 = ld_shared_v4(smem_u32(&ms->red_max_t[rb][16 * pass + hl][0]));
    tm = unord(max(max(int32_t(m4.x), int32_t(m4.y)), max(int32_t(m4.z), int32_t(m4.w))));
  }
  float mr = mref;
  if (first) {
    mr = (tm > kInitMax || tm != tm) ? tm : kInitMax;
  } else if (__any_sync(0xffffffffu, tm > mr + kLazy)) {  // the same in all four warps
    // heads whose reference moves (lanes hl and hl + 16 hold the same head)
    const uint32_t moved = __ballot_sync(0xffffffffu, tm > mr + kLazy) & 0xFFFFu;
    const float mn = tm > mr + kLazy ? tm : mr;
    const float alpha = ex2(mr - mn);  // exactly 1 for the heads that keep theirs
    mr = mn;
    lsum *= __shfl_sync(0xffffffffu, alpha, hs);
    // O holds PV of this part's earlier tiles: wait until they completed,
    // then rescale the moved heads' hi and lo columns in this lane quarter
    if (!pv_waited) {
      wait_warp(bars + kPvDone, (i - 1) & 1, ms, a);
      pv_waited = true;
    }
    tc_fence_after();
    const uint32_t ob_col = tmem + lane_base + C::o_col(ob, 0) + uint32_t(32 * pass);
    if (__popc(moved) > 4) {  // many heads: 16 columns at a time
      float al[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) al[h] = __shfl_sync(0xffffffffu, alpha, h);
#pragma unroll 1
      for (int k = 0; k < 8; ++k) {  // 4 blocks x (hi, lo)
        const uint32_t ta = ob_col + uint32_t(k >> 1) * kN + uint32_t(16 * (k & 1));
        uint32_t v[16];
        tmem_ld16(ta, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * al[h]);
        tmem_st16(ta, v);
      }
    } else {  // a few heads (the usual case once a row's maxima settle): their 8 columns each
      uint32_t mv = moved;
#pragma unroll 1
      while (mv != 0u) {
        const int h = __ffs(mv) - 1;
        mv &= mv - 1u;
        const float al_h = __shfl_sync(0xffffffffu, alpha, h);
        uint32_t v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) tmem_ld1(ob_col + uint32_t(k >> 1) * kN + uint32_t(16 * (k & 1) + h), v[k]);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tmem_st1(ob_col + uint32_t(k >> 1) * kN + uint32_t(16 * (k & 1) + h),
                   __float_as_uint(__uint_as_float(v[k]) * al_h));
      }
    }
    tmem_wait_st();
  }
  mref = mr;
  if (pass == z.first_pass) {
    // the shared extra P' buffer was last read by PV(i - 1)
    if (p_shared && i > 0 && !pv_waited) {
      wait_warp(bars + kPvDone, (i - 1) & 1, ms, a);
      pv_waited = true;
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int32_t e = max(max(ms->red_sc[z.grp][rb][0][b], ms->red_sc[z.grp][rb][1][b]),
                            max(ms->red_sc[z.grp][rb][2][b], ms->red_sc[z.grp][rb][3][b]));
      es[b] = max(e, 1) - 126;
    }
  }
  // p = 2^(x - mref).  P'_b = p * scale_b in units of the E8M0 factor
  // 2^E(h, b), E = e_h - 7 + (the tile's largest block-b scale exponent),
  // where pmax_h = 2^(tmax_h - mref_h) < 2^e_h: P'_b < 2^7.  It is formed
  // as p'' = p 2^(7 - e_h) split once into E4M3 hi + lo codes, then, per
  // block, the codes' exponent fields lowered by the key's distance m_b
  // to the tile's largest block-b scale (exact for the writer's power-of-
  // two scales; a value leaving E4M3's normal range becomes 0).  e_h is
  // kept in [-20, kLazy + 1] (a head whose tile terms all lie 2^20 below
  // its reference keeps 2^-10 relative precision on them).
  if (pass == z.first_pass) F8_TR(13, i);
  const int e_h = max(min(int((__float_as_uint(ex2(tm - mr)) >> 23) & 0xFF) - 126, int(kLazy) + 1), -20);
  const float inv_h = pow2f(7 - e_h);
#pragma unroll
  for (int h = 0; h < 16; ++h) x[h] = ex2(x[h] - __shfl_sync(0xffffffffu, mr, h));  // x = -inf (masked) gives 0
  lsum += sum16(x, lane);
  if (pass == z.first_pass) F8_TR(14, i);
  uint32_t hw0[4], lw0[4];  // codes of heads 4k .. 4k + 3
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint16_t h0_, l0_, h1_, l1_;
    const __half2 y0 = __floats2half2_rn(x[4 * k] * __shfl_sync(0xffffffffu, inv_h, 4 * k),
                                         x[4 * k + 1] * __shfl_sync(0xffffffffu, inv_h, 4 * k + 1));
    const __half2 y1 = __floats2half2_rn(x[4 * k + 2] * __shfl_sync(0xffffffffu, inv_h, 4 * k + 2),
                                         x[4 * k + 3] * __shfl_sync(0xffffffffu, inv_h, 4 * k + 3));
    split_h2(*reinterpret_cast<const uint32_t*>(&y0), h0_, l0_);
    split_h2(*reinterpret_cast<const uint32_t*>(&y1), h1_, l1_);
    hw0[k] = uint32_t(h0_) | (uint32_t(h1_) << 16);
    lw0[k] = uint32_t(l0_) | (uint32_t(l1_) << 16);
  }
  if (pass == z.first_pass) F8_TR(15, i);
#pragma unroll 1
  for (int b = 0; b < 4; ++b) {
    // (selects, not indexing: a rolled loop would put sw and es in local memory)
    const uint32_t swb = b == 0 ? sw[0] : b == 1 ? sw[1] : b == 2 ? sw[2] : sw[3];
    const int esb = b == 0 ? es[0] : b == 1 ? es[1] : b == 2 ? es[2] : es[3];
    const int bexp = int((swb >> 23) & 0xFF);  // a zero (or f32-subnormal) scale gives 0
    const int m = bexp == 0 ? 16 : min(max(esb + 126 - bexp, 0), 16);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      hw[k] = lower_codes(hw0[k], m);
      lw[k] = lower_codes(lw0[k], m);
    }
    // MN-major P' row of this key: [hi g0 | lo g0 | hi g1 | lo g1], 16 bytes each
    uint8_t* blk = smem + p_block_off<HP>(s, q, b);
    uint32_t off0 = uint32_t(lane) * kN + uint32_t(32 * pass), off1 = off0 + 16;
    off0 ^= ((off0 >> 7) & C::kPSwMask) << 4;
    off1 ^= ((off1 >> 7) & C::kPSwMask) << 4;
    *reinterpret_cast<uint4*>(blk + off0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(blk + off1) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  // P' scale factors of this tile's stage: row group g of B holds head
  // group g (hi rows then lo rows), byte b the factor of dim block b;
  // the same in every TMEM lane quarter (each warp writes its own)
  if (pass == z.first_pass) F8_TR(16, i);
  uint32_t word = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) word |= uint32_t(min(max(e_h + es[b] - 8 + 127, 1), 254)) << (8 * b);
  tmem_st1(tmem + lane_base + C::sfp_col(s) + uint32_t(pass), word);
}

template <int HP>
__global__ void __launch_bounds__(kThreads, 1) decode_fp8_kernel(const __grid_constant__ DecodeArgs a) {
  using C = Cfg<HP>;
  using Cur = Cursor<C::kRowStart>;
  constexpr int kN = C::kN;
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#ifdef SMLA_TRACE
  unsigned long long* const tr_buf = g_smla_trace_fp8;
  int tr_k = 0;
#endif
  F8_TR(1, 0);
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  Misc* ms = reinterpret_cast<Misc*>(smem + C::kOffMisc);
  const int H = a.heads;
  // head groups: CTAs 2 c and 2 c + 1 of a two-group launch take the same
  // schedule range c, heads [0, HP) and [HP, 2 HP)
  const int hg = a.head_groups;
  const int g = int(blockIdx.x) % hg;
  const int64_t G = gridDim.x / hg, c_id = blockIdx.x / hg;
  const int h0 = g * HP;
  const int Hl = min(HP, H - h0);  // heads of this group
  {
    // the schedule scan's row lengths into L2 while the barriers are set up
    // (the scan's loads then meet no DRAM latency; decode_64x16 49.4 -> 48.0 us)
    const int per = (a.n_q + kThreads - 1) / kThreads, lo = tid * per;
    if (lo < a.n_q) {
      prefetch_l2_line(a.indptr + lo);
      if (a.lens) prefetch_l2_line(a.lens + lo);
    }
  }

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bars + kKvFull + s, kLoadWarps);
      mbar_init(bars + kKvEmpty + s, kSoftmaxWarps);  // the four PV issuers
      mbar_init(bars + kSFull + s, Cfg<HP>::kQkSplit);  // [S buffer] (one or two used)
      mbar_init(bars + kSEmpty + s, Cfg<HP>::kSReaders);
      mbar_init(bars + kQEmpty + s, Cfg<HP>::kQkSplit);
      mbar_init(bars + kOFull + s, kSoftmaxWarps);
      mbar_init(bars + kOEmpty + s, 4);
      mbar_init(bars + kEpiReady + s, Cfg<HP>::kSReaders);
      mbar_init(bars + kPReady + s, kSoftmaxWarps);
      if (s == 0) mbar_init(bars + kQReady, kLoadWarps);
    }
    mbar_init(bars + kPvDone, kSoftmaxWarps);
    mbar_init(bars + kDrain, Cfg<HP>::kQkSplit + kSoftmaxWarps);
    mbar_init(bars + kStall, 1);
    mbar_init(bars + kMerge, 1);
    ms->stall = g_fp8_stall;
    ms->abort = 0;
    const uint64_t w = g_fp8_wait_ns;
    ms->wait_ns = w != 0 ? w : kWaitLimitNs;
    ms->first_row = a.n_q;
    ms->first_tile = 0;
    ms->last_row = a.n_q;
    ms->last_tile = 0;
    ms->mparts[0] = ms->mparts[1] = 0;
    ms->fast = 0;
    ms->fast_s_own = 0;
    ms->late = 0;
#ifdef SMLA_TRACE
    for (int k = 0; k < 8; ++k) ms->merge_t[k] = 0;
#endif
    ms->n_tiles = 0;
    ms->n_merge = 0;
    fence_mbar_init();
  }
  if (warp == kAuxWarp0) {
    tmem_alloc(&ms->tmem_base, 512);
    tmem_relinquish();
  }
  // zeroed staging descriptors (read by the softmax warps' early combine run)
  static_assert(kMaxInKernelParts * kMaxHP <= kThreads, "one descriptor entry per thread");
  if (tid < kMaxInKernelParts * kMaxHP) ms->cb_ml[tid / kMaxHP][tid % kMaxHP] = make_float2(0.f, 0.f);
  if (tid < kMaxInKernelParts) ms->cb_row[tid] = 0;
  F8_TR(6, 0);

  // ---- schedule: slot counts of all rows, their prefix, this CTA's first row
  {
    const int n = a.n_q;
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min(tid * per, n), hi = min(lo + per, n);
    int64_t local = 0;
#pragma unroll 1
    for (int r = lo; r < hi; ++r) local += C::kRowStart + kTileSlots * Cur::tiles_of(row_len(a, r));
    int64_t x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) ms->scan[warp] = x;
    __syncthreads();
    F8_TR(7, 0);
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
    F8_TR(8, 0);
    const int64_t Tt = ms->total_tiles;
    const int64_t b = cbeg(c_id, Tt, G), e = cbeg(c_id + 1, Tt, G);
    int64_t P = ms->scan[32 + warp] + x - local;
    int32_t mine = 0;
#pragma unroll 1
    for (int r = lo; r < hi; ++r) {
      const int32_t nt_r = Cur::tiles_of(row_len(a, r));
      const int64_t w = C::kRowStart + int64_t(kTileSlots) * nt_r;
      const int64_t F = P + C::kRowStart;                   // the row's first tile slot
      const int64_t L = F + int64_t(kTileSlots) * (nt_r - 1);  // and its last one
      // the row of this CTA's first tile: the first row whose last tile is
      // at or after b (the previous row's last tile slot is P - kTileSlots)
      if (L >= b && P - kTileSlots < b) {
        ms->first_row = r;
        ms->first_tile = P;
      }
      // the row of its last tile: the row whose first tile is before e and
      // the next row's first tile not
      if (F < e && P + w + C::kRowStart >= e) {
        ms->last_row = r;
        ms->last_tile = P;
      }
      int32_t lo_t, hi_t;
      tiles_in(F, nt_r, b, e, lo_t, hi_t);
      if (hi_t > lo_t) mine += hi_t - lo_t;
      if (blockIdx.x == 0 && a.row_tile) a.row_tile[r] = P;
      P += w;
    }
    if (blockIdx.x == 0 && tid == 0 && a.row_tile) a.row_tile[n] = Tt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (lane == 0 && mine != 0) atomicAdd(&ms->n_tiles, mine);
    F8_TR(9, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int64_t T = ms->total_tiles;
  const int64_t cb = cbeg(c_id, T, G), ce = cbeg(c_id + 1, T, G);
  const int32_t n_tiles = ms->n_tiles;
  const int32_t row0 = ms->first_row;
  const int64_t P0 = ms->first_tile;
  const uint32_t tmem = ms->tmem_base;
  const uint32_t smem_base = smem_u32(smem);
  F8_TR(2, 0);

  if (warp < kSoftmaxWarps) {
    // =================== softmax ===================
    const int q = warp;              // TMEM lane quarter: keys 32 q .. 32 q + 31 of a tile
    const int t = 32 * q + lane;     // this thread's key row of the tile
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    // the P' blocks of this warp's keys live in the shared extra buffer (32 heads, chunks 2, 3)
    const bool p_shared = 4 * q >= C::kPInRope;
    const int hs = (lane >> 1) & 15;  // head (of a pass) of this lane's sum of p (see sum16)
    float mref[C::kPass];  // reference max of head 16 pass + (lane & 15)
    float lsum[C::kPass];  // sum of p of head 16 pass + hs over this warp's keys of the part
    int nv = 0;
#pragma unroll
    for (int p = 0; p < C::kPass; ++p) {
      mref[p] = kInitMax;
      lsum[p] = 0.f;
    }
    // The end merge's combine runs once per launch, at its end, when every
    // instruction fetch that misses waits behind the other CTAs' gathers: run
    // it now without its stores (on zeroed staging descriptors) while the
    // first tiles are in flight, so that its code is in the caches then
    if (n_tiles > 0) combine_staged(a, smem, ms, kMaxInKernelParts, 0, 0, 4, t, 32 * kSoftmaxWarps, true);
    Cur c;
    c.init(a, row0, P0, cb, ce);
    int pi = 0;  // row part index within this CTA
    for (int i = 0; i < n_tiles; ++i, c.advance(a)) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const bool first = c.first(), last = c.last();
      const int ob = pi % C::kNO;
      const uint8_t* st = smem + s * kStageBytes;
      const int rb = i & 1;  // reduction buffer (a warp may run one tile ahead)
      if (first) {
#pragma unroll
        for (int p = 0; p < C::kPass; ++p) lsum[p] = 0.f;
        nv = 0;
      }
      if (i == 0 && ms->stall) wait_warp(bars + kStall, 0, ms, a);
      const int sb = i % C::kSBuf;                  // S buffer
      const uint32_t sph = (i / C::kSBuf) & 1;
      wait_warp(bars + kSFull + sb, sph, ms, a);
      wait_warp(bars + kKvFull + s, ph, ms, a);  // (already complete) orders the loaders' ids and scales
      F8_TR(10, i);
      tc_fence_after();
      PassCtx z;
      z.valid = tile_key(st, t, lane, q, 0, rb, ms, z.sw);
      nv += z.valid;
      z.a = &a;
      z.smem = smem;
      z.ms = ms;
      z.bars = bars;
      z.tmem = tmem;
      z.lane_base = lane_base;
      z.q = q;
      z.lane = lane;
      z.i = i;
      z.s = s;
      z.sb = sb;
      z.rb = rb;
      z.ob = ob;
      z.first = first;
      z.p_shared = p_shared;
      z.grp = 0;
      z.bar_id = 1;
      z.first_pass = 0;
      z.last_pass = C::kPassA - 1;
#ifdef SMLA_TRACE
      z.tr_buf = tr_buf;
      z.tr_k = &tr_k;
#endif
      bool pv_waited = false;
      int es[4];  // the tile's block-b scales < 2^es_b
#pragma unroll
      for (int pass = 0; pass < C::kPassA; ++pass) softmax_pass<HP>(z, pass, mref[pass], lsum[pass], pv_waited, es);
      tmem_wait_st();
      F8_TR(17, i);
      fence_proxy_async_smem();
      tc_fence_before();
      named_barrier(1, 32 * kSoftmaxWarps);  // the tile's P' and its scale factors are written
      // (32 heads: and the aux warps' heads 16..31)
      if constexpr (C::kSplitPass) wait_warp(bars + kPReady + s, ph, ms, a);
      F8_TR(12, i);
      {
        // PV of the tile: warp q issues dim block b = q (four MMA chains in
        // flight, one per O block)
        if (first) wait_warp(bars + kOEmpty + ob, ((pi / C::kNO) & 1) ^ 1, ms, a);
        tc_fence_after();
        F8_TR(60, i);
        if (lane == 0) {
          const uint32_t st32 = smem_base + s * kStageBytes;
          const int b = q;
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            // V^T: dims of block b (M, contiguous) x keys 32 ch .. (K, rows)
            const uint64_t ad = smem_desc(st32 + b * kChunk + ch * 4096, 16384, 1024, kSw128);
            const uint64_t bd = smem_desc(smem_base + p_block_off<HP>(s, ch, b), 8 * kN, 8 * kN, C::kPSw);
            mma_mxf8_ss(tmem + C::o_col(ob, b), ad, bd, idesc_mxf8(128, kN, 1, 1, 0, b), tmem + C::kColSfv,
                        tmem + C::sfp_col(s), (first && ch == 0) ? 0u : 1u);
          }
          mma_commit(bars + kPvDone);
          mma_commit(bars + kKvEmpty + s);
          if (last) mma_commit(bars + kOFull + ob);
        }
        __syncwarp();
        F8_TR(61, i);
      }
      if (last) {
        // the part's l and count over its keys, for the aux warps' epilogue
#pragma unroll
        for (int pass = 0; pass < C::kPassA; ++pass)
          if ((lane & 1) == 0) ms->red_l[q][16 * pass + hs] = lsum[pass];
        const int32_t nvw = __reduce_add_sync(0xffffffffu, nv);
        if (lane == 0) ms->red_nv[q] = nvw;
        // the (m, l) slot of this O buffer was read by the epilogue kNO parts ago
        wait_warp(bars + kOEmpty + ob, ((pi / C::kNO) & 1) ^ 1, ms, a);
        named_barrier(1, 32 * kSoftmaxWarps);
        if (q == 0) {
#pragma unroll
          for (int pass = 0; pass < C::kPassA; ++pass) {
            if (lane < 16) {
              const int h = 16 * pass + lane;
              ms->part_m[ob][h] = mref[pass];
              ms->part_l[ob][h] = ms->red_l[0][h] + ms->red_l[1][h] + ms->red_l[2][h] + ms->red_l[3][h];
            }
          }
          if (lane == 0) ms->part_nv[ob] = ms->red_nv[0] + ms->red_nv[1] + ms->red_nv[2] + ms->red_nv[3];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + kEpiReady + ob);
        ++pi;
      }
    }
    // the drain barrier completes once every MMA issued here has (the warp
    // that frees TMEM waits for it)
    if (lane == 0) mma_commit(bars + kDrain);
    __syncwarp();
  } else if (warp < kLoadWarp0) {
    // =================== aux: scale factors, q staging, epilogues ===================
    const int q = warp - kAuxWarp0;  // TMEM lane quarter
    const int ta = 32 * q + lane;    // 0..127
    const uint32_t lane_base = uint32_t(32 * q) << 16;
    const AuxCtx actx{&a, smem, ms, bars, tmem, lane_base, H, h0, Hl, hg, g, lane, ta, c_id, G, T};
    float mref_b = kInitMax;  // 32 heads: reference max of head 16 + (lane & 15)
    float lsum_b = 0.f;       //   and the sum of p of head 16 + ((lane >> 1) & 15) over the part's keys
    (void)mref_b;
    (void)lsum_b;
    // V^T scale factors: 1 (E8M0 127) for every dim row and key block
    {
      uint32_t v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = 0x7F7F7F7Fu;
      tmem_st16(tmem + lane_base + C::kColSfv, v);
      tmem_wait_st();
    }
    // q of a row -> [q_hi | q_lo] E4M3 (K-major, 128-byte swizzled) with an
    // E8M0 factor per (head, 32 dims) that brings the block's largest |q| to
    // [2^7, 2^8); q_rope (bf16) copied as it is; then the factors into TMEM.
    Cur c;
    c.init(a, row0, P0, cb, ce);
    if (n_tiles > 0) aux_stage_q<HP>(actx, c.row, 0, 128, 2, true);
    if (q < 2 && n_tiles > 0) {
      // the CTAs sharing this CTA's first (q = 0) and last (q = 1) row, for
      // a merge at the end (lane j looks at CTA ca + j; no waits, while the
      // first tile is still in flight)
      const int32_t r = q == 0 ? row0 : ms->last_row;
      if (r < a.n_q) {
        const int64_t Pr = (q == 0 ? P0 : ms->last_tile) + C::kRowStart;
        const int32_t nt = Cur::tiles_of(row_len(a, r));
        const int64_t ca = cof(Pr, T, G), cz = cof(Pr + int64_t(kTileSlots) * (nt - 1), T, G);
        int32_t n = 0;
        for (int64_t c0 = ca; c0 <= cz; c0 += 32) {
          const int64_t cc = c0 + lane;
          const bool in = cc <= cz && holds(cc, Pr, nt, T, G);
          const uint32_t m = __ballot_sync(0xffffffffu, in);
          const int j = n + __popc(m & ((1u << lane) - 1u));
          if (in && j < kMaxInKernelParts) ms->mslot[q][j] = slot_of(cc, Pr, T, G);
          n += __popc(m);
        }
        if (lane == 0) {
          ms->mparts[q] = n;
          ms->mP[q] = Pr;
          ms->mca[q] = ca;
          ms->mcz[q] = cz;
          ms->mnt[q] = nt;
        }
      }
    }
    named_barrier(2, 128);  // (the epilogues read the lists)
    Cur prev = c;
    int pi = 0;  // part of tile i
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      const uint8_t* st = smem + s * kStageBytes;
      // (1) the tile's record scale factors: row t = key, column 4 g + j holds
      // rows 32 j + lane, every byte the E8M0 of scale block g
      wait_warp(bars + kKvFull + s, ph, ms, a);
      F8_TR(40, i);
      {
        uint32_t v[16];
        bool foreign = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(st + kOffSc + 16 * (32 * j + lane));
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int gk = 0; gk < 4; ++gk) {
            const uint32_t e = (w[gk] >> 23) & 0xFFu;
            // a positive normal power of two (any the writer makes) or zero
            foreign |= !(w[gk] == 0u || ((w[gk] & 0x807FFFFFu) == 0u && e != 0u && e != 0xFFu));
            v[4 * gk + j] = e * 0x01010101u;
          }
        }
        tmem_st16(tmem + lane_base + C::kColSfa + 16 * s, v);
        tmem_wait_st();
        if (__any_sync(0xffffffffu, foreign) && lane == 0 && a.status) atomicOr(a.status, SMLA_STATUS_FOREIGN_SCALE);
      }
      tc_fence_before();
      named_barrier(2, 128);  // every lane quarter's factors are in TMEM
      F8_TR(41, i);
      if (q < C::kQkSplit) {
        // QK of the tile: aux warp q issues latent K-steps kLatSteps q ..
        // and its share of the rope K-steps into accumulator q
        const int qb = pi % C::kNQ;
        const int kbeg = q * C::kLatSteps;
        const int rbeg = q * (4 / C::kQkSplit);
        const int sb = i % C::kSBuf;
        const uint32_t sph = (i / C::kSBuf) & 1;
        wait_warp(bars + kSEmpty + sb, sph ^ 1, ms, a);
        // 32 heads: a new part's q, staged by the loader warps
        if (C::kSplitPass && i > 0 && c.first()) wait_warp(bars + kQReady, uint32_t((pi - 1) & 1), ms, a);
        tc_fence_after();
        F8_TR(30, i);
        if (lane == 0) {
          const uint32_t st32 = smem_base + s * kStageBytes;
          const uint32_t qs = smem_base + C::kOffQ + qb * C::kQBytes;
          const uint32_t d = tmem + C::s_col(sb, q);
          // latent: K-steps of 32 E4M3 (K-chunk kc = 128 dims = scale block kc).
          // The descriptors of this issuer's first K-step, stepped by constant
          // offsets of their start-address field (shared addresses < 256 KB:
          // the 14-bit field never carries)
          const int kc0 = kbeg >> 2;
          uint64_t ad = smem_desc(st32 + kc0 * kChunk, 16, 1024, kSw128);
          uint64_t bd = smem_desc(qs + kc0 * C::kQLatChunk, 16, 1024, kSw128);
          uint32_t sfa = tmem + C::kColSfa + 16 * s + 4 * kc0, sfb = tmem + C::kColSfq + 16 * qb + 4 * kc0;
#pragma unroll 1
          for (int j = 0; j < C::kLatSteps; ++j) {
            const int sub = j & 3;
            mma_mxf8_ss(d, ad, bd, idesc_mxf8(128, kN, 0, 0, sub, sub), sfa, sfb, j > 0 ? 1u : 0u);
            const bool next_chunk = sub == 3;  // 32 bytes on, or the next 128-dim K-chunk
            ad += next_chunk ? uint64_t((kChunk - 96) >> 4) : 2u;
            bd += next_chunk ? uint64_t((C::kQLatChunk - 96) >> 4) : 2u;
            sfa += next_chunk ? 4u : 0u;
            sfb += next_chunk ? 4u : 0u;
          }
          {
            // rope: K-steps of 16 bf16 into the q_hi columns
            const uint64_t ar0 = smem_desc(st32 + kOffRope + 32 * rbeg, 16, 1024, kSw128);
            const uint64_t br0 = smem_desc(qs + C::kQOffRope + 32 * rbeg, 16, 1024, kSw128);
#pragma unroll
            for (int r = 0; r < 4 / C::kQkSplit; ++r)
              mma_f16_ss(d, ar0 + uint64_t(2 * r), br0 + uint64_t(2 * r), idesc_bf16(128, HP, 0, 0), 1u);
          }
          mma_commit(bars + kSFull + sb);
          if (c.last()) mma_commit(bars + kQEmpty + qb);
        }
        __syncwarp();
        F8_TR(31, i);
      }
      if (i == n_tiles - 1 && i > 0 && c.last() && !c.whole()) {
        // The CTA's final part, shared with other CTAs, ends with this tile.
        // If the other parts have all arrived (their tickets are in), this
        // CTA completes the row: their O rows are copied now into the stage
        // of the previous tile (free once that tile's PV has completed) and
        // merged in this part's epilogue, without a partial of this part.
        const int xi = pi == 0 ? 0 : 1;
        const int parts = ms->mparts[xi];
        const int rows_bytes = Hl * kLatent * 4;
        if (parts >= 2 && parts <= kMaxInKernelParts && (parts - 1) * rows_bytes <= kStageBytes) {
          if (ta == 0) ms->fast = ld_acquire_gpu(a.ticket + int64_t(c.row) * hg + g) == parts - 1;
          named_barrier(2, 128);
          if (ms->fast) {
            const int sp = (i - 1) & 1;
            wait_warp(bars + kKvEmpty + sp, ((i - 1) >> 1) & 1, ms, a);  // PV(i - 1) has completed
            const int64_t own = slot_of(c_id, c.P, T, G);
            int jj = 0;
            if (ta == 0) {
              fence_proxy_async_global();  // (the other parts' partials are read by the async proxy)
              mbar_arrive_expect_tx(bars + kMerge, uint32_t((parts - 1) * rows_bytes));
            }
            for (int j = 0; j < parts; ++j) {
              const int64_t sl = ms->mslot[xi][j];
              if (sl == own || jj >= parts - 1) continue;
              if (ta == 0) {
                ms->cb_row[1 + jj] = uint32_t(sp * kStageBytes + jj * rows_bytes);
                bulk_g2s(smem_base + uint32_t(sp * kStageBytes + jj * rows_bytes), a.o_part + (sl * H + h0) * kLatent,
                         uint32_t(rows_bytes), bars + kMerge);
              }
              if (ta < Hl) ms->cb_ml[1 + jj][ta] = __ldcg(reinterpret_cast<const float2*>(a.ml_part) + sl * H + h0 + ta);
              if (ta == 32 * jj) ms->fnv[jj] = __ldcg(a.nv_part + sl);
              ++jj;
            }
            if (ta == 0) ms->fast_s_own = i & 1;
            F8_TR(45, i);
          }
          named_barrier(2, 128);
        }
      }
      // (2) the previous part's epilogue, once this part has started
      if (i > 0 && c.first()) {
        aux_epilogue<HP>(actx, prev, pi - 1, false);
        F8_TR(42, i);
      }
      if constexpr (C::kSplitPass) {
        // (2b) 32 heads: the softmax of heads 16..31 of the tile (the softmax
        // warps take heads 0..15 at the same time)
        const bool first = c.first(), last = c.last();
        const int ob = pi % C::kNO;
        const int rb = i & 1;
        const int sb = i % C::kSBuf;
        if (first) lsum_b = 0.f;
        wait_warp(bars + kSFull + sb, (i / C::kSBuf) & 1, ms, a);
        tc_fence_after();
        PassCtx z;
        z.valid = tile_key(st, ta, lane, q, 1, rb, ms, z.sw);
        z.a = &a;
        z.smem = smem;
        z.ms = ms;
        z.bars = bars;
        z.tmem = tmem;
        z.lane_base = lane_base;
        z.q = q;
        z.lane = lane;
        z.i = i;
        z.s = s;
        z.sb = sb;
        z.rb = rb;
        z.ob = ob;
        z.first = first;
        z.p_shared = 4 * q >= C::kPInRope;
        z.grp = 1;
        z.bar_id = 2;
        z.first_pass = 1;
        z.last_pass = 1;
#ifdef SMLA_TRACE
        z.tr_buf = tr_buf;
        z.tr_k = &tr_k;
#endif
        bool pv_waited = false;
        int es[4];
        softmax_pass<HP>(z, 1, mref_b, lsum_b, pv_waited, es);
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + kPReady + s);  // this warp's P' rows and factors are written
        if (last) {
          // the part's l of heads 16..31, and their (m, l) for the epilogue
          if ((lane & 1) == 0) ms->red_l[q][16 + ((lane >> 1) & 15)] = lsum_b;
          wait_warp(bars + kOEmpty + ob, ((pi / C::kNO) & 1) ^ 1, ms, a);
          named_barrier(2, 128);
          if (q == 0 && lane < 16) {
            const int h = 16 + lane;
            ms->part_m[ob][h] = mref_b;
            ms->part_l[ob][h] = ms->red_l[0][h] + ms->red_l[1][h] + ms->red_l[2][h] + ms->red_l[3][h];
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + kEpiReady + ob);
        }
      }
      // (3) the next part's q, as soon as its buffer is free (32 heads: the
      // loader warps stage it, see there)
      if (!C::kSplitPass && c.last() && i + 1 < n_tiles) {
        const int qb = (pi + 1) % C::kNQ;
        wait_warp(bars + kQEmpty + qb, (((pi + 1) / C::kNQ) & 1) ^ 1, ms, a);
        aux_stage_q<HP>(actx, c.row + 1, qb, 128, 2, true);
        F8_TR(43, i);
      }
      if (c.last()) {
        prev = c;
        ++pi;
      }
      c.advance(a);
    }
    if (pi > 0) aux_epilogue<HP>(actx, prev, pi - 1, true);
    F8_TR(44, 0);
    if (q < C::kQkSplit && lane == 0) mma_commit(bars + kDrain);
    __syncwarp();
  } else {
    // =================== loaders ===================
    const int lw = warp - kLoadWarp0;
    const int kc = lane >> 3, c16 = lane & 7;
    // raw entry of key lw + 8 lane (lanes 0-15) of a cursor's tile, or -1
    auto raw_of = [&](const Cur& cu) -> int32_t {
      const int32_t tk = lw + kLoadWarps * lane;
      if (!cu.live || lane >= kKeysPerLoader) return -1;
      const int32_t p = cu.p0() + tk;
      const int64_t off = cu.beg + p;
      if (p >= cu.p1() || off < 0 || off >= a.n_indices) return -1;
      return __ldg(a.indices + off);
    };
    Cur c;
    c.init(a, row0, P0, cb, ce);
    int32_t raw = raw_of(c);
    F8_TR(52, 0);
    bool oob = false;
    int pl = 0;  // 32 heads: the part of tile i
    (void)pl;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i & 1;
      const uint32_t ph = (i >> 1) & 1;
      if (wait_warp(bars + kKvEmpty + s, ph ^ 1, ms, a)) {
        F8_TR(50, i);
        int32_t id = raw;
        if (id >= a.n_kv_rows) {
          oob = true;
          id = -1;
        }
        if (id < 0) id = -1;
        uint8_t* st = smem + s * kStageBytes;
        const uint32_t st32 = smem_base + s * kStageBytes;
#pragma unroll 4
        for (int j = 0; j < kKeysPerLoader; ++j) {
          const int t = lw + kLoadWarps * j;
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
        if (lane < kKeysPerLoader) *reinterpret_cast<int32_t*>(st + kOffIds + 4 * (lw + kLoadWarps * lane)) = id;
        fence_proxy_async_smem();
        cp_async_mbar_arrive(bars + kKvFull + s);
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + kKvFull + s);
        F8_TR(51, i);
      }
      if constexpr (C::kSplitPass) {
        // 32 heads: a new part's q, staged here while the aux warps (which
        // also run half of the softmax) finish the previous part's last tile;
        // its buffer is free once that tile's QK has completed
        if (i > 0 && c.first()) {
          const int qb = pl % C::kNQ;
          wait_warp(bars + kQEmpty + qb, ((pl / C::kNQ) & 1) ^ 1, ms, a);
          const AuxCtx lx{&a, smem, ms, bars, tmem, uint32_t(32 * (lw & 3)) << 16, H, h0, Hl, hg, g, lane,
                          tid - 32 * kLoadWarp0, c_id, G, T};
          aux_stage_q<HP>(lx, c.row, qb, 32 * kLoadWarps, 3, lw < 4);
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + kQReady);
        }
        if (c.last()) ++pl;
      }
      c.advance(a);
      raw = raw_of(c);  // the next tile's entries, loaded while this one lands
    }
    if (__any_sync(0xffffffffu, oob) && lane == 0 && a.status) atomicOr(a.status, SMLA_STATUS_INDEX_OOB);
    cp_async_wait_all();
  }

  F8_TR(3, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == kAuxWarp0) {
    // every MMA of the CTA has completed before TMEM is freed (also after a
    // timeout: this wait has its own limit)
    if (lane == 0 && !mbar_wait(bars + kDrain, 0, kWaitLimitNs)) set_abort(ms, a.status);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // ---- rows completed here: [P2] stage_combine of their parts, with the sink
  F8_TR(4, ms->n_merge);
  if (ms->n_merge > 0) end_merge(a, smem, bars + kMerge, ms, tid, h0, Hl, hg, g, T, G);
  F8_TR(5, 0);
#ifdef SMLA_TRACE
  if (tid == 0 && tr_buf != nullptr) {
    for (int k = 0; k < 6; ++k)
      tr_buf[(size_t(blockIdx.x) * 20 + 19) * 256 + k] = (ms->merge_t[k] & 0xFFFFFFFFFFFFull) | (uint64_t(70 + k) << 48);
  }
#endif
}

}  // namespace

bool fp8_kernel_supports(int num_heads) { return num_heads >= 1 && num_heads <= 2 * kMaxHP; }

int fp8_tile_len() { return kTK; }

cudaError_t fp8_set_wait_limit(uint64_t ns, int stall) {
  const int32_t st = stall ? 1 : 0;
  const cudaError_t e = cudaMemcpyToSymbol(g_fp8_wait_ns, &ns, sizeof(ns));
  return e != cudaSuccess ? e : cudaMemcpyToSymbol(g_fp8_stall, &st, sizeof(st));
}

int fp8_head_groups(int num_heads) { return num_heads > kMaxHP ? 2 : 1; }

template <int HP>
static cudaError_t launch_fp8_hp(const DecodeLaunch& L) {
  constexpr int smem = smem_total<HP>();
  cudaError_t e = cudaFuncSetAttribute(decode_fp8_kernel<HP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  DecodeArgs args = make_decode_args(L);
  args.row_start_slots = Cfg<HP>::kRowStart;  // (read by the merge kernel)
  args.tile_slots = kTileSlots;
  e = launch_trim(L, args);
  if (e != cudaSuccess) return e;
  decode_fp8_kernel<HP><<<L.plan.grid * L.plan.head_groups, kThreads, smem, L.stream>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess || !L.plan.merge_kernel) return e;
  return launch_merge(L, args);
}

cudaError_t launch_decode_fp8(const DecodeLaunch& L) {
  if (L.plan.grid <= 0) return cudaSuccess;
  return L.p.num_heads <= 16 ? launch_fp8_hp<16>(L) : launch_fp8_hp<32>(L);
}

}  // namespace smla
