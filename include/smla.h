/*
 * smla.h -- sparse multi-head latent attention (MLA) decode over packed
 * fp8_ds_mla KV records, for NVIDIA GB300 (sm_103a).  C ABI of libsmla.so.
 *
 * What is computed follows these pages:
 *   [P1] "vllm.models.kimi_k3.amd.ops.flydsl_sparse_mla_gfx950" (FlyDSL sparse
 *        MLA forward over fp8_ds_mla records, gfx950): module docstring
 *        (record layout, CSR tiles and masking, preconditions, writer rule)
 *        and the epilogue of build_sparse_mla_fp8ds_module (output and LSE).
 *   [P2] "vllm.models.deepseek_v41.amd.mono.attention.back" (K2 back):
 *        stage_split (per-chunk partial, max, sum) and stage_combine (chunk
 *        merge with the per-head sink).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers on the current CUDA device.  The
 *     library never allocates, frees, or synchronises; every call is
 *     asynchronous on `stream` (a cudaStream_t passed as void*, NULL = the
 *     legacy default stream).  The caller owns every buffer.
 *   - Return value: SMLA_OK (0) or a negative smla_status.  Argument errors are
 *     detected on the host before anything is enqueued.  A non-zero status
 *     from a launch is SMLA_ERR_LAUNCH.  smla_strerror() names each code.
 *   - Integers are little-endian; strides are in elements of the tensor's type.
 */
#ifndef SMLA_H
#define SMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Record layout, [P1] module docstring "Record (656 B)": bytes [0, 512) hold
 * 512 E4M3 latent values, [512, 528) four little-endian f32 power-of-two
 * scales (scale b covers latent dims [128 b, 128 b + 128)), [528, 656) the
 * 64 bf16 RoPE dims.  656 = 41 * 16, so every record is 16-byte aligned when
 * the cache base is. */
#define SMLA_RECORD_BYTES 656
#define SMLA_LATENT_DIM 512
#define SMLA_ROPE_DIM 64
#define SMLA_QK_DIM 576
#define SMLA_SCALE_BLOCK 128
#define SMLA_MAX_HEADS 64

typedef enum smla_status {
  SMLA_OK = 0,
  SMLA_ERR_NULL = -1,       /* a required pointer is NULL */
  SMLA_ERR_SHAPE = -2,      /* a size is out of range (n_q < 0, heads not in [1, 64], ...) */
  SMLA_ERR_STRIDE = -3,     /* a stride overlaps rows/heads or is negative */
  SMLA_ERR_ALIGN = -4,      /* a pointer or stride breaks the alignment rules below */
  SMLA_ERR_WORKSPACE = -5,  /* workspace missing or smaller than smla_decode_workspace_size */
  SMLA_ERR_SPLITS = -6,     /* num_splits outside [0, SMLA_MAX_SPLITS] */
  SMLA_ERR_DEVICE = -7,     /* no CUDA device, or the current device is not sm_103 */
  SMLA_ERR_LAUNCH = -8      /* a kernel launch failed (see cudaGetLastError) */
} smla_status;

/* Bits a decode call ORs into *status (when status != NULL). */
#define SMLA_STATUS_INDEX_OOB 0x1   /* an index >= n_kv_rows was met and masked */
#define SMLA_STATUS_TIMEOUT 0x2     /* an in-kernel pipeline wait gave up: results invalid */
#define SMLA_STATUS_SMEM_LAYOUT 0x4 /* the kernel could not align its shared memory and
                                       computed nothing: results invalid */
#define SMLA_STATUS_FOREIGN_SCALE 0x8 /* native-fp8 kernel: a gathered record holds a block
                                         scale that is neither zero nor a positive normal
                                         power of two (smla_pack_records never writes one);
                                         the rows holding it are not computed exactly: run
                                         SMLA_KERNEL_TENSOR_CORE_BF16 on such caches */

#define SMLA_MAX_SPLITS 64

/* Arguments of one decode call.
 *
 * Row r's keys are the CSR slice indices[indptr[r] : indptr[r + 1]] ([P1]
 * module docstring, "Tiles").  Its length is max(indptr[r+1] - indptr[r], 0),
 * further capped at max(lens[r], 0) when lens != NULL.  Position p of the
 * slice contributes iff its offset indptr[r] + p lies in [0, n_indices) and
 * 0 <= indices[offset] < n_kv_rows.  Entries < 0 are masked with or without
 * has_invalid ([P1] "Tiles": masked positions contribute nothing); an entry
 * >= n_kv_rows, which [P1] lists as a precondition the host cannot check, is
 * masked the same way here, never dereferenced, and flagged in *status.
 * Duplicate entries count once per position.
 *
 * For each row r and head h, over the contributing keys t:
 *   k_t[d] = e4m3(rec_t[d]) * scale_t[d / 128]   (d < 512), bf16 rope (512 <= d < 576)
 *   s_t    = sm_scale * sum_{d < 576} q[r, h, d] * k_t[d]
 *   m = max_t s_t,  l = sum_t exp(s_t - m)
 *   lse[r, h] = m + ln(l)                          ([P1] epilogue; the sink is
 *                                                  not part of the LSE)
 *   out[r, h, d] = sum_t exp(s_t - m) k_t[d] / (l + exp(sink[h] - m))   (d < 512)
 * with the sink term absent when sink == NULL (it enters the denominator once,
 * as [P2] stage_combine folds it).  A row with no contributing key gives
 * out = 0 and lse = -inf, sink or not ([P1] epilogue).
 *
 * Layouts and alignment:
 *   q        bf16, element [r][h][d] at q + r*q_stride_row + h*q_stride_head + d;
 *            16-byte aligned base, strides multiples of 8 elements.
 *   kv_cache uint8 [n_kv_rows][656], 16-byte aligned.  Row ids are 64-bit
 *            byte offsets, so caches beyond 4 GiB work; n_kv_rows <= 2^31.
 *   indices  int32 [n_indices]; indptr int32 [n_q + 1]; lens int32 [n_q] or NULL.
 *   sink     f32 [num_heads] or NULL, in the natural-log units of s_t.
 *   out      bf16, element [r][h][d] at out + r*out_stride_row + h*out_stride_head + d;
 *            16-byte aligned base, strides multiples of 8 elements.
 *   lse      f32 [n_q][num_heads] contiguous, or NULL.
 *   n_valid  int32 [n_q] or NULL: number of contributing keys of each row.
 *   status   int32 [1] or NULL: SMLA_STATUS_* bits are ORed in (never cleared).
 */
typedef struct smla_decode_params {
  int32_t n_q;
  int32_t num_heads;
  const void* q;
  int64_t q_stride_row;
  int64_t q_stride_head;
  const void* kv_cache;
  int64_t n_kv_rows;
  const int32_t* indices;
  int64_t n_indices;
  const int32_t* indptr;
  const int32_t* lens;
  /* Planning hints; results never depend on them.  max_row_len: an upper
   * bound of the rows' slice lengths known on the host (e.g. top-k); <= 0 means
   * unknown (n_indices / n_q is used).  has_invalid: rows may end in -1
   * padding ([P1] "Tiles", has_invalid).  Masked entries contribute nothing
   * either way; with has_invalid the tensor-core plan first trims each row to
   * its last entry >= 0 (a pass with a warp per row, plan.trim_kernel = 1) so
   * that the decode skips tiles of padding. */
  int32_t max_row_len;
  int32_t has_invalid;
  float sm_scale;
  const float* sink;
  void* out;
  int64_t out_stride_row;
  int64_t out_stride_head;
  float* lse;
  int32_t* n_valid;
  int32_t* status;
  /* Split-KV control ([P2] stage_split / stage_combine).  0 lets the planner
   * choose from the row length, the batch and the SM count.  k >= 1: the
   * CUDA-core kernel cuts every row into k chunks; the tensor-core kernel
   * spreads the tiles over n_q * k CTAs (about k parts per row). */
  int32_t num_splits;
  /* Which kernel runs the call (all compute the same definition):
   *   SMLA_KERNEL_TENSOR_CORE (0, default): the native-fp8 kernel for the head
   *     counts it supports (1..16), else the bf16 tensor-core kernel;
   *   SMLA_KERNEL_CUDA_CORE (1): an fp32 CUDA-core kernel kept as a cross-check;
   *   SMLA_KERNEL_TENSOR_CORE_BF16 (2): tcgen05 kind::f16 on latents dequantised
   *     to bf16 (exact for power-of-two scales up to 2^7, any scale accepted);
   *   SMLA_KERNEL_TENSOR_CORE_FP8 (3): tcgen05 kind::mxf8f6f4 on the E4M3 bytes as
   *     they are, the block scales as E8M0 scale factors (heads 1..16; a call
   *     with more heads returns SMLA_ERR_SHAPE).  Needs writer-format scales:
   *     zero or positive normal powers of two; others set
   *     SMLA_STATUS_FOREIGN_SCALE. */
  int32_t kernel;
} smla_decode_params;

#define SMLA_KERNEL_TENSOR_CORE 0
#define SMLA_KERNEL_CUDA_CORE 1
#define SMLA_KERNEL_TENSOR_CORE_BF16 2
#define SMLA_KERNEL_TENSOR_CORE_FP8 3

/* How a decode call with given params is laid out on the GPU.
 *
 * Tensor-core kernels (bf16: tile_len 64; native fp8: tile_len 128): a
 * persistent, balanced schedule.  Each row r is cut into
 * T_r = max(1, ceil(len_r / tile_len)) tiles of tile_len slice positions
 * and takes s + k T_r slots of a schedule space, rows in order (s slots stand
 * for the cost of starting a row: its epilogue and q staging; bf16 kernel:
 * k = 1 slot per tile and s = 2; native-fp8 kernel: k = 2, s = 1, i.e. half
 * a tile), so that tile t of row r starts at slot R_r + k t with
 * R_r = s + sum_{r' < r} (s + k T_r').  CTA c of G = grid takes the slots
 * [b_c, e_c) with b_c = floor(c W / G), W the slot total, and the tiles whose
 * first slot lies there, and streams through them across row boundaries.
 * A row lying wholly inside one CTA's range is finished there; a row shared
 * by CTAs c_a..c_b (the CTAs holding its first and last tile) gets
 * one partial per CTA, stored in workspace slot 2 c + (R_r < b_c ? 0 : 1), and
 * is merged from those slots ([P2] stage_combine).  bf16 kernel: by a second,
 * small kernel launched right after (merge_kernel = 1 whenever grid > 1; a
 * warp merges one head of a row).  Native-fp8 kernel (with more than 32
 * heads two CTAs, head groups of 32, share each slot range): a row of up to 4
 * parts is merged inside the decode launch by the CTA whose part arrives last
 * (per-row ticket); when the other parts had all arrived before that CTA's
 * final part ended, it merges from its own O without writing that part's
 * partial.  Rows of more parts, possible only when ceil(grid / n_q) + 1 > 4,
 * are left to the merge kernel (merge_kernel = 1 then).
 * CUDA-core kernel: one CTA per (row, chunk); chunk c of a row covers slice
 * positions [c chunk_len, (c + 1) chunk_len), the last chunk everything after;
 * partial slot r * num_splits + c; the last chunk to finish merges.
 *
 * Tensor-core kernel with has_invalid: a pass before the decode (warp per
 * row, 512 slice positions per step from the end) writes each row's length
 * trimmed to its last entry >= 0 into the workspace, and the decode schedules
 * those lengths (trim_kernel = 1).
 *
 * Fields: kernel (the SMLA_KERNEL_* that runs: 1, 2 or 3), grid (CTAs of the decode launch), tile_len
 * (keys per tile), num_splits and chunk_len (CUDA-core kernel only),
 * partial_slots, merge_kernel, trim_kernel, workspace_bytes.  num_sms > 0 makes the plan
 * pure host arithmetic (no CUDA call); num_sms = 0 asks the current device. */
typedef struct smla_plan_info {
  int32_t kernel;
  int32_t grid;
  int32_t tile_len;
  int32_t num_splits;
  int32_t chunk_len;
  int32_t partial_slots;
  int32_t merge_kernel;
  int32_t trim_kernel;
  int32_t head_groups;
  int64_t workspace_bytes;
} smla_plan_info;

int smla_plan(const smla_decode_params* params, int32_t num_sms, smla_plan_info* plan);

/* Workspace bytes smla_decode needs for these params on the current device
 * (0 when none; also 0 for invalid params).
 *
 * Layout (each part 256-byte aligned), S = plan.partial_slots:
 *   ticket   int32 [2 n_q]       per-row (and head group) arrival counters (CUDA-core and
 *                                native-fp8 kernels)
 *   row_tile int64 [n_q + 1]     tensor-core kernel: first slot of every row, then W
 *   o_part   f32 [S][H][512]     unnormalised partial sum_t 2^(x_t - m) v_t of a row part
 *   ml_part f32 [S][H][2]        (m, l) of x_t = s_t * log2(e): m is the part's reference
 *                                maximum (its max, or at most 24 (bf16 kernel) or 16 (native
 *                                fp8) below it), l = sum_t 2^(x_t - m);
 *                                m = -inf, l = 0 for a part without keys
 *   nv_part int32 [S]            contributing keys of the part
 *   lens    int32 [n_q]          trimmed row lengths (only when plan.trim_kernel)
 * The ticket counters must be zero when a call starts (e.g. allocate the
 * workspace zeroed); every completed call returns them to zero.  A call with
 * other sizes may have written partials over that region, so re-zero bytes
 * [0, 8 n_q) before reusing a workspace across calls of different n_q,
 * num_heads, kernel or plan.  Calls that share a workspace must be ordered
 * (same stream); a call that reports SMLA_STATUS_TIMEOUT leaves it undefined. */
size_t smla_decode_workspace_size(const smla_decode_params* params);

/* Sparse MLA decode (the definition above): one decode launch, preceded by
 * the row-trim pass when plan.trim_kernel = 1 and followed by the merge kernel
 * when plan.merge_kernel = 1.  Each CTA gathers its tiles' records,
 * dequantises them to bf16 (exact), runs QK over 576 dims and PV over 512 dims
 * on the tcgen05 tensor cores with an online softmax in between, and writes
 * out / lse of its whole rows and partials of shared rows (see smla_plan).
 * `workspace` may be NULL only when smla_decode_workspace_size() returns 0.
 * Accuracy: q, k and v enter the products exactly when every block scale is a
 * positive normal power of two up to 2^7 (all scales smla_pack_records
 * writes); a block with any other f32 scale (zero, negative, not a power of
 * two, above 2^7) has each latent value e4m3 * scale formed in f32 and
 * rounded once to bf16 (exact where that product is a bf16), on a slower
 * path.  p is rounded to bf16, sums are f32, out is rounded to bf16 (round to
 * nearest even). */
int smla_decode(const smla_decode_params* params, void* workspace, size_t workspace_bytes,
                void* stream);

/* Bytes of the fixed device array behind smla_decode_noalloc: 64 MiB per
 * device.  A default tensor-core plan on a 152-SM GPU needs about 40 MiB at 64
 * heads (304 partial slots x 64 heads x 2 KiB) plus 12 bytes per query row. */
#define SMLA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* smla_decode without a caller-supplied workspace, for callers that cannot
 * allocate device memory at call time: code running inside another runtime's
 * memory pool or allocation-free serving loop, where a cudaMalloc (or a
 * framework allocation) on the call path is not allowed or would stall other
 * work.  The pages describe no such entry point; it is an addition of this
 * library.
 *
 * Same params, outputs, accuracy and launches as smla_decode; the split-KV
 * workspace (the layout of smla_decode_workspace_size) lives instead in a
 * file-scope device array of SMLA_NOALLOC_SCRATCH_BYTES bytes inside
 * libsmla.so.  The call allocates nothing.
 *   - Set-up: the first call on a device (the current device) looks up the
 *     device address of that array once (cudaGetSymbolAddress, which may load
 *     the library's module on that device).  Make that first call before any
 *     stream capture.
 *   - Limit: a call whose workspace would exceed SMLA_NOALLOC_SCRATCH_BYTES
 *     returns SMLA_ERR_WORKSPACE and launches nothing (use smla_decode with a
 *     workspace of smla_decode_workspace_size bytes instead).
 *   - Sharing: every call on a device uses the same array and leaves its last
 *     contents there.  Calls whose work may overlap on the GPU (different
 *     streams without an ordering event) race on it and give wrong results;
 *     order them.  With the CUDA-core and native-fp8 kernels the call first
 *     clears the ticket counters (bytes [0, 8 n_q)) on `stream`; the bf16
 *     tensor-core kernel writes every part of the array it reads and needs
 *     nothing cleared.
 * Errors as smla_decode, plus SMLA_ERR_DEVICE when the set-up fails. */
int smla_decode_noalloc(const smla_decode_params* params, void* stream);

/* The record writer ([P1] module docstring, "Preconditions": vLLM's
 * concat_and_cache_ds_mla rule).  For each of n records:
 *   scale_b = pow2ceil(max(amax_b, 1e-4) / 448), amax_b = max |latent[128 b .. 128 b + 127]|
 *   bytes [0, 512)   = E4M3(latent_d / scale_{d/128}), round to nearest even, saturating
 *   bytes [512, 528) = the four scales as f32
 *   bytes [528, 656) = the 64 rope bf16 values, bit for bit
 * latent: bf16 [n][latent_stride] (first 512 used), rope: bf16 [n][rope_stride]
 * (first 64 used), kv_out: uint8 [n][656].  Pointers 16-byte aligned, strides
 * multiples of 8 elements.  scale <= 2^7 holds iff |latent| <= 57344. */
int smla_pack_records(const void* latent, int64_t latent_stride, const void* rope,
                      int64_t rope_stride, int64_t n, void* kv_out, void* stream);

/* Name of a status code. */
const char* smla_strerror(int status);

/* SMLA_OK when the current CUDA device can run the kernels (sm_103). */
int smla_device_check(void);

/* Limit, in ns, of every in-kernel pipeline wait of the tensor-core kernels
 * launched after this call on the current device (process-wide); 0 restores
 * the default of 2 s.  A wait that runs out sets SMLA_STATUS_TIMEOUT: the CTA
 * then skips its remaining waits, still issues its pending copies and MMAs,
 * waits (2 s at most each) until they have completed, frees its tensor memory
 * and exits, so that the CUDA context stays usable.  out, lse, n_valid and the
 * workspace are then undefined (re-zero the ticket region before the next
 * call).  stall_first_wait = 1 makes the first softmax wait of every CTA wait
 * on a barrier that nothing signals, so that it runs out after the limit: a
 * test of that path, with no fault and no hang; 0 for normal operation.
 * Returns SMLA_ERR_DEVICE off sm_103, SMLA_ERR_LAUNCH when the values cannot
 * be set. */
int smla_set_wait_limit(uint64_t limit_ns, int stall_first_wait);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_H */
