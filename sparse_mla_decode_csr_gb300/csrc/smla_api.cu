// C-ABI entry points of libsmla.so: argument checks, the split planner, the
// workspace layout, and the kernel launches.  Everything here is host code;
// the arithmetic of the method lives in the kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "smla.h"
#include "smla_internal.h"

namespace smla {

namespace {

constexpr int kTile = 64;  // keys per pipeline tile (planning granule)

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_sm_count(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_DEVICE;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return SMLA_ERR_DEVICE;
  *num_sms = n;
  return SMLA_OK;
}

// Cost of a split count in "tile times" of the slowest CTA: waves of CTAs
// times tiles per CTA, plus the partial write/read of split rows expressed in
// tiles of gathered bytes (partials are mostly L2 traffic, hence the 1/4).
double split_cost(int64_t n_q, int heads, int64_t tiles, int s, int num_sms) {
  int64_t units = n_q * s;
  int64_t waves = (units + num_sms - 1) / num_sms;
  int64_t per_cta = (tiles + s - 1) / s;
  double partial = 0.0;
  if (s > 1) partial = 0.25 * (2.0 * heads * kLatent * 4.0) / (double(kTile) * kRecordBytes);
  return double(waves) * (double(per_cta) + partial);
}

}  // namespace

WorkspaceLayout workspace_layout(int32_t n_q, int32_t heads, int32_t slots, bool trim_lens) {
  WorkspaceLayout w{};
  w.lens_off = -1;
  if (slots <= 0 && !trim_lens) return w;
  int64_t off = 0;
  w.ticket_off = off;
  off = align256(off + int64_t(n_q) * 2 * 4);  // per row and head group
  w.rowtile_off = off;
  off = align256(off + (int64_t(n_q) + 1) * 8);
  w.o_off = off;
  off = align256(off + int64_t(slots) * heads * kLatent * 4);
  w.ml_off = off;
  off = align256(off + int64_t(slots) * heads * 2 * 4);
  w.nv_off = off;
  off = align256(off + int64_t(slots) * 4);
  if (trim_lens) {  // trimmed row lengths (has_invalid pre-pass), after everything else
    w.lens_off = off;
    off = align256(off + int64_t(n_q) * 4);
  }
  w.total = off;
  return w;
}

int check_decode_params(const smla_decode_params* p) {
  if (p == nullptr) return SMLA_ERR_NULL;
  if (p->n_q < 0 || p->num_heads < 1 || p->num_heads > SMLA_MAX_HEADS) return SMLA_ERR_SHAPE;
  if (p->n_kv_rows < 0 || p->n_kv_rows > (int64_t(1) << 31) || p->n_indices < 0) return SMLA_ERR_SHAPE;
  if (p->num_splits < 0 || p->num_splits > SMLA_MAX_SPLITS) return SMLA_ERR_SPLITS;
  if (p->kernel < SMLA_KERNEL_TENSOR_CORE || p->kernel > SMLA_KERNEL_TENSOR_CORE_FP8) return SMLA_ERR_SHAPE;
  if (p->kernel == SMLA_KERNEL_TENSOR_CORE_FP8 && !fp8_kernel_supports(p->num_heads)) return SMLA_ERR_SHAPE;
  if (p->n_q == 0) return SMLA_OK;
  if (!p->q || !p->indptr || !p->out) return SMLA_ERR_NULL;
  if (p->n_kv_rows > 0 && !p->kv_cache) return SMLA_ERR_NULL;
  if (p->n_indices > 0 && !p->indices) return SMLA_ERR_NULL;
  if (p->q_stride_head < SMLA_QK_DIM && p->num_heads > 1) return SMLA_ERR_STRIDE;
  if (p->q_stride_row < int64_t(p->num_heads - 1) * p->q_stride_head + SMLA_QK_DIM && p->n_q > 1)
    return SMLA_ERR_STRIDE;
  if (p->out_stride_head < SMLA_LATENT_DIM && p->num_heads > 1) return SMLA_ERR_STRIDE;
  if (p->out_stride_row < int64_t(p->num_heads - 1) * p->out_stride_head + SMLA_LATENT_DIM && p->n_q > 1)
    return SMLA_ERR_STRIDE;
  if (p->q_stride_row < 0 || p->q_stride_head < 0 || p->out_stride_row < 0 || p->out_stride_head < 0)
    return SMLA_ERR_STRIDE;
  if (!aligned16(p->q) || !aligned16(p->out) || (p->kv_cache && !aligned16(p->kv_cache)))
    return SMLA_ERR_ALIGN;
  if ((p->q_stride_row | p->q_stride_head | p->out_stride_row | p->out_stride_head) & 7)
    return SMLA_ERR_ALIGN;
  if (!std::isfinite(p->sm_scale)) return SMLA_ERR_SHAPE;
  return SMLA_OK;
}

}  // namespace smla

using namespace smla;

extern "C" {

const char* smla_strerror(int status) {
  switch (status) {
    case SMLA_OK: return "ok";
    case SMLA_ERR_NULL: return "a required pointer is NULL";
    case SMLA_ERR_SHAPE: return "a size is out of range";
    case SMLA_ERR_STRIDE: return "a stride is negative or overlaps rows/heads";
    case SMLA_ERR_ALIGN: return "a pointer or stride breaks the 16-byte alignment rules";
    case SMLA_ERR_WORKSPACE: return "workspace missing or too small";
    case SMLA_ERR_SPLITS: return "num_splits out of range";
    case SMLA_ERR_DEVICE: return "no usable sm_103 CUDA device";
    case SMLA_ERR_LAUNCH: return "kernel launch failed";
    default: return "unknown status";
  }
}

int smla_device_check(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return SMLA_ERR_DEVICE;
  return (major == 10 && minor == 3) ? SMLA_OK : SMLA_ERR_DEVICE;
}

int smla_set_wait_limit(uint64_t limit_ns, int stall_first_wait) {
  const int rc = smla_device_check();
  if (rc != SMLA_OK) return rc;
  if (smla::fp8_set_wait_limit(limit_ns, stall_first_wait) != cudaSuccess ||
      smla::tc_set_wait_limit(limit_ns, stall_first_wait) != cudaSuccess)
    return SMLA_ERR_LAUNCH;
  return SMLA_OK;
}

int smla_plan(const smla_decode_params* p, int32_t num_sms, smla_plan_info* plan) {
  if (plan == nullptr || p == nullptr) return SMLA_ERR_NULL;
  const int32_t n_q = p->n_q, num_heads = p->num_heads, num_splits = p->num_splits;
  if (n_q < 0 || num_heads < 1 || num_heads > SMLA_MAX_HEADS || p->n_indices < 0) return SMLA_ERR_SHAPE;
  if (num_splits < 0 || num_splits > SMLA_MAX_SPLITS) return SMLA_ERR_SPLITS;
  if (p->kernel < SMLA_KERNEL_TENSOR_CORE || p->kernel > SMLA_KERNEL_TENSOR_CORE_FP8) return SMLA_ERR_SHAPE;
  if (p->kernel == SMLA_KERNEL_TENSOR_CORE_FP8 && !fp8_kernel_supports(num_heads)) return SMLA_ERR_SHAPE;
  if (num_sms <= 0) {
    int rc = current_sm_count(&num_sms);
    if (rc != SMLA_OK) return rc;
  }
  int64_t row_len = p->max_row_len;
  if (row_len <= 0) row_len = n_q > 0 ? (p->n_indices + n_q - 1) / n_q : 0;
  const int64_t tiles = std::max<int64_t>(1, (row_len + kTile - 1) / kTile);
  *plan = smla_plan_info{};
  // the default picks the native-fp8 kernel where it supports the head count
  int32_t kernel = p->kernel;
  if (kernel == SMLA_KERNEL_TENSOR_CORE)
    kernel = fp8_kernel_supports(num_heads) ? SMLA_KERNEL_TENSOR_CORE_FP8 : SMLA_KERNEL_TENSOR_CORE_BF16;
  plan->kernel = kernel;
  plan->tile_len = kernel == SMLA_KERNEL_TENSOR_CORE_FP8 ? fp8_tile_len() : kTile;
  plan->head_groups = 1;
  if (kernel != SMLA_KERNEL_CUDA_CORE) {
    // persistent: one CTA per SM, tiles balanced over them; forcing k splits
    // spreads the tiles over n_q * k CTAs instead.  The native-fp8 kernel
    // takes up to 32 heads per CTA: above that two CTAs (head groups) share
    // each schedule range, and the grid counts ranges
    const int hg = kernel == SMLA_KERNEL_TENSOR_CORE_FP8 ? fp8_head_groups(num_heads) : 1;
    plan->head_groups = hg;
    int64_t g = num_splits > 0 ? int64_t(n_q) * num_splits : std::max(1, num_sms / hg);
    g = std::max<int64_t>(1, std::min<int64_t>(g, 65535 / hg));
    plan->grid = n_q > 0 ? int32_t(g) : 0;
    plan->num_splits = 0;
    plan->chunk_len = 0;
    plan->partial_slots = 2 * plan->grid;
    // rows shared between CTAs are merged by a second, parallel kernel; the
    // native-fp8 kernel merges rows of up to kMaxInKernelParts parts itself,
    // and needs the merge kernel only when rows of the top-k length would span
    // more CTAs (about grid / n_q + 1 each); it then merges only those rows
    if (kernel == SMLA_KERNEL_TENSOR_CORE_FP8)
      plan->merge_kernel = (n_q > 0 && (int64_t(plan->grid) + n_q - 1) / n_q + 1 > kMaxInKernelParts) ? 1 : 0;
    else
      plan->merge_kernel = (n_q > 0 && plan->grid > 1) ? 1 : 0;
    // rows that may end in -1 padding are trimmed first by a row-per-warp pass
    plan->trim_kernel = (n_q > 0 && p->has_invalid) ? 1 : 0;
    plan->workspace_bytes =
        n_q > 0 ? workspace_layout(n_q, num_heads, plan->partial_slots, plan->trim_kernel != 0).total : 0;
    return SMLA_OK;
  }
  int s = 1;
  if (num_splits > 0) {
    s = num_splits;
  } else if (n_q > 0) {
    int s_max = int(std::min<int64_t>(tiles, SMLA_MAX_SPLITS));
    double best = split_cost(n_q, num_heads, tiles, 1, num_sms);
    for (int c = 2; c <= s_max; ++c) {
      double cost = split_cost(n_q, num_heads, tiles, c, num_sms);
      if (cost < best * 0.98) {  // more splits only for a clear gain
        best = cost;
        s = c;
      }
    }
  }
  const int64_t per_chunk_tiles = (tiles + s - 1) / s;
  plan->num_splits = s;
  plan->chunk_len = int32_t(std::min<int64_t>(per_chunk_tiles * kTile, INT32_MAX / 2));
  plan->grid = int32_t(int64_t(n_q) * s);
  plan->partial_slots = s > 1 ? n_q * s : 0;
  plan->merge_kernel = 0;
  plan->trim_kernel = 0;
  plan->workspace_bytes = workspace_layout(n_q, num_heads, plan->partial_slots, false).total;
  return SMLA_OK;
}

size_t smla_decode_workspace_size(const smla_decode_params* params) {
  smla_plan_info plan{};
  if (smla_plan(params, 0, &plan) != SMLA_OK) return 0;
  return size_t(plan.workspace_bytes);
}

int smla_decode(const smla_decode_params* params, void* workspace, size_t workspace_bytes,
                void* stream) {
  int rc = check_decode_params(params);
  if (rc != SMLA_OK) return rc;
  if (params->n_q == 0) return SMLA_OK;
  rc = smla_device_check();
  if (rc != SMLA_OK) return rc;
  DecodeLaunch L{};
  L.p = *params;
  rc = smla_plan(params, 0, &L.plan);
  if (rc != SMLA_OK) return rc;
  L.ws = workspace_layout(params->n_q, params->num_heads, L.plan.partial_slots, L.plan.trim_kernel != 0);
  if (L.ws.total > 0 && (workspace == nullptr || int64_t(workspace_bytes) < L.ws.total))
    return SMLA_ERR_WORKSPACE;
  if (L.ws.total > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SMLA_ERR_ALIGN;
  L.workspace = workspace;
  L.stream = static_cast<cudaStream_t>(stream);
  cudaError_t err = L.plan.kernel == SMLA_KERNEL_CUDA_CORE ? launch_decode_simt(L)
                    : L.plan.kernel == SMLA_KERNEL_TENSOR_CORE_FP8 ? launch_decode_fp8(L)
                                                                   : launch_decode_tc(L);
  return err == cudaSuccess ? SMLA_OK : SMLA_ERR_LAUNCH;
}

int smla_pack_records(const void* latent, int64_t latent_stride, const void* rope,
                      int64_t rope_stride, int64_t n, void* kv_out, void* stream) {
  if (n < 0) return SMLA_ERR_SHAPE;
  if (n == 0) return SMLA_OK;
  if (!latent || !rope || !kv_out) return SMLA_ERR_NULL;
  if (latent_stride < SMLA_LATENT_DIM || rope_stride < SMLA_ROPE_DIM) return SMLA_ERR_STRIDE;
  if (!aligned16(latent) || !aligned16(rope) || !aligned16(kv_out) || (latent_stride & 7) ||
      (rope_stride & 7))
    return SMLA_ERR_ALIGN;
  int rc = smla_device_check();
  if (rc != SMLA_OK) return rc;
  cudaError_t err = launch_pack(latent, latent_stride, rope, rope_stride, n, kv_out,
                                static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SMLA_OK : SMLA_ERR_LAUNCH;
}

}  // extern "C"
