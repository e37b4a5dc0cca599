// Internal declarations shared by the translation units of libsmla.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "smla.h"

namespace smla {

constexpr int kRecordBytes = SMLA_RECORD_BYTES;
constexpr int kLatent = SMLA_LATENT_DIM;
constexpr int kRope = SMLA_ROPE_DIM;
constexpr int kQK = SMLA_QK_DIM;
constexpr int kScaleOffset = 512;
constexpr int kRopeOffset = 528;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Rows shared by at most this many CTAs are merged inside the native-fp8
// decode kernel (by the CTA whose part completes the row); rows of more parts
// are left to the merge kernel when the plan launches it.
constexpr int kMaxInKernelParts = 4;

// Workspace offsets of one plan (see smla_decode_workspace_size in smla.h).
struct WorkspaceLayout {
  int64_t ticket_off, rowtile_off, o_off, ml_off, nv_off, lens_off, total;
};

WorkspaceLayout workspace_layout(int32_t n_q, int32_t heads, int32_t slots, bool trim_lens);

// Everything a decode kernel needs, resolved on the host.
struct DecodeLaunch {
  smla_decode_params p;
  smla_plan_info plan;
  WorkspaceLayout ws;
  void* workspace;
  cudaStream_t stream;
};

// Host-side argument checks of smla_decode (SMLA_OK or a negative status);
// nothing is enqueued.
int check_decode_params(const smla_decode_params* p);

struct DecodeArgs;

// Kernel launchers (one per translation unit).  Return a cudaError_t.
cudaError_t launch_decode_simt(const DecodeLaunch& L);
cudaError_t launch_decode_tc(const DecodeLaunch& L);
cudaError_t launch_decode_fp8(const DecodeLaunch& L);
// The row-trim pass before a tensor-core decode (when plan.trim_kernel; it
// points args.lens at the trimmed lengths) and the merge of shared rows after it.
cudaError_t launch_trim(const DecodeLaunch& L, DecodeArgs& args);
cudaError_t launch_merge(const DecodeLaunch& L, const DecodeArgs& args);
// Heads and tile length of the native-fp8 kernel.
bool fp8_kernel_supports(int num_heads);
int fp8_tile_len();
int fp8_head_groups(int num_heads);
// Pipeline wait limits of the tensor-core kernels (0: their 2 s default) and
// the timeout-path test switch (see smla_set_wait_limit).
cudaError_t fp8_set_wait_limit(uint64_t ns, int stall);
cudaError_t tc_set_wait_limit(uint64_t ns, int stall);
cudaError_t launch_pack(const void* latent, int64_t latent_stride, const void* rope,
                        int64_t rope_stride, int64_t n, void* kv_out, cudaStream_t stream);

}  // namespace smla
