// Internal declarations shared by the host API and the kernels of libkda.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kHeadDim = 128;
constexpr float kL2Eps = 1e-6f;      // l2norm epsilon inside the square root
constexpr int kWorkspaceBytes = 256;  // device status word + error detail

// Layout of the workspace (all int32):
//   [0] status: KDA_OK or the first KDA_ERR_* a kernel recorded
//   [1] block that recorded it, [2] where (a wait site or a check id)
struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* g;
  const __nv_bfloat16* beta;
  const float* A_log;
  const float* dt_bias;
  float lower_bound;
  float scale;
  const void* initial_state;   // may be null (zero state)
  const int32_t* cu_seqlens;
  __nv_bfloat16* out;
  void* final_state;
  int state_bf16;              // 0: fp32 state, 1: bf16 state
  int* status;                 // workspace
  int64_t total_tokens;
  int32_t num_seqs;
  int32_t heads;
  int32_t vsplit;              // 1, 2, 4 or 8
};

// Record a device-side error (first writer wins) with its block and site.
__device__ __forceinline__ void record_error(int* status, int code, int site) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    status[2] = site;
  }
}

cudaError_t launch_ref(const Params& p, cudaStream_t stream);
cudaError_t launch_tc(const Params& p, cudaStream_t stream);

}  // namespace kda
