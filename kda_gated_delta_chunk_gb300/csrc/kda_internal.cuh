// Internal declarations shared by the host API and the kernels of libkda.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kda.h"

namespace kda {

constexpr int kHeadDim = 128;
constexpr float kL2Eps = 1e-6f;      // l2norm epsilon inside the square root
constexpr int kWorkspaceBytes = 256;  // device status word + error detail (fused path)
constexpr int kDefaultSmCount = 152;  // GB300; sizes the workspace when no device answers

// Split path (chunk-parallel k-side kernel, then a chain kernel): one record per
// (chunk slot, head) in the workspace after a 1 KB header.  Each record is the image of
// the shared-memory operand tiles the chain kernels read, bf16 with the 128-byte swizzle
// (layouts of kda_sm100.cuh):
constexpr int kRecWQ = 0;         // [-W | Qg] MN-major, MN = 128 tokens (0-63 of -W, 64-127
                                  //           of q_raw * 2^Gam) in blocks 16 KB apart, K = dk
constexpr int kRecQKE = 32768;    // [QK; Ke]  K-major, 192 rows x K 64: rows 0-63 raw masked
                                  //           QK (r, K = s), rows 64-191 Ke (dk rows, K = token)
constexpr int kRecTB = 57344;     // T diag(b) K-major, 64 rows x K 64
constexpr int kRecVec = 65536;    // fp32: decay [128], scale/|q| [64], 1/|k| [64]
constexpr int kRecBytes = 66560;
constexpr int kSplitHeader = 1024;
constexpr int kChunk = 64;

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
  int32_t sm_count;            // multiprocessors of the device
  // token strides in elements: q/k/v/g element (t, h, d) at t * s + h * 128 + d, beta (t, h)
  // at t * s_beta + h (dense: s = H * 128, s_beta = H)
  int64_t s_q, s_k, s_v, s_g, s_beta;
  // 1: the fused kernel shares the chunk-local work with k-side helper CTAs (P = 1 only)
  int32_t helpers;
  // optional output row map: token t's output row goes to out[out_index[t]], out being
  // [out_rows, H, 128]; null: to out[t]
  const int32_t* out_index;
  int64_t out_rows;
  // tests only (kda_test_drop_one_record(1)): the helpers leave the record of the last chunk
  // of the longest sequence's head 0 unpublished, so the bounded wait of the fused CTA that
  // needs it runs out
  int32_t test_drop_record;
  // split path only, when > 0: the chain kernel runs beside the k-side kernel (programmatic
  // dependent launch).  k-side CTAs that start on an SM whose %smid is below this value leave
  // it to the chain CTAs (at most two per such SM), and each chain CTA copies a record once
  // its claim word reads kClaimStreamed
  int32_t stream_sms;
  // builds with -DKDA_PHASE_STAMPS only: per-chunk clock64 stamps of CTA 0 (32 per chunk,
  // first 64 chunks); null otherwise
  unsigned long long* stamps;
};

// Timeline stamps of the split path, in builds with -DKDA_PHASE_STAMPS only (nothing
// otherwise): word `index` of Params::stamps gets `value`.  Warp-level chain CTA b < 256:
// words 4b .. 4b+3 = start, first record ready (streamed), end (globaltimer ns), %smid.
// k-side CTA b < 512: words 1024 + 4b .. = start, end, unused, %smid (+ 65536 when the CTA
// left its SM to the chains).
#ifdef KDA_PHASE_STAMPS
#define TSTAMP(index, value)                              \
  do {                                                    \
    if (p.stamps != nullptr) p.stamps[(index)] = (value); \
  } while (0)
#else
#define TSTAMP(index, value) \
  do {                       \
  } while (0)
#endif

// A per-device one-time host step (a kernel's shared-memory attribute): the fast path is one
// atomic load; the first calls on a device serialise on a mutex, so two host threads that
// make a device's first call at the same time both see the step done.
struct PerDeviceOnce {
  static constexpr int kMax = 64;
  std::atomic<bool> done[kMax] = {};
  std::mutex mu;
  template <class Fn>
  cudaError_t run(int dev, Fn&& fn) {
    if (dev < 0 || dev >= kMax) return fn();
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu);
    if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    const cudaError_t e = fn();
    if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
    return e;
  }
};

// Record a device-side error (first writer wins) with its block and site.
__device__ __forceinline__ void record_error(int* status, int code, int site) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    status[2] = site;
  }
}

// Row of `out` that token t's output goes to: t, or out_index[t].  An index outside
// [0, out_rows) records KDA_ERR_BAD_OUT_INDEX and gives -1 (the row is not written).
__device__ __forceinline__ int64_t out_row(const Params& p, int64_t t) {
  if (!p.out_index) return t;
  const int r = p.out_index[t];
  if (r < 0 || (int64_t)r >= p.out_rows) {
    record_error(p.status, KDA_ERR_BAD_OUT_INDEX, 90);
    return -1;
  }
  return r;
}

cudaError_t launch_ref(const Params& p, cudaStream_t stream);
cudaError_t launch_tc(const Params& p, cudaStream_t stream);
// Warp-specialised fused kernel (KDA_KERNEL_PIPE): P = 1, dense outputs.
cudaError_t launch_pipe(const Params& p, cudaStream_t stream);
// Split path: k-side records for every chunk slot (launch_kside), then the chain
// per value slice; launch_split runs both.
cudaError_t launch_kside(const Params& p, cudaStream_t stream);
cudaError_t launch_chain_tc(const Params& p, cudaStream_t stream);   // P = 1
cudaError_t launch_chain_vs(const Params& p, cudaStream_t stream);   // P = 2
// Token-by-token form (decode / speculative verify); token_states may be null.
cudaError_t launch_recurrent(const Params& p, void* token_states, cudaStream_t stream);
cudaError_t launch_split(const Params& p, cudaStream_t stream);
// cuTensorMapEncodeTiled from the CUDA driver (null if unavailable)
void* tensor_map_encoder();
// Low-M projections (kda_skinny_proj): workspace bytes and launch of the two GEMMs.
size_t proj_workspace_bytes(int32_t k, int32_t n_ab);
cudaError_t launch_proj(const void* x, int64_t ldx, const void* w_ab, const void* w_b, void* y,
                        int64_t ldy, void* z, int64_t ldz, int32_t m, int32_t k, int32_t n_ab,
                        int32_t r, int32_t n_b, void* workspace, cudaStream_t stream);

// Chunk slots the split path reserves: every sequence adds at most one partial chunk.
__host__ __device__ inline int64_t split_slots(int64_t total_tokens, int32_t num_seqs) {
  return (total_tokens + kChunk - 1) / kChunk + num_seqs;
}
inline size_t split_workspace_bytes(int64_t total_tokens, int32_t heads, int32_t num_seqs) {
  return (size_t)kSplitHeader + (size_t)split_slots(total_tokens, num_seqs) * heads * kRecBytes;
}

// Fused kernel with k-side helpers: the fused CTAs (one per sequence and head) walk their
// chunks forward; helper CTAs on the remaining SMs write records for chunks taken from
// the far end, newest chunk index first.  One claim word per (slot, head) item follows
// the records: 0 free, 1 taken by a helper, 2 its record is written, 3 taken by the
// sequence's own CTA (indexed by claim_index).  The helpers' item counter sits in the header.
constexpr int kClaimFree = 0, kClaimHelper = 1, kClaimReady = 2, kClaimOwn = 3;
constexpr int kHelperCounterWord = 128;   // int index in the workspace header
constexpr int kHelperMinFreeSms = 8;      // helpers only with at least this many free SMs
// Most (sequence, head) chains AUTO gives helpers: at least kHelperMinFreeSms SMs free and
// at most 5/8 of the SMs busy (beyond that the warp-specialised kernel is faster on GB300)
inline int64_t helper_max_chains(int sms) {
  const int64_t a = (int64_t)sms - kHelperMinFreeSms, b = 5 * (int64_t)sms / 8;
  return a < b ? a : b;
}
constexpr int kHelperMaxSeqs = 128;       // ... and at most this many sequences
// Streamed split path: the k-side kernel takes items from its own counter, first chunk index
// first, and publishes each record by setting its claim word to kClaimStreamed; the chain
// CTAs copy records as they appear.  Header words: that counter, the k-side CTAs that left
// their SM to the chains, the chain CTAs that have finished, the k-side CTAs that have
// started.  The last chain CTA to finish clears the four and the claim words of the call,
// so that every call starts from zero.
constexpr int kClaimStreamed = 4;
constexpr int kStreamCounterWord = 129, kStreamYieldWord = 130, kStreamDoneWord = 131,
              kStreamStartWord = 132;
__host__ __device__ inline size_t helper_claims_offset(int64_t total_tokens, int32_t heads,
                                                       int32_t num_seqs) {
  return (size_t)kSplitHeader + (size_t)split_slots(total_tokens, num_seqs) * heads * kRecBytes;
}
// Claim word of item (slot, head): head-major, so the words that the CTAs of different
// sequences and heads claim at the same moment (the same chunk index) sit in different
// cache lines rather than contending for one.
__host__ __device__ inline int64_t claim_index(int64_t slot, int32_t head, int64_t total_tokens,
                                               int32_t num_seqs) {
  return (int64_t)head * split_slots(total_tokens, num_seqs) + slot;
}
inline size_t helper_workspace_bytes(int64_t total_tokens, int32_t heads, int32_t num_seqs) {
  return helper_claims_offset(total_tokens, heads, num_seqs) +
         (size_t)split_slots(total_tokens, num_seqs) * heads * sizeof(int);
}
// k-side helpers launched behind the fused kernel (programmatic dependent launch)
cudaError_t launch_kside_helpers(const Params& p, cudaStream_t stream);

}  // namespace kda
