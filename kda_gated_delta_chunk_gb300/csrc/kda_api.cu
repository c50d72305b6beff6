// Host side of libkda.so: argument validation, device check, value-split
// choice and kernel dispatch.  Every entry point is declared in include/kda.h.
//
// The validation mirrors the fail-fast capability gate of the FlashKDA
// backend resolver in the PR report "[Perf][GLM-5.3-Flash] Use FlashKDA for
// KDA chunked prefill" (PR #55737, "Backend selection and capability gating"
// listing): head_dim 128, bf16 activations, a bounded gate -- refused with
// an error, never a silent fallback.  It also asserts the workspace bound
// that report lists as unchecked (Risks & impact, item 2).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_test_drop_record{0};   // kda_test_drop_one_record
int g_dev_ok[kMaxDevices];      // 0 unknown, 1 supported, -1 not
int g_dev_sms[kMaxDevices];
std::mutex g_dev_mu;

int check_device(int dev, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_CUDA;
    }
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    g_dev_sms[dev] = count;
  }
  if (sms) *sms = g_dev_sms[dev];
  return g_dev_ok[dev] == 1 ? KDA_OK : KDA_ERR_UNSUPPORTED_DEVICE;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int validate(const void* q, const void* k, const void* v, const void* g, const void* beta,
             const float* A_log, const float* dt_bias, float lower_bound, float scale,
             const void* initial_state, const int32_t* cu_seqlens, void* out,
             void* final_state, int state_dtype, void* workspace, int64_t total_tokens,
             int32_t num_seqs, int32_t heads, size_t workspace_bytes) {
  if (total_tokens < 0 || num_seqs < 0 || heads <= 0) return KDA_ERR_INVALID_ARG;
  if (total_tokens > (int64_t)INT32_MAX) return KDA_ERR_INVALID_ARG;
  if ((int64_t)heads * kda::kHeadDim * total_tokens > ((int64_t)1 << 46)) return KDA_ERR_INVALID_ARG;
  if (state_dtype != KDA_STATE_F32 && state_dtype != KDA_STATE_BF16) return KDA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !std::isfinite(lower_bound)) return KDA_ERR_INVALID_ARG;
  if (lower_bound > 0.0f || lower_bound < KDA_MIN_LOWER_BOUND) return KDA_ERR_UNSAFE_LOWER_BOUND;
  if (!cu_seqlens || !A_log || !dt_bias || !workspace) return KDA_ERR_INVALID_ARG;
  if (num_seqs > 0 && !final_state) return KDA_ERR_INVALID_ARG;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_INVALID_ARG;
  if (workspace_bytes < (size_t)kda::kWorkspaceBytes) return KDA_ERR_WORKSPACE_TOO_SMALL;
  const void* a16[] = {q, k, v, g, out, initial_state, final_state, workspace, A_log, dt_bias};
  for (const void* p : a16)
    if (p && !aligned(p, 16)) return KDA_ERR_MISALIGNED;
  if (beta && !aligned(beta, 2)) return KDA_ERR_MISALIGNED;
  if (!aligned(cu_seqlens, 4)) return KDA_ERR_MISALIGNED;
  return KDA_OK;
}

bool known_kernel(int kernel) {
  return kernel == KDA_KERNEL_AUTO || kernel == KDA_KERNEL_TC || kernel == KDA_KERNEL_REF ||
         kernel == KDA_KERNEL_SPLIT || kernel == KDA_KERNEL_TC_HELPERS ||
         kernel == KDA_KERNEL_PIPE || kernel == KDA_KERNEL_SPLIT_STREAMED;
}

// Value split of the streamed split path: the narrowest value slice (P = 8, else 4, else 2)
// whose N * heads * P chain CTAs leave at least half of the SMs to the k-side kernel running
// beside it; else the unsplit tcgen05 chain (P = 1) while its N * heads CTAs leave 5/8 of the
// SMs (measured on GB300, 4096-token sequences, H = 8, plain split at P = 2 against streamed
// P = 1: 5 sequences 209.7 / 211.9 us, 6: 227.2 / 213.6, 7: 241.8 / 224.1, 8: 262.0 / 265.4,
// 9: 276.3 / 322.2); 0 when none of these holds.  AUTO takes the streamed path only for
// sequences of 32 chunks or more on average: below that the overlap saves less than the
// k-side kernel loses on the chains' SMs (graph-timed on GB300: 4 x 512 tokens, H = 4:
// 21.4 us plain, 26.4 streamed; 1 x 2048, H = 8: 48.6 and 48.3; 1 x 4096, H = 8: 97.0 and
// 84.9).
constexpr int64_t kStreamMinTokensPerSeq = 2048;
int stream_vsplit(int32_t num_seqs, int32_t heads, int sms) {
  const int64_t units = (int64_t)num_seqs * heads;
  if (units <= 0 || num_seqs > kda::kHelperMaxSeqs) return 0;
  for (int P = 8; P >= 2; P /= 2)
    if (2 * units * P <= sms) return P;
  return 8 * units <= 3 * (int64_t)sms ? 1 : 0;
}

// The path of a call: validated selectors, then AUTO resolved.  The split path (k-side
// records + chain per value slice) needs its record area in the workspace; AUTO takes it
// when the value split triggers and the workspace holds the records.  Otherwise one CTA
// per (sequence, head): the warp-specialised kernel, or, while at most 5/8 of the SMs
// would be busy, the fused kernel with k-side helper CTAs on the free ones (on GB300 at
// 2048-token sequences the helpers win up to about 90 chains and lose from about 110).
int plan(int64_t total_tokens, int32_t num_seqs, int32_t heads, size_t workspace_bytes,
         int vsplit, int kernel, int sms, int* kernel_out, int* vsplit_out, int* launches_out) {
  if (vsplit != -1 && vsplit != 1 && vsplit != 2 && vsplit != 4 && vsplit != 8)
    return KDA_ERR_INVALID_ARG;
  if (!known_kernel(kernel)) return KDA_ERR_INVALID_ARG;
  const size_t split_need = kda::split_workspace_bytes(total_tokens, heads, num_seqs);
  const size_t help_need = kda::helper_workspace_bytes(total_tokens, heads, num_seqs);
  int P = vsplit == -1 ? kda_choose_vsplit(num_seqs, heads, sms) : vsplit;
  const bool chunk_count_ok =
      ((total_tokens + kda::kChunk - 1) / kda::kChunk) * num_seqs * heads < ((int64_t)1 << 30);
  const int P_stream = stream_vsplit(num_seqs, heads, sms);
  if (kernel == KDA_KERNEL_SPLIT) {
    if (workspace_bytes < split_need) return KDA_ERR_WORKSPACE_TOO_SMALL;
  } else if (kernel == KDA_KERNEL_SPLIT_STREAMED) {
    if (vsplit == -1) P = P_stream;
    if ((P != 1 && P != 2 && P != 4 && P != 8) || num_seqs > kda::kHelperMaxSeqs || !chunk_count_ok ||
        (P > 1 ? 2 * (int64_t)num_seqs * heads * P > sms : 8 * (int64_t)num_seqs * heads > 3 * (int64_t)sms))
      return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < help_need) return KDA_ERR_WORKSPACE_TOO_SMALL;
  } else if (kernel == KDA_KERNEL_PIPE) {
    if (vsplit != -1 && vsplit != 1) return KDA_ERR_INVALID_ARG;
    P = 1;
  } else if (kernel == KDA_KERNEL_TC_HELPERS) {
    if (vsplit != -1 && vsplit != 1) return KDA_ERR_INVALID_ARG;
    if ((int64_t)num_seqs * heads >= sms || num_seqs > kda::kHelperMaxSeqs ||
        ((total_tokens + kda::kChunk - 1) / kda::kChunk) * num_seqs * heads >= ((int64_t)1 << 30))
      return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < help_need) return KDA_ERR_WORKSPACE_TOO_SMALL;
    P = 1;
  } else if (kernel == KDA_KERNEL_AUTO) {
    if (vsplit == -1 && P > 1 && P_stream > 0 && chunk_count_ok && workspace_bytes >= help_need &&
        total_tokens > 0 && total_tokens >= kStreamMinTokensPerSeq * num_seqs) {
      kernel = KDA_KERNEL_SPLIT_STREAMED;
      P = P_stream;
    } else if (P > 1 && workspace_bytes >= split_need && total_tokens > 0) {
      kernel = KDA_KERNEL_SPLIT;
    } else {
      if (vsplit == -1) P = 1;
      kernel = P == 1 ? KDA_KERNEL_PIPE : KDA_KERNEL_TC;
      // many SMs left free: helpers take the far ends of the sequences
      if (P == 1 && num_seqs > 0 && num_seqs <= kda::kHelperMaxSeqs &&
          (int64_t)num_seqs * heads <= kda::helper_max_chains(sms) &&
          ((total_tokens + kda::kChunk - 1) / kda::kChunk) * num_seqs * heads < ((int64_t)1 << 30) &&
          total_tokens >= (int64_t)4 * kda::kChunk * num_seqs && workspace_bytes >= help_need)
        kernel = KDA_KERNEL_TC_HELPERS;
    }
  }
  int launches = num_seqs == 0 ? 0 : 1;
  if ((kernel == KDA_KERNEL_SPLIT || kernel == KDA_KERNEL_SPLIT_STREAMED) && num_seqs > 0)
    launches = total_tokens > 0 ? 2 : 1;
  if (kernel == KDA_KERNEL_TC_HELPERS && num_seqs > 0 && total_tokens > 0) launches = 2;
  if (kernel_out) *kernel_out = kernel;
  if (vsplit_out) *vsplit_out = P;
  if (launches_out) *launches_out = launches;
  return KDA_OK;
}

int fwd_impl(const void* q, const void* k, const void* v, const void* g, const void* beta,
             const float* A_log, const float* dt_bias, float lower_bound, float scale,
             const void* initial_state, const int32_t* cu_seqlens, void* out, void* final_state,
             int state_dtype, void* workspace, kda_stream_t stream, int64_t total_tokens,
             int32_t num_seqs, int32_t heads, size_t workspace_bytes, int vsplit, int kernel,
             const int64_t* strides, bool scatter = false, const int32_t* out_index = nullptr,
             int64_t out_rows = 0) {
  int rc = validate(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                    cu_seqlens, out, final_state, state_dtype, workspace, total_tokens,
                    num_seqs, heads, workspace_bytes);
  if (rc != KDA_OK) return rc;
  if (scatter) {
    if (!out_index || out_rows < 0) return KDA_ERR_INVALID_ARG;
    if (!aligned(out_index, 4)) return KDA_ERR_MISALIGNED;
  }
  // token strides (elements) of q, k, v, g, beta; NULL = dense
  int64_t st[5] = {(int64_t)heads * kda::kHeadDim, (int64_t)heads * kda::kHeadDim,
                   (int64_t)heads * kda::kHeadDim, (int64_t)heads * kda::kHeadDim, heads};
  if (strides) {
    for (int i = 0; i < 5; ++i) {
      st[i] = strides[i];
      if (st[i] < (i < 4 ? (int64_t)heads * kda::kHeadDim : (int64_t)heads)) return KDA_ERR_INVALID_ARG;
      if (st[i] > ((int64_t)1 << 40) / (total_tokens > 0 ? total_tokens : 1)) return KDA_ERR_INVALID_ARG;
      if (i < 4 && (st[i] % 8) != 0) return KDA_ERR_MISALIGNED;   // 16-byte rows for TMA
    }
  }
  // selectors first: they are host-side checks and need no device
  if (vsplit != -1 && vsplit != 1 && vsplit != 2 && vsplit != 4 && vsplit != 8)
    return KDA_ERR_INVALID_ARG;
  if (!known_kernel(kernel)) return KDA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  rc = check_device(dev, &sms);
  if (rc != KDA_OK) return rc;
  int P = 1, launches = 0;
  rc = plan(total_tokens, num_seqs, heads, workspace_bytes, vsplit, kernel, sms, &kernel, &P,
            &launches);
  if (rc != KDA_OK) return rc;
  if (num_seqs == 0) return KDA_OK;

  kda::Params p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.g = static_cast<const __nv_bfloat16*>(g);
  p.beta = static_cast<const __nv_bfloat16*>(beta);
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.lower_bound = lower_bound;
  p.scale = scale;
  p.initial_state = initial_state;
  p.cu_seqlens = cu_seqlens;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.final_state = final_state;
  p.state_bf16 = state_dtype == KDA_STATE_BF16 ? 1 : 0;
  p.status = static_cast<int*>(workspace);
  p.total_tokens = total_tokens;
  p.num_seqs = num_seqs;
  p.heads = heads;
  p.vsplit = P;
  p.sm_count = sms;
  p.s_q = st[0];
  p.s_k = st[1];
  p.s_v = st[2];
  p.s_g = st[3];
  p.s_beta = st[4];
  p.helpers = (kernel == KDA_KERNEL_TC_HELPERS && total_tokens > 0) ? 1 : 0;
  p.stream_sms = (kernel == KDA_KERNEL_SPLIT_STREAMED && total_tokens > 0) ? num_seqs * heads * P : 0;
  p.test_drop_record =
      ((p.helpers || p.stream_sms > 0) && g_test_drop_record.load(std::memory_order_relaxed) != 0) ? 1 : 0;
#ifdef KDA_PHASE_STAMPS
  // stamps build: the last 16 KB of a workspace of at least 32 KB take the per-chunk stamps
  // (64 chunks x 32 slots of CTA 0)
  if (kernel == KDA_KERNEL_PIPE && workspace_bytes >= 32768)
    p.stamps = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(workspace) +
                                                     ((workspace_bytes - 16384) & ~(size_t)255));
  // ... and for the split path, the last 32 KB of a workspace at least that much larger than
  // the call's records and claim words take its timeline (TSTAMP in kda_internal.cuh)
  if ((kernel == KDA_KERNEL_SPLIT || kernel == KDA_KERNEL_SPLIT_STREAMED) &&
      workspace_bytes >= kda::helper_workspace_bytes(total_tokens, heads, num_seqs) + 33024)
    p.stamps = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(workspace) +
                                                     ((workspace_bytes - 32768) & ~(size_t)255));
#endif
  p.out_index = scatter ? out_index : nullptr;
  p.out_rows = out_rows;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err = (kernel == KDA_KERNEL_REF)     ? kda::launch_ref(p, s)
                    : (kernel == KDA_KERNEL_SPLIT || kernel == KDA_KERNEL_SPLIT_STREAMED)
                        ? kda::launch_split(p, s)
                    : (kernel == KDA_KERNEL_PIPE)  ? kda::launch_pipe(p, s)
                                                   : kda::launch_tc(p, s);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_LAUNCH_FAILED;
  }
  return KDA_OK;
}

int recurrent_impl(const void* q, const void* k, const void* v, const void* g, const void* beta,
                   const float* A_log, const float* dt_bias, float lower_bound, float scale,
                   const void* initial_state, const int32_t* cu_seqlens, void* out,
                   void* final_state, int state_dtype, void* token_states, void* workspace,
                   kda_stream_t stream, int64_t total_tokens, int32_t num_seqs, int32_t heads,
                   size_t workspace_bytes, bool scatter, const int32_t* out_index,
                   int64_t out_rows) {
  int rc = validate(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                    cu_seqlens, out, final_state, state_dtype, workspace, total_tokens,
                    num_seqs, heads, workspace_bytes);
  if (rc != KDA_OK) return rc;
  if (scatter) {
    if (!out_index || out_rows < 0) return KDA_ERR_INVALID_ARG;
    if (!aligned(out_index, 4)) return KDA_ERR_MISALIGNED;
  }
  if (token_states && !aligned(token_states, 16)) return KDA_ERR_MISALIGNED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  rc = check_device(dev, &sms);
  if (rc != KDA_OK) return rc;
  if (num_seqs == 0) return KDA_OK;
  kda::Params p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.g = static_cast<const __nv_bfloat16*>(g);
  p.beta = static_cast<const __nv_bfloat16*>(beta);
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.lower_bound = lower_bound;
  p.scale = scale;
  p.initial_state = initial_state;
  p.cu_seqlens = cu_seqlens;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.final_state = final_state;
  p.state_bf16 = state_dtype == KDA_STATE_BF16 ? 1 : 0;
  p.status = static_cast<int*>(workspace);
  p.total_tokens = total_tokens;
  p.num_seqs = num_seqs;
  p.heads = heads;
  p.vsplit = 1;
  p.sm_count = sms;
  p.s_q = p.s_k = p.s_v = p.s_g = (int64_t)heads * kda::kHeadDim;
  p.s_beta = heads;
  p.out_index = scatter ? out_index : nullptr;
  p.out_rows = out_rows;
  if (kda::launch_recurrent(p, token_states, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_LAUNCH_FAILED;
  }
  return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_workspace_size(int64_t total_tokens, int32_t heads, int32_t max_seqs) {
  if (total_tokens < 0 || heads < 0 || max_seqs < 0) return 0;
  size_t need = (size_t)kda::kWorkspaceBytes;
  // room for the split path's records whenever some batch of up to max_seqs sequences
  // would take it on this device: N sequences qualify when 2 * heads * N <= SMs
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || check_device(dev, &sms) == KDA_ERR_CUDA || sms <= 0) {
    cudaGetLastError();
    sms = kda::kDefaultSmCount;
  }
  if (heads > 0 && total_tokens > 0 && max_seqs > 0 && 2 * (int64_t)heads <= sms) {
    const int32_t n_split = (int32_t)std::min<int64_t>(max_seqs, sms / (2 * (int64_t)heads));
    need = std::max(need, kda::split_workspace_bytes(total_tokens, heads, n_split));
  }
  // ... and for the fused kernel's k-side helpers: N * heads <= helper_max_chains(SMs)
  if (heads > 0 && total_tokens > 0 && max_seqs > 0 && heads <= kda::helper_max_chains(sms)) {
    const int32_t n_help = (int32_t)std::min<int64_t>(
        std::min<int64_t>(max_seqs, kda::kHelperMaxSeqs), kda::helper_max_chains(sms) / heads);
    need = std::max(need, kda::helper_workspace_bytes(total_tokens, heads, n_help));
  }
  return (need + 15) & ~(size_t)15;
}

int kda_chunk_prefill_fwd(const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* A_log, const float* dt_bias,
                          float lower_bound, float scale, const void* initial_state,
                          const int32_t* cu_seqlens, void* out, void* final_state,
                          int state_dtype, void* workspace, kda_stream_t stream,
                          int64_t total_tokens, int32_t num_seqs, int32_t heads,
                          size_t workspace_bytes) {
  return fwd_impl(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                  cu_seqlens, out, final_state, state_dtype, workspace, stream, total_tokens,
                  num_seqs, heads, workspace_bytes, -1, KDA_KERNEL_AUTO, nullptr);
}

int kda_chunk_prefill_fwd_ex(const void* q, const void* k, const void* v, const void* g,
                             const void* beta, const float* A_log, const float* dt_bias,
                             float lower_bound, float scale, const void* initial_state,
                             const int32_t* cu_seqlens, void* out, void* final_state,
                             int state_dtype, void* workspace, kda_stream_t stream,
                             int64_t total_tokens, int32_t num_seqs, int32_t heads,
                             size_t workspace_bytes, int vsplit, int kernel) {
  return fwd_impl(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                  cu_seqlens, out, final_state, state_dtype, workspace, stream, total_tokens,
                  num_seqs, heads, workspace_bytes, vsplit, kernel, nullptr);
}

int kda_chunk_prefill_fwd_strided(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* A_log, const float* dt_bias,
                                  float lower_bound, float scale, const void* initial_state,
                                  const int32_t* cu_seqlens, void* out, void* final_state,
                                  int state_dtype, void* workspace, kda_stream_t stream,
                                  int64_t total_tokens, int32_t num_seqs, int32_t heads,
                                  size_t workspace_bytes, int64_t q_stride, int64_t k_stride,
                                  int64_t v_stride, int64_t g_stride, int64_t beta_stride,
                                  int vsplit, int kernel) {
  const int64_t strides[5] = {q_stride, k_stride, v_stride, g_stride, beta_stride};
  return fwd_impl(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                  cu_seqlens, out, final_state, state_dtype, workspace, stream, total_tokens,
                  num_seqs, heads, workspace_bytes, vsplit, kernel, strides);
}

int kda_chunk_prefill_fwd_scatter(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* A_log, const float* dt_bias,
                                  float lower_bound, float scale, const void* initial_state,
                                  const int32_t* cu_seqlens, void* out, void* final_state,
                                  int state_dtype, void* workspace, kda_stream_t stream,
                                  int64_t total_tokens, int32_t num_seqs, int32_t heads,
                                  size_t workspace_bytes, int64_t q_stride, int64_t k_stride,
                                  int64_t v_stride, int64_t g_stride, int64_t beta_stride,
                                  const int32_t* out_index, int64_t out_rows, int vsplit,
                                  int kernel) {
  const int64_t strides[5] = {q_stride, k_stride, v_stride, g_stride, beta_stride};
  return fwd_impl(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                  cu_seqlens, out, final_state, state_dtype, workspace, stream, total_tokens,
                  num_seqs, heads, workspace_bytes, vsplit, kernel, strides, true, out_index,
                  out_rows);
}


int kda_recurrent_fwd(const void* q, const void* k, const void* v, const void* g,
                      const void* beta, const float* A_log, const float* dt_bias,
                      float lower_bound, float scale, const void* initial_state,
                      const int32_t* cu_seqlens, void* out, void* final_state, int state_dtype,
                      void* token_states, void* workspace, kda_stream_t stream,
                      int64_t total_tokens, int32_t num_seqs, int32_t heads,
                      size_t workspace_bytes) {
  return recurrent_impl(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                        cu_seqlens, out, final_state, state_dtype, token_states, workspace,
                        stream, total_tokens, num_seqs, heads, workspace_bytes, false, nullptr,
                        0);
}

int kda_recurrent_fwd_scatter(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const float* A_log, const float* dt_bias,
                              float lower_bound, float scale, const void* initial_state,
                              const int32_t* cu_seqlens, void* out, void* final_state,
                              int state_dtype, void* token_states, void* workspace,
                              kda_stream_t stream, int64_t total_tokens, int32_t num_seqs,
                              int32_t heads, size_t workspace_bytes, const int32_t* out_index,
                              int64_t out_rows) {
  return recurrent_impl(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state,
                        cu_seqlens, out, final_state, state_dtype, token_states, workspace,
                        stream, total_tokens, num_seqs, heads, workspace_bytes, true, out_index,
                        out_rows);
}

size_t kda_skinny_proj_workspace_size(int32_t k, int32_t n_ab) {
  if (k <= 0 || n_ab <= 0) return 0;
  return (kda::proj_workspace_bytes(k, n_ab) + 15) & ~(size_t)15;
}

int kda_skinny_proj(const void* x, int64_t ldx, const void* w_ab, const void* w_b, void* y,
                    int64_t ldy, void* z, int64_t ldz, int32_t m, int32_t k, int32_t n_ab,
                    int32_t r, int32_t n_b, void* workspace, size_t workspace_bytes,
                    kda_stream_t stream) {
  if (!x || !w_ab || !w_b || !y || !z || !workspace) return KDA_ERR_INVALID_ARG;
  if (m < 1 || m > 16 || k < 512 || k % 512 != 0 || n_ab < 16 || n_ab % 16 != 0 || n_b < 16 ||
      n_b % 16 != 0 || r < 16 || r % 16 != 0 || r > n_ab || r > 512)
    return KDA_ERR_INVALID_ARG;
  if (ldx < k || ldy < n_ab || ldz < n_b) return KDA_ERR_INVALID_ARG;
  if ((int64_t)n_ab * k > ((int64_t)1 << 31) || (int64_t)n_b * r > ((int64_t)1 << 31))
    return KDA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_ab, 16) || !aligned(w_b, 16) || !aligned(y, 16) ||
      !aligned(z, 4) || !aligned(workspace, 16) || ldx % 8 != 0 || ldy % 8 != 0 || ldz % 2 != 0)
    return KDA_ERR_MISALIGNED;
  if (workspace_bytes < kda::proj_workspace_bytes(k, n_ab)) return KDA_ERR_WORKSPACE_TOO_SMALL;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  const int rc = check_device(dev, &sms);
  if (rc != KDA_OK) return rc;
  if (kda::launch_proj(x, ldx, w_ab, w_b, y, ldy, z, ldz, m, k, n_ab, r, n_b, workspace,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_LAUNCH_FAILED;
  }
  return KDA_OK;
}

int kda_choose_vsplit(int32_t num_seqs, int32_t heads, int32_t sm_count) {
  if (num_seqs <= 0 || heads <= 0 || sm_count <= 0) return 1;
  const int64_t units = (int64_t)num_seqs * heads;
  if (2 * units > sm_count) return 1;   // the pages' trigger: 2*H*N <= SMs
  int p = 2;
  while (p < 8 && 2 * p * units <= sm_count) p *= 2;
  return p;
}

const char* kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs an sm_103 GPU)";
    case KDA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than kda_workspace_size()";
    case KDA_ERR_UNSAFE_LOWER_BOUND: return "lower_bound outside [-5, 0]";
    case KDA_ERR_MISALIGNED: return "pointer not aligned as required";
    case KDA_ERR_LAUNCH_FAILED: return "kernel launch failed";
    case KDA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case KDA_ERR_BAD_CU_SEQLENS: return "cu_seqlens not non-decreasing from 0 or past total_tokens";
    case KDA_ERR_CUDA: return "CUDA runtime error";
    case KDA_ERR_BAD_OUT_INDEX: return "an out_index entry lies outside [0, out_rows)";
    default: return "unknown status";
  }
}

int kda_last_device_status(void* workspace, kda_stream_t stream) {
  if (!workspace) return KDA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int host[3] = {0, 0, 0};
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpy(host, workspace, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  if (host[0] != KDA_OK) {
    const int zero[3] = {0, 0, 0};
    if (cudaMemcpy(workspace, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_CUDA;
    }
  }
  return host[0];
}

int kda_device_check(int device) { return check_device(device, nullptr); }

void kda_test_drop_one_record(int on) { g_test_drop_record.store(on != 0 ? 1 : 0); }

int kda_plan_for(int64_t total_tokens, int32_t num_seqs, int32_t heads, size_t workspace_bytes,
                 int vsplit, int kernel, int32_t sm_count, int* kernel_out, int* vsplit_out,
                 int* launches_out) {
  if (total_tokens < 0 || num_seqs < 0 || heads <= 0 || sm_count <= 0) return KDA_ERR_INVALID_ARG;
  if (workspace_bytes < (size_t)kda::kWorkspaceBytes) return KDA_ERR_WORKSPACE_TOO_SMALL;
  return plan(total_tokens, num_seqs, heads, workspace_bytes, vsplit, kernel, sm_count,
              kernel_out, vsplit_out, launches_out);
}

int kda_plan(int64_t total_tokens, int32_t num_seqs, int32_t heads, size_t workspace_bytes,
             int vsplit, int kernel, int* kernel_out, int* vsplit_out, int* launches_out) {
  if (total_tokens < 0 || num_seqs < 0 || heads <= 0) return KDA_ERR_INVALID_ARG;
  if (workspace_bytes < (size_t)kda::kWorkspaceBytes) return KDA_ERR_WORKSPACE_TOO_SMALL;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  const int rc = check_device(dev, &sms);
  if (rc != KDA_OK) return rc;
  return kda_plan_for(total_tokens, num_seqs, heads, workspace_bytes, vsplit, kernel, sms,
                      kernel_out, vsplit_out, launches_out);
}

}  // extern "C"
