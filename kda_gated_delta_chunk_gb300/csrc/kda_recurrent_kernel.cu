// Token-by-token KDA (the recurrent form) for decode and speculative-verify
// steps: a few tokens per sequence, on the same state layout as the prefill.
//
// Per token (the gated delta rule with the bounded gate of the FlashKDA prefill
// PR report, PR #55737, Features & motivation; the pages route speculative
// tokens through this recurrent form so that a rejected draft can be rolled
// back, Discussion):
//   qh = scale q / |q|, kh = k / |k|, a = lb sigmoid(e^{A_log} (g + dt_bias)), b = sigmoid(beta)
//   S = diag(e^a) S;  u = b (v - S^T kh);  S += kh u^T;  out = S^T qh
// One CTA (128 threads) per (sequence, head, 32 value columns): lane l of warp w
// owns value column l and key rows 32 w .. 32 w + 31 of the 128 x 32 fp32 state
// slice, in registers.  S^T kh and S^T qh are then per-thread sums over 32 key rows
// plus one four-way combine through shared memory; the gate and the normalised
// q, k of a token are shared by the CTA.  Optionally the state after every token
// is written out (token_states), which is what a caller needs to continue from
// any accepted prefix.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int RT = 128;    // threads = key channels
constexpr int RDV = 32;    // value columns per CTA
constexpr int RSPLIT = kHeadDim / RDV;
constexpr float kLog2eR = 1.4426950408889634f;

__device__ __forceinline__ float ex2r(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_r(float x) { return 1.0f / (1.0f + ex2r(-x * kLog2eR)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(RT)
    kda_recurrent_kernel(const __grid_constant__ Params p, void* token_states) {
  __shared__ float red[4][RDV];     // per-warp column sums
  __shared__ float nrm[2][4];       // per-warp sums of squares of q, k
  __shared__ float qs[RT], ks[RT], ds[RT];   // normalised q, k and the decay of each key row
  __shared__ float ucol[RDV];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = p.heads;
  const int part = blockIdx.x % RSPLIT;
  const int h = (blockIdx.x / RSPLIT) % H;
  const int n = blockIdx.x / (RSPLIT * H);
  const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
  if (t0 < 0 || t1 < t0 || (int64_t)t1 > p.total_tokens || p.cu_seqlens[0] != 0) {
    if (tid == 0) record_error(p.status, KDA_ERR_BAD_CU_SEQLENS, 7);
    return;
  }
  const int dv0 = part * RDV, dv = dv0 + lane, dkq = 32 * warp;   // this thread: column dv,
  const size_t HD2 = (size_t)kHeadDim * kHeadDim;                  // rows dkq .. dkq + 31
  const size_t sbase = ((size_t)n * H + h) * HD2 + dv;
  const size_t hoff = (size_t)h * kHeadDim;

  // the first token's inputs are requested before the state, so their latencies overlap
  float qv = 0.f, kv = 0.f, gv = 0.f, bv = 0.f, vv = 0.f;
  auto load_token = [&](int t) {
    qv = __bfloat162float(p.q[(size_t)t * p.s_q + hoff + tid]);
    kv = __bfloat162float(p.k[(size_t)t * p.s_k + hoff + tid]);
    gv = __bfloat162float(p.g[(size_t)t * p.s_g + hoff + tid]);
    bv = __bfloat162float(p.beta[(size_t)t * p.s_beta + h]);
    vv = __bfloat162float(p.v[(size_t)t * p.s_v + hoff + dv]);
  };
  if (t0 < t1) load_token(t0);

  float S[32];   // S[j] = state[dkq + j][dv]
  if (p.initial_state) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const size_t idx = sbase + (size_t)(dkq + j) * kHeadDim;
      S[j] = p.state_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.initial_state)[idx])
                          : static_cast<const float*>(p.initial_state)[idx];
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) S[j] = 0.0f;
  }
  const float gsc = expf(p.A_log[h]);
  const float dtb = p.dt_bias[hoff + tid];
  const float lbl2 = p.lower_bound * kLog2eR;

  auto store_state = [&](void* dst_base, size_t base) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const size_t idx = base + (size_t)(dkq + j) * kHeadDim;
      if (p.state_bf16)
        static_cast<__nv_bfloat16*>(dst_base)[idx] = __float2bfloat16_rn(S[j]);
      else
        static_cast<float*>(dst_base)[idx] = S[j];
    }
  };

  for (int t = t0; t < t1; ++t) {
    // thread tid: key row tid of the token (norms, gate); the next token's inputs in flight
    const float sq = warp_sum(qv * qv), sk = warp_sum(kv * kv);
    if (lane == 0) {
      nrm[0][warp] = sq;
      nrm[1][warp] = sk;
    }
    const float dec = ex2r(lbl2 * sigmoid_r(gsc * (gv + dtb)));
    const float bt = sigmoid_r(bv), vt = vv, qraw = qv, kraw = kv;
    if (t + 1 < t1) load_token(t + 1);
    __syncthreads();
    const float iq = p.scale * rsqrtf((nrm[0][0] + nrm[0][1]) + (nrm[0][2] + nrm[0][3]) + kL2Eps);
    const float ik = rsqrtf((nrm[1][0] + nrm[1][1]) + (nrm[1][2] + nrm[1][3]) + kL2Eps);
    qs[tid] = qraw * iq;
    ks[tid] = kraw * ik;
    ds[tid] = dec;
    __syncthreads();
    // decay, then this thread's part of (S^T kh)[dv]
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      S[j] *= ds[dkq + j];
      acc = fmaf(S[j], ks[dkq + j], acc);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {   // u = b (v - S^T kh) for column dv
      const float stk = (red[0][lane] + red[1][lane]) + (red[2][lane] + red[3][lane]);
      ucol[lane] = bt * (vt - stk);
    }
    __syncthreads();
    const float u = ucol[lane];
    float o = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      S[j] = fmaf(ks[dkq + j], u, S[j]);
      o = fmaf(S[j], qs[dkq + j], o);
    }
    red[warp][lane] = o;   // warp 0 read S^T kh before the last barrier
    __syncthreads();
    if (warp == 0) {
      const float ot = (red[0][lane] + red[1][lane]) + (red[2][lane] + red[3][lane]);
      const int64_t row = out_row(p, t);
      if (row >= 0) p.out[(size_t)row * H * kHeadDim + hoff + dv] = __float2bfloat16_rn(ot);
    }
    if (token_states) store_state(token_states, ((size_t)t * H + h) * HD2 + dv);
    __syncthreads();   // red, nrm, qs, ks, ds are rewritten by the next token
  }
  store_state(p.final_state, sbase);
}

}  // namespace

cudaError_t launch_recurrent(const Params& p, void* token_states, cudaStream_t stream) {
  const long long blocks = (long long)p.num_seqs * p.heads * RSPLIT;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  kda_recurrent_kernel<<<(unsigned)blocks, RT, 0, stream>>>(p, token_states);
  return cudaGetLastError();
}

}  // namespace kda
