// Token-by-token KDA (the recurrent form) for decode and speculative-verify
// steps: a few tokens per sequence, on the same state layout as the prefill.
//
// Per token (the gated delta rule with the bounded gate of the FlashKDA prefill
// PR report, PR #55737, Features & motivation; the pages route speculative
// tokens through this recurrent form so that a rejected draft can be rolled
// back, Discussion):
//   qh = scale q / |q|, kh = k / |k|, a = lb sigmoid(e^{A_log} (g + dt_bias)), b = sigmoid(beta)
//   S = diag(e^a) S;  u = b (v - S^T kh);  S += kh u^T;  out = S^T qh
// One CTA (128 threads) per (sequence, head, 32 value columns): thread i owns key
// row i of the 128 x 32 fp32 state slice in registers.  S^T kh and S^T qh are
// reduced over the key rows with warp reduce-scatters and one cross-warp step.
// Optionally the state after every token is written out (token_states), which
// is what a caller needs to continue from any accepted prefix.
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

// v[0..31] summed over the warp's 32 lanes; lane l ends with the sum of v[l].
__device__ __forceinline__ float reduce_scatter32(float (&v)[RDV], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(RT)
    kda_recurrent_kernel(const __grid_constant__ Params p, void* token_states) {
  __shared__ float red[4][RDV];     // per-warp column sums
  __shared__ float nrm[2][4];       // per-warp sums of squares of q, k
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
  const int dk = tid, dv0 = part * RDV;
  const size_t HD2 = (size_t)kHeadDim * kHeadDim;
  const size_t srow = ((size_t)n * H + h) * HD2 + (size_t)dk * kHeadDim + dv0;

  float S[RDV];
  if (p.initial_state) {
    if (p.state_bf16) {
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(p.initial_state) + srow);
#pragma unroll
      for (int c = 0; c < RDV / 8; ++c) {
        const uint4 w = src[c];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          S[8 * c + 2 * e] = __uint_as_float(ww[e] << 16);
          S[8 * c + 2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u);
        }
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(
          static_cast<const float*>(p.initial_state) + srow);
#pragma unroll
      for (int c = 0; c < RDV / 4; ++c) {
        const float4 w = src[c];
        S[4 * c] = w.x;
        S[4 * c + 1] = w.y;
        S[4 * c + 2] = w.z;
        S[4 * c + 3] = w.w;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < RDV; ++j) S[j] = 0.0f;
  }
  const float gsc = expf(p.A_log[h]);
  const float dtb = p.dt_bias[h * kHeadDim + dk];
  const float lbl2 = p.lower_bound * kLog2eR;

  auto store_state = [&](void* dst_base, size_t row) {
    if (p.state_bf16) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst_base) + row);
#pragma unroll
      for (int c = 0; c < RDV / 8; ++c) {
        uint32_t ww[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(S[8 * c + 2 * e], S[8 * c + 2 * e + 1]);
          ww[e] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        dst[c] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(dst_base) + row);
#pragma unroll
      for (int c = 0; c < RDV / 4; ++c)
        dst[c] = make_float4(S[4 * c], S[4 * c + 1], S[4 * c + 2], S[4 * c + 3]);
    }
  };

  for (int t = t0; t < t1; ++t) {
    const float qv = __bfloat162float(p.q[(size_t)t * p.s_q + (size_t)h * kHeadDim + dk]);
    const float kv = __bfloat162float(p.k[(size_t)t * p.s_k + (size_t)h * kHeadDim + dk]);
    const float gv = __bfloat162float(p.g[(size_t)t * p.s_g + (size_t)h * kHeadDim + dk]);
    const float bv = __bfloat162float(p.beta[(size_t)t * p.s_beta + h]);
    const float vv = (lane < RDV)
                         ? __bfloat162float(p.v[(size_t)t * p.s_v + (size_t)h * kHeadDim + dv0 + lane])
                         : 0.0f;
    // norms of q and k over the 128 key channels
    const float sq = warp_sum(qv * qv), sk = warp_sum(kv * kv);
    if (lane == 0) {
      nrm[0][warp] = sq;
      nrm[1][warp] = sk;
    }
    __syncthreads();
    const float iq = p.scale * rsqrtf((nrm[0][0] + nrm[0][1]) + (nrm[0][2] + nrm[0][3]) + kL2Eps);
    const float ik = rsqrtf((nrm[1][0] + nrm[1][1]) + (nrm[1][2] + nrm[1][3]) + kL2Eps);
    const float qh = qv * iq, kh = kv * ik;
    // decay of this key row, then the partial sums of S^T kh
    const float dec = ex2r(lbl2 * sigmoid_r(gsc * (gv + dtb)));
    float w[RDV];
#pragma unroll
    for (int j = 0; j < RDV; ++j) {
      S[j] *= dec;
      w[j] = S[j] * kh;
    }
    red[warp][lane] = reduce_scatter32(w, lane);
    __syncthreads();
    if (warp == 0) {   // u = b (v - S^T kh) for column lane
      const float stk = (red[0][lane] + red[1][lane]) + (red[2][lane] + red[3][lane]);
      ucol[lane] = sigmoid_r(bv) * (vv - stk);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < RDV; ++j) {
      S[j] = fmaf(kh, ucol[j], S[j]);
      w[j] = S[j] * qh;
    }
    red[warp][lane] = reduce_scatter32(w, lane);   // warp 0 read S^T kh before the last barrier
    __syncthreads();
    if (warp == 0) {
      const float o = (red[0][lane] + red[1][lane]) + (red[2][lane] + red[3][lane]);
      p.out[(size_t)t * H * kHeadDim + (size_t)h * kHeadDim + dv0 + lane] = __float2bfloat16_rn(o);
    }
    if (token_states)
      store_state(token_states, ((size_t)t * H + h) * HD2 + (size_t)dk * kHeadDim + dv0);
    __syncthreads();   // red and nrm are rewritten by the next token
  }
  store_state(p.final_state, srow);
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
