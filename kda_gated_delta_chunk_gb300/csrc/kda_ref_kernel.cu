// Plain-CUDA-core chunked KDA prefill (KDA_KERNEL_REF).
//
// A deliberately simple kernel: fp32 throughout, chunks of 32 tokens, every
// decay factor exp2(Gam_r - Gam_s) formed element by element (so no exponent
// anchoring is needed), no tensor cores and no pipelining.  It exists to
// check the library's plumbing and the chunk algebra on the GPU
// independently of the tcgen05 kernel; it is not the fast path.
//
// Chunk algebra (per sequence n, head h, chunk of L tokens, state S entering
// it; Gam = inclusive cumsum over the chunk of the log2 decay per key
// channel; qh already carries `scale`):
//   A[r,s]  = b_r sum_d kh_r kh_s 2^(Gam_r - Gam_s)   (s < r)
//   QK[r,s] =     sum_d qh_r kh_s 2^(Gam_r - Gam_s)   (s <= r)
//   T  = (I + A)^-1;  W = T diag(b) (kh 2^Gam);  U = T diag(b) V - W S
//   O  = (qh 2^Gam) S + QK U
//   S' = diag(2^Gam_last) S + (kh 2^(Gam_last - Gam))^T U
// The gate is the one of the FlashKDA prefill PR report (PR #55737,
// Features & motivation): a = lower_bound * sigmoid(exp(A_log) (g + dt_bias)).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int RC = 32;        // chunk length
constexpr int RT = 256;       // threads per CTA
constexpr int D = kHeadDim;
constexpr int DP = D + 1;     // padded row stride (bank spread for row-varying reads)
constexpr float kLog2e = 1.4426950408889634f;

struct RefSmem {
  float qh[RC][DP];     // scale * q / |q|, then qh * 2^Gam
  float kh[RC][DP];     // k / |k|, then kh * 2^(Gam_last - Gam)
  float gam[RC][DP];    // log2 decay, then its inclusive cumsum
  float vv[RC][D];      // v (value slice)
  float kb[RC][D];      // b * kh * 2^Gam
  float w[RC][D];       // W = T kb
  float u[RC][D];       // U
  float A[RC][RC + 1];
  float Tm[RC][RC + 1];
  float QK[RC][RC + 1];
  float b[RC];
  float S[D][D];        // state slice [key channel][value column]
};

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

__global__ void __launch_bounds__(RT, 1) kda_ref_chunk_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RefSmem& sm = *reinterpret_cast<RefSmem*>(smem_raw);

  const int P = p.vsplit;
  const int DV = D / P;
  const int H = p.heads;
  const int unit = blockIdx.x;
  const int part = unit % P;
  const int h = (unit / P) % H;
  const int n = unit / (P * H);
  const int dv0 = part * DV;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  const int64_t t0 = p.cu_seqlens[n];
  const int64_t t1 = p.cu_seqlens[n + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.total_tokens || (n == 0 && t0 != 0)) {
    if (tid == 0) record_error(p.status, KDA_ERR_BAD_CU_SEQLENS, 1);
    return;
  }

  // state slice in
  const size_t sbase = ((size_t)n * H + h) * D * D;
  for (int i = tid; i < D * DV; i += RT) {
    const int d = i / DV, c = i % DV;
    float s = 0.0f;
    if (p.initial_state) {
      const size_t idx = sbase + (size_t)d * D + dv0 + c;
      s = p.state_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.initial_state)[idx])
                       : static_cast<const float*>(p.initial_state)[idx];
    }
    sm.S[d][c] = s;
  }

  const float gate_scale = expf(p.A_log[h]);
  const float lb2 = p.lower_bound * kLog2e;
  const size_t HD = (size_t)H * D;

  for (int64_t c0 = t0; c0 < t1; c0 += RC) {
    const int L = (t1 - c0 < RC) ? (int)(t1 - c0) : RC;
    __syncthreads();   // previous chunk fully consumed

    // 1. l2norm of q and k (one warp per row), v slice, gate, beta
    for (int r = warp; r < RC; r += RT / 32) {
      float qv[4], kv[4];
      float sq = 0.f, sk = 0.f;
      for (int j = 0; j < 4; ++j) {
        const int d = lane * 4 + j;
        qv[j] = kv[j] = 0.f;
        if (r < L) {
          const size_t off = (size_t)h * D + d;
          qv[j] = __bfloat162float(p.q[(size_t)(c0 + r) * p.s_q + off]);
          kv[j] = __bfloat162float(p.k[(size_t)(c0 + r) * p.s_k + off]);
        }
        sq += qv[j] * qv[j];
        sk += kv[j] * kv[j];
      }
      for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      const float iq = p.scale / sqrtf(sq + kL2Eps);
      const float ik = 1.0f / sqrtf(sk + kL2Eps);
      for (int j = 0; j < 4; ++j) {
        sm.qh[r][lane * 4 + j] = qv[j] * iq;
        sm.kh[r][lane * 4 + j] = kv[j] * ik;
      }
    }
    for (int i = tid; i < RC * D; i += RT) {
      const int r = i / D, d = i % D;
      float a2 = 0.f, vvv = 0.f;
      if (r < L) {
        const size_t idx = (size_t)(c0 + r) * p.s_g + (size_t)h * D + d;
        a2 = lb2 * sigmoidf_(gate_scale * (__bfloat162float(p.g[idx]) + p.dt_bias[h * D + d]));
        if (d < DV) vvv = __bfloat162float(p.v[(size_t)(c0 + r) * p.s_v + (size_t)h * D + dv0 + d]);
      }
      sm.gam[r][d] = a2;
      if (d < DV) sm.vv[r][d] = vvv;
    }
    if (tid < RC)
      sm.b[tid] = tid < L ? sigmoidf_(__bfloat162float(p.beta[(size_t)(c0 + tid) * p.s_beta + h])) : 0.f;
    __syncthreads();

    // 2. inclusive cumsum of the log2 decay over the chunk, per key channel
    if (tid < D) {
      float acc = 0.f;
      for (int r = 0; r < RC; ++r) {
        acc += sm.gam[r][tid];
        sm.gam[r][tid] = acc;
      }
    }
    __syncthreads();

    // 3. decay-weighted products A (strict lower, scaled by b_r) and QK (lower)
    for (int i = tid; i < RC * RC; i += RT) {
      const int r = i / RC, s = i % RC;
      float akk = 0.f, aqk = 0.f;
      if (s <= r) {
        for (int d = 0; d < D; ++d) {
          const float f = exp2f(sm.gam[r][d] - sm.gam[s][d]);
          const float ks = sm.kh[s][d] * f;
          akk += sm.kh[r][d] * ks;
          aqk += sm.qh[r][d] * ks;
        }
      }
      sm.A[r][s] = (s < r) ? sm.b[r] * akk : 0.f;
      sm.QK[r][s] = aqk;
    }
    __syncthreads();

    // 4. T = (I + A)^-1 by forward substitution, one column per thread;
    //    meanwhile kb = b * kh * 2^Gam
    if (tid < RC) {
      const int j = tid;
      float x[RC];
#pragma unroll
      for (int r = 0; r < RC; ++r) {
        float acc = (r == j) ? 1.f : 0.f;
        for (int s = j; s < r; ++s) acc -= sm.A[r][s] * x[s];
        x[r] = (r < j) ? 0.f : acc;
      }
#pragma unroll
      for (int r = 0; r < RC; ++r) sm.Tm[r][j] = x[r];
    }
    for (int i = tid; i < RC * D; i += RT) {
      const int s = i / D, d = i % D;
      sm.kb[s][d] = sm.b[s] * sm.kh[s][d] * exp2f(sm.gam[s][d]);
    }
    __syncthreads();

    // 5. W = T kb;  U = T diag(b) V;  qh <- qh * 2^Gam
    for (int i = tid; i < RC * D; i += RT) {
      const int r = i / D, d = i % D;
      float acc = 0.f;
      for (int s = 0; s <= r; ++s) acc += sm.Tm[r][s] * sm.kb[s][d];
      sm.w[r][d] = acc;
      if (d < DV) {
        float au = 0.f;
        for (int s = 0; s <= r; ++s) au += sm.Tm[r][s] * sm.b[s] * sm.vv[s][d];
        sm.u[r][d] = au;
      }
      sm.qh[r][d] *= exp2f(sm.gam[r][d]);
    }
    __syncthreads();

    // 6. U -= W S
    for (int i = tid; i < RC * DV; i += RT) {
      const int r = i / DV, c = i % DV;
      float acc = 0.f;
      for (int d = 0; d < D; ++d) acc += sm.w[r][d] * sm.S[d][c];
      sm.u[r][c] -= acc;
    }
    __syncthreads();

    // 7. O = (qh 2^Gam) S + QK U  -> out;  kh <- kh * 2^(Gam_last - Gam)
    for (int i = tid; i < RC * DV; i += RT) {
      const int r = i / DV, c = i % DV;
      if (r < L) {
        float acc = 0.f;
        for (int d = 0; d < D; ++d) acc += sm.qh[r][d] * sm.S[d][c];
        for (int s = 0; s <= r; ++s) acc += sm.QK[r][s] * sm.u[s][c];
        const int64_t row = out_row(p, c0 + r);
        if (row >= 0) p.out[(size_t)row * HD + (size_t)h * D + dv0 + c] = __float2bfloat16_rn(acc);
      }
    }
    for (int i = tid; i < RC * D; i += RT) {
      const int s = i / D, d = i % D;
      sm.kh[s][d] *= exp2f(sm.gam[RC - 1][d] - sm.gam[s][d]);
    }
    __syncthreads();

    // 8. S = diag(2^Gam_last) S + kend^T U
    for (int i = tid; i < D * DV; i += RT) {
      const int d = i / DV, c = i % DV;
      float acc = exp2f(sm.gam[RC - 1][d]) * sm.S[d][c];
      for (int s = 0; s < RC; ++s) acc += sm.kh[s][d] * sm.u[s][c];
      sm.S[d][c] = acc;
    }
  }
  __syncthreads();

  // state slice out
  for (int i = tid; i < D * DV; i += RT) {
    const int d = i / DV, c = i % DV;
    const size_t idx = sbase + (size_t)d * D + dv0 + c;
    if (p.state_bf16)
      static_cast<__nv_bfloat16*>(p.final_state)[idx] = __float2bfloat16_rn(sm.S[d][c]);
    else
      static_cast<float*>(p.final_state)[idx] = sm.S[d][c];
  }
}

}  // namespace

cudaError_t launch_ref(const Params& p, cudaStream_t stream) {
  const int smem = (int)sizeof(RefSmem);
  cudaError_t e = cudaFuncSetAttribute(kda_ref_chunk_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.num_seqs * p.heads * p.vsplit;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  kda_ref_chunk_kernel<<<(unsigned)blocks, RT, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
