// tcgen05 + TMA chunked KDA prefill (KDA_KERNEL_TC), 64-token chunks.
//
// One CTA (256 threads, ~190 KB shared memory, 512 TMEM columns) owns one
// (sequence, head, value slice) and walks the sequence's chunks in order,
// keeping the 128 x 128 fp32 state in tensor memory the whole time.
//
// Per chunk (rows r, s = tokens of the chunk; Gam = inclusive cumsum of the
// log2 decay over the chunk, per key channel; qh carries `scale`):
//   A[r,s]  = b_r sum_d kh_r kh_s 2^(Gam_r - Gam_s)   (s < r)
//   QK[r,s] =     sum_d qh_r kh_s 2^(Gam_r - Gam_s)   (s <= r)
//   T = (I + A)^-1;  W = T diag(b) (kh 2^Gam);  U' = T diag(b) V
//   U = U' - W S;    O = (qh 2^Gam) S + QK U
//   S' = diag(2^Gam_last) S + (kh 2^(Gam_last - Gam))^T U
// This is the WY/UT form of the gated delta rule with the bounded gate of
// the FlashKDA prefill PR report (PR #55737, Features & motivation:
// a = lower_bound * sigmoid(exp(A_log) (g + dt_bias)), q/k l2norm and the
// beta sigmoid inside the kernel).
//
// Exponent anchoring.  exp2(Gam_r - Gam_s) is factored into a row factor
// and a column factor so the products run on tensor cores.  The chunk is
// cut into two 32-token blocks; inside block b the cumsum is anchored at
// its 16th token, so every per-element factor stays within 2^(+-16|lb|
// log2 e), inside the fp32/bf16 range for |lb| <= 5.5.  Products between
// the blocks reuse the block-1 row operand; their column operand Kc2 carries
// 2^(B0 - c_s) * 2^(alpha_1), a product of two factors <= 1, so one MMA with
// N = 96 yields the diagonal blocks (columns 0-63) and the off-diagonal
// block (columns 64-95) together.
//
// The dense products run on tcgen05 (kind::f16: bf16 operands in shared
// memory, fp32 accumulators in TMEM), transposed so that M = 128 is the
// value (or key) channel:
//   D = [Kr; Qr] [Kc; Kc2]^T                          (A and QK, M = 128, N = 96)
//   W_b^T = Kr_b^T (T diag b)_b^T  (b = 32-token block; Kr read as an MN-major
//           operand, the per-channel block factors applied when W is converted)
//   U'^T = V^T (T diag b)^T,  O^T = S^T Qg^T,  U^T += S^T (-W)^T,
//   O^T += U^T QK^T,  S^T += U^T Ke
// S^T and U^T enter the MMAs as bf16 A operands held in TMEM.
// The unit-lower-triangular inverse T runs on CUDA cores in fp32.  Inputs
// arrive by TMA; the next chunk's q/k/g (and v) are fetched while this one
// is being processed.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int C = 64;
constexpr int D = kHeadDim;
constexpr int NT = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxRankSeqs = 128;   // longest-first ordering for up to this many sequences

// ---- shared memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_INQ = 0;                  // q tile [64][128] bf16 row-major (TMA)
constexpr int OFF_INK = 16384;              // k tile
constexpr int OFF_ING = 32768;              // g tile
constexpr int OFF_INV = 49152;              // v tile: 2 SW128 boxes [64 tok][64 dv]
constexpr int OFF_RA = 65536;               // region reused within a chunk:
constexpr int OFF_RKQ = OFF_RA;             //  [Kr; Qr] K-major 128 rows x 128 (live to W)
constexpr int OFF_CKC = OFF_RA + 32768;     //  [Kc; Kc2] K-major 96 rows x 128 (live to D)
constexpr int NS = 68;                      //  fp32 row stride of the T scratch (16-B rows)
constexpr int OFF_NM = OFF_RA + 32768;      //  N = diag(b) strict(A)  [64][NS]  (after D)
constexpr int OFF_TM = OFF_NM + 64 * NS * 4;//  T                      [64][NS]
constexpr int OFF_Y = OFF_TM + 64 * NS * 4; //  products scratch       [32][36]
constexpr int OFF_WN = OFF_RA + 32768;      //  -W MN-major, N = 64 tok, K = 128 (after T)
constexpr int OFF_TB = OFF_RA + 73728;      //  T diag(b) K-major 64 x 64
constexpr int OFF_QG = OFF_RA + 81920;      // Qg K-major 64 rows x 128 (B of O^T = S^T Qg^T)
constexpr int OFF_KE = OFF_QG + 16384;      // Ke MN-major mn = dk, k = tok (B of S^T += U^T Ke)
constexpr int OFF_QKB = OFF_KE + 16384;     // QK K-major 64 x 64 (B of O^T += U^T QK^T)
constexpr int OFF_MISC = OFF_QKB + 8192;
constexpr int OFF_INVN = OFF_MISC;          // inv |q| * scale [64], inv |k| [64]
constexpr int OFF_BETA = OFF_MISC + 512;    // b [64]
constexpr int OFF_DECAY = OFF_MISC + 768;   // 2^Gam_last [128]
constexpr int OFF_WF = OFF_MISC + 1280;     // W factors [3][128]: 2^G0, 2^G2, 2^B0
constexpr int OFF_GT = OFF_MISC + 2816;     // group totals [4][128] (also sequence lengths)
constexpr int OFF_BAR = OFF_MISC + 4864;    // 3 mbarriers
constexpr int OFF_TSLOT = OFF_MISC + 4896;  // TMEM base address
constexpr int OFF_FLAGS = OFF_MISC + 4900;  // [0] sequence chosen for this CTA
constexpr int SMEM_USED = OFF_MISC + 5120;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(OFF_Y + 32 * 36 * 4 <= OFF_TB, "T scratch overlaps T diag(b)");
static_assert(OFF_CKC + 24576 <= OFF_TB, "operands overlap T diag(b)");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

// ---- TMEM columns (fp32 unless noted; lane = value channel, or key channel for D/W)
constexpr uint32_t TM_S = 0;      // S^T        128 cols (col = dk)
constexpr uint32_t TM_SB = 128;   // S^T bf16    64 cols (A operand, 2 dk per col)
constexpr uint32_t TM_U = 192;    // U^T         64 cols (col = token)
constexpr uint32_t TM_O = 256;    // O^T         64 cols
constexpr uint32_t TM_D = 320;    // D (A|QK)    96 cols, then W0^T at +0, W1^T at +64
constexpr uint32_t TM_UB = 448;   // U^T bf16    32 cols (A operand, 2 tokens per col)
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_KK64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_KK96 = idesc_bf16(128, 96, 0, 0);
constexpr uint32_t ID_MK64 = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_KM64 = idesc_bf16(128, 64, 0, 1);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, 0, 1);

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcpf(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigm(float x) { return rcpf(1.0f + ex2f(-x * kLog2e)); }

__device__ __forceinline__ void st_u32(unsigned char* base, uint32_t off, uint32_t v) {
  *reinterpret_cast<uint32_t*>(base + off) = v;
}
__device__ __forceinline__ void st_u128(unsigned char* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}
__device__ __forceinline__ float2 ld_bf16x2(const unsigned char* base, uint32_t off) {
  const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(base + off);
  return __bfloat1622float2(v);
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void fma4(float4& acc, float a, const float4& b) {
  acc.x = fmaf(a, b.x, acc.x);
  acc.y = fmaf(a, b.y, acc.y);
  acc.z = fmaf(a, b.z, acc.z);
  acc.w = fmaf(a, b.w, acc.w);
}

// K-step descriptors
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int rows, int ks) {
  return sdesc_sw128(tile + (ks >> 2) * rows * 128 + (ks & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, uint32_t lbo, int ks) {
  return sdesc_sw128(tile + ks * 2048, lbo, 1024);
}

__global__ void __launch_bounds__(NT, 1)
    kda_tc_chunk_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_g,
                        const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* inv_q = reinterpret_cast<float*>(sm + OFF_INVN);
  float* inv_k = inv_q + 64;
  float* beta_s = reinterpret_cast<float*>(sm + OFF_BETA);
  float* decay_s = reinterpret_cast<float*>(sm + OFF_DECAY);
  float* wf = reinterpret_cast<float*>(sm + OFF_WF);
  float* gt = reinterpret_cast<float*>(sm + OFF_GT);
  int* flags = reinterpret_cast<int*>(sm + OFF_FLAGS);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);
  const uint32_t bar_qkg = sb + OFF_BAR, bar_v = bar_qkg + 8, bar_mma = bar_qkg + 16;

  // ---- work unit: (rank, head, part), longest sequence first
  const int P = p.vsplit, H = p.heads, N = p.num_seqs;
  const int unit = blockIdx.x;
  const int part = unit % P;
  const int h = (unit / P) % H;
  const int rank = unit / (P * H);
  if (N <= kMaxRankSeqs) {
    int* lens = reinterpret_cast<int*>(gt);
    for (int i = tid; i < N; i += NT) lens[i] = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
    __syncthreads();
    for (int i = tid; i < N; i += NT) {
      const int li = lens[i];
      int r = 0;
      for (int m = 0; m < N; ++m) {
        const int lm = lens[m];
        r += (lm > li) || (lm == li && m < i);
      }
      if (r == rank) flags[0] = i;
    }
    __syncthreads();
  } else if (tid == 0) {
    flags[0] = rank;
  }
  __syncthreads();
  const int n = flags[0];
  const int t0 = p.cu_seqlens[n];
  const int t1 = p.cu_seqlens[n + 1];
  if (t0 < 0 || t1 < t0 || (int64_t)t1 > p.total_tokens || p.cu_seqlens[0] != 0) {
    if (tid == 0) record_error(p.status, KDA_ERR_BAD_CU_SEQLENS, 1);
    return;
  }
  const int DV = D / P;
  const int dv_lo = part * DV, dv_hi = dv_lo + DV;

  // ---- barriers and tensor memory
  if (tid == 0) {
    mbar_init(bar_qkg, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_g);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const int my_lane = 32 * (warp & 3) + lane;     // TMEM lane this thread reads
  const int half = warp >> 2;                     // warps 4-7 take the second column half

  const size_t HD = (size_t)H * D;
  const size_t sbase = ((size_t)n * H + h) * D * D;
  const int xcol = h * D;

  if (tid == 0 && t1 > t0) {
    mbar_expect_tx(bar_qkg, 3 * 16384);
    tma_load_2d(sb + OFF_INQ, &tm_q, xcol, t0, bar_qkg);
    tma_load_2d(sb + OFF_INK, &tm_k, xcol, t0, bar_qkg);
    tma_load_2d(sb + OFF_ING, &tm_g, xcol, t0, bar_qkg);
    mbar_expect_tx(bar_v, 16384);
    tma_load_2d(sb + OFF_INV, &tm_v, xcol, t0, bar_v);
    tma_load_2d(sb + OFF_INV + 8192, &tm_v, xcol + 64, t0, bar_v);
  }

  // ---- state in: S^T[dv][dk] -> TMEM (lane = dv); this thread covers 64 key columns
  {
    const int dv = my_lane;
    const bool mine = dv >= dv_lo && dv < dv_hi && p.initial_state != nullptr;
    for (int cb = 0; cb < 2; ++cb) {
      const int dk0 = half * 64 + cb * 32;
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float s = 0.0f;
        if (mine) {
          const size_t idx = sbase + (size_t)(dk0 + j) * D + dv;
          s = p.state_bf16
                  ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.initial_state)[idx])
                  : static_cast<const float*>(p.initial_state)[idx];
        }
        r[j] = __float_as_uint(s);
      }
      tmem_st32(tmem + lane_base + TM_S + dk0, r);
    }
    tmem_wait_st();
  }

  const float gate_scale = expf(p.A_log[h]);
  const float lb2 = p.lower_bound * kLog2e;
  const int cp = tid & 63;            // channel pair of the gate/operand phase
  const int grp = tid >> 6;           // 16-row group of the gate/operand phase
  const int d0 = 2 * cp;
  const float db0 = p.dt_bias[h * D + d0], db1 = p.dt_bias[h * D + d0 + 1];
  float* Nm = reinterpret_cast<float*>(sm + OFF_NM);
  float* Tm = reinterpret_cast<float*>(sm + OFF_TM);
  float* Y = reinterpret_cast<float*>(sm + OFF_Y);

  uint32_t ph_qkg = 0, ph_v = 0, ph_mma = 0;
  bool failed = false;
  int site = 0;
  // beta logits are fetched one chunk ahead (their load latency hides behind a chunk)
  float b_raw = 0.0f;
  if (tid < C && t0 + tid < t1) b_raw = __bfloat162float(p.beta[(size_t)(t0 + tid) * H + h]);

  for (int c0 = t0; c0 < t1; c0 += C) {
    const int L = min(C, t1 - c0);
    const bool more = c0 + C < t1;

    // ---- P0: q, k, g of this chunk have landed
    {
      const bool ok = mbar_wait(bar_qkg, ph_qkg);
      ph_qkg ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 10; break; }
    }

    // ---- P1: beta and the row norms of q and k (one warp per row)
    if (tid < C) {
      beta_s[tid] = (tid < L) ? sigm(b_raw) : 0.0f;
      if (c0 + C + tid < t1) b_raw = __bfloat162float(p.beta[(size_t)(c0 + C + tid) * H + h]);
    }
    for (int r = warp * 8; r < warp * 8 + 8; ++r) {
      const uint2 qv = *reinterpret_cast<const uint2*>(sm + OFF_INQ + r * 256 + lane * 8);
      const uint2 kv = *reinterpret_cast<const uint2*>(sm + OFF_INK + r * 256 + lane * 8);
      const float2 q01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qv.x));
      const float2 q23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qv.y));
      const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.x));
      const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.y));
      float sq = q01.x * q01.x + q01.y * q01.y + q23.x * q23.x + q23.y * q23.y;
      float sk = k01.x * k01.x + k01.y * k01.y + k23.x * k23.x + k23.y * k23.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      if (lane == 0) {
        inv_q[r] = (r < L) ? p.scale * rsqrtf(sq + kL2Eps) : 0.0f;
        inv_k[r] = (r < L) ? rsqrtf(sk + kL2Eps) : 0.0f;
      }
    }

    // ---- P2a: gate -> log2 decay, cumsum inside this thread's 16-row group
    float cl0[16], cl1[16];
    {
      float run0 = 0.0f, run1 = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = grp * 16 + i;
        const float2 gv = ld_bf16x2(sm + OFF_ING, (uint32_t)(r * 256 + d0 * 2));
        float a0 = lb2 * sigm(gate_scale * (gv.x + db0));
        float a1 = lb2 * sigm(gate_scale * (gv.y + db1));
        a0 = (r < L) ? a0 : 0.0f;
        a1 = (r < L) ? a1 : 0.0f;
        run0 += a0;
        run1 += a1;
        cl0[i] = run0;
        cl1[i] = run1;
      }
      gt[grp * 128 + d0] = run0;
      gt[grp * 128 + d0 + 1] = run1;
    }
    __syncthreads();

    // ---- P2b: anchored factors and the bf16 operand tiles [Kr; Qr], [Kc; Kc2], Qg, Ke
    {
      const bool blk1 = grp >= 2;
      float mE[2], cA[2], cB[2], cX[2], cR[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float G0 = gt[d0 + c], G1 = gt[128 + d0 + c];
        const float G2 = gt[256 + d0 + c], G3 = gt[384 + d0 + c];
        const float B0 = G0 + G1, B1 = G2 + G3;
        const float Gown = blk1 ? (grp == 2 ? G2 : G3) : (grp == 0 ? G0 : G1);
        mE[c] = (grp & 1) ? 0.0f : Gown;
        // block 0: cA = 2^G0 (E -> 2^Gam), cB = 2^G1 (Ei -> 2^(B0 - c)), cR = 2^B1
        // block 1: cA = 2^G2 (E -> 2^c),   cB = 2^G3 (Ei -> 2^(B1 - c)), cR = 2^B0
        cA[c] = ex2f(blk1 ? G2 : G0);
        cB[c] = ex2f(blk1 ? G3 : G1);
        cX[c] = ex2f(G2);                 // alpha_1, folded into Kc2
        cR[c] = ex2f(blk1 ? B0 : B1);
        if (grp == 0) {
          decay_s[d0 + c] = ex2f(B0 + B1);
          wf[d0 + c] = cA[c];              // W block 0: 2^G0
          wf[128 + d0 + c] = cX[c];        // W block 1: 2^G2, then
          wf[256 + d0 + c] = ex2f(B0);     //            2^B0
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = grp * 16 + i;
        const float iq = inv_q[r], ik = inv_k[r];
        const float2 qv = ld_bf16x2(sm + OFF_INQ, (uint32_t)(r * 256 + d0 * 2));
        const float2 kv = ld_bf16x2(sm + OFF_INK, (uint32_t)(r * 256 + d0 * 2));
        const bool live = r < L;
        const float qh0 = live ? qv.x * iq : 0.0f, qh1 = live ? qv.y * iq : 0.0f;
        const float kh0 = live ? kv.x * ik : 0.0f, kh1 = live ? kv.y * ik : 0.0f;
        const float e0 = cl0[i] - mE[0], e1 = cl1[i] - mE[1];
        const float E0 = ex2f(e0), E1 = ex2f(e1);
        const float Ei0 = ex2f(-e0), Ei1 = ex2f(-e1);
        st_u32(sm, OFF_RKQ + kmajor_off(r, d0, 128), pack_bf16x2(kh0 * E0, kh1 * E1));
        st_u32(sm, OFF_RKQ + kmajor_off(64 + r, d0, 128), pack_bf16x2(qh0 * E0, qh1 * E1));
        st_u32(sm, OFF_CKC + kmajor_off(r, d0, 96), pack_bf16x2(kh0 * Ei0, kh1 * Ei1));
        float g0, g1, ke0, ke1;
        if (!blk1) {
          const float oc0 = Ei0 * cB[0], oc1 = Ei1 * cB[1];    // 2^(B0 - c_s)
          st_u32(sm, OFF_CKC + kmajor_off(64 + r, d0, 96),
                 pack_bf16x2(kh0 * (oc0 * cX[0]), kh1 * (oc1 * cX[1])));
          g0 = E0 * cA[0];
          g1 = E1 * cA[1];
          ke0 = oc0 * cR[0];
          ke1 = oc1 * cR[1];
        } else {
          g0 = (E0 * cA[0]) * cR[0];
          g1 = (E1 * cA[1]) * cR[1];
          ke0 = Ei0 * cB[0];
          ke1 = Ei1 * cB[1];
        }
        st_u32(sm, OFF_QG + kmajor_off(r, d0, 64), pack_bf16x2(qh0 * g0, qh1 * g1));
        st_u32(sm, OFF_KE + mnmajor_off(d0, r, 8192), pack_bf16x2(kh0 * ke0, kh1 * ke1));
      }
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P3: D = [Kr; Qr] [Kc; Kc2]^T on the tensor cores; fetch the next q, k, g.
    //          Warps 4-7 meanwhile make the bf16 copy of S^T and apply this chunk's decay.
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + TM_D, kdesc(sb + OFF_RKQ, 128, ks), kdesc(sb + OFF_CKC, 96, ks), ID_KK96,
                 ks > 0);
      mma_commit(bar_mma);
      if (more) {
        mbar_expect_tx(bar_qkg, 3 * 16384);
        tma_load_2d(sb + OFF_INQ, &tm_q, xcol, c0 + C, bar_qkg);
        tma_load_2d(sb + OFF_INK, &tm_k, xcol, c0 + C, bar_qkg);
        tma_load_2d(sb + OFF_ING, &tm_g, xcol, c0 + C, bar_qkg);
      }
    }
    if (half == 1) {
      for (int cb = 0; cb < 4; ++cb) {      // 32 key columns per pass
        uint32_t x[32], pk[16];
        tmem_ld32(tmem + lane_base + TM_S + cb * 32, x);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
        tmem_st16(tmem + lane_base + TM_SB + cb * 16, pk);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 dl = ld4(decay_s + cb * 32 + 4 * j4);
          x[4 * j4] = __float_as_uint(__uint_as_float(x[4 * j4]) * dl.x);
          x[4 * j4 + 1] = __float_as_uint(__uint_as_float(x[4 * j4 + 1]) * dl.y);
          x[4 * j4 + 2] = __float_as_uint(__uint_as_float(x[4 * j4 + 2]) * dl.z);
          x[4 * j4 + 3] = __float_as_uint(__uint_as_float(x[4 * j4 + 3]) * dl.w);
        }
        tmem_st32(tmem + lane_base + TM_S + cb * 32, x);
      }
      tmem_wait_st();
    }
    {
      const bool ok = mbar_wait(bar_mma, ph_mma) && mbar_wait(bar_v, ph_v);
      ph_mma ^= 1;
      ph_v ^= 1;
      tc_fence_before();
      if (__syncthreads_or(!ok)) { failed = true; site = 30; break; }
    }
    tc_fence_after();

    // ---- P4a: A rows (lanes 0-63) -> N = diag(b) strict(A); QK rows (64-127) -> bf16 tile;
    //            warps 4-7 clear v rows past the sequence end and T above the diagonal blocks
    if (half == 0) {
      // columns 0-31 come from D[:, 64:96] for rows 32-63 (the off-diagonal block)
      const int r = my_lane & 63;
      const bool use2 = r >= 32;
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + TM_D + ((cb == 0 && use2) ? 64 : 32 * cb), a);
        tmem_wait_ld();
        if (warp < 2) {
          const float br = beta_s[r];
#pragma unroll
          for (int s4 = 0; s4 < 8; ++s4) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int s = 32 * cb + 4 * s4 + e;
              v[e] = (s < r) ? br * __uint_as_float(a[4 * s4 + e]) : 0.0f;
            }
            *reinterpret_cast<float4*>(Nm + r * NS + 32 * cb + 4 * s4) =
                make_float4(v[0], v[1], v[2], v[3]);
          }
        } else {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int s = 32 * cb + c8 * 8 + e * 2;
              w[e] = pack_bf16x2(s <= r ? __uint_as_float(a[c8 * 8 + e * 2]) : 0.0f,
                                 s + 1 <= r ? __uint_as_float(a[c8 * 8 + e * 2 + 1]) : 0.0f);
            }
            st_u128(sm, OFF_QKB + kmajor_off(r, 32 * cb + c8 * 8, 64),
                    make_uint4(w[0], w[1], w[2], w[3]));
          }
        }
      }
    } else {
      const int t4 = tid - 128;
      if (L < C) {   // v rows past the sequence end -> 0 (both 64-column boxes)
        for (int idx = t4; idx < (C - L) * 16; idx += 128) {
          const int r = L + idx / 16, cc = idx % 16;
          st_u128(sm, OFF_INV + (cc >> 3) * 8192 + r * 128 + (cc & 7) * 16, make_uint4(0, 0, 0, 0));
        }
      }
      // T above the diagonal 16x16 blocks is zero
      for (int idx = t4; idx < 6 * 64; idx += 128) {
        const int b = idx >> 6, e = idx & 63;
        const int bi = (b < 3) ? 0 : (b < 5 ? 1 : 2);
        const int bj = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
        *reinterpret_cast<float4*>(Tm + (bi * 16 + (e >> 2)) * NS + bj * 16 + 4 * (e & 3)) =
            make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- P4b: T = (I + N)^-1, blocked: 16x16 diagonal blocks, then 32, then 64
    if (tid < 64) {
      const int o = (tid >> 4) * 16, j = tid & 15;
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float acc = (i == j) ? 1.0f : 0.0f;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          if (4 * q4 < i) {
            const float4 nv = ld4(Nm + (o + i) * NS + o + 4 * q4);
            if (4 * q4 + 0 < i) acc -= nv.x * x[4 * q4 + 0];
            if (4 * q4 + 1 < i) acc -= nv.y * x[4 * q4 + 1];
            if (4 * q4 + 2 < i) acc -= nv.z * x[4 * q4 + 2];
            if (4 * q4 + 3 < i) acc -= nv.w * x[4 * q4 + 3];
          }
        }
        x[i] = acc;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) Tm[(o + i) * NS + o + j] = x[i];
    }
    __syncthreads();
    if (tid < 128) {   // Y_b = N[rows of b] T[diag block of b], pairs b = (1,0) and (3,2)
      const int b = tid >> 6, i = (tid >> 2) & 15, jq = tid & 3;
      const int ro = (2 * b + 1) * 16, co = 2 * b * 16;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const float4 nv = ld4(Nm + (ro + i) * NS + co + 4 * s4);
        fma4(acc, nv.x, ld4(Tm + (co + 4 * s4 + 0) * NS + co + 4 * jq));
        fma4(acc, nv.y, ld4(Tm + (co + 4 * s4 + 1) * NS + co + 4 * jq));
        fma4(acc, nv.z, ld4(Tm + (co + 4 * s4 + 2) * NS + co + 4 * jq));
        fma4(acc, nv.w, ld4(Tm + (co + 4 * s4 + 3) * NS + co + 4 * jq));
      }
      *reinterpret_cast<float4*>(Y + (b * 16 + i) * 20 + 4 * jq) = acc;
    }
    __syncthreads();
    if (tid < 128) {   // T[lower of b] = -T[diag of b, rows] Y_b
      const int b = tid >> 6, i = (tid >> 2) & 15, jq = tid & 3;
      const int ro = (2 * b + 1) * 16, co = 2 * b * 16;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const float4 tv = ld4(Tm + (ro + i) * NS + ro + 4 * s4);
        fma4(acc, tv.x, ld4(Y + (b * 16 + 4 * s4 + 0) * 20 + 4 * jq));
        fma4(acc, tv.y, ld4(Y + (b * 16 + 4 * s4 + 1) * 20 + 4 * jq));
        fma4(acc, tv.z, ld4(Y + (b * 16 + 4 * s4 + 2) * 20 + 4 * jq));
        fma4(acc, tv.w, ld4(Y + (b * 16 + 4 * s4 + 3) * 20 + 4 * jq));
      }
      *reinterpret_cast<float4*>(Tm + (ro + i) * NS + co + 4 * jq) =
          make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
    {   // Y2 = N[32:64, 0:32] T[0:32, 0:32]
      const int i = tid >> 3, jq = tid & 7;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s4 = 0; s4 < 8; ++s4) {
        const float4 nv = ld4(Nm + (32 + i) * NS + 4 * s4);
        fma4(acc, nv.x, ld4(Tm + (4 * s4 + 0) * NS + 4 * jq));
        fma4(acc, nv.y, ld4(Tm + (4 * s4 + 1) * NS + 4 * jq));
        fma4(acc, nv.z, ld4(Tm + (4 * s4 + 2) * NS + 4 * jq));
        fma4(acc, nv.w, ld4(Tm + (4 * s4 + 3) * NS + 4 * jq));
      }
      *reinterpret_cast<float4*>(Y + i * 36 + 4 * jq) = acc;
    }
    __syncthreads();
    {   // T[32:64, 0:32] = -T[32:64, 32:64] Y2
      const int i = tid >> 3, jq = tid & 7;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s4 = 0; s4 < 8; ++s4) {
        const float4 tv = ld4(Tm + (32 + i) * NS + 32 + 4 * s4);
        fma4(acc, tv.x, ld4(Y + (4 * s4 + 0) * 36 + 4 * jq));
        fma4(acc, tv.y, ld4(Y + (4 * s4 + 1) * 36 + 4 * jq));
        fma4(acc, tv.z, ld4(Y + (4 * s4 + 2) * 36 + 4 * jq));
        fma4(acc, tv.w, ld4(Y + (4 * s4 + 3) * 36 + 4 * jq));
      }
      *reinterpret_cast<float4*>(Tm + (32 + i) * NS + 4 * jq) =
          make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
    }
    __syncthreads();
    // T diag(b) -> bf16 (K-major, row r, k = s)
    for (int idx = tid; idx < 512; idx += NT) {
      const int r = idx >> 3, c8 = idx & 7;
      const float4 t0v = ld4(Tm + r * NS + c8 * 8), t1v = ld4(Tm + r * NS + c8 * 8 + 4);
      const float4 b0v = ld4(beta_s + c8 * 8), b1v = ld4(beta_s + c8 * 8 + 4);
      st_u128(sm, OFF_TB + kmajor_off(r, c8 * 8, 64),
              make_uint4(pack_bf16x2(t0v.x * b0v.x, t0v.y * b0v.y),
                         pack_bf16x2(t0v.z * b0v.z, t0v.w * b0v.w),
                         pack_bf16x2(t1v.x * b1v.x, t1v.y * b1v.y),
                         pack_bf16x2(t1v.z * b1v.z, t1v.w * b1v.w)));
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P5: W_b^T = (Kr rows of block b)^T (T diag b)[:, b]^T for b = 0, 1 (D region);
    //          U'^T = V^T (T diag b)^T;  O^T = S^T Qg^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma_bf16(tmem + TM_D + 64 * b, mndesc(sb + OFF_RKQ + 4096 * b, 16384, ks),
                   kdesc(sb + OFF_TB, 64, 2 * b + ks), ID_MK64, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + TM_U, mndesc(sb + OFF_INV, 8192, ks), kdesc(sb + OFF_TB, 64, ks),
                 ID_MK64, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16_ts(tmem + TM_O, tmem + TM_SB + 8 * ks, kdesc(sb + OFF_QG, 64, ks), ID_KK64,
                    ks > 0);
      mma_commit(bar_mma);
    }
    {
      const bool ok = mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 50; break; }
    }
    tc_fence_after();
    if (tid == 0 && more) {   // v tile is free again
      mbar_expect_tx(bar_v, 16384);
      tma_load_2d(sb + OFF_INV, &tm_v, xcol, c0 + C, bar_v);
      tma_load_2d(sb + OFF_INV + 8192, &tm_v, xcol + 64, c0 + C, bar_v);
    }

    // ---- P6: -W = -(2^G0 W0 + 2^B0 (2^G2 W1)) -> bf16, MN-major (n = token, k = dk)
    {
      const int dk = my_lane;
      const float f0 = wf[dk], f1a = wf[128 + dk], f1b = wf[256 + dk];
      uint32_t w0[32], w1[32];
      tmem_ld32(tmem + lane_base + TM_D + half * 32, w0);
      tmem_ld32(tmem + lane_base + TM_D + 64 + half * 32, w1);
      tmem_wait_ld();
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = c8 * 8 + e * 2;
          const float x0 = f0 * __uint_as_float(w0[j]) + f1b * (f1a * __uint_as_float(w1[j]));
          const float x1 =
              f0 * __uint_as_float(w0[j + 1]) + f1b * (f1a * __uint_as_float(w1[j + 1]));
          w[e] = pack_bf16x2(-x0, -x1);
        }
        st_u128(sm, OFF_WN + mnmajor_off(half * 32 + c8 * 8, dk, 8192),
                make_uint4(w[0], w[1], w[2], w[3]));
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- P7: U^T += S^T (-W)^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16_ts(tmem + TM_U, tmem + TM_SB + 8 * ks, mndesc(sb + OFF_WN, 8192, ks), ID_KM64,
                    1);
      mma_commit(bar_mma);
    }
    {
      const bool ok = mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 70; break; }
    }
    tc_fence_after();

    // ---- P8: U^T -> bf16 operand in TMEM (2 tokens per column)
    {   // 8 warps: lane quadrant x half of the 64 token columns
      uint32_t x[32], pk[16];
      tmem_ld32(tmem + lane_base + TM_U + half * 32, x);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
      tmem_st16(tmem + lane_base + TM_UB + half * 16, pk);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();

    // ---- P9: O^T += U^T QK^T;  S^T += U^T Ke
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ts(tmem + TM_O, tmem + TM_UB + 8 * ks, kdesc(sb + OFF_QKB, 64, ks), ID_KK64, 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ts(tmem + TM_S, tmem + TM_UB + 8 * ks, mndesc(sb + OFF_KE, 8192, ks), ID_KM128,
                    1);
      mma_commit(bar_mma);
    }
    {
      const bool ok = mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 90; break; }
    }
    tc_fence_after();

    // ---- P10: O^T -> bf16 -> global rows < L of this value slice (32 tokens per warp)
    {
      const int dv = my_lane;
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + TM_O + half * 32, r);
      tmem_wait_ld();
      if (dv >= dv_lo && dv < dv_hi) {
        __nv_bfloat16* op = p.out + (size_t)(c0 + half * 32) * HD + xcol + dv;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (half * 32 + j < L) op[(size_t)j * HD] = __float2bfloat16_rn(__uint_as_float(r[j]));
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (failed) {
    if (tid == 0) record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
    // let copies still in flight finish (bounded) before the CTA exits
    mbar_wait(bar_qkg, ph_qkg);
    mbar_wait(bar_v, ph_v);
    mbar_wait(bar_mma, ph_mma);
  } else {
    // ---- state out (slice columns only)
    const int dv = my_lane;
    const bool mine = dv >= dv_lo && dv < dv_hi;
    for (int cb = 0; cb < 2; ++cb) {
      const int dk0 = half * 64 + cb * 32;
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + TM_S + dk0, r);
      tmem_wait_ld();
      if (mine) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const size_t idx = sbase + (size_t)(dk0 + j) * D + dv;
          const float s = __uint_as_float(r[j]);
          if (p.state_bf16)
            static_cast<__nv_bfloat16*>(p.final_state)[idx] = __float2bfloat16_rn(s);
          else
            static_cast<float*>(p.final_state)[idx] = s;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  }
  return fn;
}

// A [T rows][H*128 cols] bf16 view of q/k/g/v; box {box_cols, 64 rows}.
bool make_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, int64_t T, int H,
              int box_cols, bool swizzle) {
  cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)H * D * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)C};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc(const Params& p, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(kda_tc_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long blocks = (long long)p.num_seqs * p.heads * p.vsplit;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mg, mv;
  // Zero-token launches still need valid maps: point them at any 16-byte
  // aligned address; no tile is ever loaded then.
  const void* qb = p.q ? (const void*)p.q : (const void*)p.dt_bias;
  const void* kb = p.k ? (const void*)p.k : (const void*)p.dt_bias;
  const void* gb = p.g ? (const void*)p.g : (const void*)p.dt_bias;
  const void* vb = p.v ? (const void*)p.v : (const void*)p.dt_bias;
  if (!make_map(enc, &mq, qb, p.total_tokens, p.heads, D, false) ||
      !make_map(enc, &mk, kb, p.total_tokens, p.heads, D, false) ||
      !make_map(enc, &mg, gb, p.total_tokens, p.heads, D, false) ||
      !make_map(enc, &mv, vb, p.total_tokens, p.heads, 64, true))
    return cudaErrorInvalidValue;
  kda_tc_chunk_kernel<<<(unsigned)blocks, NT, SMEM_BYTES, stream>>>(p, mq, mk, mg, mv);
  return cudaGetLastError();
}

}  // namespace kda
