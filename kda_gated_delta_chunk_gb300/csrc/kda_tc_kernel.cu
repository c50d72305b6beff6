// tcgen05 + TMA chunked KDA prefill (KDA_KERNEL_TC), 64-token chunks.
//
// One CTA (256 threads, ~213 KB shared memory, 512 TMEM columns) owns one
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
//   W^T = Kg^T (T diag b)^T,  U'^T = V^T (T diag b)^T
//   U^T += S^T (-W)^T,  O^T = S^T Qg^T,  O^T += U^T QK^T,  S^T += U^T Ke
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
constexpr int OFF_RA = 65536;               // region A (88 KB), reused within a chunk:
constexpr int OFF_RKQ = OFF_RA;             //  [Kr; Qr]  K-major, 128 rows x 128
constexpr int OFF_CKC = OFF_RA + 32768;     //  [Kc; Kc2] K-major,  96 rows x 128
constexpr int OFF_TB = OFF_RA;              //  T diag(b) K-major,  64 rows x 64
constexpr int OFF_WN = OFF_RA + 8192;       //  -W        MN-major, N = 64 tok, K = 128
constexpr int OFF_SB = OFF_RA + 24576;      //  S^T bf16  K-major, 128 rows x 128
constexpr int OFF_UB = OFF_RA + 57344;      //  U^T bf16  K-major, 128 rows x 64
constexpr int OFF_OST = OFF_RA + 73728;     //  O staging [64][128] bf16 row-major
constexpr int OFF_NM = OFF_RA + 24576;      //  fp32 N = diag(b) strict(A)  [64][65]
constexpr int OFF_TM = OFF_NM + 16640;      //  fp32 T                      [64][65]
constexpr int OFF_Y = OFF_TM + 16640;       //  fp32 scratch (2x16x17 and 32x33)
constexpr int OFF_QG = OFF_RA + 90112;      // Qg  K-major 64 rows x 128   (B of O = S^T Qg^T)
constexpr int OFF_KG = OFF_QG + 16384;      // Kg  MN-major mn = dk, k = tok (A of W^T)
constexpr int OFF_KE = OFF_KG + 16384;      // Ke  MN-major mn = dk, k = tok (B of S^T += U^T Ke)
constexpr int OFF_QKB = OFF_KE + 16384;     // QK  K-major 64 rows x 64    (B of O^T += U^T QK^T)
constexpr int OFF_MISC = OFF_QKB + 8192;
constexpr int OFF_INVN = OFF_MISC;          // inv |q| * scale [64], inv |k| [64]
constexpr int OFF_BETA = OFF_MISC + 512;    // b [64]
constexpr int OFF_DECAY = OFF_MISC + 768;   // 2^Gam_last [128]
constexpr int OFF_GT = OFF_MISC + 1280;     // group totals [4][128] (also sequence lengths)
constexpr int OFF_BAR = OFF_MISC + 3328;    // 3 mbarriers
constexpr int OFF_TSLOT = OFF_MISC + 3360;  // TMEM base address
constexpr int OFF_FLAGS = OFF_MISC + 3364;  // [0] sequence chosen for this CTA
constexpr int SMEM_USED = OFF_MISC + 3584;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(OFF_Y + 6400 <= OFF_RA + 73728, "T scratch overlaps O staging");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

// ---- TMEM columns (fp32 accumulators; lane = value or key channel)
constexpr uint32_t TM_S = 0;      // S^T   128 cols (lane = dv, col = dk)
constexpr uint32_t TM_U = 128;    // U^T    64 cols (lane = dv, col = token)
constexpr uint32_t TM_O = 192;    // O^T    64 cols
constexpr uint32_t TM_D1 = 256;   // D      96 cols (lanes 0-63: A, 64-127: QK); then W^T
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
  const int col_half = warp >> 2;                 // warps 4-7 take the second half of columns

  const size_t HD = (size_t)H * D;
  const size_t sbase = ((size_t)n * H + h) * D * D;
  const int xcol = h * D;

  // first chunk's tiles
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
      const int dk0 = col_half * 64 + cb * 32;
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

    // ---- P2b: anchored factors and the bf16 operand tiles
    {
      float G[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        G[j][0] = gt[j * 128 + d0];
        G[j][1] = gt[j * 128 + d0 + 1];
      }
      const bool blk1 = grp >= 2;
      float mE[2], cA[2], cB[2], cX[2];
      for (int c = 0; c < 2; ++c) {
        const float B0 = G[0][c] + G[1][c], B1 = G[2][c] + G[3][c];
        mE[c] = (grp & 1) ? 0.0f : G[grp][c];
        // block 0: cA = 2^G0 (row -> 2^Gam), cB = 2^G1 (col -> 2^(B0 - c)), then 2^B1
        // block 1: cA = 2^G2 (row -> 2^c),   cB = 2^G3 (col -> 2^(B1 - c)), then 2^B0
        cA[c] = ex2f(blk1 ? G[2][c] : G[0][c]);
        cB[c] = ex2f(blk1 ? G[3][c] : G[1][c]);
        cX[c] = ex2f(G[2][c]);            // alpha_1, folded into Kc2
        if (grp == 0) decay_s[d0 + c] = ex2f(B0 + B1);
        G[0][c] = ex2f(blk1 ? B0 : B1);   // reuse: the cross-block factor
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
          ke0 = oc0 * G[0][0];
          ke1 = oc1 * G[0][1];
        } else {
          const float orw0 = E0 * cA[0], orw1 = E1 * cA[1];     // 2^c_r in block 1
          g0 = orw0 * G[0][0];
          g1 = orw1 * G[0][1];
          ke0 = Ei0 * cB[0];
          ke1 = Ei1 * cB[1];
        }
        st_u32(sm, OFF_QG + kmajor_off(r, d0, 64), pack_bf16x2(qh0 * g0, qh1 * g1));
        st_u32(sm, OFF_KG + mnmajor_off(d0, r, 8192), pack_bf16x2(kh0 * g0, kh1 * g1));
        st_u32(sm, OFF_KE + mnmajor_off(d0, r, 8192), pack_bf16x2(kh0 * ke0, kh1 * ke1));
      }
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P3: D = [Kr; Qr] [Kc; Kc2]^T on the tensor cores; fetch the next q, k, g
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + TM_D1, kdesc(sb + OFF_RKQ, 128, ks), kdesc(sb + OFF_CKC, 96, ks), ID_KK96,
                 ks > 0);
      mma_commit(bar_mma);
      if (more) {
        mbar_expect_tx(bar_qkg, 3 * 16384);
        tma_load_2d(sb + OFF_INQ, &tm_q, xcol, c0 + C, bar_qkg);
        tma_load_2d(sb + OFF_INK, &tm_k, xcol, c0 + C, bar_qkg);
        tma_load_2d(sb + OFF_ING, &tm_g, xcol, c0 + C, bar_qkg);
      }
    }
    {
      const bool ok = mbar_wait(bar_mma, ph_mma) && mbar_wait(bar_v, ph_v);
      ph_mma ^= 1;
      ph_v ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 30; break; }
    }
    tc_fence_after();

    // ---- P4a: A rows (lanes 0-63) -> N = diag(b) strict(A); QK rows (64-127) -> bf16 tile;
    //            warps 4-7 clear v rows past the sequence end and T above the diagonal blocks
    float* Nm = reinterpret_cast<float*>(sm + OFF_NM);
    float* Tm = reinterpret_cast<float*>(sm + OFF_TM);
    if (warp < 4) {
      uint32_t a[64], o2[32];
      tmem_ld32(tmem + lane_base + TM_D1, *reinterpret_cast<uint32_t(*)[32]>(a));
      tmem_ld32(tmem + lane_base + TM_D1 + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
      tmem_ld32(tmem + lane_base + TM_D1 + 64, o2);
      tmem_wait_ld();
      const int r = my_lane & 63;
      const bool use2 = r >= 32;
      if (warp < 2) {
        const float br = beta_s[r];
#pragma unroll
        for (int s = 0; s < 64; ++s) {
          const float v = (s < 32 && use2) ? __uint_as_float(o2[s]) : __uint_as_float(a[s]);
          Nm[r * 65 + s] = (s < r) ? br * v : 0.0f;
        }
      } else {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = c8 * 8 + e * 2;
            const float v0 = (s < 32 && use2) ? __uint_as_float(o2[s]) : __uint_as_float(a[s]);
            const float v1 =
                (s + 1 < 32 && use2) ? __uint_as_float(o2[s + 1]) : __uint_as_float(a[s + 1]);
            w[e] = pack_bf16x2(s <= r ? v0 : 0.0f, s + 1 <= r ? v1 : 0.0f);
          }
          st_u128(sm, OFF_QKB + kmajor_off(r, c8 * 8, 64), make_uint4(w[0], w[1], w[2], w[3]));
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
      // T above the diagonal blocks is zero
      for (int idx = t4; idx < 6 * 256; idx += 128) {
        const int b = idx >> 8, e = idx & 255;
        const int bi = (b < 3) ? 0 : (b < 5 ? 1 : 2);
        const int bj = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
        Tm[(bi * 16 + (e >> 4)) * 65 + bj * 16 + (e & 15)] = 0.0f;
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
        for (int s = 0; s < i; ++s) acc -= Nm[(o + i) * 65 + o + s] * x[s];
        x[i] = acc;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) Tm[(o + i) * 65 + o + j] = x[i];
    }
    __syncthreads();
    float* Y = reinterpret_cast<float*>(sm + OFF_Y);
    {   // Y_b = N[lower of pair b] T[upper of pair b], pairs (1,0) and (3,2)
      for (int idx = tid; idx < 512; idx += NT) {
        const int b = idx >> 8, i = (idx >> 4) & 15, j = idx & 15;
        const int ro = (2 * b + 1) * 16, co = 2 * b * 16;
        float acc = 0.0f;
#pragma unroll
        for (int s = 0; s < 16; ++s) acc += Nm[(ro + i) * 65 + co + s] * Tm[(co + s) * 65 + co + j];
        Y[b * 272 + i * 17 + j] = acc;
      }
    }
    __syncthreads();
    {
      for (int idx = tid; idx < 512; idx += NT) {
        const int b = idx >> 8, i = (idx >> 4) & 15, j = idx & 15;
        const int ro = (2 * b + 1) * 16, co = 2 * b * 16;
        float acc = 0.0f;
#pragma unroll
        for (int s = 0; s < 16; ++s) acc += Tm[(ro + i) * 65 + ro + s] * Y[b * 272 + s * 17 + j];
        Tm[(ro + i) * 65 + co + j] = -acc;
      }
    }
    __syncthreads();
    {   // Y2 = N[32:64, 0:32] T[0:32, 0:32]
      for (int idx = tid; idx < 1024; idx += NT) {
        const int i = idx >> 5, j = idx & 31;
        float acc = 0.0f;
#pragma unroll 8
        for (int s = 0; s < 32; ++s) acc += Nm[(32 + i) * 65 + s] * Tm[s * 65 + j];
        Y[i * 33 + j] = acc;
      }
    }
    __syncthreads();
    {   // T[32:64, 0:32] = -T[32:64, 32:64] Y2
      for (int idx = tid; idx < 1024; idx += NT) {
        const int i = idx >> 5, j = idx & 31;
        float acc = 0.0f;
#pragma unroll 8
        for (int s = 0; s < 32; ++s) acc += Tm[(32 + i) * 65 + 32 + s] * Y[s * 33 + j];
        Tm[(32 + i) * 65 + j] = -acc;
      }
    }
    __syncthreads();
    // T diag(b) -> bf16 (K-major, row r, k = s)
    for (int idx = tid; idx < 512; idx += NT) {
      const int r = idx >> 3, c8 = idx & 7;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int s = c8 * 8 + e * 2;
        w[e] = pack_bf16x2(Tm[r * 65 + s] * beta_s[s], Tm[r * 65 + s + 1] * beta_s[s + 1]);
      }
      st_u128(sm, OFF_TB + kmajor_off(r, c8 * 8, 64), make_uint4(w[0], w[1], w[2], w[3]));
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P5: W^T = Kg^T (T diag b)^T -> D1 region;  U'^T = V^T (T diag b)^T -> U
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + TM_D1, mndesc(sb + OFF_KG, 8192, ks), kdesc(sb + OFF_TB, 64, ks),
                 ID_MK64, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + TM_U, mndesc(sb + OFF_INV, 8192, ks), kdesc(sb + OFF_TB, 64, ks),
                 ID_MK64, ks > 0);
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

    // ---- P6: -W (bf16, MN-major, n = token, k = dk) from W^T; state pass:
    //          S^T -> bf16 operand, S^T <- S^T diag(2^Gam_last)
    if (warp < 4) {
      const int dk = my_lane;
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + TM_D1 + cb * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(-__uint_as_float(r[c8 * 8 + e * 2]),
                               -__uint_as_float(r[c8 * 8 + e * 2 + 1]));
          st_u128(sm, OFF_WN + mnmajor_off(cb * 32 + c8 * 8, dk, 8192),
                  make_uint4(w[0], w[1], w[2], w[3]));
        }
      }
    } else {
      const int dv = my_lane;
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + TM_S + cb * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(r[c8 * 8 + e * 2]),
                               __uint_as_float(r[c8 * 8 + e * 2 + 1]));
          st_u128(sm, OFF_SB + kmajor_off(dv, cb * 32 + c8 * 8, 128),
                  make_uint4(w[0], w[1], w[2], w[3]));
        }
#pragma unroll
        for (int j = 0; j < 32; ++j)
          r[j] = __float_as_uint(__uint_as_float(r[j]) * decay_s[cb * 32 + j]);
        tmem_st32(tmem + lane_base + TM_S + cb * 32, r);
      }
      tmem_wait_st();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- P7: U^T += S^T (-W)^T;  O^T = S^T Qg^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + TM_U, kdesc(sb + OFF_SB, 128, ks), mndesc(sb + OFF_WN, 8192, ks), ID_KM64,
                 1);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + TM_O, kdesc(sb + OFF_SB, 128, ks), kdesc(sb + OFF_QG, 64, ks), ID_KK64,
                 ks > 0);
      mma_commit(bar_mma);
    }
    {
      const bool ok = mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 70; break; }
    }
    tc_fence_after();

    // ---- P8: U^T -> bf16 operand (K-major, row dv, k = token)
    if (warp < 4) {
      const int dv = my_lane;
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + TM_U + cb * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(r[c8 * 8 + e * 2]),
                               __uint_as_float(r[c8 * 8 + e * 2 + 1]));
          st_u128(sm, OFF_UB + kmajor_off(dv, cb * 32 + c8 * 8, 128),
                  make_uint4(w[0], w[1], w[2], w[3]));
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- P9: O^T += U^T QK^T;  S^T += U^T Ke
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + TM_O, kdesc(sb + OFF_UB, 128, ks), kdesc(sb + OFF_QKB, 64, ks), ID_KK64,
                 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + TM_S, kdesc(sb + OFF_UB, 128, ks), mndesc(sb + OFF_KE, 8192, ks),
                 ID_KM128, 1);
      mma_commit(bar_mma);
    }
    {
      const bool ok = mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 90; break; }
    }
    tc_fence_after();

    // ---- P10: O^T -> bf16 staging [token][dv] -> global rows < L of this value slice
    if (warp < 4) {
      const int dv = my_lane;
      __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_OST);
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + TM_O + cb * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) ost[(cb * 32 + j) * D + dv] = __float2bfloat16_rn(__uint_as_float(r[j]));
      }
    }
    tc_fence_before();
    __syncthreads();
    for (int idx = tid; idx < C * 16; idx += NT) {
      const int r = idx >> 4, v8 = idx & 15;
      if (r < L && v8 * 8 >= dv_lo && v8 * 8 < dv_hi) {
        const uint4 val = *reinterpret_cast<const uint4*>(sm + OFF_OST + r * 256 + v8 * 16);
        *reinterpret_cast<uint4*>(p.out + (size_t)(c0 + r) * HD + xcol + v8 * 8) = val;
      }
    }
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
      const int dk0 = col_half * 64 + cb * 32;
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
