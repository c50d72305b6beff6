// Warp-specialised fused chunked KDA prefill (KDA_KERNEL_PIPE): one CTA per
// (sequence, head), 64-token chunks, the 128 x 128 fp32 state in tensor memory.
//
// The chunk step splits into a state-free half (the "k-side": gate, norms, the
// decay-weighted Gram products and the UT inverse) and the state half (the
// "chain").  The fused kernel of kda_tc_kernel.cuh runs the two halves one after
// the other; here they run on different warps at the same time:
//   warps 0-3   chain of chunk c: thread i <-> TMEM lane i <-> value channel i;
//   warps 4-11  k-side of chunk c+1: gate, cumsum, norms, operand tiles, the A|QK
//               extraction and the T -> bf16 conversion;
//   warps 12-15 k-side of chunk c+1: per-channel anchors and factors, row norms,
//               beta, the UT inverse, the k-side MMA and the input TMA.
// The k-side hands each chunk over through one shared-memory stage guarded by
// mbarriers (stage full: k-side -> chain; stage parts free: chain -> k-side).
//
// Per chunk (rows r, s = tokens; G = inclusive cumsum of the log2 decay over the
// chunk, per key channel; raw q, k rows scaled by a power of two to norm <= 1;
// inv_q = scale / |q|, inv_k = 1 / |k| carried as per-token scalars):
//   A[r,s]  = b_r inv_k_r inv_k_s  k_r.(k_s 2^(G_r - G_s))   (s < r)
//   QK[r,s] =                      q_r.(k_s 2^(G_r - G_s))   (s <= r)
//   T = (I + A)^-1
//   Kg = k 2^G,  Qg = q 2^G,  Ke = k 2^(G_last - G)
//   X = Kg S,  U = T diag(b) V - T diag(b inv_k) X            (WY/UT form, W never formed)
//   O = diag(inv_q) (Qg S + QK diag(inv_k) U)
//   S' = diag(2^G_last) S + Ke^T diag(inv_k) U
// which is the chunk form of the gated delta rule with the bounded gate
// a = lower_bound * sigmoid(exp(A_log) (g + dt_bias)), the in-kernel q/k l2norm and
// the beta sigmoid of the FlashKDA prefill PR report (vLLM PR #55737, "Use FlashKDA
// for KDA chunked prefill", Features & motivation).
//
// The chain's products, all tcgen05 kind::f16 with M = 128 = value channel:
//   [X^T | O^T]  = S_b^T [Kg | Qg]^T          (S_b = bf16 S^T in TMEM, N = 128)
//   U^T          = V^T (T diag b)^T + X_b^T T^T   (X_b = bf16(X^T diag(-b inv_k)))
//   O^T         += U_b^T QK^T,  S^T += U_b^T Ke  (U_b = bf16(U^T diag(inv_k)))
// and the k-side's: [A | QK] = [Kr; Qr] [Kc; Kc2]^T (M = 128, N = 96) over the
// exponent-anchored operands of kda_tc_kernel.cu (two 32-token blocks anchored at
// their 16th token; Kc2 carries the block-0 columns seen from block 1).
//
// Every wait is bounded (about one second); a timeout is recorded as
// KDA_ERR_DEVICE_TIMEOUT and both warp groups leave their loops in step.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_tc_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace tcc;

constexpr int PC = 64;            // chunk
constexpr int PD = kHeadDim;      // 128
constexpr int PNT = 512;
constexpr int kPipeMaxRankSeqs = 128;

// ---- shared memory (offsets from a 1024-byte aligned base)
// k-side private
constexpr int PS_INQ = 0;             // q tile: two SW128 boxes [64 tok][64 dk], 8 KB apart
constexpr int PS_INK = 16384;         // k tile
constexpr int PS_ING = 32768;         // g tile
constexpr int PS_RKQ = 49152;         // [Kr; Qr] K-major 128 rows x 128 (until the A|QK MMA ends)
constexpr int PS_CKC = 81920;         // [Kc; Kc2] K-major 96 rows x 128
constexpr int PS_NM = PS_RKQ;         // then: N = diag(b inv_k) strict(A) diag(inv_k) [64][NS]
constexpr int PS_TM = PS_NM + 64 * NS * 4;   //       T [64][NS]
constexpr int PS_Y = PS_TM + 64 * NS * 4;    //       product scratch [32][NS]
// the stage (chain operands of one chunk)
constexpr int PS_WQ = 106496;         // [Kg; Qg] K-major 128 rows (tokens) x 128 (dk)
constexpr int PS_V = 139264;          // v: two SW128 boxes [64 tok][64 dv]; after U: O staging
                                      //    [64 tok][128 dv] bf16 row-major
constexpr int PS_TB = 155648;         // T diag(b) K-major 64 x 64
constexpr int PS_TT = 163840;         // T K-major 64 x 64
constexpr int PS_QK = 172032;         // QK (masked, raw) K-major 64 x 64
constexpr int PS_KE = 180224;         // Ke MN-major: 128 dk (2 blocks of 64, 8 KB apart) x 64 tok
// small things
constexpr int PS_VEC = 196608;        // [3 by chunk % 3]: decay[128] iq[64] ik[64] nbik[64] fp32
constexpr int kVecFloats = 320;
constexpr int PS_GT = PS_VEC + 3 * kVecFloats * 4;   // quad totals, then anchor offsets [16][128]
constexpr int PS_FAC = PS_GT + 16 * 128 * 4;          // per-channel factors [6][128]
constexpr int PS_SS = PS_FAC + 6 * 128 * 4;           // row sums of squares: q [64], k [64]
constexpr int PS_RSC = PS_SS + 128 * 4;               // row power-of-two scales, bf16x2 [128]
constexpr int PS_BETA = PS_RSC + 128 * 4;             // b [64]
constexpr int PS_BAR = PS_BETA + 64 * 4;              // mbarriers
constexpr int PS_TSLOT = PS_BAR + 16 * 8;
constexpr int PS_FLAGS = PS_TSLOT + 16;
constexpr int PS_END = PS_FLAGS + 16;
constexpr int PIPE_SMEM = PS_END + 1024;
static_assert(PS_Y + 32 * NS * 4 <= PS_WQ, "T scratch overlaps the stage");
static_assert(PS_CKC + 96 * 128 * 2 <= PS_WQ, "operands overlap the stage");
static_assert(PS_KE + 16384 <= PS_VEC, "stage overlaps the vectors");
static_assert(PS_WQ % 1024 == 0 && PS_V % 1024 == 0 && PS_TB % 1024 == 0 && PS_TT % 1024 == 0 &&
                  PS_QK % 1024 == 0 && PS_KE % 1024 == 0 && PS_RKQ % 1024 == 0 &&
                  PS_CKC % 1024 == 0,
              "SW128 tiles are 1024-byte aligned");
static_assert(PIPE_SMEM <= 227 * 1024, "shared memory");

// mbarriers (8 bytes each from PS_BAR)
constexpr int B_IN = 0;      // q, k, g of the k-side's chunk landed (TMA tx)
constexpr int B_V = 1;       // v of the chain's chunk landed (TMA tx)
constexpr int B_FULL = 2;    // stage written by the k-side (1 arrival)
constexpr int B_FREEA = 3;   // chain done with [Kg; Qg], T diag(b), T (and v)
constexpr int B_FREEB = 4;   // chain done with QK, Ke
constexpr int B_KMMA = 5;    // k-side A|QK MMA done
constexpr int B_G1A = 6;     // chain: [X^T | O^T] done
constexpr int B_G1B = 7;     // chain: U^T done
constexpr int B_G2 = 8;      // chain: O^T, S^T updates done

// ---- tensor memory columns (fp32 unless noted; lane = value channel, or row for D)
constexpr uint32_t TM_XU = 0;     // X^T, then U^T   64 cols (col = token)
constexpr uint32_t TM_O = 64;     // O^T             64 cols
constexpr uint32_t TM_S = 128;    // S^T            128 cols (col = dk)
constexpr uint32_t TM_SB = 256;   // S^T bf16        64 cols (2 dk per col)
constexpr uint32_t TM_XB = 320;   // X_b^T bf16      32 cols (2 tokens per col)
constexpr uint32_t TM_UB = 352;   // U_b^T bf16      32 cols
constexpr uint32_t TM_D = 384;    // [A | QK] (k-side) 96 cols
constexpr uint32_t TM_NCOLS = 512;

constexpr uint32_t ID_D96 = idesc_bf16(128, 96, 0, 0);    // [Kr;Qr] x [Kc;Kc2]^T
constexpr uint32_t ID_G1A = idesc_bf16(128, 128, 0, 0);   // S_b x [Kg|Qg]^T
constexpr uint32_t ID_UP = idesc_bf16(128, 64, 1, 0);     // V^T (MN-major) x (T diag b)^T
constexpr uint32_t ID_N64 = idesc_bf16(128, 64, 0, 0);    // X_b x T^T,  U_b x QK^T
constexpr uint32_t ID_KE = idesc_bf16(128, 128, 0, 1);    // U_b x Ke (MN-major)

#ifdef KDA_PHASE_STAMPS
#define PSTAMP(cond, c, slot)                                                       \
  do {                                                                              \
    if ((cond) && p.stamps != nullptr && blockIdx.x == 0 && (c) < 64)               \
      p.stamps[(c) * 16 + (slot)] = (unsigned long long)clock64();                  \
  } while (0)
#else
#define PSTAMP(cond, c, slot) \
  do {                        \
  } while (0)
#endif

// barrier `id` over `count` threads with an OR reduction of `pred` (group-uniform result)
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
__device__ __forceinline__ uint4 lds128(const unsigned char* base, uint32_t off) {
  return *reinterpret_cast<const uint4*>(base + off);
}
// byte offset of the 16-byte chunk holding columns 8o..8o+7 of row r in a tile of two
// SW128 boxes [64 rows][64 cols] 8 KB apart (what a TMA box of 64 columns writes)
__device__ __forceinline__ uint32_t in_off(int r, int o) {
  return (uint32_t)((o >> 3) * 8192 + r * 128 + (((o & 7) ^ (r & 7)) << 4));
}

struct PipeMaps {
  CUtensorMap q, k, g, v;   // [T][H*128] bf16, box {64, 64}, 128-byte swizzle
  CUtensorMap out;          // [T][H*128] bf16, box {128, 64}, no swizzle
};

__global__ void __launch_bounds__(PNT, 1)
    kda_pipe_kernel(const __grid_constant__ Params p, const __grid_constant__ PipeMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* flags = reinterpret_cast<int*>(sm + PS_FLAGS);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + PS_TSLOT);
  auto bar = [&](int i) { return sb + PS_BAR + 8 * i; };

  // ---- work unit: (rank, head), longest sequence first
  const int H = p.heads, N = p.num_seqs;
  const int h = blockIdx.x % H;
  const int rank = blockIdx.x / H;
  if (N <= kPipeMaxRankSeqs) {
    int* lens = reinterpret_cast<int*>(sm + PS_GT);
    for (int i = tid; i < N; i += PNT) lens[i] = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
    __syncthreads();
    for (int i = tid; i < N; i += PNT) {
      const int li = lens[i];
      int r = 0;
      for (int m = 0; m < N; ++m) {
        const int lm = lens[m];
        r += (lm > li) || (lm == li && m < i);
      }
      if (r == rank) flags[0] = i;
    }
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
  const int nch = (t1 - t0 + PC - 1) / PC;
  const size_t HD = (size_t)H * PD;
  const size_t sbase = ((size_t)n * H + h) * PD * PD;
  const int xcol = h * PD;

  if (tid == 0) {
    mbar_init(bar(B_IN), 1);
    mbar_init(bar(B_V), 1);
    mbar_init(bar(B_FULL), 1);
    mbar_init(bar(B_FREEA), 1);
    mbar_init(bar(B_FREEB), 1);
    mbar_init(bar(B_KMMA), 1);
    mbar_init(bar(B_G1A), 1);
    mbar_init(bar(B_G1B), 1);
    mbar_init(bar(B_G2), 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), TM_NCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  float* vecs = reinterpret_cast<float*>(sm + PS_VEC);
  bool failed = false;
  int site = 0;

  if (warp < 4) {
    // =========================================================================== chain
    const int dv = tid;                                  // value channel = TMEM lane
    const uint32_t lb = (uint32_t)(32 * warp) << 16;     // lane base of this warp
    int pend = 0;   // thread 0: bit 0 v load, 1 G1A, 2 G1B, 3 G2 issued and not waited
    int cfail = 0;  // chunk at which the loop stopped (all pending phases have its parity)
    if (tid == 0) {
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.out);
      if (nch > 0) {
        mbar_expect_tx(bar(B_V), 16384);
        tma_load_2d(sb + PS_V, &maps.v, xcol, t0, bar(B_V));
        tma_load_2d(sb + PS_V + 8192, &maps.v, xcol + 64, t0, bar(B_V));
        pend |= 1;
      }
    }
    // state in: S^T[dv][dk] -> TMEM (lane = dv)
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float s = 0.0f;
        if (p.initial_state) {
          const size_t idx = sbase + (size_t)(cb * 32 + j) * PD + dv;
          s = p.state_bf16
                  ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.initial_state)[idx])
                  : static_cast<const float*>(p.initial_state)[idx];
        }
        r[j] = __float_as_uint(s);
      }
      tmem_st32(tmem + lb + TM_S + cb * 32, r);
    }
    tmem_wait_st();

    for (int c = 0; c < nch; ++c) {
      const int c0 = t0 + PC * c;
      const int L = min(PC, t1 - c0);
      const uint32_t par = (uint32_t)(c & 1);
      const float* vec = vecs + (c % 3) * kVecFloats;
      cfail = c;

      // C0: the stage and v of chunk c have landed
      bool ok = mbar_wait(bar(B_FULL), par);
      const bool v_ok = mbar_wait(bar(B_V), par);
      if (tid == 0 && v_ok) pend &= ~1;
      ok = ok && v_ok;
      PSTAMP(tid == 0, c, 0);
      if (ok && L < PC) {   // v rows past the sequence end -> 0 (they meet zero columns of
                            // T diag(b), but must not carry inf or nan into the product)
        for (int idx = tid; idx < (PC - L) * 16; idx += 128) {
          const int r = L + idx / 16, cc = idx % 16;
          *reinterpret_cast<uint4*>(sm + PS_V + (cc >> 3) * 8192 + r * 128 +
                                    (((cc & 7) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      tc_fence_after();
      // C1a: S_b = bf16(S^T)
#pragma unroll 1
      for (int cb = 0; cb < 4; cb += 2) {
        uint32_t x[32], y[32], pk[16];
        tmem_ld32(tmem + lb + TM_S + cb * 32, x);
        tmem_ld32(tmem + lb + TM_S + cb * 32 + 32, y);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
        tmem_st16(tmem + lb + TM_SB + cb * 16, pk);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(y[2 * j]), __uint_as_float(y[2 * j + 1]));
        tmem_st16(tmem + lb + TM_SB + cb * 16 + 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      if (bar_any(4, 128, !ok)) { failed = true; site = 40; break; }
      // G1a: [X^T | O^T] = S_b [Kg | Qg]^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_ts(tmem + TM_XU, tmem + TM_SB + 8 * ks, kdesc(sb + PS_WQ, 128, ks), ID_G1A,
                      ks > 0);
        mma_commit(bar(B_G1A));
        pend |= 2;
        PSTAMP(true, c, 1);
      }
      // C1b: S^T *= 2^G_last (per key column), while G1a runs
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t x[32];
        tmem_ld32(tmem + lb + TM_S + cb * 32, x);
        tmem_wait_ld();
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 dl = ld4(vec + cb * 32 + 4 * j4);
          x[4 * j4] = __float_as_uint(__uint_as_float(x[4 * j4]) * dl.x);
          x[4 * j4 + 1] = __float_as_uint(__uint_as_float(x[4 * j4 + 1]) * dl.y);
          x[4 * j4 + 2] = __float_as_uint(__uint_as_float(x[4 * j4 + 2]) * dl.z);
          x[4 * j4 + 3] = __float_as_uint(__uint_as_float(x[4 * j4 + 3]) * dl.w);
        }
        tmem_st32(tmem + lb + TM_S + cb * 32, x);
      }
      tmem_wait_st();
      // C2: X_b = bf16(X^T diag(-b inv_k))
      ok = mbar_wait(bar(B_G1A), par);
      if (tid == 0 && ok) pend &= ~2;
      PSTAMP(tid == 0, c, 2);
      tc_fence_after();
      {
        uint32_t x[32], y[32], pk[16];
        tmem_ld32(tmem + lb + TM_XU, x);
        tmem_ld32(tmem + lb + TM_XU + 32, y);
        tmem_wait_ld();
        const float* nb = vec + 256;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 f = ld4(nb + 4 * j4);
          pk[2 * j4] = pack_bf16x2(__uint_as_float(x[4 * j4]) * f.x,
                                   __uint_as_float(x[4 * j4 + 1]) * f.y);
          pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(x[4 * j4 + 2]) * f.z,
                                       __uint_as_float(x[4 * j4 + 3]) * f.w);
        }
        tmem_st16(tmem + lb + TM_XB, pk);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 f = ld4(nb + 32 + 4 * j4);
          pk[2 * j4] = pack_bf16x2(__uint_as_float(y[4 * j4]) * f.x,
                                   __uint_as_float(y[4 * j4 + 1]) * f.y);
          pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(y[4 * j4 + 2]) * f.z,
                                       __uint_as_float(y[4 * j4 + 3]) * f.w);
        }
        tmem_st16(tmem + lb + TM_XB + 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      if (bar_any(4, 128, !ok)) { failed = true; site = 41; break; }
      // G1b: U^T = V^T (T diag b)^T + X_b^T T^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + TM_XU, mndesc(sb + PS_V, 8192, ks), kdesc(sb + PS_TB, 64, ks), ID_UP,
                   ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_ts(tmem + TM_XU, tmem + TM_XB + 8 * ks, kdesc(sb + PS_TT, 64, ks), ID_N64, 1);
        mma_commit(bar(B_G1B));
        pend |= 4;
      }
      ok = mbar_wait(bar(B_G1B), par);
      if (tid == 0 && ok) {
        pend &= ~4;
        mbar_arrive(bar(B_FREEA));   // [Kg; Qg], T diag(b), T are free
      }
      PSTAMP(tid == 0, c, 3);
      tc_fence_after();
      // C3: U_b = bf16(U^T diag(inv_k))
      {
        uint32_t x[32], y[32], pk[16];
        tmem_ld32(tmem + lb + TM_XU, x);
        tmem_ld32(tmem + lb + TM_XU + 32, y);
        tmem_wait_ld();
        const float* ik = vec + 192;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 f = ld4(ik + 4 * j4);
          pk[2 * j4] = pack_bf16x2(__uint_as_float(x[4 * j4]) * f.x,
                                   __uint_as_float(x[4 * j4 + 1]) * f.y);
          pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(x[4 * j4 + 2]) * f.z,
                                       __uint_as_float(x[4 * j4 + 3]) * f.w);
        }
        tmem_st16(tmem + lb + TM_UB, pk);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 f = ld4(ik + 32 + 4 * j4);
          pk[2 * j4] = pack_bf16x2(__uint_as_float(y[4 * j4]) * f.x,
                                   __uint_as_float(y[4 * j4 + 1]) * f.y);
          pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(y[4 * j4 + 2]) * f.z,
                                       __uint_as_float(y[4 * j4 + 3]) * f.w);
        }
        tmem_st16(tmem + lb + TM_UB + 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      if (bar_any(4, 128, !ok)) { failed = true; site = 42; break; }
      // G2: O^T += U_b^T QK^T, S^T += U_b^T Ke
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_ts(tmem + TM_O, tmem + TM_UB + 8 * ks, kdesc(sb + PS_QK, 64, ks), ID_N64, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_ts(tmem + TM_S, tmem + TM_UB + 8 * ks, mndesc(sb + PS_KE, 8192, ks), ID_KE, 1);
        mma_commit(bar(B_G2));
        pend |= 8;
      }
      ok = mbar_wait(bar(B_G2), par);
      if (tid == 0 && ok) {
        pend &= ~8;
        mbar_arrive(bar(B_FREEB));   // QK, Ke are free
      }
      PSTAMP(tid == 0, c, 4);
      tc_fence_after();
      // C4: O^T diag(inv_q) -> bf16 staging [token][dv] (over v, free since G1b)
      {
        uint32_t x[32], y[32];
        tmem_ld32(tmem + lb + TM_O, x);
        tmem_ld32(tmem + lb + TM_O + 32, y);
        tmem_wait_ld();
        const float* iq = vec + 128;
        __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + PS_V);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          ost[j * PD + dv] = __float2bfloat16_rn(__uint_as_float(x[j]) * iq[j]);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          ost[(32 + j) * PD + dv] = __float2bfloat16_rn(__uint_as_float(y[j]) * iq[32 + j]);
      }
      fence_proxy_async();
      tc_fence_before();
      if (bar_any(4, 128, !ok)) { failed = true; site = 43; break; }
      if (L == PC) {
        if (tid == 0) {
          tma_store_2d(&maps.out, xcol, c0, sb + PS_V);
          bulk_commit();
          bulk_wait_read();   // the staging is read: v of the next chunk may land there
          if (c + 1 < nch) {
            mbar_expect_tx(bar(B_V), 16384);
            tma_load_2d(sb + PS_V, &maps.v, xcol, c0 + PC, bar(B_V));
            tma_load_2d(sb + PS_V + 8192, &maps.v, xcol + 64, c0 + PC, bar(B_V));
            pend |= 1;
          }
        }
      } else {   // the sequence's last chunk: rows < L only
        for (int idx = tid; idx < L * 16; idx += 128) {
          const int r = idx >> 4, v8 = idx & 15;
          *reinterpret_cast<uint4*>(p.out + (size_t)(c0 + r) * HD + xcol + v8 * 8) =
              *reinterpret_cast<const uint4*>(sm + PS_V + r * 256 + v8 * 16);
        }
      }
      PSTAMP(tid == 0, c, 5);
    }
    if (failed) {
      if (tid == 0) {
        record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
        // let copies and MMAs still in flight end (bounded) before the CTA exits
        const uint32_t fp = (uint32_t)(cfail & 1);
        if (pend & 1) mbar_wait(bar(B_V), fp);
        if (pend & 2) mbar_wait(bar(B_G1A), fp);
        if (pend & 4) mbar_wait(bar(B_G1B), fp);
        if (pend & 8) mbar_wait(bar(B_G2), fp);
      }
    } else {
      // state out
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + lb + TM_S + cb * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const size_t idx = sbase + (size_t)(cb * 32 + j) * PD + dv;
          const float s = __uint_as_float(r[j]);
          if (p.state_bf16)
            static_cast<__nv_bfloat16*>(p.final_state)[idx] = __float2bfloat16_rn(s);
          else
            static_cast<float*>(p.final_state)[idx] = s;
        }
      }
    }
    if (tid == 0) bulk_wait_all();
  } else {
    // =========================================================================== k-side
    const int kt = tid - 128;                 // 0..383
    const bool isA = kt < 256;                // warps 4-11: tiles; warps 12-15: scalars
    const int ka = kt, wa = ka >> 5;          // (group A)
    const int o = lane & 15;                  // octet: key channels 8o .. 8o+7
    const int j = 2 * wa + (lane >> 4);       // row quad: rows 4j .. 4j+3
    const int bsel = wa >> 2;                 // 32-token block of this thread's rows
    const int kb = kt - 256;                  // 0..127 (group B)
    const bool mma_thread = kb == 0, tma_thread = kb == 64;
    float* GT = reinterpret_cast<float*>(sm + PS_GT);
    float* FAC = reinterpret_cast<float*>(sm + PS_FAC);
    float* SS = reinterpret_cast<float*>(sm + PS_SS);
    uint32_t* RSC = reinterpret_cast<uint32_t*>(sm + PS_RSC);
    float* BETA = reinterpret_cast<float*>(sm + PS_BETA);
    float* Nm = reinterpret_cast<float*>(sm + PS_NM);
    float* Tm = reinterpret_cast<float*>(sm + PS_TM);
    float* Y = reinterpret_cast<float*>(sm + PS_Y);
    const float gate_scale = expf(p.A_log[h]);
    const float lb2 = p.lower_bound * kLog2e;
    const float sg = -gate_scale * kLog2e;   // sigmoid argument, log2 units: sg (g + dt_bias)
    float sgd[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sgd[e] = isA ? sg * p.dt_bias[h * PD + 8 * o + e] : 0.0f;
    int in_pend = 0;      // tma thread: an input load issued and not waited (its parity + 1)
    int kmma_pend = 0;    // the A|QK MMA issued and not waited (its parity + 1)

    auto issue_in = [&](int c) {   // q, k, g of chunk c -> the input tiles; chunk c+1 -> L2
      const int y = t0 + PC * c;
      mbar_expect_tx(bar(B_IN), 49152);
      tma_load_2d(sb + PS_INQ, &maps.q, xcol, y, bar(B_IN));
      tma_load_2d(sb + PS_INQ + 8192, &maps.q, xcol + 64, y, bar(B_IN));
      tma_load_2d(sb + PS_INK, &maps.k, xcol, y, bar(B_IN));
      tma_load_2d(sb + PS_INK + 8192, &maps.k, xcol + 64, y, bar(B_IN));
      tma_load_2d(sb + PS_ING, &maps.g, xcol, y, bar(B_IN));
      tma_load_2d(sb + PS_ING + 8192, &maps.g, xcol + 64, y, bar(B_IN));
      if (c + 1 < nch) {
        const int y1 = y + PC;
        tma_prefetch_2d(&maps.q, xcol, y1);
        tma_prefetch_2d(&maps.q, xcol + 64, y1);
        tma_prefetch_2d(&maps.k, xcol, y1);
        tma_prefetch_2d(&maps.k, xcol + 64, y1);
        tma_prefetch_2d(&maps.g, xcol, y1);
        tma_prefetch_2d(&maps.g, xcol + 64, y1);
        tma_prefetch_2d(&maps.v, xcol, y1);
        tma_prefetch_2d(&maps.v, xcol + 64, y1);
      }
      in_pend = (c & 1) + 1;
    };
    if (tma_thread) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.g);
      if (nch > 0) issue_in(0);
    }
    // raw beta logits of the next chunk, fetched a chunk ahead (group B, kb < 64)
    float b_raw = 0.0f;
    if (!isA && kb < PC && t0 + kb < t1) b_raw = __bfloat162float(p.beta[(size_t)(t0 + kb) * p.s_beta + h]);

    for (int c = 0; c < nch; ++c) {
      const int c0 = t0 + PC * c;
      const int L = min(PC, t1 - c0);
      const uint32_t par = (uint32_t)(c & 1);
      float* vec = vecs + (c % 3) * kVecFloats;
      bool ok = true;
      float cl[4][8];

      // ---- K1 (A): gate -> log2 decay, cumsum over this thread's 4 rows; sums of squares
      //              (B): beta
      if (isA) {
        ok = mbar_wait(bar(B_IN), par);
        PSTAMP(ka == 0, c, 8);
        float pss[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * j + i;
          const bool valid = r < L;
          const uint32_t off = in_off(r, o);
          const uint4 gv = lds128(sm + PS_ING, off);
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
          for (int pq = 0; pq < 4; ++pq) {
            const float2 gf = unpack_bf16x2(gw[pq]);
            float a0 = lb2 * rcpf(1.0f + ex2f(fmaf(gf.x, sg, sgd[2 * pq])));
            float a1 = lb2 * rcpf(1.0f + ex2f(fmaf(gf.y, sg, sgd[2 * pq + 1])));
            a0 = valid ? a0 : 0.0f;
            a1 = valid ? a1 : 0.0f;
            cl[i][2 * pq] = (i ? cl[i - 1][2 * pq] : 0.0f) + a0;
            cl[i][2 * pq + 1] = (i ? cl[i - 1][2 * pq + 1] : 0.0f) + a1;
          }
          const uint4 qv = lds128(sm + PS_INQ, off);
          const uint4 kv = lds128(sm + PS_INK, off);
          const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
          float sq = 0.0f, sk = 0.0f;
#pragma unroll
          for (int pq = 0; pq < 4; ++pq) {
            const float2 qf = unpack_bf16x2(qw[pq]), kf = unpack_bf16x2(kw[pq]);
            sq = fmaf(qf.x, qf.x, fmaf(qf.y, qf.y, sq));
            sk = fmaf(kf.x, kf.x, fmaf(kf.y, kf.y, sk));
          }
          pss[i] = valid ? sq : 0.0f;
          pss[4 + i] = valid ? sk : 0.0f;
        }
        // quad totals of the cumsum -> GT[j][channel]
        *reinterpret_cast<float4*>(GT + j * 128 + 8 * o) =
            make_float4(cl[3][0], cl[3][1], cl[3][2], cl[3][3]);
        *reinterpret_cast<float4*>(GT + j * 128 + 8 * o + 4) =
            make_float4(cl[3][4], cl[3][5], cl[3][6], cl[3][7]);
        // reduce the 8 partial sums over the 16 octets of the half-warp (reduce-scatter)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool up = (lane & 8) != 0;
          const float send = up ? pss[i] : pss[i + 4];
          const float keep = up ? pss[i + 4] : pss[i];
          pss[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const bool up = (lane & 4) != 0;
          const float send = up ? pss[i] : pss[i + 2];
          const float keep = up ? pss[i + 2] : pss[i];
          pss[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        {
          const bool up = (lane & 2) != 0;
          const float send = up ? pss[0] : pss[1];
          const float keep = up ? pss[1] : pss[0];
          pss[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        pss[0] += __shfl_xor_sync(0xffffffffu, pss[0], 1);
        if ((lane & 1) == 0) {
          const int k = ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
          SS[(k >> 2) * 64 + 4 * j + (k & 3)] = pss[0];
        }
      } else if (kb < PC) {
        BETA[kb] = (kb < L) ? sigm(b_raw) : 0.0f;
        b_raw = 0.0f;
        if (c0 + PC + kb < t1) b_raw = __bfloat162float(p.beta[(size_t)(c0 + PC + kb) * p.s_beta + h]);
      }
      if (bar_any(1, 384, !ok)) { failed = true; site = 20; break; }
      if (tma_thread) in_pend = 0;   // group A saw this chunk's inputs land

      // ---- K2 (B): anchors and factors per key channel; row norms and scales
      if (!isA) {
        {
          const int d = kb;
          float P[16];
          float run = 0.0f;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            run += GT[q * 128 + d];
            P[q] = run;
          }
          const float m0 = P[3], g31 = P[7], m1 = P[11], g63 = P[15];
#pragma unroll
          for (int q = 0; q < 16; ++q) GT[q * 128 + d] = (q < 8 ? m0 : m1) - (q ? P[q - 1] : 0.0f);
          FAC[0 * 128 + d] = ex2f(g31 - m0);   // Ke, Kc2 of block 0, step 1: 2^(G31 - G)
          FAC[1 * 128 + d] = ex2f(g63 - g31);  // Ke of block 0, step 2
          FAC[2 * 128 + d] = ex2f(m1 - g31);   // Kc2 step 2; Qg/Kg of block 1, step 1
          FAC[3 * 128 + d] = ex2f(m0);         // Qg/Kg of block 0
          FAC[4 * 128 + d] = ex2f(g63 - m1);   // Ke of block 1
          FAC[5 * 128 + d] = ex2f(g31);        // Qg/Kg of block 1, step 2
          vec[d] = ex2f(g63);                  // decay of the state
        }
        {
          const int r = kb & 63;
          const float ss = SS[kb];
          // ss < 2^(e+1) -> |row| < 2^ceil((e+1)/2): rows enter the operands times 2^-sh
          const int e = ((__float_as_int(ss) >> 23) & 255) - 127;
          const int sh = max(-60, min(60, (e + 2) >> 1));
          const float inv = (r < L) ? rsqrtf(ss + kL2Eps) * __int_as_float((127 + sh) << 23) : 0.0f;
          if (kb < 64)
            vec[128 + r] = p.scale * inv;
          else
            vec[192 + r] = inv;
          const uint32_t bb = (uint32_t)(127 - sh) << 7;   // bf16 bits of 2^-sh
          RSC[kb] = bb | (bb << 16);
        }
      }
      named_barrier_sync(1, 384);
      PSTAMP(ka == 0, c, 9);

      // ---- K3 (A): operand tiles: [Kr; Qr], [Kc; Kc2] (own), Kg, Qg, Ke (stage)
      if (isA) {
        float mE[8], fa[8], fb[8], fc[8], fq[8];
        {
          const float4 m_a = ld4(GT + j * 128 + 8 * o), m_b = ld4(GT + j * 128 + 8 * o + 4);
          mE[0] = m_a.x; mE[1] = m_a.y; mE[2] = m_a.z; mE[3] = m_a.w;
          mE[4] = m_b.x; mE[5] = m_b.y; mE[6] = m_b.z; mE[7] = m_b.w;
          const int ia = bsel ? 4 : 0, ib = bsel ? 2 : 1, ic = 2, iq = bsel ? 5 : 3;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            fa[e] = FAC[ia * 128 + 8 * o + e];
            fb[e] = FAC[ib * 128 + 8 * o + e];
            fc[e] = FAC[ic * 128 + 8 * o + e];
            fq[e] = FAC[iq * 128 + 8 * o + e];
          }
        }
        // the chain has finished reading [Kg; Qg] of the previous chunk
        if (c > 0) ok = mbar_wait(bar(B_FREEA), (uint32_t)((c - 1) & 1)) && ok;
        uint32_t ke[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * j + i;
          const bool valid = r < L;
          const uint32_t off = in_off(r, o);
          uint4 qv = lds128(sm + PS_INQ, off), kv = lds128(sm + PS_INK, off);
          if (!valid) qv = kv = make_uint4(0, 0, 0, 0);
          const uint32_t rq = RSC[r], rk = RSC[64 + r];
          const uint32_t q2[4] = {bmul2(qv.x, rq), bmul2(qv.y, rq), bmul2(qv.z, rq), bmul2(qv.w, rq)};
          const uint32_t k2[4] = {bmul2(kv.x, rk), bmul2(kv.y, rk), bmul2(kv.z, rk), bmul2(kv.w, rk)};
          uint32_t kr[4], qr[4], kc[4], kc2[4], kg[4], qg[4];
#pragma unroll
          for (int pq = 0; pq < 4; ++pq) {
            const int e0 = 2 * pq, e1 = 2 * pq + 1;
            const float x0 = cl[i][e0] - mE[e0], x1 = cl[i][e1] - mE[e1];
            const float E0 = ex2f(x0), E1 = ex2f(x1);
            const float Ei0 = ex2f(-x0), Ei1 = ex2f(-x1);
            const uint32_t E2 = pack_bf16x2(E0, E1), Ei2 = pack_bf16x2(Ei0, Ei1);
            kr[pq] = bmul2(k2[pq], E2);
            qr[pq] = bmul2(q2[pq], E2);
            kc[pq] = bmul2(k2[pq], Ei2);
            uint32_t gq;
            if (bsel == 0) {
              const float u0 = Ei0 * fa[e0], u1 = Ei1 * fa[e1];   // 2^(G31 - G)
              kc2[pq] = bmul2(k2[pq], pack_bf16x2(u0 * fc[e0], u1 * fc[e1]));
              ke[i][pq] = bmul2(k2[pq], pack_bf16x2(u0 * fb[e0], u1 * fb[e1]));
              gq = pack_bf16x2(E0 * fq[e0], E1 * fq[e1]);
            } else {
              ke[i][pq] = bmul2(k2[pq], pack_bf16x2(Ei0 * fa[e0], Ei1 * fa[e1]));
              gq = pack_bf16x2((E0 * fc[e0]) * fq[e0], (E1 * fc[e1]) * fq[e1]);
              kc2[pq] = 0u;
            }
            qg[pq] = bmul2(q2[pq], gq);
            kg[pq] = bmul2(k2[pq], gq);
          }
          st_u128(sm, PS_RKQ + kmajor_off(r, 8 * o, 128), make_uint4(kr[0], kr[1], kr[2], kr[3]));
          st_u128(sm, PS_RKQ + kmajor_off(64 + r, 8 * o, 128),
                  make_uint4(qr[0], qr[1], qr[2], qr[3]));
          st_u128(sm, PS_CKC + kmajor_off(r, 8 * o, 96), make_uint4(kc[0], kc[1], kc[2], kc[3]));
          if (bsel == 0)
            st_u128(sm, PS_CKC + kmajor_off(64 + r, 8 * o, 96),
                    make_uint4(kc2[0], kc2[1], kc2[2], kc2[3]));
          st_u128(sm, PS_WQ + kmajor_off(r, 8 * o, 128), make_uint4(kg[0], kg[1], kg[2], kg[3]));
          st_u128(sm, PS_WQ + kmajor_off(64 + r, 8 * o, 128),
                  make_uint4(qg[0], qg[1], qg[2], qg[3]));
        }
        // the chain has finished reading QK and Ke of the previous chunk
        if (c > 0) ok = mbar_wait(bar(B_FREEB), (uint32_t)((c - 1) & 1)) && ok;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_u128(sm, PS_KE + mnmajor_off(8 * o, 4 * j + i, 8192),
                  make_uint4(ke[i][0], ke[i][1], ke[i][2], ke[i][3]));
        fence_proxy_async();
      }
      PSTAMP(ka == 0, c, 10);
      if (bar_any(1, 384, !ok)) { failed = true; site = 21; break; }

      // ---- K4: [A | QK] on the tensor cores; the next chunk's inputs (the tiles are free)
      if (mma_thread) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tmem + TM_D, kdesc(sb + PS_RKQ, 128, ks), kdesc(sb + PS_CKC, 96, ks), ID_D96,
                   ks > 0);
        mma_commit(bar(B_KMMA));
      }
      kmma_pend = (int)par + 1;
      if (tma_thread && c + 1 < nch) issue_in(c + 1);
      ok = mbar_wait(bar(B_KMMA), par);
      if (ok) kmma_pend = 0;
      PSTAMP(ka == 0, c, 11);
      tc_fence_after();

      // ---- K5 (A): A rows -> N (fp32), QK rows -> bf16 (stage); (B): T upper blocks -> 0
      if (isA) {
        const int q4 = wa & 3, cs = wa >> 2;
        const uint32_t lbase = (uint32_t)(32 * q4) << 16;
        const int m = 32 * q4 + lane;
        const float* ik = vec + 192;
        if (q4 < 2) {
          const int r = m;
          float* nrow = Nm + r * NS + 32 * cs;
          if (q4 == 0 && cs == 1) {
#pragma unroll
            for (int s4 = 0; s4 < 8; ++s4)
              *reinterpret_cast<float4*>(nrow + 4 * s4) = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint32_t a[32];
            tmem_ld32(tmem + lbase + TM_D + (cs == 1 ? 32 : (q4 == 0 ? 0 : 64)), a);
            tmem_wait_ld();
            const float br = BETA[r] * ik[r];
#pragma unroll
            for (int s4 = 0; s4 < 8; ++s4) {
              const float4 kk = ld4(ik + 32 * cs + 4 * s4);
              const float kv4[4] = {kk.x, kk.y, kk.z, kk.w};
              float w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int s = 32 * cs + 4 * s4 + e;
                w[e] = (s < r) ? br * kv4[e] * __uint_as_float(a[4 * s4 + e]) : 0.0f;
              }
              *reinterpret_cast<float4*>(nrow + 4 * s4) = make_float4(w[0], w[1], w[2], w[3]);
            }
          }
        } else {
          const int r = m - 64;
          if (q4 == 2 && cs == 1) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8)
              st_u128(sm, PS_QK + kmajor_off(r, 32 + 8 * c8, 64), make_uint4(0, 0, 0, 0));
          } else {
            uint32_t a[32];
            tmem_ld32(tmem + lbase + TM_D + (cs == 1 ? 32 : (q4 == 2 ? 0 : 64)), a);
            tmem_wait_ld();
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int s = 32 * cs + 8 * c8 + 2 * e;
                w[e] = pack_bf16x2(s <= r ? __uint_as_float(a[8 * c8 + 2 * e]) : 0.0f,
                                   s + 1 <= r ? __uint_as_float(a[8 * c8 + 2 * e + 1]) : 0.0f);
              }
              st_u128(sm, PS_QK + kmajor_off(r, 32 * cs + 8 * c8, 64),
                      make_uint4(w[0], w[1], w[2], w[3]));
            }
          }
        }
      } else {
        // T above the diagonal 16 x 16 blocks is zero
        for (int idx = kb; idx < 6 * 64; idx += 128) {
          const int b = idx >> 6, e = idx & 63;
          const int bi = (b < 3) ? 0 : (b < 5 ? 1 : 2);
          const int bj = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
          *reinterpret_cast<float4*>(Tm + (bi * 16 + (e >> 2)) * NS + bj * 16 + 4 * (e & 3)) =
              make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      tc_fence_before();
      if (bar_any(1, 384, !ok)) { failed = true; site = 22; break; }
      PSTAMP(ka == 0, c, 12);

      // ---- K6 (B): T = (I + N)^-1: 16 x 16 diagonal blocks by substitution (fp32), then
      //               the off-diagonal blocks as tf32 warp products, 16 -> 32 -> 64
      if (!isA) {
        const int wb = kb >> 5;
        if (wb < 2) {
          const int ob = (kb >> 4) * 16, jj = kb & 15;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = (i == jj) ? 1.0f : 0.0f;
#pragma unroll
          for (int k = 0; k < 15; ++k) {
#pragma unroll
            for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-Nm[(ob + i) * NS + ob + k], x[k], x[i]);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) Tm[(ob + i) * NS + ob + jj] = x[i];
        }
        named_barrier_sync(3, 128);
        if (wb < 2) {   // pair (1,0) on warp 0 of the group, (3,2) on warp 1
          const int ro = (2 * wb + 1) * 16, co = 2 * wb * 16;
          float* Yw = Y + wb * 16 * NS;
          warp_gemm_16x16<16>(Nm + ro * NS + co, Tm + co * NS + co, Yw, 1.0f, lane);
          __syncwarp();
          warp_gemm_16x16<16>(Tm + ro * NS + ro, Yw, Tm + ro * NS + co, -1.0f, lane);
        }
        named_barrier_sync(3, 128);
        const int mi = wb >> 1, ni = wb & 1;   // Y2 = N[32:64, 0:32] T[0:32, 0:32]
        warp_gemm_16x16<32>(Nm + (32 + 16 * mi) * NS, Tm + 16 * ni, Y + 16 * mi * NS + 16 * ni,
                            1.0f, lane);
        named_barrier_sync(3, 128);            // T[32:64, 0:32] = -T[32:64, 32:64] Y2
        warp_gemm_16x16<32>(Tm + (32 + 16 * mi) * NS + 32, Y + 16 * ni,
                            Tm + (32 + 16 * mi) * NS + 16 * ni, -1.0f, lane);
      }
      named_barrier_sync(1, 384);
      PSTAMP(ka == 0, c, 13);

      // ---- K7 (A): T diag(b) and T -> bf16 (stage); (B): -b inv_k
      if (isA) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int item = ka + 256 * h2;
          const int r = item >> 3, c8 = item & 7;
          const float4 ta = ld4(Tm + r * NS + 8 * c8), tb = ld4(Tm + r * NS + 8 * c8 + 4);
          const float4 ba = ld4(BETA + 8 * c8), bb = ld4(BETA + 8 * c8 + 4);
          const uint32_t off = kmajor_off(r, 8 * c8, 64);
          st_u128(sm, PS_TB + off,
                  make_uint4(pack_bf16x2(ta.x * ba.x, ta.y * ba.y), pack_bf16x2(ta.z * ba.z, ta.w * ba.w),
                             pack_bf16x2(tb.x * bb.x, tb.y * bb.y), pack_bf16x2(tb.z * bb.z, tb.w * bb.w)));
          st_u128(sm, PS_TT + off,
                  make_uint4(pack_bf16x2(ta.x, ta.y), pack_bf16x2(ta.z, ta.w),
                             pack_bf16x2(tb.x, tb.y), pack_bf16x2(tb.z, tb.w)));
        }
        fence_proxy_async();
      } else if (kb < PC) {
        vec[256 + kb] = -BETA[kb] * vec[192 + kb];
      }
      named_barrier_sync(1, 384);
      if (mma_thread) mbar_arrive(bar(B_FULL));   // the stage of chunk c is complete
      PSTAMP(ka == 0, c, 14);
    }
    if (failed) {
      if (kt == 0) record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
      if (tma_thread && in_pend) mbar_wait(bar(B_IN), (uint32_t)(in_pend - 1));
      if (mma_thread && kmma_pend) mbar_wait(bar(B_KMMA), (uint32_t)(kmma_pend - 1));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_NCOLS);
}

typedef CUresult (*EncodeTiledFnP)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// [T rows][H*128 cols] bf16 view with a row stride of `stride` elements
bool make_pipe_map(EncodeTiledFnP enc, CUtensorMap* m, const void* base, int64_t T, int H,
                   int64_t stride, int box_cols, bool swizzle) {
  cuuint64_t dims[2] = {(cuuint64_t)H * PD, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)PC};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

PerDeviceOnce g_pipe_attr;

}  // namespace

cudaError_t launch_pipe(const Params& p, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = g_pipe_attr.run(dev, [] {
    return cudaFuncSetAttribute(kda_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PIPE_SMEM);
  });
  if (e != cudaSuccess) return e;
  if (p.vsplit != 1 || p.out_index != nullptr || p.helpers) return cudaErrorInvalidValue;
  const long long blocks = (long long)p.num_seqs * p.heads;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  EncodeTiledFnP enc = reinterpret_cast<EncodeTiledFnP>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  PipeMaps maps;
  // zero-token launches still need valid maps: any 16-byte aligned address (no tile loads)
  const void* qb = p.q ? (const void*)p.q : (const void*)p.dt_bias;
  const void* kb = p.k ? (const void*)p.k : (const void*)p.dt_bias;
  const void* gb = p.g ? (const void*)p.g : (const void*)p.dt_bias;
  const void* vb = p.v ? (const void*)p.v : (const void*)p.dt_bias;
  const void* ob = p.out ? (const void*)p.out : (const void*)p.dt_bias;
  if (!make_pipe_map(enc, &maps.q, qb, p.total_tokens, p.heads, p.s_q, 64, true) ||
      !make_pipe_map(enc, &maps.k, kb, p.total_tokens, p.heads, p.s_k, 64, true) ||
      !make_pipe_map(enc, &maps.g, gb, p.total_tokens, p.heads, p.s_g, 64, true) ||
      !make_pipe_map(enc, &maps.v, vb, p.total_tokens, p.heads, p.s_v, 64, true) ||
      !make_pipe_map(enc, &maps.out, ob, p.total_tokens, p.heads, (int64_t)p.heads * PD, PD, false))
    return cudaErrorInvalidValue;
  kda_pipe_kernel<<<(unsigned)blocks, PNT, PIPE_SMEM, stream>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace kda
