// Warp-specialised fused chunked KDA prefill (KDA_KERNEL_PIPE): one CTA per
// (sequence, head), 64-token chunks, the 128 x 128 fp32 state in tensor memory.
//
// The chunk step splits into a state-free half (the "k-side": gate, norms, the
// decay-weighted Gram products and the UT inverse) and the state half (the
// "chain").  The fused kernel of kda_tc_kernel.cuh runs the two halves one after
// the other; here they run on different warps at the same time:
//   warps 0-3   chain of chunk c: thread i <-> TMEM lane i <-> value channel i; besides
//               its own products it turns T into the bf16 operands of G1b and takes the
//               QK rows out of the k-side's accumulator (both while its MMAs run);
//   warps 4-19  k-side of chunk c+1: gate, cumsum, norms, operand tiles, the A
//               extraction and Ke on all 16 warps; per-channel anchors and factors on
//               warps 4-11 (one 32-token block each half), row scales on 12-15, beta on
//               16-17; the UT inverse on warps 4-7; one thread each issues the k-side MMA
//               and the input TMA.
// The k-side hands each chunk over through one shared-memory stage guarded by
// mbarriers (stage full: k-side -> chain; stage parts free: chain -> k-side).
//
// Per chunk (rows r, s = tokens; G = inclusive cumsum of the log2 decay over the
// chunk, per key channel; raw k rows scaled by a power of two to norm <= 1, with
// inv_k = 1 / |k| carried as a per-token scalar; q rows enter as q scale / |q|, so that
// inv_q = 1 below):
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
//   [O^T | S^T] += U_b^T [QK | Ke]             (U_b = bf16(U^T diag(inv_k)), N = 192)
// and the k-side's: [A | QK] = [Kr; Qr] [Kc; Kc2]^T (M = 128, N = 96) over the
// exponent-anchored operands of kda_tc_kernel.cu (two 32-token blocks anchored at
// their 16th token; Kc2 carries the block-0 columns seen from block 1).
//
// Every wait is bounded (about one second); a timeout is recorded as
// KDA_ERR_DEVICE_TIMEOUT and both warp groups leave their loops in step.
#include <cuda.h>

#include <type_traits>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_tc_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace tcc;

constexpr int PC = 64;            // chunk
constexpr int PD = kHeadDim;      // 128
constexpr int PNT = 640;
constexpr int kPipeMaxRankSeqs = 128;

// ---- shared memory (offsets from a 1024-byte aligned base)
// k-side private
constexpr int PS_INQ = 0;             // q tile: two SW128 boxes [64 tok][64 dk], 8 KB apart
constexpr int PS_INK = 16384;         // k tile
constexpr int PS_ING = 32768;         // g tile
constexpr int PS_RKQ = 49152;         // [Kr; Qr] K-major 128 rows x 128 (until the A|QK MMA ends)
constexpr int PS_CKC = 81920;         // [Kc; Kc2] K-major 96 rows x 128
constexpr int PS_NM = PS_RKQ;         // then: N = diag(b inv_k) strict(A) diag(inv_k) [64][NS]
constexpr int PS_Y = PS_NM + 64 * NS * 4;    //       product scratch [32][NS]
// the stage (chain operands of one chunk)
constexpr int PS_WQ = 106496;         // [Kg; Qg] K-major 128 rows (tokens) x 128 (dk)
constexpr int PS_V = 139264;          // v: two SW128 boxes [64 tok][64 dv]
constexpr int PS_TB = 155648;         // T diag(b) K-major 64 x 64
constexpr int PS_TT = 163840;         // T K-major 64 x 64
constexpr int PS_QK = 172032;         // [QK | Ke] MN-major, N = 192 in blocks of 64, 8 KB apart:
constexpr int PS_KE = 180224;         //   QK (n = row r, k = token s; masked, raw), then Ke (n = dk)
constexpr int PS_OST = PS_QK;         // the chain's O transpose scratch (2 KB per warp) once G2 has
                                      //   read QK (the chain writes QK itself)
// small things
constexpr int PS_VEC = 196608;        // [3 by chunk % 3]: decay[128] (unused)[64] ik[64] nbik[64] b[64]
constexpr int kVecFloats = 384;
constexpr int PS_GT = PS_VEC + 3 * kVecFloats * 4;   // quad totals, then anchor offsets [16][128]
constexpr int PS_FAC = PS_GT + 16 * 128 * 4;          // per-channel factors [6][128]
constexpr int PS_SS = PS_FAC + 6 * 128 * 4;           // row sums of squares: q [64], k [64]
constexpr int PS_RSC = PS_SS + 128 * 4;               // row power-of-two scales, bf16x2 [128]
constexpr int PS_BAR = PS_RSC + 128 * 4;              // mbarriers
constexpr int PS_TSLOT = PS_BAR + 16 * 8;   // (12 mbarriers used)
constexpr int PS_FLAGS = PS_TSLOT + 16;
constexpr int PS_TM = PS_FLAGS + 16;      // T [64][NS] fp32
constexpr int PS_END = PS_TM + 64 * NS * 4;
constexpr int PIPE_SMEM = PS_END + 1024;
static_assert(PS_Y + 32 * NS * 4 <= PS_CKC, "N scratch overlaps the Kc tile (read until Ke)");
static_assert(PS_TM % 16 == 0, "T rows are read as float4");
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
constexpr int B_FREEA = 3;   // chain done with [Kg; Qg]
constexpr int B_FREEB = 4;   // chain done with Ke
constexpr int B_KMMA = 5;    // k-side A|QK MMA done
constexpr int B_G1A = 6;     // chain: [X^T | O^T] done
constexpr int B_G1B = 7;     // chain: U^T done
constexpr int B_G2 = 8;      // chain: O^T, S^T updates done
constexpr int B_FREEC = 9;   // chain done with T (fp32), which it turns into its own bf16 operands
constexpr int B_DFREE = 10;  // chain done with the QK rows of the k-side's D (TMEM)
constexpr int B_FULLA = 11;  // the first part of the stage ([Kg; Qg], the chunk's vectors)

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
constexpr uint32_t ID_N64 = idesc_bf16(128, 64, 0, 0);    // X_b x T^T
constexpr uint32_t ID_G2 = idesc_bf16(128, 192, 0, 1);    // U_b x [QK | Ke] (MN-major)

#ifdef KDA_PHASE_STAMPS
// The clock is read in an asm statement with a memory clobber, so that it keeps its place
// relative to the barriers (also asm with memory clobbers) it is meant to bracket.
__device__ __forceinline__ unsigned long long stamp_clock() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t) : : "memory");
  return t;
}
#define PSTAMP(cond, c, slot)                                                       \
  do {                                                                              \
    if ((cond) && p.stamps != nullptr && blockIdx.x == 0 && (c) < 64)               \
      p.stamps[(c) * 32 + (slot)] = stamp_clock();                                  \
  } while (0)
#else
#define PSTAMP(cond, c, slot) \
  do {                        \
  } while (0)
#endif

// One thread's bounded wait for a phase: a non-blocking test first (most waits find the
// phase complete), then hardware-parked retries.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  return mbar_wait_sleep(bar, parity);
}
// The chain's MMA waits are short and on the critical path: poll first (a parked thread
// takes a while to wake), then fall back to the parked, bounded wait.
__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < 4096; ++i)
    if (mbar_test_wait(bar, parity)) return true;
  return mbar_wait_sleep(bar, parity);
}
__device__ __forceinline__ void wgemm16(const float* A, const float* B, float* dst, float sign,
                                     int lane) {
  warp_gemm_16x16<16>(A, B, dst, sign, lane);
}
__device__ __forceinline__ void wgemm32(const float* A, const float* B, float* dst, float sign,
                                     int lane) {
  warp_gemm_16x16<32>(A, B, dst, sign, lane);
}

struct PipeMaps {
  // q, k, g, v as [2H blocks of 64 cols][T rows][64 cols] bf16, box {64, 64, 2}, 128-byte
  // swizzle: one load brings the 128 columns of a head as two SW128 tiles
  CUtensorMap q, k, g, v;
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
  const int zblk = 2 * h;   // first 64-column block of this head in the 3-D views

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
    mbar_init(bar(B_FREEC), 1);
    mbar_init(bar(B_DFREE), 1);
    mbar_init(bar(B_FULLA), 1);
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
    int v_chunk = 0;   // thread 0: the chunk whose v load is pending (bit 0 of pend)
    int cfail = 0;  // chunk at which the loop stopped (all pending phases have its parity)
    if (tid == 0) {
      tma_prefetch_desc(&maps.v);
      if (nch > 0) {
        mbar_expect_tx(bar(B_V), 16384);
        tma_load_3d(sb + PS_V, &maps.v, 0, t0, zblk, bar(B_V));
        pend |= 1;
      }
    }
    // C1a: S_b = bf16(S^T), 64 key columns at a time: the operand of the next chunk's G1a,
    // made as soon as the state is final (before the first chunk, then after each G2)
    auto convert_sb = [&]() {
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t x[32], y[32], pk[16];
        tmem_ld32(tmem + lb + TM_S + hh * 64, x);
        tmem_ld32(tmem + lb + TM_S + hh * 64 + 32, y);
        tmem_wait_ld();
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2)
          pk[j2] = pack_bf16x2(__uint_as_float(x[2 * j2]), __uint_as_float(x[2 * j2 + 1]));
        tmem_st16(tmem + lb + TM_SB + hh * 32, pk);
#pragma unroll
        for (int j2 = 0; j2 < 16; ++j2)
          pk[j2] = pack_bf16x2(__uint_as_float(y[2 * j2]), __uint_as_float(y[2 * j2 + 1]));
        tmem_st16(tmem + lb + TM_SB + hh * 32 + 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      group_sync(4, 128);
    };
    // state in: S^T[dv][dk] -> TMEM (lane = dv)
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t r[32];
      if (p.initial_state == nullptr) {
#pragma unroll
        for (int j2 = 0; j2 < 32; ++j2) r[j2] = 0u;
      } else if (p.state_bf16) {
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.initial_state) + sbase +
                                   (size_t)cb * 32 * PD + dv;
#pragma unroll
        for (int j2 = 0; j2 < 32; ++j2) r[j2] = __float_as_uint(__bfloat162float(src[j2 * PD]));
      } else {
        const float* src = static_cast<const float*>(p.initial_state) + sbase + (size_t)cb * 32 * PD + dv;
#pragma unroll
        for (int j2 = 0; j2 < 32; ++j2) r[j2] = __float_as_uint(src[j2 * PD]);
      }
      tmem_st32(tmem + lb + TM_S + cb * 32, r);
    }
    tmem_wait_st();
    tc_fence_before();
    group_sync(4, 128);
    tc_fence_after();
    convert_sb();

    for (int c = 0; c < nch; ++c) {
      const int c0 = t0 + PC * c;
      const int L = min(PC, t1 - c0);
      const uint32_t par = (uint32_t)(c & 1);
      const float* vec = vecs + (c % 3) * kVecFloats;
      cfail = c;

      // C0: the first part of the stage ([Kg; Qg] and the vectors) and v of chunk c have
      //     landed (thread 0 waits; the group parks on the barrier that carries the outcome);
      //     T comes later, once the k-side has inverted it
      bool ok = true;
      if (tid == 0) {
        ok = wait_phase(bar(B_FULLA), par);
        const bool v_ok = wait_phase(bar(B_V), par);
        if (v_ok) pend &= ~1;
        ok = ok && v_ok;
      }
      if (bar_any(4, 128, !ok)) { failed = true; site = 39; break; }
      PSTAMP(tid == 0, c, 0);
      if (L < PC) {   // v rows past the sequence end -> 0 (they meet zero columns of
                      // T diag(b), but must not carry inf or nan into the product)
        for (int idx = tid; idx < (PC - L) * 16; idx += 128) {
          const int r = L + idx / 16, cc = idx % 16;
          *reinterpret_cast<uint4*>(sm + PS_V + (cc >> 3) * 8192 + r * 128 +
                                    (((cc & 7) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      tc_fence_after();
      PSTAMP(tid == 0, c, 2);
      // G1a: [X^T | O^T] = S_b [Kg | Qg]^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_ts(tmem + TM_XU, tmem + TM_SB + 8 * ks, kdesc(sb + PS_WQ, 128, ks), ID_G1A,
                      ks > 0);
        mma_commit(bar(B_G1A));
        pend |= 2;
        PSTAMP(true, c, 3);
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
      PSTAMP(tid == 0, c, 12);
      tmem_wait_st();
      if (tid == 0) {
        ok = wait_spin(bar(B_G1A), par);
        if (ok) {
          pend &= ~2;
          mbar_arrive(bar(B_FREEA));   // [Kg; Qg] is free
        }
      }
      if (bar_any(4, 128, !ok)) { failed = true; site = 40; break; }
      PSTAMP(tid == 0, c, 4);
      tc_fence_after();
      // C2: X_b = bf16(X^T diag(-b inv_k)), 32 tokens at a time
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t x[32], pk[16];
        tmem_ld32(tmem + lb + TM_XU + hh * 32, x);
        tmem_wait_ld();
        const float* nb = vec + 256 + hh * 32;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 f = ld4(nb + 4 * j4);
          pk[2 * j4] = pack_bf16x2(__uint_as_float(x[4 * j4]) * f.x,
                                   __uint_as_float(x[4 * j4 + 1]) * f.y);
          pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(x[4 * j4 + 2]) * f.z,
                                       __uint_as_float(x[4 * j4 + 3]) * f.w);
        }
        tmem_st16(tmem + lb + TM_XB + hh * 16, pk);
      }
      tmem_wait_st();
      PSTAMP(tid == 0, c, 5);
      if (tid == 0) ok = wait_phase(bar(B_FULL), par);   // T of chunk c
      if (bar_any(4, 128, !ok)) { failed = true; site = 43; break; }
      // C1c: once the k-side has handed over T (fp32): the bf16 operands of G1b, T diag(b)
      //     and T
      {
        const float* Tm = reinterpret_cast<const float*>(sm + PS_TM);
        const float* bv = vec + 320;
#pragma unroll
        for (int it = tid; it < 512; it += 128) {
          const int r = it & 63, c8 = it >> 6;   // row r, columns 8 c8 .. 8 c8 + 7
          const float4 ta = ld4(Tm + r * NS + 8 * c8), tb = ld4(Tm + r * NS + 8 * c8 + 4);
          const float4 ba = ld4(bv + 8 * c8), bb = ld4(bv + 8 * c8 + 4);
          const uint32_t off = kmajor_off(r, 8 * c8, 64);
          st_u128(sm, PS_TB + off,
                  make_uint4(pack_bf16x2(ta.x * ba.x, ta.y * ba.y), pack_bf16x2(ta.z * ba.z, ta.w * ba.w),
                             pack_bf16x2(tb.x * bb.x, tb.y * bb.y), pack_bf16x2(tb.z * bb.z, tb.w * bb.w)));
          st_u128(sm, PS_TT + off,
                  make_uint4(pack_bf16x2(ta.x, ta.y), pack_bf16x2(ta.z, ta.w),
                             pack_bf16x2(tb.x, tb.y), pack_bf16x2(tb.z, tb.w)));
        }
      }
      fence_proxy_async();   // read by G1b
      tc_fence_before();
      group_sync(4, 128);
      PSTAMP(tid == 0, c, 26);
      // G1b: U^T = V^T (T diag b)^T + X_b^T T^T
      if (tid == 0) {
        mbar_arrive(bar(B_FREEC));   // T (fp32) has been read by all four warps
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
      // C2b, while G1b runs: warps 2-3 take the QK rows (TMEM lanes 64-127 of the k-side's D)
      //     into the MN-major bf16 operand of G2, so that D is free for the k-side's next product
      if (warp >= 2) {
        const int r = 32 * (warp & 1) + lane;   // row of QK
#pragma unroll 1
        for (int cq = 0; cq < 4; ++cq) {
          uint32_t a[16];
          // columns 16 cq .. 16 cq + 15 of the row; rows 32-63 take tokens 0-31 from D[:, 64:96]
          tmem_ld16(tmem + lb + TM_D + (warp == 3 && cq < 2 ? 64 + 16 * cq : 16 * cq), a);
          tmem_wait_ld();
          // MN-major: element (r, s) at (s/8) * 1024 + (s%8) * 128 + chunk (r/8 ^ s%8)
          const uint32_t base = (uint32_t)(cq * 2048 + (r & 7) * 2);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int s2 = 16 * cq + e;
            const __nv_bfloat16 val = __float2bfloat16_rn(s2 <= r ? __uint_as_float(a[e]) : 0.0f);
            *reinterpret_cast<__nv_bfloat16*>(
                sm + PS_QK + base + (e >> 3) * 1024 + (e & 7) * 128 + ((((r >> 3) ^ e) & 7) << 4)) = val;
          }
        }
        fence_proxy_async();   // read by G2
        tc_fence_before();
        group_sync(2, 64);
        if (tid == 64) mbar_arrive(bar(B_DFREE));   // the QK rows of D are free
        PSTAMP(tid == 64, c, 27);
      } else if (tid == 0) {   // meanwhile thread 0 waits for G1b
        ok = wait_spin(bar(B_G1B), par);
        if (ok) {
          pend &= ~4;
          PSTAMP(true, c, 28);
          if (c + 1 < nch) {           // v is free: the next chunk's v
            mbar_expect_tx(bar(B_V), 16384);
            tma_load_3d(sb + PS_V, &maps.v, 0, c0 + PC, zblk, bar(B_V));
            pend |= 1;
            v_chunk = c + 1;
          }
        }
      }
      if (bar_any(4, 128, !ok)) { failed = true; site = 41; break; }
      PSTAMP(tid == 0, c, 6);
      tc_fence_after();
      // C3: U_b = bf16(U^T diag(inv_k))
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t x[32], pk[16];
        tmem_ld32(tmem + lb + TM_XU + hh * 32, x);
        tmem_wait_ld();
        const float* ik = vec + 192 + hh * 32;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 f = ld4(ik + 4 * j4);
          pk[2 * j4] = pack_bf16x2(__uint_as_float(x[4 * j4]) * f.x,
                                   __uint_as_float(x[4 * j4 + 1]) * f.y);
          pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(x[4 * j4 + 2]) * f.z,
                                       __uint_as_float(x[4 * j4 + 3]) * f.w);
        }
        tmem_st16(tmem + lb + TM_UB + hh * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      group_sync(4, 128);
      PSTAMP(tid == 0, c, 7);
      // G2: [O^T | S^T] += U_b^T [QK | Ke]^T (one N = 192 group)
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_ts(tmem + TM_O, tmem + TM_UB + 8 * ks, mndesc(sb + PS_QK, 8192, ks), ID_G2, 1);
        mma_commit(bar(B_G2));
        pend |= 8;
        ok = wait_spin(bar(B_G2), par);
        if (ok) {
          pend &= ~8;
          mbar_arrive(bar(B_FREEB));   // Ke is free
        }
      }
      if (bar_any(4, 128, !ok)) { failed = true; site = 42; break; }
      PSTAMP(tid == 0, c, 8);
      tc_fence_after();
      // C4: O -> out rows < L (O is normalised already: the q rows entered the products as
      //     q scale / |q|).  32 tokens at a time: each thread's 32 values (its value channel)
      //     go to a per-warp [32 tok][32 dv] scratch, which the warp then reads back as 32-byte
      //     row pieces for 16-byte global stores.
      {
        unsigned char* ost = sm + PS_OST + warp * 2048;
        const int tok = lane >> 1, half = lane & 1;
#pragma unroll 1
        for (int qp = 0; qp < 2; ++qp) {
          uint32_t x[32];
          tmem_ld32(tmem + lb + TM_O + qp * 32, x);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t)
            *reinterpret_cast<__nv_bfloat16*>(ost + t * 64 + lane * 2) =
                __float2bfloat16_rn(__uint_as_float(x[t]));
          __syncwarp();
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int tl = 16 * hh + tok;   // token within the 32
            const uint4 v0 = *reinterpret_cast<const uint4*>(ost + tl * 64 + half * 32);
            const uint4 v1 = *reinterpret_cast<const uint4*>(ost + tl * 64 + half * 32 + 16);
            const int r = qp * 32 + tl;
            const int64_t orow = r < L ? out_row(p, c0 + r) : -1;   // the row map, if any
            if (orow >= 0) {
              uint4* dst = reinterpret_cast<uint4*>(p.out + orow * HD + xcol + 32 * warp + 16 * half);
              dst[0] = v0;
              dst[1] = v1;
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      group_sync(4, 128);   // the O scratch (over QK) is free for the next chunk's QK
      PSTAMP(tid == 0, c, 10);
      if (c + 1 < nch) {
        tc_fence_after();
        convert_sb();
      }
    }
    if (failed) {
      if (tid == 0) {
        record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
        // let copies and MMAs still in flight end (bounded) before the CTA exits
        const uint32_t fp = (uint32_t)(cfail & 1);
        if (pend & 1) mbar_wait(bar(B_V), (uint32_t)(v_chunk & 1));
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
        if (p.state_bf16) {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.final_state) + sbase + (size_t)cb * 32 * PD + dv;
#pragma unroll
          for (int j2 = 0; j2 < 32; ++j2) dst[j2 * PD] = __float2bfloat16_rn(__uint_as_float(r[j2]));
        } else {
          float* dst = static_cast<float*>(p.final_state) + sbase + (size_t)cb * 32 * PD + dv;
#pragma unroll
          for (int j2 = 0; j2 < 32; ++j2) dst[j2 * PD] = __uint_as_float(r[j2]);
        }
      }
    }
  } else {
    // =========================================================================== k-side
    // 512 threads.  Tile phases: thread (row quad j = warp, channel quad o4 = lane) owns rows
    // 4j .. 4j+3 and key channels 4 o4 .. 4 o4 + 3.  Scalar phases and the inverse: the first
    // 128 threads (warps 4-7).
    const int kt = tid - 128;                 // 0..511
    const int j = kt >> 5;                    // row quad
    const int o4 = lane;                      // channel quad
    const int bsel = j >> 3;                  // 32-token block of this thread's rows
    const bool mma_thread = kt == 0, tma_thread = kt == 32, free_thread = kt == 64;
    float* GT = reinterpret_cast<float*>(sm + PS_GT);
    float* FAC = reinterpret_cast<float*>(sm + PS_FAC);
    float* SS = reinterpret_cast<float*>(sm + PS_SS);
    uint32_t* RSC = reinterpret_cast<uint32_t*>(sm + PS_RSC);
    float* Nm = reinterpret_cast<float*>(sm + PS_NM);
    float* Tm = reinterpret_cast<float*>(sm + PS_TM);
    float* Y = reinterpret_cast<float*>(sm + PS_Y);
    const float gate_scale = expf(p.A_log[h]);
    const float lb2 = p.lower_bound * kLog2e;
    const float sg = -gate_scale * kLog2e;   // sigmoid argument, log2 units: sg (g + dt_bias)
    const float2 sgd01 = make_float2(sg * p.dt_bias[h * PD + 4 * o4], sg * p.dt_bias[h * PD + 4 * o4 + 1]);
    const float2 sgd23 = make_float2(sg * p.dt_bias[h * PD + 4 * o4 + 2], sg * p.dt_bias[h * PD + 4 * o4 + 3]);
    // byte offsets of this thread's 8-byte piece (channels 4 o4 .. 4 o4 + 3) of row 4 j + i in a
    // 128-byte-row SW128 tile: the row part (rows 4j .. 4j + 3 share (r & 7) >> 2 = j & 1) and
    // the 64-column block part, which depends on the tile's row count
    const uint32_t xo = (uint32_t)(((o4 & 15) >> 1) ^ (4 * (j & 1)));
    auto in8_row = [&](int i) -> uint32_t {
      return (uint32_t)((4 * j + i) * 128) + ((xo ^ (uint32_t)i) << 4) + (uint32_t)((o4 & 1) << 3);
    };
    const uint32_t in_row = (uint32_t)((o4 >> 4) * 8192);      // q, k, g input tiles (64 rows)
    const uint32_t rkq_col = (uint32_t)((o4 >> 4) * 16384);    // [Kr; Qr], [Kg; Qg] (128 rows)
    const uint32_t ckc_col = (uint32_t)((o4 >> 4) * 12288);    // [Kc; Kc2] (96 rows)
    int in_pend = 0;      // tma thread: an input load issued and not waited (its parity + 1)
    int kmma_pend = 0;    // the A|QK MMA issued and not waited (its parity + 1)
    auto ld8b = [&](uint32_t off) -> uint2 { return *reinterpret_cast<const uint2*>(sm + off); };
    auto st8b = [&](uint32_t off, uint32_t a, uint32_t b) {
      *reinterpret_cast<uint2*>(sm + off) = make_uint2(a, b);
    };

    auto issue_in = [&](int c) {   // q, k, g of chunk c -> the input tiles; chunk c+1 -> L2
      const int y = t0 + PC * c;
      mbar_expect_tx(bar(B_IN), 49152);
      tma_load_3d(sb + PS_INQ, &maps.q, 0, y, zblk, bar(B_IN));
      tma_load_3d(sb + PS_INK, &maps.k, 0, y, zblk, bar(B_IN));
      tma_load_3d(sb + PS_ING, &maps.g, 0, y, zblk, bar(B_IN));
      if (c + 1 < nch) {
        tma_prefetch_3d(&maps.q, 0, y + PC, zblk);
        tma_prefetch_3d(&maps.k, 0, y + PC, zblk);
        tma_prefetch_3d(&maps.g, 0, y + PC, zblk);
        tma_prefetch_3d(&maps.v, 0, y + PC, zblk);
      }
      in_pend = (c & 1) + 1;
    };
    if (tma_thread) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.g);
      if (nch > 0) issue_in(0);
    }
    // raw beta logits of the next chunk, fetched a chunk ahead (threads 384 .. 447)
    // (kept as the raw bf16 bits, converted only when used a chunk later, so that no warp
    // waits for the global load before the barrier that ends K2)
    unsigned short b_raw = 0;
    const int bt = kt - 384;
    if (bt >= 0 && bt < PC && t0 + bt < t1) b_raw = __bfloat16_as_ushort(p.beta[(size_t)(t0 + bt) * p.s_beta + h]);

    for (int c = 0; c < nch; ++c) {
      const int c0 = t0 + PC * c;
      const int L = min(PC, t1 - c0);
      const uint32_t par = (uint32_t)(c & 1);
      float* vec = vecs + (c % 3) * kVecFloats;
      bool ok = true;
      float cl[4][4];   // inclusive cumsums of this thread's 4 rows, 4 channels

      // ---- K1: gate -> log2 decay, cumsum over this thread's 4 rows; row sums of squares
      PSTAMP(kt == 480, c, 19);
      if (mma_thread) ok = wait_phase(bar(B_IN), par);
      PSTAMP(mma_thread, c, 25);
      if (bar_any(1, 512, !ok)) { failed = true; site = 20; break; }
      if (tma_thread) in_pend = 0;
      PSTAMP(kt == 480, c, 16);
      {
        // two channels per packed fp32x2 operation throughout
        const float2 sg2 = make_float2(sg, sg), lb22 = make_float2(lb2, lb2);
        const float2 one2 = make_float2(1.0f, 1.0f), zero2 = make_float2(0.0f, 0.0f);
        float2 run0 = zero2, run1 = zero2;   // running cumsums, channels 0-1 and 2-3
        float v[8];                           // row sums of squares: q rows 0-3, k rows 0-3
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const bool valid = 4 * j + i < L;   // the same for the whole warp
          const uint32_t off = in_row + in8_row(i);
          const uint2 gv = ld8b(PS_ING + off);
          const float2 z0 = __ffma2_rn(unpack_bf16x2(gv.x), sg2, sgd01);
          const float2 z1 = __ffma2_rn(unpack_bf16x2(gv.y), sg2, sgd23);
          const float2 d0 = __fadd2_rn(make_float2(ex2f(z0.x), ex2f(z0.y)), one2);
          const float2 d1 = __fadd2_rn(make_float2(ex2f(z1.x), ex2f(z1.y)), one2);
          float2 a0 = __fmul2_rn(make_float2(rcpf(d0.x), rcpf(d0.y)), lb22);
          float2 a1 = __fmul2_rn(make_float2(rcpf(d1.x), rcpf(d1.y)), lb22);
          if (!valid) a0 = a1 = zero2;
          run0 = __fadd2_rn(run0, a0);
          run1 = __fadd2_rn(run1, a1);
          cl[i][0] = run0.x; cl[i][1] = run0.y; cl[i][2] = run1.x; cl[i][3] = run1.y;
          const uint2 qv = ld8b(PS_INQ + off), kv = ld8b(PS_INK + off);
          const float2 q01 = unpack_bf16x2(qv.x), q23 = unpack_bf16x2(qv.y);
          const float2 k01 = unpack_bf16x2(kv.x), k23 = unpack_bf16x2(kv.y);
          const float2 sq = __ffma2_rn(q23, q23, __fmul2_rn(q01, q01));
          const float2 sk = __ffma2_rn(k23, k23, __fmul2_rn(k01, k01));
          v[i] = valid ? sq.x + sq.y : 0.0f;
          v[4 + i] = valid ? sk.x + sk.y : 0.0f;
        }
        // the eight row sums over the warp's 32 channel quads, by a butterfly that halves the
        // values each lane carries at each of the first three steps: lane bit 4 picks q or k,
        // bit 3 the row pair, bit 2 the row; lanes with bits 0-1 clear end with a full sum
        const bool h4 = (lane & 16) != 0, h3 = (lane & 8) != 0, h2 = (lane & 4) != 0;
        float w4[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          w4[m] = (h4 ? v[4 + m] : v[m]) + __shfl_xor_sync(0xffffffffu, h4 ? v[m] : v[4 + m], 16);
        float w2[2];
#pragma unroll
        for (int m = 0; m < 2; ++m)
          w2[m] = (h3 ? w4[2 + m] : w4[m]) + __shfl_xor_sync(0xffffffffu, h3 ? w4[m] : w4[2 + m], 8);
        float w1 = (h2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? w2[0] : w2[1], 4);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
        if ((lane & 3) == 0) SS[(h4 ? 64 : 0) + 4 * j + (h3 ? 2 : 0) + (h2 ? 1 : 0)] = w1;
      }
      // quad totals of the cumsum -> GT[j][channel]
      *reinterpret_cast<float4*>(GT + j * 128 + 4 * o4) =
          make_float4(cl[3][0], cl[3][1], cl[3][2], cl[3][3]);
      group_sync(1, 512);
      PSTAMP(kt == 480, c, 17);

      // ---- K2: anchors and factors per key channel, one 32-token block per thread group
      //      (threads < 128: block 0, 128 .. 255: block 1); row norms and scales (256 .. 383);
      //      beta (384 .. 447)
      if (kt < 256) {
        const int d = kt & 127, blk = kt >> 7;
        float Q[8];   // inclusive prefix over the block's eight row quads
        float run = 0.0f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          run += GT[(8 * blk + q) * 128 + d];
          Q[q] = run;
        }
        float g31 = 0.0f;   // block 1: the total of block 0 (for the state decay)
        if (blk) {
#pragma unroll
          for (int q = 0; q < 8; ++q) g31 += GT[q * 128 + d];
        }
        group_sync(5, 256);   // every quad total has been read
        // anchor offsets of the block's quads: the anchor (the block's total up to its 16th
        // token) minus the total before the quad; block 0's total cancels in block 1
#pragma unroll
        for (int q = 0; q < 8; ++q) GT[(8 * blk + q) * 128 + d] = Q[3] - (q ? Q[q - 1] : 0.0f);
        if (!blk) {   // Q = G over tokens 0-31
          FAC[0 * 128 + d] = ex2f(Q[7] - Q[3]);   // Ke, Kc2 of block 0, step 1: 2^(G31 - G)
          FAC[3 * 128 + d] = ex2f(Q[3]);          // Qg/Kg of block 0
          FAC[5 * 128 + d] = ex2f(Q[7]);          // Qg/Kg of block 1, step 2: 2^G31
        } else {      // Q = G - G31 over tokens 32-63
          FAC[1 * 128 + d] = ex2f(Q[7]);          // Ke of block 0, step 2: 2^(G63 - G31)
          FAC[2 * 128 + d] = ex2f(Q[3]);          // Kc2 step 2; Qg/Kg of block 1, step 1
          FAC[4 * 128 + d] = ex2f(Q[7] - Q[3]);   // Ke of block 1
          vec[d] = ex2f(g31 + Q[7]);              // decay of the state: 2^G63
        }
      } else if (kt < 384) {
        const int rr = kt - 256, r = rr & 63;
        const float ss = SS[rr];
        // ss < 2^(e+1) -> |row| < 2^ceil((e+1)/2): rows enter the operands times 2^-sh
        const int e = ((__float_as_int(ss) >> 23) & 255) - 127;
        const int sh = max(-60, min(60, (e + 2) >> 1));
        const float rs = (r < L) ? rsqrtf(ss + kL2Eps) : 0.0f;
        if (rr < 64) {
          // q rows enter the operands as q scale / |q| (their norm is scale): O comes out of
          // the products already normalised
          RSC[rr] = pack_bf16x2(p.scale * rs, p.scale * rs);
        } else {
          vec[192 + r] = rs * __int_as_float((127 + sh) << 23);   // 1 / |k| against k 2^-sh
          const uint32_t bb = (uint32_t)(127 - sh) << 7;           // bf16 bits of 2^-sh
          RSC[rr] = bb | (bb << 16);
        }
      } else if (bt < PC) {
        vec[320 + bt] = (bt < L) ? sigm(__uint_as_float((uint32_t)b_raw << 16)) : 0.0f;   // b
        b_raw = 0;
        if (c0 + PC + bt < t1) b_raw = __bfloat16_as_ushort(p.beta[(size_t)(c0 + PC + bt) * p.s_beta + h]);
      }
      // the barrier that ends K2 also carries the wait for the chain to have read [Kg; Qg] of
      // the previous chunk (K3 overwrites it)
      if (c > 0 && mma_thread) ok = wait_phase(bar(B_FREEA), (uint32_t)((c - 1) & 1));
      if (bar_any(1, 512, !ok)) { failed = true; site = 21; break; }
      PSTAMP(kt == 480, c, 18);

      // ---- K3: operand tiles [Kr; Qr], [Kc; Kc2] (own), Kg, Qg (stage).  The warp's rows lie in
      //      one 32-token block (bsel), so the block's variant is chosen once per warp.
      {
        if (kt < PC) vec[256 + kt] = -vec[320 + kt] * vec[192 + kt];   // -b inv_k, for the chain
        const float4 mE4 = ld4(GT + j * 128 + 4 * o4);
        const float2 nm01 = make_float2(-mE4.x, -mE4.y), nm23 = make_float2(-mE4.z, -mE4.w);
        // block 0: Kc2 = Kc 2^(G31 - anchor0) 2^(anchor1 - G31), Kg = Kr 2^anchor0;
        // block 1: Kg = Kr 2^(anchor1 - G31) 2^G31 (Kc2 has no block-1 rows).  The factors are
        // applied one after the other, never multiplied together first: their product alone
        // can leave the fp32 range (2^(anchor1 - anchor0) under strong decay) while the
        // operand it scales stays representable.
        auto tiles = [&](auto blk) {
          constexpr bool B0 = decltype(blk)::value;
          const float4 fc4 = ld4(FAC + 2 * 128 + 4 * o4);
          const float4 fq4 = ld4(FAC + (B0 ? 3 : 5) * 128 + 4 * o4);
          const float4 fa4 = ld4(FAC + 0 * 128 + 4 * o4);
          // Kg/Qg: (E [fc]) fq; Kc2: (Ei fa) fc
          const float2 fc01 = make_float2(fc4.x, fc4.y), fc23 = make_float2(fc4.z, fc4.w);
          const float2 fq01 = make_float2(fq4.x, fq4.y), fq23 = make_float2(fq4.z, fq4.w);
          const float2 fa01 = make_float2(fa4.x, fa4.y), fa23 = make_float2(fa4.z, fa4.w);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = 4 * j + i;
            const uint32_t ro = in8_row(i);
            uint2 qv = ld8b(PS_INQ + in_row + ro), kv = ld8b(PS_INK + in_row + ro);
            if (r >= L) qv = kv = make_uint2(0, 0);
            const uint32_t rq = RSC[r], rk = RSC[64 + r];
            const uint32_t q2[2] = {bmul2(qv.x, rq), bmul2(qv.y, rq)};
            const uint32_t k2[2] = {bmul2(kv.x, rk), bmul2(kv.y, rk)};
            uint32_t kr[2], qr[2], kc[2], kc2[2], kg[2], qg[2];
#pragma unroll
            for (int pq = 0; pq < 2; ++pq) {
              const float2 x = __fadd2_rn(make_float2(cl[i][2 * pq], cl[i][2 * pq + 1]),
                                          pq ? nm23 : nm01);
              const float2 E = make_float2(ex2f(x.x), ex2f(x.y));
              const float2 Ei = make_float2(ex2f(-x.x), ex2f(-x.y));
              const uint32_t E2 = pack_bf16x2(E.x, E.y), Ei2 = pack_bf16x2(Ei.x, Ei.y);
              kr[pq] = bmul2(k2[pq], E2);
              qr[pq] = bmul2(q2[pq], E2);
              kc[pq] = bmul2(k2[pq], Ei2);
              const float2 gq = B0 ? __fmul2_rn(E, pq ? fq23 : fq01)
                                   : __fmul2_rn(__fmul2_rn(E, pq ? fc23 : fc01), pq ? fq23 : fq01);
              const uint32_t gq2 = pack_bf16x2(gq.x, gq.y);
              if (B0) {
                const float2 cc = __fmul2_rn(__fmul2_rn(Ei, pq ? fa23 : fa01), pq ? fc23 : fc01);
                kc2[pq] = bmul2(k2[pq], pack_bf16x2(cc.x, cc.y));
              }
              qg[pq] = bmul2(q2[pq], gq2);
              kg[pq] = bmul2(k2[pq], gq2);
            }
            st8b(PS_RKQ + rkq_col + ro, kr[0], kr[1]);
            st8b(PS_RKQ + rkq_col + 8192 + ro, qr[0], qr[1]);
            st8b(PS_CKC + ckc_col + ro, kc[0], kc[1]);
            if (B0) st8b(PS_CKC + ckc_col + 8192 + ro, kc2[0], kc2[1]);
            st8b(PS_WQ + rkq_col + ro, kg[0], kg[1]);
            st8b(PS_WQ + rkq_col + 8192 + ro, qg[0], qg[1]);
          }
        };
        if (bsel == 0)
          tiles(std::true_type{});
        else
          tiles(std::false_type{});
        PSTAMP(kt == 480, c, 20);
        fence_proxy_async();
        group_sync(1, 512);
        if (mma_thread) mbar_arrive(bar(B_FULLA));   // [Kg; Qg] and the vectors of chunk c
        PSTAMP(kt == 480, c, 21);

        // ---- K4: [A | QK] on the tensor cores, once the chain has taken the previous QK out
        //      of D; the next chunk's inputs (the input tiles are free)
        if (mma_thread) {
          if (c > 0) ok = wait_phase(bar(B_DFREE), (uint32_t)((c - 1) & 1));
          if (ok) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_bf16(tmem + TM_D, kdesc(sb + PS_RKQ, 128, ks), kdesc(sb + PS_CKC, 96, ks),
                       ID_D96, ks > 0);
            mma_commit(bar(B_KMMA));
            kmma_pend = (int)par + 1;
          }
          PSTAMP(true, c, 31);
        }
        if (tma_thread && c + 1 < nch) issue_in(c + 1);
        PSTAMP(tma_thread, c, 30);
      }
      if (mma_thread && ok) ok = wait_phase(bar(B_KMMA), par);
      if (bar_any(1, 512, !ok)) { failed = true; site = 24; break; }
      kmma_pend = 0;
      PSTAMP(kt == 480, c, 22);
      tc_fence_after();

      // ---- K5: warps with w % 4 in {0, 1} read TMEM lanes 0-63 (rows of A), a 16-column
      //      quarter of the row's 64 columns each -> N (fp32) and -b inv_k; the other eight
      //      warps form Ke = Kc 2^(G_last - anchor) (stage) once the chain's last product of
      //      the previous chunk has read Ke
      // (one barrier for both waits: Ke's buffer here, T's before K6)
      if (c > 0) {
        if (free_thread) ok = wait_phase(bar(B_FREEB), (uint32_t)((c - 1) & 1));
        if (mma_thread) ok = wait_phase(bar(B_FREEC), (uint32_t)((c - 1) & 1));
        if (bar_any(1, 512, !ok)) { failed = true; site = 25; break; }
      }
      PSTAMP(kt == 480, c, 1);
      if ((warp & 3) < 2) {
        const int q4 = warp & 3, cq = (warp - 4) >> 2;
        const uint32_t lbase = (uint32_t)(32 * q4) << 16;
        const int r = 32 * q4 + lane;
        const float* ik = vec + 192;
        uint32_t a[16];
        if (!(q4 == 0 && cq >= 2)) {   // rows < 32 have no tokens >= 32 below the diagonal
          // columns 16 cq .. 16 cq + 15 of the row; rows 32-63 take tokens 0-31 from D[:, 64:96]
          tmem_ld16(tmem + lbase + TM_D + (q4 == 1 && cq < 2 ? 64 + 16 * cq : 16 * cq), a);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) a[e] = 0u;
        }
        float* nrow = Nm + r * NS + 16 * cq;
        const float br = vec[320 + r] * ik[r];
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const float4 kk = ld4(ik + 16 * cq + 4 * s4);
          const float kv4[4] = {kk.x, kk.y, kk.z, kk.w};
          float w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s2 = 16 * cq + 4 * s4 + e;
            w[e] = (s2 < r) ? br * kv4[e] * __uint_as_float(a[4 * s4 + e]) : 0.0f;
          }
          *reinterpret_cast<float4*>(nrow + 4 * s4) = make_float4(w[0], w[1], w[2], w[3]);
        }
      } else {
        // rows 8 kk .. 8 kk + 7, channels 4 o4 .. 4 o4 + 3
        const int kk = 2 * ((warp - 4) >> 2) + (warp & 1);
        const int kb = kk >> 2;   // 32-token block
        const float4 fa4 = ld4(FAC + (kb ? 4 : 0) * 128 + 4 * o4);
        const float4 fb4 = ld4(FAC + 1 * 128 + 4 * o4);
        // block 0: 2^(G31 - anchor0) then 2^(G63 - G31), one after the other (their product
        // alone can underflow); block 1: 2^(G63 - anchor1)
        const float2 fa01 = make_float2(fa4.x, fa4.y), fa23 = make_float2(fa4.z, fa4.w);
        const float2 fb01 = make_float2(fb4.x, fb4.y), fb23 = make_float2(fb4.z, fb4.w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 8 * kk + i;
          const uint2 kcv = ld8b(PS_CKC + kmajor_off(r, 4 * o4, 96));
          float2 a = __fmul2_rn(unpack_bf16x2(kcv.x), fa01), b = __fmul2_rn(unpack_bf16x2(kcv.y), fa23);
          if (!kb) {
            a = __fmul2_rn(a, fb01);
            b = __fmul2_rn(b, fb23);
          }
          st8b(PS_KE + mnmajor_off(4 * o4, r, 8192), pack_bf16x2(a.x, a.y), pack_bf16x2(b.x, b.y));
        }
        fence_proxy_async();
      }
      tc_fence_before();
      group_sync(1, 512);
      PSTAMP(kt == 480, c, 24);

      // ---- K6 (threads < 128): T = (I + N)^-1: 16 x 16 diagonal blocks by substitution
      //      (fp32), then the off-diagonal blocks as tf32 warp products, 16 -> 32 -> 64
      if (kt < 128) {
        const int wb = kt >> 5;
        for (int idx = kt; idx < 6 * 64; idx += 128) {   // T above the diagonal blocks is zero
          const int b = idx >> 6, e = idx & 63;
          const int bi = (b < 3) ? 0 : (b < 5 ? 1 : 2);
          const int bj = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
          *reinterpret_cast<float4*>(Tm + (bi * 16 + (e >> 2)) * NS + bj * 16 + 4 * (e & 3)) =
              make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (wb < 2) {
          // warp wb: the diagonal blocks 2 wb (lanes 0-15) and 2 wb + 1 (lanes 16-31), lane =
          // column, by forward substitution four columns of N at a time (16-byte row pieces);
          // then the pair's off-diagonal block T[2wb+1][2wb] = -T[2wb+1]^ N[2wb+1][2wb] T[2wb]^
          // (^ = diagonal block), which needs nothing from the other warps
          const int ob = (lane >> 4) * 16 + 32 * wb, jj = lane & 15;
          float x[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = (i == jj) ? 1.0f : 0.0f;
#pragma unroll
          for (int k0 = 0; k0 < 16; k0 += 4) {
#pragma unroll
            for (int i = k0 + 1; i < 16; ++i) {
              const float4 nv = ld4(Nm + (ob + i) * NS + ob + k0);
              float acc = fmaf(-nv.x, x[k0], x[i]);
              if (i > k0 + 1) acc = fmaf(-nv.y, x[k0 + 1], acc);
              if (i > k0 + 2) acc = fmaf(-nv.z, x[k0 + 2], acc);
              if (i > k0 + 3) acc = fmaf(-nv.w, x[k0 + 3], acc);
              x[i] = acc;
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) Tm[(ob + i) * NS + ob + jj] = x[i];
          __syncwarp();
          const int ro = (2 * wb + 1) * 16, co = 2 * wb * 16;
          float* Yw = Y + wb * 16 * NS;
          wgemm16(Nm + ro * NS + co, Tm + co * NS + co, Yw, 1.0f, lane);
          __syncwarp();
          wgemm16(Tm + ro * NS + ro, Yw, Tm + ro * NS + co, -1.0f, lane);
          __syncwarp();
        }
        group_sync(3, 128);
        const int mi = wb >> 1, ni = wb & 1;   // Y2 = N[32:64, 0:32] T[0:32, 0:32]
        wgemm32(Nm + (32 + 16 * mi) * NS, Tm + 16 * ni, Y + 16 * mi * NS + 16 * ni, 1.0f, lane);
        group_sync(3, 128);                    // T[32:64, 0:32] = -T[32:64, 32:64] Y2
        wgemm32(Tm + (32 + 16 * mi) * NS + 32, Y + 16 * ni, Tm + (32 + 16 * mi) * NS + 16 * ni,
                -1.0f, lane);
      }
      group_sync(1, 512);
      if (mma_thread) mbar_arrive(bar(B_FULL));   // the stage of chunk c is complete
      PSTAMP(kt == 480, c, 29);
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

// [2H blocks][T rows][64 cols] bf16 view of a [T][H*128] tensor with a row stride of
// `stride` elements: dims {64, T, 2H}, strides {stride * 2, 128} bytes; box {64, 64, 2}
bool make_pipe_map(EncodeTiledFnP enc, CUtensorMap* m, const void* base, int64_t T, int H,
                   int64_t stride) {
  cuuint64_t dims[3] = {64, (cuuint64_t)(T > 0 ? T : 1), (cuuint64_t)(2 * H)};
  cuuint64_t strides[2] = {(cuuint64_t)stride * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)PC, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
  if (p.vsplit != 1 || p.helpers) return cudaErrorInvalidValue;
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
  if (!make_pipe_map(enc, &maps.q, qb, p.total_tokens, p.heads, p.s_q) ||
      !make_pipe_map(enc, &maps.k, kb, p.total_tokens, p.heads, p.s_k) ||
      !make_pipe_map(enc, &maps.g, gb, p.total_tokens, p.heads, p.s_g) ||
      !make_pipe_map(enc, &maps.v, vb, p.total_tokens, p.heads, p.s_v))
    return cudaErrorInvalidValue;
  kda_pipe_kernel<<<(unsigned)blocks, PNT, PIPE_SMEM, stream>>>(p, maps);
  return cudaGetLastError();
}

}  // namespace kda
