// Split path, second kernel: the serial inter-chunk chain for one value slice of 32 or 16
// columns (P = 4 or 8; P = 2 runs on tcgen05, kda_chain_vs_kernel.cu).
//
// The chunk-parallel k-side kernel has already written, for every (chunk, head),
// a record with -W, Qg (raw q times 2^Gam), Ke (raw k times 2^(Gam_last - Gam)),
// T diag(b), the raw masked QK, the chunk decay 2^Gam_last and the norm scalars,
// as the image of 128-byte-swizzled shared-memory tiles; it is copied in as is
// (one bulk copy) and read with ldmatrix.
// This kernel walks one sequence's chunks in order for one head and one slice of
// DV = 128 / P value columns -- the value-dimension split of "[Kimi-K3][Perf]
// Update FlashKDA for automatic K2 V-split" (PR #52458, Features & motivation),
// which gives low-parallelism batches more CTAs.  Per chunk (S: 128 x DV, fp32):
//   U  = T diag(b) V + (-W) S           (64 x DV)
//   O  = (Qg S + QK (U/|k|)) scale/|q|  -> out
//   S  = diag(2^Gam_last) S + Ke^T (U/|k|)
// The products are narrow (N = DV), so they run as warp-level mma.sync tiles
// (bf16 in, fp32 accumulate) with S held in registers by eight consumer warps; a ninth
// warp copies the records of the next chunks (one ahead, or two for the 16-column slice)
// in while this one is processed, so that no consumer stalls on issuing a copy.  On the
// streamed split path that warp first waits for each record's claim word, the k-side
// kernel running beside this one (kda_stream.cuh).
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_stream.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int NTC = 256;        // 8 consumer warps: the products, staging and stores
constexpr int NT2 = NTC + 32;   // + 1 producer warp: the record and v copies

constexpr int B_WQ = kRecWQ, B_QKE = kRecQKE, B_TB = kRecTB, B_VEC = kRecVec;
constexpr int B_V = kRecBytes + 1024;   // V slice (aligned up to 1 KB)

template <int DV>
struct ChainSmem {
  static constexpr int SP = DV + 8;                 // padded row (bf16) of the staging tiles
  // record buffers: three (records copied in two chunks ahead) where they fit, for the
  // narrowest slice; else two (one chunk ahead, the record after next prefetched to L2)
  static constexpr int BUF = B_V + ((64 * DV * 2 + 1023) / 1024) * 1024;
  static constexpr int NB = (DV == 16) ? 3 : 2;
  static constexpr int OFF_SB = NB * BUF;           // S bf16 [2][128][SP]
  static constexpr int OFF_UB = OFF_SB + 2 * 128 * SP * 2;  // U bf16 [64][SP]
  static constexpr int OFF_BAR = OFF_UB + 64 * SP * 2;
  static constexpr int OFF_MISC = OFF_BAR + 64;
  static constexpr int BYTES = OFF_MISC + 64 + 1024;
  static_assert(BUF % 1024 == 0 && 2 * NB * 8 <= 64, "record buffers and their mbarriers");
  static_assert(BYTES <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t bf2(float lo, float hi) { return pack_bf16x2(lo, hi); }

// byte offset of (row, col) in a tile of 128-byte swizzled rows written by TMA as boxes of
// 64 columns (box b of a `rows`-row tile starts at b * rows * 128)
__device__ __forceinline__ uint32_t sw128(int row, int col, int rows) {
  return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                    (col & 7) * 2);
}
// byte offset of (row, col) of a [rows][DV] bf16 tile written by TMA with the swizzle
// whose span equals the row (32, 64 or 128 bytes): address bits [4, 4+B) ^= bits [7, 7+B)
template <int DV>
__device__ __forceinline__ uint32_t swv(int row, int col) {
  constexpr int B = (DV == 16) ? 1 : (DV == 32 ? 2 : 3);
  const uint32_t off = (uint32_t)(row * DV * 2 + col * 2);
  return off ^ (((off >> 7) & ((1u << B) - 1)) << 4);
}

struct ChainMaps {
  CUtensorMap v;        // v as [T][H*128] bf16, box {DV, 64}
};

// kRowMap: outputs through the out_index row map (its own instantiation)
template <int DV, bool kRowMap>
__global__ void __launch_bounds__(NT2, 1)
    kda_chain_kernel(const __grid_constant__ Params p, const __grid_constant__ ChainMaps maps) {
  using L_ = ChainSmem<DV>;
  constexpr int SP = L_::SP;
  constexpr int P = 128 / DV;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  constexpr int NB = L_::NB;
  const uint32_t bar0 = sb + L_::OFF_BAR;   // full: one mbarrier per record buffer, 8 bytes apart
  const uint32_t empty0 = bar0 + 8 * NB;    // empty: the consumers are done with the buffer

  const int H = p.heads;
  const int unit = blockIdx.x;
  const int part = unit % P;
  const int h = (unit / P) % H;
  const int n = unit / (P * H);
  const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
  const bool streamed = p.stream_sms > 0;
  int* last_s = reinterpret_cast<int*>(sm + L_::OFF_MISC);
  if (tid == 0 && unit < 256) {
    TSTAMP(4 * unit, globaltimer_ns());
    TSTAMP(4 * unit + 3, sm_id());
  }
  if (t0 < 0 || t1 < t0 || (int64_t)t1 > p.total_tokens || p.cu_seqlens[0] != 0) {
    if (tid == 0) record_error(p.status, KDA_ERR_BAD_CU_SEQLENS, 3);
    if (streamed) stream_finish(p, tid, NT2, last_s, [] { __syncthreads(); });
    return;
  }
  if (tid == 0) {
    for (int b = 0; b < NB; ++b) {
      mbar_init(bar0 + 8 * b, 1);
      mbar_init(empty0 + 8 * b, 1);
    }
    mbar_fence_init();
  }
  __syncthreads();
  // chunk c of sequence n was stored in slot floor(t0 / 64) + n + c by the k-side kernel
  const int slot0 = (t0 >> 6) + n;
  const int nch = (t1 - t0 + kChunk - 1) / kChunk;
  const int dv0 = part * DV;
  const size_t HD = (size_t)H * 128;
  const size_t sbase = ((size_t)n * H + h) * 128 * 128;

  auto issue = [&](int i, int buf) {   // (producer lane)
    const uint32_t base = sb + buf * L_::BUF;
    const uint32_t bar = bar0 + 8 * buf;
    const int64_t rec = (int64_t)(slot0 + i) * H + h;
    const unsigned char* src =
        reinterpret_cast<const unsigned char*>(p.status) + kSplitHeader + rec * kRecBytes;
    mbar_expect_tx(bar, kRecBytes + 64 * DV * 2);
    bulk_load(base, src, kRecBytes, bar);   // the record is contiguous at both ends
    tma_load_2d(base + B_V, &maps.v, h * 128 + dv0, t0 + kChunk * i, bar);
  };

  // record + v slice of chunk i -> L2.  With three buffers the record copy itself is issued
  // two chunks ahead, and a bulk prefetch of it as well only adds work for the TMA unit.
  auto prefetch_l2 = [&](int i) {
    if constexpr (NB == 2)
      l2_prefetch(reinterpret_cast<const unsigned char*>(p.status) + kSplitHeader +
                      ((int64_t)(slot0 + i) * H + h) * kRecBytes,
                  kRecBytes);
    tma_prefetch_2d(&maps.v, h * 128 + dv0, t0 + kChunk * i);
  };

  if (warp == NTC / 32) {
    // ---- producer: copies chunk j into buffer j % NB once the consumers are done with
    //      chunk j - NB there, so that no consumer thread stalls on issuing a copy
    if (lane == 0) {
      uint32_t eph = 0;   // bit b: parity of buffer b's next "empty" phase
      int issued = 0;     // chunks 0 .. issued-1 have been copied (buffer j % NB)
      for (int j = 0; j < nch; ++j) {
        const int b = j % NB;
        if (j >= NB) {
          if (!mbar_wait(empty0 + 8 * b, (eph >> b) & 1u)) break;
          eph ^= 1u << b;
        }
        // streamed: the record is published by the k-side kernel running beside
        if (streamed && !stream_wait_record(p, slot0 + j, h, 5)) break;
        if (streamed && j == 0 && unit < 256) TSTAMP(4 * unit + 1, globaltimer_ns());
        issue(j, b);
        issued = j + 1;
        if (j + 2 < nch) prefetch_l2(j + 2);
      }
      // no copy may still be landing when the CTA exits (bounded waits; on the normal path
      // every phase has completed already): buffer b took (issued - b + NB - 1) / NB copies
#pragma unroll
      for (int b = 0; b < NB; ++b)
        if (b < issued) mbar_wait(bar0 + 8 * b, (uint32_t)(((issued - b + NB - 1) / NB - 1) & 1));
    }
    return;
  }

  // ---- state in: this warp's S rows (key channels 16w..16w+15), all DV columns
  float S[DV / 8][4];
#pragma unroll
  for (int nt = 0; nt < DV / 8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int dk = 16 * warp + g + ((e >> 1) << 3);
      const int dv = dv0 + 8 * nt + 2 * t + (e & 1);
      float s = 0.0f;
      if (p.initial_state) {
        const size_t idx = sbase + (size_t)dk * 128 + dv;
        s = p.state_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.initial_state)[idx])
                         : static_cast<const float*>(p.initial_state)[idx];
      }
      S[nt][e] = s;
    }
  auto stage_s = [&](int which) {
    unsigned char* sbf = sm + L_::OFF_SB + which * 128 * SP * 2;
#pragma unroll
    for (int nt = 0; nt < DV / 8; ++nt) {
      const int r0 = 16 * warp + g, c = 8 * nt + 2 * t;
      *reinterpret_cast<uint32_t*>(sbf + (r0 * SP + c) * 2) = bf2(S[nt][0], S[nt][1]);
      *reinterpret_cast<uint32_t*>(sbf + ((r0 + 8) * SP + c) * 2) = bf2(S[nt][2], S[nt][3]);
    }
  };
  stage_s(0);
  uint32_t phase = 0;   // bit b: parity to wait for on buffer b
  group_sync(1, NTC);

  bool failed = false;
  const int mt = warp & 3;                 // 16-token row tile of U and O
  const int ng = warp >> 2;                // which half of the n8 tiles
  constexpr int NPW = DV / 16;             // n8 tiles per warp in U and O
  for (int i = 0; i < nch; ++i) {
    const int buf = i % NB;
    const int sidx = i & 1;                  // S bf16 staging of this chunk
    const int c0 = t0 + kChunk * i;
    const int L = min(kChunk, t1 - c0);
    const bool ok = mbar_wait(bar0 + 8 * buf, (phase >> buf) & 1u);
    if (bar_any(1, NTC, !ok)) { failed = true; break; }
    phase ^= 1u << buf;
    unsigned char* rb = sm + buf * L_::BUF;
    const uint32_t rbs = smem_u32(rb);
    const float* vec = reinterpret_cast<const float*>(rb + B_VEC);   // decay[128], iq[64], ik[64]
    if (L < kChunk) {   // v rows past the sequence end -> 0
      for (int idx = tid; idx < (kChunk - L) * DV / 2; idx += NTC) {
        const int r = L + idx / (DV / 2), c = 2 * (idx % (DV / 2));
        *reinterpret_cast<uint32_t*>(rb + B_V + swv<DV>(r, c)) = 0u;
      }
      group_sync(1, NTC);
    }

    const uint32_t sbf = sb + L_::OFF_SB + sidx * 128 * SP * 2;   // S bf16 of this chunk
    const uint32_t ubf = sb + L_::OFF_UB;
    // ---- U = T diag(b) V + (-W) S and the Qg S half of O (rows 16 mt.., n8 tiles
    //      ng + 2 j).  mma.sync latency, not issue, bounds this loop, so the sums run as
    //      independent accumulator chains at most four deep: U in three partial sums (T V, the
    //      key channels 0-63 of -W S, channels 64-127), Qg S in two; the S fragments are
    //      loaded once for both products.
    float U[NPW][4], U1[NPW][4], U2[NPW][4], O[NPW][4], O1[NPW][4];
#pragma unroll
    for (int j = 0; j < NPW; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) U[j][e] = U1[j][e] = U2[j][e] = O[j][e] = O1[j][e] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a[4], aw0[4], aw1[4], aq0[4], aq1[4];
      {
        const int row = 16 * mt + (lane & 15), col = 16 * ks + 8 * (lane >> 4);
        ldsm_x4(rbs + B_TB + sw128(row, col, 64), a);   // T diag(b)
      }
      {   // -W (tokens 0-63) and Qg (tokens 64-127) of the MN-major [-W | Qg] image, transposed
        const int jj = lane >> 3;
        const int m0 = 16 * mt + 8 * (jj & 1), k = 16 * ks + 8 * (jj >> 1) + (lane & 7);
        ldsm_x4_t(rbs + B_WQ + mnmajor_off(m0, k, 16384), aw0);
        ldsm_x4_t(rbs + B_WQ + mnmajor_off(m0, k + 64, 16384), aw1);
        ldsm_x4_t(rbs + B_WQ + mnmajor_off(64 + m0, k, 16384), aq0);
        ldsm_x4_t(rbs + B_WQ + mnmajor_off(64 + m0, k + 64, 16384), aq1);
      }
      const int kb = 16 * ks + (lane & 15);
      if constexpr (NPW >= 2) {   // two adjacent n8 tiles per ldmatrix
#pragma unroll
        for (int j = 0; j < NPW; j += 2) {
          uint32_t bv[4], b0[4], b1[4];
          const int c = 8 * (NPW * ng + j) + 8 * (lane >> 4);
          ldsm_x4_t(rbs + B_V + swv<DV>(kb, c), bv);
          ldsm_x4_t(sbf + (kb * SP + c) * 2, b0);
          ldsm_x4_t(sbf + ((kb + 64) * SP + c) * 2, b1);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            mma16816(U[j + q], a, bv[2 * q], bv[2 * q + 1]);
            mma16816(U1[j + q], aw0, b0[2 * q], b0[2 * q + 1]);
            mma16816(U2[j + q], aw1, b1[2 * q], b1[2 * q + 1]);
            mma16816(O[j + q], aq0, b0[2 * q], b0[2 * q + 1]);
            mma16816(O1[j + q], aq1, b1[2 * q], b1[2 * q + 1]);
          }
        }
      } else {
        uint32_t bv[2], b0[2], b1[2];
        const int c = 8 * ng;
        ldsm_x2_t(rbs + B_V + swv<DV>(kb, c), bv);
        ldsm_x2_t(sbf + (kb * SP + c) * 2, b0);
        ldsm_x2_t(sbf + ((kb + 64) * SP + c) * 2, b1);
        mma16816(U[0], a, bv[0], bv[1]);
        mma16816(U1[0], aw0, b0[0], b0[1]);
        mma16816(U2[0], aw1, b1[0], b1[1]);
        mma16816(O[0], aq0, b0[0], b0[1]);
        mma16816(O1[0], aq1, b1[0], b1[1]);
      }
    }
    // U / |k| (per token row) -> bf16 staging
    {
      const float ik0 = vec[192 + 16 * mt + g], ik1 = vec[192 + 16 * mt + g + 8];
      unsigned char* ub = sm + L_::OFF_UB;
#pragma unroll
      for (int j = 0; j < NPW; ++j) {
        const int c = 8 * (NPW * ng + j) + 2 * t;
        float u[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = U[j][e] + (U1[j][e] + U2[j][e]);
        *reinterpret_cast<uint32_t*>(ub + ((16 * mt + g) * SP + c) * 2) =
            bf2(u[0] * ik0, u[1] * ik0);
        *reinterpret_cast<uint32_t*>(ub + ((16 * mt + g + 8) * SP + c) * 2) =
            bf2(u[2] * ik1, u[3] * ik1);
      }
    }
    group_sync(1, NTC);

    if constexpr (DV == 16) {
      // ---- 16-column slice: O = (Qg S + QK U') scale/|q| -> out and S = diag(2^Gam_last) S +
      //      Ke^T U' in one k-step loop: the two products' mma chains are independent, so their
      //      latencies overlap, and O's U' fragments are the ones S loads anyway (4% faster at
      //      DV = 16, 4% slower at DV = 32, which keeps the two loops below).  S: this warp's key
      //      rows 16 warp.., all columns; each product's tokens 32-63 go to a second accumulator.
      {
        const float d0 = vec[16 * warp + g], d1 = vec[16 * warp + g + 8];
        float S2[DV / 8][4];
  #pragma unroll
        for (int nt = 0; nt < DV / 8; ++nt) {
          S[nt][0] *= d0;
          S[nt][1] *= d0;
          S[nt][2] *= d1;
          S[nt][3] *= d1;
          S2[nt][0] = S2[nt][1] = S2[nt][2] = S2[nt][3] = 0.0f;
        }
  #pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t aq[4], ak[4];
          {
            const int col = 16 * ks + 8 * (lane >> 4);
            ldsm_x4(rbs + B_QKE + sw128(16 * mt + (lane & 15), col, 192), aq);        // QK rows
            ldsm_x4(rbs + B_QKE + sw128(64 + 16 * warp + (lane & 15), col, 192), ak);  // Ke^T
          }
          {   // both n8 tiles of U' in one ldmatrix; O takes this warp's tile ng
            uint32_t b[4];
            const int k = 16 * ks + (lane & 15), c = 8 * (lane >> 4);
            ldsm_x4_t(ubf + (k * SP + c) * 2, b);
            const uint32_t bo0 = ng ? b[2] : b[0], bo1 = ng ? b[3] : b[1];   // (no indexing by ng)
            mma16816((ks & 1) ? O1[0] : O[0], aq, bo0, bo1);
            mma16816(ks < 2 ? S[0] : S2[0], ak, b[0], b[1]);
            mma16816(ks < 2 ? S[1] : S2[1], ak, b[2], b[3]);
          }
        }
        const int r0 = 16 * mt + g;
        const float iq0 = vec[128 + r0], iq1 = vec[128 + r0 + 8];
        int64_t row0 = c0 + r0, row1 = c0 + r0 + 8;
        bool w0 = r0 < L, w1 = r0 + 8 < L;
        if (kRowMap) {
          row0 = w0 ? out_row(p, row0) : -1;
          row1 = w1 ? out_row(p, row1) : -1;
          w0 = row0 >= 0;
          w1 = row1 >= 0;
        }
  #pragma unroll
        for (int j = 0; j < NPW; ++j) {
          const int c = dv0 + 8 * (NPW * ng + j) + 2 * t;
          if (w0)
            *reinterpret_cast<uint32_t*>(p.out + (size_t)row0 * HD + h * 128 + c) =
                bf2((O[j][0] + O1[j][0]) * iq0, (O[j][1] + O1[j][1]) * iq0);
          if (w1)
            *reinterpret_cast<uint32_t*>(p.out + (size_t)row1 * HD + h * 128 + c) =
                bf2((O[j][2] + O1[j][2]) * iq1, (O[j][3] + O1[j][3]) * iq1);
        }
  #pragma unroll
        for (int nt = 0; nt < DV / 8; ++nt)
  #pragma unroll
          for (int e = 0; e < 4; ++e) S[nt][e] += S2[nt][e];
      }
    } else {
      // ---- O = (Qg S + QK U') scale/|q|  -> out
      {
  #pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t a[4];
          const int row = 16 * mt + (lane & 15), col = 16 * ks + 8 * (lane >> 4);
          ldsm_x4(rbs + B_QKE + sw128(row, col, 192), a);   // QK: rows 0-63 of [QK; Ke]
  #pragma unroll
          for (int j = 0; j < NPW; j += 2) {   // two adjacent n8 tiles per ldmatrix
            uint32_t b[4];
            const int k = 16 * ks + (lane & 15), c = 8 * (NPW * ng + j) + 8 * (lane >> 4);
            ldsm_x4_t(ubf + (k * SP + c) * 2, b);
            mma16816((ks & 1) ? O1[j] : O[j], a, b[0], b[1]);
            mma16816((ks & 1) ? O1[j + 1] : O[j + 1], a, b[2], b[3]);
          }
        }
        const int r0 = 16 * mt + g;
        const float iq0 = vec[128 + r0], iq1 = vec[128 + r0 + 8];
        int64_t row0 = c0 + r0, row1 = c0 + r0 + 8;
        bool w0 = r0 < L, w1 = r0 + 8 < L;
        if (kRowMap) {
          row0 = w0 ? out_row(p, row0) : -1;
          row1 = w1 ? out_row(p, row1) : -1;
          w0 = row0 >= 0;
          w1 = row1 >= 0;
        }
  #pragma unroll
        for (int j = 0; j < NPW; ++j) {
          const int c = dv0 + 8 * (NPW * ng + j) + 2 * t;
          if (w0)
            *reinterpret_cast<uint32_t*>(p.out + (size_t)row0 * HD + h * 128 + c) =
                bf2((O[j][0] + O1[j][0]) * iq0, (O[j][1] + O1[j][1]) * iq0);
          if (w1)
            *reinterpret_cast<uint32_t*>(p.out + (size_t)row1 * HD + h * 128 + c) =
                bf2((O[j][2] + O1[j][2]) * iq1, (O[j][3] + O1[j][3]) * iq1);
        }
      }

      // ---- S = diag(2^Gam_last) S + Ke^T U'   (this warp: key rows 16 warp.., all columns;
      //      tokens 32-63 of the product in a second accumulator)
      {
        const float d0 = vec[16 * warp + g], d1 = vec[16 * warp + g + 8];
        float S2[DV / 8][4];
  #pragma unroll
        for (int nt = 0; nt < DV / 8; ++nt) {
          S[nt][0] *= d0;
          S[nt][1] *= d0;
          S[nt][2] *= d1;
          S[nt][3] *= d1;
          S2[nt][0] = S2[nt][1] = S2[nt][2] = S2[nt][3] = 0.0f;
        }
  #pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t a[4];
          {   // A = Ke^T: rows 64 + dk of [QK; Ke], K = token
            const int row = 16 * warp + (lane & 15), col = 16 * ks + 8 * (lane >> 4);
            ldsm_x4(rbs + B_QKE + sw128(64 + row, col, 192), a);
          }
  #pragma unroll
          for (int nt = 0; nt < DV / 8; nt += 2) {   // two n8 tiles per ldmatrix
            uint32_t b[4];
            const int k = 16 * ks + (lane & 15), c = 8 * nt + 8 * (lane >> 4);
            ldsm_x4_t(ubf + (k * SP + c) * 2, b);
            mma16816(ks < 2 ? S[nt] : S2[nt], a, b[0], b[1]);
            mma16816(ks < 2 ? S[nt + 1] : S2[nt + 1], a, b[2], b[3]);
          }
        }
  #pragma unroll
        for (int nt = 0; nt < DV / 8; ++nt)
  #pragma unroll
          for (int e = 0; e < 4; ++e) S[nt][e] += S2[nt][e];
      }
    }
    stage_s(sidx ^ 1);
    group_sync(1, NTC);
    if (tid == 0) mbar_arrive(empty0 + 8 * buf);   // every consumer is done with the buffer
  }

  if (failed) {   // (the producer lets the copies in flight land before it exits)
    if (tid == 0) record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, 4);
    if (streamed) stream_finish(p, tid, NTC, last_s, [] { group_sync(1, NTC); });
    return;
  }
  // ---- state out
#pragma unroll
  for (int nt = 0; nt < DV / 8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int dk = 16 * warp + g + ((e >> 1) << 3);
      const int dv = dv0 + 8 * nt + 2 * t + (e & 1);
      const size_t idx = sbase + (size_t)dk * 128 + dv;
      if (p.state_bf16)
        static_cast<__nv_bfloat16*>(p.final_state)[idx] = __float2bfloat16_rn(S[nt][e]);
      else
        static_cast<float*>(p.final_state)[idx] = S[nt][e];
    }
  if (tid == 0 && unit < 256) TSTAMP(4 * unit + 2, globaltimer_ns());
  if (streamed) stream_finish(p, tid, NTC, last_s, [] { group_sync(1, NTC); });
}

}  // namespace

// host side ----------------------------------------------------------------
namespace {
typedef CUresult (*EncodeTiledFn2)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_chain_maps(ChainMaps* m, const Params& p, int dv) {
  EncodeTiledFn2 enc = reinterpret_cast<EncodeTiledFn2>(tensor_map_encoder());
  if (!enc) return false;
  const cuuint32_t es[2] = {1, 1};
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.heads * 128, (cuuint64_t)(p.total_tokens > 0 ? p.total_tokens : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)p.s_v * 2};
    cuuint32_t box[2] = {(cuuint32_t)dv, 64};
    const CUtensorMapSwizzle sw = dv == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                           : (dv == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                       : CU_TENSOR_MAP_SWIZZLE_128B);
    if (enc(&m->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(p.v), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int DV>
cudaError_t launch_chain_dv(const Params& p, cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  constexpr int smem = ChainSmem<DV>::BYTES;
  e = attr_once.run(dev, [&]() -> cudaError_t {
    for (auto fn : {kda_chain_kernel<DV, false>, kda_chain_kernel<DV, true>}) {
      const cudaError_t r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  ChainMaps maps;
  if (!make_chain_maps(&maps, p, DV)) return cudaErrorInvalidValue;
  const long long blocks = (long long)p.num_seqs * p.heads * (128 / DV);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(NT2);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.stream_sms > 0 ? 1 : 0;   // streamed: beside the k-side kernel
  if (p.out_index) return cudaLaunchKernelEx(&cfg, kda_chain_kernel<DV, true>, p, maps);
  return cudaLaunchKernelEx(&cfg, kda_chain_kernel<DV, false>, p, maps);
}

}  // namespace

cudaError_t launch_split(const Params& p, cudaStream_t stream) {
  if (p.vsplit != 1 && p.vsplit != 2 && p.vsplit != 4 && p.vsplit != 8) return cudaErrorInvalidValue;
  // streamed (the chain beside the k-side kernel): with SMs to spare
  if (p.stream_sms > 0 &&
      (p.stream_sms != p.num_seqs * p.heads * p.vsplit || p.stream_sms >= p.sm_count))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_kside(p, stream);
  if (e != cudaSuccess) return e;
  // P = 2 on tcgen05 (kda_chain_vs_kernel.cu); the narrower slices keep the warp-level
  // products of this file, which measured 12-23% faster there (per-instruction tcgen05
  // overheads do not shrink with N = 32 or 16)
  switch (p.vsplit) {
    case 1: e = launch_chain_tc(p, stream); break;
    case 2: e = launch_chain_vs(p, stream); break;
    case 4: e = launch_chain_dv<32>(p, stream); break;
    default: e = launch_chain_dv<16>(p, stream); break;
  }
  if (e != cudaSuccess && p.stream_sms > 0) {
    // streamed, and the chain that clears the call's claim words and counters did not start:
    // clear them behind the k-side kernel, so that no later call reads this call's records
    // as its own (the launch error is still returned)
    cudaGetLastError();
    unsigned char* ws = reinterpret_cast<unsigned char*>(p.status);
    cudaMemsetAsync(ws + kStreamCounterWord * sizeof(int), 0,
                    (kStreamStartWord - kStreamCounterWord + 1) * sizeof(int), stream);
    cudaMemsetAsync(ws + helper_claims_offset(p.total_tokens, p.heads, p.num_seqs), 0,
                    (size_t)split_slots(p.total_tokens, p.num_seqs) * p.heads * sizeof(int), stream);
  }
  return e;
}

}  // namespace kda
