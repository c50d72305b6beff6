// Split path, second kernel for a value dimension split in two (P = 2): the serial
// inter-chunk chain of one value slice, on tcgen05.
//
// The value-dimension split is the one of "[Kimi-K3][Perf] Update FlashKDA for automatic K2
// V-split" (PR #52458, Features & motivation): P CTAs per (sequence, head), each owning
// DV = 128 / P value columns of the state.  Here each slice CTA keeps its state slice
// S (128 key channels x DV value channels, fp32) in tensor memory with lane = key channel,
// so that every product has M = 128 rows and N = DV columns.  Per chunk, from the record
// the k-side kernel wrote (-W, Qg, T diag(b), QK, Ke and the per-token scalars):
//   X    = [-W; Qg] S_b             rows 0-63: -W S, rows 64-127: Qg S     (S_b = bf16 S)
//   Y    = [T diag(b); *] V         rows 0-63: T diag(b) V
//   U_b  = bf16((X + Y)[rows 0-63] diag(1/|k|))                          (64 tokens x DV)
//   X   += [*; QK] U_b              rows 64-127: O = Qg S + QK U_b
//   S    = diag(2^Gam_last) S + Ke^T U_b
//   out  = O diag(scale/|q|)
// which is the chunk recurrence of the gated delta rule in the WY/UT form of the FlashKDA
// prefill PR report (PR #55737, Features & motivation), restricted to DV value columns.
//
// The A operands are the record images as they land in shared memory: M = 128 stacks two
// 64-row products, and the rows marked * are the neighbouring 8 KB of the stage (record
// bytes or the v tile).  Their products land only in accumulator rows that are never
// read (Y rows 64-127; X rows 0-63 after U_b has been taken out), and an MMA row depends
// only on its own A row.  S_b, U_b (written here) and the v tile (TMA) are MN-major B
// operands: K rows of 128 bytes in the 128-byte swizzle, of which the first DV columns are
// the operand.  X is double-buffered, so that O of chunk c is drained while the first
// products of chunk c+1 run; a producer warp copies the records and v tiles in, two stages
// deep, so that no consumer stalls on issuing a copy.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_stream.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

// 8 consumer warps: warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 and value columns
// [DV/2 (w / 4), DV/2 (w / 4 + 1)) of the slice; a ninth warp copies the records in
constexpr int NTC4 = 256;
constexpr int NT4 = NTC4 + 32;

// ---- shared memory (offsets from a 1024-byte aligned base)
constexpr int VS_V = kRecBytes + 1024;        // v tile [64 tok][64 cols] SW128 after the record
constexpr int VS_STAGE = VS_V + 8192;         // record + v of one chunk
constexpr int VS_SB = 2 * VS_STAGE;           // S_b: MN-major [128 dk][DV] in 128-byte rows
constexpr int VS_UB = VS_SB + 16384;          // U_b: MN-major [64 tok][DV] in 128-byte rows
constexpr int VS_BAR = VS_UB + 8192;          // full[2], empty[2], g1, g2
constexpr int VS_TSLOT = VS_BAR + 48;
constexpr int VS_USED = VS_TSLOT + 16;
constexpr int VS_BYTES = VS_USED + 1024;
static_assert(VS_V % 1024 == 0 && VS_STAGE % 1024 == 0 && VS_SB % 1024 == 0 &&
                  VS_UB % 1024 == 0,
              "SW128 tiles are 1024-byte aligned");
// the stacked A operands read 8 KB past T diag(b) and 8 KB before QK: inside the stage
static_assert(kRecTB + 16384 <= VS_STAGE && kRecQKE >= 8192, "stacked operand rows");
static_assert(VS_BYTES <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint64_t kdesc4(uint32_t tile, int ks) {   // K-major, K = 64
  return sdesc_sw128(tile + ks * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc4(uint32_t tile, uint32_t lbo, int ks) {   // MN-major
  return sdesc_sw128(tile + ks * 2048, lbo, 1024);
}
// byte offset of 16-byte piece j (columns 8j .. 8j+7) of K row k of an MN-major SW128 tile
__device__ __forceinline__ uint32_t mn_piece(int k, int j) {
  return (uint32_t)((k >> 3) * 1024 + (k & 7) * 128 + ((j ^ (k & 7)) << 4));
}

// DV consecutive TMEM columns of this thread's lane (16 at a time)
template <int DV>
__device__ __forceinline__ void tmem_ld_dv(uint32_t taddr, uint32_t (&r)[DV]) {
#pragma unroll
  for (int b = 0; b < DV / 16; ++b)
    tmem_ld16(taddr + 16 * b, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * b));
}
template <int DV>
__device__ __forceinline__ void tmem_st_dv(uint32_t taddr, const uint32_t (&r)[DV]) {
#pragma unroll
  for (int b = 0; b < DV / 16; ++b)
    tmem_st16(taddr + 16 * b, *reinterpret_cast<const uint32_t(*)[16]>(r + 16 * b));
}

struct ChainVsMaps {
  CUtensorMap v;   // v as [T][H*128] bf16, box {64 cols, 64 rows}, 128-byte swizzle
};

template <int DV, bool kRowMap>
__global__ void __launch_bounds__(NT4, 1)
    kda_chain_vs_kernel(const __grid_constant__ Params p, const __grid_constant__ ChainVsMaps maps) {
  static_assert(DV % 32 == 0, "two column halves of 16 or more");
  constexpr int P = 128 / DV;
  constexpr int DH = DV / 2;   // columns per thread
  constexpr uint32_t T_X0 = 0, T_Y = 2 * DV, T_S = 3 * DV, T_COLS = 4 * DV;
  // [-W; Qg] (MN-major) x S_b;  K-major A x MN-major B (T diag b, QK, Ke against V, U_b)
  constexpr uint32_t ID_MN = idesc_bf16(128, DV, 1, 1);
  constexpr uint32_t ID_KM = idesc_bf16(128, DV, 0, 1);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + VS_TSLOT);
  const uint32_t bar_full0 = sb + VS_BAR, bar_empty0 = bar_full0 + 16;
  const uint32_t bar_g1 = bar_full0 + 32, bar_g2 = bar_full0 + 40;

  const int H = p.heads;
  const int unit = blockIdx.x;
  const int part = unit % P;
  const int h = (unit / P) % H;
  const int n = unit / (P * H);
  const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
  const bool streamed = p.stream_sms > 0;
  int* last_s = reinterpret_cast<int*>(sm + VS_TSLOT + 4);
  if (t0 < 0 || t1 < t0 || (int64_t)t1 > p.total_tokens || p.cu_seqlens[0] != 0) {
    if (tid == 0) record_error(p.status, KDA_ERR_BAD_CU_SEQLENS, 6);
    if (streamed) stream_finish(p, tid, NT4, last_s, [] { __syncthreads(); });
    return;
  }
  const int nch = (t1 - t0 + kChunk - 1) / kChunk;
  const int slot0 = (t0 >> 6) + n;   // chunk c of sequence n sits in slot floor(t0 / 64) + n + c
  const int dv0 = part * DV;
  const size_t HD = (size_t)H * 128;
  const size_t sbase = ((size_t)n * H + h) * 128 * 128;
  const int xcol = h * 128 + dv0;

  if (tid == 0) {
    mbar_init(bar_full0, 1);
    mbar_init(bar_full0 + 8, 1);
    mbar_init(bar_empty0, 1);
    mbar_init(bar_empty0 + 8, 1);
    mbar_init(bar_g1, 1);
    mbar_init(bar_g2, 1);
    mbar_fence_init();
    tma_prefetch_desc(&maps.v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), T_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int q4 = warp & 3;
  const uint32_t lb = (uint32_t)(32 * q4) << 16;   // this warp's TMEM lane quadrant
  const int row = 32 * q4 + lane;                  // TMEM lane: key channel, or accumulator row
  const int ch = DH * (warp >> 2);                 // first column of this thread's half

  auto rec_src = [&](int i) {
    return reinterpret_cast<const unsigned char*>(p.status) + kSplitHeader +
           ((int64_t)(slot0 + i) * H + h) * kRecBytes;
  };
  auto issue = [&](int i) {   // (producer) record + v columns [dv0, dv0 + 64) of chunk i -> stage i & 1
    const uint32_t st = sb + (i & 1) * VS_STAGE;
    const uint32_t bar = bar_full0 + 8 * (i & 1);
    mbar_expect_tx(bar, kRecBytes + 8192);
    bulk_load(st, rec_src(i), kRecBytes, bar);   // the record is contiguous at both ends
    tma_load_2d(st + VS_V, &maps.v, xcol, t0 + kChunk * i, bar);
  };
  auto prefetch_l2 = [&](int i) {
    l2_prefetch(rec_src(i), kRecBytes);
    tma_prefetch_2d(&maps.v, xcol, t0 + kChunk * i);
  };
  if (warp == NTC4 / 32) {
    // ---- producer: copies chunk j into stage j & 1 once the consumers are done with chunk
    //      j - 2 there, so that no consumer stalls on issuing a copy
    if (lane == 0) {
      uint32_t eph = 0;   // bit b: parity of stage b's next "empty" phase
      int issued = 0;
      for (int j = 0; j < nch; ++j) {
        const int b = j & 1;
        if (j >= 2) {
          if (!mbar_wait(bar_empty0 + 8 * b, (eph >> b) & 1u)) break;
          eph ^= 1u << b;
        }
        // streamed: the record is published by the k-side kernel running beside
        if (streamed && !stream_wait_record(p, slot0 + j, h, 7)) break;
        issue(j);
        issued = j + 1;
        if (j + 1 < nch) prefetch_l2(j + 1);
      }
      // no copy may still be landing when the CTA exits (bounded; on the normal path every
      // phase has completed already): stage b took (issued - b + 1) / 2 copies
      for (int b = 0; b < 2; ++b)
        if (b < issued) mbar_wait(bar_full0 + 8 * b, (uint32_t)(((issued - b + 1) / 2 - 1) & 1));
    }
    return;
  }

  // ---- state in: row (key channel) `row` of the slice, this thread's DH values -> TMEM
  {
    uint32_t r[DH];
#pragma unroll
    for (int j = 0; j < DH; ++j) r[j] = 0u;
    if (p.initial_state) {
      const size_t idx = sbase + (size_t)row * 128 + dv0 + ch;
      if (p.state_bf16) {
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(p.initial_state) + idx);
#pragma unroll
        for (int j = 0; j < DH / 8; ++j) {
          const uint4 w = src[j];
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            r[8 * j + 2 * e] = ww[e] << 16;
            r[8 * j + 2 * e + 1] = ww[e] & 0xFFFF0000u;
          }
        }
      } else {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.initial_state) + idx);
#pragma unroll
        for (int j = 0; j < DH / 4; ++j) {
          const float4 w = src[j];
          r[4 * j] = __float_as_uint(w.x);
          r[4 * j + 1] = __float_as_uint(w.y);
          r[4 * j + 2] = __float_as_uint(w.z);
          r[4 * j + 3] = __float_as_uint(w.w);
        }
      }
    }
    tmem_st_dv<DH>(tmem + lb + T_S + ch, r);
    tmem_wait_st();
  }

  // O of a finished chunk (warps with q4 >= 2: X rows 64-127 = its tokens) -> out
  auto drain_o = [&](uint32_t tx, int c0, int L, float iq, int64_t orow) {
    const int t = row - 64;
    uint32_t x[DH];
    tmem_ld_dv<DH>(tmem + lb + tx + ch, x);
    tmem_wait_ld();
    const int64_t orw = kRowMap ? orow : (int64_t)(c0 + t);
    if (t < L && orw >= 0) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)orw * HD + xcol + ch);
#pragma unroll
      for (int j = 0; j < DH / 8; ++j)
        dst[j] = make_uint4(pack_bf16x2(__uint_as_float(x[8 * j]) * iq, __uint_as_float(x[8 * j + 1]) * iq),
                            pack_bf16x2(__uint_as_float(x[8 * j + 2]) * iq, __uint_as_float(x[8 * j + 3]) * iq),
                            pack_bf16x2(__uint_as_float(x[8 * j + 4]) * iq, __uint_as_float(x[8 * j + 5]) * iq),
                            pack_bf16x2(__uint_as_float(x[8 * j + 6]) * iq, __uint_as_float(x[8 * j + 7]) * iq));
    }
  };

  uint32_t phase = 0;   // bit b: parity of stage b's next fill
  uint32_t ph_mma = 0;  // one fill per chunk of both bar_g1 and bar_g2
  int mma_out = 0;      // 1: group 1 committed and not waited, 2: group 2 (thread 0)
  bool failed = false;
  int site = 0;
  // the previous chunk's O drain: its scalars, kept past the reuse of its stage
  float iq_prev = 0.0f;
  int64_t orow_prev = -1;
  int L_prev = 0;

  for (int i = 0; i < nch; ++i) {
    const int buf = i & 1;
    const int c0 = t0 + kChunk * i;
    const int L = min(kChunk, t1 - c0);
    const uint32_t st = sb + buf * VS_STAGE;
    unsigned char* stp = sm + buf * VS_STAGE;
    const float* vec = reinterpret_cast<const float*>(stp + kRecVec);   // decay, iq, ik
    const uint32_t tx = T_X0 + (uint32_t)(buf * DV);

    // ---- 1. the record and v of this chunk have landed; the next chunk's fetch goes into
    //      the other stage (its last reader, group 2 of the previous chunk, has completed)
    {
      const bool ok = tid != 0 || mbar_wait(bar_full0 + 8 * buf, (phase >> buf) & 1u);
      if (bar_any(1, NTC4, !ok)) { failed = true; site = 61; break; }
      phase ^= 1u << buf;
    }
    if (L < kChunk) {   // v rows past the sequence end -> 0
      for (int idx = tid; idx < (kChunk - L) * 8; idx += NTC4)
        *reinterpret_cast<uint4*>(stp + VS_V + (L + idx / 8) * 128 + (idx % 8) * 16) =
            make_uint4(0, 0, 0, 0);
    }

    // ---- 2. S_b = bf16(S) (MN-major K row = key channel); S *= 2^Gam_last[key channel]
    {
      uint32_t s[DH];
      tmem_ld_dv<DH>(tmem + lb + T_S + ch, s);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < DH / 8; ++j)
        *reinterpret_cast<uint4*>(sm + VS_SB + mn_piece(row, ch / 8 + j)) =
            make_uint4(pack_bf16x2(__uint_as_float(s[8 * j]), __uint_as_float(s[8 * j + 1])),
                       pack_bf16x2(__uint_as_float(s[8 * j + 2]), __uint_as_float(s[8 * j + 3])),
                       pack_bf16x2(__uint_as_float(s[8 * j + 4]), __uint_as_float(s[8 * j + 5])),
                       pack_bf16x2(__uint_as_float(s[8 * j + 6]), __uint_as_float(s[8 * j + 7])));
      const float d = vec[row];
#pragma unroll
      for (int j = 0; j < DH; ++j) s[j] = __float_as_uint(__uint_as_float(s[j]) * d);
      tmem_st_dv<DH>(tmem + lb + T_S + ch, s);
      tmem_wait_st();
    }
    fence_proxy_async();   // S_b and the zeroed v rows are read by the tensor cores
    tc_fence_before();
    group_sync(1, NTC4);   // (A)

    // ---- 3. X = [-W; Qg] S_b, Y = [T diag(b); *] V; meanwhile O of the previous chunk
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + tx, mndesc4(st + kRecWQ, 16384, ks), mndesc4(sb + VS_SB, 8192, ks), ID_MN,
                 ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + T_Y, kdesc4(st + kRecTB, ks), mndesc4(st + VS_V, 8192, ks), ID_KM, ks > 0);
      mma_commit(bar_g1);
      mma_out = 1;
    }
    if (i > 0 && q4 >= 2) {
      tc_fence_after();
      drain_o(T_X0 + (uint32_t)((buf ^ 1) * DV), c0 - kChunk, L_prev, iq_prev, orow_prev);
    }
    if (q4 >= 2) {   // this chunk's scalars for its own drain (the stage is reused)
      iq_prev = vec[128 + row - 64];
      orow_prev = (kRowMap && row - 64 < L) ? out_row(p, c0 + row - 64) : -1;
    }
    L_prev = L;
    {
      bool ok = true;
      if (tid == 0) {
        ok = mbar_wait(bar_g1, ph_mma);
        if (ok) mma_out = 0;
      }
      tc_fence_before();
      if (bar_any(1, NTC4, !ok)) { failed = true; site = 62; break; }   // (B)
    }
    tc_fence_after();

    // ---- 4. U_b = bf16((X + Y) diag(1/|k|)), rows 0-63 (warps with q4 < 2: tokens)
    if (q4 < 2) {
      uint32_t x[DH], y[DH];
      tmem_ld_dv<DH>(tmem + lb + tx + ch, x);
      tmem_ld_dv<DH>(tmem + lb + T_Y + ch, y);
      tmem_wait_ld();
      const float ik = vec[192 + row];
#pragma unroll
      for (int j = 0; j < DH / 8; ++j) {
        float u[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          u[e] = (__uint_as_float(x[8 * j + e]) + __uint_as_float(y[8 * j + e])) * ik;
        *reinterpret_cast<uint4*>(sm + VS_UB + mn_piece(row, ch / 8 + j)) =
            make_uint4(pack_bf16x2(u[0], u[1]), pack_bf16x2(u[2], u[3]), pack_bf16x2(u[4], u[5]),
                       pack_bf16x2(u[6], u[7]));
      }
      fence_proxy_async();   // U_b is read by the tensor cores
    }
    tc_fence_before();
    group_sync(1, NTC4);   // (C)

    // ---- 5. X += [*; QK] U_b (O in rows 64-127), S += Ke^T U_b
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + tx, kdesc4(st + kRecQKE - 8192, ks), mndesc4(sb + VS_UB, 8192, ks), ID_KM, 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + T_S, kdesc4(st + kRecQKE + 8192, ks), mndesc4(sb + VS_UB, 8192, ks), ID_KM, 1);
      mma_commit(bar_g2);
      mma_out = 2;
    }
    {
      bool ok = true;
      if (tid == 0) {
        ok = mbar_wait(bar_g2, ph_mma);
        if (ok) mma_out = 0;
      }
      tc_fence_before();
      if (bar_any(1, NTC4, !ok)) { failed = true; site = 63; break; }   // (D)
      ph_mma ^= 1u;
      if (tid == 0) mbar_arrive(bar_empty0 + 8 * buf);   // the stage is free for chunk i + 2
    }
    tc_fence_after();
  }

  if (failed) {
    if (tid == 0) {
      record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
      // let MMAs still in flight finish (bounded) before the CTA exits (the producer does the
      // same for its copies)
      if (mma_out == 1) mbar_wait(bar_g1, ph_mma);
      if (mma_out == 2) mbar_wait(bar_g2, ph_mma);
    }
  } else {
    if (nch > 0 && q4 >= 2)   // O of the last chunk
      drain_o(T_X0 + (uint32_t)(((nch - 1) & 1) * DV), t0 + kChunk * (nch - 1), L_prev, iq_prev,
              orow_prev);
    // ---- state out
    uint32_t r[DH];
    tmem_ld_dv<DH>(tmem + lb + T_S + ch, r);
    tmem_wait_ld();
    const size_t idx = sbase + (size_t)row * 128 + dv0 + ch;
    if (p.state_bf16) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.final_state) + idx);
#pragma unroll
      for (int j = 0; j < DH / 8; ++j)
        dst[j] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * j]), __uint_as_float(r[8 * j + 1])),
                            pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                            pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                            pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.final_state) + idx);
#pragma unroll
      for (int j = 0; j < DH / 4; ++j)
        dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                             __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    }
  }
  tc_fence_before();
  group_sync(1, NTC4);
  if (warp == 0) tmem_dealloc(tmem, T_COLS);
  if (streamed) stream_finish(p, tid, NTC4, last_s, [] { group_sync(1, NTC4); });
}

typedef CUresult (*EncodeTiledFn4)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int DV>
cudaError_t launch_chain_vs_dv(const Params& p, cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = attr_once.run(dev, [&]() -> cudaError_t {
    for (auto fn : {kda_chain_vs_kernel<DV, false>, kda_chain_vs_kernel<DV, true>}) {
      const cudaError_t r = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, VS_BYTES);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.num_seqs * p.heads * (128 / DV);
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  EncodeTiledFn4 enc = reinterpret_cast<EncodeTiledFn4>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  ChainVsMaps maps;
  const void* vb = p.v ? (const void*)p.v : (const void*)p.dt_bias;
  cuuint64_t dims[2] = {(cuuint64_t)p.heads * 128, (cuuint64_t)(p.total_tokens > 0 ? p.total_tokens : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)p.s_v * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  if (enc(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(vb), dims, strides, box,
          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(NT4);
  cfg.dynamicSmemBytes = VS_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.stream_sms > 0 ? 1 : 0;   // streamed: beside the k-side kernel
  if (p.out_index) return cudaLaunchKernelEx(&cfg, kda_chain_vs_kernel<DV, true>, p, maps);
  return cudaLaunchKernelEx(&cfg, kda_chain_vs_kernel<DV, false>, p, maps);
}

}  // namespace

// P = 2 only: at DV = 32 and 16 this kernel measured 12-23% slower than the warp-level
// chain of kda_chain_kernel.cu (20 MMAs, two commit round trips and four barriers a chunk
// cost the same whatever N, and every slice CTA copies the whole record)
cudaError_t launch_chain_vs(const Params& p, cudaStream_t stream) {
  return p.vsplit == 2 ? launch_chain_vs_dv<64>(p, stream) : cudaErrorInvalidValue;
}

}  // namespace kda
