// Split path, second kernel for an unsplit value dimension (P = 1): the serial
// inter-chunk chain on tcgen05, one CTA (256 threads) per (sequence, head).
//
// The k-side kernel left, per (chunk, head), the shared-memory image of the
// operand tiles this kernel needs ([-W | Qg], [QK; Ke], T diag(b), decay and norm
// scalars).  Each record and the chunk's v tile are fetched (bulk copy + TMA)
// into one of two stages while the previous chunk runs.  The 128 x 128 fp32
// state stays in tensor memory, transposed (lane = value channel):
//   [U^T | O^T]  = S^T [-W | Qg]^T        one MMA group, N = 128 (U = -W S, O = Qg S)
//   U^T         += V^T (T diag(b))^T      (U' of the WY/UT form)
//   U_b^T        = bf16(U^T diag(1/|k|))
//   S^T          = S^T diag(2^Gam_last)   (before the group below)
//   [O^T | S^T] += U_b^T [QK; Ke]^T       one MMA group, N = 192
//   out          = O diag(scale/|q|)      (drained while the next chunk starts)
// which is the chunk recurrence of the gated delta rule in the form the FlashKDA
// prefill PR report describes (PR #55737, Features & motivation), with the state
// read and written once per sequence.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_stream.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int NT3 = 256;
constexpr int D3 = kHeadDim;
constexpr int kMaxRankSeqs3 = 128;

// ---- shared memory (offsets from a 1024-byte aligned base)
constexpr int STAGE_V = kRecBytes + 1024;           // v tile after the record image
constexpr int STAGE_BYTES = STAGE_V + 16384;        // record + v [64 tok][128 dv] (2 SW128 boxes)
constexpr int OFF_STAGE0 = 0;
constexpr int OFF_STAGE1 = STAGE_BYTES;
constexpr int OFF_OST = 2 * STAGE_BYTES;            // O staging [64 tok][128 dv] bf16
constexpr int OFF_MISC3 = OFF_OST + 16384;
constexpr int OFF_BAR3 = OFF_MISC3;                 // full[2], mma, u
constexpr int OFF_TSLOT3 = OFF_MISC3 + 32;
constexpr int OFF_FLAGS3 = OFF_MISC3 + 48;
constexpr int OFF_LENS3 = OFF_MISC3 + 64;           // sequence lengths for the ordering
constexpr int OFF_IQ3 = OFF_LENS3 + 4 * kMaxRankSeqs3;   // scale/|q| of the last two chunks [2][64]
constexpr int OFF_OROW3 = OFF_IQ3 + 2 * 64 * 4;      // out rows of the last two chunks [2][64]
constexpr int SMEM3_USED = OFF_OROW3 + 2 * 64 * 4;
constexpr int SMEM3_BYTES = SMEM3_USED + 1024;
static_assert(STAGE_V % 1024 == 0 && STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(SMEM3_BYTES <= 227 * 1024, "shared memory");

// ---- tensor memory columns
constexpr uint32_t T_U = 0;      // U^T   64 cols (col = token)
constexpr uint32_t T_O = 64;     // O^T   64 cols
constexpr uint32_t T_S = 128;    // S^T  128 cols (col = dk)
constexpr uint32_t T_SB = 256;   // S^T bf16, 64 cols (2 dk per col)
constexpr uint32_t T_UB = 320;   // U_b^T bf16, 32 cols (2 tokens per col)
constexpr uint32_t T_COLS = 512;

constexpr uint32_t ID_G1 = idesc_bf16(128, 128, 0, 1);   // [U|O]  = SB  x [-W | Qg]^T
// (tcgen05 MMAs of M = 128 cost about the same per instruction for N = 64 and 128, so the
// two products that share the A operand S^T run as one N = 128 group)
constexpr uint32_t ID_G2 = idesc_bf16(128, 192, 0, 0);   // [O|S]  += UB  x [QK; Ke]^T
constexpr uint32_t ID_UP = idesc_bf16(128, 64, 1, 0);    // U      += V^T x (T diag b)^T

__device__ __forceinline__ uint64_t kdesc3(uint32_t tile, int rows, int ks) {
  return sdesc_sw128(tile + (ks >> 2) * rows * 128 + (ks & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mndesc3(uint32_t tile, uint32_t lbo, int ks) {
  return sdesc_sw128(tile + ks * 2048, lbo, 1024);
}
__device__ __forceinline__ float4 ld4s(const float* p) { return *reinterpret_cast<const float4*>(p); }

struct ChainTcMaps {
  CUtensorMap v;   // v as [T][H*128] bf16, box {64, 64}, 128-byte swizzle
};

// kRowMap: outputs go through the out_index row map (a separate instantiation, so that
// the dense kernel carries none of it)
template <bool kRowMap>
__global__ void __launch_bounds__(NT3, 1)
    kda_chain_tc_kernel(const __grid_constant__ Params p, const __grid_constant__ ChainTcMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* flags = reinterpret_cast<int*>(sm + OFF_FLAGS3);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT3);
  const uint32_t bar_full0 = sb + OFF_BAR3, bar_full1 = bar_full0 + 8, bar_mma = bar_full0 + 16;
  const uint32_t bar_u = bar_full0 + 24;

  // ---- work unit: (rank, head), longest sequence first
  const int H = p.heads, N = p.num_seqs;
  const int h = blockIdx.x % H;
  const int rank = blockIdx.x / H;
  if (N <= kMaxRankSeqs3) {
    int* lens = reinterpret_cast<int*>(sm + OFF_LENS3);
    for (int i = tid; i < N; i += NT3) lens[i] = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
    __syncthreads();
    for (int i = tid; i < N; i += NT3) {
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
  const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
  const bool streamed = p.stream_sms > 0;
  int* last_s = flags + 1;
  if (t0 < 0 || t1 < t0 || (int64_t)t1 > p.total_tokens || p.cu_seqlens[0] != 0) {
    if (tid == 0) record_error(p.status, KDA_ERR_BAD_CU_SEQLENS, 5);
    if (streamed) stream_finish(p, tid, NT3, last_s, [] { __syncthreads(); });
    return;
  }
  const int nch = (t1 - t0 + kChunk - 1) / kChunk;
  const int slot0 = (t0 >> 6) + n;   // chunk c of sequence n sits in slot floor(t0 / 64) + n + c
  const size_t HD = (size_t)H * D3;
  const size_t sbase = ((size_t)n * H + h) * D3 * D3;
  const int xcol = h * D3;

  if (tid == 0) {
    mbar_init(bar_full0, 1);
    mbar_init(bar_full1, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_u, 1);
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
  const int q4 = warp & 3;                      // TMEM lane quadrant
  const int half = warp >> 2;                   // column half of this warp
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int my_lane = 32 * q4 + lane;           // value channel dv of this thread

  auto issue = [&](int i) {                     // record + v of chunk i -> stage i & 1
    const uint32_t base = sb + ((i & 1) ? OFF_STAGE1 : OFF_STAGE0);
    const uint32_t bar = (i & 1) ? bar_full1 : bar_full0;
    const unsigned char* src = reinterpret_cast<const unsigned char*>(p.status) + kSplitHeader +
                               ((int64_t)(slot0 + i) * H + h) * kRecBytes;
    mbar_expect_tx(bar, kRecBytes + 16384);
    bulk_load(base, src, kRecBytes, bar);   // the record is contiguous at both ends
    tma_load_2d(base + STAGE_V, &maps.v, xcol, t0 + kChunk * i, bar);
    tma_load_2d(base + STAGE_V + 8192, &maps.v, xcol + 64, t0 + kChunk * i, bar);
  };
  auto prefetch_l2 = [&](int i) {               // record + v of chunk i -> L2
    const unsigned char* src = reinterpret_cast<const unsigned char*>(p.status) + kSplitHeader +
                               ((int64_t)(slot0 + i) * H + h) * kRecBytes;
    l2_prefetch(src, kRecBytes);
    tma_prefetch_2d(&maps.v, xcol, t0 + kChunk * i);
    tma_prefetch_2d(&maps.v, xcol + 64, t0 + kChunk * i);
  };
  // streamed: each record is published by the k-side kernel running beside (thread 0 waits
  // for it before the copy; a wait that gives up stops the loop at the next barrier)
  bool rec_fail = false;
  if (tid == 0 && nch > 0) {
    if (!streamed || stream_wait_record(p, slot0, h, 8))
      issue(0);
    else
      rec_fail = true;
    if (nch > 1) prefetch_l2(1);
    if (nch > 2) prefetch_l2(2);
  }

  // ---- state in: S^T[dv][dk] -> TMEM (lane = dv); this warp covers 64 key columns, all
  //      64 loads in flight at once
  {
    const int dv = my_lane;
    const int dk0 = half * 64;
    uint32_t r[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      float s = 0.0f;
      if (p.initial_state) {
        const size_t idx = sbase + (size_t)(dk0 + j) * D3 + dv;
        s = p.state_bf16
                ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.initial_state)[idx])
                : static_cast<const float*>(p.initial_state)[idx];
      }
      r[j] = __float_as_uint(s);
    }
    tmem_st32(tmem + lane_base + T_S + dk0, *reinterpret_cast<uint32_t(*)[32]>(r));
    tmem_st32(tmem + lane_base + T_S + dk0 + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
    tmem_wait_st();
  }

  // out rows of the next chunk (threads < 64, row map only), loaded a chunk ahead
  int next_orow = -1;
  if (kRowMap && tid < kChunk && tid < t1 - t0) next_orow = (int)out_row(p, t0 + tid);
  uint32_t phase = 0;        // bit b: parity of stage b's next fill
  uint32_t ph_mma = 0;
  bool failed = false;
  int site = 0;
  int pending = (nch > 0 && !rec_fail) ? 1 : 0;   // stages with a fetch in flight (thread 0's view)
  bool mma_out = false;              // an MMA commit not yet waited for (thread 0)
  int L_prev = 0;

  // O of the previous chunk: TMEM -> bf16 staging [token][dv]; this warp: tokens
  // 32 half .. 32 half + 31 of its value channels
  auto drain_o = [&](const float* iq) {
    const int dv = my_lane;
    __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_OST);
    {
      const int cb = half;
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + T_O + cb * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 v4 = ld4s(iq + cb * 32 + 4 * j4);
        const float iv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = cb * 32 + 4 * j4 + e;
          ost[tok * D3 + dv] = __float2bfloat16_rn(__uint_as_float(r[4 * j4 + e]) * iv[e]);
        }
      }
    }
  };
  // staging -> out rows of tokens [c0, c0 + L) (all threads, 16-byte stores); with an
  // out_index map the rows come from orow[b] (chunk parity b)
  const int* orow = reinterpret_cast<const int*>(sm + OFF_OROW3);
  auto store_o = [&](int c0, int L, int b) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = tid + k * NT3;
      const int r = idx >> 4, v8 = idx & 15;
      const int64_t row = kRowMap ? (int64_t)orow[b * 64 + r] : (int64_t)(c0 + r);
      if (r < L && row >= 0) {
        const uint4 val = *reinterpret_cast<const uint4*>(sm + OFF_OST + r * 256 + v8 * 16);
        *reinterpret_cast<uint4*>(p.out + (size_t)row * HD + xcol + v8 * 8) = val;
      }
    }
  };

  for (int i = 0; i < nch; ++i) {
    const int buf = i & 1;
    const int c0 = t0 + kChunk * i;
    const int L = min(kChunk, t1 - c0);
    const uint32_t st = sb + (buf ? OFF_STAGE1 : OFF_STAGE0);
    unsigned char* stp = sm + (buf ? OFF_STAGE1 : OFF_STAGE0);
    const float* vec = reinterpret_cast<const float*>(stp + kRecVec);   // decay, iq, ik
    float* iqs = reinterpret_cast<float*>(sm + OFF_IQ3);   // [2][64], by chunk parity

    // ---- 1. the record of this chunk has landed
    {
      const bool ok = mbar_wait(buf ? bar_full1 : bar_full0, (phase >> buf) & 1u);
      if (__syncthreads_or(!ok)) { failed = true; site = 51; break; }
      phase ^= 1u << buf;
      pending &= ~(1 << buf);
    }
    // scale/|q| (and out rows) of this chunk, kept past the stage's reuse (O is drained
    // during the next chunk)
    if (tid < kChunk) {
      iqs[buf * 64 + tid] = vec[128 + tid];
      if (kRowMap) {   // this chunk's out rows (loaded a chunk ahead), then the next's
        reinterpret_cast<int*>(sm + OFF_OROW3)[buf * 64 + tid] = next_orow;
        next_orow = (c0 + kChunk + tid < t1) ? (int)out_row(p, c0 + kChunk + tid) : -1;
      }
    }
    if (L < kChunk) {   // v rows past the sequence end -> 0 (both 64-column boxes)
      for (int idx = tid; idx < (kChunk - L) * 16; idx += NT3) {
        const int r = L + idx / 16, cc = idx % 16;
        *reinterpret_cast<uint4*>(stp + STAGE_V + (cc >> 3) * 8192 + r * 128 +
                                  ((((cc & 7) ^ (r & 7))) << 4)) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();
    }

    // ---- 2. S^T -> bf16 copy, then S^T *= 2^Gam_last (this warp: 64 key columns); O(i-1)
#pragma unroll 1
    for (int cb = 0; cb < 2; ++cb) {
      const int col = half * 64 + cb * 32;
      uint32_t x[32], pk[16];
      tmem_ld32(tmem + lane_base + T_S + col, x);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
      tmem_st16(tmem + lane_base + T_SB + col / 2, pk);
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 dl = ld4s(vec + col + 4 * j4);
        x[4 * j4] = __float_as_uint(__uint_as_float(x[4 * j4]) * dl.x);
        x[4 * j4 + 1] = __float_as_uint(__uint_as_float(x[4 * j4 + 1]) * dl.y);
        x[4 * j4 + 2] = __float_as_uint(__uint_as_float(x[4 * j4 + 2]) * dl.z);
        x[4 * j4 + 3] = __float_as_uint(__uint_as_float(x[4 * j4 + 3]) * dl.w);
      }
      tmem_st32(tmem + lane_base + T_S + col, x);
    }
    tmem_wait_st();
    if (i > 0) drain_o(iqs + (buf ^ 1) * 64);   // O(i-1) -> staging before it is overwritten
    tc_fence_before();
    __syncthreads();   // (A) SB ready, S decayed, O(i-1) staged; stage buf^1 free

    // ---- 3. [U | O] = SB [-W | Qg]^T, U += V^T (T diag b)^T; prefetch chunk i+1
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16_ts(tmem + T_U, tmem + T_SB + 8 * ks, mndesc3(st + kRecWQ, 16384, ks), ID_G1, ks > 0);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + T_U, mndesc3(st + STAGE_V, 8192, ks), kdesc3(st + kRecTB, 64, ks), ID_UP, 1);
      mma_commit(bar_u);
      mma_out = true;
      if (i + 1 < nch) {
        if (!streamed || stream_wait_record(p, slot0 + i + 1, h, 8)) {
          issue(i + 1);
          pending |= 1 << (buf ^ 1);
        } else {
          rec_fail = true;
        }
      }
      if (i + 3 < nch) prefetch_l2(i + 3);
    }
    if (i > 0) store_o(c0 - kChunk, L_prev, buf ^ 1);
    {
      const bool ok = tid != 0 || (mbar_wait(bar_u, ph_mma) && !rec_fail);
      tc_fence_before();
      if (__syncthreads_or(!ok)) { failed = true; site = 53; break; }   // (B)
    }
    tc_fence_after();

    // ---- 4. U_b^T = bf16(U^T diag(1/|k|)): warp half h2 covers tokens 32 h2 .. 32 h2 + 31
    {
      uint32_t x[32], pk[16];
      tmem_ld32(tmem + lane_base + T_U + half * 32, x);
      tmem_wait_ld();
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 ik = ld4s(vec + 192 + half * 32 + 4 * j4);
        pk[2 * j4] = pack_bf16x2(__uint_as_float(x[4 * j4]) * ik.x,
                                 __uint_as_float(x[4 * j4 + 1]) * ik.y);
        pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(x[4 * j4 + 2]) * ik.z,
                                     __uint_as_float(x[4 * j4 + 3]) * ik.w);
      }
      tmem_st16(tmem + lane_base + T_UB + half * 16, pk);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();   // (C)

    // ---- 5. [O | S] += U_b [QK; Ke]^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ts(tmem + T_O, tmem + T_UB + 8 * ks, kdesc3(st + kRecQKE, 192, ks), ID_G2, 1);
      mma_commit(bar_mma);
      mma_out = true;
    }
    {
      const bool ok = tid != 0 || mbar_wait(bar_mma, ph_mma);
      tc_fence_before();
      if (__syncthreads_or(!ok)) { failed = true; site = 55; break; }   // (D)
      ph_mma ^= 1;   // one fill per chunk of both bar_u and bar_mma
      mma_out = false;
    }
    tc_fence_after();
    L_prev = L;
  }

  if (failed) {
    if (tid == 0) {
      record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
      // let fetches and MMAs still in flight finish (bounded) before the CTA exits
      if (pending & 1) mbar_wait(bar_full0, phase & 1u);
      if (pending & 2) mbar_wait(bar_full1, (phase >> 1) & 1u);
      if (mma_out) {   // the commit not waited for: bar_u at site 53, bar_mma at 55
        if (site == 53) mbar_wait(bar_u, ph_mma);
        else mbar_wait(bar_mma, ph_mma);
      }
    }
  } else {
    if (nch > 0) {   // O of the last chunk
      const int last = nch - 1;
      drain_o(reinterpret_cast<const float*>(sm + OFF_IQ3) + (last & 1) * 64);
      __syncthreads();
      store_o(t0 + kChunk * last, L_prev, last & 1);
    }
    // ---- state out
    const int dv = my_lane;
#pragma unroll 1
    for (int cb = 0; cb < 2; ++cb) {
      const int dk0 = half * 64 + cb * 32;
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + T_S + dk0, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const size_t idx = sbase + (size_t)(dk0 + j) * D3 + dv;
        const float s = __uint_as_float(r[j]);
        if (p.state_bf16)
          static_cast<__nv_bfloat16*>(p.final_state)[idx] = __float2bfloat16_rn(s);
        else
          static_cast<float*>(p.final_state)[idx] = s;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, T_COLS);
  if (streamed) stream_finish(p, tid, NT3, last_s, [] { __syncthreads(); });
}

typedef CUresult (*EncodeTiledFn3)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

cudaError_t launch_chain_tc(const Params& p, cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = attr_once.run(dev, [&]() -> cudaError_t {
    for (auto fn : {kda_chain_tc_kernel<false>, kda_chain_tc_kernel<true>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM3_BYTES);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.num_seqs * p.heads;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  EncodeTiledFn3 enc = reinterpret_cast<EncodeTiledFn3>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  ChainTcMaps maps;
  const void* vb = p.v ? (const void*)p.v : (const void*)p.dt_bias;
  cuuint64_t dims[2] = {(cuuint64_t)p.heads * D3, (cuuint64_t)(p.total_tokens > 0 ? p.total_tokens : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)p.s_v * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  if (enc(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(vb), dims, strides, box,
          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(NT3);
  cfg.dynamicSmemBytes = SMEM3_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.stream_sms > 0 ? 1 : 0;   // streamed: beside the k-side kernel
  if (p.out_index) return cudaLaunchKernelEx(&cfg, kda_chain_tc_kernel<true>, p, maps);
  return cudaLaunchKernelEx(&cfg, kda_chain_tc_kernel<false>, p, maps);
}

}  // namespace kda
