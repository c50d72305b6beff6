// Body of the tcgen05 + TMA chunked KDA prefill kernel (KDA_KERNEL_TC): shared-memory and
// tensor-memory maps and the kernel itself, compiled by kda_tc_kernel.cu (dense outputs)
// and by kda_tc_rowmap_kernel.cu (outputs through a row map).  The including file defines
// KDA_TC_KERNEL_NAME and KDA_TC_ROW_MAP.
#pragma once
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"
#include "kda_tc_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace tcc;

constexpr int C = 64;
constexpr int D = kHeadDim;
constexpr int NT = 512;
constexpr int kMaxRankSeqs = 128;   // longest-first ordering for up to this many sequences

// ---- shared memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_INQ = 0;                  // q tile [64][128] bf16 row-major (TMA)
constexpr int OFF_INK = 16384;              // k tile
constexpr int OFF_ING = 32768;              // g tile
constexpr int OFF_INV = 49152;              // v tile: 2 SW128 boxes [64 tok][64 dv]
constexpr int OFF_RA = 65536;               // region reused within a chunk:
constexpr int OFF_RKQ = OFF_RA;             //  [Kr; Qr] K-major 128 rows x 128 (live to W)
constexpr int OFF_CKC = OFF_RA + 32768;     //  [Kc; Kc2] K-major 96 rows x 128 (live to D)
constexpr int OFF_NM = OFF_RA + 32768;      //  N = diag(b) strict(A)  [64][NS]  (after D)
constexpr int OFF_TM = OFF_NM + 64 * NS * 4;//  T                      [64][NS]
constexpr int OFF_Y = OFF_TM + 64 * NS * 4; //  products scratch       [32][NS]
constexpr int OFF_WN = OFF_RA + 32768;      //  -W MN-major, N = 64 tok, K = 128 (after T)
constexpr int OFF_TB = OFF_RA + 76800;      //  T diag(b/|k|) K-major 64 x 64 (for W)
constexpr int OFF_TBU = OFF_RA + 84992;     //  T diag(b)     K-major 64 x 64 (for U')
constexpr int OFF_QG = OFF_RA + 93184;      // Qg K-major 64 rows x 128 (B of O^T = S^T Qg^T)
constexpr int OFF_QKB = OFF_QG + 16384;     // [QK; Ke] K-major 192 rows x 64: QK (r, K = s), then
constexpr int OFF_KE = OFF_QKB + 8192;      //   Ke (dk rows, K = token): B of [O^T | S^T] += U^T [QK; Ke]^T
constexpr int OFF_MISC = OFF_KE + 16384;
constexpr int OFF_INVN = OFF_MISC;          // scale / |q| [64], 1 / |k| [64]
constexpr int OFF_BETA = OFF_MISC + 512;    // b [64]
constexpr int OFF_DECAY = OFF_MISC + 768;   // 2^Gam_last [128]
constexpr int OFF_WF = OFF_MISC + 1280;     // W factors [3][128]: 2^alpha0, 2^alpha1, 2^B0
constexpr int OFF_GT = OFF_MISC + 2816;     // 8-row group totals [8][128] (also sequence lengths)
constexpr int OFF_PART = OFF_MISC + 6912;   // norm partial sums [16 warps][16]
constexpr int OFF_BAR = OFF_MISC + 7936;    // 4 mbarriers
constexpr int OFF_TSLOT = OFF_MISC + 7968;  // TMEM base address
constexpr int OFF_FLAGS = OFF_MISC + 7972;  // [0] sequence chosen for this CTA, [1] record mode
constexpr int OFF_BAR_REC = OFF_MISC + 7984;   // 2 mbarriers: record buffers 0, 1
constexpr int OFF_RSC = OFF_MISC + 8192;    // per-row power-of-two operand scales, bf16x2 [q 64][k 64]
constexpr int OFF_OROW = OFF_RSC + 512;     // out rows of the chunk's tokens [2 by chunk parity][64]
                                            // (row-map instantiation only)
constexpr int SMEM_USED = OFF_OROW;         // dense instantiation
constexpr int SMEM_BYTES = SMEM_USED + 1024;
constexpr int SMEM_BYTES_MAP = SMEM_BYTES + 512;
static_assert(OFF_Y + 32 * NS * 4 <= OFF_TB, "T scratch overlaps T diag(b)");
static_assert(OFF_CKC + 24576 <= OFF_TB, "operands overlap T diag(b)");
static_assert(OFF_TBU + 8192 <= OFF_QG, "T tiles overlap Qg");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
// Record mode (chunks whose k-side a helper CTA computed): two record images over the
// k-side regions, the v tile where it always is, O staging over the q tile.
constexpr int OFF_REC0 = OFF_RA;
constexpr int OFF_REC1 = OFF_RA + kRecBytes;
constexpr int OFF_OSTR = OFF_INQ;
static_assert(kRecBytes % 1024 == 0 && OFF_REC1 + kRecBytes <= OFF_MISC, "record buffers");
static_assert(OFF_BAR_REC + 16 <= OFF_RSC && OFF_FLAGS + 8 <= OFF_BAR_REC, "misc");
static_assert(SMEM_BYTES_MAP <= 227 * 1024, "shared memory (row map)");

// ---- TMEM columns (fp32 unless noted; lane = value channel, or key channel for D/W)
// [U^T | O^T] and [O^T | S^T] are each one contiguous accumulator
constexpr uint32_t TM_U = 0;      // U^T         64 cols (col = token)
constexpr uint32_t TM_O = 64;     // O^T         64 cols (col = token), then
constexpr uint32_t TM_S = 128;    // S^T        128 cols (col = dk)
constexpr uint32_t TM_SB = 256;   // S^T bf16    64 cols (A operand, 2 dk per col)
constexpr uint32_t TM_D = 320;    // D (A|QK)    96 cols, then W0^T at +0, W1^T at +64
constexpr uint32_t TM_UB = 448;   // U^T bf16    32 cols (A operand, 2 tokens per col)
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t ID_KK64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_KK96 = idesc_bf16(128, 96, 0, 0);
constexpr uint32_t ID_MK64 = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_KM64 = idesc_bf16(128, 64, 0, 1);
constexpr uint32_t ID_KK192 = idesc_bf16(128, 192, 0, 0);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, 0, 1);

// KDA_TC_ROW_MAP: outputs go through the out_index row map.  The body is compiled twice,
// once per translation unit: kda_tc_chunk_kernel (dense, kda_tc_kernel.cu) and
// kda_tc_chunk_kernel_rowmap (kda_tc_rowmap_kernel.cu), so the dense kernel carries none
// of the map.
__global__ void __launch_bounds__(NT, 1)
    KDA_TC_KERNEL_NAME(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_g,
                        const __grid_constant__ CUtensorMap tm_v) {
  constexpr bool kRowMap = KDA_TC_ROW_MAP;
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
  float* part = reinterpret_cast<float*>(sm + OFF_PART);
  uint32_t* rsc = reinterpret_cast<uint32_t*>(sm + OFF_RSC);
  int* orow = reinterpret_cast<int*>(sm + OFF_OROW);   // used when an out_index map is given
  int* flags = reinterpret_cast<int*>(sm + OFF_FLAGS);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TSLOT);
  const uint32_t bar_qkg = sb + OFF_BAR, bar_v = bar_qkg + 8, bar_mma = bar_qkg + 16;
  const uint32_t bar_o = bar_qkg + 24;      // O^T = S^T Qg^T, issued by warp 4
  const uint32_t bar_rec0 = sb + OFF_BAR_REC, bar_rec1 = bar_rec0 + 8;

  // ---- work unit: (rank, head, part), longest sequence first
  const int P = p.vsplit, H = p.heads, N = p.num_seqs;
  const int unit = blockIdx.x;
  const int vpart = unit % P;
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
  const int dv_lo = vpart * DV, dv_hi = dv_lo + DV;

  // ---- barriers and tensor memory
  if (tid == 0) {
    mbar_init(bar_qkg, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_rec0, 1);
    mbar_init(bar_rec1, 1);
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
  const int q4 = warp & 3;                        // TMEM lane quadrant of this warp
  const int cs = warp >> 2;                       // column slice (0..3) of this warp
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int my_lane = 32 * q4 + lane;             // TMEM lane this thread reads

  const size_t HD = (size_t)H * D;
  const size_t sbase = ((size_t)n * H + h) * D * D;
  const int xcol = h * D;
  const int nch = (t1 - t0 + C - 1) / C;

  // With helpers (P = 1): chunk c of this sequence is item (slot0, h) + c.  Its claim words
  // start free (chunk 0: this CTA's), then the helper grid may launch.  The helpers claim (compare-and-swap) from
  // the last chunk down as they start an item.  This CTA reads the word of its next chunk
  // one chunk ahead: free -> it marks the chunk its own (a plain store: an atomic here would
  // hold the next barrier for an L2 round trip) and computes it; taken -> this and every
  // later chunk come from records.  A helper that takes the chunk between the read and the
  // mark writes a record nobody reads and stops at its next claim.
  const int slot0 = (t0 >> 6) + n;
  // this CTA's claim words: chunk c at claims[c]
  int* claims = p.helpers ? reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(p.status) +
                                                   helper_claims_offset(p.total_tokens, H, N)) +
                                claim_index(slot0, h, p.total_tokens, N)
                          : nullptr;
  // chunk 0 is always this CTA's own: its inputs are fetched before the claim words are
  // written (the helpers can only start after every CTA has written its words)
  if (tid == 0 && nch > 0) {
    mbar_expect_tx(bar_qkg, 3 * 16384);
    tma_load_2d(sb + OFF_INQ, &tm_q, xcol, t0, bar_qkg);
    tma_load_2d(sb + OFF_INK, &tm_k, xcol, t0, bar_qkg);
    tma_load_2d(sb + OFF_ING, &tm_g, xcol, t0, bar_qkg);
    mbar_expect_tx(bar_v, 16384);
    tma_load_2d(sb + OFF_INV, &tm_v, xcol, t0, bar_v);
    tma_load_2d(sb + OFF_INV + 8192, &tm_v, xcol + 64, t0, bar_v);
  }
  if (claims) {
    const bool writer = tid < nch || (blockIdx.x == 0 && tid == 0);
    for (int c = tid; c < nch; c += NT) claims[c] = (c == 0) ? kClaimOwn : kClaimFree;
    if (blockIdx.x == 0 && tid == 0) p.status[kHelperCounterWord] = 0;
    if (writer) __threadfence();
    __syncthreads();
    pdl_launch_dependents();
  }
  // Record mode (one thread): wait (bounded) for the helper's record of chunk c, then copy
  // it to buffer b
  auto fetch_record = [&](int c, int b) {
    const int* w = &claims[c];
    if (!wait_flag(w, kClaimReady)) return false;
    fence_proxy_async_global();
    const unsigned char* src = reinterpret_cast<const unsigned char*>(p.status) + kSplitHeader +
                               ((int64_t)(slot0 + c) * H + h) * kRecBytes;
    const uint32_t dst = sb + (b ? OFF_REC1 : OFF_REC0), bar = b ? bar_rec1 : bar_rec0;
    mbar_expect_tx(bar, kRecBytes);
#pragma unroll
    for (int part = 0; part < 4; ++part)
      bulk_load(dst + part * 16384, src + part * 16384, 16384, bar);
    bulk_load(dst + kRecVec, src + kRecVec, kRecBytes - kRecVec, bar);
    return true;
  };

  // out rows of the next chunk to start, loaded a chunk ahead (threads < 64, row map only)
  int next_orow = -1;
  if (kRowMap && tid < C && tid < t1 - t0) next_orow = (int)out_row(p, t0 + tid);
  if (tid == 0) flags[1] = 0;   // 1: this and every later chunk from records

  // ---- state in: S^T[dv][dk] -> TMEM (lane = dv); this warp covers 32 key columns
  {
    const int dv = my_lane;
    const bool mine = dv >= dv_lo && dv < dv_hi && p.initial_state != nullptr;
    const int dk0 = cs * 32;
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
    tmem_wait_st();
  }
  __syncthreads();   // flags[1]

  const float gate_scale = expf(p.A_log[h]);
  const float lb2 = p.lower_bound * kLog2e;
  const int cp = tid & 63;            // channel pair of the gate/operand phase
  const int grp = tid >> 6;           // 8-row group of the gate/operand phase
  const int d0 = 2 * cp;
  const int blk = grp >> 2;           // 32-token block of the group
  // sigmoid argument in log2 units: -gate_scale * log2e * (g + dt_bias)
  const float sg = -gate_scale * kLog2e;
  const float sg0 = sg * p.dt_bias[h * D + d0], sg1 = sg * p.dt_bias[h * D + d0 + 1];
  float* Nm = reinterpret_cast<float*>(sm + OFF_NM);
  float* Tm = reinterpret_cast<float*>(sm + OFF_TM);
  float* Y = reinterpret_cast<float*>(sm + OFF_Y);

  uint32_t ph_qkg = 0, ph_v = 0, ph_mma = 0, ph_o = 0;
  uint32_t ph_rec = 0;        // bit b: parity of record buffer b's next fill
  int rec_pend = 0;           // record buffers with a copy in flight (thread 32's view)
  constexpr int kFetcher = 32;   // thread that fetches records (warp 1; thread 0 issues MMAs)
  int jr = 0, L_prev = 0;     // record-mode chunks done; rows of the previous one
  bool failed = false;
  int site = 0;
  // beta logits are fetched one chunk ahead (their load latency hides behind a chunk)
  float b_raw = 0.0f;
  if (tid < C && t0 + tid < t1) b_raw = __bfloat162float(p.beta[(size_t)(t0 + tid) * p.s_beta + h]);

  int c = 0;
  for (; c < nch; ++c) {
    if (flags[1]) break;   // from here on the chunks come from records (loop below)
    const int c0 = t0 + C * c;
    const int L = min(C, t1 - c0);
    const bool more = c + 1 < nch;
    // the next chunk's claim word now; the answer is needed when its inputs are fetched (P3)
    int next_claim = kClaimFree;
    if (claims && more && tid == 0) next_claim = ld_relaxed_gpu(&claims[c + 1]);


    // ---- P0: q, k, g of this chunk have landed (every thread waits for the TMA itself;
    //          a timeout is acted on at the next barrier); beta; zero q/k rows past the end
    const bool tma_ok = mbar_wait(bar_qkg, ph_qkg);
    ph_qkg ^= 1;
    if (tid < C) {
      beta_s[tid] = (tid < L) ? sigm(b_raw) : 0.0f;
      if (c0 + C + tid < t1) b_raw = __bfloat162float(p.beta[(size_t)(c0 + C + tid) * p.s_beta + h]);
      if (kRowMap) orow[(c & 1) * C + tid] = next_orow;
    }
    if (L < C) {
      for (int idx = tid; idx < (C - L) * 32; idx += NT) {
        const int r = L + (idx >> 5), c16 = idx & 31;
        st_u128(sm, (c16 < 16 ? OFF_INQ : OFF_INK) + r * 256 + (c16 & 15) * 16,
                make_uint4(0, 0, 0, 0));
      }
    }

    // ---- P2a: gate -> log2 decay, cumsum inside this thread's 8-row group
    float cl0[8], cl1[8];
    {
      float run0 = 0.0f, run1 = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = grp * 8 + i;
        const float2 gv = unpack_bf16x2(ld_u32(sm + OFF_ING, (uint32_t)(r * 256 + d0 * 2)));
        float a0 = lb2 * rcpf(1.0f + ex2f(fmaf(gv.x, sg, sg0)));
        float a1 = lb2 * rcpf(1.0f + ex2f(fmaf(gv.y, sg, sg1)));
        a0 = (r < L) ? a0 : 0.0f;
        a1 = (r < L) ? a1 : 0.0f;
        run0 += a0;
        run1 += a1;
        cl0[i] = run0;
        cl1[i] = run1;
      }
      *reinterpret_cast<float2*>(gt + grp * 128 + d0) = make_float2(run0, run1);
      // sums of squares of the group's q and k rows over this warp's 64 channels,
      // reduce-scattered: lanes 2j, 2j + 1 end with the sum of v[j] ([0, 8) q, [8, 16) k)
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = grp * 8 + i;
        const float2 qf = unpack_bf16x2(ld_u32(sm + OFF_INQ, (uint32_t)(r * 256 + d0 * 2)));
        const float2 kf = unpack_bf16x2(ld_u32(sm + OFF_INK, (uint32_t)(r * 256 + d0 * 2)));
        v[i] = fmaf(qf.x, qf.x, qf.y * qf.y);
        v[8 + i] = fmaf(kf.x, kf.x, kf.y * kf.y);
      }
#pragma unroll
      for (int o = 16, m = 8; o >= 2; o >>= 1, m >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < m; ++i) {
          const float send = up ? v[i] : v[i + m];
          const float keep = up ? v[i + m] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      if ((lane & 1) == 0) part[warp * 16 + (lane >> 1)] = v[0];
    }
    if (__syncthreads_or(!tma_ok)) { failed = true; site = 10; break; }

    // ---- P2c: norms -> scale/|q_r|, 1/|k_r|, and a power of two 2^-s_r per row with
    //           |row| 2^-s_r <= 1.  The operands are built from the rows times 2^-s_r (exact in
    //           bf16) and the scalars carry 2^s_r: the same products, but a raw row can no
    //           longer push an anchored factor (up to 2^(16 |lb| log2 e)) out of range.
    if (tid < 128) {   // row r = tid & 63 of q (tid < 64) or k; warps 2 g8, 2 g8 + 1 hold it
      const int r = tid & 63, t = tid >> 6;
      const int g8 = r >> 3, i = r & 7;
      const float ss = part[(2 * g8) * 16 + t * 8 + i] + part[(2 * g8 + 1) * 16 + t * 8 + i];
      // ss < 2^(e+1) -> |row| < 2^ceil((e+1)/2)
      const int e = ((__float_as_int(ss) >> 23) & 255) - 127;
      const int sh = max(-60, min(60, (e + 2) >> 1));
      const float inv = (r < L) ? rsqrtf(ss + kL2Eps) * __int_as_float((127 + sh) << 23) : 0.0f;
      inv_q[t * 64 + r] = (t == 0) ? p.scale * inv : inv;
      const uint32_t b = (uint32_t)(127 - sh) << 7;   // bf16 bits of 2^-sh
      rsc[t * 64 + r] = b | (b << 16);
    }
    __syncthreads();

    if (kRowMap && tid < C)   // the next chunk's out rows (used from its P0 on)
      next_orow = (more && c0 + C + tid < t1) ? (int)out_row(p, c0 + C + tid) : -1;

    // ---- P2b: anchored factors, bf16 operand tiles of the (power-of-two scaled) q, k rows
    //           (their norms are applied to the products later)
    {
      float mE[2], cA[2], cB[2], cX[2], cR[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float G[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) G[j] = gt[j * 128 + d0 + c];
        const float B0 = (G[0] + G[1]) + (G[2] + G[3]);
        const float B1 = (G[4] + G[5]) + (G[6] + G[7]);
        const float al0 = G[0] + G[1], al1 = G[4] + G[5];
        float pre = 0.0f;                          // totals of earlier groups of the block
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if ((j >> 2) == blk && j < grp) pre += G[j];
        const float al = blk ? al1 : al0;
        mE[c] = al - pre;                          // exponent of E = cl - mE
        cA[c] = ex2f(al);                          // E -> 2^c (within the block)
        cB[c] = ex2f((blk ? B1 : B0) - al);        // Ei -> 2^(B_blk - c)
        cX[c] = ex2f(al1);                         // alpha_1, folded into Kc2
        cR[c] = ex2f(blk ? B0 : B1);               // the other block's total
        if (grp == 0) {
          decay_s[d0 + c] = ex2f(B0 + B1);
          wf[d0 + c] = cA[c];                      // W block 0: 2^alpha0
          wf[128 + d0 + c] = cX[c];                // W block 1: 2^alpha1, then
          wf[256 + d0 + c] = ex2f(B0);             //            2^B0
        }
      }
      uint32_t kep[8];                             // Ke pairs (d0, d0 + 1) of the 8 rows
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = grp * 8 + i;
        const uint32_t q2 = bmul2(ld_u32(sm + OFF_INQ, (uint32_t)(r * 256 + d0 * 2)), rsc[r]);
        const uint32_t k2 = bmul2(ld_u32(sm + OFF_INK, (uint32_t)(r * 256 + d0 * 2)), rsc[64 + r]);
        const float e0 = cl0[i] - mE[0], e1 = cl1[i] - mE[1];
        const float E0 = ex2f(e0), E1 = ex2f(e1);
        const float Ei0 = ex2f(-e0), Ei1 = ex2f(-e1);
        const uint32_t E2 = pack_bf16x2(E0, E1), Ei2 = pack_bf16x2(Ei0, Ei1);
        st_u32(sm, OFF_RKQ + kmajor_off(r, d0, 128), bmul2(k2, E2));
        st_u32(sm, OFF_RKQ + kmajor_off(64 + r, d0, 128), bmul2(q2, E2));
        st_u32(sm, OFF_CKC + kmajor_off(r, d0, 96), bmul2(k2, Ei2));
        float g0, g1, ke0, ke1;
        if (blk == 0) {
          const float oc0 = Ei0 * cB[0], oc1 = Ei1 * cB[1];    // 2^(B0 - c_s)
          st_u32(sm, OFF_CKC + kmajor_off(64 + r, d0, 96),
                 bmul2(k2, pack_bf16x2(oc0 * cX[0], oc1 * cX[1])));
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
        st_u32(sm, OFF_QG + kmajor_off(r, d0, 64), bmul2(q2, pack_bf16x2(g0, g1)));
        kep[i] = bmul2(k2, pack_bf16x2(ke0, ke1));
      }
      // Ke: the 8 tokens of channel d0 (d0 + 1) form one 16-byte chunk of row d0 (d0 + 1)
      st_u128(sm, OFF_KE + kmajor_off(d0, grp * 8, 128),
              make_uint4(__byte_perm(kep[0], kep[1], 0x5410), __byte_perm(kep[2], kep[3], 0x5410),
                         __byte_perm(kep[4], kep[5], 0x5410), __byte_perm(kep[6], kep[7], 0x5410)));
      st_u128(sm, OFF_KE + kmajor_off(d0 + 1, grp * 8, 128),
              make_uint4(__byte_perm(kep[0], kep[1], 0x7632), __byte_perm(kep[2], kep[3], 0x7632),
                         __byte_perm(kep[4], kep[5], 0x7632), __byte_perm(kep[6], kep[7], 0x7632)));
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P3: D = [Kr; Qr] [Kc; Kc2]^T on the tensor cores; fetch the next q, k, g
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + TM_D, kdesc(sb + OFF_RKQ, 128, ks), kdesc(sb + OFF_CKC, 96, ks), ID_KK96,
                 ks > 0);
      mma_commit(bar_mma);
      if (more) {
        if (next_claim == kClaimFree) {
          if (claims) st_relaxed_gpu(&claims[c + 1], kClaimOwn);
          mbar_expect_tx(bar_qkg, 3 * 16384);
          tma_load_2d(sb + OFF_INQ, &tm_q, xcol, c0 + C, bar_qkg);
          tma_load_2d(sb + OFF_INK, &tm_k, xcol, c0 + C, bar_qkg);
          tma_load_2d(sb + OFF_ING, &tm_g, xcol, c0 + C, bar_qkg);
        } else {
          flags[1] = 1;   // a helper has the next chunk, hence every later one
        }
      }
    }
    {
      // one thread waits for the MMA (the others park on the barrier); all see the v tile land
      const bool ok = (tid != 0 || mbar_wait(bar_mma, ph_mma)) && mbar_wait(bar_v, ph_v);
      ph_mma ^= 1;
      ph_v ^= 1;
      tc_fence_before();
      if (__syncthreads_or(!ok)) { failed = true; site = 30; break; }
    }
    tc_fence_after();

    // ---- P4a: A rows (lanes 0-63) -> N = diag(b/|k|) strict(A) diag(1/|k|);
    //           QK rows (64-127) -> bf16 tile (raw); other warps: v tail rows, T upper blocks
    if (cs < 2) {
      const int r = my_lane & 63;
      uint32_t a[32];
      // columns 0-31 of rows 32-63 come from D[:, 64:96] (the off-diagonal block)
      tmem_ld32(tmem + lane_base + TM_D + ((cs == 0 && r >= 32) ? 64 : 32 * cs), a);
      tmem_wait_ld();
      if (q4 < 2) {
        const float br = beta_s[r] * inv_k[r];
#pragma unroll
        for (int s4 = 0; s4 < 8; ++s4) {
          const float4 ik = ld4(inv_k + 32 * cs + 4 * s4);
          const float ikv[4] = {ik.x, ik.y, ik.z, ik.w};
          float vv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = 32 * cs + 4 * s4 + e;
            vv[e] = (s < r) ? br * ikv[e] * __uint_as_float(a[4 * s4 + e]) : 0.0f;
          }
          *reinterpret_cast<float4*>(Nm + r * NS + 32 * cs + 4 * s4) =
              make_float4(vv[0], vv[1], vv[2], vv[3]);
        }
      } else {
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = 32 * cs + c8 * 8 + e * 2;
            w[e] = pack_bf16x2(s <= r ? __uint_as_float(a[c8 * 8 + e * 2]) : 0.0f,
                               s + 1 <= r ? __uint_as_float(a[c8 * 8 + e * 2 + 1]) : 0.0f);
          }
          st_u128(sm, OFF_QKB + kmajor_off(r, 32 * cs + c8 * 8, 64),
                  make_uint4(w[0], w[1], w[2], w[3]));
        }
      }
    } else {
      const int t8 = tid - 256;
      if (L < C) {   // v rows past the sequence end -> 0 (both 64-column boxes)
        for (int idx = t8; idx < (C - L) * 16; idx += 256) {
          const int r = L + idx / 16, cc = idx % 16;
          st_u128(sm, OFF_INV + (cc >> 3) * 8192 + r * 128 + (cc & 7) * 16, make_uint4(0, 0, 0, 0));
        }
      }
      // T above the diagonal 16x16 blocks is zero
      for (int idx = t8; idx < 6 * 64; idx += 256) {
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

    // ---- P4b: T = (I + N)^-1 on warps 0-1: 16x16 diagonal blocks by substitution (fp32),
    //           then the off-diagonal blocks as tf32 tensor-core products, 16 -> 32 -> 64.
    //           Warps 4-7 meanwhile make the bf16 copy of S^T and apply this chunk's decay.
    if (warp < 4) {
      if (warp < 2) {
        const int o = (tid >> 4) * 16, j = tid & 15;
        // column j of the block's inverse by forward substitution, right-looking: once x[k]
        // is final its term leaves every later row at once (each row still subtracts its
        // terms in the order k = 0, 1, ...; the dependent chain is 16 steps, not 120)
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.0f : 0.0f;
#pragma unroll
        for (int k = 0; k < 15; ++k) {
#pragma unroll
          for (int i = k + 1; i < 16; ++i) x[i] = fmaf(-Nm[(o + i) * NS + o + k], x[k], x[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tm[(o + i) * NS + o + j] = x[i];
      }
      named_barrier_sync(1, 128);
      if (warp < 2) {   // pair (1,0) on warp 0, (3,2) on warp 1: T_rc = -T_rr (N_rc T_cc)
        const int ro = (2 * warp + 1) * 16, co = 2 * warp * 16;
        float* Yw = Y + warp * 16 * NS;
        warp_gemm_16x16<16>(Nm + ro * NS + co, Tm + co * NS + co, Yw, 1.0f, lane);
        __syncwarp();
        warp_gemm_16x16<16>(Tm + ro * NS + ro, Yw, Tm + ro * NS + co, -1.0f, lane);
      }
      named_barrier_sync(1, 128);
      const int mi = warp >> 1, ni = warp & 1;   // Y2 = N[32:64, 0:32] T[0:32, 0:32]
      warp_gemm_16x16<32>(Nm + (32 + 16 * mi) * NS, Tm + 16 * ni, Y + 16 * mi * NS + 16 * ni,
                          1.0f, lane);
      named_barrier_sync(1, 128);               // T[32:64, 0:32] = -T[32:64, 32:64] Y2
      warp_gemm_16x16<32>(Tm + (32 + 16 * mi) * NS + 32, Y + 16 * ni,
                          Tm + (32 + 16 * mi) * NS + 16 * ni, -1.0f, lane);
    } else if (warp >= 4 && warp < 8) {
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {   // state pass: 32 key columns at a time
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
      // O^T = S^T Qg^T needs only the bf16 state: issue it now, it overlaps the T inverse
      tc_fence_before();
      named_barrier_sync(2, 128);
      if (tid == 128) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_ts(tmem + TM_O, tmem + TM_SB + 8 * ks, kdesc(sb + OFF_QG, 64, ks), ID_KK64,
                      ks > 0);
        mma_commit(bar_o);
      }
    }
    tc_fence_before();
    __syncthreads();
    {   // T diag(b) and T diag(b / |k|) -> bf16 (K-major, row r, k = s), 8 columns per thread
      const int r = tid >> 3, c8 = tid & 7;
      float4 t0v = ld4(Tm + r * NS + c8 * 8), t1v = ld4(Tm + r * NS + c8 * 8 + 4);
      const float4 b0v = ld4(beta_s + c8 * 8), b1v = ld4(beta_s + c8 * 8 + 4);
      const float4 k0v = ld4(inv_k + c8 * 8), k1v = ld4(inv_k + c8 * 8 + 4);
      t0v = make_float4(t0v.x * b0v.x, t0v.y * b0v.y, t0v.z * b0v.z, t0v.w * b0v.w);
      t1v = make_float4(t1v.x * b1v.x, t1v.y * b1v.y, t1v.z * b1v.z, t1v.w * b1v.w);
      const uint32_t off = kmajor_off(r, c8 * 8, 64);
      st_u128(sm, OFF_TBU + off,
              make_uint4(pack_bf16x2(t0v.x, t0v.y), pack_bf16x2(t0v.z, t0v.w),
                         pack_bf16x2(t1v.x, t1v.y), pack_bf16x2(t1v.z, t1v.w)));
      st_u128(sm, OFF_TB + off,
              make_uint4(pack_bf16x2(t0v.x * k0v.x, t0v.y * k0v.y),
                         pack_bf16x2(t0v.z * k0v.z, t0v.w * k0v.w),
                         pack_bf16x2(t1v.x * k1v.x, t1v.y * k1v.y),
                         pack_bf16x2(t1v.z * k1v.z, t1v.w * k1v.w)));
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P5: W_b^T = (raw Kr rows of block b)^T (T diag(b/|k|))[:, b]^T (D region);
    //          U'^T = V^T (T diag(b))^T
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
        mma_bf16(tmem + TM_U, mndesc(sb + OFF_INV, 8192, ks), kdesc(sb + OFF_TBU, 64, ks),
                 ID_MK64, ks > 0);
      mma_commit(bar_mma);
    }
    {
      const bool ok = tid != 0 || mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 50; break; }
    }
    tc_fence_after();
    if (tid == 0 && more) {   // v tile is free again
      mbar_expect_tx(bar_v, 16384);
      tma_load_2d(sb + OFF_INV, &tm_v, xcol, c0 + C, bar_v);
      tma_load_2d(sb + OFF_INV + 8192, &tm_v, xcol + 64, c0 + C, bar_v);
    }

    // ---- P6: -W = -(2^a0 W0 + 2^B0 (2^a1 W1)) -> bf16, MN-major (n = token, k = dk)
    {
      const int dk = my_lane;
      const float f0 = wf[dk], f1a = wf[128 + dk], f1b = wf[256 + dk];
      uint32_t w0[16], w1[16];
      tmem_ld16(tmem + lane_base + TM_D + cs * 16, w0);
      tmem_ld16(tmem + lane_base + TM_D + 64 + cs * 16, w1);
      tmem_wait_ld();
#pragma unroll
      for (int c8 = 0; c8 < 2; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = c8 * 8 + e * 2;
          const float x0 = f0 * __uint_as_float(w0[j]) + f1b * (f1a * __uint_as_float(w1[j]));
          const float x1 =
              f0 * __uint_as_float(w0[j + 1]) + f1b * (f1a * __uint_as_float(w1[j + 1]));
          w[e] = pack_bf16x2(-x0, -x1);
        }
        st_u128(sm, OFF_WN + mnmajor_off(cs * 16 + c8 * 8, dk, 8192),
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
      const bool ok = tid != 0 || mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 70; break; }
    }
    tc_fence_after();

    // ---- P8: U^T diag(1/|k|) -> bf16 operand in TMEM (2 tokens per column)
    if (cs < 2) {
      uint32_t x[32], pk[16];
      tmem_ld32(tmem + lane_base + TM_U + cs * 32, x);
      tmem_wait_ld();
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 ik = ld4(inv_k + cs * 32 + 4 * j4);
        pk[2 * j4] = pack_bf16x2(__uint_as_float(x[4 * j4]) * ik.x,
                                 __uint_as_float(x[4 * j4 + 1]) * ik.y);
        pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(x[4 * j4 + 2]) * ik.z,
                                     __uint_as_float(x[4 * j4 + 3]) * ik.w);
      }
      tmem_st16(tmem + lane_base + TM_UB + cs * 16, pk);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();

    // ---- P9: [O^T | S^T] += U^T [QK; Ke]^T, one N = 192 group (after warp 4's
    //          O^T = S^T Qg^T completed)
    bool o_ok = true;
    if (tid == 0) {
      o_ok = mbar_wait(bar_o, ph_o);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ts(tmem + TM_O, tmem + TM_UB + 8 * ks, kdesc(sb + OFF_QKB, 192, ks), ID_KK192, 1);
      mma_commit(bar_mma);
    }
    ph_o ^= 1;
    {
      const bool ok = tid != 0 || (o_ok && mbar_wait(bar_mma, ph_mma));
      ph_mma ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; site = 90; break; }
    }
    tc_fence_after();

    // ---- P10: O^T diag(scale/|q|) -> bf16 staging [token][dv] -> 16-byte global stores of
    //           rows < L of this value slice (the [Kr; Qr] tile is free by now)
    {
      const int dv = my_lane;
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + TM_O + cs * 16, r);
      tmem_wait_ld();
      __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_RKQ);
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4) {
        const float4 iq = ld4(inv_q + cs * 16 + 4 * j4);
        const float iqv[4] = {iq.x, iq.y, iq.z, iq.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * j4 + e;
          ost[(cs * 16 + j) * D + dv] = __float2bfloat16_rn(__uint_as_float(r[j]) * iqv[e]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int idx = tid + k2 * NT;
      const int r = idx >> 4, v8 = idx & 15;
      const int64_t row = kRowMap ? (int64_t)orow[(c & 1) * C + r] : (int64_t)(c0 + r);
      if (r < L && row >= 0 && v8 * 8 >= dv_lo && v8 * 8 < dv_hi) {
        const uint4 val = *reinterpret_cast<const uint4*>(sm + OFF_RKQ + r * 256 + v8 * 16);
        *reinterpret_cast<uint4*>(p.out + (size_t)row * HD + xcol + v8 * 8) = val;
      }
    }
    __syncthreads();
  }

  // ---- record mode: the chunks a helper computed the chunk-local half of ([-W | Qg],
  //      [QK; Ke], T diag(b), decay and norm scalars in its record): the chunk step of the
  //      chain kernel, one record fetched ahead
  for (; !failed && c < nch; ++c) {
    const int c0 = t0 + C * c;
    const int L = min(C, t1 - c0);
    const bool more = c + 1 < nch;
    const int buf = jr & 1;
    const uint32_t rb = sb + (buf ? OFF_REC1 : OFF_REC0);
    const float* vec = reinterpret_cast<const float*>(sm + (buf ? OFF_REC1 : OFF_REC0) + kRecVec);
    bool ok = true;
    if (tid == kFetcher && jr == 0) {   // first record-mode chunk: nothing was fetched ahead
      ok = fetch_record(c, buf);
      if (ok) rec_pend |= 1 << buf;
    }
    // R1: the record and the v tile have landed; v rows past the sequence end -> 0
    const bool got = ok && mbar_wait(buf ? bar_rec1 : bar_rec0, (ph_rec >> buf) & 1u);
    // the v tile was issued whatever happened to the record: always wait for it
    const bool v_ok = mbar_wait(bar_v, ph_v);
    ok = got && v_ok;
    if (got) {
      ph_rec ^= 1u << buf;
      if (tid == kFetcher) rec_pend &= ~(1 << buf);
    }
    ph_v ^= 1;
    if (ok && L < C) {
      for (int idx = tid; idx < (C - L) * 16; idx += NT) {
        const int r = L + idx / 16, cc = idx % 16;
        st_u128(sm, OFF_INV + (cc >> 3) * 8192 + r * 128 + (cc & 7) * 16, make_uint4(0, 0, 0, 0));
      }
      fence_proxy_async();
    }
    if (kRowMap && tid < C) orow[(c & 1) * C + tid] = next_orow;
    if (__syncthreads_or(!ok)) { failed = true; site = 80; break; }
    if (kRowMap && tid < C)   // the next chunk's out rows
      next_orow = (more && c0 + C + tid < t1) ? (int)out_row(p, c0 + C + tid) : -1;
    if (tid == 0 && c + 2 < nch) {   // v two chunks ahead -> L2 (its TMA is issued in R3 below)
      tma_prefetch_2d(&tm_v, xcol, c0 + 2 * C);
      tma_prefetch_2d(&tm_v, xcol + 64, c0 + 2 * C);
    }

    // R2: S^T -> bf16 copy, S^T *= 2^Gam_last (this warp: 32 key columns); O of the
    //     previous chunk -> staging (its scale/|q| is in the other record buffer)
    {
      uint32_t x[32], pk[16];
      tmem_ld32(tmem + lane_base + TM_S + cs * 32, x);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16x2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
      tmem_st16(tmem + lane_base + TM_SB + cs * 16, pk);
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 dl = ld4(vec + cs * 32 + 4 * j4);
        x[4 * j4] = __float_as_uint(__uint_as_float(x[4 * j4]) * dl.x);
        x[4 * j4 + 1] = __float_as_uint(__uint_as_float(x[4 * j4 + 1]) * dl.y);
        x[4 * j4 + 2] = __float_as_uint(__uint_as_float(x[4 * j4 + 2]) * dl.z);
        x[4 * j4 + 3] = __float_as_uint(__uint_as_float(x[4 * j4 + 3]) * dl.w);
      }
      tmem_st32(tmem + lane_base + TM_S + cs * 32, x);
    }
    {
      uint32_t r[16];
      if (jr > 0) {
        const float* iqp =
            reinterpret_cast<const float*>(sm + (buf ? OFF_REC0 : OFF_REC1) + kRecVec) + 128;
        tmem_ld16(tmem + lane_base + TM_O + cs * 16, r);
        tmem_wait_ld();
        __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_OSTR);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 iq = ld4(iqp + cs * 16 + 4 * j4);
          const float iqv[4] = {iq.x, iq.y, iq.z, iq.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            ost[(cs * 16 + j) * D + my_lane] = __float2bfloat16_rn(__uint_as_float(r[j]) * iqv[e]);
          }
        }
      }
      // O^T starts from zero: the group below accumulates into [U^T | O^T]
#pragma unroll
      for (int j = 0; j < 16; ++j) r[j] = 0u;
      tmem_st16(tmem + lane_base + TM_O + cs * 16, r);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();   // (A) SB ready, S decayed, O(c-1) staged, O zeroed; the other buffer is free

    // R3: U^T = V^T (T diag b)^T, then [U^T | O^T] += S^T [-W | Qg]^T (the fused kernel's
    //     order of accumulation: the same bits whichever CTA computed the chunk-local
    //     half); fetch the next record; O(c-1) -> out
    bool next_ok = true;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + TM_U, mndesc(sb + OFF_INV, 8192, ks), kdesc(rb + kRecTB, 64, ks), ID_MK64,
                 ks > 0);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16_ts(tmem + TM_U, tmem + TM_SB + 8 * ks, mndesc(rb + kRecWQ, 16384, ks), ID_KM128,
                    1);
      mma_commit(bar_mma);
    } else if (tid == kFetcher && more) {   // meanwhile: the next record, and the one after to L2
      next_ok = fetch_record(c + 1, buf ^ 1);
      if (next_ok) rec_pend |= 1 << (buf ^ 1);
      if (c + 2 < nch && ld_acquire_gpu(&claims[c + 2]) == kClaimReady)
        l2_prefetch(reinterpret_cast<const unsigned char*>(p.status) + kSplitHeader +
                        ((int64_t)(slot0 + c + 2) * H + h) * kRecBytes,
                    kRecBytes);
    }
    if (jr > 0) {
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int idx = tid + k2 * NT;
        const int r = idx >> 4, v8 = idx & 15;
        const int64_t row =
            kRowMap ? (int64_t)orow[((c - 1) & 1) * C + r] : (int64_t)(c0 - C + r);
        if (r < L_prev && row >= 0) {
          const uint4 val = *reinterpret_cast<const uint4*>(sm + OFF_OSTR + r * 256 + v8 * 16);
          *reinterpret_cast<uint4*>(p.out + (size_t)row * HD + xcol + v8 * 8) = val;
        }
      }
    }
    {
      const bool okm = next_ok && (tid != 0 || mbar_wait(bar_mma, ph_mma));
      ph_mma ^= 1;
      tc_fence_before();
      if (__syncthreads_or(!okm)) { failed = true; site = 81; break; }   // (B)
    }
    tc_fence_after();
    if (tid == 0 && more) {   // the v tile is free again
      mbar_expect_tx(bar_v, 16384);
      tma_load_2d(sb + OFF_INV, &tm_v, xcol, c0 + C, bar_v);
      tma_load_2d(sb + OFF_INV + 8192, &tm_v, xcol + 64, c0 + C, bar_v);
    }

    // R4: U^T diag(1/|k|) -> bf16 operand in TMEM
    if (cs < 2) {
      uint32_t x[32], pk[16];
      tmem_ld32(tmem + lane_base + TM_U + cs * 32, x);
      tmem_wait_ld();
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 ik = ld4(vec + 192 + cs * 32 + 4 * j4);
        pk[2 * j4] = pack_bf16x2(__uint_as_float(x[4 * j4]) * ik.x,
                                 __uint_as_float(x[4 * j4 + 1]) * ik.y);
        pk[2 * j4 + 1] = pack_bf16x2(__uint_as_float(x[4 * j4 + 2]) * ik.z,
                                     __uint_as_float(x[4 * j4 + 3]) * ik.w);
      }
      tmem_st16(tmem + lane_base + TM_UB + cs * 16, pk);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();   // (C)

    // R5: [O^T | S^T] += U^T [QK; Ke]^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_ts(tmem + TM_O, tmem + TM_UB + 8 * ks, kdesc(rb + kRecQKE, 192, ks), ID_KK192, 1);
      mma_commit(bar_mma);
    }
    {
      const bool okm = tid != 0 || mbar_wait(bar_mma, ph_mma);
      ph_mma ^= 1;
      tc_fence_before();
      if (__syncthreads_or(!okm)) { failed = true; site = 82; break; }   // (D)
    }
    tc_fence_after();
    L_prev = L;
    ++jr;
  }

  if (!failed && flags[1] && jr > 0) {   // O of the last (record-mode) chunk
    const float* iqp =
        reinterpret_cast<const float*>(sm + (((jr - 1) & 1) ? OFF_REC1 : OFF_REC0) + kRecVec) + 128;
    uint32_t r[16];
    tmem_ld16(tmem + lane_base + TM_O + cs * 16, r);
    tmem_wait_ld();
    __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(sm + OFF_OSTR);
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      const float4 iq = ld4(iqp + cs * 16 + 4 * j4);
      const float iqv[4] = {iq.x, iq.y, iq.z, iq.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * j4 + e;
        ost[(cs * 16 + j) * D + my_lane] = __float2bfloat16_rn(__uint_as_float(r[j]) * iqv[e]);
      }
    }
    __syncthreads();
    const int c0 = t0 + C * (nch - 1);
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int idx = tid + k2 * NT;
      const int r2 = idx >> 4, v8 = idx & 15;
      const int64_t row =
          kRowMap ? (int64_t)orow[((nch - 1) & 1) * C + r2] : (int64_t)(c0 + r2);
      if (r2 < L_prev && row >= 0) {
        const uint4 val = *reinterpret_cast<const uint4*>(sm + OFF_OSTR + r2 * 256 + v8 * 16);
        *reinterpret_cast<uint4*>(p.out + (size_t)row * HD + xcol + v8 * 8) = val;
      }
    }
  }
  if (failed) {
    if (tid == 0) record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
    if (tid == kFetcher) {
      if (rec_pend & 1) mbar_wait(bar_rec0, ph_rec & 1u);
      if (rec_pend & 2) mbar_wait(bar_rec1, (ph_rec >> 1) & 1u);
    }
    // let copies still in flight finish (bounded) before the CTA exits
    mbar_wait(bar_qkg, ph_qkg);
    mbar_wait(bar_v, ph_v);
    mbar_wait(bar_mma, ph_mma);
    mbar_wait(bar_o, ph_o);
  } else {
    // ---- state out (slice columns only)
    const int dv = my_lane;
    const int dk0 = cs * 32;
    uint32_t r[32];
    tmem_ld32(tmem + lane_base + TM_S + dk0, r);
    tmem_wait_ld();
    if (dv >= dv_lo && dv < dv_hi) {
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
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace
}  // namespace kda

namespace kda {
// The row-map build of the kernel above (kda_tc_rowmap_kernel.cu), launched by launch_tc
// when the call gives an out_index map.
cudaError_t launch_tc_rowmap(const Params& p, unsigned blocks, const CUtensorMap& mq,
                             const CUtensorMap& mk, const CUtensorMap& mg, const CUtensorMap& mv,
                             cudaStream_t stream);
}  // namespace kda
