// Split path, first kernel: the chunk-local (state-free) half of the chunked KDA
// step for every (chunk, head), written to the workspace as one record each.
//
// Per item (64-token chunk c, head h), with Gam the inclusive cumsum of the log2
// decay over the chunk per key channel (gate of the FlashKDA prefill PR report,
// PR #55737, Features & motivation), raw q / k (their l2 norms are folded in as
// the per-token scalars 1/|q|, 1/|k|):
//   A[r,s]  = b_r kh_r.kh_s 2^(Gam_r - Gam_s)  (s < r),  QK[r,s] = q_r.k_s 2^(Gam_r - Gam_s)  (s <= r)
//   T = (I + A)^-1,  W = T diag(b) (kh 2^Gam),  Qg = q 2^Gam,  Ke = k 2^(Gam_last - Gam)
// The record (layout in kda_internal.cuh) holds -W and Qg as one MN-major tile,
// QK and Ke as one K-major tile, T diag(b), 2^Gam_last and the norm scalars --
// exactly the shared-memory operand images the chain kernels multiply with.
//
// The products A/QK (one N = 96 MMA over the exponent-anchored operands, two
// 32-token blocks anchored at their 16th token) and W run on tcgen05; T is the
// blocked substitution + tf32 product of the fused kernel.  Items are independent,
// so the kernel is built for throughput: 256 threads, ~110 KB of shared memory and
// 128 TMEM columns per CTA, two CTAs per SM, persistent over the (slot, head)
// items; the record tiles go straight from registers to global memory as 16-byte
// chunks of the swizzled images.
//
// Helper mode (KDA_KERNEL_TC_HELPERS): launched behind the fused kernel on the SMs
// it leaves free, the CTAs take items from a shared counter, last chunk index
// first, claim each as they start it and publish the record with a release
// store; the first claim lost to the sequence's own CTA ends a helper.
//
// Streamed mode (KDA_KERNEL_SPLIT_STREAMED, Params::stream_sms > 0): the chain kernel
// is this grid's programmatic dependent and runs beside it.  Every CTA lets it start
// at once; the CTAs that start on the chains' SMs (%smid below stream_sms, at most
// two per such SM) give up the tensor-memory allocation permit, wait until the whole
// grid has started and leave; the others take items from the path's counter, first
// chunk index first, and publish each record through its claim word.
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
constexpr int NT = 256;

// ---- shared memory (offsets from a 1024-byte aligned base)
constexpr int K_INQ = 0;          // q tile [64][128] bf16 row-major (TMA)
constexpr int K_INK = 16384;      // k tile
constexpr int K_ING = 32768;      // g tile (dead after the gate)
constexpr int K_RKQ = 32768;      // [Kr; Qr] K-major 128 x 128 (over g; live until W)
constexpr int K_CKC = 65536;      // [Kc; Kc2] K-major 96 x 128 (live until the A/QK MMA ends)
constexpr int K_TM = 0;           // T   [64][NS] fp32 (over q, k after the A/QK MMA)
constexpr int K_Y = K_TM + 64 * NS * 4;      // product scratch [32][NS]
constexpr int K_NM = 65536;       // N = diag(b/|k|) strict(A) diag(1/|k|) [64][NS] (over Kc)
constexpr int K_TB = 90112;       // T diag(b/|k|) K-major 64 x 64 bf16 (B of the W MMA)
constexpr int K_MISC = 98304;
constexpr int K_INVN = K_MISC;            // scale/|q| [64], 1/|k| [64]
constexpr int K_BETA = K_MISC + 512;      // b [64]
constexpr int K_WF = K_MISC + 768;        // W factors [3][128]
constexpr int K_GT = K_MISC + 2304;       // 8-row group totals [8][128]
constexpr int K_PART = K_MISC + 6400;     // norm partial sums [8 warps][32]
constexpr int K_BAR = K_MISC + 7424;      // 2 mbarriers
constexpr int K_TSLOT = K_MISC + 7440;
constexpr int K_FLAGS = K_MISC + 7456;    // items {item, c0, t1, head, k} x 3, 8 ints apart
constexpr int K_SGD = K_MISC + 7552;      // gate terms -e^{A_log} log2e dt_bias [128], -e^{A_log} log2e
constexpr int K_RSC = K_MISC + 8192;      // per-row power-of-two operand scales, bf16x2 [q 64][k 64]
constexpr int K_MAXC = K_MISC + 8176;     // helper mode: chunks of the longest sequence
constexpr int K_CU = K_RSC + 512;         // cu_seqlens cache (batches of up to kCuCache sequences)
constexpr int kCuCache = 1023;
constexpr int K_ORD = K_CU + 4 * (kCuCache + 1);   // helper mode: sequences, longest first
constexpr int K_SMEM_USED = K_ORD + 4 * kHelperMaxSeqs;
constexpr int K_SMEM_BYTES = K_SMEM_USED + 1024;
static_assert(K_Y + 32 * NS * 4 <= K_RKQ, "T scratch overlaps [Kr; Qr]");
static_assert(K_NM + 64 * NS * 4 <= K_TB, "N overlaps T diag(b)");
static_assert(K_FLAGS + 24 * 4 <= K_SGD && K_SGD + 129 * 4 <= K_MAXC && K_MAXC + 4 <= K_RSC, "misc");
static_assert(2 * (K_SMEM_BYTES + 1024) <= 228 * 1024, "two CTAs per SM");

constexpr uint32_t TM_D = 0;      // A | QK (96 cols), then W0^T at 0, W1^T at 64
constexpr uint32_t TM_COLS = 128;
constexpr uint32_t ID_KK96 = idesc_bf16(128, 96, 0, 0);
constexpr uint32_t ID_MK64 = idesc_bf16(128, 64, 1, 0);

// (slot, head) item -> chunk; slot of chunk c of sequence n is floor(cu[n] / 64) + n + c.
// `cu` is cu_seqlens (a shared-memory copy when the batch is small enough).
__device__ bool decode_item(const Params& p, const int* cu, int it, int* c0, int* t1) {
  const int slot = it / p.heads;
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((cu[mid] >> 6) + mid <= slot)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int a = cu[lo], b = cu[lo + 1];
  const int c = slot - ((a >> 6) + lo);
  if (a < 0 || c < 0 || (int64_t)b > p.total_tokens) return false;
  const int64_t s = (int64_t)a + (int64_t)C * c;
  if (s >= b) return false;
  *c0 = (int)s;
  *t1 = b;
  return true;
}
// The k-th item of this CTA counting down from the last slot (so the records of the
// first chunks are written last and are still in L2 when the chain kernel starts):
// {item, c0, t1, head, k'} with k' the counter it was found at; item = -1 when none is left.
__device__ void find_item(const Params& p, const int* cu, int k, int total, int* out) {
  out[0] = -1;
  out[1] = out[2] = out[3] = out[4] = 0;
  for (int64_t idx = blockIdx.x + (int64_t)k * gridDim.x; idx < total; idx += gridDim.x) {
    const int it = total - 1 - (int)idx;
    int c0, t1;
    if (decode_item(p, cu, it, &c0, &t1)) {
      out[0] = it;
      out[1] = c0;
      out[2] = t1;
      out[3] = it % p.heads;
      out[4] = (int)((idx - blockIdx.x) / gridDim.x);
      return;
    }
  }
}

// Helper mode (behind the fused kernel): the next item from the shared counter, in the
// order last chunk index first, then (sequence by decreasing length, head).  It is claimed
// only when its processing starts.  `ord` lists the sequences longest first, so a
// sequence without chunk `col` ends that column for every helper.  Streamed split path:
// the same walk from the first chunk index on, with the counter of that path.
__device__ void find_helper_item(const Params& p, const int* cu, const int* ord, int max_chunks,
                                 int* out) {
  out[0] = -1;
  out[1] = out[2] = out[3] = out[4] = 0;
  const int NH = p.num_seqs * p.heads;
  const bool fwd = p.stream_sms > 0;
  int* counter = p.status + (fwd ? kStreamCounterWord : kHelperCounterWord);
  const int limit = max_chunks * NH;   // below 2^30 (checked on the host)
  while (true) {
    const int idx = atomicAdd(counter, 1);
    if (idx < 0 || idx >= limit) return;
    const int col = fwd ? idx / NH : max_chunks - 1 - idx / NH;
    const int r = idx % NH;
    const int n = ord[r / p.heads], hh = r % p.heads;
    const int a = cu[n], b = cu[n + 1];
    if (a < 0 || b < a || (int64_t)b > p.total_tokens) return;   // malformed: the fused kernel reports it
    const int64_t s = (int64_t)a + (int64_t)C * col;
    if (s >= b) {   // no chunk `col` here nor in any shorter sequence: skip to the next column
      atomicMax(counter, (idx / NH + 1) * NH);
      continue;
    }
    out[0] = ((a >> 6) + n + col) * p.heads + hh;
    out[1] = (int)s;
    out[2] = b;
    out[3] = hh;
    return;
  }
}

__device__ __forceinline__ int* helper_claim(const Params& p, int item) {
  return reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(p.status) +
                                helper_claims_offset(p.total_tokens, p.heads, p.num_seqs)) +
         claim_index(item / p.heads, item % p.heads, p.total_tokens, p.num_seqs);
}

// two bf16x2 words (token i: lo = channel d0, hi = channel d0 + 1) -> per-channel pairs
__device__ __forceinline__ uint32_t lo_pair(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x5410); }
__device__ __forceinline__ uint32_t hi_pair(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

__global__ void __launch_bounds__(NT, 2)
    kda_kside_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_g) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* inv_q = reinterpret_cast<float*>(sm + K_INVN);
  float* inv_k = inv_q + 64;
  float* beta_s = reinterpret_cast<float*>(sm + K_BETA);
  float* wf = reinterpret_cast<float*>(sm + K_WF);
  float* gt = reinterpret_cast<float*>(sm + K_GT);
  float* part = reinterpret_cast<float*>(sm + K_PART);
  float* Nm = reinterpret_cast<float*>(sm + K_NM);
  float* Tm = reinterpret_cast<float*>(sm + K_TM);
  float* Y = reinterpret_cast<float*>(sm + K_Y);
  int* flags = reinterpret_cast<int*>(sm + K_FLAGS);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + K_TSLOT);
  const uint32_t bar_in = sb + K_BAR, bar_mma = bar_in + 8;
  unsigned char* ws = reinterpret_cast<unsigned char*>(p.status) + kSplitHeader;
  const bool streamed = p.stream_sms > 0;
  if (tid == 0 && blockIdx.x < 512) {
    TSTAMP(1024 + 4 * blockIdx.x, globaltimer_ns());
    TSTAMP(1024 + 4 * blockIdx.x + 3, sm_id());
  }
  if (streamed) {
    pdl_launch_dependents();   // the chain grid may start once every k-side CTA has begun
    // leave the SMs below stream_sms to the chain CTAs (at most two CTAs per such SM yield,
    // so that at least 2 (SMs - stream_sms) of the grid's CTAs make records wherever they run)
    bool yield = false;
    if (tid == 0) {
      atomicAdd(p.status + kStreamStartWord, 1);
      if ((int)sm_id() < p.stream_sms)
        yield = atomicAdd(p.status + kStreamYieldWord, 1) < 2 * p.stream_sms;
    }
    if (__syncthreads_or(yield)) {
      // give up the tensor-memory allocation permit (the SM takes no further CTA of this
      // grid while a resident one still holds it), then hold the SM until every CTA of the
      // grid has started (a few microseconds; 20 at most), so that the CTAs still waiting to
      // be placed land beside this one, not on the SMs the chains will need later
      if (warp == 0) tmem_relinquish();
      if (tid == 0) {
        const uint64_t w0 = globaltimer_ns();
        while (ld_relaxed_gpu(p.status + kStreamStartWord) < (int)gridDim.x &&
               globaltimer_ns() - w0 < 20000ull)
          __nanosleep(128);
      }
      if (tid == 0 && blockIdx.x < 512) {
        TSTAMP(1024 + 4 * blockIdx.x + 1, globaltimer_ns());
        TSTAMP(1024 + 4 * blockIdx.x + 3, sm_id() + 65536u);
      }
      return;
    }
  }

  const int H = p.heads;
  const int total = (int)(split_slots(p.total_tokens, p.num_seqs) * H);
  const int* cu = p.cu_seqlens;
  if (p.num_seqs <= kCuCache) {
    int* cu_s = reinterpret_cast<int*>(sm + K_CU);
    for (int i = tid; i <= p.num_seqs; i += NT) cu_s[i] = p.cu_seqlens[i];
    cu = cu_s;
    __syncthreads();
  }
  // helper mode: the sequences are those of the fused kernel's batch (at most 128, so
  // cu_seqlens is in shared memory), ranked longest first, and the chunk count of the
  // longest (at most ceil(T / 64) even for malformed cu_seqlens)
  int* maxc_s = reinterpret_cast<int*>(sm + K_MAXC);
  int* ord = reinterpret_cast<int*>(sm + K_ORD);
  if (p.helpers || streamed) {
    const int N = p.num_seqs;
    if (tid == 0) *maxc_s = 0;
    __syncthreads();
    for (int i = tid; i < N; i += NT) {
      const int li = cu[i + 1] - cu[i];
      int r = 0;
      for (int m = 0; m < N; ++m) {
        const int lm = cu[m + 1] - cu[m];
        r += (lm > li) || (lm == li && m < i);
      }
      ord[r] = i;
      atomicMax(maxc_s, (li + C - 1) / C);
    }
    __syncthreads();
    if (tid == 0) {
      *maxc_s = min(*maxc_s, (int)((p.total_tokens + C - 1) / C));
      // test hook (Params::test_drop_record): the item of the counter's first index, the last
      // chunk (streamed: the first chunk) of the longest sequence's head 0, is left unpublished
      const int n0 = ord[0];
      flags[6] = ((cu[n0] >> 6) + n0 + (streamed ? 0 : *maxc_s - 1)) * H;
    }
    __syncthreads();
  }
  if (tid == 0) {
    mbar_init(bar_in, 1);
    mbar_init(bar_mma, 1);
    mbar_fence_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_g);
    flags[8] = -1;
    if (p.helpers || streamed) {   // the next item is found during T of the current one
      find_helper_item(p, cu, reinterpret_cast<const int*>(sm + K_ORD), *reinterpret_cast<const int*>(sm + K_MAXC), flags);
    } else {
      find_item(p, cu, 0, total, flags);
      if (flags[0] >= 0) find_item(p, cu, flags[4] + 1, total, flags + 8);
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int q4 = warp & 3, cs = warp >> 2;      // TMEM lane quadrant, column half
  const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
  const int my_lane = 32 * q4 + lane;

  const float lb2 = p.lower_bound * kLog2e;
  const int cp = tid & 63;          // channel pair of the gate / operand phase
  const int rq = tid >> 6;          // row quarter: rows 16 rq .. 16 rq + 15 (groups 2 rq, 2 rq + 1)
  const int d0 = 2 * cp;
  const int blk = rq >> 1;          // 32-token block of this thread's rows

  uint32_t ph_in = 0, ph_mma = 0;
  bool failed = false;
  int site = 0;

  // head parameters and beta of an item -> shared memory, one item ahead (the sigmoid
  // argument of the gate in log2 units is sgd[128] * g + sgd[channel])
  float* sgd = reinterpret_cast<float*>(sm + K_SGD);
  auto load_params = [&](int c0n, int t1n, int hn) {
    if (tid < 128) {
      const float sgn = -expf(p.A_log[hn]) * kLog2e;
      sgd[tid] = sgn * p.dt_bias[hn * D + tid];
      if (tid == 0) sgd[128] = sgn;
    } else if (tid < 128 + C) {
      const int j = tid - 128;
      const float b = (c0n + j < t1n) ? __bfloat162float(p.beta[(size_t)(c0n + j) * p.s_beta + hn]) : 0.0f;
      beta_s[j] = (c0n + j < t1n) ? sigm(b) : 0.0f;
    }
  };
  auto load_inputs = [&](int c0n, int hn) {   // thread 0: q, k, g tiles of an item
    mbar_expect_tx(bar_in, 3 * 16384);
    tma_load_2d(sb + K_INQ, &tm_q, hn * D, c0n, bar_in);
    tma_load_2d(sb + K_INK, &tm_k, hn * D, c0n, bar_in);
    tma_load_2d(sb + K_ING, &tm_g, hn * D, c0n, bar_in);
  };
  if (flags[0] >= 0) {
    if (tid == 0) load_inputs(flags[1], flags[3]);
    load_params(flags[1], flags[2], flags[3]);
  }
  __syncthreads();

#pragma unroll 1
  while (true) {
    const int item = flags[0];
    if (item < 0) break;
    const int c0 = flags[1], t1 = flags[2];
    const int L = min(C, t1 - c0);
    unsigned char* rec = ws + (size_t)item * kRecBytes;

    // ---- P0: inputs of this item (issued during the previous item); the next item's go
    //          to L2 meanwhile
    if (tid == 0 && flags[8] >= 0) {
      tma_prefetch_2d(&tm_q, flags[11] * D, flags[9]);
      tma_prefetch_2d(&tm_k, flags[11] * D, flags[9]);
      tma_prefetch_2d(&tm_g, flags[11] * D, flags[9]);
    }
    // helper mode: claim the item as its processing starts; the answer is looked at after
    // the gate phase, before anything is written to the record
    int claimed = kClaimFree;
    if (p.helpers && tid == 0) claimed = atomicCAS(helper_claim(p, item), kClaimFree, kClaimHelper);
    const float sg = sgd[128], sg0 = sgd[d0], sg1 = sgd[d0 + 1];
    const bool tma_ok = mbar_wait(bar_in, ph_in);
    ph_in ^= 1;
    if (L < C) {   // q, k rows past the sequence end -> 0
      for (int idx = tid; idx < (C - L) * 32; idx += NT) {
        const int r = L + (idx >> 5), c16 = idx & 31;
        st_u128(sm, (c16 < 16 ? K_INQ : K_INK) + r * 256 + (c16 & 15) * 16, make_uint4(0, 0, 0, 0));
      }
    }
    if (__syncthreads_or(!tma_ok)) { failed = true; site = 60; break; }

    // ---- P2a: gate -> log2 decay, cumsum inside each 8-row group of this thread; the
    //           partial sums of squares of q and k
    // (the thread's channel pair as packed fp32x2 throughout: the same roundings, half the
    // instructions)
    float2 cl[16];
    const float2 sg2 = make_float2(sg, sg), sgd = make_float2(sg0, sg1);
#pragma unroll
    for (int gh = 0; gh < 2; ++gh) {
      float2 run = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 16 * rq + 8 * gh + i;
        const float2 gv = unpack_bf16x2(ld_u32(sm + K_ING, (uint32_t)(r * 256 + d0 * 2)));
        const float2 z = __ffma2_rn(gv, sg2, sgd);
        const float2 dd = __fadd2_rn(make_float2(ex2f(z.x), ex2f(z.y)), make_float2(1.0f, 1.0f));
        float2 a = __fmul2_rn(make_float2(rcpf(dd.x), rcpf(dd.y)), make_float2(lb2, lb2));
        if (r >= L) a = make_float2(0.0f, 0.0f);
        run = __fadd2_rn(run, a);
        cl[8 * gh + i] = run;
      }
      *reinterpret_cast<float2*>(gt + (2 * rq + gh) * 128 + d0) = run;
      // sums of squares of the group's q and k rows over this warp's 64 channels,
      // reduce-scattered: lanes 2j, 2j + 1 end with the sum of v[j] ([0, 8) q, [8, 16) k)
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = 16 * rq + 8 * gh + i;
        const float2 qf = unpack_bf16x2(ld_u32(sm + K_INQ, (uint32_t)(r * 256 + d0 * 2)));
        const float2 kf = unpack_bf16x2(ld_u32(sm + K_INK, (uint32_t)(r * 256 + d0 * 2)));
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
      if ((lane & 1) == 0) part[warp * 32 + gh * 16 + (lane >> 1)] = v[0];
    }
    if (p.helpers && tid == 0) flags[5] = claimed;
    __syncthreads();
    // the sequence's own CTA took this chunk first: this helper stops (nothing in flight)
    if (p.helpers && flags[5] != kClaimFree) break;

    // ---- P2c: norms -> scale/|q_r|, 1/|k_r|, and a power of two 2^-s_r per row with
    //           |row| 2^-s_r <= 1.  The operands are built from the rows times 2^-s_r (exact in
    //           bf16) and the scalars carry 2^s_r: the same products, but a raw row can no
    //           longer push an anchored factor (up to 2^(16 |lb| log2 e)) out of range.
    uint32_t* rsc = reinterpret_cast<uint32_t*>(sm + K_RSC);
    if (tid < 128) {   // row r = tid & 63 of q (tid < 64) or k; warps 2 rq, 2 rq + 1 hold its halves
      const int r = tid & 63, t = tid >> 6;
      const int q16 = r >> 4, gh = (r >> 3) & 1, i = r & 7;
      const int pi = gh * 16 + t * 8 + i;
      const float ss = part[(2 * q16) * 32 + pi] + part[(2 * q16 + 1) * 32 + pi];
      // ss < 2^(e+1) -> |row| < 2^ceil((e+1)/2)
      const int e = ((__float_as_int(ss) >> 23) & 255) - 127;
      const int sh = max(-60, min(60, (e + 2) >> 1));
      const float inv = (r < L) ? rsqrtf(ss + kL2Eps) * __int_as_float((127 + sh) << 23) : 0.0f;
      const float val = (t == 0) ? p.scale * inv : inv;
      inv_q[t * 64 + r] = val;
      reinterpret_cast<float*>(rec + kRecVec)[128 + t * 64 + r] = val;
      const uint32_t b = (uint32_t)(127 - sh) << 7;   // bf16 bits of 2^-sh
      rsc[t * 64 + r] = b | (b << 16);
    }
    __syncthreads();

    // ---- P2b: anchored factors; [Kr; Qr], [Kc; Kc2] operand tiles (raw q, k); Qg and Ke
    //           record tiles straight to global
    {
      // per-channel factors, applied per element in fp32 and rounded once (a factor rounded
      // to bf16 per chunk would give every token the same error in that channel).  The
      // products keep the order E cA, Ei cB first: those are near 1, while cA cR or cB cX
      // alone can fall below the fp32 normal range.
      float mE[2][2], cA[2], cB[2], cX[2], cR[2];
      {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float G[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) G[j] = gt[j * 128 + d0 + c];
          const float B0 = (G[0] + G[1]) + (G[2] + G[3]);
          const float B1 = (G[4] + G[5]) + (G[6] + G[7]);
          const float al0 = G[0] + G[1], al1 = G[4] + G[5];
          const float al = blk ? al1 : al0;
#pragma unroll
          for (int gh = 0; gh < 2; ++gh) {
            const int grp = 2 * rq + gh;
            float pre = 0.0f;                      // totals of earlier groups of the block
#pragma unroll
            for (int j = 0; j < 8; ++j)
              if ((j >> 2) == blk && j < grp) pre += G[j];
            mE[gh][c] = al - pre;                  // exponent of E = cl - mE
          }
          cA[c] = ex2f(al);                        // E -> 2^c (within the block)
          cB[c] = ex2f((blk ? B1 : B0) - al);      // Ei -> 2^(B_blk - c)
          cX[c] = ex2f(al1);                       // alpha_1, folded into Kc2
          cR[c] = ex2f(blk ? B0 : B1);             // the other block's total
          if (rq == 0) {
            reinterpret_cast<float*>(rec + kRecVec)[d0 + c] = ex2f(B0 + B1);   // 2^Gam_last
            wf[d0 + c] = cA[c];                    // W block 0: 2^alpha0
            wf[128 + d0 + c] = cX[c];              // W block 1: 2^alpha1, then
            wf[256 + d0 + c] = ex2f(B0);           //            2^B0
          }
        }
      }
      const float2 cA2 = make_float2(cA[0], cA[1]), cB2 = make_float2(cB[0], cB[1]);
      const float2 cX2 = make_float2(cX[0], cX[1]), cR2 = make_float2(cR[0], cR[1]);
#pragma unroll
      for (int gh = 0; gh < 2; ++gh) {
        uint32_t qg[8], ke[8];
        const float2 nmE = make_float2(-mE[gh][0], -mE[gh][1]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ii = 8 * gh + i;
          const int r = 16 * rq + ii;
          const uint32_t q2 = bmul2(ld_u32(sm + K_INQ, (uint32_t)(r * 256 + d0 * 2)), rsc[r]);
          const uint32_t k2 = bmul2(ld_u32(sm + K_INK, (uint32_t)(r * 256 + d0 * 2)), rsc[64 + r]);
          const float2 e = __fadd2_rn(cl[ii], nmE);
          const float2 E = make_float2(ex2f(e.x), ex2f(e.y));
          const float2 Ei = make_float2(ex2f(-e.x), ex2f(-e.y));
          const uint32_t E2 = pack_bf16x2(E.x, E.y), Ei2 = pack_bf16x2(Ei.x, Ei.y);
          st_u32(sm, K_RKQ + kmajor_off(r, d0, 128), bmul2(k2, E2));
          st_u32(sm, K_RKQ + kmajor_off(64 + r, d0, 128), bmul2(q2, E2));
          st_u32(sm, K_CKC + kmajor_off(r, d0, 96), bmul2(k2, Ei2));
          float2 gg, kk;
          if (blk == 0) {
            const float2 oc = __fmul2_rn(Ei, cB2);    // 2^(B0 - c_s)
            const float2 c2 = __fmul2_rn(oc, cX2);
            st_u32(sm, K_CKC + kmajor_off(64 + r, d0, 96), bmul2(k2, pack_bf16x2(c2.x, c2.y)));
            gg = __fmul2_rn(E, cA2);
            kk = __fmul2_rn(oc, cR2);
          } else {
            gg = __fmul2_rn(__fmul2_rn(E, cA2), cR2);
            kk = __fmul2_rn(Ei, cB2);
          }
          qg[i] = bmul2(q2, pack_bf16x2(gg.x, gg.y));
          ke[i] = bmul2(k2, pack_bf16x2(kk.x, kk.y));
        }
        // 8 consecutive tokens of one channel = one 16-byte chunk of each image
        const int r0 = 16 * rq + 8 * gh;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint4 wq, wk;
          if (c == 0) {
            wq = make_uint4(lo_pair(qg[0], qg[1]), lo_pair(qg[2], qg[3]), lo_pair(qg[4], qg[5]),
                            lo_pair(qg[6], qg[7]));
            wk = make_uint4(lo_pair(ke[0], ke[1]), lo_pair(ke[2], ke[3]), lo_pair(ke[4], ke[5]),
                            lo_pair(ke[6], ke[7]));
          } else {
            wq = make_uint4(hi_pair(qg[0], qg[1]), hi_pair(qg[2], qg[3]), hi_pair(qg[4], qg[5]),
                            hi_pair(qg[6], qg[7]));
            wk = make_uint4(hi_pair(ke[0], ke[1]), hi_pair(ke[2], ke[3]), hi_pair(ke[4], ke[5]),
                            hi_pair(ke[6], ke[7]));
          }
          // Qg: MN-major (token contiguous), tokens 64.. of [-W | Qg]
          *reinterpret_cast<uint4*>(rec + kRecWQ + mnmajor_off(64 + r0, d0 + c, 16384)) = wq;
          // Ke: K-major rows 64 + dk of [QK; Ke], K = token
          *reinterpret_cast<uint4*>(rec + kRecQKE + kmajor_off(64 + d0 + c, r0, 192)) = wk;
        }
      }
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P3: D = [Kr; Qr] [Kc; Kc2]^T on the tensor cores
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + TM_D, kdesc(sb + K_RKQ, 128, ks), kdesc(sb + K_CKC, 96, ks), ID_KK96, ks > 0);
      mma_commit(bar_mma);
    }
    {
      const bool ok = tid != 0 || mbar_wait(bar_mma, ph_mma);
      tc_fence_before();
      if (__syncthreads_or(!ok)) { failed = true; site = 63; break; }
      ph_mma ^= 1;
    }
    tc_fence_after();

    // ---- P4a: A rows (lanes 0-63) -> N = diag(b/|k|) strict(A) diag(1/|k|) (smem);
    //           QK rows (64-127) -> raw masked bf16, straight into the [QK; Ke] image
    {
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
          *reinterpret_cast<uint4*>(rec + kRecQKE + kmajor_off(r, 32 * cs + c8 * 8, 192)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // T above the diagonal 16 x 16 blocks is zero
      for (int idx = tid; idx < 6 * 64; idx += NT) {
        const int b = idx >> 6, e = idx & 63;
        const int bi = (b < 3) ? 0 : (b < 5 ? 1 : 2);
        const int bj = (b < 3) ? b + 1 : (b < 5 ? b - 1 : 3);
        *reinterpret_cast<float4*>(Tm + (bi * 16 + (e >> 2)) * NS + bj * 16 + 4 * (e & 3)) =
            make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- P4b: T = (I + N)^-1 on warps 0-3 (16 x 16 diagonal blocks by substitution, then
    //           the off-diagonal blocks as tf32 products); thread 128 finds the item after next
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
    } else if (tid == 128) {
      flags[16] = -1;
      if (p.helpers || streamed)
        find_helper_item(p, cu, reinterpret_cast<const int*>(sm + K_ORD),
                         *reinterpret_cast<const int*>(sm + K_MAXC), flags + 8);
      else if (flags[8] >= 0)
        find_item(p, cu, flags[12] + 1, total, flags + 16);
    }
    __syncthreads();

    // ---- T diag(b/|k|) -> K-major bf16 (W MMA operand); T diag(b) -> record; 16 columns
    //      per thread
    {
      const int r = tid >> 2, c16 = (tid & 3) * 16;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c8 = c16 + 8 * hh;
        float4 t0v = ld4(Tm + r * NS + c8), t1v = ld4(Tm + r * NS + c8 + 4);
        const float4 b0v = ld4(beta_s + c8), b1v = ld4(beta_s + c8 + 4);
        const float4 k0v = ld4(inv_k + c8), k1v = ld4(inv_k + c8 + 4);
        t0v = make_float4(t0v.x * b0v.x, t0v.y * b0v.y, t0v.z * b0v.z, t0v.w * b0v.w);
        t1v = make_float4(t1v.x * b1v.x, t1v.y * b1v.y, t1v.z * b1v.z, t1v.w * b1v.w);
        const uint32_t off = kmajor_off(r, c8, 64);
        *reinterpret_cast<uint4*>(rec + kRecTB + off) =
            make_uint4(pack_bf16x2(t0v.x, t0v.y), pack_bf16x2(t0v.z, t0v.w),
                       pack_bf16x2(t1v.x, t1v.y), pack_bf16x2(t1v.z, t1v.w));
        st_u128(sm, K_TB + off,
                make_uint4(pack_bf16x2(t0v.x * k0v.x, t0v.y * k0v.y),
                           pack_bf16x2(t0v.z * k0v.z, t0v.w * k0v.w),
                           pack_bf16x2(t1v.x * k1v.x, t1v.y * k1v.y),
                           pack_bf16x2(t1v.z * k1v.z, t1v.w * k1v.w)));
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- P5: W_b^T = (raw Kr rows of block b)^T (T diag(b/|k|))[:, b]^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          mma_bf16(tmem + TM_D + 64 * b, mndesc(sb + K_RKQ + 4096 * b, 16384, ks),
                   kdesc(sb + K_TB, 64, 2 * b + ks), ID_MK64, ks > 0);
      mma_commit(bar_mma);
    }
    {
      const bool ok = tid != 0 || mbar_wait(bar_mma, ph_mma);
      tc_fence_before();
      if (__syncthreads_or(!ok)) { failed = true; site = 65; break; }
      ph_mma ^= 1;
    }
    tc_fence_after();
    // the input tiles, beta and the gate terms of this item are no longer read: fetch and
    // load the next item's
    if (flags[8] >= 0) {
      if (tid == 0) load_inputs(flags[9], flags[11]);
      load_params(flags[9], flags[10], flags[11]);
    }

    // ---- P6: -W = -(2^a0 W0 + 2^B0 (2^a1 W1)) -> bf16, MN-major tokens 0-63 of [-W | Qg]
    {
      const int dk = my_lane;
      const float f0 = wf[dk], f1a = wf[128 + dk], f1b = wf[256 + dk];
      uint32_t w0[32], w1[32];
      tmem_ld32(tmem + lane_base + TM_D + cs * 32, w0);
      tmem_ld32(tmem + lane_base + TM_D + 64 + cs * 32, w1);
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
        *reinterpret_cast<uint4*>(rec + kRecWQ + mnmajor_off(cs * 32 + c8 * 8, dk, 16384)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    if (tid == 0) {   // next item becomes the current one (the one after: found during T)
#pragma unroll
      for (int i = 0; i < 5; ++i) {
        flags[i] = flags[8 + i];
        flags[8 + i] = flags[16 + i];
      }
    }
    tc_fence_before();
    __syncthreads();
    if ((p.helpers || streamed) && tid == 0 && !(p.test_drop_record && item == flags[6])) {
      __threadfence();   // publish the record (the barrier orders every thread's part of it
      st_release_gpu(helper_claim(p, item), streamed ? kClaimStreamed : kClaimReady);   // before this fence)
    }
  }

  if (failed && tid == 0) {
    record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
    if (site == 60) mbar_wait(bar_in, ph_in ^ 1);   // let the input copies land (bounded)
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TM_COLS);
  if (tid == 0 && blockIdx.x < 512) TSTAMP(1024 + 4 * blockIdx.x + 1, globaltimer_ns());
  // a helper grid completes only after the fused kernel it serves
  if (p.helpers) pdl_wait();
}

typedef CUresult (*EncodeTiledFnK)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_in_map(EncodeTiledFnK enc, CUtensorMap* m, const void* base, int64_t T, int H,
                 int64_t stride) {
  cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
  cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)C};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_kside(const Params& p, cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = attr_once.run(dev, [&]() -> cudaError_t {
    e = cudaFuncSetAttribute(kda_kside_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             K_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int64_t items = split_slots(p.total_tokens, p.num_seqs) * p.heads;
  if (items <= 0 || p.total_tokens == 0) return cudaSuccess;
  if (items > 0x7fffffffLL - 4096) return cudaErrorInvalidValue;
  EncodeTiledFnK enc = reinterpret_cast<EncodeTiledFnK>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mg;
  if (!make_in_map(enc, &mq, p.q, p.total_tokens, p.heads, p.s_q) ||
      !make_in_map(enc, &mk, p.k, p.total_tokens, p.heads, p.s_k) ||
      !make_in_map(enc, &mg, p.g, p.total_tokens, p.heads, p.s_g))
    return cudaErrorInvalidValue;
  const int64_t cap = 2 * (int64_t)p.sm_count;
  // streamed: two CTAs per SM, of which those on the chains' SMs step aside
  const int64_t grid = (items < cap && p.stream_sms == 0) ? items : cap;
  if (p.stream_sms > 0 && (p.num_seqs > kHelperMaxSeqs ||
                           ((p.total_tokens + C - 1) / C) * p.num_seqs * p.heads >= (1 << 30)))
    return cudaErrorInvalidValue;
  kda_kside_kernel<<<(unsigned)grid, NT, K_SMEM_BYTES, stream>>>(p, mq, mk, mg);
  return cudaGetLastError();
}

// Two helper CTAs per SM that the fused kernel (one CTA per sequence and head) leaves free,
// launched as its programmatic dependent: they start once every fused CTA has cleared its
// claim words, run beside it, and the grid completes after it.
cudaError_t launch_kside_helpers(const Params& p, cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = attr_once.run(dev, [&]() -> cudaError_t {
    e = cudaFuncSetAttribute(kda_kside_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             K_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int64_t free_sms = (int64_t)p.sm_count - (int64_t)p.num_seqs * p.heads;
  if (p.total_tokens == 0 || free_sms <= 0 || p.num_seqs > kHelperMaxSeqs ||
      ((p.total_tokens + C - 1) / C) * p.num_seqs * p.heads >= (1 << 30))
    return cudaErrorInvalidValue;
  EncodeTiledFnK enc = reinterpret_cast<EncodeTiledFnK>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mg;
  if (!make_in_map(enc, &mq, p.q, p.total_tokens, p.heads, p.s_q) ||
      !make_in_map(enc, &mk, p.k, p.total_tokens, p.heads, p.s_k) ||
      !make_in_map(enc, &mg, p.g, p.total_tokens, p.heads, p.s_g))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * free_sms));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = K_SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kda_kside_kernel, p, mq, mk, mg);
}

}  // namespace kda
