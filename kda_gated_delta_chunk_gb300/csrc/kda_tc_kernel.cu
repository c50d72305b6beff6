// tcgen05 + TMA chunked KDA prefill (KDA_KERNEL_TC), 64-token chunks.
//
// One CTA (512 threads, ~209 KB shared memory, 512 TMEM columns) owns one
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
// log2 e).  Products between the blocks reuse the block-1 row operand; their
// column operand Kc2 carries 2^(B0 - c_s) * 2^(alpha_1), a product of two
// factors <= 1, so one MMA with N = 96 yields the diagonal blocks (columns
// 0-63) and the off-diagonal block (columns 64-95) together.  At the block
// boundary Kc2's factor is 2^(alpha_1) >= 2^(-16|lb| log2 e): with |lb| <= 5
// that is >= 2^-116, leaving 2^10 of headroom above the smallest normal
// number for the smaller entries of a row.  q and k rows enter scaled by a
// power of two to |row| <= 1, so the factors bound the operands.
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
//
// With k-side helpers (KDA_KERNEL_TC_HELPERS) the CTAs of the k-side kernel
// run on the SMs this grid leaves free, as its programmatic dependent: they
// compute the chunk-local half of chunks taken from the end of each sequence
// and write it as a record.  Once this CTA meets a chunk a helper has taken,
// it reads that chunk and every later one from records (the chunk step of the
// chain kernel: [U^T | O^T] and [O^T | S^T] as single accumulators), with the
// same order of accumulation as above, so the result does not depend on which
// CTA computed which chunk.
#define KDA_TC_KERNEL_NAME kda_tc_chunk_kernel
#define KDA_TC_ROW_MAP false
#include "kda_tc_kernel.cuh"

namespace kda {
namespace {

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // looked up once (a function-local static: initialised once even when threads race)
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    cudaGetLastError();
    return nullptr;
  }();
  return fn;
}

// A [T rows][H*128 cols] bf16 view of q/k/g/v with a row stride of `stride` elements;
// box {box_cols, 64 rows}.
bool make_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, int64_t T, int H,
              int64_t stride, int box_cols, bool swizzle) {
  cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)C};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

void* tensor_map_encoder() { return reinterpret_cast<void*>(encode_fn()); }

cudaError_t launch_tc(const Params& p, cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = attr_once.run(dev, [&]() -> cudaError_t {
    e = cudaFuncSetAttribute(kda_tc_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
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
  if (!make_map(enc, &mq, qb, p.total_tokens, p.heads, p.s_q, D, false) ||
      !make_map(enc, &mk, kb, p.total_tokens, p.heads, p.s_k, D, false) ||
      !make_map(enc, &mg, gb, p.total_tokens, p.heads, p.s_g, D, false) ||
      !make_map(enc, &mv, vb, p.total_tokens, p.heads, p.s_v, 64, true))
    return cudaErrorInvalidValue;
  if (p.out_index) {
    e = launch_tc_rowmap(p, (unsigned)blocks, mq, mk, mg, mv, stream);
  } else {
    kda_tc_chunk_kernel<<<(unsigned)blocks, NT, SMEM_BYTES, stream>>>(p, mq, mk, mg, mv);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || !p.helpers) return e;
  return launch_kside_helpers(p, stream);
}

}  // namespace kda
