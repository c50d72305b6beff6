// The low-M projections in front of KDA: two "skinny" GEMMs of a decode or small prefill
// step (m <= 16 token rows), bf16 operands, fp32 accumulation, bf16 results:
//   Y = X W_ab^T                  X [m, k], W_ab [n_ab, k]        ->  Y [m, n_ab]
//   Z = bf16(Y[:, :r]) W_b^T      W_b [n_b, r]                    ->  Z [m, n_b]
// These are the shapes of the Kimi-K3 low-M KDA projection overlap in the vLLM PR report
// "[Bugfix] Fix Kimi-K3 KDA projection overlap compile on Hopper" (Implementation
// breakdown and the skinny-GEMM test listing): hidden 7168 -> 144 with the first 128
// columns feeding the 128 -> 1536 up-projection, m from 1 to 14.
//
// Both GEMMs are bound by reading the weights.  The first splits K over CTAs: a CTA owns 16
// output columns and 512 of K, stages its X and W_ab tiles with cp.async and runs
// m16n8k16 tensor-core MMAs (tokens padded to 16 rows); the K-block partial sums go to the
// workspace and the last CTA of each column block (an arrival counter) adds them in K-block
// order -- deterministic -- and writes Y.  The second GEMM is launched as the first's
// programmatic dependent: its CTAs fetch their W_b rows while the first runs, then wait for
// it (griddepcontrol.wait) and read Y.
#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int PM = 16;           // token rows of an MMA tile
constexpr int PKB = 512;         // K per CTA of the first GEMM
constexpr int PKS = PKB + 8;     // shared-memory row stride (elements): ldmatrix without conflicts
constexpr int PNT = 256;         // threads of the first GEMM's CTAs
constexpr int PNT2 = 64;         // ... of the second's (two warps: two 8-column tiles)

struct ProjParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* w_ab;
  const __nv_bfloat16* w_b;
  __nv_bfloat16* y;
  __nv_bfloat16* z;
  int64_t ldx, ldy, ldz;
  int m, k, n_ab, r, n_b;
  int* count;    // [n_ab / 16] arrival counters (zero between calls)
  float* part;   // [k / 512][16][n_ab] K-block partial sums
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
// D += A (16 x 16, row) B (16 x 8, col), bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// A CTA: output columns [16 nb, 16 nb + 16) over K block kb.  Warp w multiplies the
// 8-column tile (w & 1) over the K quarter (w >> 1) of the block.
__global__ void __launch_bounds__(PNT) kda_proj_n_kernel(const __grid_constant__ ProjParams pp) {
  pdl_launch_dependents();   // the second GEMM may start fetching its weights
  extern __shared__ __align__(16) unsigned char smp[];
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smp);   // [16][PKS]
  __nv_bfloat16* ws = xs + PM * PKS;                            // [16][PKS]
  float* red = reinterpret_cast<float*>(ws + PM * PKS);         // [4 K quarters][16][16]
  int* last = reinterpret_cast<int*>(red + 4 * 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nkb = pp.k / PKB;
  const int nb = blockIdx.x / nkb, kb = blockIdx.x % nkb;

  // X rows (tokens >= m read as zero) and W_ab rows of the tile, in 16-byte chunks
  constexpr int CPR = PKB / 8;   // chunks per row
  for (int i = tid; i < 2 * PM * CPR; i += PNT) {
    const int t = i / (PM * CPR), row = (i / CPR) % PM, ch = i % CPR;
    __nv_bfloat16* dst = (t ? ws : xs) + row * PKS + ch * 8;
    if (t == 0 && row >= pp.m) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const __nv_bfloat16* src =
        t ? pp.w_ab + (size_t)(16 * nb + row) * pp.k + (size_t)kb * PKB + ch * 8
          : pp.x + (size_t)row * pp.ldx + (size_t)kb * PKB + ch * 8;
    cp_async16(smem_u32(dst), src);
  }
  cp_async_wait_all();
  __syncthreads();

  float c[4] = {0.f, 0.f, 0.f, 0.f};
  const int n8 = warp & 1, kq = warp >> 1;
  constexpr int SPQ = PKB / 64;   // k16 steps per K quarter
#pragma unroll
  for (int s = 0; s < SPQ; ++s) {
    const int k0 = (SPQ * kq + s) * 16;
    uint32_t a[4], b[2];
    ldsm4(smem_u32(xs + (lane & 15) * PKS + k0 + (lane >> 4) * 8), a);
    ldsm2(smem_u32(ws + (8 * n8 + (lane & 7)) * PKS + k0 + ((lane >> 3) & 1) * 8), b);
    mma_bf16_16816(c, a, b);
  }
  {   // accumulator (token lane / 4 (+ 8), column 8 n8 + 2 (lane % 4) (+ 1)) -> K-quarter slab
    float* rq = red + kq * 256;
    const int tr = lane >> 2, tc = 8 * n8 + 2 * (lane & 3);
    rq[tr * 16 + tc] = c[0];
    rq[tr * 16 + tc + 1] = c[1];
    rq[(tr + 8) * 16 + tc] = c[2];
    rq[(tr + 8) * 16 + tc + 1] = c[3];
  }
  __syncthreads();
  const int tok = tid >> 4, col = tid & 15;
  {
    const float v = (red[tid] + red[256 + tid]) + (red[512 + tid] + red[768 + tid]);
    pp.part[((size_t)kb * PM + tok) * pp.n_ab + 16 * nb + col] = v;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *last = atomicAdd(&pp.count[nb], 1) == nkb - 1;
  __syncthreads();
  if (!*last) return;
  // the last CTA of the column block: the K blocks in order, then Y
  __threadfence();
  float s = 0.0f;   // K-block order; the loads of a group of 8 are in flight together
  const float* src = pp.part + (size_t)tok * pp.n_ab + 16 * nb + col;
  const size_t bstride = (size_t)PM * pp.n_ab;
  for (int b0 = 0; b0 < nkb; b0 += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (b0 + j < nkb) ? __ldcg(src + (b0 + j) * bstride) : 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
  }
  if (tok < pp.m) pp.y[(size_t)tok * pp.ldy + 16 * nb + col] = __float2bfloat16_rn(s);
  if (tid == 0) pp.count[nb] = 0;   // ready for the next call
}

// A CTA: output columns [16 nb, 16 nb + 16) of Z; warp w the 8-column tile w.
__global__ void __launch_bounds__(PNT2) kda_proj_k_kernel(const __grid_constant__ ProjParams pp) {
  extern __shared__ __align__(16) unsigned char smp[];
  const int RS = pp.r + 8;
  __nv_bfloat16* wbs = reinterpret_cast<__nv_bfloat16*>(smp);   // [16][RS]
  __nv_bfloat16* ys = wbs + PM * RS;                             // [16][RS]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = blockIdx.x;
  const int cpr = pp.r / 8;   // 16-byte chunks per row
  // W_b rows: they do not depend on the first GEMM
  for (int i = tid; i < PM * cpr; i += PNT2) {
    const int row = i / cpr, ch = i % cpr;
    cp_async16(smem_u32(wbs + row * RS + ch * 8), pp.w_b + (size_t)(16 * nb + row) * pp.r + ch * 8);
  }
  pdl_wait();   // the first GEMM has completed and Y is visible
  for (int i = tid; i < PM * cpr; i += PNT2) {
    const int row = i / cpr, ch = i % cpr;
    __nv_bfloat16* dst = ys + row * RS + ch * 8;
    if (row < pp.m)
      cp_async16(smem_u32(dst), pp.y + (size_t)row * pp.ldy + ch * 8);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  cp_async_wait_all();
  __syncthreads();
  float c[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < pp.r; k0 += 16) {
    uint32_t a[4], b[2];
    ldsm4(smem_u32(ys + (lane & 15) * RS + k0 + (lane >> 4) * 8), a);
    ldsm2(smem_u32(wbs + (8 * warp + (lane & 7)) * RS + k0 + ((lane >> 3) & 1) * 8), b);
    mma_bf16_16816(c, a, b);
  }
  const int tr = lane >> 2, n = 16 * nb + 8 * warp + 2 * (lane & 3);
  if (tr < pp.m)
    *reinterpret_cast<__nv_bfloat162*>(pp.z + (size_t)tr * pp.ldz + n) = __floats2bfloat162_rn(c[0], c[1]);
  if (tr + 8 < pp.m)
    *reinterpret_cast<__nv_bfloat162*>(pp.z + (size_t)(tr + 8) * pp.ldz + n) =
        __floats2bfloat162_rn(c[2], c[3]);
}

}  // namespace

size_t proj_workspace_bytes(int32_t k, int32_t n_ab) {
  if (k <= 0 || n_ab <= 0) return 0;
  const size_t counters = (((size_t)(n_ab / 16) * sizeof(int) + 255) / 256) * 256;
  return 256 + counters + (size_t)(k / PKB) * PM * n_ab * sizeof(float);
}

int proj_smem_first() { return 2 * PM * PKS * 2 + 4 * 256 * 4 + 16; }

cudaError_t launch_proj(const void* x, int64_t ldx, const void* w_ab, const void* w_b, void* y,
                        int64_t ldy, void* z, int64_t ldz, int32_t m, int32_t k, int32_t n_ab,
                        int32_t r, int32_t n_b, void* workspace, cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int smem1 = proj_smem_first();
  e = attr_once.run(dev, [&]() -> cudaError_t {
    e = cudaFuncSetAttribute(kda_proj_n_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_proj_k_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             2 * PM * (512 + 8) * 2);
    if (e != cudaSuccess) return e;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  ProjParams pp;
  pp.x = static_cast<const __nv_bfloat16*>(x);
  pp.w_ab = static_cast<const __nv_bfloat16*>(w_ab);
  pp.w_b = static_cast<const __nv_bfloat16*>(w_b);
  pp.y = static_cast<__nv_bfloat16*>(y);
  pp.z = static_cast<__nv_bfloat16*>(z);
  pp.ldx = ldx;
  pp.ldy = ldy;
  pp.ldz = ldz;
  pp.m = m;
  pp.k = k;
  pp.n_ab = n_ab;
  pp.r = r;
  pp.n_b = n_b;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const size_t counters = (((size_t)(n_ab / 16) * sizeof(int) + 255) / 256) * 256;
  pp.count = reinterpret_cast<int*>(ws + 256);
  pp.part = reinterpret_cast<float*>(ws + 256 + counters);
  const unsigned blocks1 = (unsigned)((n_ab / 16) * (k / PKB));
  kda_proj_n_kernel<<<blocks1, PNT, smem1, stream>>>(pp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_b / 16));
  cfg.blockDim = dim3(PNT2);
  cfg.dynamicSmemBytes = 2 * PM * (r + 8) * 2;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kda_proj_k_kernel, pp);
}

}  // namespace kda
