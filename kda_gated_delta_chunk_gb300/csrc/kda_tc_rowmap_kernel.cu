// The fused tcgen05 prefill kernel writing its outputs through an out_index row map
// (kda_chunk_prefill_fwd_scatter): the body of kda_tc_kernel.cuh compiled as a kernel of
// its own, so that the dense kernel in kda_tc_kernel.cu carries none of the map.
#define KDA_TC_KERNEL_NAME kda_tc_chunk_kernel_rowmap
#define KDA_TC_ROW_MAP true
#include "kda_tc_kernel.cuh"

namespace kda {

cudaError_t launch_tc_rowmap(const Params& p, unsigned blocks, const CUtensorMap& mq,
                             const CUtensorMap& mk, const CUtensorMap& mg, const CUtensorMap& mv,
                             cudaStream_t stream) {
  static PerDeviceOnce attr_once;   // the shared-memory attribute, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = attr_once.run(dev, [&]() -> cudaError_t {
    e = cudaFuncSetAttribute(kda_tc_chunk_kernel_rowmap,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES_MAP);
    if (e != cudaSuccess) return e;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  kda_tc_chunk_kernel_rowmap<<<blocks, NT, SMEM_BYTES_MAP, stream>>>(p, mq, mk, mg, mv);
  return cudaGetLastError();
}

}  // namespace kda
