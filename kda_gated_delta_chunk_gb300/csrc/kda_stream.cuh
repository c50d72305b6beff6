// Device side of the streamed split path shared by the chain kernels: the chain grid runs
// beside the k-side grid (programmatic dependent launch) and copies each record once the
// k-side kernel has published it through its claim word (kClaimStreamed, kda_internal.cuh).
#pragma once

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {

// Producer thread of a chain CTA, before it copies record (slot, head): waits (acquire,
// about a second at most) for the record's claim word, then orders its bulk copy after the
// k-side kernel's generic stores.  False (with KDA_ERR_DEVICE_TIMEOUT recorded at `site`)
// when the wait gives up.
__device__ __forceinline__ bool stream_wait_record(const Params& p, int64_t slot, int head,
                                                   int site) {
  const int* claim =
      reinterpret_cast<const int*>(reinterpret_cast<const unsigned char*>(p.status) +
                                   helper_claims_offset(p.total_tokens, p.heads, p.num_seqs)) +
      claim_index(slot, head, p.total_tokens, p.num_seqs);
  if (!sm100::wait_flag(claim, kClaimStreamed)) {
    record_error(p.status, KDA_ERR_DEVICE_TIMEOUT, site);
    return false;
  }
  sm100::fence_proxy_async_global();
  return true;
}

// At the end of every chain CTA (threads 0 .. nthr-1 of it; `sync` is a barrier over them):
// once the k-side grid has completed, the last chain CTA to finish clears the claim words of
// the call and the path's counters, so that the next call starts from zero.  `last_s` is a
// shared-memory word.
template <typename Sync>
__device__ void stream_finish(const Params& p, int tid, int nthr, int* last_s, Sync sync) {
  if (tid == 0) {
    sm100::pdl_wait();
    __threadfence();
    *last_s = atomicAdd(p.status + kStreamDoneWord, 1) == (int)gridDim.x - 1;
  }
  sync();
  if (!*last_s) return;
  __threadfence();
  int* claims = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(p.status) +
                                       helper_claims_offset(p.total_tokens, p.heads, p.num_seqs));
  const int64_t items = split_slots(p.total_tokens, p.num_seqs) * p.heads;
  for (int64_t i = tid; i < items; i += nthr) claims[i] = kClaimFree;
  if (tid == 0) {
    p.status[kStreamCounterWord] = 0;
    p.status[kStreamYieldWord] = 0;
    p.status[kStreamDoneWord] = 0;
    p.status[kStreamStartWord] = 0;
  }
}

}  // namespace kda
