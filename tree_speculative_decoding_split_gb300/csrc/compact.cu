// K4: KV compaction after acceptance, one CTA per (request, KV head); the moves themselves are
// in compact.cuh (shared with the acceptance kernels that fold compaction into their tail).
// Paged caches map each logical slot through the request's block table (the moves are the same,
// between physical rows).

#include "common.cuh"
#include "compact.cuh"
#include "kernels.cuh"

namespace spectree {

// One CTA per (request, KV head).
__global__ void __launch_bounds__(128) compact_kv_kernel(const CompactParams c, const int32_t* __restrict__ path,
                                                         const int32_t* __restrict__ accept_len) {
  __shared__ uint4 s_buf[kCompactBufChunks];
  __shared__ int s_pth[kCompactBufChunks / 8];
  const int b = blockIdx.x / c.Hkv, g = blockIdx.x % c.Hkv;
  compact_request(c, path + (size_t)b * c.path_cap, accept_len[b], b, g, c.Hkv, s_buf, s_pth);
}

void launch_compact_kv(const CompactParams& c, const int32_t* path, const int32_t* accept_len, int B,
                       cudaStream_t stream) {
  compact_kv_kernel<<<B * c.Hkv, 128, 0, stream>>>(c, path, accept_len);
}

}  // namespace spectree
