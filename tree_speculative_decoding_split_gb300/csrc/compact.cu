// K4: KV compaction after acceptance.
//
// Candidates after a rejection are discarded and the accepted prefix is kept (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "棄却サンプリング").  The
// accepted path's K/V rows are gathered from their tree slots L + path[j] to L + j, in place.
// One CTA per (request, KV head); the row copies go in increasing j with a barrier between
// rows.  That order is hazard-free: path[j] >= j for a root path in topological order, so the
// only destination slot a later row can read from (L + path[j'] = L + j with j > j') belongs
// to a row that is written after row j' has been read.

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

__global__ void __launch_bounds__(128) compact_kv_kernel(
    uint8_t* __restrict__ k, uint8_t* __restrict__ v, int row_bytes, const int32_t* __restrict__ prefix_len,
    const int32_t* __restrict__ path, const int32_t* __restrict__ accept_len, int Hkv, long long L_cap,
    int path_cap, int32_t* __restrict__ src_slot, int32_t* __restrict__ new_len, int32_t* dev_status) {
  const int b = blockIdx.x / Hkv, g = blockIdx.x % Hkv, tid = threadIdx.x;
  const long long L = prefix_len[b];
  const int len = accept_len[b];
  const int32_t* pth = path + (size_t)b * path_cap;
  __shared__ int s_err;
  if (tid == 0) {
    int err = 0;
    if (len < 0 || len >= path_cap || L < 0 || pth[0] != 0) {
      err = (len >= path_cap) ? SPEC_ERR_CAPACITY : SPEC_ERR_BAD_TREE;
    } else {
      for (int j = 1; j <= len; ++j)
        if (pth[j] <= pth[j - 1]) { err = SPEC_ERR_BAD_TREE; break; }
      if (!err && L + pth[len] >= L_cap) err = SPEC_ERR_CAPACITY;
    }
    s_err = err;
  }
  __syncthreads();
  if (s_err) {
    if (g == 0) {
      if (tid == 0) {
        set_status(dev_status, s_err);
        if (new_len) new_len[b] = (int)L;
      }
      if (src_slot)
        for (int j = tid; j < path_cap; j += blockDim.x) src_slot[(size_t)b * path_cap + j] = -1;
    }
    return;
  }
  const int chunks = row_bytes / 16;
  const size_t head_off = ((size_t)b * Hkv + g) * (size_t)L_cap;
  for (int j = 1; j <= len; ++j) {
    const size_t src = head_off + (size_t)(L + pth[j]);
    const size_t dst = head_off + (size_t)(L + j);
    if (src != dst) {
      for (int c = tid; c < 2 * chunks; c += blockDim.x) {
        uint8_t* base = (c < chunks) ? k : v;
        const int cc = (c < chunks) ? c : c - chunks;
        const uint4 val = *reinterpret_cast<const uint4*>(base + src * row_bytes + cc * 16);
        *reinterpret_cast<uint4*>(base + dst * row_bytes + cc * 16) = val;
      }
    }
    __syncthreads();
  }
  if (g == 0) {
    if (src_slot)
      for (int j = tid; j < path_cap; j += blockDim.x)
        src_slot[(size_t)b * path_cap + j] = (j <= len) ? (int)(L + pth[j]) : -1;
    if (tid == 0 && new_len) new_len[b] = (int)(L + 1 + len);
  }
}

void launch_compact_kv(void* k, void* v, int elem_bytes, const int32_t* prefix_len,
                       const int32_t* path, const int32_t* accept_len, int B, int Hkv, int d,
                       long long L_cap, int path_cap, int32_t* src_slot, int32_t* new_len,
                       int32_t* dev_status, cudaStream_t stream) {
  compact_kv_kernel<<<B * Hkv, 128, 0, stream>>>(static_cast<uint8_t*>(k), static_cast<uint8_t*>(v),
                                                d * elem_bytes, prefix_len, path, accept_len, Hkv,
                                                L_cap, path_cap, src_slot, new_len, dev_status);
}

}  // namespace spectree
