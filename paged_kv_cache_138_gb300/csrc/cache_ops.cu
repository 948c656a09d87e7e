// Cache-consistency kernels for sm_103a: reshape_and_cache (scatter of new
// K/V rows to their slots), the device slot mapping and copy_blocks (the
// copy-on-write block copy).  All are bit-exact data movement with 16-byte
// vector accesses; each checks the indices it reads and skips a bad one after
// recording it in dev_err.
#include <algorithm>

#include "pkv_device.cuh"

namespace pkv {
namespace cache {

constexpr int kThreads = 256;

// One thread moves one 16-byte vector of K and the matching vector of V.
// The cache [num_blocks, bs, Hkv, D] viewed as rows of Hkv*D halves has the
// token of slot `slot` at row `slot` (block slot/bs, offset slot%bs).
__global__ void __launch_bounds__(kThreads)
    reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             const int64_t* __restrict__ slots, uint4* __restrict__ kc,
                             uint4* __restrict__ vc, int64_t total, int row_vecs,
                             int64_t num_slots, int32_t* dev_err) {
  // a programmatically dependent launch that follows (the attention kernel)
  // may place its CTAs while this grid runs; it reads nothing before this
  // grid has completed
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (idx >= total) return;
  const int64_t i = idx / row_vecs;
  const int c = static_cast<int>(idx - i * row_vecs);
  const int64_t slot = __ldg(slots + i);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (c == 0) report(dev_err, PKV_DEV_BAD_SLOT);
    return;
  }
  const uint4 kv = __ldg(k + i * row_vecs + c);
  const uint4 vv = __ldg(v + i * row_vecs + c);
  kc[slot * row_vecs + c] = kv;
  vc[slot * row_vecs + c] = vv;
}

__global__ void __launch_bounds__(kThreads)
    slot_mapping_kernel(const int32_t* __restrict__ tables, const int32_t* __restrict__ positions,
                        int num_seqs, int max_blocks, int block_size, int64_t num_blocks,
                        int64_t* __restrict__ slots, int32_t* dev_err) {
  const int s = blockIdx.x * kThreads + threadIdx.x;
  if (s >= num_seqs) return;
  const int32_t pos = __ldg(positions + s);
  int64_t slot = -1;
  if (pos >= 0) {
    const int32_t logical = pos / block_size;
    if (logical >= max_blocks) {
      report(dev_err, PKV_DEV_BAD_POSITION);
    } else {
      const int32_t b = __ldg(tables + static_cast<int64_t>(s) * max_blocks + logical);
      if (b < 0 || b >= num_blocks)
        report(dev_err, PKV_DEV_BAD_BLOCK_ID);
      else
        slot = static_cast<int64_t>(b) * block_size + pos % block_size;
    }
  }
  slots[s] = slot;
}

constexpr int kMaxLayersPerLaunch = 64;
struct LayerPtrs {
  uint4* k[kMaxLayersPerLaunch];
  uint4* v[kMaxLayersPerLaunch];
};

// grid (pairs x chunks, layers, 2 caches): a CTA copies one chunk of one block
// of one cache, each thread keeping kCopyUnroll 16-byte loads in flight.  A
// 128 KB block (16 tokens x 32 heads x 256 B) is 4 chunks, so a step's few
// hundred copy-on-write pairs still give every SM several CTAs: one CTA per
// block left the copy latency-bound.
constexpr int kCopyUnroll = 8;
constexpr int64_t kCopyChunkVecs = static_cast<int64_t>(kThreads) * kCopyUnroll;

__global__ void __launch_bounds__(kThreads)
    copy_blocks_kernel(const __grid_constant__ LayerPtrs ptrs, const int64_t* __restrict__ pairs,
                       int64_t block_vecs, int chunks, int64_t num_blocks, int32_t* dev_err) {
  // a programmatically dependent launch that follows (the attention kernel)
  // may place its CTAs while this grid runs; it reads nothing before this
  // grid has completed
  asm volatile("griddepcontrol.launch_dependents;");
  const int pair = blockIdx.x / chunks, chunk = blockIdx.x % chunks, layer = blockIdx.y;
  const int64_t src = __ldg(pairs + 2 * pair), dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && chunk == 0 && layer == 0 && blockIdx.z == 0)
      report(dev_err, PKV_DEV_BAD_BLOCK_ID);
    return;
  }
  if (src == dst) return;
  uint4* base = blockIdx.z ? ptrs.v[layer] : ptrs.k[layer];
  const int64_t lo = chunk * kCopyChunkVecs;
  const int64_t hi = min(block_vecs, lo + kCopyChunkVecs);
  const uint4* __restrict__ from = base + src * block_vecs;
  uint4* __restrict__ to = base + dst * block_vecs;
  int64_t i = lo + threadIdx.x;
  for (; i + (kCopyUnroll - 1) * kThreads < hi; i += kCopyUnroll * kThreads) {
    uint4 r[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) r[u] = __ldg(from + i + u * kThreads);
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) to[i + u * kThreads] = r[u];
  }
  for (; i < hi; i += kThreads) to[i] = __ldg(from + i);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace cache
}  // namespace pkv

extern "C" int pkv_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping,
                                     void* k_cache, void* v_cache, int num_tokens,
                                     int num_kv_heads, int head_dim, int block_size,
                                     int64_t num_blocks, int32_t* dev_err, void* stream) {
  using namespace pkv::cache;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(num_kv_heads) * head_dim) % 8 != 0) return PKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  const int64_t row_vecs64 = static_cast<int64_t>(num_kv_heads) * head_dim / 8;
  if (row_vecs64 > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const int row_vecs = static_cast<int>(row_vecs64);
  const int64_t total = static_cast<int64_t>(num_tokens) * row_vecs;
  const int64_t blocks = (total + kThreads - 1) / kThreads;
  if (blocks > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  reshape_and_cache_kernel<<<static_cast<unsigned>(blocks), kThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), total, row_vecs,
      num_blocks * block_size, dev_err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_slot_mapping(const int32_t* block_tables, const int32_t* positions,
                                int num_seqs, int max_blocks_per_seq, int block_size,
                                int64_t num_blocks, int64_t* slot_mapping, int32_t* dev_err,
                                void* stream) {
  using namespace pkv::cache;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!block_tables || !positions || !slot_mapping) return PKV_ERR_INVALID_ARG;
  slot_mapping_kernel<<<(num_seqs + kThreads - 1) / kThreads, kThreads, 0,
                        static_cast<cudaStream_t>(stream)>>>(
      block_tables, positions, num_seqs, max_blocks_per_seq, block_size, num_blocks, slot_mapping,
      dev_err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                               const int64_t* block_pairs, int num_pairs, int64_t block_bytes,
                               int64_t num_blocks, int32_t* dev_err, void* stream) {
  using namespace pkv::cache;
  if (num_layers < 0 || num_pairs < 0 || block_bytes <= 0 || num_blocks <= 0)
    return PKV_ERR_INVALID_ARG;
  if (block_bytes % 16 != 0) return PKV_ERR_INVALID_ARG;
  if (num_layers == 0 || num_pairs == 0) return PKV_OK;
  if (!k_caches || !v_caches || !block_pairs) return PKV_ERR_INVALID_ARG;
  const int64_t block_vecs = block_bytes / 16;
  const int64_t chunks = (block_vecs + kCopyChunkVecs - 1) / kCopyChunkVecs;
  if (static_cast<int64_t>(num_pairs) * chunks > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  for (int base = 0; base < num_layers; base += kMaxLayersPerLaunch) {
    const int n = std::min(kMaxLayersPerLaunch, num_layers - base);
    LayerPtrs ptrs;
    for (int i = 0; i < kMaxLayersPerLaunch; ++i) ptrs.k[i] = ptrs.v[i] = nullptr;
    for (int i = 0; i < n; ++i) {
      void* kp = k_caches[base + i];
      void* vp = v_caches[base + i];
      if (!kp || !vp || !aligned16(kp) || !aligned16(vp)) return PKV_ERR_INVALID_ARG;
      ptrs.k[i] = static_cast<uint4*>(kp);
      ptrs.v[i] = static_cast<uint4*>(vp);
    }
    copy_blocks_kernel<<<dim3(static_cast<unsigned>(num_pairs * chunks), n, 2), kThreads, 0,
                         static_cast<cudaStream_t>(stream)>>>(
        ptrs, block_pairs, block_vecs, static_cast<int>(chunks), num_blocks, dev_err);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// ---- swap_blocks: whole blocks between two pools --------------------------------------
namespace pkv {
namespace cache {

struct PoolPtrs {
  const uint4* src[kMaxLayersPerLaunch];
  uint4* dst[kMaxLayersPerLaunch];
};

// grid (pairs, pools): one CTA copies one block of one pool.  Either side may be
// host memory the GPU can address (pinned and mapped), which makes this the
// device<->host swap of a preempted sequence's blocks.
__global__ void __launch_bounds__(kThreads)
    swap_blocks_kernel(const __grid_constant__ PoolPtrs ptrs, const int64_t* __restrict__ pairs,
                       int64_t block_vecs, int64_t src_num_blocks, int64_t dst_num_blocks,
                       int32_t* dev_err) {
  const int pair = blockIdx.x, pool = blockIdx.y;
  const int64_t src = __ldg(pairs + 2 * pair), dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
    if (threadIdx.x == 0 && pool == 0) report(dev_err, PKV_DEV_BAD_BLOCK_ID);
    return;
  }
  const uint4* __restrict__ from = ptrs.src[pool] + src * block_vecs;
  uint4* __restrict__ to = ptrs.dst[pool] + dst * block_vecs;
  constexpr int kUnroll = 8;
  int64_t i = threadIdx.x;
  for (; i + (kUnroll - 1) * kThreads < block_vecs; i += kUnroll * kThreads) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = from[i + u * kThreads];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) to[i + u * kThreads] = r[u];
  }
  for (; i < block_vecs; i += kThreads) to[i] = from[i];
}

}  // namespace cache
}  // namespace pkv

extern "C" int pkv_swap_blocks(const void* const* src_pools, void* const* dst_pools,
                               int num_pools, const int64_t* block_pairs, int num_pairs,
                               int64_t block_bytes, int64_t src_num_blocks,
                               int64_t dst_num_blocks, int32_t* dev_err, void* stream) {
  using namespace pkv::cache;
  if (num_pools < 0 || num_pairs < 0 || block_bytes <= 0 || src_num_blocks <= 0 ||
      dst_num_blocks <= 0 || block_bytes % 16 != 0)
    return PKV_ERR_INVALID_ARG;
  if (num_pools == 0 || num_pairs == 0) return PKV_OK;
  if (!src_pools || !dst_pools || !block_pairs) return PKV_ERR_INVALID_ARG;
  for (int base = 0; base < num_pools; base += kMaxLayersPerLaunch) {
    const int n = std::min(kMaxLayersPerLaunch, num_pools - base);
    PoolPtrs ptrs;
    for (int i = 0; i < kMaxLayersPerLaunch; ++i) {
      ptrs.src[i] = nullptr;
      ptrs.dst[i] = nullptr;
    }
    for (int i = 0; i < n; ++i) {
      const void* sp = src_pools[base + i];
      void* dp = dst_pools[base + i];
      if (!sp || !dp || !aligned16(sp) || !aligned16(dp)) return PKV_ERR_INVALID_ARG;
      ptrs.src[i] = static_cast<const uint4*>(sp);
      ptrs.dst[i] = static_cast<uint4*>(dp);
    }
    swap_blocks_kernel<<<dim3(num_pairs, n), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        ptrs, block_pairs, block_bytes / 16, src_num_blocks, dst_num_blocks, dev_err);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

// ---- self-test of the bounded wait ------------------------------------------------
namespace pkv {
namespace cache {

// One thread waits on an mbarrier that nothing arrives on: the wait must give up
// after limit_ns, report PKV_DEV_WAIT_TIMEOUT and return (no hang, no trap).
__global__ void bounded_wait_selftest_kernel(int32_t* dev_err, uint64_t limit_ns,
                                             int32_t* landed) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  *landed = mbar_wait_bounded(&bar, 0, dev_err, limit_ns) ? 1 : 0;
}

}  // namespace cache
}  // namespace pkv

extern "C" int pkv_selftest_bounded_wait(int32_t* dev_err, int32_t* landed, int limit_ms,
                                         void* stream) {
  if (!dev_err || !landed || limit_ms <= 0 || limit_ms > 2000) return PKV_ERR_INVALID_ARG;
  pkv::cache::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      dev_err, static_cast<uint64_t>(limit_ms) * 1000000ull, landed);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
