// Paged decode attention: host entry points and the split merge kernel.
// The split kernel itself (design notes included) is attention_kernel.cuh,
// instantiated per block size in attention_bs*.cu.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "attention_kernel.cuh"

namespace pkv {
namespace attn {

// Log-sum-exp merge of the splits of each (sequence, query head) row: one
// warp per row, kMergeRows rows per CTA; lane i reads split i's (m, l) (32 at
// a time) for the maximum, then every lane accumulates dims 4 i .. 4 i + 3 of
// the weighted partials with float4 loads.  Rows whose only split wrote the
// output directly are skipped.
constexpr int kMergeRows = 8;

__global__ void __launch_bounds__(kMergeRows * 32) paged_attention_merge_kernel(const Params p) {
  // a programmatically dependent launch that follows (the attention kernel)
  // may place its CTAs while this grid runs; it reads nothing before this
  // grid has completed
  asm volatile("griddepcontrol.launch_dependents;");
  // launched as a programmatic dependent of the attention kernel: CTAs may be
  // resident before it finishes; wait here until its writes are visible (a
  // no-op for an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeRows + (threadIdx.x >> 5);
  if (row >= static_cast<int64_t>(p.num_seqs) * p.num_q_heads) return;
  const int s = static_cast<int>(row / p.num_q_heads);
  int L = __ldg(p.context_lens + s);
  const int cap = p.max_blocks * p.block_size;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int ntiles = (L + kTile - 1) / kTile;
  const int own_begin = min(shared_tiles_of(p, s), ntiles);
  const int shared_splits = shared_slots_of(p, own_begin);
  const int nsplit = shared_splits + splits_for_tiles(p, ntiles - own_begin);
  if (nsplit == 0 || (nsplit == 1 && shared_splits == 0)) return;
  const float* ml = p.part_ml + row * p.max_splits * 2;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + row * p.max_splits * kHeadDim);
  float M = -INFINITY;
  for (int i = lane; i < nsplit; i += 32) M = fmaxf(M, ml[2 * i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int i = 0; i < nsplit; ++i) {
      const float c = exp2_approx(ml[2 * i] - M);
      const float4 v = po[i * (kHeadDim / 4) + lane];
      num.x += c * v.x;
      num.y += c * v.y;
      num.z += c * v.z;
      num.w += c * v.w;
      den += c * ml[2 * i + 1];
    }
  }
  store_out4(p.out + row * kHeadDim + 4 * lane, den, num);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// The cache [num_blocks * BS rows, Hkv, 128] as a 3-D tensor; a box is
// min(BS, 16) rows x 1 head x 64 dims (128 B inner extent, 128-byte swizzle).
bool make_cache_map(CUtensorMap* map, const void* base, int num_kv_heads, int64_t num_blocks,
                    int block_size) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(num_kv_heads),
                        static_cast<cuuint64_t>(num_blocks) * block_size};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                           static_cast<cuuint64_t>(num_kv_heads) * kHeadDim * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(block_size < kTile ? block_size : kTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool supported_block_size(int bs) { return bs == 8 || bs == 16 || bs == 32 || bs == 64; }

// Stride of the split grid's sequence order: the first value coprime with S
// at or above 0.618 S (1 for S <= 2), so that y -> y * stride % S permutes the
// sequences and batch neighbours land far apart.
int seq_stride_for(int num_seqs) {
  if (num_seqs <= 2) return 1;
  auto gcd = [](int a, int b) {
    while (b) {
      const int t = a % b;
      a = b;
      b = t;
    }
    return a;
  };
  int k = static_cast<int>(0.618 * num_seqs);
  if (k < 1) k = 1;
  while (gcd(k, num_seqs) != 1) ++k;
  return k;
}

// Shared validation + launch of both entry points.
struct Groups {
  const int32_t* first = nullptr;
  const int32_t* seq_group = nullptr;
  const int32_t* shared = nullptr;
  int num_groups = 0;
  int max_shared_tokens = 0;
  int max_own_tokens = 0;  // longest stretch past a group's shared prefix
};

int decode(void* out, const void* q, const void* k_new, const void* v_new, const void* k_cache,
           const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
           int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
           int64_t num_blocks, int max_blocks_per_seq, float scale, void* workspace,
           size_t workspace_bytes, int32_t* dev_err, void* stream, bool fused,
           const Groups& groups = Groups(), const int32_t* cow_block = nullptr,
           const int32_t* cow_src = nullptr) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || !supported_block_size(block_size)) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_INVALID_ARG;
  if (fused && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
  if ((cow_block != nullptr) != (cow_src != nullptr) || (cow_block && !fused))
    return PKV_ERR_INVALID_ARG;
  const uintptr_t align = reinterpret_cast<uintptr_t>(k_cache) |
                          reinterpret_cast<uintptr_t>(v_cache) |
                          reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new);
  if ((align & 15) || (reinterpret_cast<uintptr_t>(q) & 3)) return PKV_ERR_INVALID_ARG;
  if (num_blocks > INT32_MAX / block_size || num_seqs > 65535 || num_kv_heads > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const bool grouped = groups.first != nullptr;
  if (grouped) {
    if (!groups.seq_group || !groups.shared || groups.num_groups <= 0 ||
        groups.num_groups > 65535 || groups.max_shared_tokens < 0 ||
        groups.max_own_tokens < 0)
      return PKV_ERR_INVALID_ARG;
    if (groups.max_shared_tokens % kTile || groups.max_shared_tokens % block_size)
      return PKV_ERR_INVALID_ARG;
  }
  const size_t need =
      grouped ? pkv_paged_attention_grouped_workspace_bytes(num_seqs, num_q_heads,
                                                            max_blocks_per_seq, block_size,
                                                            head_dim, groups.max_shared_tokens)
              : pkv_paged_attention_workspace_bytes(num_seqs, num_q_heads, max_blocks_per_seq,
                                                    block_size, head_dim);
  if (need > 0 && (!workspace || workspace_bytes < need)) return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 15) return PKV_ERR_INVALID_ARG;
  // split length of this launch (the workspace bound assumes the shortest)
  const int partition =
      partition_tiles_for(num_seqs, num_kv_heads, max_blocks_per_seq, block_size);
  const int own_splits = max_splits_for(max_blocks_per_seq, block_size, partition);
  const int shared_splits =
      grouped ? (tiles_for_tokens(groups.max_shared_tokens) + partition - 1) / partition : 0;

  Params p;
  p.out = static_cast<__half*>(out);
  p.q = static_cast<const __half*>(q);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.max_splits = own_splits + shared_splits;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = need ? p.part_o + static_cast<size_t>(num_seqs) * num_q_heads * p.max_splits *
                                    kHeadDim
                   : nullptr;
  p.dev_err = dev_err;
  p.k_new = static_cast<const __half*>(k_new);
  p.v_new = static_cast<const __half*>(v_new);
  p.k_cache = static_cast<__half*>(const_cast<void*>(k_cache));
  p.v_cache = static_cast<__half*>(const_cast<void*>(v_cache));
  p.num_blocks = num_blocks;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.block_size = block_size;
  p.seq_group = grouped ? groups.seq_group : nullptr;
  p.group_first = groups.first;
  p.group_shared = groups.shared;
  p.cow_block = cow_block;
  p.cow_src = cow_src;
  p.num_groups = groups.num_groups;
  p.own_tiles_cap = (tiles_for_tokens(groups.max_own_tokens) + partition - 1) / partition *
                    partition;
  p.shared_splits_cap = shared_splits;
  p.seq_stride = seq_stride_for(num_seqs);
  {
    // the last split plane is visited in zigzag order of length when its
    // units can reach half a split (shorter remainders do not shape the tail)
    const int64_t table_tiles =
        tiles_for_tokens(static_cast<int64_t>(max_blocks_per_seq) * block_size);
    const int64_t last_plane_tiles =
        table_tiles - static_cast<int64_t>(own_splits - 1) * partition;
    p.rank_by_length = num_seqs <= kMaxRankedSeqs && 2 * last_plane_tiles >= partition;
  }
  p.partition_tiles = partition;
  p.scale_log2 = scale * 1.4426950408889634f;

  CUtensorMap mk, mv;
  if (!make_cache_map(&mk, k_cache, num_kv_heads, num_blocks, block_size) ||
      !make_cache_map(&mv, v_cache, num_kv_heads, num_blocks, block_size))
    return PKV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PKV_OK;
  if (grouped) {
    // own units: sequences never run past max_own_tokens beyond their shared
    // prefix (a sequence outside any group counts all its tokens as its own)
    const int own = (tiles_for_tokens(groups.max_own_tokens) + partition - 1) / partition;
    // spread the shared units over the first half of the grid when own units
    // are at most half as long (measured on forked samples: +3 %); else first
    const int64_t n_shared = static_cast<int64_t>(num_kv_heads) * groups.num_groups * shared_splits;
    const int64_t n_total = n_shared + static_cast<int64_t>(num_kv_heads) * num_seqs * own;
    int stride = 1;
    if (n_shared > 0 && 2 * static_cast<int64_t>(groups.max_own_tokens) <= groups.max_shared_tokens)
      stride = static_cast<int>(std::max<int64_t>(1, n_total / 2 / n_shared));
    switch (block_size) {
      case 8: rc = launch_grouped_step<8>(G, fused, mk, mv, p, shared_splits, own, stride, st); break;
      case 16:
        rc = launch_grouped_step<16>(G, fused, mk, mv, p, shared_splits, own, stride, st);
        break;
      case 32:
        rc = launch_grouped_step<32>(G, fused, mk, mv, p, shared_splits, own, stride, st);
        break;
      default:
        rc = launch_grouped_step<64>(G, fused, mk, mv, p, shared_splits, own, stride, st);
        break;
    }
  } else {
    switch (block_size) {
      case 8: rc = launch_split<8>(G, fused, mk, mv, p, own_splits, st); break;
      case 16: rc = launch_split<16>(G, fused, mk, mv, p, own_splits, st); break;
      case 32: rc = launch_split<32>(G, fused, mk, mv, p, own_splits, st); break;
      default: rc = launch_split<64>(G, fused, mk, mv, p, own_splits, st); break;
    }
  }
  if (rc != PKV_OK) return rc;
  if (p.max_splits > 1) {
    // programmatic dependent launch: the merge grid is scheduled while the
    // attention kernel's last CTAs run and starts the moment it completes
    const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.num_q_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + kMergeRows - 1) / kMergeRows));
    cfg.blockDim = dim3(kMergeRows * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, paged_attention_merge_kernel, p) != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace attn
}  // namespace pkv

extern "C" size_t pkv_paged_attention_workspace_bytes(int num_seqs, int num_q_heads,
                                                      int max_blocks_per_seq, int block_size,
                                                      int head_dim) {
  using namespace pkv::attn;
  if (num_seqs <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
      head_dim != kHeadDim)
    return 0;
  const int splits = max_splits_for(max_blocks_per_seq, block_size);
  if (splits <= 1) return 0;
  return static_cast<size_t>(num_seqs) * num_q_heads * splits * (kHeadDim + 2) * sizeof(float);
}

extern "C" int pkv_paged_attention_split_tokens(int num_seqs, int num_kv_heads,
                                                int max_blocks_per_seq, int block_size) {
  using namespace pkv::attn;
  if (num_seqs <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
      !supported_block_size(block_size))
    return PKV_ERR_INVALID_ARG;
  return partition_tiles_for(num_seqs, num_kv_heads, max_blocks_per_seq, block_size) * kTile;
}

extern "C" size_t pkv_paged_attention_grouped_workspace_bytes(int num_seqs, int num_q_heads,
                                                              int max_blocks_per_seq,
                                                              int block_size, int head_dim,
                                                              int max_shared_tokens) {
  using namespace pkv::attn;
  if (num_seqs <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
      head_dim != kHeadDim || max_shared_tokens < 0)
    return 0;
  const int splits = max_splits_for(max_blocks_per_seq, block_size) +
                     (tiles_for_tokens(max_shared_tokens) + kPartitionTiles - 1) / kPartitionTiles;
  return static_cast<size_t>(num_seqs) * num_q_heads * splits * (kHeadDim + 2) * sizeof(float);
}

extern "C" int pkv_paged_attention_decode_grouped(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* group_first,
    const int32_t* seq_group, const int32_t* group_shared, int num_groups, int max_shared_tokens,
    int max_own_tokens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int64_t num_blocks, int max_blocks_per_seq, float scale, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* stream) {
  pkv::attn::Groups gr;
  gr.first = group_first;
  gr.seq_group = seq_group;
  gr.shared = group_shared;
  gr.num_groups = num_groups;
  gr.max_shared_tokens = max_shared_tokens;
  gr.max_own_tokens = max_own_tokens;
  if (!group_first) return PKV_ERR_INVALID_ARG;
  return pkv::attn::decode(out, q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                           max_blocks_per_seq, scale, workspace, workspace_bytes, dev_err, stream,
                           false, gr);
}

extern "C" int pkv_paged_attention_decode_grouped_fused(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
    void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    const int32_t* group_first, const int32_t* seq_group, const int32_t* group_shared,
    int num_groups, int max_shared_tokens, int max_own_tokens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int max_blocks_per_seq,
    float scale, void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  pkv::attn::Groups gr;
  gr.first = group_first;
  gr.seq_group = seq_group;
  gr.shared = group_shared;
  gr.num_groups = num_groups;
  gr.max_shared_tokens = max_shared_tokens;
  gr.max_own_tokens = max_own_tokens;
  if (!group_first) return PKV_ERR_INVALID_ARG;
  return pkv::attn::decode(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                           max_blocks_per_seq, scale, workspace, workspace_bytes, dev_err, stream,
                           true, gr);
}

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int64_t num_blocks,
                                          int max_blocks_per_seq, float scale, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_err,
                                          void* stream) {
  return pkv::attn::decode(out, q, nullptr, nullptr, k_cache, v_cache, block_tables, context_lens,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                           max_blocks_per_seq, scale, workspace, workspace_bytes, dev_err, stream,
                           false);
}

extern "C" int pkv_paged_attention_decode_fused(void* out, const void* q, const void* k_new,
                                                const void* v_new, void* k_cache, void* v_cache,
                                                const int32_t* block_tables,
                                                const int32_t* context_lens, int num_seqs,
                                                int num_q_heads, int num_kv_heads, int head_dim,
                                                int block_size, int64_t num_blocks,
                                                int max_blocks_per_seq, float scale,
                                                void* workspace, size_t workspace_bytes,
                                                int32_t* dev_err, void* stream) {
  return pkv::attn::decode(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                           max_blocks_per_seq, scale, workspace, workspace_bytes, dev_err, stream,
                           true);
}

extern "C" int pkv_paged_attention_decode_fused_cow(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, const int32_t* cow_block,
    const int32_t* cow_src, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, int max_blocks_per_seq, float scale, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!cow_block || !cow_src) return PKV_ERR_INVALID_ARG;
  return pkv::attn::decode(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                           max_blocks_per_seq, scale, workspace, workspace_bytes, dev_err, stream,
                           true, pkv::attn::Groups(), cow_block, cow_src);
}

extern "C" int pkv_paged_attention_decode_grouped_fused_cow(
    void* out, const void* q, const void* k_new, const void* v_new, void* k_cache,
    void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
    const int32_t* group_first, const int32_t* seq_group, const int32_t* group_shared,
    int num_groups, int max_shared_tokens, int max_own_tokens, const int32_t* cow_block,
    const int32_t* cow_src, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, int max_blocks_per_seq, float scale, void* workspace,
    size_t workspace_bytes, int32_t* dev_err, void* stream) {
  pkv::attn::Groups gr;
  gr.first = group_first;
  gr.seq_group = seq_group;
  gr.shared = group_shared;
  gr.num_groups = num_groups;
  gr.max_shared_tokens = max_shared_tokens;
  gr.max_own_tokens = max_own_tokens;
  if (!group_first || !cow_block || !cow_src) return PKV_ERR_INVALID_ARG;
  return pkv::attn::decode(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                           num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                           max_blocks_per_seq, scale, workspace, workspace_bytes, dev_err, stream,
                           true, gr, cow_block, cow_src);
}

// ---- allocation-free variant ------------------------------------------------------
// Some callers cannot call cudaMalloc or any allocating routine: a plugin whose
// host framework owns all device memory and hands out none, or code on a
// latency-critical path where an allocation's implicit device synchronisation
// is not acceptable.  For them the split partials live in a fixed scratch
// array in this module's device memory instead of a caller workspace.
namespace pkv {
namespace attn {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device

// Held by every device that loads this library, until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch in the current context.  It is looked up
// again on every call made outside stream capture (the lookup allocates
// nothing), so a context created anew on the device -- after
// cudaDeviceReset, or another driver context made current -- gets the
// array's address in that context, not a stale one.  A call made while its
// stream is being captured uses the address the device's last uncaptured
// call found (the first call on a device must therefore come before any
// capture).
void* static_scratch_ptr(cudaStream_t stream) {
  static std::atomic<void*> ptrs[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return nullptr;
  if (cap != cudaStreamCaptureStatusNone) return ptrs[dev].load(std::memory_order_acquire);
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
  ptrs[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace attn
}  // namespace pkv

extern "C" int pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                                  const void* v_cache,
                                                  const int32_t* block_tables,
                                                  const int32_t* context_lens, int num_seqs,
                                                  int num_q_heads, int num_kv_heads, int head_dim,
                                                  int block_size, int64_t num_blocks,
                                                  int max_blocks_per_seq, float scale,
                                                  int32_t* dev_err, void* stream) {
  using namespace pkv::attn;
  const size_t need = pkv_paged_attention_workspace_bytes(num_seqs, num_q_heads,
                                                          max_blocks_per_seq, block_size,
                                                          head_dim);
  if (need > kStaticScratchBytes) return PKV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = static_scratch_ptr(static_cast<cudaStream_t>(stream));
    if (!scratch) return PKV_ERR_CUDA;
  }
  return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                                    num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                    num_blocks, max_blocks_per_seq, scale, scratch,
                                    need > 0 ? kStaticScratchBytes : 0, dev_err, stream);
}
