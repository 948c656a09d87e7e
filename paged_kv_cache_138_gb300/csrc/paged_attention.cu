// Paged decode attention for sm_103a.
//
// What it computes ("qaqbuyan: vLLM PagedAttention", `paged_attention`; slot
// rule of "P06 BlockManager"): for every sequence s and query head h,
//   out[s,h] = softmax(scale * q[s,h] . K_s^T) V_s
// over the L = context_lens[s] tokens whose K/V rows sit in physical blocks
// block_tables[s][t / 16], row t % 16.
//
// How (GB300 design, not the pages' sketch):
//  * One CTA per (KV head g, sequence s, split of up to 32 physical blocks).
//    The G = Hq / Hkv query heads that read KV head g are handled together, so
//    every K/V byte is read from HBM once per step.
//  * Each of the 4 warps streams its own blocks of the split (warp w takes
//    blocks w, w+4, ...) through a private 3-stage ring in shared memory.  A
//    stage is one physical block of one KV head: four TMA tiles of 16 rows x
//    64 dims (K lo/hi, V lo/hi), 8 KB, 128-byte swizzled, completion counted on
//    one mbarrier.  Lane 0 refills a stage as soon as the warp is done with it.
//  * QK: lane (t, half) = (lane % 16, lane / 16) dots token t with 64 dims of
//    each of the G queries (q pre-scaled by scale*log2 e, fp32 in smem); one
//    shuffle joins the halves.  Packed fp32x2 FMAs.
//  * Online softmax in base 2 per warp, with a lazy rescale: the running max
//    only moves when a block max exceeds it by more than 8, so most blocks do
//    no rescaling and every weight stays <= 2^8.
//  * PV: lane owns 4 of the 128 output dims for each query, weights broadcast
//    from smem; tokens past L are never multiplied (no 0 * garbage).
//  * The 4 warps' (m, l, o) are merged in smem.  Sequences that need one split
//    write fp16 output directly; longer ones write fp32 partials that a second
//    small kernel merges by log-sum-exp.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "pkv_device.cuh"

namespace pkv {
namespace attn {

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kPartitionBlocks = 32;                    // physical blocks per CTA
constexpr int kHalfTileBytes = kBlockSize * 64 * 2;     // 16 rows x 128 B
constexpr int kStageBytes = 4 * kHalfTileBytes;         // K lo, K hi, V lo, V hi
constexpr float kRescaleThreshold = 8.0f;               // log2 units

struct Smem {
  static constexpr int stages = 0;
  static constexpr int stages_bytes = kWarps * kStages * kStageBytes;
  static constexpr int bars = stages + stages_bytes;                  // u64 [warps][stages]
  static constexpr int ml = bars + kWarps * kStages * 8;              // float [warps][8][2]
  static constexpr int total = ml + kWarps * 8 * 2 * 4;
  static constexpr int alloc = total + 1024;                          // alignment slack
  static_assert(kWarps * 8 * kHeadDim * 4 <= stages_bytes, "merge buffer must fit");
};

struct Params {
  __half* out;
  const __half* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;   // [S, Hq, max_splits, 128]
  float* part_ml;  // [S, Hq, max_splits, 2]  (max, sum) in log2 units
  int32_t* dev_err;
  int64_t num_blocks;
  int num_seqs, num_q_heads, num_kv_heads, max_blocks, max_splits;
  float scale_log2;
};

__device__ __forceinline__ int clamp_context(const Params& p, int s, bool may_report) {
  int L = __ldg(p.context_lens + s);
  const int cap = p.max_blocks * kBlockSize;
  if (L < 0 || L > cap) {
    if (may_report) report(p.dev_err, PKV_DEV_BAD_CONTEXT_LEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

// Shared-memory byte offset of 16-byte chunk c (0..15 over the 128 dims) of
// row `row` in a stage half pair starting at `base` (K: base 0, V: base 2):
// each 64-dim half is a [16 rows x 128 B] TMA box with the 128-byte swizzle
// (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t tile_chunk(uint32_t stage, int base, int row, int c) {
  return stage + (base + (c >> 3)) * kHalfTileBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// One physical block (16 tokens) of one KV head for the G query heads of the
// warp, on the tensor cores.  Rows of the 16-row MMA tile are query heads
// (only the first G are real, the rest are zero), columns are tokens:
//   S = Q K^T  : 8 k-steps over the 128 dims x 2 token halves  (16 MMAs)
//   P = 2^(S * scale * log2 e - m), fp16                        (online softmax)
//   O += P V   : 16 dim tiles of 8                              (16 MMAs)
// Lane layout (m16n8k16): lane holds query row lane / 4; tokens
// 2 * (lane % 4) + {0, 1} (+ 8); output dims 8 * nd + 2 * (lane % 4) + {0, 1}.
__device__ __forceinline__ void process_block(uint32_t st, const uint32_t (&qa)[8][2], int valid,
                                              int lane, float scale_log2, float& m, float& l,
                                              float (&o)[16][4]) {
  constexpr unsigned kFull = 0xffffffffu;
  const int r8 = lane & 7, mi = lane >> 3;
  // ---- S = Q K^T -------------------------------------------------------------
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  const int ktok = r8 + ((mi >> 1) << 3);  // matrices: (t0-7,lo) (t0-7,hi) (t8-15,lo) (t8-15,hi)
#pragma unroll
  for (int kc = 0; kc < 8; ++kc) {
    uint32_t b00, b01, b10, b11;
    ldsm_x4(tile_chunk(st, 0, ktok, 2 * kc + (mi & 1)), b00, b01, b10, b11);
    mma_16816_top(s0, qa[kc][0], qa[kc][1], b00, b01);
    mma_16816_top(s1, qa[kc][0], qa[kc][1], b10, b11);
  }
  // ---- online softmax on this lane's row ------------------------------------------
  const int tq = 2 * (lane & 3);
  const float x0 = tq < valid ? s0[0] * scale_log2 : -INFINITY;
  const float x1 = tq + 1 < valid ? s0[1] * scale_log2 : -INFINITY;
  const float x2 = tq + 8 < valid ? s1[0] * scale_log2 : -INFINITY;
  const float x3 = tq + 9 < valid ? s1[1] * scale_log2 : -INFINITY;
  float bm = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
  bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
  if (bm > m + kRescaleThreshold) {  // the 4 lanes of a row agree
    const float alpha = exp2_approx(m - bm);
    l *= alpha;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      o[nd][0] *= alpha;
      o[nd][1] *= alpha;
    }
    m = bm;
  }
  const float p0 = exp2_approx(x0 - m), p1 = exp2_approx(x1 - m);
  const float p2 = exp2_approx(x2 - m), p3 = exp2_approx(x3 - m);
  l += (p0 + p1) + (p2 + p3);
  const uint32_t pa0 = pack_half2(p0, p1), pa2 = pack_half2(p2, p3);
  // ---- rows past the context may hold anything (NaN): zero them, as 0 * NaN
  // would poison the sums -------------------------------------------------------------
  if (valid < kBlockSize) {
    const int n = (kBlockSize - valid) * 16;  // 16-byte chunks to clear
    for (int i = lane; i < n; i += 32) {
      const int row = valid + (i >> 4), c = i & 15;
      st_shared_zero16(st + (2 + (c >> 3)) * kHalfTileBytes + row * 128 + ((c & 7) << 4));
    }
    fence_proxy_async_smem();
    __syncwarp();
  }
  // ---- O += P V ----------------------------------------------------------------------
  const int vtok = r8 + ((mi & 1) << 3);  // matrices: (t0-7,c) (t8-15,c) (t0-7,c+1) (t8-15,c+1)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t v0, v1, v2, v3;
    ldsm_x4_trans(tile_chunk(st, 2, vtok, 2 * j + (mi >> 1)), v0, v1, v2, v3);
    mma_16816_top(o[2 * j], pa0, pa2, v0, v1);
    mma_16816_top(o[2 * j + 1], pa0, pa2, v2, v3);
  }
}

template <int G>
__global__ void __launch_bounds__(kThreads, 2)
    paged_attention_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                 const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  static_assert(G >= 1 && G <= 8, "query rows of the MMA tile");
  constexpr unsigned kFull = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int g = blockIdx.x, s = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads;
  const int h0 = g * G;

  const int L = clamp_context(p, s, threadIdx.x == 0 && g == 0 && split == 0);
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int nsplit = (nblk + kPartitionBlocks - 1) / kPartitionBlocks;
  if (L == 0) {
    if (split == 0) {
      __half* o = p.out + (static_cast<int64_t>(s) * Hq + h0) * kHeadDim;
      for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) o[i] = __float2half_rn(0.f);
    }
    return;
  }
  const int blk_begin = split * kPartitionBlocks;
  if (blk_begin >= nblk) return;
  const int n_here = min(kPartitionBlocks, nblk - blk_begin);
  // warp w streams local blocks w, w + 4, ...; lane j holds the id of its j-th
  const int my_count = warp < n_here ? (n_here - warp + kWarps - 1) / kWarps : 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars) + warp * kStages;
  const uint32_t ring = smem_u32(smem + Smem::stages + warp * kStages * kStageBytes);

  int32_t my_id = -1;
  if (lane < my_count) {
    my_id = __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks + blk_begin + warp +
                  lane * kWarps);
    if (my_id < 0 || my_id >= p.num_blocks) {
      report(p.dev_err, PKV_DEV_BAD_BLOCK_ID);
      my_id = -1;
    }
  }
  if (lane == 0) {
    if (warp == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
    }
    for (int j = 0; j < kStages; ++j) mbar_init(&bars[j], 1);
    fence_barrier_init();
  }
  __syncwarp();

  auto issue = [&](int k, int32_t b) {  // lane 0 only: local block k, physical id b
    uint64_t* bar = &bars[k % kStages];
    uint8_t* st = smem + Smem::stages + (warp * kStages + k % kStages) * kStageBytes;
    if (b < 0) {  // reported already: complete the phase without data
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, kStageBytes);
    const int row = b * kBlockSize;
    tma_load_3d(st, &tmap_k, 0, g, row, bar);
    tma_load_3d(st + kHalfTileBytes, &tmap_k, 64, g, row, bar);
    tma_load_3d(st + 2 * kHalfTileBytes, &tmap_v, 0, g, row, bar);
    tma_load_3d(st + 3 * kHalfTileBytes, &tmap_v, 64, g, row, bar);
  };

  int issued = min(kStages, my_count);
#pragma unroll
  for (int k = 0; k < kStages; ++k) {
    const int32_t b = __shfl_sync(kFull, my_id, k);
    if (lane == 0 && k < issued) issue(k, b);
  }

  // q of this lane's row as m16n8k16 A fragments (raw fp16; scale applied to S)
  uint32_t qa[8][2];
  const int qrow = lane >> 2;
  if (qrow < G) {
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(
        p.q + (static_cast<int64_t>(s) * Hq + h0 + qrow) * kHeadDim);
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      qa[kc][0] = __ldg(qp + 8 * kc + (lane & 3));
      qa[kc][1] = __ldg(qp + 8 * kc + 4 + (lane & 3));
    }
  } else {
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) qa[kc][0] = qa[kc][1] = 0u;
  }

  float m = -INFINITY, l = 0.f;
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  bool ok = true;
  for (int k = 0; k < issued; ++k) {
    const int stage = k % kStages;
    const bool landed = mbar_wait_bounded(&bars[stage], (k / kStages) & 1, p.dev_err);
    ok = __all_sync(kFull, ok && landed) != 0;
    const int32_t b = __shfl_sync(kFull, my_id, k);
    if (ok && b >= 0) {
      const int valid = min(kBlockSize, L - (blk_begin + warp + k * kWarps) * kBlockSize);
      process_block(ring + stage * kStageBytes, qa, valid, lane, p.scale_log2, m, l, o);
    }
    __syncwarp();
    const int32_t nb = __shfl_sync(kFull, my_id, issued < 32 ? issued : 0);
    if (ok && issued < my_count) {
      if (lane == 0) issue(issued, nb);
      ++issued;
    }
  }
  l += __shfl_xor_sync(kFull, l, 1);
  l += __shfl_xor_sync(kFull, l, 2);

  // ---- merge the 4 warps' partial softmax states ------------------------------
  __syncthreads();  // every issued tile has landed (or timed out); ring is free
  float* ml = reinterpret_cast<float*>(smem + Smem::ml);
  float* ob = reinterpret_cast<float*>(smem + Smem::stages);
  if (qrow < G) {
    if ((lane & 3) == 0) {
      ml[(warp * 8 + qrow) * 2] = m;
      ml[(warp * 8 + qrow) * 2 + 1] = l;
    }
    float* orow = ob + (warp * 8 + qrow) * kHeadDim + 2 * (lane & 3);
#pragma unroll
    for (int nd = 0; nd < 16; ++nd)
      *reinterpret_cast<float2*>(orow + nd * 8) = make_float2(o[nd][0], o[nd][1]);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * kHeadDim; e += kThreads) {
    const int gi = e / kHeadDim, d = e % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[(w * 8 + gi) * 2]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float c = exp2_approx(ml[(w * 8 + gi) * 2] - M);
        num += c * ob[(w * 8 + gi) * kHeadDim + d];
        den += c * ml[(w * 8 + gi) * 2 + 1];
      }
    }
    const int64_t row = static_cast<int64_t>(s) * Hq + h0 + gi;
    if (nsplit == 1) {
      p.out[row * kHeadDim + d] = __float2half_rn(den > 0.f ? num / den : 0.f);
    } else {
      const int64_t slot = row * p.max_splits + split;
      p.part_o[slot * kHeadDim + d] = num;
      if (d == 0) {
        p.part_ml[slot * 2] = M;
        p.part_ml[slot * 2 + 1] = den;
      }
    }
  }
}

// Log-sum-exp merge of the splits of one (sequence, query head); 128 threads,
// one output dim each.  Rows that needed a single split were written directly.
__global__ void __launch_bounds__(kHeadDim)
    paged_attention_merge_kernel(const Params p) {
  const int h = blockIdx.x, s = blockIdx.y, d = threadIdx.x;
  const int L = clamp_context(p, s, false);
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int nsplit = (nblk + kPartitionBlocks - 1) / kPartitionBlocks;
  if (nsplit <= 1) return;
  const int64_t row = static_cast<int64_t>(s) * p.num_q_heads + h;
  const float* ml = p.part_ml + row * p.max_splits * 2;
  const float* po = p.part_o + row * p.max_splits * kHeadDim;
  float M = -INFINITY;
  for (int i = 0; i < nsplit; ++i) M = fmaxf(M, ml[2 * i]);
  float num = 0.f, den = 0.f;
  if (M != -INFINITY) {
    for (int i = 0; i < nsplit; ++i) {
      const float c = exp2_approx(ml[2 * i] - M);
      num += c * po[i * kHeadDim + d];
      den += c * ml[2 * i + 1];
    }
  }
  p.out[row * kHeadDim + d] = __float2half_rn(den > 0.f ? num / den : 0.f);
}

// ---- host side ------------------------------------------------------------------

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

// The cache [num_blocks * 16 rows, Hkv, 128] as a 3-D tensor; a box is 16 rows
// x 1 head x 64 dims (128 B inner extent, 128-byte swizzle).
bool make_cache_map(CUtensorMap* map, const void* base, int num_kv_heads, int64_t num_blocks) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(num_kv_heads),
                        static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                           static_cast<cuuint64_t>(num_kv_heads) * kHeadDim * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBlockSize)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int max_splits_for(int max_blocks) { return (max_blocks + kPartitionBlocks - 1) / kPartitionBlocks; }

template <int G>
int launch(const CUtensorMap& mk, const CUtensorMap& mv, const Params& p, cudaStream_t stream) {
  // The shared-memory opt-in is per device; remember it for up to 64 devices.
  static std::atomic<uint8_t> opted_in[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(paged_attention_split_kernel<G>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem::alloc) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev >= 0 && dev < 64) opted_in[dev].store(1, std::memory_order_release);
  }
  dim3 grid(p.num_kv_heads, p.num_seqs, p.max_splits);
  paged_attention_split_kernel<G><<<grid, kThreads, Smem::alloc, stream>>>(mk, mv, p);
  if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  if (p.max_splits > 1) {
    paged_attention_merge_kernel<<<dim3(p.num_q_heads, p.num_seqs), kHeadDim, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
  }
  return PKV_OK;
}

}  // namespace attn
}  // namespace pkv

extern "C" size_t pkv_paged_attention_workspace_bytes(int num_seqs, int num_q_heads,
                                                      int max_blocks_per_seq, int head_dim) {
  using namespace pkv::attn;
  if (num_seqs <= 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || head_dim != kHeadDim)
    return 0;
  const int splits = max_splits_for(max_blocks_per_seq);
  if (splits <= 1) return 0;
  return static_cast<size_t>(num_seqs) * num_q_heads * splits * (kHeadDim + 2) * sizeof(float);
}

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int64_t num_blocks,
                                          int max_blocks_per_seq, float scale, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_err,
                                          void* stream) {
  using namespace pkv::attn;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PKV_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return PKV_ERR_INVALID_ARG;
  if (num_blocks > INT32_MAX / kBlockSize || num_seqs > 65535 || num_kv_heads > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * kBlockSize > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const size_t need = pkv_paged_attention_workspace_bytes(num_seqs, num_q_heads,
                                                          max_blocks_per_seq, head_dim);
  if (need > 0 && (!workspace || workspace_bytes < need)) return PKV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 15) return PKV_ERR_INVALID_ARG;

  Params p;
  p.out = static_cast<__half*>(out);
  p.q = static_cast<const __half*>(q);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.max_splits = max_splits_for(max_blocks_per_seq);
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = need ? p.part_o + static_cast<size_t>(num_seqs) * num_q_heads * p.max_splits *
                                    kHeadDim
                   : nullptr;
  p.dev_err = dev_err;
  p.num_blocks = num_blocks;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.scale_log2 = scale * 1.4426950408889634f;

  CUtensorMap mk, mv;
  if (!make_cache_map(&mk, k_cache, num_kv_heads, num_blocks) ||
      !make_cache_map(&mv, v_cache, num_kv_heads, num_blocks))
    return PKV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (G) {
    case 1: return launch<1>(mk, mv, p, st);
    case 2: return launch<2>(mk, mv, p, st);
    case 4: return launch<4>(mk, mv, p, st);
    default: return launch<8>(mk, mv, p, st);
  }
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

// Device address of g_static_scratch on the current device, looked up once per
// device (host code may not use the symbol itself as a device pointer).
void* static_scratch_ptr() {
  static std::atomic<void*> ptrs[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  void* p = ptrs[dev].load(std::memory_order_acquire);
  if (p) return p;
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
                                                          max_blocks_per_seq, head_dim);
  if (need > kStaticScratchBytes) return PKV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = static_scratch_ptr();
    if (!scratch) return PKV_ERR_CUDA;
  }
  return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                                    num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                    num_blocks, max_blocks_per_seq, scale, scratch,
                                    need > 0 ? kStaticScratchBytes : 0, dev_err, stream);
}
