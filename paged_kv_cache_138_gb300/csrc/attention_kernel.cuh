// Paged decode attention kernels for sm_103a (template; instantiated per block
// size in attention_bs*.cu).
//
// What it computes ("qaqbuyan: vLLM PagedAttention", `paged_attention`; slot
// rule of "P06 BlockManager"): for every sequence s and query head h,
//   out[s,h] = softmax(scale * q[s,h] . K_s^T) V_s
// over the L = context_lens[s] tokens; token t's K/V row is row t % BS of
// physical block block_tables[s][t / BS].
//
// How (GB300 design, not the pages' sketch):
//  * The unit of work is a 16-token tile.  One CTA per (KV head g, sequence s,
//    split of up to 32 tiles = 512 tokens).  The G = Hq / Hkv query heads that
//    read KV head g are handled together, so every K/V byte leaves HBM once.
//  * Each of the 4 warps streams its own tiles of the split (warp w takes tiles
//    w, w+4, ...) through a private 3-stage ring in shared memory.  A stage is
//    one tile of one KV head: K and V, each as two 64-dim TMA boxes (128-byte
//    swizzle), 8 KB, completion counted on one mbarrier with a bounded wait.
//    A tile is a 16-row window of a block (BS >= 16) or two 8-row blocks
//    (BS = 8); lane 0 refills a stage as soon as the warp is done with it.
//  * Per tile, S = Q K^T and O += P V run on mma.sync m16n8k16 fragments read
//    with ldmatrix from the swizzled tiles (query heads are the MMA rows).
//  * Online softmax in base 2 per query row with a lazy rescale: the running
//    max only moves when a tile max exceeds it by more than 8, so most tiles
//    skip rescaling and every weight stays <= 2^8 (exact in fp16 range).
//  * The 4 warps' (m, l, o) are merged in shared memory.  Sequences that need
//    one split write fp16 output directly; longer ones write fp32 partials that
//    a second small kernel merges by log-sum-exp.
//  * FUSED: the CTA that holds the sequence's last tile also performs the
//    cache write of the new token (position L - 1): it stores k_new/v_new at
//    their slot and patches the same row of its staged tile, so one launch per
//    layer replaces reshape_and_cache + attention.
#pragma once

#include <cuda.h>

#include <atomic>

#include "pkv_device.cuh"

namespace pkv {
namespace attn {

constexpr int kHeadDim = 128;
constexpr int kTile = 16;                          // tokens per stage
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;
constexpr int kPartitionTiles = 32;                // tiles per CTA split (512 tokens)
constexpr int kHalfTileBytes = kTile * 64 * 2;     // 16 rows x 128 B
constexpr int kStageBytes = 4 * kHalfTileBytes;    // K lo, K hi, V lo, V hi
constexpr float kRescaleThreshold = 8.0f;          // log2 units

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
  // fused cache write (FUSED kernels only)
  const __half* k_new;  // [S, Hkv, 128]
  const __half* v_new;
  __half* k_cache;      // [num_blocks, BS, Hkv, 128]
  __half* v_cache;
  int64_t num_blocks;
  int num_seqs, num_q_heads, num_kv_heads, max_blocks, max_splits, block_size;
  float scale_log2;
};

inline int tiles_for_tokens(int64_t tokens) { return static_cast<int>((tokens + kTile - 1) / kTile); }
inline int max_splits_for(int max_blocks, int block_size) {
  const int tiles = tiles_for_tokens(static_cast<int64_t>(max_blocks) * block_size);
  return (tiles + kPartitionTiles - 1) / kPartitionTiles;
}

template <int BS>
__device__ __forceinline__ int clamp_context(const Params& p, int s, bool may_report) {
  int L = __ldg(p.context_lens + s);
  const int cap = p.max_blocks * BS;
  if (L < 0 || L > cap) {
    if (may_report) report(p.dev_err, PKV_DEV_BAD_CONTEXT_LEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

// Shared-memory address of 16-byte chunk c (0..15 over the 128 dims) of row
// `row` of a stage: K at base 0, V at base 2; each 64-dim half is a
// [16 rows x 128 B] box with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t tile_chunk(uint32_t stage, int base, int row, int c) {
  return stage + (base + (c >> 3)) * kHalfTileBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// One 16-token tile of one KV head for the G query heads of the warp, on the
// tensor cores.  Rows of the 16-row MMA tile are query heads (only the first G
// are real, the rest are zero), columns are tokens:
//   S = Q K^T  : 8 k-steps over the 128 dims x 2 token halves  (16 MMAs)
//   P = 2^(S * scale * log2 e - m), fp16                        (online softmax)
//   O += P V   : 16 dim tiles of 8                              (16 MMAs)
// Lane layout (m16n8k16): lane holds query row lane / 4; tokens
// 2 * (lane % 4) + {0, 1} (+ 8); output dims 8 * nd + 2 * (lane % 4) + {0, 1}.
__device__ __forceinline__ void process_tile(uint32_t st, const uint32_t (&qa)[8][2], int valid,
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
  if (valid < kTile) {
    const int n = (kTile - valid) * 16;  // 16-byte chunks to clear
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

// Physical block ids of local tile j of a warp (second id only when BS == 8).
struct TileIds {
  int32_t a, b;
};

template <int G, int BS, bool FUSED>
__global__ void __launch_bounds__(kThreads, 2)
    paged_attention_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                 const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  static_assert(G >= 1 && G <= 8, "query rows of the MMA tile");
  static_assert(BS == 8 || BS == 16 || BS == 32 || BS == 64, "block sizes with a kernel");
  constexpr unsigned kFull = 0xffffffffu;
  constexpr int kBlocksPerTile = BS < kTile ? kTile / BS : 1;  // 2 for BS = 8
  constexpr int kBoxRows = BS < kTile ? BS : kTile;
  constexpr uint32_t kBoxBytes = kBoxRows * 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int g = blockIdx.x, s = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads;
  const int h0 = g * G;

  const int L = clamp_context<BS>(p, s, threadIdx.x == 0 && g == 0 && split == 0);
  const int ntiles = (L + kTile - 1) / kTile;
  const int nsplit = (ntiles + kPartitionTiles - 1) / kPartitionTiles;
  if (L == 0) {
    if (split == 0) {
      __half* o = p.out + (static_cast<int64_t>(s) * Hq + h0) * kHeadDim;
      for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) o[i] = __float2half_rn(0.f);
    }
    return;
  }
  const int tile_begin = split * kPartitionTiles;
  if (tile_begin >= ntiles) return;
  const int n_here = min(kPartitionTiles, ntiles - tile_begin);
  // warp w streams local tiles w, w + 4, ...; lane j holds the ids of its j-th
  const int my_count = warp < n_here ? (n_here - warp + kWarps - 1) / kWarps : 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars) + warp * kStages;
  const uint32_t ring = smem_u32(smem + Smem::stages + warp * kStages * kStageBytes);

  const int32_t* trow = p.block_tables + static_cast<int64_t>(s) * p.max_blocks;
  TileIds my_ids = {-1, -1};
  if (lane < my_count) {
    const int tile = tile_begin + warp + lane * kWarps;
    const int first_tok = tile * kTile;
#pragma unroll
    for (int q = 0; q < kBlocksPerTile; ++q) {
      const int tok = first_tok + q * BS;
      int32_t b = -1;
      if (tok < L) {
        b = __ldg(trow + tok / BS);
        if (b < 0 || b >= p.num_blocks) {
          report(p.dev_err, PKV_DEV_BAD_BLOCK_ID);
          b = -2;  // poison the whole tile
        }
      }
      if (q == 0) my_ids.a = b; else my_ids.b = b;
    }
    if (my_ids.b == -2) my_ids.a = -2;
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

  // lane 0 only: local tile k with physical block(s) ids
  auto issue = [&](int k, TileIds ids) {
    uint64_t* bar = &bars[k % kStages];
    uint8_t* st = smem + Smem::stages + (warp * kStages + k % kStages) * kStageBytes;
    if (ids.a < 0) {  // reported already: complete the phase without data
      mbar_arrive(bar);
      return;
    }
    const int row_in_block = BS > kTile ? ((tile_begin + warp + k * kWarps) * kTile) % BS : 0;
    const int nboxes = (kBlocksPerTile == 2 && ids.b >= 0) ? 2 : 1;
    mbar_arrive_expect_tx(bar, 4 * kBoxBytes * nboxes);
#pragma unroll
    for (int q = 0; q < kBlocksPerTile; ++q) {
      if (q == 1 && nboxes == 1) break;
      const int row = (q == 0 ? ids.a : ids.b) * BS + row_in_block;
      const uint32_t off = q * kBoxBytes;
      tma_load_3d(st + off, &tmap_k, 0, g, row, bar);
      tma_load_3d(st + kHalfTileBytes + off, &tmap_k, 64, g, row, bar);
      tma_load_3d(st + 2 * kHalfTileBytes + off, &tmap_v, 0, g, row, bar);
      tma_load_3d(st + 3 * kHalfTileBytes + off, &tmap_v, 64, g, row, bar);
    }
  };
  auto ids_of = [&](int k) {
    TileIds t;
    t.a = __shfl_sync(kFull, my_ids.a, k);
    t.b = __shfl_sync(kFull, my_ids.b, k);
    return t;
  };

  int issued = min(kStages, my_count);
#pragma unroll
  for (int k = 0; k < kStages; ++k) {
    const TileIds t = ids_of(k);
    if (lane == 0 && k < issued) issue(k, t);
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

  // the new token (FUSED): its tile, its row within the tile
  const int new_tile = (L - 1) / kTile, new_row = (L - 1) % kTile;

  float m = -INFINITY, l = 0.f;
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  bool ok = true;
  for (int k = 0; k < issued; ++k) {
    const int stage = k % kStages;
    const bool landed = mbar_wait_bounded(&bars[stage], (k / kStages) & 1, p.dev_err);
    ok = __all_sync(kFull, ok && landed) != 0;
    const TileIds t = ids_of(k);
    const int tile = tile_begin + warp + k * kWarps;
    if (ok && t.a >= 0) {
      const uint32_t st = ring + stage * kStageBytes;
      if (FUSED && tile == new_tile) {
        // cache write of the new token: global slot and the staged row
        const int32_t blk = (BS < kTile && new_row >= BS) ? t.b : t.a;
        const int row_in_block = (L - 1) % BS;
        const int c = lane & 15;
        const bool is_v = lane >= 16;
        const int64_t src = (static_cast<int64_t>(s) * p.num_kv_heads + g) * kHeadDim + c * 8;
        const uint4 val = *reinterpret_cast<const uint4*>((is_v ? p.v_new : p.k_new) + src);
        const int64_t dst =
            ((static_cast<int64_t>(blk) * BS + row_in_block) * p.num_kv_heads + g) * kHeadDim +
            c * 8;
        *reinterpret_cast<uint4*>((is_v ? p.v_cache : p.k_cache) + dst) = val;
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                         tile_chunk(st, is_v ? 2 : 0, new_row, c)),
                     "r"(val.x), "r"(val.y), "r"(val.z), "r"(val.w)
                     : "memory");
        fence_proxy_async_smem();
        __syncwarp();
      }
      const int valid = min(kTile, L - tile * kTile);
      process_tile(st, qa, valid, lane, p.scale_log2, m, l, o);
    }
    __syncwarp();
    const TileIds nt = ids_of(issued < 32 ? issued : 0);
    if (ok && issued < my_count) {
      if (lane == 0) issue(issued, nt);
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

// ---- host side: launch of one instantiation ---------------------------------------
template <int G, int BS, bool FUSED>
int launch_one(const CUtensorMap& mk, const CUtensorMap& mv, const Params& p,
               cudaStream_t stream) {
  // The shared-memory opt-in is per device; remember it for up to 64 devices.
  static std::atomic<uint8_t> opted_in[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(paged_attention_split_kernel<G, BS, FUSED>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem::alloc) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev >= 0 && dev < 64) opted_in[dev].store(1, std::memory_order_release);
  }
  dim3 grid(p.num_kv_heads, p.num_seqs, p.max_splits);
  paged_attention_split_kernel<G, BS, FUSED><<<grid, kThreads, Smem::alloc, stream>>>(mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Host launcher of the split kernel for one block size (attention_bs*.cu).
template <int BS>
int launch_split(int G, bool fused, const CUtensorMap& mk, const CUtensorMap& mv, const Params& p,
                 cudaStream_t stream);

#define PKV_DEFINE_LAUNCH_SPLIT(BSV)                                                          \
  template <>                                                                                 \
  int launch_split<BSV>(int G, bool fused, const CUtensorMap& mk, const CUtensorMap& mv,      \
                        const Params& p, cudaStream_t st) {                                   \
    switch (G) {                                                                              \
      case 1: return fused ? launch_one<1, BSV, true>(mk, mv, p, st)                          \
                           : launch_one<1, BSV, false>(mk, mv, p, st);                        \
      case 2: return fused ? launch_one<2, BSV, true>(mk, mv, p, st)                          \
                           : launch_one<2, BSV, false>(mk, mv, p, st);                        \
      case 4: return fused ? launch_one<4, BSV, true>(mk, mv, p, st)                          \
                           : launch_one<4, BSV, false>(mk, mv, p, st);                        \
      case 8: return fused ? launch_one<8, BSV, true>(mk, mv, p, st)                          \
                           : launch_one<8, BSV, false>(mk, mv, p, st);                        \
      default: return PKV_ERR_UNSUPPORTED;                                                    \
    }                                                                                         \
  }

}  // namespace attn
}  // namespace pkv
