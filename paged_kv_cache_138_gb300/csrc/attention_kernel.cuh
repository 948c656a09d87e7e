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
//    split of up to T tiles), T = 128, 64 or 32 (2048, 1024 or 512 tokens) per
//    launch: the largest that still gives the grid enough CTAs (see
//    partition_tiles_for).  A CTA's set-up, drain and cross-warp merge cost the
//    same whatever its length, so long splits amortise them; a batch too small
//    to fill the GPU with long splits gets short ones.  The G = Hq / Hkv query heads that
//    read KV head g are handled together, so every K/V byte leaves HBM once.
//  * Each of the 4 warps streams its own tiles of the split (warp w takes tiles
//    w, w+4, ...) through a private 2-stage ring in shared memory.  A stage is
//    one tile of one KV head: K and V, each as two 64-dim TMA boxes (128-byte
//    swizzle), 8 KB, completion counted on one mbarrier with a bounded wait.
//    A tile is a 16-row window of a block (BS >= 16) or two 8-row blocks
//    (BS = 8); lane 0 refills a stage as soon as the warp is done with it.
//    Three CTAs share an SM (66 KB of shared memory each): 12 warps x 2 stages
//    keep 192 KB in flight per SM, and while one CTA sets up or merges the
//    other two keep streaming.
//  * Per tile, S = Q K^T and O += P V run on mma.sync m16n8k16 fragments read
//    with ldmatrix from the swizzled tiles (query heads are the MMA rows).
//  * Online softmax in base 2 per query row with a lazy rescale: the running
//    max only moves when a tile max exceeds it by more than 8, so most tiles
//    skip rescaling and every weight stays <= 2^8 (exact in fp16 range).  The
//    weights are rounded to fp16 once, for the P.V product, and the running
//    sum adds those same fp16 values.
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
#include <climits>

#include "pkv_device.cuh"

namespace pkv {
namespace attn {

constexpr int kHeadDim = 128;
constexpr int kTile = 16;                          // tokens per stage
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kCtasPerSm = 3;                      // 3 x (4 x 2 x 8 KB rings) per SM
constexpr int kPartitionTiles = 32;                // shortest split T (512 tokens)
constexpr int kMaxPartitionTiles = 128;            // longest split: 32 tiles per warp
constexpr int kHalfTileBytes = kTile * 64 * 2;     // 16 rows x 128 B
constexpr int kStageBytes = 4 * kHalfTileBytes;    // K lo, K hi, V lo, V hi
constexpr float kRescaleThreshold = 8.0f;          // log2 units

struct Smem {
  static constexpr int stages = 0;
  static constexpr int stages_bytes = kWarps * kStages * kStageBytes;
  static constexpr int bars = stages + stages_bytes;                  // u64 [warps][stages]
  static constexpr int ml = bars + kWarps * kStages * 8;              // float [warps][16][2]
  static constexpr int total = ml + kWarps * 16 * 2 * 4;
  static constexpr int alloc = total + 1024;                          // alignment slack
  static_assert(kWarps * 16 * kHeadDim * 4 <= stages_bytes, "merge buffer must fit");
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
  // shared-prefix groups (grouped launches only; seq_group == nullptr otherwise)
  const int32_t* seq_group;     // [S] group of each sequence
  const int32_t* group_first;   // [num_groups + 1] first sequence of each group
  const int32_t* group_shared;  // [num_groups] tokens the whole group shares
  // copy-on-write folded into a fused launch (nullptr otherwise): sequence s
  // gets logical block cow_block[s] (-1: none) as a copy of physical block
  // cow_src[s] before its new token is written there
  const int32_t* cow_block;     // [S]
  const int32_t* cow_src;       // [S]
  int64_t num_blocks;
  int num_seqs, num_q_heads, num_kv_heads, max_blocks, max_splits, block_size, num_groups;
  int own_tiles_cap;  // grouped launches: own tiles the grid covers per sequence
  int shared_splits_cap;  // grouped launches: split slots reserved for a shared prefix
  int seq_stride;     // split grid: row y of the grid is sequence (y * seq_stride) % S
  int rank_by_length;  // split grid: last split plane in zigzag_rank order of length
  int partition_tiles;  // T: tiles per split (32, 64 or 128)
  float scale_log2;
};

inline int tiles_for_tokens(int64_t tokens) { return static_cast<int>((tokens + kTile - 1) / kTile); }
inline int max_splits_for(int max_blocks, int block_size, int partition_tiles = kPartitionTiles) {
  const int tiles = tiles_for_tokens(static_cast<int64_t>(max_blocks) * block_size);
  return (tiles + partition_tiles - 1) / partition_tiles;
}

// Split length T of a launch: the longest of 128, 64, 32 tiles for which
// the grid's upper bound S x Hkv x ceil(tiles of the longest table / T) still
// reaches kMinSplitUnits CTAs (a few waves of three CTAs on each of 152 SMs).
constexpr int64_t kMinSplitUnits = 1024;
inline int partition_tiles_for(int num_seqs, int num_kv_heads, int max_blocks, int block_size) {
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_kv_heads;
  for (int t = kMaxPartitionTiles; t > kPartitionTiles; t /= 2)
    if (rows * max_splits_for(max_blocks, block_size, t) >= kMinSplitUnits) return t;
  return kPartitionTiles;
}

// Tiles a sequence shares with its group (0 outside grouped launches) and the
// split slots those take in the workspace.  The shared part ends on a tile
// boundary (a group whose shared length is not a multiple of 16 is reported by
// its shared units).  A group id out of range counts as no shared prefix; the
// sequence's own units report it.
__device__ __forceinline__ int shared_tiles_of(const Params& p, int s) {
  if (!p.seq_group) return 0;
  const int grp = __ldg(p.seq_group + s);
  if (grp < 0 || grp >= p.num_groups) return 0;
  return max(__ldg(p.group_shared + grp), 0) / kTile;
}
__device__ __forceinline__ int splits_for_tiles(const Params& p, int tiles) {
  return (tiles + p.partition_tiles - 1) / p.partition_tiles;
}
// Workspace slots of a sequence's shared prefix: one per split of it, never
// more than the launch reserved (a group sharing more tokens than the launch
// was sized for is reported; its rows then stay inside their own slots).
__device__ __forceinline__ int shared_slots_of(const Params& p, int shared_tiles) {
  return min(splits_for_tiles(p, shared_tiles), p.shared_splits_cap);
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
  const uint32_t pa0 = pack_half2(p0, p1), pa2 = pack_half2(p2, p3);
  // the sum takes the fp16 weights the P.V product uses, so numerator and
  // denominator weigh every token alike (one dominant token returns its V row)
  l += sum_half2(pa0) + sum_half2(pa2);
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


__device__ __forceinline__ void mma_16816_full(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same tile with all 16 MMA rows real (a shared-prefix group: one row per
// (member sequence, query head)).  Every token of a shared tile is valid.
// Lane holds rows r0 = lane / 4 and r1 = r0 + 8: m[0], l[0] and o[nd][0..1]
// belong to r0; m[1], l[1] and o[nd][2..3] to r1.
__device__ __forceinline__ void process_tile16(uint32_t st, const uint32_t (&qa)[8][4], int lane,
                                               float scale_log2, float (&m)[2], float (&l)[2],
                                               float (&o)[16][4]) {
  constexpr unsigned kFull = 0xffffffffu;
  const int r8 = lane & 7, mi = lane >> 3;
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  const int ktok = r8 + ((mi >> 1) << 3);
#pragma unroll
  for (int kc = 0; kc < 8; ++kc) {
    uint32_t b00, b01, b10, b11;
    ldsm_x4(tile_chunk(st, 0, ktok, 2 * kc + (mi & 1)), b00, b01, b10, b11);
    mma_16816_full(s0, qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b00, b01);
    mma_16816_full(s1, qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], b10, b11);
  }
  uint32_t pa[4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float x0 = s0[2 * r] * scale_log2, x1 = s0[2 * r + 1] * scale_log2;
    const float x2 = s1[2 * r] * scale_log2, x3 = s1[2 * r + 1] * scale_log2;
    float bm = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
    if (bm > m[r] + kRescaleThreshold) {
      const float alpha = exp2_approx(m[r] - bm);
      l[r] *= alpha;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        o[nd][2 * r] *= alpha;
        o[nd][2 * r + 1] *= alpha;
      }
      m[r] = bm;
    }
    const float p0 = exp2_approx(x0 - m[r]), p1 = exp2_approx(x1 - m[r]);
    const float p2 = exp2_approx(x2 - m[r]), p3 = exp2_approx(x3 - m[r]);
    pa[r] = pack_half2(p0, p1);       // a0 (row r0) / a1 (row r1): tokens 2(lane%4)..
    pa[2 + r] = pack_half2(p2, p3);   // a2 / a3: tokens 8 + 2(lane%4)..
    l[r] += sum_half2(pa[r]) + sum_half2(pa[2 + r]);   // the fp16 weights, as in P.V
  }
  const int vtok = r8 + ((mi & 1) << 3);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t v0, v1, v2, v3;
    ldsm_x4_trans(tile_chunk(st, 2, vtok, 2 * j + (mi >> 1)), v0, v1, v2, v3);
    mma_16816_full(o[2 * j], pa[0], pa[1], pa[2], pa[3], v0, v1);
    mma_16816_full(o[2 * j + 1], pa[0], pa[1], pa[2], pa[3], v2, v3);
  }
}

// Physical block ids of one tile (second id only when BS == 8).
struct TileIds {
  int32_t a, b;
};

// The per-warp TMA pipeline over the tiles tile_begin + warp + 4 j of one
// table row: lane j keeps the ids of the warp's j-th tile, lane 0 keeps
// kStages tiles in flight, run() hands every landed tile to a callback.
template <int BS>
struct TileStream {
  static constexpr unsigned kFull = 0xffffffffu;
  static constexpr int kBlocksPerTile = BS < kTile ? kTile / BS : 1;  // 2 for BS = 8
  static constexpr int kBoxRows = BS < kTile ? BS : kTile;
  static constexpr uint32_t kBoxBytes = kBoxRows * 128;

  uint8_t* stages;        // this warp's ring
  uint64_t* bars;
  const CUtensorMap* tk;
  const CUtensorMap* tv;
  int warp, lane, g, tile_begin, my_count, issued;
  bool timed_out;  // a bounded wait of run() gave up (warp-uniform)
  TileIds my_ids;

  // ids_limit: tokens at or past it have no block (the context length).
  // Logical block cow_blk (-1: none) is read from physical block cow_from
  // instead of the table's entry (copy-on-write folded into the launch).
  __device__ __forceinline__ void init(uint8_t* smem, const CUtensorMap* tk_, const CUtensorMap* tv_,
                                       int g_, const int32_t* trow, int tile_begin_, int n_here,
                                       int ids_limit, const Params& p, int cow_blk = -1,
                                       int32_t cow_from = -1) {
    warp = threadIdx.x >> 5;
    lane = threadIdx.x & 31;
    tk = tk_;
    tv = tv_;
    g = g_;
    tile_begin = tile_begin_;
    my_count = warp < n_here ? (n_here - warp + kWarps - 1) / kWarps : 0;
    timed_out = false;
    stages = smem + Smem::stages + warp * kStages * kStageBytes;
    bars = reinterpret_cast<uint64_t*>(smem + Smem::bars) + warp * kStages;
    my_ids.a = my_ids.b = -1;
    if (lane < my_count) {
      const int first_tok = (tile_begin + warp + lane * kWarps) * kTile;
#pragma unroll
      for (int q = 0; q < kBlocksPerTile; ++q) {
        const int tok = first_tok + q * BS;
        int32_t b = -1;
        if (tok < ids_limit && tok / BS == cow_blk) {
          b = cow_from;  // checked by the caller
        } else if (tok < ids_limit) {
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
        prefetch_tmap(tk);
        prefetch_tmap(tv);
      }
      for (int j = 0; j < kStages; ++j) mbar_init(&bars[j], 1);
      fence_barrier_init();
    }
    __syncwarp();
    issued = min(kStages, my_count);
#pragma unroll
    for (int k = 0; k < kStages; ++k) {
      const TileIds t = ids_of(k);
      if (lane == 0 && k < issued) issue(k, t);
    }
  }

  __device__ __forceinline__ TileIds ids_of(int k) const {
    TileIds t;
    t.a = __shfl_sync(kFull, my_ids.a, k);
    t.b = __shfl_sync(kFull, my_ids.b, k);
    return t;
  }

  // lane 0 only: local tile k with physical block(s) ids
  __device__ __forceinline__ void issue(int k, TileIds ids) {
    uint64_t* bar = &bars[k % kStages];
    uint8_t* st = stages + (k % kStages) * kStageBytes;
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
      tma_load_3d(st + off, tk, 0, g, row, bar);
      tma_load_3d(st + kHalfTileBytes + off, tk, 64, g, row, bar);
      tma_load_3d(st + 2 * kHalfTileBytes + off, tv, 0, g, row, bar);
      tma_load_3d(st + 3 * kHalfTileBytes + off, tv, 64, g, row, bar);
    }
  }

  // f(stage smem address, tile index, ids) for every tile that landed.
  template <class F>
  __device__ __forceinline__ void run(int32_t* dev_err, F&& f) {
    bool ok = true;
    for (int k = 0; k < issued; ++k) {
      const int stage = k % kStages;
      const bool landed = mbar_wait_bounded(&bars[stage], (k / kStages) & 1, dev_err);
      ok = __all_sync(kFull, ok && landed) != 0;
      const TileIds t = ids_of(k);
      if (ok && t.a >= 0) f(smem_u32(stages + stage * kStageBytes), tile_begin + warp + k * kWarps, t);
      __syncwarp();
      const TileIds nt = ids_of(issued < 32 ? issued : 0);
      if (ok && issued < my_count) {
        if (lane == 0) issue(issued, nt);
        ++issued;
      }
    }
    timed_out = !ok;
  }
};

// Combine the 4 warps' (m, l, o) of `rows` query rows held in shared memory
// (ml [warps][16][2], ob [warps][16][128]) and hand each row's (M, den, num)
// to emit(row, d, M, den, num4) for dims d .. d + 3.  Warp w takes rows w,
// w + 4, ...; lane i dims 4 i .. 4 i + 3 (one 16-byte read per warp's
// partial), so up to 4 rows merge in one pass.  Per element the arithmetic
// is the warps' weights exp2(m_w - M) in warp order, as one thread per
// element would do it.
template <class Emit>
__device__ __forceinline__ void merge_warps(const float* ml, const float* ob, int rows, Emit&& emit) {
  const int lane = threadIdx.x & 31;
  for (int r = threadIdx.x >> 5; r < rows; r += kWarps) {
    float mw[kWarps];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      mw[w] = ml[(w * 16 + r) * 2];
      M = fmaxf(M, mw[w]);
    }
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float c = exp2_approx(mw[w] - M);
        const float4 v = *reinterpret_cast<const float4*>(ob + (w * 16 + r) * kHeadDim + 4 * lane);
        num.x += c * v.x;
        num.y += c * v.y;
        num.z += c * v.z;
        num.w += c * v.w;
        den += c * ml[(w * 16 + r) * 2 + 1];
      }
    }
    emit(r, 4 * lane, M, den, num);
  }
}

__device__ __forceinline__ void store_partial(const Params& p, int64_t row, int slot, int d,
                                              float M, float den, float4 num) {
  const int64_t at = row * p.max_splits + slot;
  *reinterpret_cast<float4*>(p.part_o + at * kHeadDim + d) = num;
  if (d == 0) {
    p.part_ml[at * 2] = M;
    p.part_ml[at * 2 + 1] = den;
  }
}

// fp16 output of dims d .. d + 3 of a row (one 8-byte store)
__device__ __forceinline__ void store_out4(__half* o, float den, float4 num) {
  const bool ok = den > 0.f;
  const __half2 a = __floats2half2_rn(ok ? num.x / den : 0.f, ok ? num.y / den : 0.f);
  const __half2 b = __floats2half2_rn(ok ? num.z / den : 0.f, ok ? num.w / den : 0.f);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(o) = u;
}

// Copy-on-write from the staged tile: staged rows first_row .. first_row +
// rows - 1 (K and V of KV head g) are stored as rows dst_row .. dst_row +
// rows - 1 of block `dst`, one 16-byte chunk per lane and step; the
// half-warps write 256 contiguous bytes each.  A block of at most 16 rows is
// staged whole by one tile; a longer one by one tile per 16 rows.
template <int BS>
__device__ __forceinline__ void store_staged_rows(uint32_t st, const Params& p, int g,
                                                  int32_t dst, int first_row, int dst_row,
                                                  int rows, int lane) {
  for (int i = lane; i < rows * 32; i += 32) {
    const int r = i >> 5, c = i & 15;
    const bool is_v = (i >> 4) & 1;
    uint4 val;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                 : "r"(tile_chunk(st, is_v ? 2 : 0, first_row + r, c)));
    const int64_t at =
        ((static_cast<int64_t>(dst) * BS + dst_row + r) * p.num_kv_heads + g) * kHeadDim + c * 8;
    *reinterpret_cast<uint4*>((is_v ? p.v_cache : p.k_cache) + at) = val;
  }
  __syncwarp();  // every lane has read the stage before it changes again
}

// Copy-on-write of the rows of a block past every tile the launch streams
// (a block longer than 16 rows whose last rows lie past the context): rows
// from_row .. BS - 1 of block `src`, K and V of KV head g, copied to block
// `dst` with 16-byte loads and stores.
template <int BS>
__device__ __forceinline__ void copy_block_tail(const Params& p, int g, int32_t src, int32_t dst,
                                                int from_row, int lane) {
  const int64_t block_elems = static_cast<int64_t>(BS) * p.num_kv_heads * kHeadDim;
  for (int i = lane; i < (BS - from_row) * 32; i += 32) {
    const int r = from_row + (i >> 5), c = i & 15;
    __half* base = ((i >> 4) & 1) ? p.v_cache : p.k_cache;
    const int64_t off = (static_cast<int64_t>(r) * p.num_kv_heads + g) * kHeadDim + c * 8;
    const uint4 val = *reinterpret_cast<const uint4*>(base + src * block_elems + off);
    *reinterpret_cast<uint4*>(base + dst * block_elems + off) = val;
  }
}

// One CTA per (KV head, sequence, split of its own tiles).  In grouped launches
// a sequence's own tiles start after the prefix its group shares, and its
// partials go after the group's shared splits.
template <int G, int BS, bool FUSED>
__device__ __forceinline__ void split_body(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                           const Params& p, uint8_t* smem, int g, int s,
                                           int split) {
  static_assert(G >= 1 && G <= 8, "query rows of the MMA tile");
  static_assert(BS == 8 || BS == 16 || BS == 32 || BS == 64, "block sizes with a kernel");
  constexpr unsigned kFull = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads;
  const int h0 = g * G;

  // the group's shared length first: its two dependent loads then overlap the
  // context length's
  const int shared_tiles = shared_tiles_of(p, s);
  const int L = clamp_context<BS>(p, s, threadIdx.x == 0 && g == 0 && split == 0);
  const int ntiles = (L + kTile - 1) / kTile;
  const int own_begin = min(shared_tiles, ntiles);
  const int shared_splits = shared_slots_of(p, own_begin);
  const int nsplit = shared_splits + splits_for_tiles(p, ntiles - own_begin);
  if (L == 0) {
    if (split == 0) {
      __half* o = p.out + (static_cast<int64_t>(s) * Hq + h0) * kHeadDim;
      for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) o[i] = __float2half_rn(0.f);
    }
    return;
  }
  if (p.seq_group && split == 0 && threadIdx.x == 0) {
    const int grp = __ldg(p.seq_group + s);
    // no such group, a longer shared prefix than the launch reserved, or more
    // own tokens than the grid covers
    if (grp < 0 || grp >= p.num_groups || splits_for_tiles(p, own_begin) > p.shared_splits_cap ||
        ntiles - own_begin > p.own_tiles_cap)
      report(p.dev_err, PKV_DEV_BAD_GROUP);
  }
  // FUSED in a grouped launch: the new token must fall in the sequence's own
  // tiles (the only ones its own units stream); in a shared tile it would be
  // a token written into a block its whole group reads
  if (FUSED && p.seq_group && split == 0 && threadIdx.x == 0 && (L - 1) / kTile < own_begin)
    report(p.dev_err, PKV_DEV_BAD_GROUP);
  const int tile_begin = own_begin + split * p.partition_tiles;
  if (tile_begin >= ntiles) return;
  const int n_here = min(p.partition_tiles, ntiles - tile_begin);

  // copy-on-write folded into the launch (FUSED): the block must hold some
  // of the sequence's own tokens; the units whose tiles hold it read the
  // source block instead and store the staged rows as the block's (tiles
  // cow_tile_lo .. cow_tile_hi; one tile for BS <= 16)
  int cow_blk = -1, cow_tile_lo = -1, cow_tile_hi = -2;
  int32_t cow_from = -1, cow_to = -1;
  if constexpr (FUSED) {
    if (p.cow_block) {
      const int cb = __ldg(p.cow_block + s);
      if (cb >= 0) {
        const bool may_report = threadIdx.x == 0 && g == 0 && split == 0;
        const int32_t from = __ldg(p.cow_src + s);
        if (cb >= p.max_blocks || cb * BS >= L || cb * BS < own_begin * kTile) {
          if (may_report) report(p.dev_err, PKV_DEV_BAD_POSITION);
        } else {
          const int32_t to = __ldg(p.block_tables + static_cast<int64_t>(s) * p.max_blocks + cb);
          if (from < 0 || from >= p.num_blocks || to < 0 || to >= p.num_blocks) {
            if (may_report) report(p.dev_err, PKV_DEV_BAD_BLOCK_ID);
          } else {
            cow_blk = cb;
            cow_tile_lo = cb * BS / kTile;
            cow_tile_hi = (cb * BS + BS - 1) / kTile;
            cow_from = from;
            cow_to = to;
          }
        }
      }
    }
  }

  TileStream<BS> ts;
  ts.init(smem, &tmap_k, &tmap_v, g, p.block_tables + static_cast<int64_t>(s) * p.max_blocks,
          tile_begin, n_here, L, p, cow_blk, cow_from);

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

  // the new token (FUSED): its tile, its row within the tile; the warp that
  // will hold that tile loads the token's K (lanes 0-15) / V (16-31) now, so
  // the load is done by the time the tile lands
  const int new_tile = (L - 1) / kTile, new_row = (L - 1) % kTile;
  uint4 new_val = make_uint4(0u, 0u, 0u, 0u);
  if (FUSED && new_tile >= tile_begin && new_tile < tile_begin + n_here &&
      (new_tile - tile_begin) % kWarps == warp) {
    const int64_t src =
        (static_cast<int64_t>(s) * p.num_kv_heads + g) * kHeadDim + (lane & 15) * 8;
    new_val = *reinterpret_cast<const uint4*>((lane >= 16 ? p.v_new : p.k_new) + src);
  }

  float m = -INFINITY, l = 0.f;
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  ts.run(p.dev_err, [&](uint32_t st, int tile, TileIds t) {
    if (FUSED && tile == new_tile) {
      // cache write of the new token: global slot and the staged row (a
      // block being copied is written at its copy, not at its source)
      int32_t blk = (BS < kTile && new_row >= BS) ? t.b : t.a;
      if ((L - 1) / BS == cow_blk) blk = cow_to;
      const int row_in_block = (L - 1) % BS;
      const int c = lane & 15;
      const bool is_v = lane >= 16;
      const uint4 val = new_val;
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
    if constexpr (FUSED) {
      // the copied block, new token included, before process_tile zeroes the
      // V rows past the context in the stage
      if (tile >= cow_tile_lo && tile <= cow_tile_hi) {
        if constexpr (BS <= kTile) {
          store_staged_rows<BS>(st, p, g, cow_to, (cow_blk * BS) % kTile, 0, BS, lane);
        } else {
          const int dst_row = tile * kTile - cow_blk * BS;
          store_staged_rows<BS>(st, p, g, cow_to, 0, dst_row, kTile, lane);
          // the context's last tile: the block's rows past it are streamed
          // by no unit, so this one copies them from the source
          if (tile == (L - 1) / kTile && dst_row + kTile < BS)
            copy_block_tail<BS>(p, g, cow_from, cow_to, dst_row + kTile, lane);
        }
      }
    }
    process_tile(st, qa, min(kTile, L - tile * kTile), lane, p.scale_log2, m, l, o);
  });
  l += __shfl_xor_sync(kFull, l, 1);
  l += __shfl_xor_sync(kFull, l, 2);

  // ---- merge the 4 warps' partial softmax states ------------------------------
  // every issued tile has landed and the ring is free -- unless a bounded wait
  // gave up: boxes may then still be in flight into the ring, which the merge
  // reuses, so the CTA leaves without merging or storing (PKV_DEV_WAIT_TIMEOUT
  // is reported; the launch's outputs are undefined)
  if (__syncthreads_or(ts.timed_out)) return;
  float* ml = reinterpret_cast<float*>(smem + Smem::ml);
  float* ob = reinterpret_cast<float*>(smem + Smem::stages);
  if (qrow < G) {
    if ((lane & 3) == 0) {
      ml[(warp * 16 + qrow) * 2] = m;
      ml[(warp * 16 + qrow) * 2 + 1] = l;
    }
    float* orow = ob + (warp * 16 + qrow) * kHeadDim + 2 * (lane & 3);
#pragma unroll
    for (int nd = 0; nd < 16; ++nd)
      *reinterpret_cast<float2*>(orow + nd * 8) = make_float2(o[nd][0], o[nd][1]);
  }
  __syncthreads();
  merge_warps(ml, ob, G, [&](int gi, int d, float M, float den, float4 num) {
    const int64_t row = static_cast<int64_t>(s) * Hq + h0 + gi;
    if (nsplit == 1)
      store_out4(p.out + row * kHeadDim + d, den, num);
    else
      store_partial(p, row, shared_splits + split, d, M, den, num);
  });
}

// Shared prefix of a group: one CTA per (KV head, group, split of the shared
// tiles) streams each shared tile once for every member, the members' query
// heads being the 16 rows of the MMA tile (members x G <= 16).  It writes one
// partial per member row into the group's first split slots; the members' own
// tiles go through paged_attention_split_kernel and the merge kernel combines.
template <int G, int BS>
__device__ __forceinline__ void shared_body(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                            const Params& p, uint8_t* smem, int g, int grp,
                                            int split) {
  constexpr unsigned kFull = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads;

  const int first = __ldg(p.group_first + grp);
  const int last = __ldg(p.group_first + grp + 1);
  const int shared = __ldg(p.group_shared + grp);
  const int members = last - first;
  const int rows = members * G;
  // a malformed group is reported and skipped: members inside the batch, at
  // most 16 MMA rows, a shared length on a tile boundary within the tables
  if (first < 0 || members < 0 || last > p.num_seqs || rows > 16 || shared % kTile != 0 ||
      shared > p.max_blocks * BS) {
    if (threadIdx.x == 0 && g == 0 && split == 0) report(p.dev_err, PKV_DEV_BAD_GROUP);
    return;
  }
  if (shared <= 0 || members == 0) return;
  const int shared_tiles = shared / kTile;
  const int tile_begin = split * p.partition_tiles;
  if (tile_begin >= shared_tiles) return;
  const int n_here = min(p.partition_tiles, shared_tiles - tile_begin);

  // the leader's blocks stream for the whole group: issue them first
  const int32_t* lead = p.block_tables + static_cast<int64_t>(first) * p.max_blocks;
  TileStream<BS> ts;
  ts.init(smem, &tmap_k, &tmap_v, g, lead, tile_begin, n_here, shared, p);

  // A fragments of rows r0 = lane/4 and r1 = r0 + 8: row r is member r / G,
  // query head g*G + r % G
  uint32_t qa[8][4];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = (lane >> 2) + 8 * half;
    if (r < rows) {
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<int64_t>(first + r / G) * Hq + g * G + r % G) * kHeadDim);
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        qa[kc][half] = __ldg(qp + 8 * kc + (lane & 3));
        qa[kc][2 + half] = __ldg(qp + 8 * kc + 4 + (lane & 3));
      }
    } else {
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) qa[kc][half] = qa[kc][2 + half] = 0u;
    }
  }

  // while the first tiles are in flight: every member must belong to this
  // group, hold at least the shared tokens and map them to the leader's
  // blocks (loads only in the loop, so the unrolled iterations overlap)
  {
    const int blk_lo = tile_begin * kTile / BS;
    // blocks holding the unit's tiles (the last one partly for BS > 16)
    const int nblk = ((tile_begin + n_here) * kTile + BS - 1) / BS - blk_lo;
    const int total = members * nblk;
    bool bad = false;
#pragma unroll 4
    for (int i = threadIdx.x; i < total; i += kThreads) {
      const int mem = i / nblk, b = blk_lo + i % nblk;
      bad |= __ldg(p.block_tables + static_cast<int64_t>(first + mem) * p.max_blocks + b) !=
             __ldg(lead + b);
    }
    if (threadIdx.x < members)
      bad |= __ldg(p.context_lens + first + threadIdx.x) < shared ||
             __ldg(p.seq_group + first + threadIdx.x) != grp;
    if (bad) report(p.dev_err, PKV_DEV_BAD_GROUP);
  }

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  ts.run(p.dev_err, [&](uint32_t st, int, TileIds) {
    process_tile16(st, qa, lane, p.scale_log2, m, l, o);
  });
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(kFull, l[r], 1);
    l[r] += __shfl_xor_sync(kFull, l[r], 2);
  }

  // as in split_body: after a wait that gave up, neither merge nor store
  if (__syncthreads_or(ts.timed_out)) return;
  float* ml = reinterpret_cast<float*>(smem + Smem::ml);
  float* ob = reinterpret_cast<float*>(smem + Smem::stages);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = (lane >> 2) + 8 * half;
    if (r < rows) {
      if ((lane & 3) == 0) {
        ml[(warp * 16 + r) * 2] = m[half];
        ml[(warp * 16 + r) * 2 + 1] = l[half];
      }
      float* orow = ob + (warp * 16 + r) * kHeadDim + 2 * (lane & 3);
#pragma unroll
      for (int nd = 0; nd < 16; ++nd)
        *reinterpret_cast<float2*>(orow + nd * 8) =
            make_float2(o[nd][2 * half], o[nd][2 * half + 1]);
    }
  }
  __syncthreads();
  merge_warps(ml, ob, rows, [&](int r, int d, float M, float den, float4 num) {
    const int64_t row = static_cast<int64_t>(first + r / G) * Hq + g * G + r % G;
    store_partial(p, row, split, d, M, den, num);
  });
}

__device__ __forceinline__ uint8_t* aligned_smem() {
  extern __shared__ uint8_t smem_raw[];
  return smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
}

// Batches of at most kThreads sequences are visited longest first.
constexpr int kMaxRankedSeqs = kThreads;

// The sequence of rank y when the batch is ordered by decreasing context
// length, ties by batch index (a permutation of 0..S-1).  The lengths are
// staged in the merge area of shared memory (unused until the merge), padded
// to kMaxRankedSeqs with INT_MIN (never ahead of a real entry); each thread
// ranks one sequence against them, four per 16-byte read, and the one whose
// rank is y names itself.
__device__ __forceinline__ int ranked_sequence(const Params& p, uint8_t* smem, int y) {
  __shared__ int picked;
  int32_t* lens = reinterpret_cast<int32_t*>(smem + Smem::ml);
  static_assert(kMaxRankedSeqs == kThreads, "one thread per ranked sequence");
  static_assert(kMaxRankedSeqs * 4 <= Smem::total - Smem::ml, "lengths fit the merge area");
  static_assert(Smem::ml % 16 == 0, "16-byte reads of the staged lengths");
  const int t = threadIdx.x, n = p.num_seqs;
  const int32_t mine = t < n ? __ldg(p.context_lens + t) : INT_MIN;
  lens[t] = mine;
  __syncthreads();
  if (t < n) {
    const int4* l4 = reinterpret_cast<const int4*>(lens);
    int rank = 0;
#pragma unroll 8
    for (int j4 = 0; j4 < (n + 3) / 4; ++j4) {
      const int4 v = l4[j4];
      const int j = 4 * j4;
      rank += (v.x > mine) | ((v.x == mine) & (j < t));
      rank += (v.y > mine) | ((v.y == mine) & (j + 1 < t));
      rank += (v.z > mine) | ((v.z == mine) & (j + 2 < t));
      rank += (v.w > mine) | ((v.w == mine) & (j + 3 < t));
    }
    if (rank == y) picked = t;
  }
  __syncthreads();
  return picked;
}

// Rank visited at row y of n: longest, shortest, second longest, second
// shortest, ... (the two ends meet at the median length).
__device__ __forceinline__ int zigzag_rank(int y, int n) {
  return (y & 1) ? n - 1 - (y >> 1) : (y >> 1);
}

// grid (KV heads, sequences, splits).  CTAs start in grid order (all first
// splits, then all second splits, ...), so the last split plane makes the
// last waves, where SMs fall idle one by one.  Two orders of the rows:
//  * rank_by_length (at most kMaxRankedSeqs sequences, and a last plane whose
//    units can reach half a split: the host checks the table width), on the
//    last plane only: rows alternate between the longest and the shortest
//    sequences not yet visited (zigzag_rank), so long units start first,
//    every short unit's set-up and merge run beside a long unit's streaming,
//    and the grid ends on units of median length rather than on a random
//    long one or a crowd of short, latency-bound ones (longest first alone
//    measured -5.5 % on a batch of many very short sequences).  Ranking every
//    plane measured slower on batches with several splits (each CTA's ranking
//    delays its first load, and the earlier planes' units are mostly whole
//    splits anyway), as did ranking a last plane of short remainders;
//  * every other plane, and every plane of other batches: row y takes
//    sequence (y * seq_stride) % S, a stride coprime with S near 0.618 S: a
//    batch ordered by length (as continuous batching tends to keep it: older
//    requests are longer) would otherwise start all its short units back to
//    back, and a CTA with a short unit spends most of its life in set-up and
//    merge.
template <int G, int BS, bool FUSED>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    paged_attention_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                 const __grid_constant__ CUtensorMap tmap_v, const Params p) {
  // launched as a programmatic dependent of the stream's previous kernel: the
  // CTAs may be placed while it finishes; nothing is read before this wait,
  // which returns once that kernel has completed and its writes are visible
  // (a no-op after any other operation)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint8_t* smem = aligned_smem();
  const int y = blockIdx.y;
  const int s = (p.rank_by_length && blockIdx.z == gridDim.z - 1)
                    ? ranked_sequence(p, smem, zigzag_rank(y, p.num_seqs))
                    : static_cast<int>(static_cast<int64_t>(y) * p.seq_stride % p.num_seqs);
  split_body<G, BS, FUSED>(tmap_k, tmap_v, p, smem, blockIdx.x, s, blockIdx.z);
}

// One launch for a grouped step, 1-D grid of the shared-prefix units (KV
// head, group, shared split) and the members' own units (KV head, sequence,
// own split).  The shared units are the long ones and start early: grid
// positions 0, k, 2k, ... (k = shared_stride) hold them and the own units
// fill the rest in order.  With k = 1 they all come first; when own units are
// much shorter than shared ones the host spreads the shared units over the
// first half of the grid, so that every SM pairs a long unit with short ones
// instead of running the shared units together and then only short units,
// whose set-up and drain nothing hides.  The own units keep the batch order:
// visiting them in zigzag_rank order of length measured 2.9 % slower on
// forked samples (the samples of one prompt, adjacent in the batch, read
// their shared copy-on-write source close together, while it is still in
// L2).  FUSED: the own unit holding a sequence's last tile also writes its
// new token to the cache.
template <int G, int BS, bool FUSED>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    paged_attention_grouped_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                   const __grid_constant__ CUtensorMap tmap_v, const Params p,
                                   int shared_splits, int own_splits, int shared_stride) {
  // launched as a programmatic dependent of the stream's previous kernel: the
  // CTAs may be placed while it finishes; nothing is read before this wait,
  // which returns once that kernel has completed and its writes are visible
  // (a no-op after any other operation)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint8_t* smem = aligned_smem();
  int u = blockIdx.x;
  const int n_shared = p.num_kv_heads * p.num_groups * shared_splits;
  if (u % shared_stride == 0 && u / shared_stride < n_shared)
    u /= shared_stride;  // the (u / k)-th shared unit
  else
    u += n_shared - min(n_shared, u / shared_stride + 1);  // own units after the shared ones
  if (u < n_shared) {
    const int g = u % p.num_kv_heads;
    u /= p.num_kv_heads;
    shared_body<G, BS>(tmap_k, tmap_v, p, smem, g, u % p.num_groups, u / p.num_groups);
  } else {
    u -= n_shared;
    const int g = u % p.num_kv_heads;
    u /= p.num_kv_heads;
    split_body<G, BS, FUSED>(tmap_k, tmap_v, p, smem, g, u % p.num_seqs, u / p.num_seqs);
  }
}

// ---- host side: launch of one instantiation ---------------------------------------
// The shared-memory opt-in is per kernel and per device; cudaFuncSetAttribute is
// cheap but not free, so each kernel instantiation remembers it in its own
// flags (one per device, up to 64).
template <class Kernel>
int opt_in_smem(Kernel kernel, std::atomic<uint8_t> (&opted_in)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= 64 || !opted_in[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::alloc) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    if (dev >= 0 && dev < 64) opted_in[dev].store(1, std::memory_order_release);
  }
  return PKV_OK;
}

template <int G, int BS, bool FUSED>
int launch_one(const CUtensorMap& mk, const CUtensorMap& mv, const Params& p, int private_splits,
               cudaStream_t stream) {
  static std::atomic<uint8_t> opted_in[64];
  const int rc = opt_in_smem(paged_attention_split_kernel<G, BS, FUSED>, opted_in);
  if (rc != PKV_OK) return rc;
  // programmatic dependent launch: see the wait at the kernel's entry
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_kv_heads, p.num_seqs, private_splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem::alloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_attention_split_kernel<G, BS, FUSED>, mk, mv, p) ==
                 cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

template <int G, int BS, bool FUSED>
int launch_grouped(const CUtensorMap& mk, const CUtensorMap& mv, const Params& p,
                   int shared_splits, int own_splits, int shared_stride, cudaStream_t stream) {
  static std::atomic<uint8_t> opted_in[64];
  const int rc = opt_in_smem(paged_attention_grouped_kernel<G, BS, FUSED>, opted_in);
  if (rc != PKV_OK) return rc;
  const int64_t units = static_cast<int64_t>(p.num_kv_heads) *
                        (static_cast<int64_t>(p.num_groups) * shared_splits +
                         static_cast<int64_t>(p.num_seqs) * own_splits);
  if (units <= 0) return PKV_OK;
  if (units > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  // programmatic dependent launch: see the wait at the kernel's entry
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem::alloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, paged_attention_grouped_kernel<G, BS, FUSED>, mk, mv, p,
                            shared_splits, own_splits, shared_stride) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

// Host launchers for one block size (defined in attention_bs*.cu).
template <int BS>
int launch_split(int G, bool fused, const CUtensorMap& mk, const CUtensorMap& mv, const Params& p,
                 int private_splits, cudaStream_t stream);
template <int BS>
int launch_grouped_step(int G, bool fused, const CUtensorMap& mk, const CUtensorMap& mv,
                        const Params& p, int shared_splits, int own_splits, int shared_stride,
                        cudaStream_t stream);

#define PKV_CASE_G(GV, BSV)                                                                   \
  case GV:                                                                                    \
    return fused ? launch_one<GV, BSV, true>(mk, mv, p, ps, st)                               \
                 : launch_one<GV, BSV, false>(mk, mv, p, ps, st);
#define PKV_CASE_GROUPED(GV, BSV)                                                             \
  case GV:                                                                                    \
    return fused ? launch_grouped<GV, BSV, true>(mk, mv, p, ss, os, sk, st)                   \
                 : launch_grouped<GV, BSV, false>(mk, mv, p, ss, os, sk, st);
#define PKV_DEFINE_LAUNCH_SPLIT(BSV)                                                          \
  template <>                                                                                 \
  int launch_split<BSV>(int G, bool fused, const CUtensorMap& mk, const CUtensorMap& mv,      \
                        const Params& p, int ps, cudaStream_t st) {                           \
    switch (G) {                                                                              \
      PKV_CASE_G(1, BSV)                                                                      \
      PKV_CASE_G(2, BSV)                                                                      \
      PKV_CASE_G(4, BSV)                                                                      \
      PKV_CASE_G(8, BSV)                                                                      \
      default: return PKV_ERR_UNSUPPORTED;                                                    \
    }                                                                                         \
  }                                                                                           \
  template <>                                                                                 \
  int launch_grouped_step<BSV>(int G, bool fused, const CUtensorMap& mk,                      \
                               const CUtensorMap& mv, const Params& p, int ss, int os,        \
                               int sk, cudaStream_t st) {                                     \
    switch (G) {                                                                              \
      PKV_CASE_GROUPED(1, BSV)                                                                \
      PKV_CASE_GROUPED(2, BSV)                                                                \
      PKV_CASE_GROUPED(4, BSV)                                                                \
      PKV_CASE_GROUPED(8, BSV)                                                                \
      default: return PKV_ERR_UNSUPPORTED;                                                    \
    }                                                                                         \
  }

}  // namespace attn
}  // namespace pkv
