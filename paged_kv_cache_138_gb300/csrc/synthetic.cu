// Synthetic inputs drawn on the device: standard-normal fp16 values for the
// q / K / V rows a decode server's model would produce.  No part of paged
// attention or of the cache kernels; benchmarks and the model-less serving
// driver use it so that drawing a step's values costs one short launch.
//
// Element j of the stream keyed by `seed` (j counted from 0 across calls via
// `offset`): pair p = j / 2 takes the p-th output of SplitMix64 started at
// state `seed` (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014: state += 0x9e3779b97f4a7c15, then the
// variant-13 finaliser), splits its 64 bits into u1 = (bits 40..63 + 1) / 2^24
// in (0, 1] and u2 = bits 16..39 / 2^24 in [0, 1), and applies the Box-Muller
// transform (Box and Muller, 1958): r = sqrt(-2 ln u1), element 2p gets
// r cos(2 pi u2) and element 2p + 1 gets r sin(2 pi u2), rounded to fp16.
// A thread draws each pair once and stores 8 values with one 16-byte store.
#include <algorithm>

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {
namespace synth {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;  // one 16-byte store

__device__ __forceinline__ uint64_t splitmix64_output(uint64_t seed, uint64_t p) {
  uint64_t z = seed + (p + 1) * 0x9e3779b97f4a7c15ull;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// Both values of pair p.  The angle is taken as 2 pi u2 - pi, inside the
// interval where the hardware sine/cosine is accurate to ~2^-21 absolute, and
// the signs flipped back: cos(t + pi) = -cos t, sin(t + pi) = -sin t.
__device__ __forceinline__ float2 normal_pair(uint64_t seed, uint64_t p) {
  const uint64_t w = splitmix64_output(seed, p);
  const float u1 = static_cast<float>((w >> 40) + 1) * (1.0f / 16777216.0f);
  const float u2 = static_cast<float>((w >> 16) & 0xFFFFFFull) * (1.0f / 16777216.0f);
  const float r = sqrtf(-2.0f * logf(u1));   // logf(u1) <= 0 for u1 <= 1
  float s, c;
  __sincosf(6.28318530718f * u2 - 3.14159265359f, &s, &c);
  return make_float2(-r * c, -r * s);
}

__device__ __forceinline__ float normal_at(uint64_t seed, uint64_t j) {
  const float2 v = normal_pair(seed, j >> 1);
  return (j & 1) ? v.y : v.x;
}

__global__ void __launch_bounds__(kThreads)
    fill_normal_f16_kernel(__half* __restrict__ dst, int64_t n, uint64_t seed, uint64_t offset) {
  // a programmatically dependent launch that follows (the attention kernel)
  // may place its CTAs while this grid runs; it reads nothing before this
  // grid has completed
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads * kPerThread;
  for (int64_t base = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) * kPerThread;
       base < n; base += stride) {
    if (base + kPerThread <= n) {
      __align__(16) __half2 h[kPerThread / 2];
      if ((offset & 1) == 0) {         // the thread's elements are whole pairs
        const uint64_t p0 = (offset + base) >> 1;
#pragma unroll
        for (int e = 0; e < kPerThread / 2; ++e) h[e] = __float22half2_rn(normal_pair(seed, p0 + e));
      } else {
#pragma unroll
        for (int e = 0; e < kPerThread / 2; ++e)
          h[e] = __floats2half2_rn(normal_at(seed, offset + base + 2 * e),
                                   normal_at(seed, offset + base + 2 * e + 1));
      }
      *reinterpret_cast<uint4*>(dst + base) = *reinterpret_cast<const uint4*>(h);
    } else {
      for (int64_t e = base; e < n; ++e) dst[e] = __float2half_rn(normal_at(seed, offset + e));
    }
  }
}

}  // namespace synth
}  // namespace pkv

extern "C" int pkv_fill_normal_f16(void* dst, int64_t n, uint64_t seed, uint64_t offset,
                                   void* stream) {
  using namespace pkv::synth;
  if (n < 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!dst || (reinterpret_cast<uintptr_t>(dst) & 15) != 0) return PKV_ERR_INVALID_ARG;
  const int64_t threads = (n + kPerThread - 1) / kPerThread;
  // at most 8 resident 256-thread CTAs on each of the 152 SMs; more work loops
  const int64_t blocks = std::min<int64_t>((threads + kThreads - 1) / kThreads, 152 * 8);
  fill_normal_f16_kernel<<<static_cast<unsigned>(blocks), kThreads, 0,
                           static_cast<cudaStream_t>(stream)>>>(static_cast<__half*>(dst), n,
                                                                seed, offset);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
