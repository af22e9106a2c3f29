// philox.cuh -- Philox4x64-10 counter-based generator (Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC'11), written on the device from
// the published definition: ten rounds of the 4x64 Philox S-box, the key bumped by a
// Weyl sequence between rounds.
#pragma once

#include <stdint.h>

namespace dfs {

__device__ __forceinline__ void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull;
  constexpr uint64_t kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull;
  constexpr uint64_t kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t lo0 = kM0 * c[0], hi0 = __umul64hi(kM0, c[0]);
    const uint64_t lo1 = kM1 * c[2], hi1 = __umul64hi(kM1, c[2]);
    const uint64_t n0 = hi1 ^ c[1] ^ k0;
    const uint64_t n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// Uniform (2j+1) * 2^-24 with j = the top 23 bits of the word: exact in fp32.
__device__ __forceinline__ float u01_from_word(uint64_t w) {
  return static_cast<float>(2u * static_cast<uint32_t>(w >> 41) + 1u) * 0x1p-24f;
}

// Uniform of Philox stream s at draft position t of request b: counter (0, t, b, s), word 0.
// Streams: 0 the acceptance tests, 1 the redraws, 3 the path draws.
__device__ __forceinline__ float uniform_stream(uint64_t seed, int b, int t, uint64_t s) {
  uint64_t c[4] = {0ull, static_cast<uint64_t>(t), static_cast<uint64_t>(b), s};
  philox4x64_10(c, seed, 0ull);
  return u01_from_word(c[0]);
}

// Accept-test uniform of draft position t of request b: counter (0, t, b, 0), word 0.
__device__ __forceinline__ float uniform_accept(uint64_t seed, int b, int t) {
  return uniform_stream(seed, b, t, 0ull);
}

// The redraw's one uniform for draft position t of request b (the draw from row t - 1, or
// from the bonus row when t = L): counter (0, t, b, 1), word 0.
__device__ __forceinline__ float uniform_redraw(uint64_t seed, int b, int t) {
  return uniform_stream(seed, b, t, 1ull);
}

// Path-draw uniform of the sampled traversal at draft position t of request b: counter
// (0, t, b, 3), word 0.
__device__ __forceinline__ float uniform_path(uint64_t seed, int b, int t) {
  return uniform_stream(seed, b, t, 3ull);
}

}  // namespace dfs
