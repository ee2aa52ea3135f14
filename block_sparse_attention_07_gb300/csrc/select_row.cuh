// Block selection of one row by one warp ("MiniMax M3 vLLM サポート：…",
// section "MSA 実行プロセス", step 2: top-k blocks with local_blocks=1;
// "MiniMax-M3.1-Flash Day-0 対応", section "MSAの仕組み": 16 blocks of 128
// tokens). Used where the selection runs inside another kernel (the fused
// select + sparse-GQA launch); the standalone selection kernel uses a whole CTA
// per row with the same keys.
//
// Candidate n of a row becomes the 64-bit key (order-preserving image of its
// fp32 score) << 32 | ~n: "higher score, then lower block id" is plain
// unsigned order and every key is distinct.
#pragma once

#include "msa_device.cuh"

namespace msa {

// Monotone map fp32 -> uint32 (NaN is treated as -inf).
__device__ __forceinline__ uint32_t order_key(float s) {
  if (s != s) s = -INFINITY;
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t make_key(float s, int n) {
  return (static_cast<uint64_t>(order_key(s)) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - n);
}

__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v), src);
  const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

constexpr int kWarpSurvCap = 128;   // survivors a warp stages in shared memory
constexpr int kWarpBatch = 8;       // candidates per lane loaded together (independent loads in flight)

// Keys of candidates base + lane + 32 u, u < kWarpBatch (0 past the row's end).
__device__ __forceinline__ void warp_load_keys(const float* sr, int ell, int base, int lane,
                                               uint64_t (&k)[kWarpBatch]) {
  float v[kWarpBatch];
#pragma unroll
  for (int u = 0; u < kWarpBatch; ++u) {
    const int n = base + lane + 32 * u;
    v[u] = n < ell ? sr[n] : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kWarpBatch; ++u) {
    const int n = base + lane + 32 * u;
    k[u] = n < ell ? make_key(v[u], n) : 0ull;
  }
}

// The warp's keys >= t compacted (in candidate order) into surv; returns their
// number (only the first kWarpSurvCap are stored).
__device__ __forceinline__ int warp_collect(const float* sr, int ell, uint64_t t, uint64_t* surv, int lane) {
  int s = 0;
  for (int base = 0; base < ell; base += 32 * kWarpBatch) {
    uint64_t k[kWarpBatch];
    warp_load_keys(sr, ell, base, lane, k);
#pragma unroll
    for (int u = 0; u < kWarpBatch; ++u) {
      const bool keep = k[u] != 0ull && k[u] >= t;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const int at = s + __popc(m & ((1u << lane) - 1u));
        if (at < kWarpSurvCap) surv[at] = k[u];
      }
      s += __popc(m);
    }
  }
  return s;
}

// out[0..K) = the ascending ids of the top take = min(K - 1, ell) candidates
// n < ell of the score row sr, plus the local block ell, then -1 padding.
// surv: kWarpSurvCap words, chosen: 16 ints of this warp's shared memory.
static __device__ void warp_select_row(const float* sr, int ell, int K, int32_t* out, uint64_t* surv, int* chosen,
                                       int lane) {
  const int take = min(K - 1, ell);
  if (take > 0) {
    // 1. lane maxima; the take-th largest of them (when at least take lanes
    //    hold candidates) has take keys at or above it, so it bounds the row's
    //    take-th largest key from below
    uint64_t tmax = 0ull;
    for (int base = 0; base < ell; base += 32 * kWarpBatch) {
      uint64_t k[kWarpBatch];
      warp_load_keys(sr, ell, base, lane, k);
#pragma unroll
      for (int u = 0; u < kWarpBatch; ++u) tmax = k[u] > tmax ? k[u] : tmax;
    }
    uint64_t t = 0ull;
    if (__popc(__ballot_sync(0xffffffffu, tmax != 0ull)) >= take) {
      int rank = 0;
      for (int q = 0; q < 32; ++q) rank += shfl64(tmax, q) > tmax ? 1 : 0;
      const uint32_t hit = __ballot_sync(0xffffffffu, tmax != 0ull && rank == take - 1);
      t = shfl64(tmax, __ffs(hit) - 1);
    }
    // 2. survivors
    int s = warp_collect(sr, ell, t, surv, lane);
    if (s > kWarpSurvCap) {
      // exact take-th largest key by a bitwise search over the row
      uint64_t tx = 0ull;
      for (int bit = 63; bit >= 0; --bit) {
        const uint64_t c = tx | (1ull << bit);
        int cnt = 0;
        for (int base = 0; base < ell; base += 32 * kWarpBatch) {
          uint64_t k[kWarpBatch];
          warp_load_keys(sr, ell, base, lane, k);
#pragma unroll
          for (int u = 0; u < kWarpBatch; ++u) cnt += (k[u] != 0ull && k[u] >= c) ? 1 : 0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        if (cnt >= take) tx = c;
      }
      s = warp_collect(sr, ell, tx, surv, lane);   // exactly take keys
    }
    __syncwarp();
    // 3. a survivor's rank is the number of survivors above it
    for (int i = lane; i < s; i += 32) {
      const uint64_t ki = surv[i];
      int r = 0;
      for (int m = 0; m < s; ++m) r += surv[m] > ki ? 1 : 0;
      if (r < take) chosen[r] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(ki));
    }
    __syncwarp();
  }
  // 4. ascending ids of the chosen blocks plus the local block
  const int mine = lane < take ? chosen[lane] : (lane == take ? ell : INT32_MAX);
  int pos = 0;
  for (int q = 0; q <= take; ++q) pos += __shfl_sync(0xffffffffu, mine, q) < mine ? 1 : 0;
  if (lane <= take) out[pos] = mine;
  for (int e = take + 1 + lane; e < K; e += 32) out[e] = -1;
  __syncwarp();
}

}  // namespace msa
