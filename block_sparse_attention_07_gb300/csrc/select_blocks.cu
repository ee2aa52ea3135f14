// Stage 2 of MSA decode: top-k block selection with the local block kept.
//
// "MiniMax M3 vLLM サポート：…" (agentlenshq.com), section "MSA 実行プロセス",
// step 2: the top-k blocks are chosen, local_blocks=1 keeping the block that
// holds the query token. "MiniMax-M3.1-Flash Day-0 対応", section "MSAの仕組み":
// 16 blocks of 128 tokens, at most 2,048 keys per query.
//
// One warp per (request, position, index head). Each candidate n becomes the
// 64-bit key (order-preserving image of its fp32 score) << 32 | ~n, so "higher
// score, then lower block id" is plain unsigned order, every key is distinct
// and the selection is exact.
//   1. One pass over the row: each lane keeps the largest key of its strided
//      slice. The take-th largest of the 32 lane maxima, T0, has at least
//      `take` keys >= it, so the answer lies in {key >= T0}.
//   2. A second pass appends the keys >= T0 to a per-warp buffer in shared
//      memory (typically a few dozen).
//   3. Each survivor's rank is the number of survivors above it; ranks below
//      `take` are the chosen blocks. (If the survivors overflow the buffer, an
//      exact bitwise search for the take-th largest key replaces T0.)
//   4. The chosen ids plus the local block are written in ascending order.
#include "msa_internal.h"

namespace msa {

constexpr uint32_t kFullMask = 0xffffffffu;
constexpr int kSelWarps = 4;
constexpr int kSurvCap = 256;

struct SelParams {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* selected;
  uint32_t* flags;
  int B, Q, I, NB, K;
};

// Monotone map fp32 -> uint32 (NaN is treated as -inf).
__device__ __forceinline__ uint32_t order_key(float s) {
  if (s != s) s = -INFINITY;
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t make_key(float s, int n) {
  return (static_cast<uint64_t>(order_key(s)) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - n);
}

__device__ __forceinline__ uint64_t cand_key(const float* row, int n) { return make_key(__ldg(row + n), n); }

__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(kFullMask, static_cast<uint32_t>(v), src);
  const uint32_t hi = __shfl_sync(kFullMask, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Number of keys >= t in the row (warp-wide).
__device__ int count_at_least(const float* row, int ell, uint64_t t, int lane) {
  int c = 0;
  for (int n = lane; n < ell; n += 32) c += cand_key(row, n) >= t ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFullMask, c, o);
  return c;
}

// Appends the row's keys >= t to buf (at most cap are stored); returns how many there are.
__device__ int collect_at_least(const float* row, int ell, uint64_t t, int lane, uint64_t* buf, int cap) {
  int s = 0;
  for (int base = 0; base < ell; base += 32) {
    const int n = base + lane;
    const uint64_t k = n < ell ? cand_key(row, n) : 0ull;
    const bool keep = n < ell && k >= t;
    const uint32_t bal = __ballot_sync(kFullMask, keep);
    const int at = s + __popc(bal & ((1u << lane) - 1u));
    if (keep && at < cap) buf[at] = k;
    s += __popc(bal);
  }
  return s;
}

__global__ void __launch_bounds__(32 * kSelWarps) select_blocks_kernel(SelParams p) {
  __shared__ uint64_t surv[kSelWarps][kSurvCap];
  __shared__ int chosen[kSelWarps][16];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kSelWarps + wib;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Q * p.I;
  if (row >= rows) return;
  const int b = static_cast<int>(row / (static_cast<int64_t>(p.Q) * p.I));
  const int j = static_cast<int>((row / p.I) % p.Q);
  int32_t* out = p.selected + row * p.K;
  const int L = p.seq_lens[b];
  if (L < p.Q || L > p.NB * kBlock || L < 1) {
    if (lane == 0) set_flag(p.flags, MSA_FLAG_BAD_SEQLEN);
    for (int e = lane; e < p.K; e += 32) out[e] = -1;
    return;
  }
  const int ell = (L - p.Q + j) / kBlock;        // local block = number of candidates
  const int take = min(p.K - 1, ell);
  const float* sr = p.scores + row * p.NB;

  if (take > 0) {
    // 1. lane maxima (16 loads in flight per lane)
    uint64_t lmax = 0ull;
    for (int base = 0; base < ell; base += 32 * 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int n = base + lane + 32 * u;
        v[u] = n < ell ? __ldg(sr + n) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int n = base + lane + 32 * u;
        const uint64_t k = make_key(v[u], n);
        if (n < ell && k > lmax) lmax = k;
      }
    }
    // the take-th largest lane maximum (real keys are distinct and > 0)
    int rank = 0;
    for (int q = 0; q < 32; ++q) rank += shfl64(lmax, q) > lmax ? 1 : 0;
    const uint32_t hit = __ballot_sync(kFullMask, rank == take - 1);
    uint64_t t0 = shfl64(lmax, __ffs(hit) - 1);

    // 2. survivors
    int s = collect_at_least(sr, ell, t0, lane, surv[wib], kSurvCap);
    if (s > kSurvCap) {
      // exact take-th largest key by a bitwise search, then exactly `take` survivors
      uint64_t t = 0ull;
      for (int bit = 63; bit >= 0; --bit) {
        const uint64_t c = t | (1ull << bit);
        if (count_at_least(sr, ell, c, lane) >= take) t = c;
      }
      s = collect_at_least(sr, ell, t, lane, surv[wib], kSurvCap);
    }
    __syncwarp();
    // 3. rank of each survivor among the survivors
    for (int i = lane; i < s; i += 32) {
      const uint64_t ki = surv[wib][i];
      int r = 0;
      for (int m = 0; m < s; ++m) r += surv[wib][m] > ki ? 1 : 0;
      if (r < take) chosen[wib][r] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(ki));
    }
    __syncwarp();
  }
  // 4. ascending ids of the take chosen blocks plus the local block
  const int mine = lane < take ? chosen[wib][lane] : (lane == take ? ell : INT32_MAX);
  int pos = 0;
  for (int q = 0; q <= take; ++q) pos += __shfl_sync(kFullMask, mine, q) < mine ? 1 : 0;
  if (lane <= take) out[pos] = mine;
  for (int e = take + 1 + lane; e < p.K; e += 32) out[e] = -1;
}

cudaError_t launch_select_blocks(const SelectArgs& a, cudaStream_t stream, DispatchRecord* rec) {
  SelParams p{a.scores, a.seq_lens, a.selected, a.flags, a.B, a.Q, a.I, a.NB, a.K};
  const int64_t rows = static_cast<int64_t>(a.B) * a.Q * a.I;
  const int64_t grid = (rows + kSelWarps - 1) / kSelWarps;
  select_blocks_kernel<<<static_cast<unsigned>(grid), 32 * kSelWarps, 0, stream>>>(p);
  rec->set("select_blocks threshold_rank grid=%lld block=%d rows=%lld topk=%d", static_cast<long long>(grid),
           32 * kSelWarps, static_cast<long long>(rows), a.K);
  return cudaGetLastError();
}

}  // namespace msa
