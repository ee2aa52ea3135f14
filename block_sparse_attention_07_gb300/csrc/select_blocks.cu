// Stage 2 of MSA decode: top-k block selection with the local block kept.
//
// "MiniMax M3 vLLM サポート：…" (agentlenshq.com), section "MSA 実行プロセス",
// step 2: the top-k blocks are chosen, local_blocks=1 keeping the block that
// holds the query token. "MiniMax-M3.1-Flash Day-0 対応", section "MSAの仕組み":
// 16 blocks of 128 tokens, at most 2,048 keys per query.
//
// One warp per (request, position, index head). Each candidate becomes a
// 64-bit key (order-preserving image of the fp32 score << 32 | ~block id), so
// "higher score, then lower id" is plain unsigned order and the selection is
// exact. Every lane keeps its own sorted top-(k-1) of a strided slice; the
// warp then pops the k-1 largest heads with two 32-bit warp max reductions
// each, adds the local block and writes the ids in ascending order.
#include "msa_internal.h"

namespace msa {

constexpr int kMaxTop = 15;  // topk - 1 for topk <= 16
constexpr uint32_t kFullMask = 0xffffffffu;

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

__global__ void __launch_bounds__(256) select_blocks_kernel(SelParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
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

  uint64_t top[kMaxTop];
#pragma unroll
  for (int q = 0; q < kMaxTop; ++q) top[q] = 0ull;  // below every real key
  for (int n = lane; n < ell; n += 32) {
    const uint64_t key = (static_cast<uint64_t>(order_key(sr[n])) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - n);
    if (key > top[kMaxTop - 1]) {
#pragma unroll
      for (int q = kMaxTop - 1; q > 0; --q) top[q] = key > top[q - 1] ? top[q - 1] : (key > top[q] ? key : top[q]);
      top[0] = key > top[0] ? key : top[0];
    }
  }

  int mine = -1;
  for (int r = 0; r < take; ++r) {
    const uint32_t hi = static_cast<uint32_t>(top[0] >> 32);
    const uint32_t mhi = __reduce_max_sync(kFullMask, hi);
    const uint32_t lo = hi == mhi ? static_cast<uint32_t>(top[0]) : 0u;
    const uint32_t mlo = __reduce_max_sync(kFullMask, lo);
    if (hi == mhi && lo == mlo) {
#pragma unroll
      for (int q = 0; q < kMaxTop - 1; ++q) top[q] = top[q + 1];
      top[kMaxTop - 1] = 0ull;
    }
    if (lane == r) mine = static_cast<int>(0xFFFFFFFFu - mlo);
  }
  if (lane == take) mine = ell;
  // Ascending order of the take+1 ids held by lanes 0..take.
  int rank = 0;
  for (int q = 0; q <= take; ++q) {
    const int other = __shfl_sync(kFullMask, mine, q);
    rank += (lane <= take && other < mine) ? 1 : 0;
  }
  if (lane <= take) out[rank] = mine;
  for (int e = take + 1 + lane; e < p.K; e += 32) out[e] = -1;
}

cudaError_t launch_select_blocks(const SelectArgs& a, cudaStream_t stream, DispatchRecord* rec) {
  SelParams p{a.scores, a.seq_lens, a.selected, a.flags, a.B, a.Q, a.I, a.NB, a.K};
  const int64_t rows = static_cast<int64_t>(a.B) * a.Q * a.I;
  const int64_t grid = (rows + 7) / 8;
  select_blocks_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(p);
  rec->set("select_blocks warp_topk grid=%lld block=256 rows=%lld topk=%d", static_cast<long long>(grid),
           static_cast<long long>(rows), a.K);
  return cudaGetLastError();
}

}  // namespace msa
