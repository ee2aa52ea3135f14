// Stage 2 of MSA decode: top-k block selection with the local block kept.
//
// "MiniMax M3 vLLM サポート：…" (agentlenshq.com), section "MSA 実行プロセス",
// step 2: the top-k blocks are chosen, local_blocks=1 keeping the block that
// holds the query token. "MiniMax-M3.1-Flash Day-0 対応", section "MSAの仕組み":
// 16 blocks of 128 tokens, at most 2,048 keys per query.
//
// One 256-thread CTA per (request, position, index head). Each candidate n
// becomes the 64-bit key (order-preserving image of its fp32 score) << 32 | ~n,
// so "higher score, then lower block id" is plain unsigned order, every key is
// distinct and the selection is exact.
//   1. Every thread takes the candidates n = tid + 256 i and keeps their
//      largest key. In a warp whose lanes hold at least `take` candidates, the
//      take-th largest lane maximum T_w has `take` keys of that warp at or above
//      it, so the row's take-th largest key is >= T_w; T = max_w T_w is a lower
//      bound for it.
//   2. The keys >= T (typically take to 2 x take of them) are appended to a
//      shared buffer. (If more than the buffer holds, an exact bitwise search
//      for the take-th largest key replaces T.)
//   3. A survivor's rank is the number of survivors above it; ranks below
//      `take` are the chosen blocks.
//   4. The chosen ids plus the local block are written in ascending order.
#include "msa_internal.h"
#include "select_row.cuh"

namespace msa {

constexpr uint32_t kFullMask = 0xffffffffu;
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBatch = 8;          // candidates per thread per batch of loads
constexpr int kSurvCap = 512;

struct SelParams {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* selected;
  uint32_t* flags;
  int B, Q, I, NB, K;
};

// Loads this thread's keys of batch `base` (0 where there is no candidate).
__device__ __forceinline__ void load_batch(const float* row, int ell, int base, uint64_t (&k)[kBatch]) {
  float v[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int n = base + static_cast<int>(threadIdx.x) + kSelThreads * u;
    v[u] = n < ell ? __ldg(row + n) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int n = base + static_cast<int>(threadIdx.x) + kSelThreads * u;
    k[u] = n < ell ? make_key(v[u], n) : 0ull;
  }
}

// Appends every key >= t to buf through the shared counter *cnt (stores at most kSurvCap).
__device__ void collect(const float* row, int ell, uint64_t t, uint64_t* buf, int* cnt) {
  for (int base = 0; base < ell; base += kSelThreads * kBatch) {
    uint64_t k[kBatch];
    load_batch(row, ell, base, k);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (k[u] != 0ull && k[u] >= t) {
        const int at = atomicAdd(cnt, 1);
        if (at < kSurvCap) buf[at] = k[u];
      }
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) select_blocks_kernel(SelParams p) {
  __shared__ uint64_t surv[kSurvCap];
  __shared__ uint64_t wthr[kSelWarps];
  __shared__ int chosen[16];
  __shared__ int cnt;
  __shared__ int tally;
  griddep_launch_dependents();
  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int b = static_cast<int>(row / (static_cast<int64_t>(p.Q) * p.I));
  const int j = static_cast<int>((row / p.I) % p.Q);
  int32_t* out = p.selected + row * p.K;
  const int L = p.seq_lens[b];
  if (L < p.Q || L > p.NB * kBlock || L < 1) {
    if (tid == 0) set_flag(p.flags, MSA_FLAG_BAD_SEQLEN);
    for (int e = tid; e < p.K; e += kSelThreads) out[e] = -1;
    return;
  }
  const int ell = (L - p.Q + j) / kBlock;        // local block = number of candidates
  const int take = min(p.K - 1, ell);
  const float* sr = p.scores + row * p.NB;

  if (take > 0) {
    if (tid == 0) cnt = 0;
    // 1. per-thread maximum, then each warp's take-th largest lane maximum
    uint64_t tmax = 0ull;
    for (int base = 0; base < ell; base += kSelThreads * kBatch) {
      uint64_t k[kBatch];
      load_batch(sr, ell, base, k);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) tmax = k[u] > tmax ? k[u] : tmax;
    }
    const int lanes_with = __popc(__ballot_sync(kFullMask, tmax != 0ull));
    uint64_t tw = 0ull;
    if (lanes_with >= take) {
      int rank = 0;
      for (int q = 0; q < 32; ++q) rank += shfl64(tmax, q) > tmax ? 1 : 0;
      const uint32_t hit = __ballot_sync(kFullMask, tmax != 0ull && rank == take - 1);
      tw = shfl64(tmax, __ffs(hit) - 1);
    }
    if (lane == 0) wthr[warp] = tw;
    __syncthreads();
    uint64_t t = 0ull;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) t = wthr[w] > t ? wthr[w] : t;

    // 2. survivors
    collect(sr, ell, t, surv, &cnt);
    __syncthreads();
    int s = cnt;
    if (s > kSurvCap) {
      // exact take-th largest key by a bitwise search over the row
      uint64_t tx = 0ull;
      for (int bit = 63; bit >= 0; --bit) {
        const uint64_t c = tx | (1ull << bit);
        if (tid == 0) tally = 0;
        __syncthreads();
        int mine = 0;
        for (int base = 0; base < ell; base += kSelThreads * kBatch) {
          uint64_t k[kBatch];
          load_batch(sr, ell, base, k);
#pragma unroll
          for (int u = 0; u < kBatch; ++u) mine += (k[u] != 0ull && k[u] >= c) ? 1 : 0;
        }
        if (mine) atomicAdd(&tally, mine);
        __syncthreads();
        if (tally >= take) tx = c;
        __syncthreads();
      }
      if (tid == 0) cnt = 0;
      __syncthreads();
      collect(sr, ell, tx, surv, &cnt);
      __syncthreads();
      s = cnt;
    }
    // 3. rank of each survivor among the survivors
    for (int i = tid; i < s; i += kSelThreads) {
      const uint64_t ki = surv[i];
      int r = 0;
      for (int m = 0; m < s; ++m) r += surv[m] > ki ? 1 : 0;
      if (r < take) chosen[r] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(ki));
    }
    __syncthreads();
  }
  // 4. ascending ids of the take chosen blocks plus the local block
  if (warp == 0) {
    const int mine = lane < take ? chosen[lane] : (lane == take ? ell : INT32_MAX);
    int pos = 0;
    for (int q = 0; q <= take; ++q) pos += __shfl_sync(kFullMask, mine, q) < mine ? 1 : 0;
    if (lane <= take) out[pos] = mine;
  }
  for (int e = take + 1 + tid; e < p.K; e += kSelThreads) out[e] = -1;
}

cudaError_t launch_select_blocks(const SelectArgs& a, cudaStream_t stream, DispatchRecord* rec) {
  SelParams p{a.scores, a.seq_lens, a.selected, a.flags, a.B, a.Q, a.I, a.NB, a.K};
  const int64_t rows = static_cast<int64_t>(a.B) * a.Q * a.I;
  const cudaError_t err =
      launch_pdl(select_blocks_kernel, dim3(static_cast<unsigned>(rows)), dim3(kSelThreads), 0, stream, p);
  if (err != cudaSuccess) return err;
  rec->set("select_blocks threshold_rank cta_per_row grid=%lld block=%d topk=%d", static_cast<long long>(rows),
           kSelThreads, a.K);
  return cudaGetLastError();
}

}  // namespace msa
