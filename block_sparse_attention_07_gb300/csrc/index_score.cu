// Stage 1 of MSA decode: block scoring by the index heads.
//
// "MiniMax M3 vLLM サポート：…" (agentlenshq.com), section "MSA 実行プロセス",
// step 1: a small index head scores every candidate KV block. The block score
// is the maximum over the block's tokens of s_t * (q_idx . k_t). Following
// "vLLM、AMD Instinct MI355X上で…" (news.ainew.jp), question 2, each index key
// is loaded once for all query positions of its request, and no positive
// score scale is applied.
//
// FP8 / NVFP4 paths: a persistent kernel, one CTA per SM (two for NVFP4 keys,
// whose pages are half the size). Work units are the (request, block) pairs
// that some position of the request can select; seven eighths of them are
// split evenly over the CTAs and the rest handed out at run time (below).
// A producer thread streams each unit's page (I heads x 128 tokens x 128 B of
// E4M3 keys, contiguous, plus I x 512 B of per-token scales) into a ring of
// shared-memory stages with bulk copies completed on mbarriers. One consumer
// warp group per index head (each warp takes a share of the page's 128 tokens)
// turns 16 tokens x 16 dims of keys into an fp16 mma A
// fragment (cvt e4m3x2 -> f16x2 is exact), multiplies by the Q positions'
// index queries (the 8 columns of m16n8k16; fp16 after an exact power-of-two
// rescale of each query row), applies the per-token scale and keeps the running
// max. The dims a thread feeds to the mma are a fixed permutation of 0..127,
// applied identically to keys and queries, so each thread reads whole 16-byte
// runs of a key row. The warps of a head merge their column maxima through a
// shared-memory slot per stage: the last to arrive (by a ticket counter) writes
// the score, so none waits for another.
#include <atomic>

#include "insert_rows.cuh"

namespace msa {

constexpr int kIdxStages = 3;       // 66.5 KB pages (FP8 keys, 4 heads), one CTA per SM
constexpr int kIdxStagesFp4 = 3;    // 36 KB pages (NVFP4 keys, 4 heads), two CTAs per SM
constexpr int kFp4CtasPerSm = 2;    // two independent pipelines per SM hide more of the per-page latency
constexpr int kMaxIdxHeads = 4;
constexpr int kWarpsPerHead = 2;    // consumer warps per index head (each takes a share of the page's tokens)
constexpr int kTilesPerWarp = kBlock / 16 / kWarpsPerHead;
constexpr int kIdxThreads = 32 * (1 + kWarpsPerHead * kMaxIdxHeads);
constexpr uint32_t kFull = 0xffffffffu;

struct IdxParams {
  const void* q;
  const void* keys;
  const void* scale;        // fp32 per token (FP8 keys) or E4M3 per 16 values (NVFP4 keys)
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* scores;
  uint32_t* flags;
  float global_scale;       // NVFP4 keys: fp32 per-tensor scale
  int B, Q, I, NB, P;
  int ins_on;               // 1: also insert the step's new tokens (one per request, Q = 1)
  uint64_t epoch;           // grows from call to call; tags the work-queue words
  int slot;                 // the call's work-queue slot
  InsertParams ins;
};

// Work split of the FP8 / NVFP4 kernels: the first units are divided evenly
// over the CTAs; the last 1 / kDynShare of them are handed out at run time in
// chunks of kDynChunk consecutive units, so CTAs whose pages arrived faster
// take more and all end together. The queue is one pair of words per launch
// slot: the next chunk and the CTAs that have finished, each holding
// epoch << kCountBits | count. Epochs grow from call to call, so each CTA first
// raises both words to at least that base (a word left by an earlier call
// restarts from 0) and then counts with plain atomic adds. The CTA that
// finishes last sets both words back to the base, so a replay of a captured
// graph (whose epoch is fixed at capture) starts from 0. Direct calls take the
// slots 0 .. kQueueSlots - 1 in turn and launches captured into a graph the
// slots after them, so a direct call never raises a captured launch's words.
constexpr int kDynShare = 8;
constexpr int kDynChunk = 2;
constexpr int kQueueSlots = 64;
constexpr int kCountBits = 24;        // counts stay below 2^23 (units / kDynChunk, CTAs)
__device__ unsigned long long g_idx_queue[2 * kQueueSlots][2];

__device__ __forceinline__ unsigned long long epoch_base(uint64_t epoch) {
  return static_cast<unsigned long long>(epoch) << kCountBits;
}
// The count at w before adding one, or -1 if the word belongs to another epoch (flagged).
__device__ __forceinline__ int64_t epoch_fetch_add(unsigned long long* w, uint64_t epoch, uint32_t* flags) {
  const unsigned long long old = atomicAdd(w, 1ull);
  if ((old >> kCountBits) != static_cast<unsigned long long>(epoch)) {
    set_flag(flags, MSA_FLAG_TIMEOUT);
    return -1;
  }
  return static_cast<int64_t>(old & ((1ull << kCountBits) - 1));
}

// The insert fused into the index launch (one query position): token t is
// request t's token at position L_t - 1, so it lands in the request's local
// block, which this launch never scores. A token whose slot is not that
// position is flagged (MSA_FLAG_BAD_SLOT) and skipped; a negative slot is a
// padding token and is skipped silently. The consumer warps take the
// (token, head) rows before their first page arrives; the attention that
// reads the new K/V waits for this whole launch.
__device__ __noinline__ void fused_insert(const IdxParams& p, int64_t cw, int64_t ncw, int lane) {
  const InsertParams& ins = p.ins;
  const int64_t total = static_cast<int64_t>(ins.T) * ins.G;
  for (int64_t w = cw; w < total; w += ncw) {
    const int t = static_cast<int>(w / ins.G), h = static_cast<int>(w % ins.G);
    const int64_t slot = ins.slots[t];
    if (slot < 0) continue;
    const int L = p.seq_lens[t];
    bool ok = L >= 1 && L <= p.NB * kBlock;
    if (ok) {
      const int page = p.block_table[static_cast<int64_t>(t) * p.NB + (L - 1) / kBlock];
      ok = page >= 0 && page < p.P && slot == static_cast<int64_t>(page) * kBlock + (L - 1) % kBlock;
    }
    if (!ok) {
      if (lane == 0) set_flag(p.flags, MSA_FLAG_BAD_SLOT);
      continue;
    }
    insert_row(ins, t, h, lane);
  }
}

// Blocks of request b that some query position can select: every n < l_last,
// l_last being the local block of the last position. -1 for an invalid length.
__device__ __forceinline__ int units_of(int L, int Q, int NB) {
  if (L < Q || L > NB * kBlock || L < 1) return -1;
  return (L - 1) / kBlock;
}

// Exclusive prefix of units_of over the batch, computed by one warp into pref[0..B].
__device__ void build_prefix(const IdxParams& p, int* pref, bool report) {
  const int lane = threadIdx.x & 31;
  int run = 0;
  if (lane == 0) pref[0] = 0;
  for (int base = 0; base < p.B; base += 32) {
    const int b = base + lane;
    int u = 0;
    if (b < p.B) {
      u = units_of(p.seq_lens[b], p.Q, p.NB);
      if (u < 0) {
        if (report) set_flag(p.flags, MSA_FLAG_BAD_SEQLEN);
        u = 0;
      }
    }
    int incl = u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    if (b < p.B) pref[b + 1] = run + incl;
    run += __shfl_sync(kFull, incl, 31);
  }
}

// Largest b with pref[b] <= u (u < pref[B]).
__device__ __forceinline__ int find_request(const int* pref, int B, int64_t u) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Sets scores[b, j, g, n] = -inf for every n >= units(b) (never written by a
// unit); warp `first` of `count` takes every count-th row of NB scores, its
// lanes adjacent scores.
__device__ void fill_tails(const IdxParams& p, const int* pref, int64_t first, int64_t count) {
  const int lane = threadIdx.x & 31;
  const int rows_per_b = p.Q * p.I;
  const int64_t rows = static_cast<int64_t>(rows_per_b) * p.B;
  for (int64_t r = first; r < rows; r += count) {
    const int b = static_cast<int>(r / rows_per_b);
    float* row = p.scores + r * p.NB;
    for (int n = pref[b + 1] - pref[b] + lane; n < p.NB; n += 32) row[n] = -INFINITY;
  }
}

// Bytes of one page of index keys / key scales, per index head.
template <bool kFp4Keys>
__host__ __device__ constexpr uint32_t key_bytes_per_head() { return kFp4Keys ? kBlock * kDim / 2 : kBlock * kDim; }
template <bool kFp4Keys>
__host__ __device__ constexpr uint32_t scale_bytes_per_head() { return kFp4Keys ? kBlock * kDim / 16 : kBlock * 4; }

// kFp4Keys = false: E4M3 keys + fp32 per-token scale. true: NVFP4 keys (E2M1
// pairs, E4M3 scale per 16 values, fp32 global scale).
// kGroupCols (NVFP4 keys, one query position): the 8 mma columns are the 8
// scale groups of the key row instead of query positions. Column n of the B
// operand holds the query's dims of group n and zeros elsewhere, so the
// accumulator is the per-group partial dot product q . code, and the block
// scales multiply those fp32 partials rather than every decoded key value.
template <int kStages, bool kFp4Keys, bool kGroupCols>
__global__ void __launch_bounds__(kIdxThreads, kFp4Keys ? kFp4CtasPerSm : 1) index_score_fp8_kernel(IdxParams p) {
  extern __shared__ __align__(1024) uint8_t smem_fp8[];
  uint8_t* smem = smem_fp8;
  const int I = p.I;
  const uint32_t key_bytes = static_cast<uint32_t>(I) * key_bytes_per_head<kFp4Keys>();
  const uint32_t scale_bytes = static_cast<uint32_t>(I) * scale_bytes_per_head<kFp4Keys>();
  const uint32_t stage_bytes = key_bytes + scale_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  int* valid = reinterpret_cast<int*>(empty + kStages);
  float* part = reinterpret_cast<float*>(valid + kStages);          // [stage][head][warp of pair][8 columns]
  uint32_t* ticket = reinterpret_cast<uint32_t*>(part + kStages * kMaxIdxHeads * kWarpsPerHead * 8);
  int* sunit = reinterpret_cast<int*>(ticket + kStages * kMaxIdxHeads);   // unit of each stage, -1: no more
  int* pref = sunit + kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  griddep_wait();
  if (warp == 0) build_prefix(p, pref, blockIdx.x == 0);
  if (threadIdx.x == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kWarpsPerHead * I);
    }
    fence_mbar_init();
  }
  for (int x = threadIdx.x; x < kStages * kMaxIdxHeads; x += blockDim.x) ticket[x] = 0u;
  __syncthreads();
  if (warp > 0) {
    // the consumer warps fill the score tails (and insert) while the producer starts streaming
    const int64_t nc = blockDim.x / 32 - 1;
    fill_tails(p, pref, static_cast<int64_t>(blockIdx.x) * nc + (warp - 1), nc * gridDim.x);
    if (p.ins_on) fused_insert(p, static_cast<int64_t>(blockIdx.x) * nc + (warp - 1), nc * gridDim.x, lane);
  }

  const int64_t U = pref[p.B];
  const int64_t S = U - U / kDynShare;                 // units [S, U) go through the queue
  const int64_t u0 = S * blockIdx.x / gridDim.x, u1 = S * (blockIdx.x + 1) / gridDim.x;
  const int64_t n_static = u1 - u0;
  const int b_first = u0 < U ? find_request(pref, p.B, u0) : 0;
  unsigned long long* queue = g_idx_queue[p.slot];

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    // The whole warp fetches the page ids of the next 32 units at once (one
    // chunk ahead); lane 0 issues the copies and records each stage's unit.
    // Then the queue's chunks, and a last stage marked -1.
    const uint64_t pol = l2_evict_first_policy();
    const uint8_t* keys = static_cast<const uint8_t*>(p.keys);
    auto page_of = [&](int64_t u, int64_t end) -> int {
      if (u >= end) return -1;
      const int bb = find_request(pref, p.B, u);
      return p.block_table[static_cast<int64_t>(bb) * p.NB + (u - pref[bb])];
    };
    int64_t i = 0;
    bool ok = true;
    // lane 0: waits for stage i to be free, then fills it with unit u's page (u < 0: the end mark)
    auto issue = [&](int64_t u, int page) {
      if (lane == 0) {
        const int s = static_cast<int>(i % kStages);
        if (!mbar_wait(smem_addr(&empty[s]), static_cast<uint32_t>(((i / kStages) & 1) ^ 1))) {
          set_flag(p.flags, MSA_FLAG_TIMEOUT);
          ok = false;
        } else {
          const uint32_t fb = smem_addr(&full[s]);
          sunit[s] = static_cast<int>(u);
          if (u < 0 || page < 0 || page >= p.P) {
            if (u >= 0) set_flag(p.flags, MSA_FLAG_BAD_PAGE);
            valid[s] = 0;
            mbar_arrive(fb);
          } else {
            valid[s] = 1;
            const uint32_t dst = smem_addr(smem + s * stage_bytes);
            mbar_arrive_expect_tx(fb, stage_bytes);
            bulk_g2s(dst, keys + static_cast<int64_t>(page) * key_bytes, key_bytes, fb, pol);
            bulk_g2s(dst + key_bytes, static_cast<const uint8_t*>(p.scale) + static_cast<int64_t>(page) * scale_bytes,
                     scale_bytes, fb, pol);
          }
        }
      }
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      ++i;
    };
    int cur = page_of(u0 + lane, u1);
    for (int64_t base = u0; base < u1 && ok; base += 32) {
      const int nxt = page_of(base + 32 + lane, u1);
      const int n = static_cast<int>(u1 - base < 32 ? u1 - base : 32);
      for (int k = 0; k < n && ok; ++k) issue(base + k, __shfl_sync(kFull, cur, k));
      cur = nxt;
    }
    if (lane == 0) {
      atomicMax(&queue[0], epoch_base(p.epoch));
      atomicMax(&queue[1], epoch_base(p.epoch));
    }
    while (ok) {
      int64_t c0 = -1;
      if (lane == 0) {
        const int64_t cnt = epoch_fetch_add(&queue[0], p.epoch, p.flags);
        c0 = cnt < 0 ? -1 : S + cnt * kDynChunk;
        if (c0 >= U) c0 = -1;
      }
      c0 = __shfl_sync(kFull, c0, 0);
      if (c0 < 0) break;
      const int64_t c1 = c0 + kDynChunk < U ? c0 + kDynChunk : U;
      const int pg = page_of(c0 + lane, c1);
      for (int64_t u = c0; u < c1 && ok; ++u) issue(u, __shfl_sync(kFull, pg, static_cast<int>(u - c0)));
    }
    if (ok) issue(-1, -1);
    if (lane == 0) {
      // this CTA takes no more chunks; the last to finish clears the queue words
      const int64_t done = epoch_fetch_add(&queue[1], p.epoch, p.flags);
      if (done == static_cast<int64_t>(gridDim.x) - 1) {
        atomicExch(&queue[0], epoch_base(p.epoch));
        atomicExch(&queue[1], epoch_base(p.epoch));
      }
      // Do not leave while copies into this CTA's shared memory may be in flight.
      const int64_t first = i > kStages ? i - kStages : 0;
      for (int64_t k = first; k < i; ++k)
        if (!mbar_wait(smem_addr(&full[k % kStages]), static_cast<uint32_t>((k / kStages) & 1))) break;
    }
    return;
  }

  // ------------------------------------------------------------ consumers --
  const int g = (warp - 1) / kWarpsPerHead, slice = (warp - 1) % kWarpsPerHead;
  const int t0 = slice * kTilesPerWarp;
  const int gr = lane >> 2, c = lane & 3;
  const uint16_t* qbase = static_cast<const uint16_t*>(p.q);
  uint32_t qb[8][2];
  float inv_col0 = 0.f, inv_col1 = 0.f;
  int ell_col0 = 0, ell_col1 = 0;
  int cur_b = -1;
  int b = b_first;
  // the index-query fragments of request b (loaded when the request changes)
  auto load_query = [&]() {
    const int L = p.seq_lens[b];
    // Index-query fragment of position gr for this request and head.
    float qv[32];
    if (kGroupCols || gr < p.Q) {
      // dims this thread feeds to the mma: FP8 keys 16c..16c+15 and 64+16c..64+16c+15
      // (two 16-byte runs of a key row), NVFP4 keys 32c..32c+31 (one 16-byte run)
      const uint16_t* qp = qbase + ((static_cast<int64_t>(b) * p.Q + (kGroupCols ? 0 : gr)) * I + g) * kDim;
      const int o0 = kFp4Keys ? 32 * c : 16 * c, o1 = kFp4Keys ? 32 * c + 16 : 64 + 16 * c;
      const uint4 a0 = *reinterpret_cast<const uint4*>(qp + o0);
      const uint4 a1 = *reinterpret_cast<const uint4*>(qp + o0 + 8);
      const uint4 a2 = *reinterpret_cast<const uint4*>(qp + o1);
      const uint4 a3 = *reinterpret_cast<const uint4*>(qp + o1 + 8);
      const uint32_t w[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                              a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        qv[2 * k] = bf16_bits_to_f32(w[k] & 0xFFFF);
        qv[2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) qv[k] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(qv[k]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    const int sh = fp16_shift_for(amax);
    const float f = exp2_int(sh);
    const float inv = (kGroupCols || gr < p.Q) ? exp2_int(-sh) * (kFp4Keys ? p.global_scale : 1.f) : 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      // k-step s covers this thread's dims 32c+4s..32c+4s+3 (group 2c + s/4)
      const bool live = !kGroupCols || gr == 2 * c + (s >> 2);
      qb[s][0] = live ? pack_f16x2(qv[4 * s] * f, qv[4 * s + 1] * f) : 0u;
      qb[s][1] = live ? pack_f16x2(qv[4 * s + 2] * f, qv[4 * s + 3] * f) : 0u;
    }
    if (kGroupCols) {
      inv_col0 = inv_col1 = inv;
    } else {
      inv_col0 = __shfl_sync(kFull, inv, 8 * c);
      inv_col1 = __shfl_sync(kFull, inv, 8 * c + 4);
    }
    ell_col0 = (L - p.Q + 2 * c) / kBlock;
    ell_col1 = (L - p.Q + 2 * c + 1) / kBlock;
    cur_b = b;
  };
  for (int64_t i = 0;; ++i) {
    // units of the static range are known in advance, so their request's
    // queries load while the page is in flight; a queue unit is read from its stage
    const int s = static_cast<int>(i % kStages);
    int64_t u;
    if (i < n_static) {
      u = u0 + i;
      while (u >= pref[b + 1]) ++b;
      if (b != cur_b) load_query();
      if (!mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>((i / kStages) & 1))) {
        if (lane == 0) set_flag(p.flags, MSA_FLAG_TIMEOUT);
        break;
      }
    } else {
      if (!mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>((i / kStages) & 1))) {
        if (lane == 0) set_flag(p.flags, MSA_FLAG_TIMEOUT);
        break;
      }
      u = sunit[s];
      if (u < 0) break;                          // no more units
      if (u < pref[b] || u >= pref[b + 1]) b = find_request(pref, p.B, u);
      if (b != cur_b) load_query();
    }
    const int n = static_cast<int>(u - pref[b]);
    float m0 = -INFINITY, m1 = -INFINITY;
    if (valid[s] && !kFp4Keys) {
      const uint8_t* kb = smem + s * stage_bytes + g * (kBlock * kDim);
      const float* sc = reinterpret_cast<const float*>(smem + s * stage_bytes + key_bytes) + g * kBlock;
#pragma unroll 2
      for (int t = t0; t < t0 + kTilesPerWarp; ++t) {
        const uint8_t* r0 = kb + (16 * t + gr) * kDim + 16 * c;
        const uint4 x0 = *reinterpret_cast<const uint4*>(r0);
        const uint4 x1 = *reinterpret_cast<const uint4*>(r0 + 64);
        const uint4 y0 = *reinterpret_cast<const uint4*>(r0 + 8 * kDim);
        const uint4 y1 = *reinterpret_cast<const uint4*>(r0 + 8 * kDim + 64);
        const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t yw[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t a[4] = {e4m3x2_to_f16x2(static_cast<uint16_t>(xw[k] & 0xFFFF)),
                                 e4m3x2_to_f16x2(static_cast<uint16_t>(yw[k] & 0xFFFF)),
                                 e4m3x2_to_f16x2(static_cast<uint16_t>(xw[k] >> 16)),
                                 e4m3x2_to_f16x2(static_cast<uint16_t>(yw[k] >> 16))};
          mma_f16(acc, a, qb[k][0], qb[k][1]);
        }
        const float s0 = sc[16 * t + gr], s1 = sc[16 * t + gr + 8];
        m0 = fmaxf(m0, fmaxf(acc[0] * s0, acc[2] * s1));
        m1 = fmaxf(m1, fmaxf(acc[1] * s0, acc[3] * s1));
      }
    } else if (valid[s] && kGroupCols) {
      // NVFP4 keys, one position: acc[0..1] = row r0's partials of groups 2c,
      // 2c+1, acc[2..3] the same for row r1; scaled, summed over the 4 threads
      // of the row, then maxed.
      const uint8_t* kb = smem + s * stage_bytes + g * (kBlock * kDim / 2);
      const uint8_t* sb = smem + s * stage_bytes + key_bytes + g * (kBlock * kDim / 16);
#pragma unroll
      for (int t = t0; t < t0 + kTilesPerWarp; ++t) {
        const int r0 = 16 * t + gr, r1 = r0 + 8;
        const uint4 x = *reinterpret_cast<const uint4*>(kb + r0 * (kDim / 2) + 16 * c);
        const uint4 y = *reinterpret_cast<const uint4*>(kb + r1 * (kDim / 2) + 16 * c);
        const uint32_t sx = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sb + r0 * (kDim / 16) + 2 * c));
        const uint32_t sy = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sb + r1 * (kDim / 16) + 2 * c));
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t hx[4], hy[4];
          e2m1x8_to_f16x2x4(xw[j], hx);
          e2m1x8_to_f16x2x4(yw[j], hy);
          const uint32_t a0[4] = {hx[0], hy[0], hx[1], hy[1]};
          const uint32_t a1[4] = {hx[2], hy[2], hx[3], hy[3]};
          mma_f16(acc, a0, qb[2 * j][0], qb[2 * j][1]);
          mma_f16(acc, a1, qb[2 * j + 1][0], qb[2 * j + 1][1]);
        }
        const __half2 hsx = *reinterpret_cast<const __half2*>(&sx);
        const __half2 hsy = *reinterpret_cast<const __half2*>(&sy);
        float v0 = acc[0] * __low2float(hsx) + acc[1] * __high2float(hsx);
        float v1 = acc[2] * __low2float(hsy) + acc[3] * __high2float(hsy);
        v0 += __shfl_xor_sync(kFull, v0, 1);
        v1 += __shfl_xor_sync(kFull, v1, 1);
        v0 += __shfl_xor_sync(kFull, v0, 2);
        v1 += __shfl_xor_sync(kFull, v1, 2);
        m0 = fmaxf(m0, fmaxf(v0, v1));
      }
    } else if (valid[s]) {
      // NVFP4 keys: 64 B of E2M1 pairs per token row, 8 E4M3 scales; e2m1 x e4m3
      // is exact in fp16, so the fragment is the decoded key up to the global scale.
      const uint8_t* kb = smem + s * stage_bytes + g * (kBlock * kDim / 2);
      const uint8_t* sb = smem + s * stage_bytes + key_bytes + g * (kBlock * kDim / 16);
#pragma unroll 2
      for (int t = t0; t < t0 + kTilesPerWarp; ++t) {
        const int r0 = 16 * t + gr, r1 = r0 + 8;
        const uint4 x = *reinterpret_cast<const uint4*>(kb + r0 * (kDim / 2) + 16 * c);
        const uint4 y = *reinterpret_cast<const uint4*>(kb + r1 * (kDim / 2) + 16 * c);
        const uint32_t sx = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sb + r0 * (kDim / 16) + 2 * c));
        const uint32_t sy = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(sb + r1 * (kDim / 16) + 2 * c));
        const __half2 sx0 = __half2half2(__ushort_as_half(static_cast<unsigned short>(sx & 0xFFFF)));
        const __half2 sx1 = __half2half2(__ushort_as_half(static_cast<unsigned short>(sx >> 16)));
        const __half2 sy0 = __half2half2(__ushort_as_half(static_cast<unsigned short>(sy & 0xFFFF)));
        const __half2 sy1 = __half2half2(__ushort_as_half(static_cast<unsigned short>(sy >> 16)));
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t xl, xh, yl, yh;
          e2m1x4_to_f16x2x2(static_cast<uint16_t>(xw[k >> 1] >> (16 * (k & 1))), xl, xh);
          e2m1x4_to_f16x2x2(static_cast<uint16_t>(yw[k >> 1] >> (16 * (k & 1))), yl, yh);
          const __half2 scx = k < 4 ? sx0 : sx1, scy = k < 4 ? sy0 : sy1;
          __half2 h0 = __hmul2(*reinterpret_cast<__half2*>(&xl), scx);
          __half2 h1 = __hmul2(*reinterpret_cast<__half2*>(&yl), scy);
          __half2 h2 = __hmul2(*reinterpret_cast<__half2*>(&xh), scx);
          __half2 h3 = __hmul2(*reinterpret_cast<__half2*>(&yh), scy);
          const uint32_t a[4] = {*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                                 *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3)};
          mma_f16(acc, a, qb[k][0], qb[k][1]);
        }
        m0 = fmaxf(m0, fmaxf(acc[0], acc[2]));
        m1 = fmaxf(m1, fmaxf(acc[1], acc[3]));
      }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      m0 = fmaxf(m0, __shfl_xor_sync(kFull, m0, o));
      m1 = fmaxf(m1, __shfl_xor_sync(kFull, m1, o));
    }
    // Merge with the other warps of the head. Each writes its maxima to the
    // slot of (stage, head), then takes a ticket; the last ticket holder of the
    // unit (every unit takes exactly kWarpsPerHead tickets) reads the other
    // parts and writes the score. The slot is reused only after every warp has
    // released the stage, which each does after its last read of the slot.
    bool writer = true;
    if constexpr (kWarpsPerHead > 1) {
      float* slot = part + (s * kMaxIdxHeads + g) * (kWarpsPerHead * 8);
      if (gr == 0) {
        slot[slice * 8 + 2 * c] = m0;
        slot[slice * 8 + 2 * c + 1] = m1;
      }
      __syncwarp();
      uint32_t tk = 0;
      if (lane == 0) {
        __threadfence_block();
        tk = atomicAdd(&ticket[s * kMaxIdxHeads + g], 1u);
        __threadfence_block();
      }
      writer = __shfl_sync(kFull, tk, 0) % kWarpsPerHead == kWarpsPerHead - 1;
      __syncwarp();
      if (writer && gr == 0) {
        const volatile float* other = slot;
#pragma unroll
        for (int h = 0; h < kWarpsPerHead; ++h) {
          if (h == slice) continue;
          m0 = fmaxf(m0, other[h * 8 + 2 * c]);
          m1 = fmaxf(m1, other[h * 8 + 2 * c + 1]);
        }
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    if (writer && gr == 0) {
      const int64_t base = (static_cast<int64_t>(b) * p.Q) * I + g;
      const int j0 = 2 * c, j1 = 2 * c + 1;
      if (j0 < p.Q) p.scores[(base + static_cast<int64_t>(j0) * I) * p.NB + n] = n < ell_col0 ? m0 * inv_col0 : -INFINITY;
      if (j1 < p.Q) p.scores[(base + static_cast<int64_t>(j1) * I) * p.NB + n] = n < ell_col1 ? m1 * inv_col1 : -INFINITY;
    }
  }
}

// fp32 keys and queries (small workloads): one 128-thread CTA per (request,
// block, index head). Thread t scores token t of the block against the Q
// positions' index queries (in shared memory) with plain fp32 FMAs, eight
// 16-byte loads of its key row in flight at a time; the block's maximum per
// position is taken over the CTA by shuffles and shared memory.
__global__ void __launch_bounds__(kBlock) index_score_f32_kernel(IdxParams p) {
  extern __shared__ __align__(16) uint8_t smem_f32[];
  uint8_t* smem = smem_f32;
  int* pref = reinterpret_cast<int*>(smem);
  float* qsh = reinterpret_cast<float*>(smem + ((static_cast<size_t>(p.B) + 1) * 4 + 15) / 16 * 16);
  float* red = qsh + 8 * kDim;                      // [4 warps][8 positions]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  griddep_wait();
  if (p.ins_on) fused_insert(p, static_cast<int64_t>(blockIdx.x) * 4 + warp, static_cast<int64_t>(gridDim.x) * 4, lane);
  if (warp == 0) build_prefix(p, pref, blockIdx.x == 0);
  __syncthreads();
  fill_tails(p, pref, static_cast<int64_t>(blockIdx.x) * 4 + warp, static_cast<int64_t>(gridDim.x) * 4);
  const int64_t total = static_cast<int64_t>(pref[p.B]) * p.I;
  const float* qg = static_cast<const float*>(p.q);
  const float* keys = static_cast<const float*>(p.keys);
  for (int64_t task = blockIdx.x; task < total; task += gridDim.x) {
    const int64_t v = task / p.I;
    const int g = static_cast<int>(task % p.I);
    const int b = find_request(pref, p.B, v);
    const int n = static_cast<int>(v - pref[b]);
    const int L = p.seq_lens[b];
    __syncthreads();                                // previous task done with qsh / red
    for (int x = threadIdx.x; x < p.Q * kDim; x += blockDim.x) {
      const int j = x / kDim, d = x % kDim;
      qsh[x] = qg[((static_cast<int64_t>(b) * p.Q + j) * p.I + g) * kDim + d];
    }
    __syncthreads();
    const int page = p.block_table[static_cast<int64_t>(b) * p.NB + n];
    float dot[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) dot[j] = 0.f;
    const bool ok = page >= 0 && page < p.P;
    if (!ok) {
      if (threadIdx.x == 0) set_flag(p.flags, MSA_FLAG_BAD_PAGE);
    } else {
      const float4* row = reinterpret_cast<const float4*>(
          keys + ((static_cast<int64_t>(page) * p.I + g) * kBlock + threadIdx.x) * kDim);
      for (int d8 = 0; d8 < kDim / 4; d8 += 8) {
        float4 kv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) kv[u] = row[d8 + u];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j < p.Q) {
              const float4 qj = *reinterpret_cast<const float4*>(qsh + j * kDim + 4 * (d8 + u));
              dot[j] = fmaf(kv[u].x, qj.x, dot[j]);
              dot[j] = fmaf(kv[u].y, qj.y, dot[j]);
              dot[j] = fmaf(kv[u].z, qj.z, dot[j]);
              dot[j] = fmaf(kv[u].w, qj.w, dot[j]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float m = ok ? dot[j] : -INFINITY;
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      if (lane == 0) red[warp * 8 + j] = m;
    }
    __syncthreads();
    if (threadIdx.x < p.Q) {
      const int j = threadIdx.x;
      const float val = fmaxf(fmaxf(red[j], red[8 + j]), fmaxf(red[16 + j], red[24 + j]));
      const int ell = (L - p.Q + j) / kBlock;
      p.scores[((static_cast<int64_t>(b) * p.Q + j) * p.I + g) * p.NB + n] = n < ell ? val : -INFINITY;
    }
  }
}

cudaError_t launch_index_score(const IndexArgs& a, const InsertArgs* ins, cudaStream_t stream, DispatchRecord* rec) {
  IdxParams p{a.q, a.keys, a.scale, a.block_table, a.seq_lens, a.scores, a.flags, a.global_scale,
              a.B, a.Q, a.I, a.NB, a.P};
  p.ins_on = 0;
  static std::atomic<uint64_t> epoch{1};
  static std::atomic<uint32_t> captured{0};
  p.epoch = epoch.fetch_add(1);                      // grows from call to call (queue words, above)
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) capture = cudaStreamCaptureStatusNone;
  p.slot = capture == cudaStreamCaptureStatusActive ? kQueueSlots + static_cast<int>(captured.fetch_add(1) % kQueueSlots)
                                                    : static_cast<int>(p.epoch % kQueueSlots);
  if (ins != nullptr) {
    if (a.Q != 1) return cudaErrorInvalidValue;   // the caller checks it
    p.ins_on = 1;
    p.ins = make_insert_params(*ins);
  }
  const int sms = device_sm_count();
  cudaError_t err;
  if (a.fp8 || a.fp4) {
    const int stages = a.fp4 ? kIdxStagesFp4 : kIdxStages;
    const size_t stage = a.fp4 ? static_cast<size_t>(a.I) * (key_bytes_per_head<true>() + scale_bytes_per_head<true>())
                               : static_cast<size_t>(a.I) * (key_bytes_per_head<false>() + scale_bytes_per_head<false>());
    const size_t smem = stages * stage + 2 * stages * 8 + stages * 4 +
                        stages * kMaxIdxHeads * (kWarpsPerHead * 8 * 4 + 4) + stages * 4 + (a.B + 1) * 4;
    auto kern = !a.fp4 ? index_score_fp8_kernel<kIdxStages, false, false>
                : a.Q == 1 ? index_score_fp8_kernel<kIdxStagesFp4, true, true>
                           : index_score_fp8_kernel<kIdxStagesFp4, true, false>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int grid = a.fp4 ? kFp4CtasPerSm * sms : sms;
    const int block = 32 * (1 + kWarpsPerHead * a.I);
    err = launch_pdl(kern, dim3(grid), dim3(block), smem, stream, p);
    if (err != cudaSuccess) return err;
    rec->set("%sindex_score %s grid=%d block=%d smem=%zu stages=%d q_len=%d idx_heads=%d", p.ins_on ? "insert+" : "",
             !a.fp4 ? "fp8_mma_f16" : a.Q == 1 ? "nvfp4_group_cols_mma_f16" : "nvfp4_mma_f16", grid, block, smem,
             stages, a.Q, a.I);
  } else {
    const size_t smem = ((static_cast<size_t>(a.B) + 1) * 4 + 15) / 16 * 16 + 8 * kDim * 4 + 4 * 8 * 4;
    err = cudaFuncSetAttribute(index_score_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int grid = sms * 8;                   // grid-stride over (request, block, head) tasks
    err = launch_pdl(index_score_f32_kernel, dim3(grid), dim3(kBlock), smem, stream, p);
    if (err != cudaSuccess) return err;
    rec->set("%sindex_score f32_fma grid=%d block=%d smem=%zu q_len=%d idx_heads=%d", p.ins_on ? "insert+" : "", grid,
             kBlock, smem, a.Q, a.I);
  }
  return cudaGetLastError();
}

}  // namespace msa
