// Stage 3 of MSA decode: sparse GQA over the selected blocks, split-K, with a
// log-sum-exp combine.
//
// "MiniMax M3 vLLM サポート：…" (agentlenshq.com), section "MSA 実行プロセス",
// step 3: online-softmax attention over the selected KV blocks only; section
// "EAGLE3 を用いた投機的デコード": a decode-only split-K path that serves every
// decode_query_len. "vLLM、AMD Instinct MI355X上で…", question 1: 64 query
// heads share 4 KV heads, so the 16 heads of a KV head form one M=16 tile.
//
// Four forms, all persistent, all with bounded waits and no traps:
//   sparse_gqa_kernel<bf16 | FP8>: work items are (row, selection slot) pairs,
//     row = (request, KV head, position), positions of one (request, KV head)
//     adjacent; every CTA owns whole rows. A producer warp fetches each
//     selected page through 2-D tensor maps with 128-byte swizzle
//     (conflict-free ldmatrix); each of four consumer warps owns 32 tokens of
//     every block; QK^T and PV run on m16n8k16 tensor-core mma. At a row's end
//     the CTA merges its warps' online-softmax states and writes the output.
//   sparse_gqa_fp4_kernel (NVFP4): eight consumer warps of 16 tokens; each
//     row split over the CTAs of a thread-block cluster that merge in
//     distributed shared memory, or (when the rows' clusters do not all fit
//     at once) item ranges balanced over the SMs, split rows merged by the
//     CTA that delivers the last partial.
//   sparse_gqa_union_kernel (bf16, several query positions): the union of a
//     (request, KV head) group's blocks streamed once, one warp per position.
//   sparse_gqa_tc_kernel (bf16, opt-in): the tile on tcgen05 with S and O in
//     tensor memory.
#include <cuda.h>

#include <atomic>
#include <cstdlib>
#include <cstring>

#include "msa_internal.h"
#include "select_row.cuh"

namespace msa {

// K/V cache formats (template argument of the kernel).
constexpr int kKvBf16 = 0, kKvFp8 = 2;
template <int kKv>
constexpr int stages_for() { return kKv == kKvBf16 ? 3 : 6; }   // 64 KB bf16 / 32 KB FP8 pages
constexpr int kTokPerWarp = 32;                  // tokens of every block that one consumer warp owns
constexpr int kCWarps = kBlock / kTokPerWarp;    // consumer warps (one per SM sub-partition)
constexpr int kNT = kTokPerWarp / 8;             // QK^T n-tiles of 8 tokens per warp
constexpr int kKK = kTokPerWarp / 16;            // PV k-steps of 16 tokens per warp
constexpr int kCombWarps = kCWarps;              // states staged in shared memory at a row's end
static_assert(kCWarps == 4, "the row merge runs on 4 warps x 32 threads");
constexpr int kBoxBytes = kBlock * 64 * 2;       // 128 rows x 128 B (64 fp16/bf16)
constexpr int kTileBytes = 4 * kBoxBytes;        // K lo/hi + V lo/hi = 64 KB
constexpr int kFp4StageBytes = 2 * (kBlock * kDim / 2 + kBlock * kDim / 16);  // 18 KB
constexpr int kFp8BoxBytes = kBlock * kDim;      // 128 rows x 128 E4M3 codes
constexpr int kFp8StageBytes = 2 * kFp8BoxBytes; // K + V = 32 KB
template <int kKv>
constexpr uint32_t stage_bytes_for() {
  return kKv == kKvBf16 ? kTileBytes : kFp8StageBytes;
}
constexpr uint32_t kAll = 0xffffffffu;
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleSlack = 8.f;    // log2 units: probabilities below 256 before normalisation

struct GqaParams {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* selected;
  const float* scores;          // non-null: the CTAs select their rows' blocks from these first
  int32_t* sel_out;             // (and write them here; the same buffer as `selected`)
  uint16_t* out;
  float* lse;
  float* ws;
  uint32_t* flags;
  const uint8_t* k4;
  const uint8_t* v4;
  const uint8_t* ks;
  const uint8_t* vs;
  unsigned long long* tickets;  // one per row, after the partials in the workspace
  float k_global, v_global;
  float scale_log2;
  uint32_t epoch;               // differs on every call; tags the tickets
  int B, Q, H, G, NB, P, K;
  int row_aligned;  // 1: every CTA owns whole rows; 0: balanced item ranges, rows may be split
  int cluster_n;    // NVFP4 only: > 1 = each row split over one cluster of this many CTAs
  int64_t W;        // items = B * G * Q * K
};

struct SmemLayout {
  uint32_t stages, tiles, comb_o, comb_ml, bars, zero;
  uint32_t total;
};

template <int kKv>
__host__ __device__ constexpr SmemLayout gqa_layout() {
  SmemLayout s{};
  s.stages = 0;
  s.tiles = s.stages + stages_for<kKv>() * stage_bytes_for<kKv>();
  s.comb_o = s.tiles;
  s.comb_ml = s.comb_o + kCombWarps * kGroup * kDim * 4;
  s.bars = s.comb_ml + kCombWarps * kGroup * 2 * 4;
  s.zero = s.bars + (2 * stages_for<kKv>() + 2) * 8 + 16;    // after the last-arriver flag
  s.total = s.zero + 16;                                       // 16 zero bytes: the V row of a masked token
  return s;
}

// First CTA whose item range contains item x (ranges are [W*c/C, W*(c+1)/C)).
__host__ __device__ __forceinline__ int cta_of(int64_t x, int64_t W, int C) {
  return static_cast<int>(((x + 1) * C + W - 1) / W) - 1;
}

struct RowPos {
  int b, g, j;
};

// (request, KV head, position) of enumeration row r; positions are adjacent.
// Rows and items fit in 32 bits (at most 4096 x 8 x 4 rows of 16 slots).
__device__ __forceinline__ RowPos row_pos(const GqaParams& p, int64_t r64) {
  const uint32_t r = static_cast<uint32_t>(r64);
  const uint32_t rq = r / static_cast<uint32_t>(p.Q);
  RowPos o;
  o.j = static_cast<int>(r - rq * static_cast<uint32_t>(p.Q));
  o.b = static_cast<int>(rq / static_cast<uint32_t>(p.G));
  o.g = static_cast<int>(rq - static_cast<uint32_t>(o.b) * static_cast<uint32_t>(p.G));
  return o;
}

struct ItemInfo {
  int blk, page, valid, g;
};

// Selected block, page and validity of item x (x >= x1: an empty slot). Checks
// the device-side invariants; only the producer reports problems.
__device__ __forceinline__ ItemInfo load_item(const GqaParams& p, int64_t x, int64_t x1, bool report) {
  ItemInfo it{-1, -1, 0, 0};
  if (x >= x1) return it;
  const uint32_t r = static_cast<uint32_t>(x) / static_cast<uint32_t>(p.K);
  const int e = static_cast<int>(static_cast<uint32_t>(x) - r * static_cast<uint32_t>(p.K));
  const RowPos rp = row_pos(p, r);
  it.g = rp.g;
  const int L = p.seq_lens[rp.b];          // loaded alongside the selection, not after it
  it.blk = p.selected[((static_cast<int64_t>(rp.b) * p.Q + rp.j) * p.G + rp.g) * p.K + e];
  if (it.blk < 0) return it;
  if (L < p.Q || L > p.NB * kBlock || L < 1) {
    if (report) set_flag(p.flags, MSA_FLAG_BAD_SEQLEN);
    return it;
  }
  if (it.blk > (L - p.Q + rp.j) / kBlock) {
    if (report) set_flag(p.flags, MSA_FLAG_BAD_BLOCK);
    return it;
  }
  it.page = p.block_table[static_cast<int64_t>(rp.b) * p.NB + it.blk];
  if (it.page < 0 || it.page >= p.P) {
    if (report) set_flag(p.flags, MSA_FLAG_BAD_PAGE);
    return it;
  }
  it.valid = 1;
  return it;
}

// Counts this CTA's partial of a row: the ticket word holds (epoch << 32 | count)
// and a count from another epoch is read as 0, so the workspace needs no
// initialisation. Returns true for the CTA that delivers the last partial,
// which also clears the word: no other CTA of this launch touches it again,
// and a replay of a captured graph (whose epoch is fixed at capture) starts
// from zero.
__device__ bool ticket_is_last(const GqaParams& p, int64_t row, int nslots) {
  unsigned long long* t = p.tickets + row;
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(t);
  for (int tries = 0; tries < (1 << 20); ++tries) {
    const uint32_t cnt = static_cast<uint32_t>(cur >> 32) == p.epoch ? static_cast<uint32_t>(cur) : 0u;
    const unsigned long long nw = (static_cast<unsigned long long>(p.epoch) << 32) | (cnt + 1u);
    const unsigned long long prev = atomicCAS(t, cur, nw);
    if (prev == cur) {
      const bool last = static_cast<int>(cnt + 1u) == nslots;
      if (last) atomicExch(t, 0ull);
      return last;
    }
    cur = prev;
  }
  set_flag(p.flags, MSA_FLAG_TIMEOUT);
  return false;
}

// Consumer-group barrier on an mbarrier (count = 4 warps), bounded in time.
__device__ __forceinline__ bool group_sync(uint32_t bar, uint32_t& phase, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase);
  phase ^= 1;
  return ok;
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Thread-block cluster helpers. The barrier is the non-aligned form, so threads
// of a warp may reach it from different places; every thread of the cluster
// arrives at it, and each reaches it after bounded waits only.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }
// Asynchronous stores into another CTA's shared memory (`addr` from
// cluster_map), each completing its bytes on the mbarrier at `rbar` in that CTA.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, float a, float b, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(addr), "f"(a), "f"(b), "r"(rbar)
               : "memory");
}
// Non-blocking test of an mbarrier phase (try_wait may suspend the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

__device__ __forceinline__ uint32_t swz(uint32_t box, int row, int chunk) {
  return box + row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <int kKv>
__global__ void __launch_bounds__(32 * (1 + kCWarps), 1)
    sparse_gqa_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr bool kFp8 = kKv == kKvFp8;
  static_assert(kKv == kKvBf16 || kKv == kKvFp8, "four-warp form: bf16 or FP8 K/V");
  static_assert(!kFp8 || kNT == 4, "the FP8 fragment loads take 4 n-tiles per ldmatrix.x4");
  constexpr SmemLayout Ly = gqa_layout<kKv>();
  constexpr uint32_t kStageBytes = stage_bytes_for<kKv>();
  constexpr int kGqaStages = stages_for<kKv>();
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base_addr = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_addr - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Ly.bars);
  uint64_t* empty = full + kGqaStages;
  uint64_t* gbar = empty + kGqaStages;   // [0]: partials written, [1]: partials read
  float* comb_o = reinterpret_cast<float*>(sm + Ly.comb_o);
  float* comb_m = reinterpret_cast<float*>(sm + Ly.comb_ml);
  float* comb_l = comb_m + kCombWarps * kGroup;
  int* last_flag = reinterpret_cast<int*>(sm + Ly.bars + (2 * kGqaStages + 2) * 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGqaStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kCWarps);
    }
    mbar_init(smem_addr(&gbar[0]), kCWarps);
    mbar_init(smem_addr(&gbar[1]), kCWarps);
    fence_mbar_init();
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    st_shared_zero16(base_addr + Ly.zero);
  }
  __syncthreads();
  griddep_wait();

  const int C = gridDim.x;
  int64_t x0, x1;
  if (p.row_aligned) {
    const int64_t rows = p.W / p.K;
    x0 = rows * blockIdx.x / C * p.K;
    x1 = rows * (blockIdx.x + 1) / C * p.K;
  } else {
    x0 = p.W * blockIdx.x / C;
    x1 = p.W * (blockIdx.x + 1) / C;
  }
  if (x0 >= x1) return;

  if (p.scores != nullptr) {
    // Stage 2 inside this launch: every warp selects rows this CTA touches
    // (rows shared with other CTAs get the same result from each), staging its
    // survivors in the row-merge buffer, unused until a row ends.
    uint64_t* surv = reinterpret_cast<uint64_t*>(sm + Ly.comb_o) + warp * (kWarpSurvCap + 8);
    int* chosen = reinterpret_cast<int*>(surv + kWarpSurvCap);
    const int64_t r_last = (x1 - 1) / p.K;
    for (int64_t r = x0 / p.K + warp; r <= r_last; r += blockDim.x >> 5) {
      const RowPos rp = row_pos(p, r);
      const int64_t row_off = (static_cast<int64_t>(rp.b) * p.Q + rp.j) * p.G + rp.g;
      int32_t* out = p.sel_out + row_off * p.K;
      const int L = p.seq_lens[rp.b];
      if (L < p.Q || L > p.NB * kBlock || L < 1) {           // (flagged by the item loads below)
        for (int e = lane; e < p.K; e += 32) out[e] = -1;
        continue;
      }
      warp_select_row(p.scores + row_off * p.NB, (L - p.Q + rp.j) / kBlock, p.K, out, surv, chosen, lane);
    }
    __syncthreads();                  // the item loads below read these rows back
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    // The warp fetches the next 32 items' block, page and validity at once
    // (one chunk ahead); lane 0 issues the copies.
    ItemInfo cur = load_item(p, x0 + lane, x1, true);
    int64_t i = 0;
    int s = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t base = x0; base < x1 && ok; base += 32) {
      const ItemInfo nxt = load_item(p, base + 32 + lane, x1, true);
      const int n = static_cast<int>(x1 - base < 32 ? x1 - base : 32);
      for (int k = 0; k < n; ++k) {
        if (!__shfl_sync(kAll, cur.valid, k)) continue;
        const int page = __shfl_sync(kAll, cur.page, k);
        const int g = __shfl_sync(kAll, cur.g, k);
        if (lane == 0) {
          if (!mbar_wait(smem_addr(&empty[s]), phase ^ 1u)) {
            set_flag(p.flags, MSA_FLAG_TIMEOUT);
            ok = false;
          } else {
            const uint32_t fb = smem_addr(&full[s]);
            const uint32_t dst = base_addr + Ly.stages + s * kStageBytes;
            const int64_t ph = static_cast<int64_t>(page) * p.G + g;   // (page, kv head) slab
            mbar_arrive_expect_tx(fb, kStageBytes);
            if (kFp8) {
              const int y = static_cast<int>(ph * kBlock);
              tma_load_2d(dst, &tk, 0, y, fb);
              tma_load_2d(dst + kFp8BoxBytes, &tv, 0, y, fb);
            } else {
              const int y = static_cast<int>(ph * kBlock);
              tma_load_2d(dst, &tk, 0, y, fb);
              tma_load_2d(dst + kBoxBytes, &tk, 64, y, fb);
              tma_load_2d(dst + 2 * kBoxBytes, &tv, 0, y, fb);
              tma_load_2d(dst + 3 * kBoxBytes, &tv, 64, y, fb);
            }
          }
        }
        ok = __shfl_sync(kAll, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++i;
        if (++s == kGqaStages) { s = 0; phase ^= 1u; }
      }
      cur = nxt;
    }
    if (lane == 0) {
      const int64_t first = i > kGqaStages ? i - kGqaStages : 0;
      for (int64_t k = first; k < i; ++k)
        if (!mbar_wait(smem_addr(&full[k % kGqaStages]), static_cast<uint32_t>((k / kGqaStages) & 1))) break;
    }
    return;
  }

  // -------------------------------------------------------------- consumers --
  const int w = warp - 1;          // token slice [kTokPerWarp w, kTokPerWarp (w + 1)) of every block
  const int ct = threadIdx.x - 32; // 0 .. 32 kCWarps - 1; the first 128 merge a row's states
  const int gr = lane >> 2, c = lane & 3;
  uint32_t gph[2] = {0u, 0u};

  uint32_t qf[8][4];
  float o[16][4];
  float m_r[2], l_r[2], mul_r[2];
  int64_t seg_row = -1;
  int seg_b = 0, seg_g = 0, seg_j = 0, seg_p = 0, seg_ell = 0;
  bool ok = true;

  auto begin_segment = [&](int64_t r) {
    const RowPos rp = row_pos(p, r);
    seg_row = r;
    seg_b = rp.b; seg_g = rp.g; seg_j = rp.j;
    const int L = p.seq_lens[rp.b];
    seg_p = L - p.Q + rp.j;
    seg_ell = seg_p / kBlock;
    const uint16_t* qh = p.q + ((static_cast<int64_t>(rp.b) * p.Q + rp.j) * p.H + static_cast<int64_t>(rp.g) * kGroup) * kDim;
    // The bf16 query words are the mma A fragments as loaded: qf[s] holds rows
    // gr / gr + 8 at dims 16 s + 2 c (+1) and 16 s + 8 + 2 c (+1). With FP8
    // keys the k-slots of step s are dims 16 s + 4 c .. 16 s + 4 c + 3 instead
    // (the four bytes one ldmatrix lane receives of a key row).
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (kFp8) {
          const uint2 wq = *reinterpret_cast<const uint2*>(qh + (gr + 8 * r) * kDim + 16 * s + 4 * c);
          qf[s][r] = wq.x;
          qf[s][2 + r] = wq.y;
        } else {
          const uint16_t* row = qh + (gr + 8 * r) * kDim + 16 * s + 2 * c;
          qf[s][r] = *reinterpret_cast<const uint32_t*>(row);
          qf[s][2 + r] = *reinterpret_cast<const uint32_t*>(row + 8);
        }
      }
    }
    if (kFp8) {
      // fp16 operands: rescale each query row by an exact power of two that
      // keeps it inside the fp16 range; the logit multiplier undoes it.
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float amax = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t wq = qf[s][2 * h + r];
            amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(wq & 0xFFFF)), fabsf(bf16_bits_to_f32(wq >> 16))));
          }
        }
        amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 2));
        const int sh = fp16_shift_for(amax);
        const float f = exp2_int(sh);
        mul_r[r] = p.scale_log2 * p.k_global * exp2_int(-sh);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t wq = qf[s][2 * h + r];
            qf[s][2 * h + r] = pack_f16x2(bf16_bits_to_f32(wq & 0xFFFF) * f, bf16_bits_to_f32(wq >> 16) * f);
          }
        }
      }
    } else {
      mul_r[0] = mul_r[1] = p.scale_log2;
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m_r[0] = m_r[1] = -INFINITY;
    l_r[0] = l_r[1] = 0.f;
  };

  // Stages this warp's state (o, m, l) of the current row in slot k.
  auto stage_state = [&](int k, const float (&lt)[2]) {
    float* mo = comb_o + k * kGroup * kDim;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      if (kFp8) {
        // n-tile n holds the even (n even) or odd dims of chunk n / 2: column
        // 2 c + e is dim 16 (n / 2) + 4 c + 2 e + (n & 1)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = 16 * (n >> 1) + 4 * c + 2 * e + (n & 1);
          mo[gr * kDim + d] = o[n][e];
          mo[(gr + 8) * kDim + d] = o[n][2 + e];
        }
      } else {
        *reinterpret_cast<float2*>(mo + gr * kDim + 8 * n + 2 * c) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(mo + (gr + 8) * kDim + 8 * n + 2 * c) = make_float2(o[n][2], o[n][3]);
      }
    }
    if (c == 0) {
      comb_m[k * kGroup + gr] = m_r[0];
      comb_m[k * kGroup + gr + 8] = m_r[1];
      comb_l[k * kGroup + gr] = lt[0];
      comb_l[k * kGroup + gr + 8] = lt[1];
    }
  };

  // Merges the warps' states of the current row; writes the final output when
  // this CTA covered the whole row, a split-K partial otherwise. Every consumer
  // warp takes every barrier; the merge itself runs on the first 128 threads.
  auto end_segment = [&]() -> bool {
    float lt[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float v = l_r[r];
      v += __shfl_xor_sync(kAll, v, 1);
      v += __shfl_xor_sync(kAll, v, 2);
      lt[r] = v;
    }
    stage_state(w, lt);
    if (!group_sync(smem_addr(&gbar[0]), gph[0], lane)) return false;
    const bool merger = ct < kCombWarps * 32;
    const int hh = (ct >> 3) & (kGroup - 1), d0 = (ct & 7) * 16;
    float M = -INFINITY;
    float Ls = 0.f;
    float acc[16];
    if (merger) {
#pragma unroll
      for (int k = 0; k < kCombWarps; ++k) M = fmaxf(M, comb_m[k * kGroup + hh]);
      float fw[kCombWarps];
#pragma unroll
      for (int k = 0; k < kCombWarps; ++k) {
        fw[k] = M == -INFINITY ? 0.f : ex2_approx(comb_m[k * kGroup + hh] - M);
        Ls += fw[k] * comb_l[k * kGroup + hh];
      }
#pragma unroll
      for (int d = 0; d < 16; ++d) {
        float v = 0.f;
#pragma unroll
        for (int k = 0; k < kCombWarps; ++k) v += fw[k] * comb_o[(k * kGroup + hh) * kDim + d0 + d];
        acc[d] = v * (kFp8 ? p.v_global : 1.f);
      }
    }
    const int64_t r = seg_row;
    const bool whole = x0 <= r * p.K && (r + 1) * p.K <= x1;
    const int64_t head = (static_cast<int64_t>(seg_b) * p.Q + seg_j) * p.H + static_cast<int64_t>(seg_g) * kGroup + hh;
    auto write_out = [&](const float (&v)[16], float mm, float ll) {
      const float inv = ll > 0.f ? 1.f / ll : 0.f;
      uint32_t packed[8];
#pragma unroll
      for (int d = 0; d < 8; ++d) packed[d] = pack_bf16x2(v[2 * d] * inv, v[2 * d + 1] * inv);
      uint4* dst = reinterpret_cast<uint4*>(p.out + head * kDim + d0);
      dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
      if (p.lse != nullptr && (ct & 7) == 0) p.lse[head] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
    };
    if (whole) {
      if (merger) write_out(acc, M, Ls);
      return group_sync(smem_addr(&gbar[1]), gph[1], lane);
    }
    // Split row: publish this CTA's partial; the CTA that delivers the last
    // one merges them all.
    const int first = cta_of(r * p.K, p.W, C);
    const int nslots = cta_of(r * p.K + p.K - 1, p.W, C) - first + 1;
    float* rowp = p.ws + r * p.K * static_cast<int64_t>(kPartialFloats);
    float* part = rowp + (static_cast<int>(blockIdx.x) - first) * static_cast<int64_t>(kPartialFloats);
    if (merger) {
      float4* dst = reinterpret_cast<float4*>(part + hh * kDim + d0);
#pragma unroll
      for (int d = 0; d < 4; ++d) dst[d] = make_float4(acc[4 * d], acc[4 * d + 1], acc[4 * d + 2], acc[4 * d + 3]);
      if ((ct & 7) == 0) {
        part[kGroup * kDim + hh] = M;
        part[kGroup * kDim + kGroup + hh] = Ls;
      }
    }
    if (!group_sync(smem_addr(&gbar[1]), gph[1], lane)) return false;
    if (ct == 0) {
      fence_acq_rel_gpu();                       // publish the CTA's partial (after the barrier above)
      const bool last = ticket_is_last(p, r, nslots);
      if (last) fence_acq_rel_gpu();             // see the other CTAs' partials
      *last_flag = last ? 1 : 0;
    }
    if (!group_sync(smem_addr(&gbar[0]), gph[0], lane)) return false;
    if (*last_flag && merger) {
      float M2 = -INFINITY;
      for (int q = 0; q < nslots; ++q) M2 = fmaxf(M2, __ldcg(rowp + q * kPartialFloats + kGroup * kDim + hh));
      float L2 = 0.f;
      float v[16];
#pragma unroll
      for (int d = 0; d < 16; ++d) v[d] = 0.f;
      if (M2 != -INFINITY) {
        for (int q = 0; q < nslots; ++q) {
          const float* pq = rowp + q * kPartialFloats;
          const float f = ex2_approx(__ldcg(pq + kGroup * kDim + hh) - M2);
          L2 += f * __ldcg(pq + kGroup * kDim + kGroup + hh);
#pragma unroll
          for (int d4 = 0; d4 < 4; ++d4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(pq + hh * kDim + d0) + d4);
            v[4 * d4] += f * x.x;
            v[4 * d4 + 1] += f * x.y;
            v[4 * d4 + 2] += f * x.z;
            v[4 * d4 + 3] += f * x.w;
          }
        }
      }
      write_out(v, M2, L2);
    }
    return true;
  };

  // QK^T of this warp's tokens for the tile at kt (K lo / K hi boxes).
  // ldmatrix addresses within a tile, per thread. A row's 16-byte chunk q sits
  // at row * 128 + ((q ^ (row & 7)) << 4) of its box; every row this thread
  // addresses has row & 7 == lane & 7, so only the chunk's low bits vary with
  // the loop indices and the rest are compile-time offsets.
  //   QK^T (K boxes): row 8 nt + (lane & 7) of the warp's slice, chunk 4 (sp & 1) + (lane >> 3)
  //   PV (V boxes):   row 16 kk + 8 ((lane >> 3) & 1) + (lane & 7), chunk 2 (np & 3) + (lane >> 4)
  const uint32_t warp_rows = static_cast<uint32_t>(kTokPerWarp * w) * 128u;
  uint32_t k_off[2], v_off[4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    k_off[h] = warp_rows + (lane & 7) * 128u + ((((4 * h) + (lane >> 3)) ^ (lane & 7)) << 4);
#pragma unroll
  for (int h = 0; h < 4; ++h)
    v_off[h] = warp_rows + (8 * ((lane >> 3) & 1) + (lane & 7)) * 128u + ((((2 * h) + (lane >> 4)) ^ (lane & 7)) << 4);

  const uint32_t lane_x = (lane & 7) << 4;     // FP8 tiles: XOR of the 128-byte swizzle for this lane's rows
  const uint32_t k8_row = (static_cast<uint32_t>(kTokPerWarp * w) + 8u * (lane >> 3) + (lane & 7)) * 128u;
  const uint32_t v8_row = (static_cast<uint32_t>(kTokPerWarp * w) + 8u * ((lane >> 3) & 1) + (lane & 7)) * 128u;

  auto qk = [&](uint32_t kt, float (&sc)[kNT][4]) {
    if (kFp8) {
      // FP8 K: one ldmatrix.x4 per 16-dim chunk q gives lane (gr, c) the codes
      // of dims 16 q + 4 c .. + 3 of token row gr of each of the 4 n-tiles
      // (matrix m = n-tile m); two exact cvts make its b0 / b1 fragments.
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t r[4];
        ldsm_x4(kt + k8_row + ((static_cast<uint32_t>(q) << 4) ^ lane_x), r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
          mma_f16(sc[nt], qf[q], e4m3x2_to_f16x2(static_cast<uint16_t>(r[nt] & 0xFFFF)),
                  e4m3x2_to_f16x2(static_cast<uint16_t>(r[nt] >> 16)));
      }
      return;
    }
    // ---- S = Q K^T for this warp's tokens (kNT n-tiles of 8 tokens). The
    // n-tiles are independent accumulation chains, interleaved per pair of
    // k-steps so that the mma latencies overlap.
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int sp = 0; sp < 4; ++sp) {
      const uint32_t kb = kt + (sp >> 1) * kBoxBytes + k_off[sp & 1];
      uint32_t b[kNT][4];
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) ldsm_x4(kb + nt * 8 * 128, b[nt][0], b[nt][1], b[nt][2], b[nt][3]);
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        mma_bf16(sc[nt], qf[2 * sp], b[nt][0], b[nt][1]);
      }
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        mma_bf16(sc[nt], qf[2 * sp + 1], b[nt][2], b[nt][3]);
      }
    }
  };

  // Causal limit and the first half of the online softmax for one tile: block
  // maxima and, when the reference max rises, the rescale of the accumulators.
  auto softmax_prep = [&](float (&sc)[kNT][4], int it_blk) {
    // ---- causal limit inside the local block
    if (it_blk == seg_ell) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int t0 = it_blk * kBlock + kTokPerWarp * w + 8 * nt + 2 * c;
        if (t0 > seg_p) { sc[nt][0] = -INFINITY; sc[nt][2] = -INFINITY; }
        if (t0 + 1 > seg_p) { sc[nt][1] = -INFINITY; sc[nt][3] = -INFINITY; }
      }
    }
    // ---- online softmax (log2 domain), rows gr and gr + 8. The reference max
    // m_r is raised only when a block's max exceeds it by more than
    // kRescaleSlack, so the unnormalised probabilities stay below 2^kRescaleSlack
    // and most blocks leave the output accumulator unscaled (the final division
    // by l makes the choice of reference immaterial up to rounding).
    float bmax[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) mx = fmaxf(mx, fmaxf(sc[nt][2 * r], sc[nt][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
      bmax[r] = mx * mul_r[r];
    }
    const bool raise0 = bmax[0] > m_r[0] + kRescaleSlack, raise1 = bmax[1] > m_r[1] + kRescaleSlack;
    if (__any_sync(kAll, raise0 || raise1)) {
      float alpha[2] = {1.f, 1.f};
      if (raise0) { alpha[0] = ex2_approx(m_r[0] - bmax[0]); m_r[0] = bmax[0]; }
      if (raise1) { alpha[1] = ex2_approx(m_r[1] - bmax[1]); m_r[1] = bmax[1]; }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        l_r[r] *= alpha[r];
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][2 * r] *= alpha[r];
          o[n][2 * r + 1] *= alpha[r];
        }
      }
    }
  };

  // Second half: probabilities, row sums and O += P V from the V boxes at kt.
  // V rows of tokens past the causal limit (in the local block) may hold any
  // bytes, NaN patterns included (cache slots not written yet): their
  // probabilities are 0, but 0 x NaN is NaN, so the ldmatrix lanes of those
  // rows read a 16-byte zero row instead. (Zeroing them in the stage, which
  // the next tensor copy overwrites, raced with that copy.)
  auto softmax_pv = [&](uint32_t kt, const float (&sc)[kNT][4], int it_blk) {
    float pr[kNT][4];
    // p = 2^(s * mul - m): masked logits (-inf) give 0 since mul > 0; while the
    // reference is still -inf every logit so far is -inf, and 0 stands in for it.
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float neg_ref = m_r[r] == -INFINITY ? 0.f : -m_r[r];
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pv = ex2_approx(fmaf(sc[nt][2 * r + e], mul_r[r], neg_ref));
          pr[nt][2 * r + e] = pv;
          ls += pv;
        }
      }
      l_r[r] += ls;
    }
    // ---- O += P V (kKK k-steps of 16 tokens, 16 n-tiles of 8 dims)
    const bool local = it_blk == seg_ell;
#pragma unroll
    for (int kk = 0; kk < kKK; ++kk) {
      // the V row this lane addresses in each ldmatrix.x4.trans: token
      // 16 kk + 8 ((lane >> 3) & 1) + (lane & 7) of the warp's slice; past the
      // causal limit the lane points at a 16-byte zero row instead
      const bool zrow = local && it_blk * kBlock + kTokPerWarp * w + 16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7) > seg_p;
      const uint32_t zaddr = base_addr + Ly.zero;
      uint32_t a[4];
      if (kFp8) {
        a[0] = pack_f16x2(pr[2 * kk][0], pr[2 * kk][1]);
        a[1] = pack_f16x2(pr[2 * kk][2], pr[2 * kk][3]);
        a[2] = pack_f16x2(pr[2 * kk + 1][0], pr[2 * kk + 1][1]);
        a[3] = pack_f16x2(pr[2 * kk + 1][2], pr[2 * kk + 1][3]);
      } else {
        a[0] = pack_bf16x2(pr[2 * kk][0], pr[2 * kk][1]);
        a[1] = pack_bf16x2(pr[2 * kk][2], pr[2 * kk][3]);
        a[2] = pack_bf16x2(pr[2 * kk + 1][0], pr[2 * kk + 1][1]);
        a[3] = pack_bf16x2(pr[2 * kk + 1][2], pr[2 * kk + 1][3]);
      }
      if (kFp8) {
        // FP8 V: one ldmatrix.x4.trans per chunk pair (matrices: tokens 0-7 and
        // 8-15 of the k-step, for chunks 2 qp and 2 qp + 1) gives lane (gr, c)
        // tokens 2c, 2c+1 of dims 2 gr, 2 gr + 1 of a chunk; a byte permute
        // pairs the two tokens of each dim, and exact cvts make the fragments
        // of the chunk's even-dim (n-tile 2 chunk) and odd-dim (2 chunk + 1)
        // n-tiles.
        const uint32_t vt = kt + kFp8BoxBytes + kk * 16 * 128 + v8_row;
#pragma unroll
        for (int qp = 0; qp < 4; ++qp) {
          uint32_t v[4];
          const uint32_t va = vt + (((static_cast<uint32_t>(2 * qp) + (lane >> 4)) << 4) ^ lane_x);
          ldsm_x4_t(zrow ? zaddr : va, v[0], v[1], v[2], v[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t t0 = __byte_perm(v[2 * h], 0, 0x3120), t1 = __byte_perm(v[2 * h + 1], 0, 0x3120);
            const int n = 2 * (2 * qp + h);
            mma_f16(o[n], a, e4m3x2_to_f16x2(static_cast<uint16_t>(t0 & 0xFFFF)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(t1 & 0xFFFF)));
            mma_f16(o[n + 1], a, e4m3x2_to_f16x2(static_cast<uint16_t>(t0 >> 16)),
                    e4m3x2_to_f16x2(static_cast<uint16_t>(t1 >> 16)));
          }
        }
        continue;
      }
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b0, b1, b2, b3;
        const uint32_t va = kt + (2 + (np >> 2)) * kBoxBytes + kk * 16 * 128 + v_off[np & 3];
        ldsm_x4_t(zrow ? zaddr : va, b0, b1, b2, b3);
        mma_bf16(o[2 * np], a, b0, b1);
        mma_bf16(o[2 * np + 1], a, b2, b3);
      }
    }
  };

  // Item cursor: `cur` holds the infos of items base .. base + 31, `nxt` of the
  // 32 after them (loaded one chunk ahead).
  ItemInfo cur = load_item(p, x0 + lane, x1, false);
  ItemInfo nxt = load_item(p, x0 + 32 + lane, x1, false);
  int64_t base = x0;
  int kx = 0;
  int64_t xrow = x0 / p.K;                    // row and slot of the current item, advanced by one per item
  int xslot = static_cast<int>(x0 - xrow * p.K);
  int s = 0;
  uint32_t phase = 0;
  float sc[kNT][4];
  while (ok && base + kx < x1) {
    if (xrow != seg_row) {
      if (seg_row >= 0 && !end_segment()) { ok = false; break; }
      begin_segment(xrow);
    }
    const int valid = __shfl_sync(kAll, cur.valid, kx);
    const int it_blk = __shfl_sync(kAll, cur.blk, kx);
    if (++xslot == p.K) { xslot = 0; ++xrow; }
    if (++kx == 32) {
      kx = 0;
      base += 32;
      cur = nxt;
      nxt = load_item(p, base + 32 + lane, x1, false);
    }
    if (!valid) continue;
    const uint32_t kt = base_addr + Ly.stages + s * kStageBytes;   // bf16: K lo, K hi, V lo, V hi; FP8: K, V
    if (!mbar_wait(smem_addr(&full[s]), phase)) { ok = false; break; }
    qk(kt, sc);
    softmax_prep(sc, it_blk);
    softmax_pv(kt, sc, it_blk);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    if (++s == kGqaStages) { s = 0; phase ^= 1u; }
  }
  if (ok && seg_row >= 0) ok = end_segment();
  if (!ok && lane == 0) set_flag(p.flags, MSA_FLAG_TIMEOUT);
}

// ---------------------------------------------------------------------------
// NVFP4 K/V ("MiniMax-M3.1-Flash Day-0 対応", section "何が新しいか": E2M1
// values with an E4M3 scale per 16 and an fp32 global scale, 576 bytes per
// token per layer). The conversion to fp16 operands, not the copy of a block's
// 18 KB, sets the pace, so every block is spread over eight consumer warps of
// 16 tokens (two warps per SM sub-partition, which overlap each other's
// dependency chains). There is no producer warp: warp 0 also issues the
// copies, up to the stage count ahead of its own progress, and waits for a
// free stage only for the block it needs next. K codes are converted straight
// into mma operands: lane (r, c) of an n-tile loads the 16 code bytes
// 16c .. 16c + 15 of token r (dims 32c .. 32c + 31), so k-step s of the product
// takes dims 32c + 4s .. + 3 from every lane, and the query fragments are
// loaded with the same dims. V is expanded (E2M1 x E4M3 is exact in fp16) into
// the warp's rows of a swizzled fp16 tile, rows past the causal limit written
// as zeros, and read with ldmatrix.trans for P V; the stage is released after
// Q K^T. The fp32 global scales multiply the logits and the output.
// Work split: with few rows (every row's cluster resident at once), row r
// runs on cluster r of n = 2, 4 or 8 CTAs, CTA q taking slots [q K / n,
// (q + 1) K / n) and finalising heads [q, q + 1) 16 / n; the other CTAs push
// their merged partials of those heads into its receive buffer with st.async
// stores that complete bytes on its exchange barrier. Otherwise item ranges
// are balanced over the CTAs and split rows merged through the workspace, as
// in sparse_gqa_kernel. (The same eight-warp form for FP8 K/V measured slower
// than four warps on whole rows, 32.3 against 24.8 us on 32 x 32K: there the
// tensor and ALU pipes are both near saturation.)

constexpr int kF4Warps = 8;
constexpr int kF4Tok = kBlock / kF4Warps;          // 16 tokens per warp and block
constexpr int kF4Stages = 6;
constexpr uint32_t kF4Codes = kBlock * kDim / 2;   // 8 KB of E2M1 codes per K or V block
constexpr uint32_t kF4Scales = kBlock * kDim / 16; // 1 KB of E4M3 scales

// A cluster row's receive buffer: per sending CTA and finalised head, the 128
// output sums, then m and l (a 528-byte stride keeps the vector stores aligned).
constexpr int kXStride = kDim + 4;
constexpr uint32_t kXRecvBytes = 7 * 2 * kXStride * 4;   // the largest of (n - 1) x (16 / n) heads, n = 2, 4, 8
__host__ __device__ constexpr uint32_t cluster_expected_bytes(int n) {
  return static_cast<uint32_t>((n - 1) * (kGroup / n) * (kGroup * 32 + 8));   // 16 x 32 B + m, l per head
}

struct F4Layout {
  uint32_t stages, vtile, comb_o, comb_ml, xrecv, bars, total;
};
__host__ __device__ constexpr F4Layout f4_layout() {
  F4Layout s{};
  s.stages = 0;
  s.vtile = kF4Stages * kFp4StageBytes;                     // fp16 V: two 128-row x 64-dim swizzled boxes
  s.comb_o = s.vtile + 2 * kBoxBytes;
  s.comb_ml = s.comb_o + kF4Warps * kGroup * kDim * 4;
  s.xrecv = s.comb_ml + kF4Warps * kGroup * 2 * 4;
  s.bars = s.xrecv + kXRecvBytes;
  s.total = s.bars + (2 * kF4Stages + 2) * 8 + 16 + 8;      // + the last-arriver flag, the cluster exchange barrier
  return s;
}

__global__ void __launch_bounds__(32 * kF4Warps, 1) sparse_gqa_fp4_kernel(GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr uint32_t kStageBytes = kFp4StageBytes;
  constexpr F4Layout Ly = f4_layout();
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base_addr = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_addr - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Ly.bars);
  uint64_t* empty = full + kF4Stages;
  uint64_t* gbar = empty + kF4Stages;        // [0]: states staged, [1]: states read
  float* comb_o = reinterpret_cast<float*>(sm + Ly.comb_o);
  float* comb_m = reinterpret_cast<float*>(sm + Ly.comb_ml);
  float* comb_l = comb_m + kF4Warps * kGroup;
  int* last_flag = reinterpret_cast<int*>(sm + Ly.bars + (2 * kF4Stages + 2) * 8);
  uint64_t* xbar = reinterpret_cast<uint64_t*>(sm + Ly.bars + (2 * kF4Stages + 2) * 8 + 16);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, c = lane & 3;
  const bool clustered = p.cluster_n > 1;

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4Stages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kF4Warps);
    }
    mbar_init(smem_addr(&gbar[0]), kF4Warps);
    mbar_init(smem_addr(&gbar[1]), kF4Warps);
    if (clustered) {
      // armed now with the bytes the other CTAs will store into the receive buffer
      mbar_init(smem_addr(xbar), 1);
      mbar_arrive_expect_tx(smem_addr(xbar), cluster_expected_bytes(p.cluster_n));
    }
    fence_mbar_init();
  }
  __syncthreads();
  // The other CTAs store into this CTA's receive buffer only after every CTA
  // of the cluster passed this point (waited for at the row's end).
  if (clustered) cluster_arrive_relaxed();
  griddep_wait();

  const int C = gridDim.x;
  const uint32_t crank = clustered ? cluster_rank() : 0u;
  int64_t x0, x1;
  if (clustered) {
    // one row per cluster, its slots split evenly over the cluster's CTAs (K >= cluster_n)
    const int64_t r = blockIdx.x / p.cluster_n;
    x0 = r * p.K + static_cast<int64_t>(p.K) * crank / p.cluster_n;
    x1 = r * p.K + static_cast<int64_t>(p.K) * (crank + 1) / p.cluster_n;
  } else {
    x0 = p.W * blockIdx.x / C;
    x1 = p.W * (blockIdx.x + 1) / C;
    if (x0 >= x1) return;
  }
  if (p.scores != nullptr) {
    // Stage 2 inside this launch: every warp selects rows this CTA touches
    // (rows shared with other CTAs get the same result from each), staging its
    // survivors in the row-merge buffer, unused until a row ends.
    uint64_t* surv = reinterpret_cast<uint64_t*>(sm + Ly.comb_o) + w * (kWarpSurvCap + 8);
    int* chosen = reinterpret_cast<int*>(surv + kWarpSurvCap);
    for (int64_t r = x0 / p.K + w; r <= (x1 - 1) / p.K; r += kF4Warps) {
      const RowPos rp = row_pos(p, r);
      const int64_t row_off = (static_cast<int64_t>(rp.b) * p.Q + rp.j) * p.G + rp.g;
      int32_t* out = p.sel_out + row_off * p.K;
      const int L = p.seq_lens[rp.b];
      if (L < p.Q || L > p.NB * kBlock || L < 1) {           // (flagged by the item loads below)
        for (int e = lane; e < p.K; e += 32) out[e] = -1;
        continue;
      }
      warp_select_row(p.scores + row_off * p.NB, (L - p.Q + rp.j) / kBlock, p.K, out, surv, chosen, lane);
    }
    __syncthreads();                  // the item loads below read these rows back
  }
  const uint64_t pol = l2_evict_first_policy();
  uint32_t gph[2] = {0u, 0u};
  bool ok = true;

  // Item cursor (every warp): `cur` holds the infos of items base .. base + 31,
  // `nxt` the next 32. Warp 0 reports bad items (it also issues their copies).
  ItemInfo cur = load_item(p, x0 + lane, x1, w == 0);
  ItemInfo nxt = load_item(p, x0 + 32 + lane, x1, w == 0);
  int64_t base = x0;
  int kx = 0;

  // Copy issue (warp 0): item ia is the next to examine, `is` counts the valid
  // items whose copies were issued; the consumers have used `cs` valid items.
  int64_t ia = x0;
  int is = 0, cs = 0;
  auto issue_upto = [&](int need) {
    // issues the valid items' copies in order: waiting for a free stage until
    // `need` are issued, then while a stage is already free, at most
    // kF4Stages items ahead of this warp (items past the 64 loaded infos wait
    // for a later call)
    while (ok && ia < x1 && ia < base + 64 && is < cs + kF4Stages) {
      const int k = static_cast<int>(ia - base);
      const int valid = __shfl_sync(kAll, k < 32 ? cur.valid : nxt.valid, k & 31);
      const int page = __shfl_sync(kAll, k < 32 ? cur.page : nxt.page, k & 31);
      const int g = __shfl_sync(kAll, k < 32 ? cur.g : nxt.g, k & 31);
      if (!valid) { ++ia; continue; }
      const int s = is % kF4Stages;
      const uint32_t par = (static_cast<uint32_t>(is / kF4Stages) & 1u) ^ 1u;
      int go = 0;
      if (lane == 0) {
        if (is < need) go = mbar_wait(smem_addr(&empty[s]), par) ? 1 : -1;
        else go = mbar_test_wait(smem_addr(&empty[s]), par) ? 1 : 0;
        if (go == 1) {
          const uint32_t fb = smem_addr(&full[s]);
          const uint32_t dst = base_addr + Ly.stages + s * kStageBytes;
          const int64_t ph = static_cast<int64_t>(page) * p.G + g;
          mbar_arrive_expect_tx(fb, kStageBytes);
          bulk_g2s(dst, p.k4 + ph * kF4Codes, kF4Codes, fb, pol);
          bulk_g2s(dst + kF4Codes, p.ks + ph * kF4Scales, kF4Scales, fb, pol);
          bulk_g2s(dst + kF4Codes + kF4Scales, p.v4 + ph * kF4Codes, kF4Codes, fb, pol);
          bulk_g2s(dst + 2 * kF4Codes + kF4Scales, p.vs + ph * kF4Scales, kF4Scales, fb, pol);
        }
      }
      go = __shfl_sync(kAll, go, 0);
      if (go < 0) { set_flag(p.flags, MSA_FLAG_TIMEOUT); ok = false; break; }
      if (go == 0) break;
      ++ia;
      ++is;
    }
  };

  if (w == 0) issue_upto(0);        // the first copies, before the first row's query loads

  uint32_t qf[8][4];
  float o[16][4];
  float m_r[2], l_r[2], mul_r[2];
  int64_t seg_row = -1;
  int seg_b = 0, seg_g = 0, seg_j = 0, seg_p = 0, seg_ell = 0;

  auto begin_segment = [&](int64_t r) {
    const RowPos rp = row_pos(p, r);
    seg_row = r;
    seg_b = rp.b; seg_g = rp.g; seg_j = rp.j;
    seg_p = p.seq_lens[rp.b] - p.Q + rp.j;
    seg_ell = seg_p / kBlock;
    const uint16_t* qh = p.q + ((static_cast<int64_t>(rp.b) * p.Q + rp.j) * p.H + static_cast<int64_t>(rp.g) * kGroup) * kDim;
    // k-step s, lane c: dims 32c + 4s .. + 3 (a0/a1: the first two, a2/a3: the last two)
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint2 wq = *reinterpret_cast<const uint2*>(qh + (gr + 8 * r) * kDim + 32 * c + 4 * s);
        qf[s][r] = wq.x;
        qf[s][2 + r] = wq.y;
      }
    }
    // fp16 operands: each query row scaled by an exact power of two into range
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float amax = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t wq = qf[s][2 * h + r];
          amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(wq & 0xFFFF)), fabsf(bf16_bits_to_f32(wq >> 16))));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, 2));
      const int sh = fp16_shift_for(amax);
      const float f = exp2_int(sh);
      mul_r[r] = p.scale_log2 * p.k_global * exp2_int(-sh);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t wq = qf[s][2 * h + r];
          qf[s][2 * h + r] = pack_f16x2(bf16_bits_to_f32(wq & 0xFFFF) * f, bf16_bits_to_f32(wq >> 16) * f);
        }
      }
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m_r[0] = m_r[1] = -INFINITY;
    l_r[0] = l_r[1] = 0.f;
  };

  // Merges the eight warps' states of the current row; writes the output when
  // the CTA covered the whole row, a split-K partial otherwise (the CTA that
  // delivers a row's last partial merges them all, or in a cluster every CTA
  // its share of the heads).
  bool cluster_done = false;          // this thread took part in the cluster's exchange
  auto end_segment = [&]() -> bool {
    float lt[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float v = l_r[r];
      v += __shfl_xor_sync(kAll, v, 1);
      v += __shfl_xor_sync(kAll, v, 2);
      lt[r] = v;
    }
    {
      float* mo = comb_o + w * kGroup * kDim;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        *reinterpret_cast<float2*>(mo + gr * kDim + 8 * n + 2 * c) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2*>(mo + (gr + 8) * kDim + 8 * n + 2 * c) = make_float2(o[n][2], o[n][3]);
      }
      if (c == 0) {
        comb_m[w * kGroup + gr] = m_r[0];
        comb_m[w * kGroup + gr + 8] = m_r[1];
        comb_l[w * kGroup + gr] = lt[0];
        comb_l[w * kGroup + gr + 8] = lt[1];
      }
    }
    if (!group_sync(smem_addr(&gbar[0]), gph[0], lane)) return false;
    // 256 threads: head hh = tid / 16, dims d0 .. d0 + 7
    const int tid = threadIdx.x;
    const int hh = tid >> 4, d0 = (tid & 15) * 8;
    float M = -INFINITY, Ls = 0.f;
    float acc[8];
#pragma unroll
    for (int k = 0; k < kF4Warps; ++k) M = fmaxf(M, comb_m[k * kGroup + hh]);
#pragma unroll
    for (int d = 0; d < 8; ++d) acc[d] = 0.f;
#pragma unroll
    for (int k = 0; k < kF4Warps; ++k) {
      const float fw = M == -INFINITY ? 0.f : ex2_approx(comb_m[k * kGroup + hh] - M);
      Ls += fw * comb_l[k * kGroup + hh];
      const float4 a = *reinterpret_cast<const float4*>(comb_o + (k * kGroup + hh) * kDim + d0);
      const float4 b = *reinterpret_cast<const float4*>(comb_o + (k * kGroup + hh) * kDim + d0 + 4);
      acc[0] += fw * a.x; acc[1] += fw * a.y; acc[2] += fw * a.z; acc[3] += fw * a.w;
      acc[4] += fw * b.x; acc[5] += fw * b.y; acc[6] += fw * b.z; acc[7] += fw * b.w;
    }
#pragma unroll
    for (int d = 0; d < 8; ++d) acc[d] *= p.v_global;
    const int64_t r = seg_row;
    const bool whole = x0 <= r * p.K && (r + 1) * p.K <= x1;
    const int64_t head = (static_cast<int64_t>(seg_b) * p.Q + seg_j) * p.H + static_cast<int64_t>(seg_g) * kGroup + hh;
    auto write_out = [&](const float (&v)[8], float mm, float ll) {
      const float inv = ll > 0.f ? 1.f / ll : 0.f;
      uint4 pk;
      pk.x = pack_bf16x2(v[0] * inv, v[1] * inv);
      pk.y = pack_bf16x2(v[2] * inv, v[3] * inv);
      pk.z = pack_bf16x2(v[4] * inv, v[5] * inv);
      pk.w = pack_bf16x2(v[6] * inv, v[7] * inv);
      *reinterpret_cast<uint4*>(p.out + head * kDim + d0) = pk;
      if (p.lse != nullptr && (tid & 15) == 0) p.lse[head] = ll > 0.f ? (mm + log2f(ll)) * kLn2 : -INFINITY;
    };
    if (clustered) {
      // CTA q finalises heads [q, q + 1) * 16 / cluster_n. Every other CTA
      // stores its partials of those heads straight into q's receive buffer
      // (asynchronous stores that complete bytes on q's exchange barrier, armed
      // at the start); q waits for the barrier, merges in sender order and
      // writes the output.
      const int hpc = kGroup / p.cluster_n;
      const int dest = hh / hpc, hl = hh - dest * hpc;
      const int me = static_cast<int>(crank);
      const uint32_t xrecv = base_addr + Ly.xrecv;
      cluster_done = true;
      cluster_wait();                     // every CTA's exchange barrier is armed
      if (dest != me) {
        const int j = me < dest ? me : me - 1;                  // this CTA's sender slot at dest
        const uint32_t slot = xrecv + static_cast<uint32_t>((j * hpc + hl) * kXStride) * 4u;
        const uint32_t rbar = cluster_map(smem_addr(xbar), dest);
        st_async_v4(cluster_map(slot + d0 * 4, dest), acc[0], acc[1], acc[2], acc[3], rbar);
        st_async_v4(cluster_map(slot + d0 * 4 + 16, dest), acc[4], acc[5], acc[6], acc[7], rbar);
        if ((tid & 15) == 0) st_async_v2(cluster_map(slot + kDim * 4, dest), M, Ls, rbar);
      }
      bool got = true;
      if (dest == me) {
        got = mbar_wait(smem_addr(xbar), 0u);
        const float* xr = reinterpret_cast<const float*>(sm + Ly.xrecv);
        for (int j = 0; got && j < p.cluster_n - 1; ++j) {
          const float* pq = xr + (j * hpc + hl) * kXStride;
          const float Mq = pq[kDim], Lq = pq[kDim + 1];
          if (Mq == -INFINITY) continue;
          const float4 a = *reinterpret_cast<const float4*>(pq + d0);
          const float4 b = *reinterpret_cast<const float4*>(pq + d0 + 4);
          const float Mn = fmaxf(M, Mq);
          const float fs = M == -INFINITY ? 0.f : ex2_approx(M - Mn), fq = ex2_approx(Mq - Mn);
          Ls = fs * Ls + fq * Lq;
          acc[0] = fs * acc[0] + fq * a.x; acc[1] = fs * acc[1] + fq * a.y;
          acc[2] = fs * acc[2] + fq * a.z; acc[3] = fs * acc[3] + fq * a.w;
          acc[4] = fs * acc[4] + fq * b.x; acc[5] = fs * acc[5] + fq * b.y;
          acc[6] = fs * acc[6] + fq * b.z; acc[7] = fs * acc[7] + fq * b.w;
          M = Mn;
        }
        if (got) write_out(acc, M, Ls);
      }
      // no CTA leaves while another may still store into it
      cluster_arrive_relaxed();
      cluster_wait();
      return got;
    }
    if (whole) {
      write_out(acc, M, Ls);
      return group_sync(smem_addr(&gbar[1]), gph[1], lane);
    }
    const int first = cta_of(r * p.K, p.W, C);
    const int nslots = cta_of(r * p.K + p.K - 1, p.W, C) - first + 1;
    float* rowp = p.ws + r * p.K * static_cast<int64_t>(kPartialFloats);
    float* part = rowp + (static_cast<int>(blockIdx.x) - first) * static_cast<int64_t>(kPartialFloats);
    {
      float4* dst = reinterpret_cast<float4*>(part + hh * kDim + d0);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      if ((tid & 15) == 0) {
        part[kGroup * kDim + hh] = M;
        part[kGroup * kDim + kGroup + hh] = Ls;
      }
    }
    if (!group_sync(smem_addr(&gbar[1]), gph[1], lane)) return false;
    if (tid == 32) {              // not warp 0's lane 0, whose bulk copies may still be in flight
      fence_acq_rel_gpu();
      const bool last = ticket_is_last(p, r, nslots);
      if (last) fence_acq_rel_gpu();
      *last_flag = last ? 1 : 0;
    }
    if (!group_sync(smem_addr(&gbar[0]), gph[0], lane)) return false;
    if (*last_flag) {
      float M2 = -INFINITY;
      for (int q = 0; q < nslots; ++q) M2 = fmaxf(M2, __ldcg(rowp + q * kPartialFloats + kGroup * kDim + hh));
      float L2 = 0.f;
      float v[8];
#pragma unroll
      for (int d = 0; d < 8; ++d) v[d] = 0.f;
      if (M2 != -INFINITY) {
        for (int q = 0; q < nslots; ++q) {
          const float* pq = rowp + q * kPartialFloats;
          const float f = ex2_approx(__ldcg(pq + kGroup * kDim + hh) - M2);
          L2 += f * __ldcg(pq + kGroup * kDim + kGroup + hh);
          const float4 a = __ldcg(reinterpret_cast<const float4*>(pq + hh * kDim + d0));
          const float4 b = __ldcg(reinterpret_cast<const float4*>(pq + hh * kDim + d0 + 4));
          v[0] += f * a.x; v[1] += f * a.y; v[2] += f * a.z; v[3] += f * a.w;
          v[4] += f * b.x; v[5] += f * b.y; v[6] += f * b.z; v[7] += f * b.w;
        }
      }
      write_out(v, M2, L2);
    }
    return true;
  };

  const uint32_t vtile = base_addr + Ly.vtile;
  uint32_t v_off[4];
#pragma unroll
  for (int h = 0; h < 4; ++h)
    v_off[h] = (static_cast<uint32_t>(kF4Tok * w) + 8 * ((lane >> 3) & 1) + (lane & 7)) * 128u +
               ((((2 * h) + (lane >> 4)) ^ (lane & 7)) << 4);

  int s = 0;
  uint32_t phase = 0;
  int64_t xrow = x0 / p.K;
  int xslot = static_cast<int>(x0 - xrow * p.K);
  while (ok && base + kx < x1) {
    if (xrow != seg_row) {
      if (seg_row >= 0 && !end_segment()) { ok = false; break; }
      begin_segment(xrow);
    }
    const int valid = __shfl_sync(kAll, cur.valid, kx);
    const int it_blk = __shfl_sync(kAll, cur.blk, kx);
    if (++xslot == p.K) { xslot = 0; ++xrow; }
    if (!valid) {
      if (++kx == 32) { kx = 0; base += 32; cur = nxt; nxt = load_item(p, base + 32 + lane, x1, w == 0); }
      continue;
    }
    if (w == 0) issue_upto(cs + 1);                 // this item's copy, and more while stages are free
    if (!mbar_wait(smem_addr(&full[s]), phase)) { ok = false; break; }
    const uint8_t* st = sm + Ly.stages + s * kStageBytes;
    const int tb = it_blk * kBlock + kF4Tok * w;   // first token of this warp's rows
    // ---- V rows of this warp -> fp16 tile (rows past the causal limit as zeros)
    {
      const int row = kF4Tok * w + (lane >> 1), hh = lane & 1;
      const uint8_t* vc = st + kF4Codes + kF4Scales + row * 64 + 32 * hh;
      const uint4 c0 = *reinterpret_cast<const uint4*>(vc);
      const uint4 c1 = *reinterpret_cast<const uint4*>(vc + 16);
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(st + 2 * kF4Codes + kF4Scales + row * 8 + 4 * hh);
      const bool live = tb + (lane >> 1) <= seg_p;
      const uint32_t s01 = e4m3x2_to_f16x2(static_cast<uint16_t>(sw & 0xFFFF));
      const uint32_t s23 = e4m3x2_to_f16x2(static_cast<uint16_t>(sw >> 16));
      const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const uint32_t box = vtile + hh * kBoxBytes;
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {               // 16 dims: scale group 4 hh + gg
        const uint32_t sg = gg < 2 ? s01 : s23;
        const __half2 scl = __half2half2(__ushort_as_half(static_cast<unsigned short>((gg & 1) ? (sg >> 16) : (sg & 0xFFFF))));
#pragma unroll
        for (int k = 0; k < 2; ++k) {                // 8 dims -> one 16-byte chunk
          uint32_t h[4];
          e2m1x8_to_f16x2x4(words[2 * gg + k], h);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h[e]), scl);
            h[e] = live ? *reinterpret_cast<uint32_t*>(&v) : 0u;
          }
          const uint32_t a = swz(box, row, 2 * gg + k);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                       "r"(h[3])
                       : "memory");
        }
      }
    }
    // ---- S = Q K^T for the warp's 16 tokens, K codes converted in registers
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const int t = kF4Tok * w + 8 * nt + gr;
      const uint4 cw = *reinterpret_cast<const uint4*>(st + t * 64 + 16 * c);
      const uint32_t s2 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(st + kF4Codes + t * 8 + 2 * c));
      const __half2 sa = __half2half2(__ushort_as_half(static_cast<unsigned short>(s2 & 0xFFFF)));
      const __half2 sb = __half2half2(__ushort_as_half(static_cast<unsigned short>(s2 >> 16)));
      const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {               // word q4: k-steps 2 q4 and 2 q4 + 1
        uint32_t h[4];
        e2m1x8_to_f16x2x4(words[q4], h);
        const __half2 scl = q4 < 2 ? sa : sb;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h[e]), scl);
          h[e] = *reinterpret_cast<uint32_t*>(&v);
        }
        mma_f16(sc[nt], qf[2 * q4], h[0], h[1]);
        mma_f16(sc[nt], qf[2 * q4 + 1], h[2], h[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[s]));   // codes no longer needed
    ++cs;
    if (++s == kF4Stages) { s = 0; phase ^= 1u; }
    if (w == 0) issue_upto(cs);
    // ---- causal limit, online softmax (log2 domain), P V
    if (it_blk == seg_ell) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int t0 = tb + 8 * nt + 2 * c;
        if (t0 > seg_p) { sc[nt][0] = -INFINITY; sc[nt][2] = -INFINITY; }
        if (t0 + 1 > seg_p) { sc[nt][1] = -INFINITY; sc[nt][3] = -INFINITY; }
      }
    }
    float bmax[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = fmaxf(fmaxf(sc[0][2 * r], sc[0][2 * r + 1]), fmaxf(sc[1][2 * r], sc[1][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
      bmax[r] = mx * mul_r[r];
    }
    const bool raise0 = bmax[0] > m_r[0] + kRescaleSlack, raise1 = bmax[1] > m_r[1] + kRescaleSlack;
    if (__any_sync(kAll, raise0 || raise1)) {
      float alpha[2] = {1.f, 1.f};
      if (raise0) { alpha[0] = ex2_approx(m_r[0] - bmax[0]); m_r[0] = bmax[0]; }
      if (raise1) { alpha[1] = ex2_approx(m_r[1] - bmax[1]); m_r[1] = bmax[1]; }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        l_r[r] *= alpha[r];
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[n][2 * r] *= alpha[r];
          o[n][2 * r + 1] *= alpha[r];
        }
      }
    }
    float pr[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float neg_ref = m_r[r] == -INFINITY ? 0.f : -m_r[r];
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pv = ex2_approx(fmaf(sc[nt][2 * r + e], mul_r[r], neg_ref));
          pr[nt][2 * r + e] = pv;
          ls += pv;
        }
      }
      l_r[r] += ls;
    }
    {
      uint32_t a[4];
      a[0] = pack_f16x2(pr[0][0], pr[0][1]);
      a[1] = pack_f16x2(pr[0][2], pr[0][3]);
      a[2] = pack_f16x2(pr[1][0], pr[1][1]);
      a[3] = pack_f16x2(pr[1][2], pr[1][3]);
      __syncwarp();                                   // the warp's V rows are in the tile
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vtile + (np >> 2) * kBoxBytes + v_off[np & 3], b0, b1, b2, b3);
        mma_f16(o[2 * np], a, b0, b1);
        mma_f16(o[2 * np + 1], a, b2, b3);
      }
      __syncwarp();                                   // before the next block's expansion overwrites the rows
    }
    if (++kx == 32) { kx = 0; base += 32; cur = nxt; nxt = load_item(p, base + 32 + lane, x1, w == 0); }
  }
  if (ok && seg_row >= 0) ok = end_segment();
  if (clustered && !cluster_done) {
    // a wait gave up before the row's exchange (the other CTAs' waits for
    // this CTA's partials then give up too, flagged): still pass the cluster
    // barriers that they wait on before leaving
    cluster_wait();
    cluster_arrive_relaxed();
    cluster_wait();
  }
  if (!ok && lane == 0) set_flag(p.flags, MSA_FLAG_TIMEOUT);
  if (w == 0 && lane == 0) {
    // no copy of this CTA may still be in flight when it exits
    for (int k = is > kF4Stages ? is - kF4Stages : 0; k < is; ++k)
      if (!mbar_wait(smem_addr(&full[k % kF4Stages]), static_cast<uint32_t>((k / kF4Stages) & 1))) break;
  }
}

// ---------------------------------------------------------------------------
// Several query positions per request (speculative verification: "MiniMax M3
// vLLM サポート：…", section "EAGLE3 を用いた投機的デコード", every draft
// position of a request in one decode pass). The positions of one (request,
// KV head) pair share their local block and often more, so this form streams
// the union of their selected blocks once instead of once per position. One
// CTA owns a (request, KV head) group: a producer warp copies each union block
// (bf16 K and V, 64 KB) into a stage, and consumer warp j attends for query
// position j over the blocks of its own selection, all 128 tokens of each in
// four 32-token slices, with its own online softmax and causal limit. A stage
// is released once every position that selected its block has used it; when
// the producer fills a stage it arrives in advance for the positions that did
// not select the block. Each position's output is complete in one warp, so
// there is no split-K merge. Every wait is bounded.

constexpr int kUnWarps = 8;                      // consumer warps: one per query position (q_len <= 8)
constexpr int kUnStages = 3;                     // 64 KB bf16 K/V tiles
constexpr int kUnMaxNB = 8192;                   // block bitmaps kept in shared memory up to this many blocks
constexpr int kUnAhead = 1;                      // union blocks prefetched into L2 beyond the stages (1: measured best)

struct UnLayout {
  uint32_t stages, surv, bits, ubits, prefix, ulist, tags, bars, zero, total;
};

// nw = 32-bit words per block bitmap (ceil(NB / 32)).
__host__ __device__ inline UnLayout un_layout(int nw) {
  UnLayout s{};
  s.stages = 0;
  s.surv = kUnStages * kTileBytes;                               // fused selection: each warp's survivors
  s.bits = s.surv + (1 + kUnWarps) * (kWarpSurvCap + 8) * 8;     // [kUnWarps][nw] selected blocks per position
  s.ubits = s.bits + kUnWarps * nw * 4;                          // [nw] their union
  s.prefix = s.ubits + nw * 4;                                   // [nw] union blocks in the words before
  s.ulist = s.prefix + nw * 4;                                   // [kUnWarps * 16] union blocks in ascending order
  s.tags = s.ulist + kUnWarps * 16 * 4;                          // [kUnStages] union index held by each stage, abort word
  s.bars = (s.tags + (kUnStages + 2) * 4 + 7) & ~7u;
  s.zero = (s.bars + 2 * kUnStages * 8 + 15) & ~15u;            // 16 zero bytes: the V row of a token past L - 1
  s.total = s.zero + 16;
  return s;
}

__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Waits until *tag == n (a stage filled with union block n), bounded in time.
__device__ __forceinline__ bool wait_tag(const volatile int* tag, int n) {
  if (*tag == n) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (*tag == n) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__global__ void __launch_bounds__(32 * (1 + kUnWarps), 1)
    sparse_gqa_union_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                            GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base_addr = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_addr - raw);
  const int nw = (p.NB + 31) >> 5;
  const UnLayout Ly = un_layout(nw);
  uint32_t* bits = reinterpret_cast<uint32_t*>(sm + Ly.bits);
  uint32_t* ubits = reinterpret_cast<uint32_t*>(sm + Ly.ubits);
  int* prefix = reinterpret_cast<int*>(sm + Ly.prefix);
  int* ulist = reinterpret_cast<int*>(sm + Ly.ulist);
  volatile int* tags = reinterpret_cast<volatile int*>(sm + Ly.tags);
  volatile int* abort_flag = tags + kUnStages;
  volatile int* group_total = tags + kUnStages + 1;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Ly.bars);
  uint64_t* empty = full + kUnStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kUnStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kUnWarps);
      tags[s] = -1;
    }
    *abort_flag = 0;
    st_shared_zero16(base_addr + Ly.zero);
    fence_mbar_init();
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  __syncthreads();
  griddep_wait();

  const int groups = p.B * p.G;
  const int j = warp - 1;                       // consumers: query position
  const int gr = lane >> 2, c = lane & 3;
  int n_base = 0;                               // union index of the group's first block (counted over the CTA's groups)
  int n_issued = 0;                             // producer: union blocks whose copies it issued
  bool ok = true;

  // ldmatrix offsets inside a 32-token slice (slice q adds q * 4096 bytes,
  // which keeps every row's 128-byte swizzle phase)
  uint32_t k_off[2], v_off[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) k_off[h] = (lane & 7) * 128u + ((((4 * h) + (lane >> 3)) ^ (lane & 7)) << 4);
#pragma unroll
  for (int h = 0; h < 4; ++h)
    v_off[h] = (8 * ((lane >> 3) & 1) + (lane & 7)) * 128u + ((((2 * h) + (lane >> 4)) ^ (lane & 7)) << 4);

  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int b = grp / p.G, g = grp - b * p.G;
    const int L = p.seq_lens[b];
    const bool len_ok = L >= p.Q && L >= 1 && L <= p.NB * kBlock;
    // 1. (fused) selection of the group's rows; bitmaps cleared
    for (int i = threadIdx.x; i < kUnWarps * nw; i += blockDim.x) bits[i] = 0u;
    if (p.scores != nullptr && warp < p.Q) {
      const int64_t row_off = (static_cast<int64_t>(b) * p.Q + warp) * p.G + g;
      int32_t* out = p.sel_out + row_off * p.K;
      uint64_t* surv = reinterpret_cast<uint64_t*>(sm + Ly.surv) + warp * (kWarpSurvCap + 8);
      if (!len_ok) {
        for (int e = lane; e < p.K; e += 32) out[e] = -1;
      } else {
        warp_select_row(p.scores + row_off * p.NB, (L - p.Q + warp) / kBlock, p.K, out, surv,
                        reinterpret_cast<int*>(surv + kWarpSurvCap), lane);
      }
    }
    __syncthreads();
    // 2. each position's valid selected blocks into its bitmap
    if (j >= 0 && j < p.Q) {
      if (!len_ok) {
        if (j == 0 && lane == 0) set_flag(p.flags, MSA_FLAG_BAD_SEQLEN);
      } else {
        const int ell = (L - p.Q + j) / kBlock;
        const int32_t* sel = p.selected + ((static_cast<int64_t>(b) * p.Q + j) * p.G + g) * p.K;
        for (int e = lane; e < p.K; e += 32) {
          const int blk = sel[e];
          if (blk < 0) continue;
          if (blk > ell) { set_flag(p.flags, MSA_FLAG_BAD_BLOCK); continue; }
          const int page = p.block_table[static_cast<int64_t>(b) * p.NB + blk];
          if (page < 0 || page >= p.P) { set_flag(p.flags, MSA_FLAG_BAD_PAGE); continue; }
          atomicOr(&bits[j * nw + (blk >> 5)], 1u << (blk & 31));
        }
      }
    }
    __syncthreads();
    // 3. union and its running count per word (producer warp)
    if (warp == 0) {
      int run = 0;
      for (int w0 = 0; w0 < nw; w0 += 32) {
        const int w = w0 + lane;
        uint32_t u = 0u;
        if (w < nw)
          for (int q = 0; q < p.Q; ++q) u |= bits[q * nw + w];
        const int cnt = __popc(u);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(kAll, incl, o);
          if (lane >= o) incl += t;
        }
        if (w < nw) {
          ubits[w] = u;
          prefix[w] = run + incl - cnt;
          int at = run + incl - cnt;             // the union's blocks in ascending order (at most 8 x 16)
          for (uint32_t v = u; v != 0u; v &= v - 1u) ulist[at++] = (w << 5) + __ffs(v) - 1;
        }
        run += __shfl_sync(kAll, incl, 31);
      }
      if (lane == 0) *group_total = run;
    }
    __syncthreads();
    const int total = *group_total;

    if (warp == 0) {
      // ------------------------------------------------------------ producer --
      // Union block i goes to stage (n_base + i) % kUnStages. Lane 0 also asks
      // L2 for the K and V slabs of block i + kUnStages + kUnAhead - 1, so that
      // when a stage frees its copy finds the data close by.
      auto l2_prefetch = [&](int i) {
        if (i < total) {
          const int page = p.block_table[static_cast<int64_t>(b) * p.NB + ulist[i]];
          const int64_t off = (static_cast<int64_t>(page) * p.G + g) * (kBlock * kDim * 2);
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.k4 + off), "r"(kBlock * kDim * 2) : "memory");
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.v4 + off), "r"(kBlock * kDim * 2) : "memory");
        }
      };
      if (lane == 0)
        for (int i = kUnStages; i < kUnStages + kUnAhead - 1; ++i) l2_prefetch(i);
      for (int i = 0; i < total && ok; ++i) {
        if (lane == 0) {
          const int n = n_base + i;
          const int s = n % kUnStages;
          const uint32_t ph = static_cast<uint32_t>(n / kUnStages) & 1u;
          if (!mbar_wait(smem_addr(&empty[s]), ph ^ 1u)) {
            set_flag(p.flags, MSA_FLAG_TIMEOUT);
            ok = false;
          } else {
            const int blk = ulist[i];
            const int w = blk >> 5, bit = blk & 31;
            int users = 0;
            for (int q = 0; q < p.Q; ++q) users += (bits[q * nw + w] >> bit) & 1;
            tags[s] = n;
            if (users < kUnWarps) mbar_arrive_n(smem_addr(&empty[s]), static_cast<uint32_t>(kUnWarps - users));
            const int page = p.block_table[static_cast<int64_t>(b) * p.NB + blk];
            const int y = static_cast<int>((static_cast<int64_t>(page) * p.G + g) * kBlock);
            const uint32_t fb = smem_addr(&full[s]);
            const uint32_t dst = base_addr + Ly.stages + s * kTileBytes;
            mbar_arrive_expect_tx(fb, kTileBytes);
            tma_load_2d(dst, &tk, 0, y, fb);
            tma_load_2d(dst + kBoxBytes, &tk, 64, y, fb);
            tma_load_2d(dst + 2 * kBoxBytes, &tv, 0, y, fb);
            tma_load_2d(dst + 3 * kBoxBytes, &tv, 64, y, fb);
            l2_prefetch(i + kUnStages + kUnAhead - 1);
          }
        }
        ok = __shfl_sync(kAll, ok ? 1 : 0, 0) != 0;
        if (ok) n_issued = n_base + i + 1;
      }
    } else if (j < p.Q) {
      // ------------------------------------------------- consumer: position j --
      const int pj = L - p.Q + j;                 // causal limit of position j (valid when len_ok)
      const int ell = pj / kBlock;
      const int last_blk = (L - 1) / kBlock;      // block holding the last cached token
      uint32_t qf[8][4];
      float o[16][4];
      float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
      const float mul = p.scale_log2;
#pragma unroll
      for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      if (len_ok) {
        const uint16_t* qh =
            p.q + ((static_cast<int64_t>(b) * p.Q + j) * p.H + static_cast<int64_t>(g) * kGroup) * kDim;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint16_t* row = qh + (gr + 8 * r) * kDim + 16 * s + 2 * c;
            qf[s][r] = *reinterpret_cast<const uint32_t*>(row);
            qf[s][2 + r] = *reinterpret_cast<const uint32_t*>(row + 8);
          }
        }
      }
      for (int w = 0; w < nw && ok && len_ok; ++w) {
        uint32_t mine = bits[j * nw + w];
        const uint32_t uw = ubits[w];
        const int pw = prefix[w];
        while (mine != 0u) {
          const int bit = __ffs(mine) - 1;
          mine &= mine - 1u;
          const int blk = (w << 5) + bit;
          const int n = n_base + pw + __popc(uw & ((1u << bit) - 1u));
          const int s = n % kUnStages;
          if (!wait_tag(tags + s, n) ||
              !mbar_wait(smem_addr(&full[s]), static_cast<uint32_t>(n / kUnStages) & 1u)) {
            ok = false;
            break;
          }
          const uint32_t kt = base_addr + Ly.stages + s * kTileBytes;
#pragma unroll 1
          for (int qs = 0; qs < kBlock / kTokPerWarp; ++qs) {
            const uint32_t ks = kt + qs * (kTokPerWarp * 128u);
            float sc[kNT][4];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int sp = 0; sp < 4; ++sp) {
              const uint32_t kb = ks + (sp >> 1) * kBoxBytes + k_off[sp & 1];
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {          // two n-tiles at a time: 9 warps leave 168 registers
                uint32_t bq[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                  ldsm_x4(kb + (2 * h2 + nt) * 8 * 128, bq[nt][0], bq[nt][1], bq[nt][2], bq[nt][3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) mma_bf16(sc[2 * h2 + nt], qf[2 * sp], bq[nt][0], bq[nt][1]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) mma_bf16(sc[2 * h2 + nt], qf[2 * sp + 1], bq[nt][2], bq[nt][3]);
              }
            }
            const int tbase = blk * kBlock + qs * kTokPerWarp;
            if (blk == ell) {                       // causal limit of this position
#pragma unroll
              for (int nt = 0; nt < kNT; ++nt) {
                const int t0 = tbase + 8 * nt + 2 * c;
                if (t0 > pj) { sc[nt][0] = -INFINITY; sc[nt][2] = -INFINITY; }
                if (t0 + 1 > pj) { sc[nt][1] = -INFINITY; sc[nt][3] = -INFINITY; }
              }
            }
            // online softmax, log2 domain (as in sparse_gqa_kernel)
            float bmax[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              float mx = -INFINITY;
#pragma unroll
              for (int nt = 0; nt < kNT; ++nt) mx = fmaxf(mx, fmaxf(sc[nt][2 * r], sc[nt][2 * r + 1]));
              mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
              mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
              bmax[r] = mx * mul;
            }
            const bool raise0 = bmax[0] > m_r[0] + kRescaleSlack, raise1 = bmax[1] > m_r[1] + kRescaleSlack;
            if (__any_sync(kAll, raise0 || raise1)) {
              float alpha[2] = {1.f, 1.f};
              if (raise0) { alpha[0] = ex2_approx(m_r[0] - bmax[0]); m_r[0] = bmax[0]; }
              if (raise1) { alpha[1] = ex2_approx(m_r[1] - bmax[1]); m_r[1] = bmax[1]; }
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                l_r[r] *= alpha[r];
#pragma unroll
                for (int n2 = 0; n2 < 16; ++n2) {
                  o[n2][2 * r] *= alpha[r];
                  o[n2][2 * r + 1] *= alpha[r];
                }
              }
            }
            float pr[kNT][4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const float neg_ref = m_r[r] == -INFINITY ? 0.f : -m_r[r];
              float ls = 0.f;
#pragma unroll
              for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float pv = ex2_approx(fmaf(sc[nt][2 * r + e], mul, neg_ref));
                  pr[nt][2 * r + e] = pv;
                  ls += pv;
                }
              }
              l_r[r] += ls;
            }
            // V rows past the last cached token may hold any bytes (never
            // written): every position gives them probability 0, and the
            // ldmatrix lanes of those rows read a 16-byte zero row instead
            // (0 x NaN is NaN)
#pragma unroll
            for (int kk = 0; kk < kKK; ++kk) {
              const bool zrow = blk == last_blk && tbase + 16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7) > L - 1;
              uint32_t a[4];
              a[0] = pack_bf16x2(pr[2 * kk][0], pr[2 * kk][1]);
              a[1] = pack_bf16x2(pr[2 * kk][2], pr[2 * kk][3]);
              a[2] = pack_bf16x2(pr[2 * kk + 1][0], pr[2 * kk + 1][1]);
              a[3] = pack_bf16x2(pr[2 * kk + 1][2], pr[2 * kk + 1][3]);
#pragma unroll
              for (int np = 0; np < 8; ++np) {
                uint32_t b0, b1, b2, b3;
                const uint32_t va = ks + (2 + (np >> 2)) * kBoxBytes + kk * 16 * 128 + v_off[np & 3];
                ldsm_x4_t(zrow ? base_addr + Ly.zero : va, b0, b1, b2, b3);
                mma_bf16(o[2 * np], a, b0, b1);
                mma_bf16(o[2 * np + 1], a, b2, b3);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
        }
      }
      // position j's output: 16 heads of KV head g
      float lt[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float v = l_r[r];
        v += __shfl_xor_sync(kAll, v, 1);
        v += __shfl_xor_sync(kAll, v, 2);
        lt[r] = v;
      }
      const int64_t head0 = (static_cast<int64_t>(b) * p.Q + j) * p.H + static_cast<int64_t>(g) * kGroup;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float inv = lt[r] > 0.f ? 1.f / lt[r] : 0.f;
        uint16_t* orow = p.out + (head0 + gr + 8 * r) * kDim + 2 * c;
#pragma unroll
        for (int n2 = 0; n2 < 16; ++n2)
          *reinterpret_cast<uint32_t*>(orow + 8 * n2) = pack_bf16x2(o[n2][2 * r] * inv, o[n2][2 * r + 1] * inv);
        if (p.lse != nullptr && c == 0)
          p.lse[head0 + gr + 8 * r] = lt[r] > 0.f ? (m_r[r] + log2f(lt[r])) * kLn2 : -INFINITY;
      }
    }
    if (!ok) *abort_flag = 1;
    n_base += total;
    __syncthreads();                 // the next group rebuilds the bitmaps
    if (*abort_flag) break;
  }
  if (*abort_flag && lane == 0) set_flag(p.flags, MSA_FLAG_TIMEOUT);
  if (warp == 0 && lane == 0) {
    // no copy of this CTA may still be in flight when it exits
    const int first = n_issued > kUnStages ? n_issued - kUnStages : 0;
    for (int k = first; k < n_issued; ++k)
      if (!mbar_wait(smem_addr(&full[k % kUnStages]), static_cast<uint32_t>((k / kUnStages) & 1))) break;
  }
}

// ---------------------------------------------------------------------------
// bf16 K/V on the fifth-generation tensor cores. The 16-head tile is below
// tcgen05's minimum M, so both products run transposed:
//   S^T = K Q^T   (M = 128 tokens, N = 16 heads, K = 128 dims)
//   O^T = V^T P^T (M = 128 dims,   N = 16 heads, K = 128 tokens)
// A is the TMA-loaded, 128-byte-swizzled K tile (K-major) or V tile (read
// MN-major); B is the row's query or the block's probabilities, staged in
// shared memory in the same swizzled K-major form. S (double-buffered) and O
// accumulate in TMEM. One thread of the MMA warp issues the MMAs; its commits
// release the K/V stage and the P buffer. The four softmax warps own one token
// each of S (TMEM lane = token) and one head dim each of O (lane = dim).
// Whole rows per CTA; every wait is bounded.

constexpr int kTcWarps = 6;                      // producer, 4 softmax warps, MMA warp
constexpr int kTcMmaWarp = 5;
constexpr uint32_t kTcCols = 64;                 // TMEM columns: S[2] (16 each) + O (16)
constexpr uint32_t kTcO = 32;                    // O's first column
constexpr int kTcStages = 3;

struct TcLayout {
  uint32_t stages, q, p, red, vote, lsum, bars, tslot, total;
};
__host__ __device__ constexpr TcLayout tc_layout() {
  TcLayout s{};
  s.stages = 0;                                  // kTcStages x 64 KB (K lo, K hi, V lo, V hi)
  s.q = s.stages + kTcStages * kTileBytes;       // 2 x 4 KB: query of the row, 16 heads x 128 dims
  s.p = s.q + 2 * 4096;                          // 2 x 4 KB: P of the block, 16 heads x 128 tokens
  s.red = s.p + 2 * 4096;                        // [2][4 warps][16] block maxima
  s.vote = s.red + 2 * 4 * 16 * 4;               // [2][4] raise votes
  s.lsum = s.vote + 2 * 4 * 4;                   // [4 warps][16] row sums
  s.bars = s.lsum + 4 * 16 * 4;                  // 20 mbarriers
  s.tslot = s.bars + 20 * 8;                     // TMEM base address
  s.total = s.tslot + 16;
  return s;
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand (the layout
// the TMA boxes have: 16-byte chunk c of row r at ((c ^ (r & 7)) << 4), rows
// 128 B apart, 8-row groups 1024 B apart): start address, leading and stride
// byte offsets (16-byte units), descriptor version 1, swizzle mode 2.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A/B
// major-ness (0: K-major, 1: MN-major), N / 8, M / 16.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1 : 0) : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                 "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__global__ void __launch_bounds__(32 * kTcWarps, 1)
    sparse_gqa_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr TcLayout Ly = tc_layout();
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base_addr = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_addr - raw);
  const uint32_t bars = base_addr + Ly.bars;
  // mbarriers: full[3], empty[3], s_full[2], s_free[2], p_full[2], p_free[2], q_full[2], o_full, o_free, done
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (3 + s); };
  auto s_full = [&](int b) { return bars + 8u * (6 + b); };
  auto s_free = [&](int b) { return bars + 8u * (8 + b); };
  auto p_full = [&](int b) { return bars + 8u * (10 + b); };
  auto p_free = [&](int b) { return bars + 8u * (12 + b); };
  auto q_full = [&](int b) { return bars + 8u * (14 + b); };
  const uint32_t o_full = bars + 8u * 16, o_free = bars + 8u * 17, done_bar = bars + 8u * 18;
  const uint32_t gbar = bars + 8u * 19;      // softmax-warp group sync (bounded, unlike bar.sync)
  float* red = reinterpret_cast<float*>(sm + Ly.red);
  volatile int* vote = reinterpret_cast<volatile int*>(sm + Ly.vote);
  float* lsum = reinterpret_cast<float*>(sm + Ly.lsum);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);               // a commit after the block's P.V
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_free(b), kCWarps);
      mbar_init(p_full(b), kCWarps);
      mbar_init(p_free(b), 1);
      mbar_init(q_full(b), kCWarps);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, kCWarps);
    mbar_init(done_bar, 1);
    mbar_init(gbar, kCWarps);
    fence_mbar_init();
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  if (warp == kTcMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(base_addr + Ly.tslot), "r"(kTcCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + Ly.tslot);
  griddep_wait();

  const int C = gridDim.x;
  const int64_t rows_all = p.W / p.K;
  const int64_t x0 = rows_all * blockIdx.x / C * p.K;
  const int64_t x1 = rows_all * (blockIdx.x + 1) / C * p.K;
  const int64_t r0 = x0 / p.K;

  if (x0 < x1 && p.scores != nullptr) {
    // Stage 2 inside this launch (as in the mma.sync kernel); the survivors go
    // to the third stage, which no copy has been issued to yet.
    uint64_t* surv = reinterpret_cast<uint64_t*>(sm + Ly.stages + 2 * kTileBytes) + warp * (kWarpSurvCap + 8);
    int* chosen = reinterpret_cast<int*>(surv + kWarpSurvCap);
    for (int64_t r = r0 + warp; r * p.K < x1; r += kTcWarps) {
      const RowPos rp = row_pos(p, r);
      const int64_t row_off = (static_cast<int64_t>(rp.b) * p.Q + rp.j) * p.G + rp.g;
      int32_t* out = p.sel_out + row_off * p.K;
      const int L = p.seq_lens[rp.b];
      if (L < p.Q || L > p.NB * kBlock || L < 1) {
        for (int e = lane; e < p.K; e += 32) out[e] = -1;
        continue;
      }
      warp_select_row(p.scores + row_off * p.NB, (L - p.Q + rp.j) / kBlock, p.K, out, surv, chosen, lane);
    }
    __syncthreads();
  }

  bool ok = true;
  if (x0 < x1 && warp == 0) {
    // ------------------------------------------------------------ producer --
    ItemInfo cur = load_item(p, x0 + lane, x1, true);
    int64_t i = 0;
    int s = 0;
    uint32_t phase = 0;
    for (int64_t base = x0; base < x1 && ok; base += 32) {
      const ItemInfo nxt = load_item(p, base + 32 + lane, x1, true);
      const int n = static_cast<int>(x1 - base < 32 ? x1 - base : 32);
      for (int k = 0; k < n; ++k) {
        if (!__shfl_sync(kAll, cur.valid, k)) continue;
        const int page = __shfl_sync(kAll, cur.page, k);
        const int g = __shfl_sync(kAll, cur.g, k);
        if (lane == 0) {
          if (!mbar_wait(empty(s), phase ^ 1u)) {
            set_flag(p.flags, MSA_FLAG_TIMEOUT);
            ok = false;
          } else {
            const uint32_t fb = full(s);
            const uint32_t dst = base_addr + Ly.stages + s * kTileBytes;
            const int y = static_cast<int>((static_cast<int64_t>(page) * p.G + g) * kBlock);
            mbar_arrive_expect_tx(fb, kTileBytes);
            tma_load_2d(dst, &tk, 0, y, fb);
            tma_load_2d(dst + kBoxBytes, &tk, 64, y, fb);
            tma_load_2d(dst + 2 * kBoxBytes, &tv, 0, y, fb);
            tma_load_2d(dst + 3 * kBoxBytes, &tv, 64, y, fb);
          }
        }
        ok = __shfl_sync(kAll, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++i;
        if (++s == kTcStages) { s = 0; phase ^= 1u; }
      }
      cur = nxt;
    }
    if (lane == 0) {          // the last copies land before the CTA's teardown
      const int64_t first = i > kTcStages ? i - kTcStages : 0;
      for (int64_t k = first; k < i; ++k)
        if (!mbar_wait(full(static_cast<int>(k % kTcStages)), static_cast<uint32_t>((k / kTcStages) & 1))) break;
    }
  } else if (x0 < x1 && warp == kTcMmaWarp) {
    // ----------------------------------------------------------- MMA warp --
    constexpr uint32_t id_qk = tc_idesc_bf16(128, 16, 0, 0);
    constexpr uint32_t id_pv = tc_idesc_bf16(128, 16, 1, 0);
    const bool leader = lane == 0;
    ItemInfo cur = load_item(p, x0 + lane, x1, false);
    ItemInfo nxt = load_item(p, x0 + 32 + lane, x1, false);
    int64_t base = x0;
    int kx = 0;
    int64_t n = 0;                 // valid items so far
    int64_t rv = 0;                // rows with a valid item so far
    int64_t cur_row = -1;
    bool row_first = true;
    bool pend = false, pend_first = false;
    int64_t pend_n = 0, pend_rv = 0;
    auto issue_pv = [&](int64_t m, bool first, bool last, int64_t mrv) -> bool {
      if (first && mrv >= 1 && !mbar_wait(o_free, static_cast<uint32_t>((mrv - 1) & 1))) return false;
      if (!mbar_wait(p_full(static_cast<int>(m & 1)), static_cast<uint32_t>((m >> 1) & 1))) return false;
      tc_fence_after();
      if (leader) {
        const uint32_t vt = base_addr + Ly.stages + static_cast<uint32_t>(m % kTcStages) * kTileBytes + 2 * kBoxBytes;
        const uint32_t pt = base_addr + Ly.p + static_cast<uint32_t>(m & 1) * 4096u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tmem + kTcO, tc_desc(vt + kk * 2048u, kBoxBytes, 1024), tc_desc(pt + (kk >> 2) * 2048u + (kk & 3) * 32u, 16, 1024),
                 id_pv, !(first && kk == 0));
        tc_commit(empty(static_cast<int>(m % kTcStages)));
        tc_commit(p_free(static_cast<int>(m & 1)));
        if (last) tc_commit(o_full);
      }
      __syncwarp();
      return true;
    };
    while (ok && base + kx < x1) {
      const int64_t x = base + kx;
      const int valid = __shfl_sync(kAll, cur.valid, kx);
      if (++kx == 32) {
        kx = 0;
        base += 32;
        cur = nxt;
        nxt = load_item(p, base + 32 + lane, x1, false);
      }
      const int64_t row = x / p.K;
      if (row != cur_row) {
        if (pend) { ok = issue_pv(pend_n, pend_first, true, pend_rv); pend = false; if (!ok) break; }
        cur_row = row;
        row_first = true;
      }
      if (!valid) continue;
      const int64_t krow = row - r0;
      const int s = static_cast<int>(n % kTcStages);
      if (!mbar_wait(full(s), static_cast<uint32_t>((n / kTcStages) & 1))) { ok = false; break; }
      if (row_first && !mbar_wait(q_full(static_cast<int>(krow & 1)), static_cast<uint32_t>((krow >> 1) & 1))) { ok = false; break; }
      if (n >= 2 && !mbar_wait(s_free(static_cast<int>(n & 1)), static_cast<uint32_t>(((n - 2) >> 1) & 1))) { ok = false; break; }
      tc_fence_after();
      if (leader) {
        const uint32_t kt = base_addr + Ly.stages + static_cast<uint32_t>(s) * kTileBytes;
        const uint32_t qt = base_addr + Ly.q + static_cast<uint32_t>(krow & 1) * 4096u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma(tmem + static_cast<uint32_t>(n & 1) * 16u,
                 tc_desc(kt + (kk >> 2) * kBoxBytes + (kk & 3) * 32u, 16, 1024),
                 tc_desc(qt + (kk >> 2) * 2048u + (kk & 3) * 32u, 16, 1024), id_qk, kk > 0);
        tc_commit(s_full(static_cast<int>(n & 1)));
      }
      __syncwarp();
      if (pend) { ok = issue_pv(pend_n, pend_first, false, pend_rv); if (!ok) break; }
      if (row_first) ++rv;
      pend = true; pend_n = n; pend_first = row_first; pend_rv = rv - 1;
      row_first = false;
      ++n;
    }
    if (ok && pend) ok = issue_pv(pend_n, pend_first, true, pend_rv);
    if (leader) {             // every MMA has finished before TMEM is freed
      tc_commit(done_bar);
      mbar_wait(done_bar, 0);
    }
    __syncwarp();
  } else if (x0 < x1) {
    // ------------------------------------------------------- softmax warps --
    const int sw = warp - 1;                 // 0 .. 3
    const int ct = threadIdx.x - 32;         // 0 .. 127
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int t = 32 * (warp & 3) + lane;    // token of S / dim of O this thread owns
    const float mul = p.scale_log2;
    float m_ref[16], l_part[16];
    int64_t seg_row = -1;
    int seg_b = 0, seg_g = 0, seg_j = 0, seg_p = 0, seg_ell = 0;
    bool seg_valid = false;
    int64_t n = 0, rv = 0;
    uint32_t gph = 0;
    auto gsync = [&]() -> bool { return group_sync(gbar, gph, lane); };

    auto begin_row = [&](int64_t r) {
      const RowPos rp = row_pos(p, r);
      seg_row = r;
      seg_b = rp.b; seg_g = rp.g; seg_j = rp.j;
      seg_p = p.seq_lens[rp.b] - p.Q + rp.j;
      seg_ell = seg_p / kBlock;
      seg_valid = false;
#pragma unroll
      for (int h = 0; h < 16; ++h) { m_ref[h] = -INFINITY; l_part[h] = 0.f; }
      // the row's query, 16 heads x 128 dims, as the swizzled K-major B operand
      const int64_t krow = r - r0;
      const uint16_t* qh = p.q + ((static_cast<int64_t>(rp.b) * p.Q + rp.j) * p.H + static_cast<int64_t>(rp.g) * kGroup) * kDim;
      const uint32_t qt = base_addr + Ly.q + static_cast<uint32_t>(krow & 1) * 4096u;
      for (int i = ct; i < 256; i += 128) {
        const int h = i >> 4, c = i & 15;
        st_shared_v4(qt + (c >> 3) * 2048u + h * 128u + ((((c & 7) ^ (h & 7))) << 4),
                     reinterpret_cast<const uint4*>(qh)[h * 16 + c]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full(static_cast<int>(krow & 1)));
    };
    auto end_row = [&]() -> bool {
      const int64_t head0 = (static_cast<int64_t>(seg_b) * p.Q + seg_j) * p.H + static_cast<int64_t>(seg_g) * kGroup;
      float Lt[16];
      uint32_t o[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) { Lt[h] = 0.f; o[h] = 0u; }
      if (seg_valid) {
        if (!mbar_wait(o_full, static_cast<uint32_t>((rv - 1) & 1))) return false;
        tc_fence_after();
        tc_ld16(tmem + kTcO + lane_base, o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          float v = l_part[h];
#pragma unroll
          for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(kAll, v, s);
          if (lane == 0) lsum[sw * 16 + h] = v;
        }
        if (!gsync()) return false;
#pragma unroll
        for (int h = 0; h < 16; ++h) Lt[h] = lsum[h] + lsum[16 + h] + lsum[32 + h] + lsum[48 + h];
        if (!gsync()) return false;   // lsum is rewritten at the next row end
      }
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float ll = seg_valid ? Lt[h] : 0.f;
        const float v = ll > 0.f ? __uint_as_float(o[h]) / ll : 0.f;
        p.out[(head0 + h) * kDim + t] = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFF);
        if (p.lse != nullptr && ct == h) p.lse[head0 + h] = ll > 0.f ? (m_ref[h] + log2f(ll)) * kLn2 : -INFINITY;
      }
      return true;
    };

    ItemInfo cur = load_item(p, x0 + lane, x1, false);
    ItemInfo nxt = load_item(p, x0 + 32 + lane, x1, false);
    int64_t base = x0;
    int kx = 0;
    bool row_first = true;
    while (ok && base + kx < x1) {
      const int64_t x = base + kx;
      const int valid = __shfl_sync(kAll, cur.valid, kx);
      const int it_blk = __shfl_sync(kAll, cur.blk, kx);
      if (++kx == 32) {
        kx = 0;
        base += 32;
        cur = nxt;
        nxt = load_item(p, base + 32 + lane, x1, false);
      }
      const int64_t row = x / p.K;
      if (row != seg_row) {
        if (seg_row >= 0 && !end_row()) { ok = false; break; }
        begin_row(row);
        row_first = true;
      }
      if (!valid) continue;
      if (!seg_valid) { seg_valid = true; ++rv; }
      const int b2 = static_cast<int>(n & 1);
      // S of this block: 16 heads of token t
      if (!mbar_wait(s_full(b2), static_cast<uint32_t>((n >> 1) & 1))) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[16];
      tc_ld16(tmem + static_cast<uint32_t>(b2) * 16u + lane_base, sr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(b2));
      const bool masked = it_blk == seg_ell && it_blk * kBlock + t > seg_p;
      float xs[16];
      bool raise = false;
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        xs[h] = masked ? -INFINITY : __uint_as_float(sr[h]) * mul;
        raise = raise || xs[h] > m_ref[h] + kRescaleSlack;
      }
      const uint32_t wv = __ballot_sync(kAll, raise);
      if (lane == 0) vote[b2 * 4 + sw] = wv != 0u;
      if (!gsync()) { ok = false; break; }
      if (vote[b2 * 4] | vote[b2 * 4 + 1] | vote[b2 * 4 + 2] | vote[b2 * 4 + 3]) {
        // exact block maxima per head, then a raised reference where they
        // exceed it by more than the slack (uniform over the CTA)
        float bm[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          float v = xs[h];
#pragma unroll
          for (int s = 16; s > 0; s >>= 1) v = fmaxf(v, __shfl_xor_sync(kAll, v, s));
          bm[h] = v;
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < 16; ++h) red[(b2 * 4 + sw) * 16 + h] = bm[h];
        }
        if (!gsync()) { ok = false; break; }
        float alpha[16];
        bool any_alpha = false;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float* rh = red + b2 * 64 + h;
          const float M = fmaxf(fmaxf(rh[0], rh[16]), fmaxf(rh[32], rh[48]));
          const float mn = M > m_ref[h] + kRescaleSlack ? M : m_ref[h];
          alpha[h] = m_ref[h] == -INFINITY ? 0.f : ex2_approx(m_ref[h] - mn);
          any_alpha = any_alpha || mn != m_ref[h];
          m_ref[h] = mn;
          l_part[h] *= alpha[h];
        }
        if (any_alpha && !row_first) {
          // O *= alpha once the previous block's P.V has landed
          if (!mbar_wait(p_free(static_cast<int>((n - 1) & 1)), static_cast<uint32_t>(((n - 1) >> 1) & 1))) { ok = false; break; }
          tc_fence_after();
          uint32_t o[16];
          tc_ld16(tmem + kTcO + lane_base, o);
#pragma unroll
          for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
          tc_st16(tmem + kTcO + lane_base, o);
          tc_fence_before();
        }
      }
      // P of this block into the free P buffer (the P.V two blocks back has read it)
      if (n >= 2 && !mbar_wait(p_free(b2), static_cast<uint32_t>(((n - 2) >> 1) & 1))) { ok = false; break; }
      const uint32_t pt = base_addr + Ly.p + static_cast<uint32_t>(b2) * 4096u + static_cast<uint32_t>(t >> 6) * 2048u;
      const int chunk = (t & 63) >> 3;
      const uint32_t within = static_cast<uint32_t>(t & 7) * 2u;
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float pv = ex2_approx(xs[h] - m_ref[h]);
        l_part[h] += pv;
        st_shared_u16(pt + h * 128u + ((chunk ^ (h & 7)) << 4) + within,
                      static_cast<uint16_t>(pack_bf16x2(pv, 0.f) & 0xFFFF));
      }
      if (masked) {
        // a never-written slot may hold NaN: zero this token's V row, since
        // 0 x NaN would reach O through the product
        const uint32_t vrow = base_addr + Ly.stages + static_cast<uint32_t>(n % kTcStages) * kTileBytes +
                              2 * kBoxBytes + static_cast<uint32_t>(t) * 128u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          st_shared_zero16(vrow + 16u * i);
          st_shared_zero16(vrow + kBoxBytes + 16u * i);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(b2));
      row_first = false;
      ++n;
    }
    if (ok && seg_row >= 0) ok = end_row();
  }
  if (!ok && lane == 0) set_flag(p.flags, MSA_FLAG_TIMEOUT);

  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcCols) : "memory");
  }
}

// ---------------------------------------------------------------------------
// The union form on the fifth-generation tensor cores. With several query
// positions per request the 16 heads of the 8 positions of a (request, KV
// head) group make an M = 128 tile, tcgen05's native shape: S = Q K^T
// (M = 128 query rows, N = 128 tokens, K = 128 dims) and O += P V (N = 128
// dims, K = 128 tokens), one pair of MMAs per union block for every position
// at once. Q and P are the A operands, held in tensor memory (bf16 pairs per
// 32-bit column); K and V are the B operands, read from the TMA-loaded
// 128-byte-swizzled stage (K K-major, V MN-major); S (two buffers, P written
// over the buffer's first 64 columns) and O accumulate in tensor memory.
// Roles: a producer warp (copies, L2 prefetch), an MMA warp (one thread issues,
// commits release the stage and the S/P buffer), and four softmax warps whose
// thread r owns query row r (position r / 16, head r % 16): its 128 logits of
// a block sit in its registers, so the online softmax needs no exchange. A
// position that did not select a block gets P = 0 for it. The output
// accumulator is rescaled in tensor memory only when a row's maximum rises by
// more than 2^8. V rows past the last cached token are zeroed in the stage
// before P V (their probability is 0, but they may hold NaN patterns). One
// CTA per group; every wait is bounded.

constexpr int kTuWarps = 6;                      // producer, MMA warp, 4 softmax warps
constexpr int kTuMmaWarp = 1;
constexpr int kTuStages = 3;
constexpr uint32_t kTuCols = 512;                // TMEM: Q (64) | S0 (128) | S1 (128) | O (128)
constexpr uint32_t kTuQ = 0, kTuS = 64, kTuO = 320;

struct TuLayout {
  uint32_t stages, surv, bits, ubits, prefix, ulist, umask, misc, bars, total;
};
__host__ __device__ inline TuLayout tu_layout(int nw) {
  TuLayout s{};
  s.stages = 0;
  s.surv = kTuStages * kTileBytes;                                // fused selection: each warp's survivors
  s.bits = s.surv + kTuWarps * (kWarpSurvCap + 8) * 8;            // [8][nw] selected blocks per position
  s.ubits = s.bits + kUnWarps * nw * 4;                           // [nw] union
  s.prefix = s.ubits + nw * 4;                                    // [nw] union blocks in the words before
  s.ulist = s.prefix + nw * 4;                                    // [128] union blocks, ascending
  s.umask = s.ulist + kUnWarps * 16 * 4;                          // [128] positions that selected each
  s.misc = s.umask + kUnWarps * 16;                               // group total, abort, TMEM base
  s.bars = (s.misc + 16 + 7) & ~7u;                               // 16 mbarriers
  s.total = s.bars + 16 * 8;
  return s;
}

__device__ __forceinline__ void tc_mma_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
               ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc ? 1 : 0) : "memory");
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
                 "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                 "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
               "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                 "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
                 "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
                 "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}

__global__ void __launch_bounds__(32 * kTuWarps, 1)
    sparse_gqa_union_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                               GqaParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base_addr = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base_addr - raw);
  const int nw = (p.NB + 31) >> 5;
  const TuLayout Ly = tu_layout(nw);
  uint32_t* bits = reinterpret_cast<uint32_t*>(sm + Ly.bits);
  uint32_t* ubits = reinterpret_cast<uint32_t*>(sm + Ly.ubits);
  int* prefix = reinterpret_cast<int*>(sm + Ly.prefix);
  int* ulist = reinterpret_cast<int*>(sm + Ly.ulist);
  uint8_t* umask = sm + Ly.umask;
  volatile int* group_total = reinterpret_cast<volatile int*>(sm + Ly.misc);
  volatile int* abort_flag = group_total + 1;
  const uint32_t tslot = base_addr + Ly.misc + 8;
  const uint32_t bars = base_addr + Ly.bars;
  // mbarriers: full[3], empty[3], s_full[2], p_full[2], sbuf_free[2], q_full, o_full, o_free, done
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (3 + s); };
  auto s_full = [&](int b) { return bars + 8u * (6 + b); };
  auto p_full = [&](int b) { return bars + 8u * (8 + b); };
  auto sbuf_free = [&](int b) { return bars + 8u * (10 + b); };
  const uint32_t q_full = bars + 8u * 12, o_full = bars + 8u * 13, o_free = bars + 8u * 14, done_bar = bars + 8u * 15;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTuStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);                   // a commit after the block's P V
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(p_full(b), 4);                  // the softmax warps
      mbar_init(sbuf_free(b), 1);               // a commit after the P V that read the buffer
    }
    mbar_init(q_full, 4);
    mbar_init(o_full, 1);
    mbar_init(o_free, 4);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  if (warp == kTuMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tslot), "r"(kTuCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + Ly.misc + 8);
  griddep_wait();

  const int groups = p.B * p.G;
  int n_base = 0;         // union index of the group's first block, counted over the CTA's groups
  int gq = 0;             // groups with at least one block this CTA has done (they use the Q / O barriers)
  int n_issued = 0;       // producer: copies issued
  bool ok = true;

  for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
    const int b = grp / p.G, g = grp - b * p.G;
    const int L = p.seq_lens[b];
    const bool len_ok = L >= p.Q && L >= 1 && L <= p.NB * kBlock;
    // 1. (fused) selection of the group's rows; bitmaps cleared
    for (int i = threadIdx.x; i < kUnWarps * nw; i += blockDim.x) bits[i] = 0u;
    if (p.scores != nullptr) {
      uint64_t* surv = reinterpret_cast<uint64_t*>(sm + Ly.surv) + warp * (kWarpSurvCap + 8);
      for (int j = warp; j < p.Q; j += kTuWarps) {
        const int64_t row_off = (static_cast<int64_t>(b) * p.Q + j) * p.G + g;
        int32_t* out = p.sel_out + row_off * p.K;
        if (!len_ok) {
          for (int e = lane; e < p.K; e += 32) out[e] = -1;
        } else {
          warp_select_row(p.scores + row_off * p.NB, (L - p.Q + j) / kBlock, p.K, out, surv,
                          reinterpret_cast<int*>(surv + kWarpSurvCap), lane);
        }
      }
    }
    __syncthreads();
    // 2. each position's valid selected blocks into its bitmap
    for (int j = warp; j < p.Q; j += kTuWarps) {
      if (!len_ok) {
        if (j == 0 && lane == 0) set_flag(p.flags, MSA_FLAG_BAD_SEQLEN);
        continue;
      }
      const int ell = (L - p.Q + j) / kBlock;
      const int32_t* sel = p.selected + ((static_cast<int64_t>(b) * p.Q + j) * p.G + g) * p.K;
      for (int e = lane; e < p.K; e += 32) {
        const int blk = sel[e];
        if (blk < 0) continue;
        if (blk > ell) { set_flag(p.flags, MSA_FLAG_BAD_BLOCK); continue; }
        const int page = p.block_table[static_cast<int64_t>(b) * p.NB + blk];
        if (page < 0 || page >= p.P) { set_flag(p.flags, MSA_FLAG_BAD_PAGE); continue; }
        atomicOr(&bits[j * nw + (blk >> 5)], 1u << (blk & 31));
      }
    }
    __syncthreads();
    // 3. union, its running count per word, the ascending list and each block's positions
    if (warp == 0) {
      int run = 0;
      for (int w0 = 0; w0 < nw; w0 += 32) {
        const int w = w0 + lane;
        uint32_t u = 0u;
        if (w < nw)
          for (int q = 0; q < p.Q; ++q) u |= bits[q * nw + w];
        const int cnt = __popc(u);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(kAll, incl, o);
          if (lane >= o) incl += t;
        }
        if (w < nw) {
          ubits[w] = u;
          prefix[w] = run + incl - cnt;
          int at = run + incl - cnt;
          for (uint32_t v = u; v != 0u; v &= v - 1u) {
            const int bit = __ffs(v) - 1;
            uint32_t m = 0u;
            for (int q = 0; q < p.Q; ++q) m |= ((bits[q * nw + w] >> bit) & 1u) << q;
            umask[at] = static_cast<uint8_t>(m);
            ulist[at++] = (w << 5) + bit;
          }
        }
        run += __shfl_sync(kAll, incl, 31);
      }
      if (lane == 0) *group_total = run;
    }
    __syncthreads();
    const int total = *group_total;
    const int last_blk = (L - 1) / kBlock;

    if (warp == 0) {
      // ------------------------------------------------------------ producer --
      auto l2_prefetch = [&](int i) {
        if (i < total) {
          const int page = p.block_table[static_cast<int64_t>(b) * p.NB + ulist[i]];
          const int64_t off = (static_cast<int64_t>(page) * p.G + g) * (kBlock * kDim * 2);
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.k4 + off), "r"(kBlock * kDim * 2) : "memory");
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.v4 + off), "r"(kBlock * kDim * 2) : "memory");
        }
      };
      if (lane == 0)
        for (int i = kTuStages; i < kTuStages + kUnAhead - 1; ++i) l2_prefetch(i);
      for (int i = 0; i < total && ok; ++i) {
        if (lane == 0) {
          const int n = n_base + i;
          const int s = n % kTuStages;
          if (!mbar_wait(empty(s), (static_cast<uint32_t>(n / kTuStages) & 1u) ^ 1u)) {
            set_flag(p.flags, MSA_FLAG_TIMEOUT);
            ok = false;
          } else {
            const int page = p.block_table[static_cast<int64_t>(b) * p.NB + ulist[i]];
            const int y = static_cast<int>((static_cast<int64_t>(page) * p.G + g) * kBlock);
            const uint32_t dst = base_addr + Ly.stages + s * kTileBytes;
            mbar_arrive_expect_tx(full(s), kTileBytes);
            tma_load_2d(dst, &tk, 0, y, full(s));
            tma_load_2d(dst + kBoxBytes, &tk, 64, y, full(s));
            tma_load_2d(dst + 2 * kBoxBytes, &tv, 0, y, full(s));
            tma_load_2d(dst + 3 * kBoxBytes, &tv, 64, y, full(s));
            l2_prefetch(i + kTuStages + kUnAhead - 1);
            n_issued = n + 1;
          }
        }
        ok = __shfl_sync(kAll, ok ? 1 : 0, 0) != 0;
      }
      n_issued = __shfl_sync(kAll, n_issued, 0);
    } else if (warp == kTuMmaWarp) {
      // ----------------------------------------------------------- MMA warp --
      constexpr uint32_t id_s = tc_idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t id_o = tc_idesc_bf16(128, 128, 0, 1);
      const bool leader = lane == 0;
      auto issue_pv = [&](int i) -> bool {      // O += P V of union block i
        const int n = n_base + i, bb = n & 1, s = n % kTuStages;
        if (!mbar_wait(p_full(bb), static_cast<uint32_t>(n >> 1) & 1u)) return false;
        if (i == 0 && gq > 0 && !mbar_wait(o_free, static_cast<uint32_t>(gq - 1) & 1u)) return false;
        tc_fence_after();
        if (leader) {
          const uint32_t vt = base_addr + Ly.stages + static_cast<uint32_t>(s) * kTileBytes + 2 * kBoxBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_ta(tmem + kTuO, tmem + kTuS + 128u * bb + 8u * kk, tc_desc(vt + kk * 2048u, kBoxBytes, 1024), id_o,
                      !(i == 0 && kk == 0));
          tc_commit(empty(s));
          tc_commit(sbuf_free(bb));
          if (i == total - 1) tc_commit(o_full);
        }
        __syncwarp();
        return true;
      };
      if (total > 0 && !mbar_wait(q_full, static_cast<uint32_t>(gq) & 1u)) ok = false;
      for (int i = 0; i < total && ok; ++i) {
        const int n = n_base + i, bb = n & 1, s = n % kTuStages;
        if (!mbar_wait(full(s), static_cast<uint32_t>(n / kTuStages) & 1u)) { ok = false; break; }
        if (n >= 2 && !mbar_wait(sbuf_free(bb), static_cast<uint32_t>((n - 2) >> 1) & 1u)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
          const uint32_t kt = base_addr + Ly.stages + static_cast<uint32_t>(s) * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_ta(tmem + kTuS + 128u * bb, tmem + kTuQ + 8u * kk,
                      tc_desc(kt + (kk >> 2) * kBoxBytes + (kk & 3) * 32u, 16, 1024), id_s, kk > 0);
          tc_commit(s_full(bb));
        }
        __syncwarp();
        if (i > 0 && !issue_pv(i - 1)) { ok = false; break; }
      }
      if (ok && total > 0 && !issue_pv(total - 1)) ok = false;
    } else {
      // ------------------------------------------------------- softmax warps --
      const int r = 32 * (warp & 3) + lane;    // query row = TMEM lane
      const int j = r >> 4, h = r & 15;
      const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
      const bool row_live = len_ok && j < p.Q;
      const int pj = L - p.Q + j;
      const int ell = pj / kBlock;
      const float mul = p.scale_log2;
      const uint32_t wmask = 3u << (2 * (warp & 3));   // the two positions of this warp's rows
      float m_ref = -INFINITY, l_sum = 0.f;
      const int64_t head = (static_cast<int64_t>(b) * p.Q + (j < p.Q ? j : 0)) * p.H + static_cast<int64_t>(g) * kGroup + h;
      if (total > 0) {
        // the group's queries into tensor memory: row r = (position j, head h), bf16 pairs per column
        const uint4* qr = reinterpret_cast<const uint4*>(p.q + head * kDim);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t qv[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 v = row_live ? qr[half * 8 + k] : make_uint4(0u, 0u, 0u, 0u);
            qv[4 * k] = v.x; qv[4 * k + 1] = v.y; qv[4 * k + 2] = v.z; qv[4 * k + 3] = v.w;
          }
          tc_st32(tmem + lane_base + kTuQ + 32u * half, qv);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
      }
      for (int i = 0; i < total && ok; ++i) {
        const int n = n_base + i, bb = n & 1, s = n % kTuStages;
        const int blk = ulist[i];
        const uint32_t um = umask[i];
        const uint32_t sbuf = tmem + lane_base + kTuS + 128u * bb;
        if (!mbar_wait(s_full(bb), static_cast<uint32_t>(n >> 1) & 1u)) { ok = false; break; }
        tc_fence_after();
        if (um & wmask) {
          const bool mine = ((um >> j) & 1u) != 0 && row_live;
          uint32_t sr[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tc_ld32(sbuf + 32u * q, sr[q]);
          // logits (log2 units), causal limit of this position, row maximum
          float mx = -INFINITY;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int t = blk * kBlock + 32 * q + k;
              float x = __uint_as_float(sr[q][k]) * mul;
              if (!mine || (blk == ell && t > pj)) x = -INFINITY;
              sr[q][k] = __float_as_uint(x);
              mx = fmaxf(mx, x);
            }
          }
          const bool raise = mx > m_ref + kRescaleSlack;
          const float m_new = raise ? mx : m_ref;
          const float alpha = (raise && m_ref != -INFINITY) ? ex2_approx(m_ref - m_new) : 1.f;
          if (__any_sync(kAll, raise && m_ref != -INFINITY)) {
            // O *= alpha once the previous block's P V has landed
            if (n >= 1 && !mbar_wait(sbuf_free((n - 1) & 1), static_cast<uint32_t>((n - 1) >> 1) & 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t ov[32];
              tc_ld32(tmem + lane_base + kTuO + 32u * q, ov);
#pragma unroll
              for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
              tc_st32(tmem + lane_base + kTuO + 32u * q, ov);
            }
          }
          m_ref = m_new;
          l_sum *= alpha;
          // P = 2^(x - m) in bf16 pairs over the buffer's first 64 columns
          const float neg_ref = m_ref == -INFINITY ? 0.f : -m_ref;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float p0 = ex2_approx(__uint_as_float(sr[q][2 * k]) + neg_ref);
              const float p1 = ex2_approx(__uint_as_float(sr[q][2 * k + 1]) + neg_ref);
              l_sum += p0 + p1;
              pk[k] = pack_bf16x2(p0, p1);
            }
            tc_st16(sbuf + 16u * q, pk);
          }
        } else {
          uint32_t zz[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) zz[k] = 0u;
#pragma unroll
          for (int q = 0; q < 4; ++q) tc_st16(sbuf + 16u * q, zz);
        }
        // V rows past the last cached token: zeros (thread r takes token row r)
        if (blk == last_blk && blk * kBlock + r > L - 1) {
          const uint32_t vrow = base_addr + Ly.stages + static_cast<uint32_t>(s) * kTileBytes + 2 * kBoxBytes +
                                static_cast<uint32_t>(r) * 128u;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            st_shared_zero16(vrow + 16u * k);
            st_shared_zero16(vrow + kBoxBytes + 16u * k);
          }
        }
        fence_proxy_async_smem();
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(bb));
      }
      // the group's output rows
      if (ok && total > 0) {
        if (!mbar_wait(o_full, static_cast<uint32_t>(gq) & 1u)) {
          ok = false;
        } else {
          tc_fence_after();
          const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t ov[32];
            tc_ld32(tmem + lane_base + kTuO + 32u * q, ov);
            if (row_live) {
              uint32_t pk[16];
#pragma unroll
              for (int k = 0; k < 16; ++k)
                pk[k] = pack_bf16x2(__uint_as_float(ov[2 * k]) * inv, __uint_as_float(ov[2 * k + 1]) * inv);
              uint4* dst = reinterpret_cast<uint4*>(p.out + head * kDim + 32 * q);
#pragma unroll
              for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free);
        }
      }
      if (row_live && total == 0) {                // no block: output 0, lse -inf
        uint4* dst = reinterpret_cast<uint4*>(p.out + head * kDim);
        for (int k = 0; k < 16; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (row_live && p.lse != nullptr) p.lse[head] = l_sum > 0.f ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
    }
    if (!ok) *abort_flag = 1;
    n_base += total;
    if (total > 0) ++gq;
    __syncthreads();                 // the next group rebuilds the bitmaps and the queries
    if (*abort_flag) break;
  }
  if (*abort_flag && lane == 0) set_flag(p.flags, MSA_FLAG_TIMEOUT);
  if (warp == 0 && lane == 0) {
    // no copy of this CTA may still be in flight when it exits
    for (int k = n_issued > kTuStages ? n_issued - kTuStages : 0; k < n_issued; ++k)
      if (!mbar_wait(full(k % kTuStages), static_cast<uint32_t>((k / kTuStages) & 1))) break;
  }
  if (warp == kTuMmaWarp && lane == 0) {     // every MMA has finished before TMEM is freed
    tc_commit(done_bar);
    mbar_wait(done_bar, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kTuMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTuCols) : "memory");
  }
}

size_t gqa_workspace_bytes(int B, int Q, int G, int K) {
  const size_t rows = static_cast<size_t>(B) * Q * G;
  return rows * K * kPartialFloats * sizeof(float) + rows * sizeof(unsigned long long);
}

// cuTensorMapEncodeTiled from the driver, looked up through the runtime so the
// library does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D map over a cache [P*G*BS rows, 128 dims] with 128-row boxes of 128 bytes
// and 128 B swizzle: bf16 (64-dim boxes, two per row) or FP8 codes (one box).
static cudaError_t make_kv_map(CUtensorMap* map, const void* base, int64_t rows, bool fp8) {
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim) * (fp8 ? 1 : 2)};
  const cuuint32_t box[2] = {fp8 ? 128u : 64u, static_cast<cuuint32_t>(kBlock)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The tcgen05 form of the bf16 tile is opt-in: MSA_BF16_ATTENTION=tcgen05 in
// the environment when the call is made (read on every call, so a captured
// graph keeps the kernel chosen at capture). With 16 heads per KV head its
// per-block hand-offs (S in TMEM, a CTA-wide rescale vote, P through shared
// memory) cost more than the register-resident mma.sync tile saves: on the
// 32 x 32K bf16 workload the launch takes 46.7 us against 31.2.
static bool bf16_tcgen05_selected() {
  const char* e = getenv("MSA_BF16_ATTENTION");
  return e != nullptr && strcmp(e, "tcgen05") == 0;
}

// With several query positions and bf16 K/V, the union form (one CTA per
// (request, KV head), each block read once) is used when there are at least
// three groups for every four SMs; with fewer the per-position rows spread
// better over the SMs. MSA_MULTIPOS_ATTENTION=union, =union_mma or =rows in the
// environment (read on every call) forces one form.
// The union form runs on tcgen05 (sparse_gqa_union_tc_kernel);
// MSA_MULTIPOS_ATTENTION=union_mma selects its mma.sync form instead.
static bool multipos_union_tc_selected() {
  const char* e = getenv("MSA_MULTIPOS_ATTENTION");
  return e == nullptr || strcmp(e, "union_mma") != 0;
}

static bool multipos_union_selected(const GqaArgs& a, int sms) {
  if (a.Q < 2 || a.NB > kUnMaxNB) return false;
  const char* e = getenv("MSA_MULTIPOS_ATTENTION");
  if (e != nullptr && (strcmp(e, "union") == 0 || strcmp(e, "union_mma") == 0)) return true;
  if (e != nullptr && strcmp(e, "rows") == 0) return false;
  return 4ll * a.B * a.G >= 3ll * sms;
}

// How many clusters of `cn` NVFP4 CTAs can be resident at once on this device
// (cached per device and size).
static int fp4_max_active_clusters(int cn, size_t smem) {
  static std::atomic<int> cache[64][3];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const int slot = cn == 2 ? 0 : cn == 4 ? 1 : 2;
  if (dev < 64) {
    const int v = cache[dev][slot].load();
    if (v > 0) return v - 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cn * 64));
  cfg.blockDim = dim3(32 * kF4Warps);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cn);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, sparse_gqa_fp4_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;                          // not cached: a later call asks again
  }
  if (dev < 64) cache[dev][slot].store(n + 1);
  return n;
}

// NVFP4 rows are split over the CTAs of a thread-block cluster and merged
// through distributed shared memory when every row's cluster can be resident at
// once: the largest cluster of 8, 4 or 2 CTAs (at most K, so every CTA has a
// slot) that allows it. Otherwise item ranges are balanced over the SMs and
// split rows merge through the workspace. MSA_NVFP4_SPLIT=tickets, =cluster2,
// =cluster4 or =cluster8 in the environment (read on every call) forces a form.
static int fp4_cluster_size(int64_t rows, int K, size_t smem) {
  const char* e = getenv("MSA_NVFP4_SPLIT");
  if (e != nullptr && strcmp(e, "tickets") == 0) return 1;
  if (e != nullptr && strncmp(e, "cluster", 7) == 0) {
    const int forced = atoi(e + 7);
    if (forced == 2 || forced == 4 || forced == 8) return forced <= K ? forced : 1;
  }
  for (int cn = 8; cn >= 2; cn /= 2) {
    if (cn > K) continue;
    if (rows <= fp4_max_active_clusters(cn, smem)) return cn;
  }
  return 1;
}

cudaError_t launch_sparse_gqa(const GqaArgs& a, cudaStream_t stream, DispatchRecord* rec) {
  GqaParams p;
  p.q = a.q;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.selected = a.selected;
  p.scores = a.scores;
  p.sel_out = const_cast<int32_t*>(a.selected);
  p.out = a.out;
  p.lse = a.lse;
  p.ws = a.workspace;
  p.flags = a.flags;
  p.k4 = static_cast<const uint8_t*>(a.k);
  p.v4 = static_cast<const uint8_t*>(a.v);
  p.ks = a.k_scale;
  p.vs = a.v_scale;
  p.k_global = a.k_global;
  p.v_global = a.v_global;
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  p.B = a.B; p.Q = a.Q; p.H = a.H; p.G = a.G; p.NB = a.NB; p.P = a.P; p.K = a.K;
  p.W = static_cast<int64_t>(a.B) * a.G * a.Q * a.K;
  p.cluster_n = 0;
  if (p.W == 0) {
    rec->set("sparse_gqa empty");
    return cudaSuccess;
  }
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  const int64_t cache_rows = static_cast<int64_t>(a.P) * a.G * kBlock;
  cudaError_t err;
  if (!a.nvfp4) {
    if ((err = make_kv_map(&tk, a.k, cache_rows, a.fp8 != 0)) != cudaSuccess) return err;
    if ((err = make_kv_map(&tv, a.v, cache_rows, a.fp8 != 0)) != cudaSuccess) return err;
  }
  // Work split. bf16 and FP8 pages (64 / 32 KB per block) stream best when
  // every CTA owns whole rows: no split-K partials, no merge. NVFP4 pages (18 KB) are latency
  // bound per block, so their item ranges are balanced exactly over all SMs
  // and the CTAs that share a row merge through the workspace.
  const int sms = device_sm_count();
  const int64_t rows = p.W / p.K;
  int C;
  if (!a.nvfp4) {
    p.row_aligned = 1;
    C = static_cast<int>(rows < sms ? rows : sms);
  } else {
    p.row_aligned = 0;
    C = static_cast<int>(p.W < sms ? p.W : sms);
  }
  const size_t smem = (a.fp8 ? gqa_layout<kKvFp8>().total : gqa_layout<kKvBf16>().total) + 1024;
  static std::atomic<uint32_t> epoch{1};
  p.epoch = epoch.fetch_add(1);
  if (p.epoch == 0) p.epoch = epoch.fetch_add(1);    // 0 never tags a ticket
  p.tickets = reinterpret_cast<unsigned long long*>(a.workspace + (p.W / p.K) * p.K * kPartialFloats);
  if (!a.nvfp4 && !a.fp8 && !bf16_tcgen05_selected() && multipos_union_selected(a, sms)) {
    // several positions, bf16 K/V: the union of each group's blocks, one CTA per group
    const int nw = (a.NB + 31) / 32;
    if (multipos_union_tc_selected()) {
      const size_t tsm = tu_layout(nw).total + 1024;
      const int64_t ngroups = static_cast<int64_t>(a.B) * a.G;
      const int TC = static_cast<int>(ngroups < sms ? ngroups : sms);
      err = cudaFuncSetAttribute(sparse_gqa_union_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(tsm));
      if (err != cudaSuccess) return err;
      err = launch_pdl(sparse_gqa_union_tc_kernel, dim3(TC), dim3(32 * kTuWarps), tsm, stream, tk, tv, p);
      rec->set("%ssparse_gqa bf16_tma_tcgen05 union_of_positions grid=%d block=%d smem=%zu stages=%d groups=%lld",
               a.scores != nullptr ? "select+" : "", TC, 32 * kTuWarps, tsm, kTuStages,
               static_cast<long long>(ngroups));
      return err != cudaSuccess ? err : cudaGetLastError();
    }
    const size_t usmem = un_layout(nw).total + 1024;
    const int64_t groups = static_cast<int64_t>(a.B) * a.G;
    const int UC = static_cast<int>(groups < sms ? groups : sms);
    err = cudaFuncSetAttribute(sparse_gqa_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(usmem));
    if (err != cudaSuccess) return err;
    err = launch_pdl(sparse_gqa_union_kernel, dim3(UC), dim3(32 * (1 + kUnWarps)), usmem, stream, tk, tv, p);
    rec->set("%ssparse_gqa bf16_tma_mma union_of_positions grid=%d block=%d smem=%zu stages=%d groups=%lld",
             a.scores != nullptr ? "select+" : "", UC, 32 * (1 + kUnWarps), usmem, kUnStages,
             static_cast<long long>(groups));
    return err != cudaSuccess ? err : cudaGetLastError();
  }
  if (!a.nvfp4 && !a.fp8 && bf16_tcgen05_selected()) {
    // bf16 K/V on the tcgen05 kernel, when selected (whole rows)
    const size_t tsmem = tc_layout().total + 1024;
    err = cudaFuncSetAttribute(sparse_gqa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(tsmem));
    if (err != cudaSuccess) return err;
    err = launch_pdl(sparse_gqa_tc_kernel, dim3(C), dim3(32 * kTcWarps), tsmem, stream, tk, tv, p);
    rec->set("%ssparse_gqa bf16_tma_tcgen05 persistent whole_rows grid=%d block=%d smem=%zu stages=%d items=%lld",
             a.scores != nullptr ? "select+" : "", C, 32 * kTcWarps, tsmem, kTcStages, static_cast<long long>(p.W));
    return err != cudaSuccess ? err : cudaGetLastError();
  }
  if (a.nvfp4) {
    // NVFP4 K/V: eight consumer warps, balanced item ranges
    constexpr size_t wsmem = f4_layout().total + 1024;
    err = cudaFuncSetAttribute(sparse_gqa_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(wsmem));
    if (err != cudaSuccess) return err;
    const int cn = fp4_cluster_size(rows, a.K, wsmem);
    if (cn > 1) {
      p.cluster_n = cn;
      const int64_t grid = rows * cn;
      err = launch_pdl_cluster(sparse_gqa_fp4_kernel, dim3(static_cast<unsigned>(grid)), dim3(32 * kF4Warps), wsmem,
                               stream, cn, p);
      rec->set("%ssparse_gqa nvfp4_regk_f16_mma 8warps cluster_split_dsmem_combine cluster=%d grid=%lld block=%d "
               "smem=%zu stages=%d items=%lld",
               a.scores != nullptr ? "select+" : "", cn, static_cast<long long>(grid), 32 * kF4Warps, wsmem,
               kF4Stages, static_cast<long long>(p.W));
      return err != cudaSuccess ? err : cudaGetLastError();
    }
    err = launch_pdl(sparse_gqa_fp4_kernel, dim3(C), dim3(32 * kF4Warps), wsmem, stream, p);
    rec->set("%ssparse_gqa nvfp4_regk_f16_mma 8warps persistent split_k_fused_combine grid=%d block=%d smem=%zu "
             "stages=%d items=%lld",
             a.scores != nullptr ? "select+" : "", C, 32 * kF4Warps, wsmem, kF4Stages,
             static_cast<long long>(p.W));
    return err != cudaSuccess ? err : cudaGetLastError();
  }
  auto kern = a.fp8 ? sparse_gqa_kernel<kKvFp8> : sparse_gqa_kernel<kKvBf16>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  err = launch_pdl(kern, dim3(C), dim3(32 * (1 + kCWarps)), smem, stream, tk, tv, p);
  rec->set("%ssparse_gqa %s persistent %s grid=%d block=%d smem=%zu stages=%d items=%lld",
           a.scores != nullptr ? "select+" : "",
           a.fp8 ? "fp8_tma_cvt_f16_mma" : "bf16_tma_mma",
           p.row_aligned ? "whole_rows" : "split_k_fused_combine", C, 32 * (1 + kCWarps), smem,
           a.fp8 ? stages_for<kKvFp8>() : stages_for<kKvBf16>(),
           static_cast<long long>(p.W));
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace msa
