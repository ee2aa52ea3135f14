// Cache insertion and quantisation: writes new tokens' K/V (bf16 copy, FP8 E4M3
// with a per-tensor scale, or NVFP4)
// and index keys (fp32 copy or FP8 E4M3 + per-token scale) into the paged
// caches. One warp per (token, head); every step of the quantisers is an IEEE
// round-to-nearest fp32 operation so the bytes are a pure function of the input.
#include <cmath>
#include <cstring>

#include "insert_rows.cuh"

namespace msa {

__global__ void __launch_bounds__(256) kv_insert_kernel(InsertParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = static_cast<int64_t>(p.T) * p.G;
  for (int64_t w = warp; w < total; w += nwarps)
    insert_row(p, static_cast<int>(w / p.G), static_cast<int>(w % p.G), lane);
}

// ------------------------------------------- QK-norm + RoPE + cache insert --
// "MiniMax-M3.1-Flash Day-0 対応", section "最適化と数値" (QKV GEMM + norm + RoPE
// + KV insert fused) and "MiniMax M3 vLLM サポート：…", section "カーネル融合"
// (QKNorm + RoPE + KV insertion in one kernel). kPrologueParts CTAs per token,
// each taking every kPrologueParts-th head row (query heads, key heads, V heads,
// index query heads, index key heads). A CTA computes the token's 64 rotary
// (cos, sin) pairs (angle pos * theta^(-2i/128) with the inverse frequencies
// from the host in double precision, reduced modulo 2 pi in double so large
// positions keep their phase, then an fp32 sincos), while each warp loads all
// of its rows; then per row: RMSNorm (fp32, IEEE sqrt and division), rotation
// of the pairs (i, i + 64) — lane l holds dims 4l..4l+3, its partner lane
// l ^ 16 the other half — rounding to bf16, and the query goes to its output,
// the key (and V, unrotated) through the cache's quantiser. Index rows take the
// same path with their own weights unless the layer reuses another layer's
// selection (null index pointers).
constexpr int kPrologueParts = 4;
constexpr int kPrologueWarps = 8;
constexpr int kPrologueRowsPerWarp = 3;   // ceil(80 rows / (4 parts x 8 warps))

struct PrologueParams {
  InsertParams ins;
  const uint16_t* q;          // bf16 [T, H, D]
  const uint16_t* idx_q;      // bf16 [T, I, D] or null
  uint16_t* q_out;
  uint16_t* idx_q_out;
  const int32_t* positions;   // [T]
  const float* wq;
  const float* wk;
  const float* wiq;
  const float* wik;
  float eps;
  int H, I;
  double inv_freq[kDim / 2];  // theta^(-2i/D)
};

__global__ void __launch_bounds__(32 * kPrologueWarps) qk_norm_rope_insert_kernel(const __grid_constant__ PrologueParams pp) {
  __shared__ float2 cs[kDim / 2];
  griddep_launch_dependents();
  griddep_wait();
  const InsertParams& p = pp.ins;
  const int t = blockIdx.x / kPrologueParts, part = blockIdx.x % kPrologueParts;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool with_idx = pp.idx_q != nullptr;
  const int nq = pp.H, nk = p.G, ni = with_idx ? pp.I : 0;
  const int rows = nq + 2 * nk + 2 * ni;     // q heads, k heads, v heads, index q heads, index k heads

  // this warp's rows, loaded before anything waits on them
  int kind[kPrologueRowsPerWarp], head[kPrologueRowsPerWarp];
  float x[kPrologueRowsPerWarp][4];
#pragma unroll
  for (int j = 0; j < kPrologueRowsPerWarp; ++j) {
    const int r = part + kPrologueParts * (warp + kPrologueWarps * j);
    kind[j] = -1;
    if (r >= rows) continue;
    int k, h;                                  // 0 q, 1 k, 2 v, 3 index q, 4 index k
    if (r < nq) { k = 0; h = r; }
    else if (r < nq + nk) { k = 1; h = r - nq; }
    else if (r < nq + 2 * nk) { k = 2; h = r - nq - nk; }
    else if (r < nq + 2 * nk + ni) { k = 3; h = r - nq - 2 * nk; }
    else { k = 4; h = r - nq - 2 * nk - ni; }
    kind[j] = k;
    head[j] = h;
    const uint16_t* src = k == 0 ? pp.q + (static_cast<int64_t>(t) * nq + h) * kDim
                        : k == 1 ? p.k_new + (static_cast<int64_t>(t) * nk + h) * kDim
                        : k == 2 ? p.v_new + (static_cast<int64_t>(t) * nk + h) * kDim
                        : k == 3 ? pp.idx_q + (static_cast<int64_t>(t) * pp.I + h) * kDim
                                 : static_cast<const uint16_t*>(p.idx_new) + (static_cast<int64_t>(t) * pp.I + h) * kDim;
    load_bf16x4(src + 4 * lane, x[j]);
  }
  if (threadIdx.x < kDim / 2) {
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    const double ang = static_cast<double>(pp.positions[t]) * pp.inv_freq[threadIdx.x];
    const double red = fma(-rint(ang * (1.0 / kTwoPi)), kTwoPi, ang);     // |red| <= pi
    float sn, cn;
    sincosf(static_cast<float>(red), &sn, &cn);
    cs[threadIdx.x] = make_float2(cn, sn);
  }
  __syncthreads();
  const int64_t slot = p.slots[t];
  const float rms_scale = 1.0f / kDim;
#pragma unroll
  for (int j = 0; j < kPrologueRowsPerWarp; ++j) {
    const int k = kind[j], h = head[j];
    if (k < 0) continue;
    if (k != 2) {
      // RMSNorm
      float ss = x[j][0] * x[j][0] + x[j][1] * x[j][1] + x[j][2] * x[j][2] + x[j][3] * x[j][3];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rinv = __fdiv_rn(1.0f, __fsqrt_rn(__fmaf_rn(ss, rms_scale, pp.eps)));
      const float* wv = k == 0 ? pp.wq : k == 1 ? pp.wk : k == 3 ? pp.wiq : pp.wik;
      const float4 wt = *reinterpret_cast<const float4*>(wv + 4 * lane);
      const float y0 = x[j][0] * rinv * wt.x, y1 = x[j][1] * rinv * wt.y;
      const float y2 = x[j][2] * rinv * wt.z, y3 = x[j][3] * rinv * wt.w;
      const float yv[4] = {y0, y1, y2, y3};
      // rotary: lane l < 16 holds y_i (i = 4l + e), lane l + 16 holds y_{i+64};
      // the results are rounded to bf16, the values the caches and outputs hold
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, yv[e], 16);
        const float2 c = cs[(4 * lane + e) & (kDim / 2 - 1)];
        const float z = lane < 16 ? yv[e] * c.x - other * c.y : other * c.y + yv[e] * c.x;
        x[j][e] = bf16_bits_to_f32(static_cast<uint16_t>(pack_bf16x2(z, 0.f) & 0xFFFF));
      }
    }
    if (k == 0 || k == 3) {
      uint16_t* dst = k == 0 ? pp.q_out + (static_cast<int64_t>(t) * nq + h) * kDim
                             : pp.idx_q_out + (static_cast<int64_t>(t) * pp.I + h) * kDim;
      *reinterpret_cast<uint2*>(dst + 4 * lane) = make_uint2(pack_bf16x2(x[j][0], x[j][1]), pack_bf16x2(x[j][2], x[j][3]));
      continue;
    }
    const int64_t row = slot_row(p, slot, h, k == 4 ? pp.I : p.G, lane);
    if (row < 0) continue;
    if (k == 4) store_idx_row(p, row, x[j], lane);
    else store_kv_row(p, k == 2, row, x[j], lane);
  }
}

cudaError_t launch_kv_insert(const InsertArgs& a, cudaStream_t stream, DispatchRecord* rec) {
  const InsertParams p = make_insert_params(a);
  const int64_t warps = static_cast<int64_t>(a.T) * a.G;
  int64_t blocks = (warps + 7) / 8;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const cudaError_t err = launch_pdl(kv_insert_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
  if (err != cudaSuccess) return err;
  rec->set("kv_insert %s%s grid=%lld block=256 tokens=%d", a.kv_nvfp4 ? "nvfp4" : a.kv_fp8 ? "fp8" : "bf16",
           a.idx_new ? (a.idx_fp4 ? "+idx_nvfp4" : a.idx_fp8 ? "+idx_fp8" : "+idx_f32") : "",
           static_cast<long long>(blocks), a.T);
  return cudaGetLastError();
}

cudaError_t launch_qk_norm_rope_insert(const PrologueArgs& a, cudaStream_t stream, DispatchRecord* rec) {
  PrologueParams pp;
  memset(&pp, 0, sizeof(pp));
  pp.ins = make_insert_params(a.ins);
  pp.ins.idx_new_bf16 = 1;
  pp.q = static_cast<const uint16_t*>(a.q);
  pp.idx_q = static_cast<const uint16_t*>(a.idx_q);
  pp.q_out = static_cast<uint16_t*>(a.q_out);
  pp.idx_q_out = static_cast<uint16_t*>(a.idx_q_out);
  pp.positions = a.positions;
  pp.wq = a.wq; pp.wk = a.wk; pp.wiq = a.wiq; pp.wik = a.wik;
  pp.eps = a.eps;
  pp.H = a.H;
  pp.I = a.I;
  for (int i = 0; i < kDim / 2; ++i) pp.inv_freq[i] = pow(static_cast<double>(a.theta), -2.0 * i / kDim);
  const int rows = a.H + 2 * a.ins.G + (a.idx_q ? 2 * a.I : 0);
  if (rows > kPrologueParts * kPrologueWarps * kPrologueRowsPerWarp) return cudaErrorInvalidValue;
  const cudaError_t err = launch_pdl(qk_norm_rope_insert_kernel, dim3(static_cast<unsigned>(a.ins.T) * kPrologueParts),
                                     dim3(32 * kPrologueWarps), 0, stream, pp);
  if (err != cudaSuccess) return err;
  rec->set("qk_norm_rope_insert %s%s grid=%d block=256 heads=%d+%d+%d", a.ins.kv_nvfp4 ? "nvfp4" : a.ins.kv_fp8 ? "fp8" : "bf16",
           a.idx_q ? (a.ins.idx_fp4 ? "+idx_nvfp4" : "+idx_fp8") : "", a.ins.T * kPrologueParts, a.H, a.ins.G,
           a.idx_q ? a.I : 0);
  return cudaGetLastError();
}

}  // namespace msa
