// Cache insertion and quantisation: writes new tokens' K/V (bf16 copy, FP8 E4M3
// with a per-tensor scale, or NVFP4)
// and index keys (fp32 copy or FP8 E4M3 + per-token scale) into the paged
// caches. One warp per (token, head); every step of the quantisers is an IEEE
// round-to-nearest fp32 operation so the bytes are a pure function of the input.
#include "msa_internal.h"

namespace msa {

struct InsertParams {
  const uint16_t* k_new;      // bf16 [T, G, D]
  const uint16_t* v_new;
  const void* idx_new;        // [T, G, D] f32 or bf16, or null
  int idx_new_bf16;
  const int64_t* slots;       // [T]
  int T, G;
  int64_t num_slots;          // P * BS
  int kv_nvfp4;
  int kv_fp8;
  void* k; void* v;           // caches
  uint8_t* k_scale; uint8_t* v_scale;
  float k_global, v_global;
  int idx_fp8;
  int idx_fp4;
  void* idx_keys;             // f32 / u8 [P, G, BS, D], or u8 [P, G, BS, D/2] NVFP4
  float* idx_scale;           // fp8: [P, G, BS]
  uint8_t* idx_block_scale;   // nvfp4: [P, G, BS, D/16]
  float idx_global;
  uint32_t* flags;
};

// NVFP4: lane owns 4 consecutive values; 4 lanes form one 16-value group.
__device__ __forceinline__ void quant_nvfp4_vals(const float (&x)[4], uint8_t* codes, uint8_t* scales, float g,
                                                 int lane) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  const float sb_in = __fdiv_rn(__fdiv_rn(a, 6.0f), g);
  const uint8_t sb_code = static_cast<uint8_t>(f32x2_to_e4m3x2(sb_in, 0.f) & 0xFF);
  const float denom = __fmul_rn(e4m3_to_f32(sb_code), g);
  uint16_t packed = 0;
  if (denom > 0.f) {
    float y[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) y[i] = __fdiv_rn(x[i], denom);
    y[4] = y[5] = y[6] = y[7] = 0.f;
    packed = static_cast<uint16_t>(f32x8_to_e2m1x8(y) & 0xFFFF);
  }
  *reinterpret_cast<uint16_t*>(codes + 2 * lane) = packed;
  if ((lane & 3) == 0) scales[lane >> 2] = sb_code;
}

__device__ __forceinline__ void quant_nvfp4_row(const uint16_t* src, uint8_t* codes, uint8_t* scales, float g,
                                                int lane) {
  const uint2 raw = *reinterpret_cast<const uint2*>(src + 4 * lane);
  const float x[4] = {bf16_bits_to_f32(raw.x & 0xFFFF), bf16_bits_to_f32(raw.x >> 16),
                      bf16_bits_to_f32(raw.y & 0xFFFF), bf16_bits_to_f32(raw.y >> 16)};
  quant_nvfp4_vals(x, codes, scales, g, lane);
}

__global__ void __launch_bounds__(256) kv_insert_kernel(InsertParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t total = static_cast<int64_t>(p.T) * p.G;
  for (int64_t w = warp; w < total; w += nwarps) {
    const int t = static_cast<int>(w / p.G);
    const int h = static_cast<int>(w % p.G);
    const int64_t slot = p.slots[t];
    if (slot < 0) continue;
    if (slot >= p.num_slots) {
      if (lane == 0) set_flag(p.flags, MSA_FLAG_BAD_SLOT);
      continue;
    }
    const int64_t page = slot / kBlock, off = slot % kBlock;
    const int64_t row = (page * p.G + h) * kBlock + off;   // (page, head, offset) row of any [P, G, BS, ...] cache
    const int64_t src = (static_cast<int64_t>(t) * p.G + h) * kDim;

    if (p.kv_fp8) {
      // code = E4M3_RNE_satfinite(x / s), one fp32 RN division per value
      const uint2 kk = *reinterpret_cast<const uint2*>(p.k_new + src + 4 * lane);
      const uint2 vv = *reinterpret_cast<const uint2*>(p.v_new + src + 4 * lane);
      auto enc = [](uint2 raw, float s) -> uint32_t {
        const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(bf16_bits_to_f32(raw.x & 0xFFFF), s),
                                            __fdiv_rn(bf16_bits_to_f32(raw.x >> 16), s));
        const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(bf16_bits_to_f32(raw.y & 0xFFFF), s),
                                            __fdiv_rn(bf16_bits_to_f32(raw.y >> 16), s));
        return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      };
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.k) + row * kDim + 4 * lane) = enc(kk, p.k_global);
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.v) + row * kDim + 4 * lane) = enc(vv, p.v_global);
    } else if (!p.kv_nvfp4) {
      const uint2 kk = *reinterpret_cast<const uint2*>(p.k_new + src + 4 * lane);
      const uint2 vv = *reinterpret_cast<const uint2*>(p.v_new + src + 4 * lane);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.k) + row * kDim + 4 * lane) = kk;
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.v) + row * kDim + 4 * lane) = vv;
    } else {
      quant_nvfp4_row(p.k_new + src, static_cast<uint8_t*>(p.k) + row * (kDim / 2), p.k_scale + row * (kDim / 16),
                      p.k_global, lane);
      quant_nvfp4_row(p.v_new + src, static_cast<uint8_t*>(p.v) + row * (kDim / 2), p.v_scale + row * (kDim / 16),
                      p.v_global, lane);
    }

    if (p.idx_new != nullptr) {
      float x[4];
      if (p.idx_new_bf16) {
        const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.idx_new) + src + 4 * lane);
        x[0] = bf16_bits_to_f32(raw.x & 0xFFFF); x[1] = bf16_bits_to_f32(raw.x >> 16);
        x[2] = bf16_bits_to_f32(raw.y & 0xFFFF); x[3] = bf16_bits_to_f32(raw.y >> 16);
      } else {
        const float4 raw = *reinterpret_cast<const float4*>(static_cast<const float*>(p.idx_new) + src + 4 * lane);
        x[0] = raw.x; x[1] = raw.y; x[2] = raw.z; x[3] = raw.w;
      }
      if (p.idx_fp4) {
        quant_nvfp4_vals(x, static_cast<uint8_t*>(p.idx_keys) + row * (kDim / 2),
                         p.idx_block_scale + row * (kDim / 16), p.idx_global, lane);
      } else if (!p.idx_fp8) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.idx_keys) + row * kDim + 4 * lane) =
            make_float4(x[0], x[1], x[2], x[3]);
      } else {
        float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float s = __fdiv_rn(a, 448.0f);
        uint32_t word = 0;
        if (s > 0.f) {
          const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
          const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
          word = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.idx_keys) + row * kDim + 4 * lane) = word;
        if (lane == 0) p.idx_scale[row] = s;
      }
    }
  }
}

cudaError_t launch_kv_insert(const InsertArgs& a, cudaStream_t stream, DispatchRecord* rec) {
  InsertParams p;
  p.k_new = static_cast<const uint16_t*>(a.k_new);
  p.v_new = static_cast<const uint16_t*>(a.v_new);
  p.idx_new = a.idx_new;
  p.idx_new_bf16 = a.idx_new_bf16;
  p.slots = a.slots;
  p.T = a.T;
  p.G = a.G;
  p.num_slots = a.num_slots;
  p.kv_nvfp4 = a.kv_nvfp4;
  p.kv_fp8 = a.kv_fp8;
  p.k = a.k; p.v = a.v;
  p.k_scale = static_cast<uint8_t*>(a.k_scale);
  p.v_scale = static_cast<uint8_t*>(a.v_scale);
  p.k_global = a.k_global; p.v_global = a.v_global;
  p.idx_fp8 = a.idx_fp8;
  p.idx_fp4 = a.idx_fp4;
  p.idx_keys = a.idx_keys;
  p.idx_scale = a.idx_scale;
  p.idx_block_scale = static_cast<uint8_t*>(a.idx_block_scale);
  p.idx_global = a.idx_global;
  p.flags = a.flags;
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

}  // namespace msa
