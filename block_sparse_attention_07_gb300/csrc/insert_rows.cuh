// Cache insertion rows: the parameters of an insert and the row writers that
// quantise one (token, head) row into the paged caches (bf16 copy, FP8 E4M3
// with a per-tensor scale, or NVFP4 for K/V; fp32 copy, FP8 E4M3 with a
// per-token scale, or NVFP4 for index keys). Every step of the quantisers is an
// IEEE round-to-nearest fp32 operation, so the bytes are a pure function of the
// input. Used by the insert kernels and by the index kernel's fused insert.
#pragma once

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

// The row writers below take one (token, head) row of D = 128 values, 4 per
// lane (dims 4 lane .. 4 lane + 3), as fp32 values (bf16-exact for bf16, FP8 and
// NVFP4 caches) and store it into row `row` of a [P, heads, BS, ...] cache.

// K or V row into the K/V cache (bf16 copy, FP8 E4M3 with the tensor scale, NVFP4).
__device__ __forceinline__ void store_kv_row(const InsertParams& p, bool is_v, int64_t row, const float (&x)[4],
                                             int lane) {
  void* base = is_v ? p.v : p.k;
  if (p.kv_fp8) {
    // code = E4M3_RNE_satfinite(x / s), one fp32 RN division per value
    const float s = is_v ? p.v_global : p.k_global;
    const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
    const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(base) + row * kDim + 4 * lane) =
        static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  } else if (!p.kv_nvfp4) {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(base) + row * kDim + 4 * lane) =
        make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
  } else {
    quant_nvfp4_vals(x, static_cast<uint8_t*>(base) + row * (kDim / 2),
                     (is_v ? p.v_scale : p.k_scale) + row * (kDim / 16), is_v ? p.v_global : p.k_global, lane);
  }
}

// Index key row into the index cache (fp32 copy, FP8 E4M3 + per-(token, head)
// scale s = amax / 448, or NVFP4).
__device__ __forceinline__ void store_idx_row(const InsertParams& p, int64_t row, const float (&x)[4], int lane) {
  if (p.idx_fp4) {
    quant_nvfp4_vals(x, static_cast<uint8_t*>(p.idx_keys) + row * (kDim / 2), p.idx_block_scale + row * (kDim / 16),
                     p.idx_global, lane);
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

__device__ __forceinline__ void load_bf16x4(const uint16_t* src, float (&x)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(src);
  x[0] = bf16_bits_to_f32(raw.x & 0xFFFF);
  x[1] = bf16_bits_to_f32(raw.x >> 16);
  x[2] = bf16_bits_to_f32(raw.y & 0xFFFF);
  x[3] = bf16_bits_to_f32(raw.y >> 16);
}

// Cache row of a slot, or -1 (negative slot: skip; out of range: skip and flag).
__device__ __forceinline__ int64_t slot_row(const InsertParams& p, int64_t slot, int h, int heads, int lane) {
  if (slot < 0) return -1;
  if (slot >= p.num_slots) {
    if (lane == 0) set_flag(p.flags, MSA_FLAG_BAD_SLOT);
    return -1;
  }
  return ((slot / kBlock) * heads + h) * kBlock + slot % kBlock;   // (page, head, offset) row
}

// One (token t, head h) insert: K and V rows, and the index key row when the
// insert carries index keys. Returns false when the slot was skipped.
__device__ __forceinline__ bool insert_row(const InsertParams& p, int t, int h, int lane) {
  const int64_t row = slot_row(p, p.slots[t], h, p.G, lane);
  if (row < 0) return false;
  const int64_t src = (static_cast<int64_t>(t) * p.G + h) * kDim + 4 * lane;
  float x[4];
  load_bf16x4(p.k_new + src, x);
  store_kv_row(p, false, row, x, lane);
  load_bf16x4(p.v_new + src, x);
  store_kv_row(p, true, row, x, lane);
  if (p.idx_new != nullptr) {
    if (p.idx_new_bf16) {
      load_bf16x4(static_cast<const uint16_t*>(p.idx_new) + src, x);
    } else {
      const float4 raw = *reinterpret_cast<const float4*>(static_cast<const float*>(p.idx_new) + src);
      x[0] = raw.x; x[1] = raw.y; x[2] = raw.z; x[3] = raw.w;
    }
    store_idx_row(p, row, x, lane);
  }
  return true;
}

// Device parameters of an insert from its host arguments.
inline InsertParams make_insert_params(const InsertArgs& a) {
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
  return p;
}

}  // namespace msa
