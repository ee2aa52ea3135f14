// Internal interface between the C ABI (msa_api.cu) and the kernel launchers.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>
#include <utility>

#include "msa_device.cuh"

namespace msa {

// Thread-local record of what actually launched ("configured != executed").
struct DispatchRecord {
  char text[512];
  void set(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(text, sizeof(text), fmt, ap);
    va_end(ap);
  }
};

int device_sm_count();

// Launches a kernel with programmatic stream serialisation: it may begin while
// the previous kernel on the stream is still running, and waits for it with
// griddep_wait() before touching memory that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl for a grid of thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                               int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct InsertArgs {
  const void* k_new;
  const void* v_new;
  const void* idx_new;
  int idx_new_bf16;
  const int64_t* slots;
  int T, G;
  int64_t num_slots;
  int kv_nvfp4;
  int kv_fp8;
  void* k;
  void* v;
  void* k_scale;
  void* v_scale;
  float k_global, v_global;
  int idx_fp8;
  int idx_fp4;
  void* idx_keys;
  float* idx_scale;
  void* idx_block_scale;
  float idx_global;
  uint32_t* flags;
};

struct IndexArgs {
  const void* q;          // [B, Q, I, D] f32 or bf16
  const void* keys;       // [P, I, BS, D] f32 / u8 E4M3, or [P, I, BS, D/2] NVFP4
  const void* scale;      // fp8: fp32 [P, I, BS]; nvfp4: E4M3 [P, I, BS, D/16]
  float global_scale;     // nvfp4 only
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* scores;          // [B, Q, I, NB]
  uint32_t* flags;
  int B, Q, I, NB, P;
  int fp8, fp4;
};

struct SelectArgs {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* selected;
  uint32_t* flags;
  int B, Q, I, NB, K;
};

struct GqaArgs {
  const uint16_t* q;       // bf16 [B, Q, H, D]
  int nvfp4;
  int fp8;
  const void* k;           // bf16 [P, G, BS, D], u8 E4M3 [P, G, BS, D] or u8 [P, G, BS, D/2]
  const void* v;
  const uint8_t* k_scale;  // nvfp4 [P, G, BS, D/16]
  const uint8_t* v_scale;
  float k_global, v_global;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* selected;  // [B, Q, G, K]; written first when scores is set
  const float* scores;      // [B, Q, I, NB] or null (fused selection)
  uint16_t* out;            // bf16 [B, Q, H, D]
  float* lse;               // [B, Q, H] or null
  float* workspace;
  uint32_t* flags;
  int B, Q, H, G, NB, P, K;
  float softmax_scale;
};

// Floats per split-K partial: o [16 heads][128 dims], then m [16], then l [16].
// The workspace holds rows x topk partials, then one 64-bit ticket per row.
constexpr int kPartialFloats = kGroup * kDim + 2 * kGroup;

size_t gqa_workspace_bytes(int B, int Q, int G, int K);

cudaError_t launch_kv_insert(const InsertArgs& a, cudaStream_t stream, DispatchRecord* rec);

// QK-norm + RoPE + insert: the insert's arguments (k_new / v_new / idx_new are
// the un-normalised bf16 projections) plus the queries and the norm / rotary
// parameters.
struct PrologueArgs {
  InsertArgs ins;
  const void* q;            // bf16 [T, H, D]
  const void* idx_q;        // bf16 [T, I, D] or null (layer reusing a selection)
  void* q_out;
  void* idx_q_out;
  const int32_t* positions;
  const float* wq;
  const float* wk;
  const float* wiq;
  const float* wik;
  float eps;
  float theta;
  int H, I;
};
cudaError_t launch_qk_norm_rope_insert(const PrologueArgs& a, cudaStream_t stream, DispatchRecord* rec);
// ins: the step's insert run inside the same launch (FP8 / NVFP4 index keys,
// one query position, token t = request t's token at position L_t - 1), or null.
cudaError_t launch_index_score(const IndexArgs& a, const InsertArgs* ins, cudaStream_t stream, DispatchRecord* rec);
cudaError_t launch_select_blocks(const SelectArgs& a, cudaStream_t stream, DispatchRecord* rec);
cudaError_t launch_sparse_gqa(const GqaArgs& a, cudaStream_t stream, DispatchRecord* rec);

}  // namespace msa
