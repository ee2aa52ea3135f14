// C ABI of libmsa.so (declared in include/msa.h): host-side validation,
// the thread-local dispatch record, and the launches. Nothing here allocates
// device memory and nothing synchronises except msa_read_device_flags.
#include <cstring>

#include "msa_internal.h"

namespace msa {

static thread_local DispatchRecord g_record = {"(no launch yet)"};

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// One thread waits on an mbarrier that nothing arrives at, through the bounded
// wait every kernel of the library uses; when the wait gives up it records
// MSA_FLAG_TIMEOUT and the kernel returns. No copy targets the barrier or the
// CTA's shared memory, so giving up leaves nothing in flight.
__global__ void bounded_wait_selftest_kernel(uint32_t* flags) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  if (!mbar_wait(b, 0)) set_flag(flags, MSA_FLAG_TIMEOUT);
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape rules shared by every entry point.
static msa_status_t check_dims(const msa_dims_t* d) {
  if (d == nullptr) return MSA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->q_len < 1 || d->n_heads < 1 || d->n_kv_heads < 1 || d->n_idx_heads < 1 ||
      d->head_dim < 1 || d->block_size < 1 || d->max_blocks_per_seq < 1 || d->num_pages < 1 || d->topk < 1 ||
      d->local_blocks < 0)
    return MSA_ERR_INVALID_ARG;
  if (!(d->softmax_scale > 0.f) || d->softmax_scale != d->softmax_scale) return MSA_ERR_INVALID_ARG;
  if (d->head_dim != kDim || d->block_size != kBlock || d->local_blocks != 1) return MSA_ERR_UNSUPPORTED;
  if (d->n_idx_heads != d->n_kv_heads || d->n_heads != d->n_kv_heads * kGroup) return MSA_ERR_UNSUPPORTED;
  if (d->topk > 16 || d->q_len > 8 || d->n_idx_heads > 4 || d->batch > 4096) return MSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->max_blocks_per_seq) * kBlock > INT32_MAX) return MSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->num_pages) * d->n_kv_heads * kBlock > INT32_MAX) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

static msa_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

}  // namespace msa

using namespace msa;

extern "C" {

int msa_abi_version(void) { return MSA_ABI_VERSION; }

const char* msa_status_string(msa_status_t s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
    case MSA_ERR_DEVICE_FLAG: return "MSA_ERR_DEVICE_FLAG";
  }
  return "MSA_ERR_UNKNOWN";
}

msa_status_t msa_get_last_dispatch(char* buf, size_t len) {
  if (buf == nullptr || len == 0) return MSA_ERR_INVALID_ARG;
  strncpy(buf, g_record.text, len - 1);
  buf[len - 1] = '\0';
  return MSA_OK;
}

// Validates the caches of an insert and fills the shared launch arguments
// (everything but the source rows). idx_bf16_only: index sources must be bf16.
static msa_status_t insert_targets(const msa_dims_t* dims, bool with_idx, msa_dtype_t idx_new_dtype,
                                   const msa_kv_cache_t* cache, const msa_index_cache_t* idx_cache,
                                   uint32_t* dev_flags, InsertArgs& a) {
  if (cache == nullptr || dev_flags == nullptr || cache->k == nullptr || cache->v == nullptr) return MSA_ERR_INVALID_ARG;
  if (!aligned16(cache->k) || !aligned16(cache->v)) return MSA_ERR_INVALID_ARG;
  memset(&a, 0, sizeof(a));
  if (cache->dtype == MSA_NVFP4) {
    if (cache->k_scale == nullptr || cache->v_scale == nullptr) return MSA_ERR_INVALID_ARG;
    if (!(cache->k_global > 0.f) || !(cache->v_global > 0.f) || cache->k_global > 3.0e38f ||
        cache->v_global > 3.0e38f)
      return MSA_ERR_INVALID_ARG;
    a.kv_nvfp4 = 1;
  } else if (cache->dtype == MSA_FP8_E4M3) {
    if (!(cache->k_global > 0.f) || !(cache->v_global > 0.f) || cache->k_global > 3.0e38f ||
        cache->v_global > 3.0e38f)
      return MSA_ERR_INVALID_ARG;
    a.kv_fp8 = 1;
  } else if (cache->dtype != MSA_BF16) {
    return MSA_ERR_UNSUPPORTED;
  }
  if (with_idx) {
    if (idx_cache == nullptr || idx_cache->keys == nullptr || !aligned16(idx_cache->keys)) return MSA_ERR_INVALID_ARG;
    if (idx_cache->dtype == MSA_FP8_E4M3) {
      if (idx_cache->scale == nullptr) return MSA_ERR_INVALID_ARG;
      if (idx_new_dtype != MSA_F32 && idx_new_dtype != MSA_BF16) return MSA_ERR_UNSUPPORTED;
      a.idx_fp8 = 1;
    } else if (idx_cache->dtype == MSA_NVFP4) {
      if (idx_cache->block_scale == nullptr) return MSA_ERR_INVALID_ARG;
      if (!(idx_cache->global_scale > 0.f) || idx_cache->global_scale > 3.0e38f) return MSA_ERR_INVALID_ARG;
      if (idx_new_dtype != MSA_F32 && idx_new_dtype != MSA_BF16) return MSA_ERR_UNSUPPORTED;
      a.idx_fp4 = 1;
      a.idx_block_scale = idx_cache->block_scale;
      a.idx_global = idx_cache->global_scale;
    } else if (idx_cache->dtype == MSA_F32) {
      if (idx_new_dtype != MSA_F32) return MSA_ERR_UNSUPPORTED;
    } else {
      return MSA_ERR_UNSUPPORTED;
    }
    a.idx_new_bf16 = idx_new_dtype == MSA_BF16;
    a.idx_keys = idx_cache->keys;
    a.idx_scale = idx_cache->scale;
  }
  a.G = dims->n_kv_heads;
  a.num_slots = static_cast<int64_t>(dims->num_pages) * kBlock;
  a.k = cache->k;
  a.v = cache->v;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.k_global = cache->k_global;
  a.v_global = cache->v_global;
  a.flags = dev_flags;
  return MSA_OK;
}

msa_status_t msa_kv_insert_quant(const msa_dims_t* dims, const void* k_new, const void* v_new,
                                 const void* idx_k_new, msa_dtype_t idx_new_dtype, const int64_t* slot_mapping,
                                 int32_t num_tokens, const msa_kv_cache_t* cache,
                                 const msa_index_cache_t* idx_cache, uint32_t* dev_flags, void* stream) {
  msa_status_t st = check_dims(dims);
  if (st != MSA_OK) return st;
  if (num_tokens < 0 || cache == nullptr || dev_flags == nullptr) return MSA_ERR_INVALID_ARG;
  if (num_tokens == 0) {
    g_record.set("kv_insert empty");
    return MSA_OK;
  }
  if (k_new == nullptr || v_new == nullptr || slot_mapping == nullptr) return MSA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || (idx_k_new != nullptr && !aligned16(idx_k_new)))
    return MSA_ERR_INVALID_ARG;
  InsertArgs a;
  st = insert_targets(dims, idx_k_new != nullptr, idx_new_dtype, cache, idx_cache, dev_flags, a);
  if (st != MSA_OK) return st;
  a.k_new = k_new;
  a.v_new = v_new;
  a.idx_new = idx_k_new;
  a.slots = slot_mapping;
  a.T = num_tokens;
  return cuda_status(launch_kv_insert(a, static_cast<cudaStream_t>(stream), &g_record));
}

msa_status_t msa_qk_norm_rope_insert(const msa_dims_t* dims, const void* q, const void* k, const void* v,
                                     const void* idx_q, const void* idx_k, const int32_t* positions,
                                     const int64_t* slot_mapping, int32_t num_tokens, const msa_norm_rope_t* nr,
                                     void* q_out, void* idx_q_out, const msa_kv_cache_t* cache,
                                     const msa_index_cache_t* idx_cache, uint32_t* dev_flags, void* stream) {
  msa_status_t st = check_dims(dims);
  if (st != MSA_OK) return st;
  if (num_tokens < 0 || nr == nullptr || cache == nullptr || dev_flags == nullptr) return MSA_ERR_INVALID_ARG;
  const bool with_idx = idx_q != nullptr || idx_k != nullptr;
  if (with_idx && (idx_q == nullptr || idx_k == nullptr || idx_q_out == nullptr || nr->idx_q_weight == nullptr ||
                   nr->idx_k_weight == nullptr))
    return MSA_ERR_INVALID_ARG;
  if (!(nr->eps >= 0.f) || nr->eps > 1.f || !(nr->rope_theta > 1.f) || nr->rope_theta > 3.0e38f)
    return MSA_ERR_INVALID_ARG;
  if (num_tokens == 0) {
    g_record.set("qk_norm_rope_insert empty");
    return MSA_OK;
  }
  if (q == nullptr || k == nullptr || v == nullptr || positions == nullptr || slot_mapping == nullptr ||
      q_out == nullptr || nr->q_weight == nullptr || nr->k_weight == nullptr)
    return MSA_ERR_INVALID_ARG;
  const void* ptrs16[] = {q, k, v, q_out, nr->q_weight, nr->k_weight};
  for (const void* ptr : ptrs16)
    if (!aligned16(ptr)) return MSA_ERR_INVALID_ARG;
  if (with_idx && (!aligned16(idx_q) || !aligned16(idx_k) || !aligned16(idx_q_out) || !aligned16(nr->idx_q_weight) ||
                   !aligned16(nr->idx_k_weight)))
    return MSA_ERR_INVALID_ARG;
  if (with_idx && idx_cache != nullptr && idx_cache->dtype == MSA_F32) return MSA_ERR_UNSUPPORTED;
  PrologueArgs a;
  memset(&a, 0, sizeof(a));
  st = insert_targets(dims, with_idx, MSA_BF16, cache, idx_cache, dev_flags, a.ins);
  if (st != MSA_OK) return st;
  a.ins.k_new = k;
  a.ins.v_new = v;
  a.ins.idx_new = idx_k;
  a.ins.idx_new_bf16 = 1;
  a.ins.slots = slot_mapping;
  a.ins.T = num_tokens;
  a.q = q;
  a.idx_q = with_idx ? idx_q : nullptr;
  a.q_out = q_out;
  a.idx_q_out = with_idx ? idx_q_out : nullptr;
  a.positions = positions;
  a.wq = nr->q_weight;
  a.wk = nr->k_weight;
  a.wiq = nr->idx_q_weight;
  a.wik = nr->idx_k_weight;
  a.eps = nr->eps;
  a.theta = nr->rope_theta;
  a.H = dims->n_heads;
  a.I = dims->n_idx_heads;
  return cuda_status(launch_qk_norm_rope_insert(a, static_cast<cudaStream_t>(stream), &g_record));
}

// Validation and arguments of the index-score step (shared by the fused insert).
static msa_status_t index_args(const msa_dims_t* dims, const void* idx_q, msa_dtype_t q_dtype,
                               const msa_index_cache_t* idx_cache, const int32_t* block_table,
                               const int32_t* seq_lens, float* scores, uint32_t* dev_flags, IndexArgs& a) {
  msa_status_t st = check_dims(dims);
  if (st != MSA_OK) return st;
  if (idx_q == nullptr || idx_cache == nullptr || idx_cache->keys == nullptr || block_table == nullptr ||
      seq_lens == nullptr || scores == nullptr || dev_flags == nullptr)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(idx_q) || !aligned16(idx_cache->keys)) return MSA_ERR_INVALID_ARG;
  a.fp8 = 0;
  a.fp4 = 0;
  a.scale = nullptr;
  a.global_scale = 1.f;
  if (idx_cache->dtype == MSA_FP8_E4M3) {
    if (q_dtype != MSA_BF16) return MSA_ERR_UNSUPPORTED;
    if (idx_cache->scale == nullptr || !aligned16(idx_cache->scale)) return MSA_ERR_INVALID_ARG;
    a.fp8 = 1;
    a.scale = idx_cache->scale;
  } else if (idx_cache->dtype == MSA_NVFP4) {
    if (q_dtype != MSA_BF16) return MSA_ERR_UNSUPPORTED;
    if (idx_cache->block_scale == nullptr || !aligned16(idx_cache->block_scale)) return MSA_ERR_INVALID_ARG;
    if (!(idx_cache->global_scale > 0.f) || idx_cache->global_scale > 3.0e38f) return MSA_ERR_INVALID_ARG;
    a.fp4 = 1;
    a.scale = idx_cache->block_scale;
    a.global_scale = idx_cache->global_scale;
  } else if (idx_cache->dtype == MSA_F32) {
    if (q_dtype != MSA_F32) return MSA_ERR_UNSUPPORTED;
  } else {
    return MSA_ERR_UNSUPPORTED;
  }
  a.q = idx_q;
  a.keys = idx_cache->keys;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.scores = scores;
  a.flags = dev_flags;
  a.B = dims->batch;
  a.Q = dims->q_len;
  a.I = dims->n_idx_heads;
  a.NB = dims->max_blocks_per_seq;
  a.P = dims->num_pages;
  return MSA_OK;
}

msa_status_t msa_index_score(const msa_dims_t* dims, const void* idx_q, msa_dtype_t q_dtype,
                             const msa_index_cache_t* idx_cache, const int32_t* block_table,
                             const int32_t* seq_lens, float* scores, uint32_t* dev_flags, void* stream) {
  IndexArgs a;
  const msa_status_t st = index_args(dims, idx_q, q_dtype, idx_cache, block_table, seq_lens, scores, dev_flags, a);
  if (st != MSA_OK) return st;
  return cuda_status(launch_index_score(a, nullptr, static_cast<cudaStream_t>(stream), &g_record));
}

msa_status_t msa_insert_index_score(const msa_dims_t* dims, const void* k_new, const void* v_new,
                                    const void* idx_k_new, const int64_t* slot_mapping,
                                    const msa_kv_cache_t* cache, const void* idx_q,
                                    const msa_index_cache_t* idx_cache, const int32_t* block_table,
                                    const int32_t* seq_lens, float* scores, uint32_t* dev_flags, void* stream) {
  // the index query and the new index keys are fp32 with an fp32 index cache, bf16 otherwise
  const msa_dtype_t idx_dt = idx_cache != nullptr && idx_cache->dtype == MSA_F32 ? MSA_F32 : MSA_BF16;
  IndexArgs a;
  msa_status_t st = index_args(dims, idx_q, idx_dt, idx_cache, block_table, seq_lens, scores, dev_flags, a);
  if (st != MSA_OK) return st;
  if (dims->q_len != 1) return MSA_ERR_UNSUPPORTED;
  if (cache == nullptr || k_new == nullptr || v_new == nullptr || idx_k_new == nullptr || slot_mapping == nullptr)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(idx_k_new)) return MSA_ERR_INVALID_ARG;
  InsertArgs ins;
  st = insert_targets(dims, true, idx_dt, cache, idx_cache, dev_flags, ins);
  if (st != MSA_OK) return st;
  ins.k_new = k_new;
  ins.v_new = v_new;
  ins.idx_new = idx_k_new;
  ins.slots = slot_mapping;
  ins.T = dims->batch;
  return cuda_status(launch_index_score(a, &ins, static_cast<cudaStream_t>(stream), &g_record));
}

msa_status_t msa_select_blocks(const msa_dims_t* dims, const float* scores, const int32_t* seq_lens,
                               int32_t* selected, uint32_t* dev_flags, void* stream) {
  msa_status_t st = check_dims(dims);
  if (st != MSA_OK) return st;
  if (scores == nullptr || seq_lens == nullptr || selected == nullptr || dev_flags == nullptr)
    return MSA_ERR_INVALID_ARG;
  SelectArgs a{scores, seq_lens, selected, dev_flags, dims->batch, dims->q_len, dims->n_idx_heads,
               dims->max_blocks_per_seq, dims->topk};
  return cuda_status(launch_select_blocks(a, static_cast<cudaStream_t>(stream), &g_record));
}

size_t msa_sparse_gqa_workspace_size(const msa_dims_t* dims, msa_dtype_t kv_dtype) {
  (void)kv_dtype;
  if (check_dims(dims) != MSA_OK) return 0;
  return gqa_workspace_bytes(dims->batch, dims->q_len, dims->n_kv_heads, dims->topk);
}

static msa_status_t sparse_gqa_common(const msa_dims_t* dims, const void* q, const msa_kv_cache_t* cache,
                                      const int32_t* block_table, const int32_t* seq_lens, const int32_t* selected,
                                      const float* scores, void* out, float* lse, void* workspace,
                                      size_t workspace_bytes, uint32_t* dev_flags, void* stream) {
  msa_status_t st = check_dims(dims);
  if (st != MSA_OK) return st;
  if (q == nullptr || cache == nullptr || cache->k == nullptr || cache->v == nullptr || block_table == nullptr ||
      seq_lens == nullptr || selected == nullptr || out == nullptr || dev_flags == nullptr)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(cache->k) || !aligned16(cache->v)) return MSA_ERR_INVALID_ARG;
  GqaArgs a;
  memset(&a, 0, sizeof(a));
  if (cache->dtype == MSA_NVFP4) {
    if (cache->k_scale == nullptr || cache->v_scale == nullptr || !aligned16(cache->k_scale) ||
        !aligned16(cache->v_scale))
      return MSA_ERR_INVALID_ARG;
    if (!(cache->k_global > 0.f) || !(cache->v_global > 0.f)) return MSA_ERR_INVALID_ARG;
    a.nvfp4 = 1;
  } else if (cache->dtype == MSA_FP8_E4M3) {
    if (!(cache->k_global > 0.f) || !(cache->v_global > 0.f) || cache->k_global > 3.0e38f ||
        cache->v_global > 3.0e38f)
      return MSA_ERR_INVALID_ARG;
    a.fp8 = 1;
  } else if (cache->dtype != MSA_BF16) {
    return MSA_ERR_UNSUPPORTED;
  }
  const size_t need = gqa_workspace_bytes(dims->batch, dims->q_len, dims->n_kv_heads, dims->topk);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MSA_ERR_WORKSPACE;
  a.q = static_cast<const uint16_t*>(q);
  a.k = cache->k;
  a.v = cache->v;
  a.k_scale = static_cast<const uint8_t*>(cache->k_scale);
  a.v_scale = static_cast<const uint8_t*>(cache->v_scale);
  a.k_global = cache->k_global;
  a.v_global = cache->v_global;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.selected = selected;
  a.scores = scores;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.workspace = static_cast<float*>(workspace);
  a.flags = dev_flags;
  a.B = dims->batch;
  a.Q = dims->q_len;
  a.H = dims->n_heads;
  a.G = dims->n_kv_heads;
  a.NB = dims->max_blocks_per_seq;
  a.P = dims->num_pages;
  a.K = dims->topk;
  a.softmax_scale = dims->softmax_scale;
  return cuda_status(launch_sparse_gqa(a, static_cast<cudaStream_t>(stream), &g_record));
}

msa_status_t msa_sparse_gqa_decode(const msa_dims_t* dims, const void* q, const msa_kv_cache_t* cache,
                                   const int32_t* block_table, const int32_t* seq_lens, const int32_t* selected,
                                   void* out, float* lse, void* workspace, size_t workspace_bytes,
                                   uint32_t* dev_flags, void* stream) {
  return sparse_gqa_common(dims, q, cache, block_table, seq_lens, selected, nullptr, out, lse, workspace,
                           workspace_bytes, dev_flags, stream);
}

msa_status_t msa_select_sparse_gqa_decode(const msa_dims_t* dims, const void* q, const msa_kv_cache_t* cache,
                                          const int32_t* block_table, const int32_t* seq_lens, const float* scores,
                                          int32_t* selected, void* out, float* lse, void* workspace,
                                          size_t workspace_bytes, uint32_t* dev_flags, void* stream) {
  if (scores == nullptr) return MSA_ERR_INVALID_ARG;
  return sparse_gqa_common(dims, q, cache, block_table, seq_lens, selected, scores, out, lse, workspace,
                           workspace_bytes, dev_flags, stream);
}

msa_status_t msa_selftest_bounded_wait(uint32_t* dev_flags, void* stream) {
  if (dev_flags == nullptr) return MSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(dev_flags);
  const cudaError_t err = cudaGetLastError();
  g_record.set("selftest bounded_wait grid=1 block=32");
  return err == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

msa_status_t msa_read_device_flags(const uint32_t* dev_flags, uint32_t* host_flags, void* stream) {
  if (dev_flags == nullptr || host_flags == nullptr) return MSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_flags, dev_flags, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MSA_ERR_CUDA;
  return *host_flags != 0 ? MSA_ERR_DEVICE_FLAG : MSA_OK;
}

}  // extern "C"
