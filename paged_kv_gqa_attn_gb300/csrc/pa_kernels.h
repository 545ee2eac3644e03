// Host-side launchers of the paged-attention kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_device.cuh"

namespace pa {

// Split-KV launch geometry: grid = (max_partitions, num_kv_heads, num_seqs).
struct Launch {
  int head_dim;
  int group;  // num_q_heads / num_kv_heads
  bool fp8;
  cudaStream_t stream;
};

// Each returns cudaSuccess or the launch error.  Unsupported combinations return
// cudaErrorInvalidConfiguration (the caller has already checked them).
cudaError_t launch_decode(const AttnParams& p, const Launch& l);
// Decode on mma.sync (same grid, partitions and partial layout as launch_decode): E4M3 caches for
// every group, bf16 caches for groups of 1, 2 and 4.  tk / tv: 2-D TMA maps of the K and V pools
// viewed as [num_blocks * Hkv * bs, d] with 16-row boxes of 128-byte rows and the 128-byte swizzle
// (bf16: 64-dim boxes, as for verify; E4M3 d = 128: one box per page), or for E4M3 d = 64 one box
// of 64-byte rows with the 64-byte swizzle.
cudaError_t launch_decode_mma(const AttnParams& p, const Launch& l, const CUtensorMap& tk, const CUtensorMap& tv);
// Verify: planner + persistent tcgen05 kernel + segment merge, all on l.stream.  `scratch` holds
// verify_scratch_bytes(...) bytes; ncta = verify_resident_ctas(num_sms) persistent CTAs.
// tk / tv: 2-D TMA maps of the bf16 K and V pools viewed as [num_blocks * Hkv * bs, d] with
// 16 x 64 boxes and the 128-byte swizzle.
int verify_resident_ctas(int num_sms);
size_t verify_scratch_bytes(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim, int ncta);
cudaError_t launch_verify_tc(const AttnParams& p, const Launch& l, void* scratch, int ncta, const CUtensorMap& tk,
                             const CUtensorMap& tv);
cudaError_t launch_merge(const AttnParams& p, const Launch& l);
// Paged prefill (varlen queries, p.query_start_loc / p.total_q set; p.q_len = the host bound on
// any sequence's new rows): a planner orders the (sequence, 128-row tile) pairs by work, then one
// tcgen05 CTA per (kv head, pair).  scratch holds prefill_scratch_bytes(...) bytes.
size_t prefill_scratch_bytes(int num_seqs, int max_q_len, int group);
// Verify / tree verify (p.tree_mask) with bf16 caches and 65-128 rows per kv head on the prefill
// kernel split like decode: grid (partition, kv head, sequence) from p.pages_per_partition (a
// multiple of 4 pages) / p.max_partitions, partials in p.part_o / p.part_lse for launch_merge.
cudaError_t launch_verify_split(const AttnParams& p, const Launch& l, const CUtensorMap& tk, const CUtensorMap& tv);
cudaError_t launch_prefill_tc(const AttnParams& p, const Launch& l, int max_q_len, void* scratch, const CUtensorMap& tk,
                              const CUtensorMap& tv);
// KV append (bf16 scatter, or fp8 with per-(block, head) rescaling); arguments already checked.
cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const int32_t* block_table, const int32_t* context_lens, int num_seqs, int n_new,
                          int max_blocks_per_seq, int num_blocks, int num_kv_heads, int head_dim, bool fp8,
                          float* k_scale, float* v_scale, unsigned* err, cudaStream_t stream);

// Speculative acceptance: scan kernel over vocabulary chunks, then the pick kernel (programmatic
// dependent).  chunk_sums holds accept_scratch_bytes(num_seqs, vocab) bytes.
size_t accept_scratch_bytes(int num_seqs, int vocab);
cudaError_t launch_accept(const float* p, const float* q, const int32_t* draft, const float* u_accept,
                          const uint32_t* words, int num_seqs, int num_draft, int vocab, int32_t* out_tokens,
                          int32_t* num_accepted, void* scratch, unsigned* err, cudaStream_t stream);
// Programmatic dependent launch of `fn` on `st` (cudaLaunchKernelExC with the
// programmatic-stream-serialisation attribute).
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, int smem, cudaStream_t st, void** args);

// Raise a kernel's dynamic shared-memory limit on the current device (first call per device
// and kernel only; later calls are a table lookup).
cudaError_t set_smem_once(const void* kernel, int bytes);

// Host-side argument checks of paged_attn_decode (a pa_status), and the current device's
// error-word address; neither allocates.
int validate_decode_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                         const int32_t* context_lens, int num_seqs, int max_blocks_per_seq, int num_blocks,
                         int max_context_len, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int kv_dtype, const float* k_scale, const float* v_scale,
                         const void* out);
cudaError_t error_word_address(unsigned** out);

}  // namespace pa
