// Log-sum-exp merge of split-KV partitions.
//
// Partition p of a row holds o_p = (sum_j 2^(s_j - m_p) v_j) / l_p and lse_p = m_p + log2(l_p)
// over its tokens (scores in base-2 units).  The row's softmax over all tokens is the
// weighted mix o = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M), M = max_p lse_p: the same
// rescaling the online softmax applies between tiles (studybook fde-roadmap ch.10, section
// 10.1.2, tiling + online softmax), applied once across partitions.
#include "pa_kernels.h"

namespace pa {
namespace {

// One pass over a row's partitions, kBatch per turn with their loads issued together; the running
// maximum M rescales what was summed before it grew (log-sum-exp rule).
template <int D, int kBatch>
__device__ __forceinline__ void merge_partitions(const float* lse, const float* po, int nparts, int lane, float& M,
                                                 float& wsum, float (&acc)[D / 32]) {
  constexpr int kDPL = D / 32;
  for (int q0 = 0; q0 < nparts; q0 += kBatch) {
    float lq[kBatch];
    float vv[kBatch][kDPL];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int q = min(q0 + k, nparts - 1);
      lq[k] = q0 + k < nparts ? lse[q] : -INFINITY;
      const float* src = po + (size_t)q * D + lane * kDPL;
      if constexpr (kDPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        vv[k][0] = v.x; vv[k][1] = v.y; vv[k][2] = v.z; vv[k][3] = v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        vv[k][0] = v.x; vv[k][1] = v.y;
      }
    }
    float mb = M;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) mb = fmaxf(mb, lq[k]);
    if (mb == -INFINITY) continue;  // nothing with mass yet
    const float alpha = M == -INFINITY ? 0.f : fast_exp2(M - mb);
    wsum *= alpha;
#pragma unroll
    for (int e = 0; e < kDPL; ++e) acc[e] *= alpha;
    M = mb;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const float w = lq[k] == -INFINITY ? 0.f : fast_exp2(lq[k] - M);
      wsum += w;
#pragma unroll
      for (int e = 0; e < kDPL; ++e) acc[e] += w * vv[k][e];
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const AttnParams p) {
  constexpr int kDPL = D / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads;
  const long rows = (long)p.num_seqs * p.q_len * Hq;
  const long row = (long)blockIdx.x * 4 + warp;  // (b, i, h) flattened
  if (row >= rows) return;
  const int b = (int)(row / ((long)p.q_len * Hq));
  const int L = context_len(p, b, false);
  if (L <= 0) return;
  const int npages = (L + 15) / 16;
  const int nparts = (npages + p.pages_per_partition - 1) / p.pages_per_partition;
  if (nparts <= 1) return;  // the attention kernel wrote this row directly
  // launched as a programmatic dependent of the attention kernel: wait for its partials
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* lse = p.part_lse + row * p.max_partitions;
  const float* po = p.part_o + row * p.max_partitions * D;

  float M = -INFINITY, wsum = 0.f;
  float acc[kDPL];
#pragma unroll
  for (int e = 0; e < kDPL; ++e) acc[e] = 0.f;
  // a few partitions: eight per turn; many (long contexts): thirty-two per turn, fewer round trips
  if (nparts <= 8)
    merge_partitions<D, 8>(lse, po, nparts, lane, M, wsum, acc);
  else
    merge_partitions<D, 32>(lse, po, nparts, lane, M, wsum, acc);
  __nv_bfloat16* dst = p.out + row * D + lane * kDPL;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int e = 0; e < kDPL; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}

}  // namespace

cudaError_t launch_merge(const AttnParams& p, const Launch& l) {
  const long rows = (long)p.num_seqs * p.q_len * p.num_q_heads;
  const unsigned blocks = (unsigned)((rows + 3) / 4);
  if (blocks == 0) return cudaSuccess;
  // programmatic dependent launch: the merge grid is scheduled while the attention kernel's
  // last CTAs run and waits (griddepcontrol.wait) for their partials before reading them
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (l.head_dim == 128) return cudaLaunchKernelEx(&cfg, merge_kernel<128>, p);
  if (l.head_dim == 64) return cudaLaunchKernelEx(&cfg, merge_kernel<64>, p);
  return cudaErrorInvalidConfiguration;
}

}  // namespace pa
