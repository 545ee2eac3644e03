// Device helpers shared by the paged-attention kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace pa {

// Bits of the per-device error word.
constexpr unsigned kErrBlockId = 1u;       // a block-table entry outside [0, num_blocks)
constexpr unsigned kErrShortContext = 2u;  // a row that sees no token, or a context above the bound
constexpr unsigned kErrTimeout = 4u;       // an mbarrier wait hit its iteration limit
constexpr unsigned kErrBadInput = 8u;      // a token id outside the vocabulary, or a distribution with no mass

// Upper bounds before a wait gives up (a page copy lands in microseconds).  kWaitLimit counts
// mbarrier.try_wait polls, each of which suspends the thread for up to a hardware time limit
// while the phase is incomplete (3.8 us per poll measured on GB300): 2^18 polls is about one
// second.  kSpinLimit counts iterations of the issuer loops that probe several barriers with the
// non-suspending mbarrier.test_wait (tens of ns each): 2^22 iterations is a fraction of a second.
constexpr uint32_t kWaitLimit = 1u << 18;
constexpr uint32_t kSpinLimit = 1u << 22;

constexpr float kLog2e = 1.4426950408889634f;

// Arguments of every attention kernel.  Pointers are device pointers.
struct AttnParams {
  const __nv_bfloat16* q;       // [B, q_len, Hq, d]
  const uint8_t* k_cache;       // [NB, Hkv, bs, d] (bf16 or E4M3 bytes)
  const uint8_t* v_cache;
  const int32_t* block_table;   // [B, max_blocks_per_seq]
  const int32_t* context_lens;  // [B]
  const float* k_scale;         // [NB, Hkv] (fp8 only)
  const float* v_scale;
  __nv_bfloat16* out;           // [B, q_len, Hq, d]
  float* part_o;                // [B, q_len, Hq, P, d]  normalised partial outputs
  float* part_lse;              // [B, q_len, Hq, P]     log2 of each partition's softmax mass
  const uint32_t* tree_mask;    // [B, q_len] ancestor bitmasks over the new tokens, or null (causal)
  const int32_t* query_start_loc;  // [B + 1] packed query rows per sequence (prefill), or null
  unsigned* err;                // per-device error word
  int num_seqs;
  int max_blocks_per_seq;
  int num_blocks;
  int q_len;
  int num_q_heads;
  int num_kv_heads;
  int pages_per_partition;
  int max_partitions;
  int max_context_len;          // host-side bound; longer contexts are clamped and flagged
  int total_q;                  // rows of the packed q / out (prefill)
  float scale_log2;             // scale * log2(e): scores are kept in base-2 units
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier + bulk asynchronous copy (TMA unit) -------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of one phase (never suspends the thread: for loops that poll several
// barriers, where a suspended probe of one would miss another one completing).
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

// Bounded wait on one phase of an mbarrier.  Returns false when `limit` polls did not see it.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t limit = kWaitLimit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// One contiguous global -> shared copy through the TMA unit, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---- arithmetic ------------------------------------------------------------------------------

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

union F2U {
  float2 f;
  unsigned long long u;
};

// d = a * b + c on a pair of fp32 lanes (one sm_100-family FFMA2 instruction).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  F2U ua, ub, uc, ud;
  ua.f = a;
  ub.f = b;
  uc.f = c;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(ud.u) : "l"(ua.u), "l"(ub.u), "l"(uc.u));
  return ud.f;
}

// Two packed bf16 -> two fp32 (a bf16 is the upper half of a binary32: exact).
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// acc.x += low bf16 of w, acc.y += high bf16 of w, in fp32: the sm_100-family mixed-precision add
// (the bf16 operand widens exactly, one rounding of the sum), bit for bit
// ffma2(bf16x2_to_f2(w), {1, 1}, acc) without the two unpacking instructions.
__device__ __forceinline__ float2 add_bf16x2_f2(uint32_t w, float2 acc) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
  return acc;
}

// Two packed E4M3 bytes (low byte first) -> two fp32, through the hardware e4m3x2 -> f16x2
// conversion (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t w) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(w));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ void record_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// context_lens[b], clamped to the host-side bound the grid and scratch were sized for (a longer
// context would index past its block-table row); thread 0 of partition 0 flags the clamp.
__device__ __forceinline__ int context_len(const AttnParams& p, int b, bool flag) {
  int L = p.context_lens[b];
  if (L > p.max_context_len) {
    if (flag) record_error(p.err, kErrShortContext);
    L = p.max_context_len;
  }
  return L;
}

// Last step of a split-KV partition: combine the per-warp online-softmax states that the CTA's
// warps left in shared memory (wacc [W][G][D] unnormalised outputs, wm [W][G] running maxima and
// wl [W][G] sums, base 2) and store either the finished bf16 rows (the sequence has one
// partition) or the normalised partial output and its log2-sum-exp for the merge kernel.
template <int G, int D, int W>
__device__ __forceinline__ void store_partition(const AttnParams& p, const float* wacc, const float* wm,
                                                const float* wl, int b, int g, int part, int nparts) {
  const int Hq = p.num_q_heads;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx / D;
    const int dd = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w * G + h]);
    float o = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float f = fast_exp2(wm[w * G + h] - M);
        lsum += f * wl[w * G + h];
        o += f * wacc[(w * G + h) * D + dd];
      }
      o = o / lsum;
    }
    const int qh = g * G + h;
    if (nparts == 1) {
      p.out[((size_t)b * Hq + qh) * D + dd] = __float2bfloat16(o);
    } else {
      const size_t row = ((size_t)b * Hq + qh) * p.max_partitions + part;
      p.part_o[row * D + dd] = o;
      if (dd == 0) p.part_lse[row] = (M == -INFINITY) ? -INFINITY : M + __log2f(lsum);
    }
  }
}

}  // namespace pa
