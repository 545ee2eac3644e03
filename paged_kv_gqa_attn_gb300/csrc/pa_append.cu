// Append the new tokens' K and V to the paged cache (the step before attention).
//
// Each decode (or verify) step stores the K and V it computed for its new token(s) so that later
// steps read them from the cache (studybook fde-roadmap ch.10, sections 10.2.2 and 10.3.2); in a
// paged cache the slot of position j is slot j % bs of block block_table[b][j / bs]
// (section 10.12.2; aegloslab servingai 5.3.7).  context_lens counts the new tokens: sequence
// b's n_new tokens take positions [L_b - n_new, L_b).
//
// bf16 caches take the rows as they are.  fp8 (E4M3) caches keep one fp32 scale per (physical
// block, kv head) equal to amax / 448 over the block's valid tokens (section 10.8.2): an append
// recomputes amax over the block's older tokens (decoded with the old scale) and the new ones,
// re-encodes the older tokens when the scale changes, and encodes the new ones; all arithmetic
// fp32, rounding to E4M3 nearest-even with saturation (cvt.rn.satfinite).
//
// The blocks written are assumed to belong to their sequence alone (a block shared with another
// sequence is copied before it is written: the scheduler's job).
#include "pa_kernels.h"

namespace pa {
namespace {

struct AppendParams {
  const __nv_bfloat16* k_new;  // [B, n_new, Hkv, d]
  const __nv_bfloat16* v_new;
  uint8_t* k_cache;            // [NB, Hkv, bs, d]
  uint8_t* v_cache;
  const int32_t* block_table;
  const int32_t* context_lens;
  float* k_scale;              // [NB, Hkv] (fp8)
  float* v_scale;
  unsigned* err;
  int num_seqs, n_new, max_blocks_per_seq, num_blocks, num_kv_heads;
};

__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  uint32_t h2;
  const uint16_t w = b;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(w));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}

// Two floats -> two E4M3 codes (round to nearest even, saturate finite values at +-448).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// bf16: a scatter, one thread per 16-byte piece of a new row; consecutive threads take
// consecutive pieces of the source [B, n_new, Hkv, d] (K pieces, then V pieces).
template <int D>
__global__ void __launch_bounds__(256) append_bf16_kernel(const AppendParams p) {
  constexpr int kChunks = D * 2 / 16;
  const int64_t per_side = (int64_t)p.num_seqs * p.n_new * p.num_kv_heads * kChunks;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 2 * per_side) return;
  const bool is_v = i >= per_side;
  const int64_t r = is_v ? i - per_side : i;
  const int c = (int)(r % kChunks);
  const int64_t row = r / kChunks;  // (b * n_new + t) * Hkv + g
  const int g = (int)(row % p.num_kv_heads);
  const int64_t bt = row / p.num_kv_heads;
  const int t = (int)(bt % p.n_new);
  const int b = (int)(bt / p.n_new);
  const int L = p.context_lens[b];
  const int j = L - p.n_new + t;
  if (L < p.n_new || L > p.max_blocks_per_seq * 16) {  // shorter than the new rows, or past the table
    record_error(p.err, kErrShortContext);
    return;
  }
  const int pb = p.block_table[(size_t)b * p.max_blocks_per_seq + j / 16];
  if (pb < 0 || pb >= p.num_blocks) {
    record_error(p.err, kErrBlockId);
    return;
  }
  const __nv_bfloat16* src = is_v ? p.v_new : p.k_new;
  uint8_t* cache = is_v ? p.v_cache : p.k_cache;
  const uint4 v = *reinterpret_cast<const uint4*>(src + row * D + c * 8);
  *reinterpret_cast<uint4*>(cache + ((((size_t)pb * p.num_kv_heads + g) * 16 + j % 16) * D + c * 8) * 2) = v;
}

// fp8: one CTA per (kv head, sequence, K or V) walks the one or two blocks the new tokens land in.
template <int D>
__global__ void __launch_bounds__(128) append_fp8_kernel(const AppendParams p) {
  __shared__ float vals[16 * D];  // the block's valid tokens, decoded / new, fp32
  __shared__ float red[4];
  const int g = blockIdx.x, b = blockIdx.y;
  const bool is_v = blockIdx.z == 1;
  const int L = p.context_lens[b];
  const int first = L - p.n_new;
  if (first < 0 || L > p.max_blocks_per_seq * 16) {
    if (threadIdx.x == 0) record_error(p.err, kErrShortContext);
    return;
  }
  const __nv_bfloat16* src = is_v ? p.v_new : p.k_new;
  uint8_t* cache = is_v ? p.v_cache : p.k_cache;
  float* scales = is_v ? p.v_scale : p.k_scale;
  for (int blk = first / 16; blk <= (L - 1) / 16; ++blk) {
    const int pb = p.block_table[(size_t)b * p.max_blocks_per_seq + blk];
    if (pb < 0 || pb >= p.num_blocks) {
      if (threadIdx.x == 0) record_error(p.err, kErrBlockId);
      continue;
    }
    const int lo = blk * 16;
    const int s0 = max(first - lo, 0);   // slots [0, s0): older tokens
    const int s1 = min(L - lo, 16);      // slots [s0, s1): new tokens
    uint8_t* page = cache + ((size_t)pb * p.num_kv_heads + g) * 16 * D;
    const float old_scale = scales[(size_t)pb * p.num_kv_heads + g];
    float amax = 0.f;
    for (int idx = threadIdx.x; idx < s1 * D; idx += blockDim.x) {
      const int sl = idx / D, c = idx - sl * D;
      float v;
      if (sl < s0) {
        v = e4m3_to_f32(page[idx]) * old_scale;
      } else {
        v = __bfloat162float(src[(((size_t)b * p.n_new + (lo + sl - first)) * p.num_kv_heads + g) * D + c]);
      }
      vals[idx] = v;
      amax = fmaxf(amax, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float new_scale = amax > 0.f ? amax / 448.f : 1.f;
    const int from = (s0 > 0 && new_scale != old_scale) ? 0 : s0;  // re-encode older tokens?
    for (int idx = threadIdx.x * 2 + from * D; idx < s1 * D; idx += blockDim.x * 2) {
      const uint16_t two = f32x2_to_e4m3x2(vals[idx] / new_scale, vals[idx + 1] / new_scale);
      *reinterpret_cast<uint16_t*>(page + idx) = two;
    }
    __syncthreads();  // every thread has read old_scale and vals before they change
    if (threadIdx.x == 0) scales[(size_t)pb * p.num_kv_heads + g] = new_scale;
  }
}

template <int D>
cudaError_t launch_d(const AppendParams& p, bool fp8, cudaStream_t st) {
  if (fp8) {
    append_fp8_kernel<D><<<dim3(p.num_kv_heads, p.num_seqs, 2), 128, 0, st>>>(p);
  } else {
    const int64_t threads = 2LL * p.num_seqs * p.n_new * p.num_kv_heads * (D * 2 / 16);
    append_bf16_kernel<D><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const int32_t* block_table, const int32_t* context_lens, int num_seqs, int n_new,
                          int max_blocks_per_seq, int num_blocks, int num_kv_heads, int head_dim, bool fp8,
                          float* k_scale, float* v_scale, unsigned* err, cudaStream_t stream) {
  AppendParams p;
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.k_cache = static_cast<uint8_t*>(k_cache);
  p.v_cache = static_cast<uint8_t*>(v_cache);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.err = err;
  p.num_seqs = num_seqs;
  p.n_new = n_new;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.num_kv_heads = num_kv_heads;
  if (head_dim == 128) return launch_d<128>(p, fp8, stream);
  if (head_dim == 64) return launch_d<64>(p, fp8, stream);
  return cudaErrorInvalidConfiguration;
}

}  // namespace pa
