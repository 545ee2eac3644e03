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

// Two floats -> two E4M3 codes (round to nearest even, saturate finite values at +-448).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// bf16: a scatter.  One CTA per new token (b, t) moves that token's K and V rows for every kv
// head, 16 bytes per thread; the source loads are issued before the dependent context-length
// and block-table loads so that both round trips overlap.
template <int D>
__global__ void __launch_bounds__(128) append_bf16_kernel(const AppendParams p) {
  constexpr int kC = D / 8;  // 16-byte pieces per head row
  constexpr int kPer = 4;    // pieces in flight per thread
  const int row = blockIdx.x;  // b * n_new + t
  const int b = row / p.n_new, t = row - b * p.n_new;
  const int per_side = p.num_kv_heads * kC;
  const int total = 2 * per_side;
  const uint4* ksrc = reinterpret_cast<const uint4*>(p.k_new) + (size_t)row * per_side;
  const uint4* vsrc = reinterpret_cast<const uint4*>(p.v_new) + (size_t)row * per_side;
  for (int base = 0; base < total; base += kPer * blockDim.x) {
    uint4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      if (i < total) v[k] = i < per_side ? ksrc[i] : vsrc[i - per_side];
    }
    const int L = p.context_lens[b];
    if (L < p.n_new || L > p.max_blocks_per_seq * 16) {  // shorter than the new rows, or past the table
      if (threadIdx.x == 0) record_error(p.err, kErrShortContext);
      return;
    }
    const int j = L - p.n_new + t;
    const int pb = p.block_table[(size_t)b * p.max_blocks_per_seq + j / 16];
    if (pb < 0 || pb >= p.num_blocks) {
      if (threadIdx.x == 0) record_error(p.err, kErrBlockId);
      return;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = base + k * blockDim.x + threadIdx.x;
      if (i < total) {
        const bool is_v = i >= per_side;
        const int r = is_v ? i - per_side : i;
        const int g = r / kC, c = r - g * kC;
        uint4* dst = reinterpret_cast<uint4*>(is_v ? p.v_cache : p.k_cache) +
                     (((size_t)pb * p.num_kv_heads + g) * 16 + (j & 15)) * kC + c;
        *dst = v[k];
      }
    }
  }
}

// E4M3 codes (16, in a uint4) -> floats, exactly (through f16).
__device__ __forceinline__ void e4m3x16_to_f32(const uint4 w, float* f) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t h2;
      const uint16_t pair = static_cast<uint16_t>(words[k] >> (16 * h));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
      f[4 * k + 2 * h] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
      f[4 * k + 2 * h + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
    }
  }
}

// fp8: one CTA per (kv head, sequence, K or V) walks the one or two blocks the new tokens land
// in.  Thread i owns bytes [16 i, 16 i + 16) of the (block, head) page: 16 codes of one token.
// The values stay in registers between the amax reduction and the encode.
template <int D>
__global__ void __launch_bounds__(128) append_fp8_kernel(const AppendParams p) {
  static_assert(16 * D / 16 <= 128, "one 16-byte piece per thread");
  constexpr int kPieces = D;  // 16 tokens x D bytes / 16
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
  const int i = threadIdx.x;
  const int sl = i * 16 / D, c0 = i * 16 - sl * D;  // token slot and first dim of this piece
  for (int blk = first / 16; blk <= (L - 1) / 16; ++blk) {
    const int pb = p.block_table[(size_t)b * p.max_blocks_per_seq + blk];
    if (pb < 0 || pb >= p.num_blocks) {
      if (threadIdx.x == 0) record_error(p.err, kErrBlockId);
      continue;
    }
    const int lo = blk * 16;
    const int s0 = max(first - lo, 0);  // slots [0, s0): older tokens
    const int s1 = min(L - lo, 16);     // slots [s0, s1): new tokens
    uint4* page = reinterpret_cast<uint4*>(cache + ((size_t)pb * p.num_kv_heads + g) * 16 * D);
    const float old_scale = scales[(size_t)pb * p.num_kv_heads + g];
    float f[16];
    float amax = 0.f;
    const bool mine = i < kPieces && sl < s1;
    if (mine) {
      if (sl < s0) {
        e4m3x16_to_f32(page[i], f);
#pragma unroll
        for (int k = 0; k < 16; ++k) f[k] *= old_scale;
      } else {
        const uint4* s4 = reinterpret_cast<const uint4*>(
            src + (((size_t)b * p.n_new + (lo + sl - first)) * p.num_kv_heads + g) * D + c0);
        const uint4 a = s4[0], c = s4[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          f[2 * k] = __uint_as_float(w[k] << 16);
          f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(f[k]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float new_scale = amax > 0.f ? amax / 448.f : 1.f;
    // older tokens are re-encoded only when the scale moved
    if (mine && (sl >= s0 || new_scale != old_scale)) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint16_t lo2 = f32x2_to_e4m3x2(f[4 * k] / new_scale, f[4 * k + 1] / new_scale);
        const uint16_t hi2 = f32x2_to_e4m3x2(f[4 * k + 2] / new_scale, f[4 * k + 3] / new_scale);
        w[k] = (uint32_t)lo2 | ((uint32_t)hi2 << 16);
      }
      page[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();  // every thread has read old_scale and red before they change
    if (threadIdx.x == 0) scales[(size_t)pb * p.num_kv_heads + g] = new_scale;
  }
}

template <int D>
cudaError_t launch_d(const AppendParams& p, bool fp8, cudaStream_t st) {
  if (fp8) {
    append_fp8_kernel<D><<<dim3(p.num_kv_heads, p.num_seqs, 2), 128, 0, st>>>(p);
  } else {
    append_bf16_kernel<D><<<(unsigned)(p.num_seqs * p.n_new), 128, 0, st>>>(p);
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
