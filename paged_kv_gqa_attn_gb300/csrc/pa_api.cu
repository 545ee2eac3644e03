// C ABI of the paged-attention library: argument checks, split-KV planning, scratch, launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "paged_attn.h"
#include "pa_kernels.h"

// Per-device error word written by the kernels (see pa::kErr*).
__device__ unsigned int g_pa_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxForcedPartitions = 4096;
constexpr int kAutoMaxPartitions = 64;
constexpr int kAutoPagesCap = 64;      // longest partition the automatic plan aims for (bf16)
// E4M3: 256 pages (1 MiB of K and V per CTA); long_fp8 (4 x 131072 tokens): 32 partitions of 256
// pages 167.6 us, 64 of 128 173.9 us, 48 of 171 174.4 us, 38 of 216 181.8 us, 19 of 432 174.6 us
constexpr int kAutoPagesCapE4M3 = 256;
// CTAs per SM the automatic plan aims for: a few waves of the 3 resident bf16 decode CTAs per SM;
// E4M3 CTAs stream half the bytes per page, so their fixed start and epilogue weigh twice as much
// and fewer, longer partitions win (llama8b_decode shape with E4M3: 2 partitions 50.0 us, 3 51.3,
// 4 51.5, 8 57.0; bf16: 3 partitions 85.1 us, 2 86.6, 4 85.6).
constexpr int kCtasPerSmTarget = 8;
constexpr int kCtasPerSmTargetE4M3 = 4;

std::atomic<int> g_forced_partitions{0};

struct DeviceState {
  bool ready = false;
  unsigned* err = nullptr;
  int num_sms = 0;
  cudaMemPool_t pool = nullptr;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_pa_error_word) != cudaSuccess) return PA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PA_ERR_CUDA;
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return PA_ERR_CUDA;
    uint64_t keep = UINT64_MAX;  // keep freed scratch cached in this library's pool
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    s.err = static_cast<unsigned*>(ptr);
    s.num_sms = sms;
    s.pool = pool;
    s.ready = true;
  }
  *out = &s;
  return PA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link needed).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// The pool [NB * Hkv * bs, d] bf16 as a 2-D TMA map with 16-token x 64-dim boxes, 128-B swizzle.
int encode_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int num_kv_heads, int block_size,
                    int head_dim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)num_blocks * num_kv_heads * block_size};
  cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)block_size};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// The E4M3 pool [NB * Hkv * bs, d] bytes as a 2-D TMA map with one 16 x d box per page, swizzled by
// its row width (128 B rows: 128-byte swizzle; 64 B rows: 64-byte swizzle).
int encode_e4m3_pool_map(CUtensorMap* map, const void* pool, int num_blocks, int num_kv_heads, int block_size,
                         int head_dim) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)num_blocks * num_kv_heads * block_size};
  cuuint64_t strides[1] = {(cuuint64_t)head_dim};
  cuuint32_t box[2] = {(cuuint32_t)head_dim, (cuuint32_t)block_size};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

enum class Form { kDecode, kVerify };

int validate(Form form, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
             const int32_t* context_lens, int num_seqs, int max_blocks_per_seq, int num_blocks,
             int max_context_len, int q_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
             int kv_dtype, const float* k_scale, const float* v_scale, const void* out) {
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || max_blocks_per_seq < 1 || num_blocks < 1 || max_context_len < 0) return PA_ERR_INVALID_ARG;
  if (num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || q_len < 1) return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  if (kv_dtype == PA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size) return PA_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
    return PA_ERR_INVALID_ARG;
  if (block_size != 16 || (head_dim != 64 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  // TMA row coordinates are signed 32-bit
  if ((int64_t)num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (form == Form::kDecode) {
    if (q_len != 1) return PA_ERR_INVALID_ARG;
    if (group > 64) return PA_ERR_UNSUPPORTED;  // other groups take the verify kernel's 64 rows
  } else {
    if (q_len > 16) return PA_ERR_INVALID_ARG;
    // up to 64 rows per kv head: the verify kernel; 65-128: the split prefill kernel
    if (group * q_len > 128) return PA_ERR_UNSUPPORTED;
  }
  return PA_OK;
}

int run(Form form, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
        const int32_t* context_lens, const uint32_t* tree_mask, int num_seqs, int max_blocks_per_seq,
        int num_blocks, int max_context_len, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
        int block_size, float scale, int kv_dtype, const float* k_scale, const float* v_scale, void* out,
        void* stream) {
  int st = validate(form, q, k_cache, v_cache, block_table, context_lens, num_seqs, max_blocks_per_seq,
                    num_blocks, max_context_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                    kv_dtype, k_scale, v_scale, out);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return PA_OK;
  DeviceState* dev = nullptr;
  st = device_state(&dev);
  if (st != PA_OK) return st;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  pa::AttnParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.tree_mask = tree_mask;
  p.err = dev->err;
  p.num_seqs = num_seqs;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.q_len = q_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.max_context_len = max_context_len;
  p.scale_log2 = scale * pa::kLog2e;

  pa::Launch l;
  l.head_dim = head_dim;
  l.group = num_q_heads / num_kv_heads;
  l.fp8 = kv_dtype == PA_KV_FP8_E4M3;
  l.stream = s;

  cudaError_t e;
  void* scratch = nullptr;
  // Decode runs the warp-level mma.sync kernel (split-KV partitions + merge) for groups of 1, 2, 4
  // and 8 query heads; verify, and decode with any other group (up to 64: 3, 5, 7, 16 ...), the
  // tcgen05 kernel (balanced persistent split + merge), decode as its q_len = 1 rows.
  // Verify with more than the verify kernel's 64 rows per kv head (bf16, up to 128) runs the
  // chunked-prefill kernel split into partitions like decode, with the same merge.
  const bool mma_group = l.group == 1 || l.group == 2 || l.group == 4 || l.group == 8;
  const bool wide_verify = form == Form::kVerify && l.group * q_len > 64;
  const bool on_tensor_cores = (form == Form::kVerify && !wide_verify) || (form == Form::kDecode && !mma_group);
  if (on_tensor_cores) {
    // balanced persistent split: planner, tcgen05 kernel, segment merge
    const int ncta = pa::verify_resident_ctas(dev->num_sms);
    const size_t bytes = pa::verify_scratch_bytes(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim, ncta);
    if (cudaMallocFromPoolAsync(&scratch, bytes, dev->pool, s) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_NO_MEMORY;
    }
    // bf16 pages move as 2-D tensor boxes; E4M3 V pages as plain bulk copies, and E4M3 K pages
    // as 2-D boxes in the swizzled layout the E4M3 products read (head_dim 128) or as bulk copies
    CUtensorMap tk = {}, tv = {};
    int r1 = PA_OK, r2 = PA_OK;
    if (!l.fp8) {
      r1 = encode_pool_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
      r2 = encode_pool_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim);
    } else if (head_dim == 128) {
      r1 = encode_e4m3_pool_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
    }
    e = (r1 == PA_OK && r2 == PA_OK) ? pa::launch_verify_tc(p, l, scratch, ncta, tk, tv) : cudaErrorInvalidValue;
  } else {
    int ppp = 0, nparts = 0;
    st = paged_attn_plan(dev->num_sms, num_seqs, num_kv_heads, max_context_len, block_size, q_len, kv_dtype, &ppp,
                         &nparts);
    if (st != PA_OK) return st;
    if (wide_verify && ppp % 4 != 0) {  // the prefill kernel walks whole 64-token steps
      const int pages = (max_context_len + block_size - 1) / block_size;
      ppp = (ppp + 3) / 4 * 4;
      nparts = pages > 0 ? (pages + ppp - 1) / ppp : 1;
    }
    p.pages_per_partition = ppp;
    p.max_partitions = nparts;
    if (nparts > 1) {
      const size_t rows = (size_t)num_seqs * q_len * num_q_heads * nparts;
      const size_t bytes = rows * head_dim * sizeof(float) + rows * sizeof(float);
      if (cudaMallocFromPoolAsync(&scratch, bytes, dev->pool, s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_NO_MEMORY;
      }
      p.part_o = static_cast<float*>(scratch);
      p.part_lse = p.part_o + rows * head_dim;
    }
    // 2-D TMA maps of the pools (bf16: 16 x 64-dim boxes; E4M3: one 16 x d box per page)
    CUtensorMap tk = {}, tv = {};
    const int r1 = l.fp8 ? encode_e4m3_pool_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim)
                         : encode_pool_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim);
    const int r2 = l.fp8 ? encode_e4m3_pool_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim)
                         : encode_pool_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim);
    if (r1 != PA_OK || r2 != PA_OK)
      e = cudaErrorInvalidValue;
    else
      e = wide_verify ? pa::launch_verify_split(p, l, tk, tv) : pa::launch_decode_mma(p, l, tk, tv);
    if (e == cudaSuccess && nparts > 1) e = pa::launch_merge(p, l);
  }
  if (scratch) cudaFreeAsync(scratch, s);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

namespace pa {

cudaError_t set_smem_once(const void* kernel, int bytes) {
  struct Entry {
    const void* kernel;
    int device;
  };
  static Entry done[512];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < n; ++i)
    if (done[i].kernel == kernel && done[i].device == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n < 512) done[n++] = {kernel, dev};
  return e;
}

int validate_decode_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                         const int32_t* context_lens, int num_seqs, int max_blocks_per_seq, int num_blocks,
                         int max_context_len, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int kv_dtype, const float* k_scale, const float* v_scale,
                         const void* out) {
  return validate(Form::kDecode, q, k_cache, v_cache, block_table, context_lens, num_seqs, max_blocks_per_seq,
                  num_blocks, max_context_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype,
                  k_scale, v_scale, out);
}

// Launch `fn` so that it may start while the previous kernel on `st` finishes (programmatic
// dependent launch); the kernel calls griddepcontrol.wait before it reads that kernel's output.
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, int smem, cudaStream_t st, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t error_word_address(unsigned** out) {
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_pa_error_word);
  if (e == cudaSuccess) *out = static_cast<unsigned*>(ptr);
  return e;
}

}  // namespace pa

extern "C" {

int paged_attn_plan(int num_sms, int num_seqs, int num_kv_heads, int max_context_len, int block_size, int q_len,
                    int kv_dtype, int* pages_per_partition, int* max_partitions) {
  (void)q_len;
  if (!pages_per_partition || !max_partitions || num_sms < 1 || num_seqs < 0 || num_kv_heads < 1 ||
      max_context_len < 0 || block_size < 1)
    return PA_ERR_INVALID_ARG;
  const int64_t max_pages = ((int64_t)max_context_len + block_size - 1) / block_size;
  const int64_t pages = max_pages > 0 ? max_pages : 1;
  int64_t P;
  const int forced = g_forced_partitions.load();
  if (forced > 0) {
    P = forced < pages ? forced : pages;
    const int64_t ppp = (pages + P - 1) / P;
    *pages_per_partition = (int)ppp;
    *max_partitions = (int)((pages + ppp - 1) / ppp);
    return PA_OK;
  }
  const int64_t units = (int64_t)(num_seqs > 0 ? num_seqs : 1) * num_kv_heads;
  const int64_t target = (int64_t)(kv_dtype == PA_KV_FP8_E4M3 ? kCtasPerSmTargetE4M3 : kCtasPerSmTarget) * num_sms;
  P = (target + units - 1) / units;
  // E4M3: when one partition per (sequence, kv head) already fills 80 % of the target, splitting
  // costs more (a merge, twice the fixed start and end per CTA) than the idle slots it fills
  // (llama8b-shaped decode 48.2 -> 46.8 us, groups of 8 52.9 -> 48.9 us)
  if (kv_dtype == PA_KV_FP8_E4M3 && units * 5 >= target * 4) P = 1;
  const int64_t cap = kv_dtype == PA_KV_FP8_E4M3 ? kAutoPagesCapE4M3 : kAutoPagesCap;
  const int64_t by_cap = (pages + cap - 1) / cap;
  if (by_cap > P) P = by_cap;
  if (P > kAutoMaxPartitions) P = kAutoMaxPartitions;
  if (P > pages) P = pages;
  if (P < 1) P = 1;
  int64_t ppp = (pages + P - 1) / P;
  ppp = (ppp + 3) / 4 * 4;
  *pages_per_partition = (int)ppp;
  *max_partitions = (int)((pages + ppp - 1) / ppp);
  return PA_OK;
}

int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                      const int32_t* context_lens, int num_seqs, int max_blocks_per_seq, int num_blocks,
                      int max_context_len, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, float scale, int kv_dtype, const float* k_scale, const float* v_scale,
                      void* out, void* stream) {
  return run(Form::kDecode, q, k_cache, v_cache, block_table, context_lens, nullptr, num_seqs, max_blocks_per_seq,
             num_blocks, max_context_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size, scale, kv_dtype,
             k_scale, v_scale, out, stream);
}

int paged_attn_verify(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                      const int32_t* context_lens, int num_seqs, int max_blocks_per_seq, int num_blocks,
                      int max_context_len, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, float scale, int kv_dtype, const float* k_scale, const float* v_scale,
                      void* out, void* stream) {
  return run(Form::kVerify, q, k_cache, v_cache, block_table, context_lens, nullptr, num_seqs, max_blocks_per_seq,
             num_blocks, max_context_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size, scale, kv_dtype,
             k_scale, v_scale, out, stream);
}

int paged_attn_tree_verify(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                           const int32_t* context_lens, const uint32_t* tree_mask, int num_seqs,
                           int max_blocks_per_seq, int num_blocks, int max_context_len, int q_len, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, float scale, int kv_dtype,
                           const float* k_scale, const float* v_scale, void* out, void* stream) {
  if (!tree_mask) return PA_ERR_INVALID_ARG;
  return run(Form::kVerify, q, k_cache, v_cache, block_table, context_lens, tree_mask, num_seqs,
             max_blocks_per_seq, num_blocks, max_context_len, q_len, num_q_heads, num_kv_heads, head_dim, block_size,
             scale, kv_dtype, k_scale, v_scale, out, stream);
}

int paged_attn_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* context_lens, const int32_t* query_start_loc, int num_seqs, int total_q,
                       int max_q_len, int max_blocks_per_seq, int num_blocks, int max_context_len, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, float scale, int kv_dtype,
                       const float* k_scale, const float* v_scale, void* out, void* stream) {
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !query_start_loc || !out)
    return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
      max_context_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || block_size < 1) return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  if (kv_dtype == PA_KV_FP8_E4M3 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * block_size) return PA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) % 16 != 0) return PA_ERR_INVALID_ARG;
  // bf16 pages move as 2-D tensor boxes, E4M3 pages as 16-byte-aligned bulk copies
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return PA_ERR_INVALID_ARG;
  const int group = num_q_heads / num_kv_heads;
  if (block_size != 16 || (head_dim != 64 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
  if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_seqs * num_kv_heads > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (((int64_t)max_q_len + 128 / group - 1) / (128 / group) > 65535) return PA_ERR_UNSUPPORTED;  // tile < 2^16
  if ((int64_t)num_seqs * ((max_q_len + 128 / group - 1) / (128 / group)) * num_kv_heads > 0x7fffffffLL)
    return PA_ERR_UNSUPPORTED;  // one CTA per (tile, kv head)
  // TMA row coordinates are signed 32-bit
  if ((int64_t)num_blocks * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return PA_OK;
  DeviceState* dev = nullptr;
  int st = device_state(&dev);
  if (st != PA_OK) return st;
  pa::AttnParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.query_start_loc = query_start_loc;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.err = dev->err;
  p.num_seqs = num_seqs;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.q_len = max_q_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.max_context_len = max_context_len;
  p.total_q = total_q;
  p.scale_log2 = scale * pa::kLog2e;
  pa::Launch l;
  l.head_dim = head_dim;
  l.group = group;
  l.fp8 = kv_dtype == PA_KV_FP8_E4M3;
  l.stream = static_cast<cudaStream_t>(stream);
  // bf16: 2-D TMA maps of the pools; E4M3: K pages as 2-D boxes in the swizzled layout the E4M3
  // products read (head_dim 128), V pages (and head_dim 64 K pages) as bulk copies
  CUtensorMap tk = {}, tv = {};
  if (!l.fp8 && (encode_pool_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim) != PA_OK ||
                 encode_pool_map(&tv, v_cache, num_blocks, num_kv_heads, block_size, head_dim) != PA_OK))
    return PA_ERR_CUDA;
  if (l.fp8 && head_dim == 128 &&
      encode_e4m3_pool_map(&tk, k_cache, num_blocks, num_kv_heads, block_size, head_dim) != PA_OK)
    return PA_ERR_CUDA;
  void* scratch = nullptr;
  if (cudaMallocFromPoolAsync(&scratch, pa::prefill_scratch_bytes(num_seqs, max_q_len, group), dev->pool, l.stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_NO_MEMORY;
  }
  const cudaError_t e = pa::launch_prefill_tc(p, l, max_q_len, scratch, tk, tv);
  cudaFreeAsync(scratch, l.stream);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int paged_attn_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int32_t* block_table, const int32_t* context_lens, int num_seqs, int n_new,
                         int max_blocks_per_seq, int num_blocks, int num_kv_heads, int head_dim, int block_size,
                         int kv_dtype, float* k_scale, float* v_scale, void* stream) {
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !context_lens) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || n_new < 0 || max_blocks_per_seq < 1 || num_blocks < 1 || num_kv_heads < 1 ||
      head_dim < 1 || block_size < 1)
    return PA_ERR_INVALID_ARG;
  if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3) return PA_ERR_INVALID_ARG;
  const bool fp8 = kv_dtype == PA_KV_FP8_E4M3;
  if (fp8 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  if ((int64_t)n_new > (int64_t)max_blocks_per_seq * block_size) return PA_ERR_INVALID_ARG;
  if (block_size != 16 || (head_dim != 64 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_seqs * n_new > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;  // one CTA per new token
  // rows are moved in 16-byte pieces
  const uintptr_t align = (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_cache | (uintptr_t)v_cache;
  if (align % 16 != 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || n_new == 0) return PA_OK;
  DeviceState* dev = nullptr;
  int st = device_state(&dev);
  if (st != PA_OK) return st;
  cudaError_t e = pa::launch_append(k_new, v_new, k_cache, v_cache, block_table, context_lens, num_seqs, n_new,
                                    max_blocks_per_seq, num_blocks, num_kv_heads, head_dim, fp8, k_scale, v_scale,
                                    dev->err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int paged_attn_spec_accept(const float* p, const float* q, const int32_t* draft_tokens, const float* u_accept,
                           const uint32_t* u_sample, int num_seqs, int num_draft, int vocab_size,
                           int32_t* out_tokens, int32_t* num_accepted, void* stream) {
  if (!p || !u_sample || !out_tokens || !num_accepted) return PA_ERR_INVALID_ARG;
  if (num_draft > 0 && (!q || !draft_tokens || !u_accept)) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_draft < 0 || vocab_size < 1) return PA_ERR_INVALID_ARG;
  if (num_draft > 31 || vocab_size > (1 << 21) || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  DeviceState* dev = nullptr;
  int st = device_state(&dev);
  if (st != PA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  if (cudaMallocFromPoolAsync(&scratch, pa::accept_scratch_bytes(num_seqs, vocab_size), dev->pool, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_NO_MEMORY;
  }
  cudaError_t e = pa::launch_accept(p, q, draft_tokens, u_accept, u_sample, num_seqs, num_draft, vocab_size,
                                    out_tokens, num_accepted, scratch, dev->err, s);
  cudaFreeAsync(scratch, s);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int paged_attn_check_device_errors(void* stream) {
  DeviceState* dev = nullptr;
  int st = device_state(&dev);
  if (st != PA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, dev->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemset(dev->err, 0, sizeof word) != cudaSuccess) return PA_ERR_CUDA;
  if (word & (pa::kErrBlockId | pa::kErrShortContext | pa::kErrBadInput)) return PA_ERR_DEVICE_BOUNDS;
  if (word & pa::kErrTimeout) return PA_ERR_DEVICE_TIMEOUT;
  return PA_OK;
}

const char* paged_attn_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case PA_ERR_CUDA: return "CUDA runtime or launch error";
    case PA_ERR_NO_MEMORY: return "split-KV scratch allocation failed";
    case PA_ERR_DEVICE_BOUNDS: return "device: index out of range, context shorter than q_len, or invalid device-side input";
    case PA_ERR_DEVICE_TIMEOUT: return "device: asynchronous copy wait timed out";
    case PA_ERR_SCRATCH_LIMIT: return "shape needs more split-KV scratch than the static array holds";
    default: return "unknown status";
  }
}

int paged_attn_set_max_partitions(int p) {
  if (p < 0 || p > kMaxForcedPartitions) return PA_ERR_INVALID_ARG;
  g_forced_partitions.store(p);
  return PA_OK;
}

int paged_attn_version(void) { return 100; }

}  // extern "C"
