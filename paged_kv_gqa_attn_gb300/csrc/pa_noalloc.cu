// paged_attn_decode_static_scratch: decode that allocates nothing.
//
// Some callers cannot allocate device memory while they serve: a host framework whose memory
// manager reserved the GPU's memory up front and hands out no more, or a real-time loop whose
// rules forbid allocation after start-up.  The ordinary entry point takes its split-KV scratch
// from a stream-ordered pool; this variant keeps the partials in a fixed array that lives in the
// library's device image instead, so a call makes no allocation of any kind.
//
// The array below is a file-scope __device__ variable: every GPU that loads this library holds
// kStaticScratchBytes for it until the process exits.  In host code its name is only a host-side
// stand-in, not a device address, so the kernels are given the address that
// cudaGetSymbolAddress returns, looked up once per device (with that device current) on the
// first call made on it.  Make that first call before capturing any stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "paged_attn.h"
#include "pa_kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = 32u << 20;  // 32 MiB of split-KV partials per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct StaticScratchDevice {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_static_scratch
  unsigned* err = nullptr;           // device address of the library's error word
  int num_sms = 0;
};
StaticScratchDevice g_devices[kMaxDevices];
std::mutex g_mu;

// Once per device, with that device current: resolve the array's device address.
int static_scratch_device(StaticScratchDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  StaticScratchDevice& d = g_devices[dev];
  if (!d.ready) {
    // A failed look-up returns PA_ERR_CUDA with the runtime's last error cleared, so the next
    // launch check of this or any other call does not report it again.
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    unsigned* err = nullptr;
    if (pa::error_word_address(&err) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    d.scratch = static_cast<unsigned char*>(ptr);
    d.err = err;
    d.num_sms = sms;
    d.ready = true;
  }
  *out = &d;
  return PA_OK;
}

}  // namespace

extern "C" size_t paged_attn_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" int paged_attn_decode_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* block_table, const int32_t* context_lens,
                                                int num_seqs, int max_blocks_per_seq, int num_blocks,
                                                int max_context_len, int q_len, int num_q_heads, int num_kv_heads,
                                                int head_dim, int block_size, float scale, int kv_dtype,
                                                const float* k_scale, const float* v_scale, void* out,
                                                void* stream) {
  int st = pa::validate_decode_args(q, k_cache, v_cache, block_table, context_lens, num_seqs, max_blocks_per_seq,
                                    num_blocks, max_context_len, q_len, num_q_heads, num_kv_heads, head_dim,
                                    block_size, kv_dtype, k_scale, v_scale, out);
  if (st != PA_OK) return st;
  const int group = num_q_heads / num_kv_heads;  // the CUDA-core kernel's groups
  if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  StaticScratchDevice* dev = nullptr;
  st = static_scratch_device(&dev);
  if (st != PA_OK) return st;

  int ppp = 0, nparts = 0;
  st = paged_attn_plan(dev->num_sms, num_seqs, num_kv_heads, max_context_len, block_size, q_len, kv_dtype, &ppp,
                       &nparts);
  if (st != PA_OK) return st;

  pa::AttnParams p = {};
  if (nparts > 1) {
    // partial outputs [B, q_len, Hq, P, d] then log2-sum-exps [B, q_len, Hq, P], all fp32.  Nothing
    // needs clearing: the merge reads only partitions that this call's decode kernel wrote.
    const size_t rows = (size_t)num_seqs * q_len * num_q_heads * nparts;
    const size_t bytes = rows * head_dim * sizeof(float) + rows * sizeof(float);
    if (bytes > kStaticScratchBytes) return PA_ERR_SCRATCH_LIMIT;
    p.part_o = reinterpret_cast<float*>(dev->scratch);
    p.part_lse = p.part_o + rows * head_dim;
  }
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.err = dev->err;
  p.num_seqs = num_seqs;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.q_len = q_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.pages_per_partition = ppp;
  p.max_partitions = nparts;
  p.max_context_len = max_context_len;
  p.scale_log2 = scale * pa::kLog2e;

  pa::Launch l;
  l.head_dim = head_dim;
  l.group = num_q_heads / num_kv_heads;
  l.fp8 = kv_dtype == PA_KV_FP8_E4M3;
  l.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = pa::launch_decode(p, l);
  if (e == cudaSuccess && nparts > 1) e = pa::launch_merge(p, l);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
