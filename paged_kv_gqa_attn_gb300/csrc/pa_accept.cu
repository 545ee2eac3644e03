// Speculative acceptance: the step after verify that turns the target's distributions into the
// tokens a round emits.
//
// Speculative sampling (studybook fde-roadmap ch.10, section 10.6.2; aegloslab servingai 5.3.10;
// sirzzang "Speculative Decoding", verification): draft token x_i (drawn from q_i) is accepted
// when p_i(x_i) >= q_i(x_i), else with probability p_i(x_i) / q_i(x_i); the first rejection
// ends the round with a token drawn from norm(max(0, p_i - q_i)); a round that accepts all K
// drafts adds a bonus token drawn from p_{K+1}.
//
// The uniforms are inputs: u_accept[b][i] in [0, 1) (accept iff p >= q or u < p / q, an IEEE
// fp32 division) and one 32-bit word per sequence for the draw.  A draw from weights r is the
// inverse CDF in 2^-40 fixed point: w(x) = floor(min(r, 1) * 2^40), Z = sum w,
// T = floor(Z * word / 2^32), token = first x whose inclusive prefix of w exceeds T.  The sums
// are integers, so the token does not depend on how the vocabulary is split across threads.
//
// Two kernels.  scan: grid (vocabulary chunk, sequence); every CTA finds the first rejection
// (one warp, a lane per draft) and sums the weights of its 4096-entry chunk of the row the draw
// uses (the residual, or p_{K+1}).  pick (programmatic dependent, one CTA per sequence): prefix
// of the chunk sums, the chunk holding T, a rescan of that chunk (from L2) for the token, and the
// outputs.  Only one vocabulary row (two for a residual) is read per sequence.
#include "pa_kernels.h"

namespace pa {
namespace {

constexpr int kChunk = 4096;                  // vocabulary entries per scan CTA
constexpr int kThreads = 256;
constexpr int kPer = kChunk / kThreads;       // 16 entries per thread
constexpr int kMaxChunks = 2 * kThreads;      // vocabularies up to 2^21 entries
constexpr float kFix = 1099511627776.0f;      // 2^40

struct AcceptParams {
  const float* p;          // [B, K+1, V] target probabilities
  const float* q;          // [B, K, V]   draft probabilities
  const int32_t* draft;    // [B, K]
  const float* u_accept;   // [B, K]
  const uint32_t* words;   // [B]
  int32_t* out_tokens;     // [B, K+1]
  int32_t* num_accepted;   // [B]
  unsigned long long* chunk_sums;  // [B, nchunks]
  unsigned* err;
  int num_seqs, K, V, nchunks;
};

__device__ __forceinline__ unsigned long long fixed_weight(float r) {
  r = fminf(fmaxf(r, 0.f), 1.f);  // exact; r * 2^40 is exact and the conversion truncates (= floor)
  return static_cast<unsigned long long>(r * kFix);
}

// The 16 entries a thread handles, as indices into the row, in four contiguous quads.
//  scan layout: quad j of thread t starts at c * kChunk + j * (4 * kThreads) + 4 t (coalesced);
//  run layout:  entries c * kChunk + 16 t + k (a thread's entries are consecutive, as a prefix
//               over threads in thread order needs).
__device__ __forceinline__ int scan_index(int c, int k) {
  return c * kChunk + (k >> 2) * (4 * kThreads) + 4 * (int)threadIdx.x + (k & 3);
}
__device__ __forceinline__ int run_index(int c, int k) { return c * kChunk + kPer * (int)threadIdx.x + k; }

// Load the 16 entries idx[] of a row with every load issued up front: indices past the row are
// clamped to a valid address (their weight is masked later).  kVec: 16-byte loads of the quads
// (needs 16-byte aligned rows, i.e. V % 4 == 0 and an aligned base).
template <bool kVec>
__device__ __forceinline__ void load16(const float* __restrict__ row, int V, const int (&idx)[kPer],
                                       float (&v)[kPer]) {
  if constexpr (kVec) {
#pragma unroll
    for (int j = 0; j < kPer / 4; ++j) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(row + min(idx[4 * j], V - 4)));
      v[4 * j] = f.x;
      v[4 * j + 1] = f.y;
      v[4 * j + 2] = f.z;
      v[4 * j + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPer; ++k) v[k] = __ldg(row + min(idx[k], V - 1));
  }
}

// Fixed-point weights of the 16 entries: the residual max(0, p - q) (one fp32 subtraction), or p
// when qr is null; 0 past the row.
template <bool kVec>
__device__ __forceinline__ void weights16(const float* pr, const float* qr, int V, const int (&idx)[kPer],
                                          unsigned long long (&w)[kPer]) {
  float pv[kPer];
  load16<kVec>(pr, V, idx, pv);
  if (qr) {
    float qv[kPer];
    load16<kVec>(qr, V, idx, qv);
#pragma unroll
    for (int k = 0; k < kPer; ++k) w[k] = idx[k] < V ? fixed_weight(pv[k] - qv[k]) : 0ull;
  } else {
#pragma unroll
    for (int k = 0; k < kPer; ++k) w[k] = idx[k] < V ? fixed_weight(pv[k]) : 0ull;
  }
}

// First rejected draft (K if all are accepted), or -1 if a draft token is outside [0, V).
// Called by one whole warp; lane i tests draft i.
__device__ int first_rejection(const AcceptParams& a, int b) {
  const int lane = threadIdx.x & 31;
  bool rej = false, bad = false;
  if (lane < a.K) {
    const int x = a.draft[(size_t)b * a.K + lane];
    if (x < 0 || x >= a.V) {
      bad = true;
    } else {
      const float pv = a.p[((size_t)b * (a.K + 1) + lane) * a.V + x];
      const float qv = a.q[((size_t)b * a.K + lane) * a.V + x];
      const float u = a.u_accept[(size_t)b * a.K + lane];
      rej = !(pv >= qv || u < __fdiv_rn(pv, qv));
    }
  }
  if (__any_sync(0xffffffffu, bad)) return -1;
  const unsigned m = __ballot_sync(0xffffffffu, rej);
  return m ? __ffs(m) - 1 : a.K;
}

struct DrawRow {
  const float* pr;
  const float* qr;  // null: the weights are p itself
};

__device__ __forceinline__ DrawRow draw_row(const AcceptParams& a, int b, int i) {
  if (i < a.K) return {a.p + ((size_t)b * (a.K + 1) + i) * a.V, a.q + ((size_t)b * a.K + i) * a.V};
  return {a.p + ((size_t)b * (a.K + 1) + a.K) * a.V, nullptr};
}

__device__ __forceinline__ unsigned long long shfl_up_u64(unsigned long long v, int d) {
  const unsigned lo = __shfl_up_sync(0xffffffffu, (unsigned)v, d);
  const unsigned hi = __shfl_up_sync(0xffffffffu, (unsigned)(v >> 32), d);
  return ((unsigned long long)hi << 32) | lo;
}

// Exclusive prefix of v over the CTA's threads (thread order); *total gets the sum.  All threads.
__device__ unsigned long long block_exclusive_scan(unsigned long long v, unsigned long long* total) {
  __shared__ unsigned long long warp_tot[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long o = shfl_up_u64(inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  unsigned long long before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const unsigned long long t = warp_tot[w];
    if (w < warp) before += t;
    all += t;
  }
  __syncthreads();  // warp_tot may be reused by the next call
  *total = all;
  return before + inc - v;
}

__device__ unsigned long long block_sum(unsigned long long v) {
  unsigned long long total;
  block_exclusive_scan(v, &total);
  return total;
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads) accept_scan_kernel(const AcceptParams a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int s_rej;
  const int c = blockIdx.x, b = blockIdx.y;
  if (threadIdx.x < 32) {
    const int r = first_rejection(a, b);
    if (threadIdx.x == 0) s_rej = r;
  }
  __syncthreads();
  const int rej = s_rej;
  if (rej < 0) return;  // the pick kernel reports it
  const DrawRow row = draw_row(a, b, rej);
  int idx[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) idx[k] = scan_index(c, k);
  unsigned long long w[kPer];
  weights16<kVec>(row.pr, row.qr, a.V, idx, w);
  unsigned long long sum = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) sum += w[k];
  sum = block_sum(sum);
  if (threadIdx.x == 0) a.chunk_sums[(size_t)b * a.nchunks + c] = sum;
}

// Token at offset t (0 <= t < chunk weight) inside chunk c: thread-contiguous 16-entry runs,
// a CTA scan of the run sums, then a walk of the one run that crosses t.
template <bool kVec>
__device__ int find_in_chunk(const DrawRow& row, int V, int c, unsigned long long t) {
  __shared__ int s_tok;
  int idx[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) idx[k] = run_index(c, k);
  unsigned long long w[kPer];
  weights16<kVec>(row.pr, row.qr, V, idx, w);
  unsigned long long run = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) run += w[k];
  if (threadIdx.x == 0) s_tok = -1;
  unsigned long long total;
  const unsigned long long before = block_exclusive_scan(run, &total);  // has a barrier after s_tok's init
  if (before <= t && t < before + run) {
    unsigned long long acc = before;
    int tok = -1;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      acc += w[k];
      if (tok < 0 && acc > t) tok = idx[k];
    }
    s_tok = tok;
  }
  __syncthreads();
  return s_tok;
}

// Chunk holding offset T given per-thread pairs of chunk sums; returns the chunk and the offset
// inside it through shared memory.
__device__ int find_chunk(const unsigned long long* sums, int nchunks, unsigned long long T,
                          unsigned long long* t_in_chunk) {
  __shared__ int s_c;
  __shared__ unsigned long long s_t;
  const int c0 = threadIdx.x * 2;
  const unsigned long long a0 = c0 < nchunks ? sums[c0] : 0ull;
  const unsigned long long a1 = c0 + 1 < nchunks ? sums[c0 + 1] : 0ull;
  if (threadIdx.x == 0) s_c = -1;
  unsigned long long total;
  const unsigned long long before = block_exclusive_scan(a0 + a1, &total);
  if (before <= T && T < before + a0) {
    s_c = c0;
    s_t = T - before;
  } else if (before + a0 <= T && T < before + a0 + a1) {
    s_c = c0 + 1;
    s_t = T - before - a0;
  }
  __syncthreads();
  *t_in_chunk = s_t;
  return s_c;
}

template <bool kVec>
__global__ void __launch_bounds__(kThreads) accept_pick_kernel(const AcceptParams a) {
  __shared__ int s_rej;
  __shared__ unsigned long long s_sums[kMaxChunks];
  const int b = blockIdx.x;
  // the decision reads only inputs: it overlaps the tail of the scan kernel
  if (threadIdx.x < 32) {
    const int r = first_rejection(a, b);
    if (threadIdx.x == 0) s_rej = r;
  }
  __syncthreads();
  const int rej = s_rej;
  int32_t* out = a.out_tokens + (size_t)b * (a.K + 1);
  if (rej < 0) {
    for (int i = threadIdx.x; i <= a.K; i += blockDim.x) out[i] = -1;
    if (threadIdx.x == 0) {
      a.num_accepted[b] = -1;
      record_error(a.err, kErrBadInput);
    }
    return;
  }
  DrawRow row = draw_row(a, b, rej);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int c = threadIdx.x; c < a.nchunks; c += blockDim.x) s_sums[c] = a.chunk_sums[(size_t)b * a.nchunks + c];
  __syncthreads();
  unsigned long long Z = 0;
  {
    unsigned long long part = 0;
    for (int c = threadIdx.x; c < a.nchunks; c += blockDim.x) part += s_sums[c];
    Z = block_sum(part);
  }
  if (Z == 0 && row.qr) {
    // the residual has no mass (possible only through rounding of the inputs): draw from p_i
    row.qr = nullptr;
    for (int c = 0; c < a.nchunks; ++c) {
      int idx[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) idx[k] = scan_index(c, k);
      unsigned long long w[kPer];
      weights16<kVec>(row.pr, nullptr, a.V, idx, w);
      unsigned long long part = 0;
#pragma unroll
      for (int k = 0; k < kPer; ++k) part += w[k];
      part = block_sum(part);
      if (threadIdx.x == 0) s_sums[c] = part;
    }
    __syncthreads();
    unsigned long long part = 0;
    for (int c = threadIdx.x; c < a.nchunks; c += blockDim.x) part += s_sums[c];
    Z = block_sum(part);
  }
  int tok = -1;
  if (Z > 0) {
    const unsigned long long T = __umul64hi(Z, (unsigned long long)a.words[b] << 32);
    unsigned long long t = 0;
    const int c = find_chunk(s_sums, a.nchunks, T, &t);
    tok = find_in_chunk<kVec>(row, a.V, c, t);
  } else if (threadIdx.x == 0) {
    record_error(a.err, kErrBadInput);
  }
  for (int i = threadIdx.x; i <= a.K; i += blockDim.x) {
    out[i] = i < rej ? a.draft[(size_t)b * a.K + i] : (i == rej ? tok : -1);
  }
  if (threadIdx.x == 0) a.num_accepted[b] = rej;
}

}  // namespace

size_t accept_scratch_bytes(int num_seqs, int vocab) {
  const size_t nchunks = ((size_t)vocab + kChunk - 1) / kChunk;
  return (size_t)num_seqs * nchunks * sizeof(unsigned long long);
}

cudaError_t launch_accept(const float* p, const float* q, const int32_t* draft, const float* u_accept,
                          const uint32_t* words, int num_seqs, int num_draft, int vocab, int32_t* out_tokens,
                          int32_t* num_accepted, void* scratch, unsigned* err, cudaStream_t stream) {
  AcceptParams a;
  a.p = p;
  a.q = q;
  a.draft = draft;
  a.u_accept = u_accept;
  a.words = words;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.chunk_sums = static_cast<unsigned long long*>(scratch);
  a.err = err;
  a.num_seqs = num_seqs;
  a.K = num_draft;
  a.V = vocab;
  a.nchunks = (vocab + kChunk - 1) / kChunk;
  if (a.nchunks > kMaxChunks) return cudaErrorInvalidConfiguration;
  // 16-byte loads when every row starts 16-byte aligned
  const bool vec = vocab % 4 == 0 && reinterpret_cast<uintptr_t>(p) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(q) % 16 == 0;
  const void* scan = vec ? reinterpret_cast<const void*>(accept_scan_kernel<true>)
                         : reinterpret_cast<const void*>(accept_scan_kernel<false>);
  const void* pick = vec ? reinterpret_cast<const void*>(accept_pick_kernel<true>)
                         : reinterpret_cast<const void*>(accept_pick_kernel<false>);
  void* args[] = {&a};
  cudaError_t e = cudaLaunchKernel(scan, dim3(a.nchunks, num_seqs), dim3(kThreads), args, 0, stream);
  if (e != cudaSuccess) return e;
  return launch_pdl(pick, dim3(num_seqs), dim3(kThreads), 0, stream, args);
}

}  // namespace pa
