// Paged GQA speculative-verify attention (q_len = K + 1 causal rows) on tensor cores, sm_103a.
//
// The verify forward scores the K draft tokens plus the bonus position in one pass, each row
// masked to the tokens up to itself (sirzzang "Speculative Decoding", parallel verification
// and its causal-mask figure).  With G query heads per kv head the G * q_len rows of one kv
// head share every K/V page, so scores and values form a real dense product:
// [rows x d] x [d x 64 tokens] and [rows x 64 tokens] x [64 tokens x d] per step.
//
// One CTA per (partition, kv head, sequence); one warp per 16-row slice of the rows.  Pages
// arrive through the TMA unit as 2-D tensor tiles of 16 tokens x 64 dims with the 128-byte
// swizzle, four pages (64 tokens) per pipeline stage, completion on an mbarrier.  Each warp
// keeps its rows' Q fragments in registers, runs S = Q K^T and O += P V with bf16 mma.sync
// (fp32 accumulate) from ldmatrix fragments, and an online softmax in base 2 between steps
// (studybook fde-roadmap ch.10, section 10.1.2).  Partials and the merge follow the decode
// kernel's split-KV scheme.
#include "pa_kernels.h"

namespace pa {
namespace {

template <int D, int MT>
struct VerifyTraits {
  static constexpr int kWarps = MT;
  static constexpr int kThreads = 32 * MT;
  static constexpr int kBS = 16;
  static constexpr int kTP = 4;                        // pages per step
  static constexpr int kStepTokens = kTP * kBS;        // 64
  static constexpr int kBoxCols = 64;                  // 64 bf16 = one 128-byte swizzle row
  static constexpr int kBoxes = D / kBoxCols;          // boxes per page
  static constexpr int kBoxBytes = kBS * 128;          // 2 KiB
  static constexpr int kPageBytes = kBoxes * kBoxBytes;
  static constexpr int kStageBytes = 2 * kTP * kPageBytes;  // K pages then V pages
  static constexpr int kStages = D == 128 ? 3 : 4;
  static constexpr int kKSteps = D / 16;               // k16 steps of S = Q K^T
  static constexpr int kOTiles = D / 8;                // n8 tiles of O
  static constexpr int kSTiles = kStepTokens / 8;      // n8 tiles of S per step (8)
  static constexpr int kSmem = kStages * kStageBytes + kStages * 8 + 1024;  // + alignment slack
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Shared-memory address of (token row t of page pg, dims [c*8, c*8+8)) in a K or V region of a
// stage, following the TMA 128-byte swizzle (16-byte chunk index XOR row % 8).
template <class T>
__device__ __forceinline__ uint32_t tile_addr(uint32_t region, int pg, int t, int dchunk) {
  const int box = dchunk >> 3;
  const int ch = dchunk & 7;
  return region + pg * T::kPageBytes + box * T::kBoxBytes + t * 128 + ((ch ^ (t & 7)) << 4);
}

template <int D, int MT>
__global__ void __launch_bounds__(32 * MT) verify_kernel(const AttnParams p,
                                                          const __grid_constant__ CUtensorMap tmk,
                                                          const __grid_constant__ CUtensorMap tmv) {
  using T = VerifyTraits<D, MT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar0 = base + T::kStages * T::kStageBytes;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int part = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int Hq = p.num_q_heads;
  const int G = Hq / p.num_kv_heads;
  const int QL = p.q_len;
  const int R = G * QL;
  const int L = context_len(p, b, part == 0 && g == 0 && threadIdx.x == 0);

  const int r0 = warp * 16 + (lane >> 2);  // this thread's two rows
  const int r1 = r0 + 8;
  const int npages = (L + T::kBS - 1) / T::kBS;
  const int ppp = p.pages_per_partition;
  const int pbeg = part * ppp;

  // rows that see no token (context shorter than q_len) come out as zeros; flag them
  if (L < QL && part == 0 && g == 0 && threadIdx.x == 0) record_error(p.err, kErrShortContext);
  if (L <= 0) {  // no page at all: zero the group's rows once
    if (part == 0) {
      for (int idx = threadIdx.x; idx < R * D; idx += T::kThreads) {
        const int r = idx / D, dd = idx - r * D;
        const int i = r / G, h = r - i * G;
        p.out[(((size_t)b * QL + i) * Hq + g * G + h) * D + dd] = __float2bfloat16(0.f);
      }
    }
    return;
  }
  if (pbeg >= npages) return;
  const int pend = min(npages, pbeg + ppp);
  const int nparts = (npages + ppp - 1) / ppp;
  const int limit_tok = min(L, pend * T::kBS);  // tokens of this partition end here
  const int nsteps = (pend - pbeg + T::kTP - 1) / T::kTP;
  const int32_t* bt = p.block_table + (size_t)b * p.max_blocks_per_seq;

  if (threadIdx.x == 0) {
    for (int s = 0; s < T::kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  __syncthreads();

  auto issue = [&](int step) {  // thread 0 only
    const int s = step % T::kStages;
    const uint32_t bar = bar0 + 8 * s;
    const uint32_t kreg = base + s * T::kStageBytes;
    const uint32_t vreg = kreg + T::kTP * T::kPageBytes;
    int bytes = 0;
    int pbs[T::kTP];
#pragma unroll
    for (int pg = 0; pg < T::kTP; ++pg) {
      const int page = pbeg + step * T::kTP + pg;
      int pb = -1;
      if (page < pend) {
        pb = bt[page];
        if (pb < 0 || pb >= p.num_blocks) {
          record_error(p.err, kErrBlockId);
          pb = -1;
        }
      }
      pbs[pg] = pb;
      if (pb >= 0) bytes += 2 * T::kPageBytes;
    }
    if (bytes == 0) {
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int pg = 0; pg < T::kTP; ++pg) {
      if (pbs[pg] < 0) continue;
      const int row = (pbs[pg] * p.num_kv_heads + g) * T::kBS;
#pragma unroll
      for (int bx = 0; bx < T::kBoxes; ++bx) {
        tma_load_2d(kreg + pg * T::kPageBytes + bx * T::kBoxBytes, &tmk, bx * T::kBoxCols, row, bar);
        tma_load_2d(vreg + pg * T::kPageBytes + bx * T::kBoxBytes, &tmv, bx * T::kBoxCols, row, bar);
      }
    }
  };
  if (threadIdx.x == 0) {
    const int n0 = nsteps < T::kStages ? nsteps : T::kStages;
    for (int st = 0; st < n0; ++st) issue(st);
  }

  // Q fragments (A operand, row-major 16 x 16 per k-step) for rows r0, r1; rows >= R are 0.
  uint32_t qa[T::kKSteps][4];
  {
    const int cq = (lane & 3) * 2;
    const __nv_bfloat16* q0 = nullptr;
    const __nv_bfloat16* q1 = nullptr;
    if (r0 < R) q0 = p.q + (((size_t)b * QL + r0 / G) * Hq + g * G + r0 % G) * D;
    if (r1 < R) q1 = p.q + (((size_t)b * QL + r1 / G) * Hq + g * G + r1 % G) * D;
#pragma unroll
    for (int ks = 0; ks < T::kKSteps; ++ks) {
      const int c = ks * 16 + cq;
      qa[ks][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + c) : 0u;
      qa[ks][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + c) : 0u;
      qa[ks][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + c + 8) : 0u;
      qa[ks][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + c + 8) : 0u;
    }
  }
  // causal limits of the two rows: row r (query index i = r / G) sees tokens j < L - QL + i + 1
  const int n_r0 = r0 < R ? L - QL + r0 / G + 1 : L;
  const int n_r1 = r1 < R ? L - QL + r1 / G + 1 : L;

  float o[T::kOTiles][4];
#pragma unroll
  for (int nt = 0; nt < T::kOTiles; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  // ldmatrix lane roles
  const int lm = lane >> 3;  // which 8x8 matrix this lane addresses
  const int lr = lane & 7;   // which row of it

  int done = 0;
  bool timed_out = false;
  for (int step = 0; step < nsteps; ++step) {
    const int s = step % T::kStages;
    const bool landed = mbar_wait(bar0 + 8 * s, (step / T::kStages) & 1);
    if (__syncthreads_or(!landed)) {
      timed_out = true;
      break;
    }
    done = step + 1;
    const uint32_t kreg = base + s * T::kStageBytes;
    const uint32_t vreg = kreg + T::kTP * T::kPageBytes;
    const int tok0 = (pbeg + step * T::kTP) * T::kBS;  // absolute index of the step's first token

    // which of the step's pages hold usable data
    unsigned page_ok = 0;
#pragma unroll
    for (int pg = 0; pg < T::kTP; ++pg) {
      const int page = pbeg + step * T::kTP + pg;
      if (page < pend) {
        const int pb = bt[page];
        if (pb >= 0 && pb < p.num_blocks) page_ok |= 1u << pg;
      }
    }
    const bool ragged = (page_ok != (1u << T::kTP) - 1) || (tok0 + T::kStepTokens > limit_tok);

    // S = Q K^T over the step's 64 tokens
    float sacc[T::kSTiles][4];
#pragma unroll
    for (int nt = 0; nt < T::kSTiles; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int tp = 0; tp < T::kSTiles / 2; ++tp) {  // pairs of n8 tiles = 16 tokens = one page
#pragma unroll
      for (int ks = 0; ks < T::kKSteps; ++ks) {
        // matrices: 0 -> tokens 0-7 dims lo, 1 -> tokens 0-7 dims hi, 2/3 -> tokens 8-15
        const int t = (lm >> 1) * 8 + lr;
        const int dchunk = ks * 2 + (lm & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(tile_addr<T>(kreg, tp, t, dchunk), b0, b1, b2, b3);
        mma_bf16(sacc[2 * tp], qa[ks], b0, b1);
        mma_bf16(sacc[2 * tp + 1], qa[ks], b2, b3);
      }
    }

    // scale to base 2, mask, online softmax
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < T::kSTiles; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = tok0 + nt * 8 + (lane & 3) * 2 + (c & 1);
        const int pg = nt >> 1;
        const bool ok = ((page_ok >> pg) & 1u) && j < limit_tok && j < ((c < 2) ? n_r0 : n_r1);
        const float v = ok ? sacc[nt][c] * p.scale_log2 : -INFINITY;
        sacc[nt][c] = v;
        if (c < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float a0 = fast_exp2(m0 - base0), a1 = fast_exp2(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
    uint32_t pa[T::kSTiles / 2][4];
#pragma unroll
    for (int nt = 0; nt < T::kSTiles; ++nt) {
      const float e0 = fast_exp2(sacc[nt][0] - base0);
      const float e1 = fast_exp2(sacc[nt][1] - base0);
      const float e2 = fast_exp2(sacc[nt][2] - base1);
      const float e3 = fast_exp2(sacc[nt][3] - base1);
      ps0 += e0 + e1;
      ps1 += e2 + e3;
      // S accumulator layout of two n8 tiles == A fragment layout of one k16 step
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(e0, e1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(e2, e3);
    }
    l0 = l0 * a0 + ps0;
    l1 = l1 * a1 + ps1;
#pragma unroll
    for (int nt = 0; nt < T::kOTiles; ++nt) {
      o[nt][0] *= a0; o[nt][1] *= a0;
      o[nt][2] *= a1; o[nt][3] *= a1;
    }

    // O += P V over the step's 64 tokens
#pragma unroll
    for (int kk = 0; kk < T::kSTiles / 2; ++kk) {  // k16 = one page
#pragma unroll
      for (int np = 0; np < T::kOTiles / 2; ++np) {  // pairs of n8 dim tiles
        // matrices: 0 -> tokens 0-7 dims lo, 1 -> tokens 8-15 dims lo, 2/3 -> dims hi
        const int t = (lm & 1) * 8 + lr;
        const int dchunk = np * 2 + (lm >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(tile_addr<T>(vreg, kk, t, dchunk), b0, b1, b2, b3);
        if (ragged) {
          // zero V of tokens that hold no data (stale stages, block tails): 0 * NaN is NaN
          const int jb = tok0 + kk * 16 + (lane & 3) * 2;
          const bool pok = (page_ok >> kk) & 1u;
          const uint32_t mlo0 = (pok && jb < limit_tok) ? 0x0000ffffu : 0u;
          const uint32_t mhi0 = (pok && jb + 1 < limit_tok) ? 0xffff0000u : 0u;
          const uint32_t mlo1 = (pok && jb + 8 < limit_tok) ? 0x0000ffffu : 0u;
          const uint32_t mhi1 = (pok && jb + 9 < limit_tok) ? 0xffff0000u : 0u;
          b0 &= (mlo0 | mhi0);
          b2 &= (mlo0 | mhi0);
          b1 &= (mlo1 | mhi1);
          b3 &= (mlo1 | mhi1);
        }
        mma_bf16(o[2 * np], pa[kk], b0, b1);
        mma_bf16(o[2 * np + 1], pa[kk], b2, b3);
      }
    }
    __syncthreads();  // every warp is done with stage s
    if (threadIdx.x == 0 && step + T::kStages < nsteps) issue(step + T::kStages);
  }
  if (timed_out && threadIdx.x == 0) {
    record_error(p.err, kErrTimeout);
    const int issued = min(nsteps, done + T::kStages);
    for (int st = done; st < issued; ++st) mbar_wait(bar0 + 8 * (st % T::kStages), (st / T::kStages) & 1);
  }

  // the merge kernel (launched as a programmatic dependent) may start its prologue now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? r1 : r0;
    if (r >= R) continue;
    const float l = half ? l1 : l0;
    const float m = half ? m1 : m0;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int i = r / G, h = r - (r / G) * G;
    const size_t orow = ((size_t)b * QL + i) * Hq + g * G + h;
    if (nparts == 1) {
      __nv_bfloat16* dst = p.out + orow * D + (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < T::kOTiles; ++nt)
        *reinterpret_cast<__nv_bfloat162*>(dst + nt * 8) =
            __floats2bfloat162_rn(o[nt][half * 2] * inv, o[nt][half * 2 + 1] * inv);
    } else {
      const size_t prow = orow * p.max_partitions + part;
      float* dst = p.part_o + prow * D + (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < T::kOTiles; ++nt)
        *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(o[nt][half * 2] * inv, o[nt][half * 2 + 1] * inv);
      if ((lane & 3) == 0) p.part_lse[prow] = (l > 0.f) ? m + __log2f(l) : -INFINITY;
    }
  }
}

template <int D, int MT>
cudaError_t launch_mt(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  using T = VerifyTraits<D, MT>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(verify_kernel<D, MT>), T::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_partitions, p.num_kv_heads, p.num_seqs);
  verify_kernel<D, MT><<<grid, T::kThreads, T::kSmem, st>>>(p, tk, tv);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_mt(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int rows,
                        cudaStream_t st) {
  switch ((rows + 15) / 16) {
    case 1: return launch_mt<D, 1>(p, tk, tv, st);
    case 2: return launch_mt<D, 2>(p, tk, tv, st);
    case 3: return launch_mt<D, 3>(p, tk, tv, st);
    case 4: return launch_mt<D, 4>(p, tk, tv, st);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace

cudaError_t launch_verify_tc(const AttnParams& p, const Launch& l, const CUtensorMap& tk,
                             const CUtensorMap& tv) {
  const int rows = l.group * p.q_len;
  if (l.head_dim == 128) return dispatch_mt<128>(p, tk, tv, rows, l.stream);
  if (l.head_dim == 64) return dispatch_mt<64>(p, tk, tv, rows, l.stream);
  return cudaErrorInvalidConfiguration;
}

}  // namespace pa
