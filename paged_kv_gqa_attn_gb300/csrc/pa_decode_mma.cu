// Paged GQA decode (q_len = 1) on the warp-level tensor-core instruction (mma.sync m16n8k16,
// fp32 accumulation), sm_103a: bf16 caches with bf16 operands, E4M3 caches with f16 operands.
//
// Why not CUDA cores: with paired fp32 FMAs the two products, the reduction of partial dot
// products across lanes and (E4M3) the decoding of every code cost 46 (bf16) to ~50 (E4M3) warp
// instructions per (token, kv head), so a warp held each page stage for microseconds of
// arithmetic and the E4M3 kernel ran issue-bound at about half the HBM rate.  Here one page costs
// 16 (E4M3, bf16 at G <= 4) or 24 (bf16 at G = 8) mma.sync plus fragment moves: ~21 warp
// instructions per (token, kv head) for bf16, and the page stages turn over at the rate the
// copies land.  The contraction is the same one (the G query heads of the group against each
// page; FlashAttention tiling with an online softmax, studybook fde-roadmap ch.10, section
// 10.1.2); nothing is reshaped to reach the tensor core.
//
// One warp's work per page: a page is the 16 x d slice of one physical block for one kv head
// (block-table gather, section 10.4.2; aegloslab servingai 5.3.7), copied by the TMA unit as 2-D
// boxes of 128-byte rows with the 128-byte swizzle (64-byte E4M3 rows at d = 64: the 64-byte
// swizzle), so that every fragment load below hits 32 distinct banks.  Then
//   S^T[16 tokens x 8] = K[16 x d] . Q^T[d x 8]         A = K (rows = tokens), B = Q
//   O^T[d x 8]        += V^T[d x 16]  . P^T[16 x 8]       A = V (rows = dims),  B = P
// with the G query heads of the group as columns.  The contraction index of the first product is
// spread so that each thread reads a quarter of each of its two K rows as whole 16-byte chunks;
// the rows of the second are ordered so that each thread reads an eighth of four V rows, and
// byte (E4M3) or 16-bit (bf16) permutes pair the values of two tokens.  The C fragment of S^T
// becomes the B fragment of P^T with one movmatrix.trans per 8 tokens.
//
// Softmax weights: E4M3 weights are f16 with each page's V scale folded in as an added
// log2|scale| (and its sign), so that they stay in (0, 2^kTau] for any scale and the running sum
// takes exp2(score - max) without it; each page's K scale multiplies its scores.  bf16 weights
// are a bf16 high part plus the rounded remainder (another bf16 column of the n-tile for G <= 4,
// a second P.V pass for G = 8): ~16 significant bits.  The running maximum is refreshed (three
// shuffles per column, the outputs rescaled) only when some score passes it by more than kTau.
// The CTA's warps (two for bf16, four for E4M3) take the partition's pages round-robin, each with
// its own ring of stages; the CTA then combines the warps and stores the rows or the partials.
#include "pa_kernels.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

// Each page is read by one CTA once per call: its TMA loads carry the L2 evict-first policy.
constexpr bool kDecodeKvEvictFirst = true;

template <int D, int G, bool FP8>
struct MmaDecodeTraits {
  // bf16: 2 warps per CTA, 6 CTAs per SM (llama8b_decode 83.8 us; 3 x 4: 84.9 us; 4 x 3: 85.1
  // us); E4M3: 4 warps, 4 CTAs per SM (long_fp8 167.4 us; 2 x 8: 179.5 us; 3 x 5: 198.7 us)
  static constexpr int kWarps = FP8 ? 4 : 2;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kBS = 16;
  static constexpr int kElt = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;          // 64, 128 or 256
  static constexpr int kPageBytes = kBS * kRowBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;  // K page then V page
  // E4M3: 3-stage rings; bf16 (pages twice the size): 2 stages
  static constexpr int kStages = FP8 ? 3 : 2;
  static constexpr int kMinBlocks = FP8 ? 4 : 6;
  static constexpr int kBoxes = kRowBytes >= 128 ? kRowBytes / 128 : 1;  // TMA boxes per page
  static constexpr int kKSteps = D / 16;              // k-steps of the score product
  static constexpr int kQKChunks = kRowBytes / 64;    // 16-byte K chunks per thread per row
  static constexpr int kQKWords = 4 * kQKChunks;
  static constexpr int kMTiles = D / 16;              // m-tiles (16 dims) of the value product
  static constexpr int kPVWords = kRowBytes / 32;     // 32-bit V words per thread per row
  // bf16 weights are a high part plus the rounded remainder: for G <= 4 the remainders take G more
  // columns of the n-tile; for G = 8 (no spare column) a second P.V pass multiplies them.
  static constexpr bool kLowPass = !FP8 && 2 * G > 8;
  static constexpr int kCols = (FP8 || kLowPass) ? G : 2 * G;
  static constexpr int kStageRegion = kWarps * kStages * kStageBytes;
  static constexpr int kBarRegion = kWarps * kStages * 8;
  static constexpr int kSmem = 1024 + kStageRegion + kBarRegion;  // 1 KiB: alignment of the swizzle
  static_assert(kWarps * G * D * 4 + 2 * kWarps * G * 4 <= kStageRegion, "merge scratch fits");
  static_assert(kCols <= 8, "the columns of the products are the 8 of one n-tile");
};

constexpr float kTau = 8.f;  // largest softmax weight, log2, before the running max is refreshed

// Byte offset of 16-byte chunk `c` of row `r` of a page as the TMA unit writes it.  Rows of 128 B
// or more arrive as boxes of 128-byte rows with the 128-byte swizzle (chunk ^ row % 8), box j
// holding chunks 8j .. 8j+7 of every row; 64-byte rows use the 64-byte swizzle
// (chunk ^ (row / 2) % 4).  Pages are 1 KiB aligned.
template <int RB>
__device__ __forceinline__ uint32_t chunk_off(int r, int c) {
  if constexpr (RB == 64)
    return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
  else
    return (c >> 3) * (16 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// The c-th K chunk of thread q: a quarter of the row, taken as chunk pairs 2q, 2q+1 of each
// 128-byte box (so that the 8 threads of a load phase hit 8 different bank groups), or chunk q
// of a 64-byte row.
template <int RB>
__device__ __forceinline__ int qk_chunk(int q, int c) {
  if constexpr (RB == 64)
    return q;
  else
    return 8 * (c >> 1) + 2 * q + (c & 1);
}

// D[16x8] += A[16x16] . B[16x8], f16 (or bf16) operands, fp32 accumulators (warp-collective).
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  if constexpr (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit elements held as mma fragments (warp-collective).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// What bf16 rounding leaves of p (rounded to bf16 again, it carries p's next 8 significant bits).
__device__ __forceinline__ float bf16_rem(float p) { return p - __bfloat162float(__float2bfloat16_rn(p)); }

// bf16 weight of column c when the low parts share the n-tile: the head's weight (rounded to bf16
// by the packing) in the first G columns, its remainder in the next G.
template <int G>
__device__ __forceinline__ float bf16_part(float p, int c) {
  return c < G ? p : bf16_rem(p);
}

template <int D, int G, bool FP8>
__global__ void __launch_bounds__((MmaDecodeTraits<D, G, FP8>::kThreads), (MmaDecodeTraits<D, G, FP8>::kMinBlocks))
    decode_mma_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  using T = MmaDecodeTraits<D, G, FP8>;
  constexpr int RB = T::kRowBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2;  // fragment row group
  const int qi = lane & 3;   // thread in the group
  const int part = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int Hq = p.num_q_heads;
  // The first two windows of block ids (below) depend only on the partition, not on the context
  // length: load them together with it, bounded by the table row, and mask them once it arrives.
  const int ppp = p.pages_per_partition;
  const int pbeg = part * ppp;
  const int first = pbeg + warp;
  const int32_t* bt = p.block_table + (size_t)b * p.max_blocks_per_seq;
  const int row0 = first + T::kWarps * lane, row1 = first + T::kWarps * (32 + lane);
  const int raw0 = row0 < p.max_blocks_per_seq ? bt[row0] : -1;
  const int raw1 = row1 < p.max_blocks_per_seq ? bt[row1] : -1;
  const int L = context_len(p, b, part == 0 && g == 0 && threadIdx.x == 0);

  if (L <= 0) {  // no token to attend to: zero the group's rows once, flag it
    if (part == 0) {
      for (int idx = threadIdx.x; idx < G * D; idx += T::kThreads)
        p.out[((size_t)b * Hq + g * G) * D + idx] = __float2bfloat16(0.f);
      if (threadIdx.x == 0) record_error(p.err, kErrShortContext);
    }
    return;
  }
  const int npages = (L + T::kBS - 1) / T::kBS;
  if (pbeg >= npages) return;
  const int pend = min(npages, pbeg + ppp);
  const int nparts = (npages + ppp - 1) / ppp;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  uint8_t* stages = smem + warp * T::kStages * T::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::kStageRegion) + warp * T::kStages;

  const int nk = first < pend ? (pend - first + T::kWarps - 1) / T::kWarps : 0;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < T::kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Block ids (and, for E4M3, K/V scales) of the warp's pages, 32 at a time in lane registers
  // (lane i of the first window holds page wb + i, the second window the next 32); read back with
  // shuffles.
  auto load_window = [&](int kb) {
    const int kk = kb + lane;
    return kk < nk ? bt[first + T::kWarps * kk] : -1;
  };
  auto load_scale = [&](const float* sc, int id) {
    return (FP8 && id >= 0 && id < p.num_blocks) ? sc[(size_t)id * p.num_kv_heads + g] : 1.f;
  };
  int wb = 0;
  int idw0 = lane < nk ? raw0 : -1;
  int idw1 = 32 + lane < nk ? raw1 : -1;
  float ksw0 = load_scale(p.k_scale, idw0), vsw0 = load_scale(p.v_scale, idw0);
  float ksw1 = load_scale(p.k_scale, idw1), vsw1 = load_scale(p.v_scale, idw1);
  auto id_of = [&](int k) {  // k in [wb, wb + 64), warp-uniform
    const int o = k - wb;
    return o < 32 ? __shfl_sync(0xffffffffu, idw0, o) : __shfl_sync(0xffffffffu, idw1, o - 32);
  };

  // whole warp: lane 0 starts the TMA copies of the warp's k-th page into stage k % kStages
  const uint64_t kv_policy = l2_evict_first_policy();
  auto issue = [&](int k) {
    const int pb = id_of(k);
    if (lane != 0) return;
    const int s = k % T::kStages;
    const uint32_t bar = smem_addr(&bars[s]);
    if (pb < 0 || pb >= p.num_blocks) {
      record_error(p.err, kErrBlockId);
      mbar_arrive(bar);
      return;
    }
    const int row = (int)(((int64_t)pb * p.num_kv_heads + g) * T::kBS);
    const uint32_t dst = smem_addr(stages + s * T::kStageBytes);
    mbar_arrive_expect_tx(bar, 2 * T::kPageBytes);
#pragma unroll
    for (int j = 0; j < T::kBoxes; ++j) {
      if (kDecodeKvEvictFirst) {
        tma_load_2d_hint(dst + j * (16 * 128), &tmk, j * (128 / T::kElt), row, bar, kv_policy);
        tma_load_2d_hint(dst + T::kPageBytes + j * (16 * 128), &tmv, j * (128 / T::kElt), row, bar, kv_policy);
      } else {
        tma_load_2d(dst + j * (16 * 128), &tmk, j * (128 / T::kElt), row, bar);
        tma_load_2d(dst + T::kPageBytes + j * (16 * 128), &tmv, j * (128 / T::kElt), row, bar);
      }
    }
  };
  {
    const int n0 = nk < T::kStages ? nk : T::kStages;
    for (int k = 0; k < n0; ++k) issue(k);
  }

  // B fragments of Q^T, column gi (E4M3: head gi; bf16: head gi % G, the first G columns for the
  // weights' high parts and the next G for their low parts).  In k-step s the thread's contraction
  // indices 2qi, 2qi+1 / 2qi+8, 2qi+9 are four consecutive dims of its K words: E4M3 word s (two
  // codes each half), bf16 words 2s and 2s+1.  E4M3: each head's row is scaled by a power of two
  // 2^k before its f16 re-encoding (f16_prescale_exp: exact, no overflow for any bf16 q), and
  // its scores by 2^-k: qdiv0 / qdiv1 = 2^-k of the score columns 2qi / 2qi+1.
  uint32_t qf[T::kKSteps][2];
  float qdiv0 = 1.f, qdiv1 = 1.f;
  {
    const bool real = gi < T::kCols;
    const __nv_bfloat16* qrow = p.q + ((size_t)b * Hq + g * G + (real ? gi % G : 0)) * D;
    uint2 xs[T::kKSteps];
    uint32_t emax = 0;
#pragma unroll
    for (int s = 0; s < T::kKSteps; ++s) {
      const int w = FP8 ? s : 2 * s;
      const int d0 = (qk_chunk<RB>(qi, w >> 2) * 16 + (w & 3) * 4) / T::kElt;
      xs[s] = real ? *reinterpret_cast<const uint2*>(qrow + d0) : make_uint2(0u, 0u);
      if constexpr (FP8) emax = max(emax, max(bf16x2_max_exp(xs[s].x), bf16x2_max_exp(xs[s].y)));
    }
    if constexpr (FP8) {
      // the 4 lanes of row gi (qi = 0..3) hold all of head gi's dims
      emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, 1));
      emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, 2));
      const int kq = f16_prescale_exp(emax);
      const float up = exp2_int(kq);
#pragma unroll
      for (int s = 0; s < T::kKSteps; ++s) {
        const float2 lo = bf16x2_to_f2(xs[s].x), hi = bf16x2_to_f2(xs[s].y);
        qf[s][0] = pack_f16(lo.x * up, lo.y * up);
        qf[s][1] = pack_f16(hi.x * up, hi.y * up);
      }
      // score column c is head c: its exponent sits in the lanes of row c (lane 4c)
      qdiv0 = exp2_int(-__shfl_sync(0xffffffffu, kq, (2 * qi) * 4));
      qdiv1 = exp2_int(-__shfl_sync(0xffffffffu, kq, (2 * qi + 1) * 4));
    } else {
#pragma unroll
      for (int s = 0; s < T::kKSteps; ++s) {
        qf[s][0] = xs[s].x;
        qf[s][1] = xs[s].y;
      }
    }
  }

  // O^T accumulators: o[i][0] / o[i][1] = the m-tile's low dim (vdim below) of columns 2qi /
  // 2qi+1, o[i][2] / o[i][3] = the dim after it.  Running max m and sum l of columns 2qi (m0, l0)
  // and 2qi+1 (m1, l1); l holds this thread's tokens only until the end.
  float o[T::kMTiles][4];
#pragma unroll
  for (int i = 0; i < T::kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  int k_done = 0;
  bool timed_out = false;
  for (int k = 0; k < nk; ++k) {
    const int s = k % T::kStages;
    const uint32_t parity = (k / T::kStages) & 1;
    const bool landed = mbar_wait(smem_addr(&bars[s]), parity);
    if (__any_sync(0xffffffffu, !landed)) {
      timed_out = true;
      break;
    }
    k_done = k + 1;
    if (k == wb + 32) {  // slide the windows (the issue below looks at most kStages ahead)
      wb += 32;
      idw0 = idw1;
      idw1 = load_window(wb + 32);
      if constexpr (FP8) {
        ksw0 = ksw1;
        vsw0 = vsw1;
        ksw1 = load_scale(p.k_scale, idw1);
        vsw1 = load_scale(p.v_scale, idw1);
      }
    }
    const int page = first + T::kWarps * k;
    const int pb = id_of(k);
    if (pb >= 0 && pb < p.num_blocks) {
      const int valid = min(T::kBS, L - page * T::kBS);
      const uint8_t* kp = stages + s * T::kStageBytes;
      const uint8_t* vp = kp + T::kPageBytes;

      // ---- S^T = K . Q^T: rows gi and gi + 8 of the page, a quarter row each ----
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        uint32_t k0[T::kQKWords], k1[T::kQKWords];
#pragma unroll
        for (int c = 0; c < T::kQKChunks; ++c) {
          const int ch = qk_chunk<RB>(qi, c);
          const uint4 x = *reinterpret_cast<const uint4*>(kp + chunk_off<RB>(gi, ch));
          const uint4 y = *reinterpret_cast<const uint4*>(kp + chunk_off<RB>(gi + 8, ch));
          k0[4 * c] = x.x; k0[4 * c + 1] = x.y; k0[4 * c + 2] = x.z; k0[4 * c + 3] = x.w;
          k1[4 * c] = y.x; k1[4 * c + 1] = y.y; k1[4 * c + 2] = y.z; k1[4 * c + 3] = y.w;
        }
#pragma unroll
        for (int st = 0; st < T::kKSteps; ++st) {
          if constexpr (FP8)
            mma_16816<false>(sc, e4m3x2_to_f16x2(k0[st]), e4m3x2_to_f16x2(k1[st]), e4m3x2_to_f16x2(k0[st] >> 16),
                             e4m3x2_to_f16x2(k1[st] >> 16), qf[st][0], qf[st][1]);
          else
            mma_16816<true>(sc, k0[2 * st], k1[2 * st], k0[2 * st + 1], k1[2 * st + 1], qf[st][0], qf[st][1]);
        }
      }

      // ---- online softmax: sc[0] / sc[1] = token gi, columns 2qi / 2qi+1; sc[2] / sc[3] = token gi+8 ----
      float ksc = p.scale_log2, lv = 0.f, rvs = 1.f;
      uint32_t neg = 0u;
      if constexpr (FP8) {
        const int o32 = k - wb;  // k is in [wb, wb + 32) here
        const float ks = __shfl_sync(0xffffffffu, ksw0, o32);
        const float vs = __shfl_sync(0xffffffffu, vsw0, o32);
        lv = __log2f(fmaxf(fabsf(vs), 0x1p-100f));
        rvs = fast_exp2(-lv);
        neg = vs < 0.f ? 0x80008000u : 0u;
        ksc *= ks;
      }
      const float ksc0 = FP8 ? ksc * qdiv0 : ksc, ksc1 = FP8 ? ksc * qdiv1 : ksc;
      float x0 = fmaf(sc[0], ksc0, lv), x1 = fmaf(sc[1], ksc1, lv);
      float x2 = fmaf(sc[2], ksc0, lv), x3 = fmaf(sc[3], ksc1, lv);
      if (valid < T::kBS) {
        if (gi >= valid) x0 = x1 = -INFINITY;
        if (gi + 8 >= valid) x2 = x3 = -INFINITY;
      }
      float lm0 = fmaxf(x0, x2), lm1 = fmaxf(x1, x3);
      if (__any_sync(0xffffffffu, lm0 > m0 + kTau || lm1 > m1 + kTau)) {
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
          lm0 = fmaxf(lm0, __shfl_xor_sync(0xffffffffu, lm0, sh));
          lm1 = fmaxf(lm1, __shfl_xor_sync(0xffffffffu, lm1, sh));
        }
        const float n0 = fmaxf(m0, lm0), n1 = fmaxf(m1, lm1);
        const float a0 = fast_exp2(m0 - n0), a1 = fast_exp2(m1 - n1);
        m0 = n0;
        m1 = n1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int i = 0; i < T::kMTiles; ++i) {
          o[i][0] *= a0;
          o[i][2] *= a0;
          o[i][1] *= a1;
          o[i][3] *= a1;
        }
      }
      const float p0 = fast_exp2(x0 - m0), p1 = fast_exp2(x1 - m1);
      const float p2 = fast_exp2(x2 - m0), p3 = fast_exp2(x3 - m1);
      l0 += (p0 + p2) * rvs;
      l1 += (p1 + p3) * rvs;
      // B fragments of P^T: b0 = tokens 2qi, 2qi+1 of column gi, b1 = tokens 2qi+8, 2qi+9
      uint32_t b0, b1, b0l = 0u, b1l = 0u;
      if constexpr (FP8) {
        b0 = movmatrix_trans(pack_f16(p0, p1) ^ neg);
        b1 = movmatrix_trans(pack_f16(p2, p3) ^ neg);
      } else if constexpr (T::kLowPass) {
        b0 = movmatrix_trans(pack_bf16(p0, p1));
        b1 = movmatrix_trans(pack_bf16(p2, p3));
        b0l = movmatrix_trans(pack_bf16(bf16_rem(p0), bf16_rem(p1)));
        b1l = movmatrix_trans(pack_bf16(bf16_rem(p2), bf16_rem(p3)));
      } else {
        b0 = movmatrix_trans(pack_bf16(bf16_part<G>(p0, 2 * qi), bf16_part<G>(p1, 2 * qi + 1)));
        b1 = movmatrix_trans(pack_bf16(bf16_part<G>(p2, 2 * qi), bf16_part<G>(p3, 2 * qi + 1)));
      }

      // ---- O^T += V^T . P^T: rows 2qi, 2qi+1, 2qi+8, 2qi+9 of the page, an eighth of each row ----
      uint32_t v[4][T::kPVWords];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = 2 * qi + (r & 1) + 8 * (r >> 1);
        if constexpr (RB == 64) {  // E4M3, d = 64: 8 bytes
          const uint2 x = *reinterpret_cast<const uint2*>(vp + chunk_off<RB>(t, gi >> 1) + 8 * (gi & 1));
          v[r][0] = x.x; v[r][1] = x.y;
        } else {  // chunk gi of every 128-byte box
#pragma unroll
          for (int j = 0; j < T::kPVWords / 4; ++j) {
            const uint4 x = *reinterpret_cast<const uint4*>(vp + chunk_off<RB>(t, 8 * j + gi));
            v[r][4 * j] = x.x; v[r][4 * j + 1] = x.y; v[r][4 * j + 2] = x.z; v[r][4 * j + 3] = x.w;
          }
        }
      }
      if (valid < T::kBS) {  // values past the context may be anything (even NaN): zero them
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int t = 2 * qi + (r & 1) + 8 * (r >> 1);
          if (t >= valid)
#pragma unroll
            for (int w = 0; w < T::kPVWords; ++w) v[r][w] = 0u;
        }
      }
#pragma unroll
      for (int w = 0; w < T::kPVWords; ++w) {
        if constexpr (FP8) {
          // byte pairs (token 2qi, 2qi+1) and (2qi+8, 2qi+9) of the word's four dims: m-tiles 2w, 2w+1
          const uint32_t xa = __byte_perm(v[0][w], v[1][w], 0x5140);
          const uint32_t ya = __byte_perm(v[0][w], v[1][w], 0x7362);
          const uint32_t xb = __byte_perm(v[2][w], v[3][w], 0x5140);
          const uint32_t yb = __byte_perm(v[2][w], v[3][w], 0x7362);
          mma_16816<false>(o[2 * w], e4m3x2_to_f16x2(xa), e4m3x2_to_f16x2(xa >> 16), e4m3x2_to_f16x2(xb),
                           e4m3x2_to_f16x2(xb >> 16), b0, b1);
          mma_16816<false>(o[2 * w + 1], e4m3x2_to_f16x2(ya), e4m3x2_to_f16x2(ya >> 16), e4m3x2_to_f16x2(yb),
                           e4m3x2_to_f16x2(yb >> 16), b0, b1);
        } else {
          // bf16 pairs (token 2qi, 2qi+1) and (2qi+8, 2qi+9) of the word's two dims: m-tile w
          const uint32_t a0 = __byte_perm(v[0][w], v[1][w], 0x5410), a1 = __byte_perm(v[0][w], v[1][w], 0x7632);
          const uint32_t a2 = __byte_perm(v[2][w], v[3][w], 0x5410), a3 = __byte_perm(v[2][w], v[3][w], 0x7632);
          mma_16816<true>(o[w], a0, a1, a2, a3, b0, b1);
          if constexpr (T::kLowPass) mma_16816<true>(o[w], a0, a1, a2, a3, b0l, b1l);
        }
      }
    }
    __syncwarp();
    if (k + T::kStages < nk) issue(k + T::kStages);
  }
  if (timed_out) {
    // let every copy this warp started land (bounded) before its stages are reused
    if (lane == 0) {
      record_error(p.err, kErrTimeout);
      const int issued = min(nk, k_done + T::kStages);
      for (int k = k_done; k < issued; ++k) mbar_wait(smem_addr(&bars[k % T::kStages]), (k / T::kStages) & 1);
    }
    __syncwarp();
  }

  // the merge kernel (launched as a programmatic dependent) may start its prologue now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // sums over the 8 row groups (each thread summed its own tokens)
#pragma unroll
  for (int sh = 4; sh < 32; sh <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
    l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
  }
  if constexpr (!FP8 && !T::kLowPass) {  // add each head's low-part column (column c + G) to its column c
    if constexpr (G == 1) {
#pragma unroll
      for (int i = 0; i < T::kMTiles; ++i) {
        o[i][0] += o[i][1];
        o[i][2] += o[i][3];
      }
    } else {
#pragma unroll
      for (int i = 0; i < T::kMTiles; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][e] += __shfl_xor_sync(0xffffffffu, o[i][e], G / 2);
    }
  }

  __syncthreads();  // every warp is done with its stages
  float* wacc = reinterpret_cast<float*>(smem);  // [kWarps][G][D]
  float* wm = wacc + T::kWarps * G * D;          // [kWarps][G]
  float* wl = wm + T::kWarps * G;                // [kWarps][G]
  const int h0 = 2 * qi, h1 = 2 * qi + 1;
  if (gi == 0) {
    if (h0 < G) {
      wm[warp * G + h0] = m0;
      wl[warp * G + h0] = l0;
    }
    if (h1 < G) {
      wm[warp * G + h1] = m1;
      wl[warp * G + h1] = l1;
    }
  }
#pragma unroll
  for (int i = 0; i < T::kMTiles; ++i) {
    // the m-tile's low dim: E4M3 d/8 * gi + 2i; bf16 word i of chunk gi of box i / 4
    const int dd = FP8 ? (D / 8) * gi + 2 * i : 64 * (i >> 2) + 8 * gi + 2 * (i & 3);
    if (h0 < G) *reinterpret_cast<float2*>(wacc + (warp * G + h0) * D + dd) = make_float2(o[i][0], o[i][2]);
    if (h1 < G) *reinterpret_cast<float2*>(wacc + (warp * G + h1) * D + dd) = make_float2(o[i][1], o[i][3]);
  }
  __syncthreads();
  store_partition<G, D, T::kWarps>(p, wacc, wm, wl, b, g, part, nparts);
}

template <int D, int G, bool FP8>
cudaError_t launch_one(const AttnParams& p, cudaStream_t stream, const CUtensorMap& tk, const CUtensorMap& tv) {
  using T = MmaDecodeTraits<D, G, FP8>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(decode_mma_kernel<D, G, FP8>), T::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_partitions, p.num_kv_heads, p.num_seqs);
  decode_mma_kernel<D, G, FP8><<<grid, T::kThreads, T::kSmem, stream>>>(p, tk, tv);
  return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t dispatch_group(const AttnParams& p, const Launch& l, const CUtensorMap& tk, const CUtensorMap& tv) {
  switch (l.group) {
    case 1: return launch_one<D, 1, FP8>(p, l.stream, tk, tv);
    case 2: return launch_one<D, 2, FP8>(p, l.stream, tk, tv);
    case 4: return launch_one<D, 4, FP8>(p, l.stream, tk, tv);
    case 8: return launch_one<D, 8, FP8>(p, l.stream, tk, tv);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace

cudaError_t launch_decode_mma(const AttnParams& p, const Launch& l, const CUtensorMap& tk, const CUtensorMap& tv) {
  if (l.head_dim == 128) return l.fp8 ? dispatch_group<128, true>(p, l, tk, tv) : dispatch_group<128, false>(p, l, tk, tv);
  if (l.head_dim == 64) return l.fp8 ? dispatch_group<64, true>(p, l, tk, tv) : dispatch_group<64, false>(p, l, tk, tv);
  return cudaErrorInvalidConfiguration;
}

}  // namespace pa
