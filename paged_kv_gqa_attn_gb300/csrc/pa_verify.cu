// Paged GQA speculative-verify attention (q_len = K + 1 causal rows) on 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), sm_103a.
//
// The verify forward scores the K draft tokens plus the bonus position in one pass, each row
// masked to the tokens up to itself (sirzzang "Speculative Decoding", parallel verification and
// its causal-mask figure).  With G query heads per kv head, the R = G * q_len rows of one kv head
// share every K/V page, so scores and values are dense products per 64-token step:
//   S[128 x 64]  = Q[128 x d] . K_step[64 x d]^T      (rows beyond R are padding)
//   O[128 x d]  += P[128 x 64] . V_step[64 x d]
// FlashAttention's tiling with an online softmax (studybook fde-roadmap ch.10, section 10.1.2).
//
// Work split (persistent, balanced).  For each kv head the pages of all sequences are laid end
// to end; the Hkv * TP pages of all heads are cut into gridDim.x equal contiguous ranges, one per
// resident CTA.  A range may cross sequence boundaries: a CTA walks its range as a list of
// segments (kv head g, sequence b, pages [p0, p1)).  A segment covering its whole sequence writes
// the final rows; otherwise it writes a partial (normalised O and log2-sum-exp) into slot
// g * B + b + c (c = CTA index), and the segment merge kernel combines the pieces with the
// log-sum-exp rule.  TP and the per-sequence page offsets (the plan) are built by every CTA from
// context_lens for up to 1022 sequences, else by verify_plan_kernel just before on the stream.
//
// Each CTA keeps its tensor memory, barriers and pipelines across segments, five warps (roles
// for a CTA whose rows sit in TMEM lanes 0-63; the second CTA on an SM mirrors warps 0-1 and 2-3
// and keeps its rows in lanes 64-127, so the two CTAs' softmax warps use different sub-partitions,
// and each sub-partition w % 4 holds one softmax warp and one producer warp of the other CTA):
//   warps 3, 2     -- TMA producers: K and V pages (2-D tensor boxes of 16 tokens x 64 dims with
//                     the 128-byte swizzle, completion on mbarriers) into a 2-stage K ring (a K
//                     tile is free once its QK is done) and a 3-stage V ring (a V tile is held
//                     until its PV, so it needs the deeper ring to hide HBM latency); the K
//                     producer also writes each step's page record (which of its pages hold a
//                     block) into a 4-step ring, so the softmax needs no global load per step;
//   warp 4, lane 0 -- MMA issuer: tcgen05.mma for both products, completion via tcgen05.commit,
//                     issuing S(k+1) ahead of PV(k) whenever it is ready first;
//   warps 0, 1     -- softmax: thread r owns query row r (TMEM lane r); it reads its 64 scores
//                     with tcgen05.ld, masks (causal limit or tree-ancestor mask over the new
//                     tokens, block tail, segment end), keeps the row max m and sum l in base 2,
//                     writes P as bf16 pairs over its S in tensor memory (P.V reads its A
//                     operand from there), and rescales its O row in TMEM only when the max grows
//                     by more than 2^8 (a stale max is exact as long as l uses the same one).
//                     Between segments it writes the next Q and drains O.
// Tensor memory holds two S buffers, so QK of step k+1 runs while the softmax works on step k.
// Shared operands use the canonical tcgen05 layouts: Q and K K-major with 128-byte swizzle
// (8-row groups 1024 B apart), V MN-major with 128-byte swizzle (64-dim atoms one region apart).
#include "pa_kernels.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

template <int D>
struct TcTraits {
  static constexpr int kBS = 16;
  static constexpr int kTP = 4;                          // pages per step
  static constexpr int kStepTokens = kTP * kBS;          // 64 = N of S, K of P.V
  static constexpr int kHalves = D / 64;                 // 64-dim swizzle atoms across d
  static constexpr int kRegion = kStepTokens * 128;      // one half: 64 token rows x 128 B
  static constexpr int kBoxBytes = kBS * 128;            // one half of one page
  static constexpr int kKTile = kHalves * kRegion;       // [half][64 token rows][128 B]
  static constexpr int kKStages = 2;                     // K ring: the tile is free after QK
  static constexpr int kVStages = 3;                     // V ring: held from its copy until PV
  static constexpr int kRows = 64;                       // rows a CTA serves (G * q_len <= 64)
  static constexpr int kQBytes = kHalves * kRows * 128;  // [half][64 rows][128 B]
  // [K 0][K 1][Q halves][V 0][V 1][V 2]: a 64-row Q half read as 128 MMA rows overhangs into the
  // next 8 KB (rows in the upper lane half) or underhangs into the 8 KB before (lower half), so
  // Q sits between other buffers.
  static constexpr int kOffK = 0;
  static constexpr int kOffQ = kOffK + kKStages * kKTile;
  static constexpr int kOffV = kOffQ + kQBytes;
  static constexpr int kOffBar = kOffV + kVStages * kKTile;
  // barriers: kfull[2], kempty[2], vfull[3], vempty[3], o_done[2], p_ready[2], s_ready[2],
  // q_ready, o_free, final, for E4M3 caches kready[2], vready[3] (tile converted to f16), and
  // rec[4] (bf16: page record of a step written)
  static constexpr int kRecSlots = 4;
  static constexpr int kNumBars = 24 + kRecSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  // bf16 page records: per step, the bits of its pages that hold a block (one 32-bit word), a
  // ring of kRecSlots steps
  static constexpr int kOffRec = kOffMisc + 16;
  static constexpr int kOffPlan = kOffRec + kRecSlots * 4;  // the CTA's own plan (B <= kOwnPlanMax)
  static constexpr int kSmem = kOffPlan + 1024 * 4 + 1024; // + slack for 1024-B alignment
  // tensor memory: two S buffers (64 fp32 columns each; P of a step overwrites its S as bf16
  // pairs and feeds P.V from there), then O
  static constexpr int kSCol = 0;
  static constexpr int kOCol = 128;
  static constexpr int kTmemCols = 256;
  static constexpr int kThreads = 160;
  // instruction descriptors (kind::f16): D fp32 (bit 4), A bf16 (bits 7-9 = 1), B bf16 (bits
  // 10-12 = 1), B major bit 16 (1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24
  static constexpr uint32_t kIdescQK =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kStepTokens >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static constexpr uint32_t kIdescPV =
      (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  // E4M3 caches: the products run on f16 operands (A and B type 0)
  static constexpr uint32_t kIdescQK16 = kIdescQK & ~((1u << 7) | (1u << 10));
  static constexpr uint32_t kIdescPV16 = kIdescPV & ~((1u << 7) | (1u << 10));
  static_assert(kOCol + D <= kTmemCols, "tensor memory layout");
};

// ---- the balanced split: a CTA's contiguous range of the (kv head, sequence page) space ------
//
// Each (kv head, sequence) segment costs kSegCost pages more than it holds: a CTA pays a pipeline
// drain and refill, a partial write and a merge for each segment it starts, so the split places
// kSegCost virtual pages in front of every segment's real pages and cuts the virtual space into
// equal ranges -- a CTA that crosses a boundary gets fewer real pages.
// plan[0] = TP (virtual pages of all sequences, one kv head), plan[1 + b] = virtual start of
// sequence b (its header, then its real pages; plan[1 + B] = TP).  Real page k of (g, b) sits at
// x = g * TP + plan[1 + b] + kSegCost + k.  A range that starts inside a header begins at the
// segment's first real page; one that ends inside a header has an empty last segment.
constexpr int kSegCost = 14;
// KV pages are read once per call: their TMA loads carry the L2 evict-first policy.
constexpr bool kKvEvictFirst = true;
// warps per CTA of the merge kernel (one warp per output row)
constexpr int kMergeWarps = 4;
// E4M3 producer warps poll their copy and conversion sides; an idle poll sleeps this long (ns)
constexpr unsigned kProducerBackoffNs = 128;
constexpr int kOwnPlanMax = 1022;  // up to this many sequences every CTA builds the plan itself

// The page prefix of the (clamped) contexts, built by all threads of a CTA into plan[0 .. B + 1]
// (the same numbers verify_plan_kernel writes): a contiguous run of sequences per thread, then a
// block-wide exclusive scan of the run sums.
__device__ __forceinline__ int plan_pages(const AttnParams& p, int b) {
  const int L = min(p.context_lens[b], p.max_context_len);
  return L > 0 ? (L + 15) / 16 + kSegCost : 0;  // real pages plus the segment's header
}

// pre >= 0: this thread's page count of sequence threadIdx.x, loaded by the caller ahead of time
// (B <= blockDim.x: one sequence per thread); pre < 0: the threads load their runs here.
__device__ void build_plan(const AttnParams& p, int32_t* plan, int pre) {
  __shared__ int warp_tot[8];
  const int B = p.num_seqs, t = threadIdx.x, nt = blockDim.x, lane = t & 31, warp = t >> 5;
  const int per = (B + nt - 1) / nt;
  const int b0 = min(B, t * per), b1 = min(B, b0 + per);
  int sum = 0;
  if (pre >= 0) sum = pre;  // per == 1: b1 - b0 <= 1 and the count was loaded at kernel entry
  else
    for (int b = b0; b < b1; ++b) sum += plan_pages(p, b);
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < nt / 32; ++w) {
    if (w < warp) before += warp_tot[w];
    total += warp_tot[w];
  }
  int run = before + inc - sum;
  if (pre >= 0) {
    if (b0 < b1) plan[1 + b0] = run;
  } else {
    for (int b = b0; b < b1; ++b) {
      plan[1 + b] = run;
      run += plan_pages(p, b);
    }
  }
  if (t == 0) {
    plan[0] = total;
    plan[1 + B] = total;
  }
  __syncthreads();
}

struct Range {
  long long x0, x1;  // [x0, x1): this CTA's pages
  long long TP;
};

// Shares of the split: a CTA of the first half of the grid weighs kShareFirst, one of the second
// half kShareSecond.  The block scheduler places the first half one CTA per SM before the
// second, so the second CTA of every SM starts later.  CTA c's range starts at
// X(c) = floor(T * u(c) / U), u(c) = the weights of the CTAs before c, U = u(ncta).
constexpr int kShareFirst = 16, kShareSecond = 16;

__device__ __forceinline__ long long share_units(int c, int ncta) {
  const int H = ncta / 2;
  return (long long)kShareFirst * min(c, H) + (long long)kShareSecond * max(c - H, 0);
}

__device__ __forceinline__ long long range_start(int c, long long T, int ncta) {
  return T * share_units(c, ncta) / share_units(ncta, ncta);
}

// every CTA's range holds at least one page
__device__ __forceinline__ bool every_range_nonempty(long long T, int ncta) {
  return T * min(kShareFirst, kShareSecond) >= share_units(ncta, ncta);
}

__device__ __forceinline__ Range cta_range(const int32_t* plan, int num_kv_heads, int c, int ncta) {
  Range r;
  r.TP = plan[0];
  const long long T = r.TP * num_kv_heads;
  r.x0 = range_start(c, T, ncta);
  r.x1 = range_start(c + 1, T, ncta);
  return r;
}

// CTA whose range holds flattened page x < T (the inverse of cta_range): the largest c with
// X(c) <= x, i.e. u(c) <= floor(((x + 1) U - 1) / T).
__device__ __forceinline__ int cta_of(long long x, long long T, int ncta) {
  const int H = ncta / 2;
  const long long v = ((x + 1) * share_units(ncta, ncta) - 1) / T;
  const long long first = (long long)kShareFirst * H;
  const long long c = v < first ? v / kShareFirst : H + (v - first) / kShareSecond;
  return (int)min(c, (long long)ncta - 1);
}

// One segment: kv head g, sequence b, its pages [p0, p1).
struct Seg {
  int g, b, p0, p1, npages;
  bool whole;  // the segment is the sequence's whole context
};

// The segment that starts at flattened page x (x < range end).
__device__ __forceinline__ Seg segment_at(const int32_t* plan, int B, const Range& rg, long long x) {
  Seg sg;
  sg.g = (int)(x / rg.TP);
  const int loc = (int)(x - (long long)sg.g * rg.TP);
  // sequence b with plan[1 + b] <= loc < plan[2 + b] (skips empty sequences)
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (plan[1 + mid] <= loc) lo = mid; else hi = mid - 1;
  }
  sg.b = lo;
  const int real0 = plan[1 + lo] + kSegCost;  // first real page of the segment
  sg.npages = plan[2 + lo] - real0;
  sg.p0 = max(loc - real0, 0);
  const long long seg_end = min(rg.x1, (long long)sg.g * rg.TP + plan[2 + lo]);
  sg.p1 = (int)(seg_end - ((long long)sg.g * rg.TP + real0));  // <= p0: the range ends in the header
  sg.whole = sg.p0 == 0 && sg.p1 == sg.npages;
  return sg;
}

__device__ __forceinline__ long long seg_end_x(const Seg& sg, const int32_t* plan, const Range& rg) {
  return min(rg.x1, (long long)sg.g * rg.TP + plan[2 + sg.b]);
}

#ifdef PA_TIMELINE
// Instrumented build only (-DPA_TIMELINE, a separate library; the product build has none of
// it): %globaltimer stamps per CTA of the last verify launch, and the end of its merge, read by
// paged_attn_timeline_read_verify.  Slots: 0 entry, 1 plan built, 2 first S seen by the softmax,
// 3 softmax done, 4 SM id, 5 segments walked, 6 steps walked, 7 exit.
constexpr int kTlCtas = 1024, kTlSlots = 8;
__device__ unsigned long long g_verify_timeline[kTlCtas * kTlSlots];
__device__ unsigned long long g_verify_merge_end;
__device__ __forceinline__ unsigned long long tl_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tl_put(int slot, unsigned long long v) {
  if (blockIdx.x < kTlCtas) g_verify_timeline[blockIdx.x * kTlSlots + slot] = v;
}
#define PA_TL_STAMP(slot) tl_put((slot), tl_now())
#define PA_TL_VALUE(slot, v) tl_put((slot), (unsigned long long)(v))
// Per-step SM-clock stamps (clock64) of 16 CTAs -- the first 8 of each half of the grid, which
// pair up on SMs -- over their first 64 steps, read by paged_attn_timeline_read_verify_steps.
enum StepSlot {
  kStVCopy = 0,  // V copy of the step issued
  kStVLanded,    // E4M3: the V warp saw the step's V bytes land
  kStConvV,      // E4M3: the V warp's conversion done
  kStConvK,      // E4M3: the K warp's conversion done
  kStQK,         // QK issued
  kStS,          // S seen by the softmax (row 0)
  kStP0,         // P written by the first softmax warp
  kStPV,         // PV issued
  kStKCopy,      // K copy issued and the step's page record written
  kStP1,         // P written by the second softmax warp
  kStSlots
};
constexpr int kStCtas = 16, kStSteps = 64;
__device__ long long g_verify_steps[kStCtas * kStSteps * kStSlots];
__device__ __forceinline__ void st_put(int step, int slot) {
  const int h = gridDim.x / 2;
  int c = -1;
  if (blockIdx.x < 8) c = blockIdx.x;
  else if (blockIdx.x >= h && blockIdx.x < h + 8) c = 8 + blockIdx.x - h;
  if (c >= 0 && step < kStSteps) g_verify_steps[(c * kStSteps + step) * kStSlots + slot] = clock64();
}
#define PA_ST(step, slot) st_put((step), (slot))
#else
#define PA_ST(step, slot) ((void)0)
#define PA_TL_STAMP(slot) ((void)0)
#define PA_TL_VALUE(slot, v) ((void)0)
#endif

template <int D, bool FP8>
__global__ void __launch_bounds__(160, 2) verify_tc_kernel(const AttnParams p, int32_t* __restrict__ plan_g,
                                                           const __grid_constant__ CUtensorMap tmk,
                                                           const __grid_constant__ CUtensorMap tmv) {
  using T = TcTraits<D>;
  // E4M3 with head_dim 128: Q.K^T on the E4M3 codes of K (kind::f8f6f4, Q split into two E4M3
  // terms), P.V on f16; head_dim 64: both products on f16 (K and V converted)
  constexpr bool kKDirect = FP8 && D == 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));  // generic pointer to `base`
  const uint32_t sQ = base + T::kOffQ;
  const uint32_t sK = base + T::kOffK;
  const uint32_t sV = base + T::kOffV;
  // barriers
  const uint32_t bar_kfull = base + T::kOffBar;     // + 8 * (step % 2): K tile landed
  const uint32_t bar_kempty = bar_kfull + 16;       // + 8 * (step % 2): QK done, K tile reusable
  const uint32_t bar_vfull = bar_kempty + 16;       // + 8 * (step % 3): V tile landed
  const uint32_t bar_vempty = bar_vfull + 24;       // + 8 * (step % 3): PV done, V tile reusable
  const uint32_t bar_o_done = bar_vempty + 24;      // + 8 * (step % 2): PV done (O updated, S/P buffer free)
  const uint32_t bar_p_ready = bar_o_done + 16;     // + 8 * (step % 2): softmax wrote P (2 warps)
  const uint32_t bar_s_ready = bar_p_ready + 16;    // + 8 * (step % 2): S of the step in tensor memory
  const uint32_t bar_q_ready = bar_s_ready + 16;    // Q of a segment written
  const uint32_t bar_o_free = bar_q_ready + 8;      // O of a segment read out
  const uint32_t bar_final = bar_o_free + 8;        // every MMA issued has completed
  const uint32_t bar_kready = bar_final + 8;        // E4M3: + 8 * (step % 2): K tile converted to f16
  const uint32_t bar_vready = bar_kready + 16;      // E4M3: + 8 * (step % 3): V tile converted to f16
  const uint32_t bar_rec = bar_vready + 24;         // bf16: + 8 * (step % 4): the step's page record written
  uint32_t* const srec = reinterpret_cast<uint32_t*>(gbase + T::kOffRec);
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + T::kOffMisc);
  volatile uint32_t* abort_flag = misc + 1;
#ifdef PA_TIMELINE
  if (threadIdx.x == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    PA_TL_STAMP(0);
    PA_TL_VALUE(4, smid);
  }
#endif

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads;
  const int Hkv = p.num_kv_heads;
  const int G = Hq / Hkv;
  const int QL = p.q_len;
  const int R = G * QL;
  const int B = p.num_seqs;
  // The plan's context lengths are loaded first (one per thread up to blockDim.x sequences), so
  // their latency overlaps the set-up below.
  int pre_pages = -1;
  if (B <= (int)blockDim.x) pre_pages = threadIdx.x < B ? plan_pages(p, threadIdx.x) : 0;

  // ---- set-up (independent of the plan): barriers, tensor memory ---------------------------
  if (threadIdx.x == 128) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
      mbar_init(bar_o_done + 8 * s, 1);
      mbar_init(bar_p_ready + 8 * s, 2);
      mbar_init(bar_s_ready + 8 * s, 1);
      mbar_init(bar_kready + 8 * s, 1);
    }
    for (int s = 0; s < 3; ++s) {
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_vempty + 8 * s, 1);
      mbar_init(bar_vready + 8 * s, kKDirect ? 2 : 1);  // head_dim 128: both producer warps convert V
    }
    for (int s = 0; s < T::kRecSlots; ++s) mbar_init(bar_rec + 8 * s, 1);
    mbar_init(bar_q_ready, 2);
    mbar_init(bar_o_free, 2);
    mbar_init(bar_final, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    if constexpr (!FP8 || kKDirect) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    if constexpr (!FP8) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + T::kOffMisc),
                 "r"(T::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t tO = tmem + T::kOCol;
  auto tS_of = [&](int step) { return tmem + T::kSCol + 64u * (uint32_t)(step & 1); };

  // The plan: up to kOwnPlanMax sequences every CTA builds it in shared memory (CTA 0 also publishes
  // it for the merge kernel, flags short or clamped contexts and zeroes the rows of empty
  // sequences); beyond that the planner kernel launched just before this one wrote it.
  const bool own_plan = B <= kOwnPlanMax;
  int32_t* splan = reinterpret_cast<int32_t*>(gbase + T::kOffPlan);
  if (own_plan) {
    build_plan(p, splan, pre_pages);
    if (blockIdx.x == 0) {
      for (int i = threadIdx.x; i < B + 2; i += blockDim.x) plan_g[i] = splan[i];
      const int row_elems = QL * Hq * D;
      for (int b = 0; b < B; ++b) {
        const int L = p.context_lens[b];
        if (threadIdx.x == 0 && (L > p.max_context_len || L < QL)) record_error(p.err, kErrShortContext);
        if (L <= 0)  // no CTA visits a sequence without tokens: its rows are zeros
          for (int i = threadIdx.x; i < row_elems; i += blockDim.x)
            p.out[(size_t)b * row_elems + i] = __float2bfloat16(0.f);
      }
    }
  } else {
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  const int32_t* plan = own_plan ? splan : plan_g;
  const Range rg = cta_range(plan, Hkv, blockIdx.x, gridDim.x);
  if (threadIdx.x == 0) PA_TL_STAMP(1);

  // Lane half: TMEM lanes 32w..32w+31 belong to warps w and w+4 (one SM sub-partition each), so
  // one CTA of an SM keeps its query rows in lanes 0-63 (softmax on warps 0, 1) and the other in
  // lanes 64-127 (softmax on warps 2, 3): two co-resident CTAs then use all four sub-partitions.
  // The block scheduler fills every SM with one CTA of the first half of the grid before it
  // places the second, so the halves of the grid pair up per SM.
  // Warp w issues on sub-partition w % 4.  The producers sit on the sub-partitions of the other
  // CTA's softmax warps (E4M3 producers convert pages, about as much ALU work per step as a
  // softmax warp) and the MMA issuer, one thread, on warp 4: each sub-partition holds one softmax
  // and one producer warp.
  const int lh = blockIdx.x >= gridDim.x / 2 ? 1 : 0;
  const int w_issue = 4;            // MMA issuer
  const int w_kprod = lh ? 1 : 3;   // K producer
  const int w_vprod = lh ? 0 : 2;   // V producer
  const bool is_softmax = warp < 4 && (warp >> 1) == lh;
  const uint32_t row_shift = (uint32_t)lh * (T::kRows * 128);  // 64 rows: A operands start that much earlier

  const Seg sg0 = segment_at(plan, B, rg, rg.x0);
  if (rg.x0 < rg.x1 && sg0.p1 > sg0.p0) {  // the range holds at least one real page
    if (warp == w_kprod || warp == w_vprod) {
      if constexpr (FP8) {
        // ======== E4M3 producers: one warp per ring.  A bulk copy lands each fp8 page of a step in
        // the upper half of the step's f16 tile; once it has landed the warp reads its rows of the
        // step into registers, then writes them back as f16 (exact) in the 128-byte-swizzled
        // layout the MMAs read, zeroing the rows of pages without a block and of tokens past the
        // context or the segment, and marks the tile converted.  With head_dim 128 the K pages
        // need no conversion (Q.K^T runs on the E4M3 codes, kind::f8f6f4): the K warp copies them
        // with 2-D tensor boxes in the swizzled layout the MMA reads, and converts half of every V
        // tile (token rows 0-31) while the V warp copies the V pages and converts the other half.
        // Copies run up to a ring ahead of the conversions: the warp polls both sides, so neither
        // waits behind the other.
        const bool is_k = warp == w_kprod;
        const int nst = is_k ? T::kKStages : T::kVStages;            // the ring this warp copies into
        const uint32_t ring = is_k ? sK : sV;
        const uint32_t bar_full = is_k ? bar_kfull : bar_vfull;    // copied bytes landed
        const uint32_t bar_free = is_k ? bar_kempty : bar_vempty;  // QK / PV of the step nst before done
        const uint8_t* cache = is_k ? p.k_cache : p.v_cache;
        // the ring this warp converts, and its token rows [c_row0, c_row0 + c_rows)
        const bool conv_v = kKDirect || !is_k;
        const int c_nst = conv_v ? T::kVStages : T::kKStages;
        const uint32_t c_ring = conv_v ? sV : sK;
        const uint32_t c_full = conv_v ? bar_vfull : bar_kfull;
        const uint32_t c_ready = conv_v ? bar_vready : bar_kready;
        const int c_row0 = kKDirect && !is_k ? 32 : 0;
        constexpr int kCRows = kKDirect ? 32 : T::kStepTokens;
        constexpr int kPageFp8 = T::kBS * D;                 // bytes of one fp8 page
        constexpr int kStageFp8 = T::kTP * kPageFp8;         // one step: half the f16 tile
        constexpr int kCPR = D / 16;                         // 16-code chunks per token row
        constexpr int kPer = kCRows * kCPR / 32;             // chunks per lane per step
        static_assert(2 * kStageFp8 == T::kKTile, "fp8 step in the upper half of its f16 tile");
        const uint64_t kv_policy = l2_evict_first_policy();
        struct Walk {
          Seg sg;
          int pstep;
          bool done;
        };
        auto advance = [&](Walk& w) {
          w.pstep += T::kTP;
          if (w.pstep < w.sg.p1) return;
          const long long x = seg_end_x(w.sg, plan, rg);
          if (x >= rg.x1) { w.done = true; return; }
          w.sg = segment_at(plan, B, rg, x);
          w.pstep = w.sg.p0;
          if (w.sg.p1 <= w.sg.p0) w.done = true;
        };
        // lane pg < kTP: block id of page pg of the step (-1 for none)
        auto page_id = [&](const Walk& w, bool flag) {
          int v = -1;
          if (lane < T::kTP && w.pstep + lane < w.sg.p1) {
            v = p.block_table[(size_t)w.sg.b * p.max_blocks_per_seq + w.pstep + lane];
            if (v < 0 || v >= p.num_blocks) {
              if (flag) record_error(p.err, kErrBlockId);
              v = -1;
            }
          }
          return v;
        };
        Walk wc{sg0, sg0.p0, false};  // copies
        Walk wv = wc;                 // conversions
        int gi = 0, gc = 0;           // steps copied, steps converted
        uint32_t idle = 0;
        while (!wv.done || !wc.done) {
          bool progressed = false;
          // (a) copy the next step's pages once its stage is free (and, when this warp converts
          // its own ring, no more than a ring ahead of the conversions)
          if (!wc.done && (gi < gc + nst || (kKDirect && is_k))) {
            bool free_ok = gi < nst;
            if (!free_ok && lane == 0)
              free_ok = mbar_test_wait(bar_free + 8 * ((gi - nst) % nst), ((gi - nst) / nst) & 1);
            if (__shfl_sync(0xffffffffu, free_ok, 0)) {
              const int v = page_id(wc, is_k);
              int pbs[T::kTP];
#pragma unroll
              for (int pg = 0; pg < T::kTP; ++pg) pbs[pg] = __shfl_sync(0xffffffffu, v, pg);
              if (lane == 0) {
                const int st = gi % nst;
                const uint32_t bar = bar_full + 8 * st;
                int npg = 0;
#pragma unroll
                for (int pg = 0; pg < T::kTP; ++pg) npg += pbs[pg] >= 0;
                if (npg == 0) {
                  mbar_arrive(bar);
                } else if (kKDirect && is_k) {
                  // E4M3 K pages as 16 x 128-byte boxes, 128-byte swizzle: the MMA's K-major layout
                  const uint32_t dst = ring + st * T::kKTile;
                  mbar_arrive_expect_tx(bar, npg * kPageFp8);
#pragma unroll
                  for (int pg = 0; pg < T::kTP; ++pg)
                    if (pbs[pg] >= 0)
                      tma_load_2d_hint(dst + pg * kPageFp8, &tmk, 0, (pbs[pg] * Hkv + wc.sg.g) * T::kBS, bar,
                                       kv_policy);
                } else {
                  const uint32_t dst = ring + st * T::kKTile + kStageFp8;
                  mbar_arrive_expect_tx(bar, npg * kPageFp8);
#pragma unroll
                  for (int pg = 0; pg < T::kTP; ++pg)
                    if (pbs[pg] >= 0) {
                      const uint8_t* src = cache + ((size_t)pbs[pg] * Hkv + wc.sg.g) * kPageFp8;
                      if (kKvEvictFirst)
                        bulk_copy_g2s_hint(dst + pg * kPageFp8, src, kPageFp8, bar, kv_policy);
                      else
                        bulk_copy_g2s(dst + pg * kPageFp8, src, kPageFp8, bar);
                    }
                }
              }
              if (lane == 0) PA_ST(gi, is_k ? kStKCopy : kStVCopy);
              ++gi;
              advance(wc);
              progressed = true;
            }
          }
          // (b) convert this warp's rows of the oldest unconverted step once its bytes have landed
          // (a step of the ring this warp does not copy has landed once its full barrier's phase
          // completed: the copying warp cannot be a phase ahead before this warp converted it)
          if (!wv.done && (gc < gi || (kKDirect && is_k))) {
            bool landed = false;
            if (lane == 0) landed = mbar_test_wait(c_full + 8 * (gc % c_nst), (gc / c_nst) & 1);
            if (__shfl_sync(0xffffffffu, landed, 0)) {
              if (lane == 0 && !is_k) PA_ST(gc, kStVLanded);
              const uint32_t tile = c_ring + (gc % c_nst) * T::kKTile;
              const uint32_t src = tile + kStageFp8;
              const unsigned okm = __ballot_sync(0xffffffffu, page_id(wv, false) >= 0) & ((1u << T::kTP) - 1u);
              const int L = context_len(p, wv.sg.b, false);
              const int rows_ok = min(L, wv.sg.p1 * T::kBS) - wv.pstep * T::kBS;  // token rows [0, rows_ok)
              // batches of 32 * kBatch chunks: a batch holds whole token rows, and the f16 write of
              // row t lands on the E4M3 bytes of row t only, so reading the batch before writing it
              // (the warp-wide barrier below) keeps every later batch's bytes intact
              constexpr int kBatch = kPer >= 4 ? kPer / 4 : 1;
#pragma unroll 1
              for (int i0 = 0; i0 < kPer; i0 += kBatch) {
                uint4 code[kBatch];
#pragma unroll
                for (int ii = 0; ii < kBatch; ++ii) {
                  const int q = lane + 32 * (i0 + ii), tr = c_row0 + q / kCPR, dc = q % kCPR;
                  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                               : "=r"(code[ii].x), "=r"(code[ii].y), "=r"(code[ii].z), "=r"(code[ii].w)
                               : "r"(src + tr * D + dc * 16)
                               : "memory");
                }
                __syncwarp();  // the batch's rows are in registers before any f16 row overwrites them
#pragma unroll
                for (int ii = 0; ii < kBatch; ++ii) {
                  const int q = lane + 32 * (i0 + ii), tr = c_row0 + q / kCPR, dc = q % kCPR;
                  const bool keep = ((okm >> (tr / T::kBS)) & 1u) && tr < rows_ok;
                  const uint32_t c4[4] = {keep ? code[ii].x : 0u, keep ? code[ii].y : 0u, keep ? code[ii].z : 0u,
                                          keep ? code[ii].w : 0u};
                  uint32_t h[8];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    h[2 * j] = e4m3x2_to_f16x2(c4[j]);
                    h[2 * j + 1] = e4m3x2_to_f16x2(c4[j] >> 16);
                  }
                  // dims [16 dc, 16 dc + 16): half dc / 4, 16-byte chunks 2 (dc % 4) and the next
                  const uint32_t row = tile + (dc >> 2) * T::kRegion + tr * 128;
                  const int c8 = (dc & 3) * 2;
                  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c8 ^ (tr & 7)) << 4)),
                               "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                               : "memory");
                  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((c8 + 1) ^ (tr & 7)) << 4)),
                               "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                               : "memory");
                }
                __syncwarp();
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(c_ready + 8 * (gc % c_nst));
              if (lane == 0) PA_ST(gc, is_k ? kStConvK : kStConvV);
              ++gc;
              advance(wv);
              progressed = true;
            }
          }
          if (progressed) {
            idle = 0;
          } else if (++idle >= kSpinLimit || ((idle & 1023u) == 0 && *abort_flag)) {
            if (lane == 0) {
              if (!*abort_flag) record_error(p.err, kErrTimeout);
              *abort_flag = 1u;
            }
            break;
          } else if (kProducerBackoffNs > 0) {
            __nanosleep(kProducerBackoffNs);  // nothing to do yet: leave the issue slots to the softmax
          }
        }
        // every copy this warp started has landed before the CTA's shared memory can go away
        if (lane == 0)
          for (int k = max(0, gi - nst); k < gi; ++k) mbar_wait(bar_full + 8 * (k % nst), (k / nst) & 1);
        __syncwarp();
      } else {
        // ======== TMA producers: one warp fills the K ring (2 stages), the other the V ring (3) =====
        const bool is_k = warp == w_kprod;
        const CUtensorMap* map = is_k ? &tmk : &tmv;
        const int nst = is_k ? T::kKStages : T::kVStages;
        const uint32_t ring = is_k ? sK : sV;
        const uint32_t bar_full = is_k ? bar_kfull : bar_vfull;
        // a stage is free once QK (K tile) or PV (V tile) of the step nst before has completed
        const uint32_t bar_free = is_k ? bar_kempty : bar_vempty;
        int gs = 0;  // steps started, over all segments
        bool alive = true;
        const uint64_t kv_policy = l2_evict_first_policy();
        for (long long x = rg.x0; alive && x < rg.x1;) {
          const Seg sg = segment_at(plan, B, rg, x);
          x = seg_end_x(sg, plan, rg);
          if (sg.p1 <= sg.p0) break;  // the range ended inside the next segment's header
          const int32_t* bt = p.block_table + (size_t)sg.b * p.max_blocks_per_seq;
          // block ids of 32 pages per lane-load: `cur` holds pages [cbase, cbase + 32)
          auto load_ids = [&](int pbase) {
            const int pg = pbase + lane;
            int v = -1;
            if (pg < sg.p1) {
              v = bt[pg];
              if (v < 0 || v >= p.num_blocks) {
                if (is_k) record_error(p.err, kErrBlockId);
                v = -1;
              }
            }
            return v;
          };
          int cbase = sg.p0;
          int cur = load_ids(cbase);
          int nxt = load_ids(cbase + 32);
          for (int pstep = sg.p0; pstep < sg.p1; pstep += T::kTP, ++gs) {
            if (pstep >= cbase + 32) {
              cbase += 32;
              cur = nxt;
              nxt = load_ids(cbase + 32);
            }
            int pbs[T::kTP];
            int npg = 0;
            uint32_t okbits = 0;
  #pragma unroll
            for (int pg = 0; pg < T::kTP; ++pg) {
              pbs[pg] = __shfl_sync(0xffffffffu, cur, (pstep - cbase + pg) & 31);
              // pages of the step past the 32-page window come from the next window
              if (pstep - cbase + pg >= 32) pbs[pg] = __shfl_sync(0xffffffffu, nxt, (pstep - cbase + pg) & 31);
              if (pstep + pg >= sg.p1) pbs[pg] = -1;
              npg += pbs[pg] >= 0;
              okbits |= (pbs[pg] >= 0 ? 1u : 0u) << pg;
            }
            if (lane == 0) {
              bool ready = true;
              if (gs >= nst)
                ready = wait_or_abort(bar_free + 8 * ((gs - nst) % nst), ((gs - nst) / nst) & 1, abort_flag, p.err);
              if (!ready) {
                alive = false;
              } else {
                const int s = gs % nst;
                const uint32_t region = ring + s * T::kKTile;
                const uint32_t bar = bar_full + 8 * s;
                if (npg == 0) {
                  mbar_arrive(bar);
                } else {
                  mbar_arrive_expect_tx(bar, npg * T::kHalves * T::kBoxBytes);
  #pragma unroll
                  for (int pg = 0; pg < T::kTP; ++pg) {
                    if (pbs[pg] < 0) continue;
                    const int row = (pbs[pg] * Hkv + sg.g) * T::kBS;
  #pragma unroll
                    for (int hh = 0; hh < T::kHalves; ++hh) {
                      if (kKvEvictFirst)
                        tma_load_2d_hint(region + hh * T::kRegion + pg * T::kBoxBytes, map, hh * 64, row, bar, kv_policy);
                      else
                        tma_load_2d(region + hh * T::kRegion + pg * T::kBoxBytes, map, hh * 64, row, bar);
                    }
                  }
                }
                if (is_k) {  // the step's page record for the softmax: pages holding a block
                  srec[gs % T::kRecSlots] = okbits;
                  mbar_arrive(bar_rec + 8 * (gs % T::kRecSlots));
                }
              }
            }
            if (lane == 0) PA_ST(gs, is_k ? kStKCopy : kStVCopy);
            alive = __shfl_sync(0xffffffffu, alive, 0);
            if (!alive) break;
          }
        }
        // every copy started has landed before the CTA's shared memory can go away
        if (lane == 0)
          for (int k = max(0, gs - nst); k < gs; ++k) mbar_wait(bar_full + 8 * (k % nst), (k / nst) & 1);
        __syncwarp();
      }
    } else if (warp == w_issue) {
      // ======================= MMA issuer ====================================================
      if (lane == 0) {
        auto mma_qk = [&](int st) {
          const uint32_t kreg = sK + (st & 1) * T::kKTile;
          if constexpr (kKDirect) {
            // S = Q_hi . K^T + Q_lo . K^T on E4M3 operands: each token row of K is one 128-byte
            // swizzled row (128 codes), 32 codes per instruction; Q_hi and Q_lo are 64-row E4M3
            // tiles one Q half apart
#pragma unroll
            for (int term = 0; term < 2; ++term)
#pragma unroll
              for (int kk = 0; kk < D / 32; ++kk)
                umma_f8(tS_of(st), smem_desc(sQ + term * (T::kRows * 128) + kk * 32 - row_shift, 16, 1024),
                        smem_desc(kreg + kk * 32, 16, 1024), T::kIdescQK16, (term > 0 || kk > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = (kk >> 2) * T::kRegion + (kk & 3) * 32;
              const uint32_t qoff = (kk >> 2) * (T::kRows * 128) + (kk & 3) * 32;
              umma_bf16(tS_of(st), smem_desc(sQ + qoff - row_shift, 16, 1024), smem_desc(kreg + koff, 16, 1024),
                        FP8 ? T::kIdescQK16 : T::kIdescQK, kk > 0 ? 1u : 0u);
            }
          }
          umma_commit(bar_s_ready + 8 * (st & 1));
          umma_commit(bar_kempty + 8 * (st & 1));
        };
        auto mma_pv = [&](int st, bool first) {
          const uint32_t vreg = sV + (st % T::kVStages) * T::kKTile;
#pragma unroll
          for (int kk = 0; kk < T::kStepTokens / 16; ++kk) {
            // A = P in tensor memory (16 tokens = 8 columns of bf16 pairs, all 128 lanes; the
            // lanes of the other half hold padding rows); B = V (MN-major: 64-dim atoms one half
            // region apart, 8-token groups 1024 B apart, 16 tokens = 2048 B per step)
            umma_bf16_tmem_a(tO, tS_of(st) + kk * 8, smem_desc(vreg + kk * 2048, T::kRegion, 1024),
                             FP8 ? T::kIdescPV16 : T::kIdescPV, (!first || kk > 0) ? 1u : 0u);
          }
          umma_commit(bar_o_done + 8 * (st & 1));
          umma_commit(bar_vempty + 8 * (st % T::kVStages));
        };
        // QK and PV each walk the segments; whichever is ready first is issued first
        long long xq = rg.x0, xp = rg.x0;   // segment starts of the two walkers
        Seg sq = segment_at(plan, B, rg, xq), sv = sq;
        int q_seg = 0, v_seg = 0;            // segment indices
        int q_step = 0, v_step = 0;          // step within the segment
        int gq = 0, gp = 0;                  // global step numbers
        bool q_done = false, v_done = false;
        uint32_t idle = 0;
        while (!v_done) {
          bool progressed = false;
          if (!q_done) {
            const bool first = q_step == 0;
            if (mbar_test_wait((FP8 && !kKDirect ? bar_kready : bar_kfull) + 8 * (gq & 1), (gq >> 1) & 1) &&
                (gq < 2 || mbar_test_wait(bar_o_done + 8 * (gq & 1), ((gq - 2) >> 1) & 1)) &&
                (!first || mbar_test_wait(bar_q_ready, q_seg & 1))) {
              tc_fence_after();
              mma_qk(gq);
              PA_ST(gq, kStQK);
              ++gq;
              progressed = true;
              if (sq.p0 + (++q_step) * T::kTP >= sq.p1) {
                xq = seg_end_x(sq, plan, rg);
                q_step = 0;
                ++q_seg;
                if (xq < rg.x1) sq = segment_at(plan, B, rg, xq);
                if (xq >= rg.x1 || sq.p1 <= sq.p0) q_done = true;
              }
            }
          }
          if (gp < gq) {
            const bool first = v_step == 0;
            if (mbar_test_wait(bar_p_ready + 8 * (gp & 1), (gp >> 1) & 1) &&
                mbar_test_wait((FP8 ? bar_vready : bar_vfull) + 8 * (gp % T::kVStages), (gp / T::kVStages) & 1) &&
                (!first || v_seg == 0 || mbar_test_wait(bar_o_free, (v_seg - 1) & 1))) {
              tc_fence_after();
              mma_pv(gp, first);
              PA_ST(gp, kStPV);
              ++gp;
              progressed = true;
              if (sv.p0 + (++v_step) * T::kTP >= sv.p1) {
                xp = seg_end_x(sv, plan, rg);
                v_step = 0;
                ++v_seg;
                if (xp < rg.x1) sv = segment_at(plan, B, rg, xp);
                if (xp >= rg.x1 || sv.p1 <= sv.p0) v_done = true;
              }
            }
          }
          if (progressed) {
            idle = 0;
          } else if (++idle >= kSpinLimit || ((idle & 1023u) == 0 && *abort_flag)) {
            if (!*abort_flag) record_error(p.err, kErrTimeout);
            *abort_flag = 1u;
            break;
          }
        }
        // every MMA this thread issued has completed before tensor memory is released
        umma_commit(bar_final);
        mbar_wait(bar_final, 0);
      }
      __syncwarp();
    } else if (is_softmax) {
      // ======================= softmax warps: thread r owns query row r =====================
      const int r = threadIdx.x - 64 * lh;
      const bool row_live = r < R;
      const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
      const int ri = r / G, rh = r - (r / G) * G;  // query index and head within the group
      // Q row r of segment sg (zeros for padding rows) as K-major 128-byte-swizzled rows.  E4M3:
      // f16 products, the row scaled by a power of two 2^k first (f16_prescale_exp: exact, no
      // overflow for any bf16 q); returns 2^-k, the factor of the row's scores (1 for bf16).
      auto write_q = [&](const Seg& sg) -> float {
        const __nv_bfloat16* qrow = nullptr;
        if (row_live) qrow = p.q + (((size_t)sg.b * QL + ri) * Hq + sg.g * G + rh) * D;
        float up = 1.f, qdiv = 1.f;
        if constexpr (FP8) {
          uint32_t emax = 0;
          if (qrow)
#pragma unroll 4
            for (int c = 0; c < D / 8; ++c) emax = max(emax, bf16x8_max_exp(*reinterpret_cast<const uint4*>(qrow + c * 8)));
          const int kq = kKDirect ? e4m3_prescale_exp(emax) : f16_prescale_exp(emax);
          up = exp2_int(kq);
          qdiv = exp2_int(-kq);
        }
        if constexpr (kKDirect) {
          // Q row r as two E4M3 terms, hi = e4m3(q 2^k) and lo = e4m3(q 2^k - hi), each a
          // K-major 128-byte swizzled row of 128 codes (16-byte chunk c = dims 16c .. 16c + 15)
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint4 a = make_uint4(0u, 0u, 0u, 0u), b2 = a;
            if (qrow) {
              a = *reinterpret_cast<const uint4*>(qrow + c * 16);
              b2 = *reinterpret_cast<const uint4*>(qrow + c * 16 + 8);
            }
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 x0 = bf16x2_to_f2(w[2 * j]), x1 = bf16x2_to_f2(w[2 * j + 1]);
              const float v0 = x0.x * up, v1 = x0.y * up, v2 = x1.x * up, v3 = x1.y * up;
              const uint32_t h01 = f32x2_to_e4m3x2(v0, v1), h23 = f32x2_to_e4m3x2(v2, v3);
              const float2 d01 = e4m3x2_to_f2((uint16_t)h01), d23 = e4m3x2_to_f2((uint16_t)h23);
              const uint32_t l01 = f32x2_to_e4m3x2(v0 - d01.x, v1 - d01.y), l23 = f32x2_to_e4m3x2(v2 - d23.x, v3 - d23.y);
              hi[j] = h01 | (h23 << 16);
              lo[j] = l01 | (l23 << 16);
            }
            const uint32_t off = r * 128 + (((uint32_t)c ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sQ + off), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]),
                         "r"(hi[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sQ + T::kRows * 128 + off), "r"(lo[0]),
                         "r"(lo[1]), "r"(lo[2]), "r"(lo[3])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_q_ready);
          return qdiv;
        }
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (qrow) v = *reinterpret_cast<const uint4*>(qrow + c * 8);
          if constexpr (FP8) {
            const float2 a = bf16x2_to_f2(v.x), b2 = bf16x2_to_f2(v.y), c2 = bf16x2_to_f2(v.z), d2 = bf16x2_to_f2(v.w);
            v = make_uint4(pack_f16(a.x * up, a.y * up), pack_f16(b2.x * up, b2.y * up), pack_f16(c2.x * up, c2.y * up),
                           pack_f16(d2.x * up, d2.y * up));
          }
          const uint32_t dst = sQ + (c >> 3) * (T::kRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_q_ready);
        return qdiv;
      };
      // E4M3: pages of a step that hold usable data (bit per page) and their K and V scales, loaded
      // a step ahead (bf16 steps read the page record the K producer wrote)
      auto step_pages_ok = [&](const Seg& sg, int pstep, float (&ksc)[T::kTP], float (&vsc)[T::kTP]) {
        const int32_t* bt = p.block_table + (size_t)sg.b * p.max_blocks_per_seq;
        unsigned okp = 0;
#pragma unroll
        for (int pg = 0; pg < T::kTP; ++pg) {
          ksc[pg] = 0.f;
          vsc[pg] = 0.f;
          if (pstep + pg < sg.p1) {
            const int pb = bt[pstep + pg];
            if (pb >= 0 && pb < p.num_blocks) {
              okp |= 1u << pg;
              if constexpr (FP8) {
                ksc[pg] = p.k_scale[(size_t)pb * Hkv + sg.g];
                vsc[pg] = p.v_scale[(size_t)pb * Hkv + sg.g];
              }
            }
          }
        }
        return okp;
      };

      bool ok = true;
      int gs = 0;     // global step
      int seg = 0;    // segment index
      Seg sg = segment_at(plan, B, rg, rg.x0);
      float qdiv_next = write_q(sg);
      float ks_next[T::kTP] = {}, vs_next[T::kTP] = {};
      unsigned pok_next = 0;
      if constexpr (FP8) pok_next = step_pages_ok(sg, sg.p0, ks_next, vs_next);
      while (ok) {
        const int L = context_len(p, sg.b, false);
        const int first_new = L - QL;  // the q_len new tokens start here
        // new tokens this row sees: bits 0..ri (causal) or its tree-ancestor mask
        const uint32_t mrow =
            row_live ? (p.tree_mask ? p.tree_mask[(size_t)sg.b * QL + ri] : ((2u << ri) - 1u)) : 0u;
        const int limit_tok = min(L, sg.p1 * T::kBS);    // tokens of this segment end here
        const long long xnext = seg_end_x(sg, plan, rg);
        const Seg sg_next = xnext < rg.x1 ? segment_at(plan, B, rg, xnext) : sg;
        const bool has_next = xnext < rg.x1 && sg_next.p1 > sg_next.p0;
        float m_used = -INFINITY, l = 0.f;
        const float qdiv = qdiv_next;  // 2^-k of this segment's Q row (E4M3)
        for (int pstep = sg.p0; pstep < sg.p1; pstep += T::kTP, ++gs) {
          const bool last = pstep + T::kTP >= sg.p1;
          const uint32_t tS = tS_of(gs) + lane_off;
          if (!(ok = wait_or_abort(bar_s_ready + 8 * (gs & 1), (gs >> 1) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          unsigned pok = pok_next;
          float ksc[T::kTP], vsc[T::kTP];
#pragma unroll
          for (int pg = 0; pg < T::kTP; ++pg) {
            ksc[pg] = ks_next[pg];
            vsc[pg] = vs_next[pg];
          }
          if constexpr (!FP8) {
            // the step's page record (written by the K producer when it copied the step's K pages)
            if (!(ok = wait_or_abort(bar_rec + 8 * (gs % T::kRecSlots), (gs / T::kRecSlots) & 1, abort_flag, p.err)))
              break;
            pok = srec[gs % T::kRecSlots];
          }
          if (gs == 0 && r == 0) PA_TL_STAMP(2);
          if (r == 0) PA_ST(gs, kStS);
          float s[T::kStepTokens];
          {
            uint32_t raw64[64];
            tmem_ld_x64(tS, raw64);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(raw64[c]);
          }
          // S of the segment's last step is out: QK of this segment is over, the Q buffer is free
          if (last && has_next) qdiv_next = write_q(sg_next);
          if constexpr (FP8) {
            if (!last) pok_next = step_pages_ok(sg, pstep + T::kTP, ks_next, vs_next);
            else if (has_next) pok_next = step_pages_ok(sg_next, sg_next.p0, ks_next, vs_next);
          }

          const int tok0 = pstep * T::kBS;
          // visibility of the step's 64 tokens as one word: context tokens up to the segment end,
          // the new tokens of this row's mask, pages that hold data.  Built once per step, so the
          // per-score test is a constant bit test; an all-ones word (interior steps) skips it.
          uint64_t vis = low_bits64(min(limit_tok, first_new) - tok0);
          {
            const int sh = first_new - tok0;  // step position of new token 0
            uint64_t nb = 0;
            if (sh >= 0 && sh < 64) nb = (uint64_t)mrow << sh;
            else if (sh < 0 && sh > -32) nb = (uint64_t)(mrow >> -sh);
            vis |= nb & low_bits64(limit_tok - tok0);
            uint64_t pm = 0;
#pragma unroll
            for (int pg = 0; pg < T::kTP; ++pg)
              if ((pok >> pg) & 1u) pm |= 0xffffull << (16 * pg);
            vis &= pm;
          }
          // Full steps with a positive scale stay in raw scores (row max before scaling, the scale
          // folded into one packed FMA per pair); masked steps scale first and mask with -inf.
          // Padding rows see nothing (their P is 0; they are never stored).
          if (!row_live) vis = 0;
          const bool raw = !FP8 && vis == ~0ull && p.scale_log2 > 0.f;
          float mxs[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) mxs[j] = -INFINITY;
          if (raw) {
#pragma unroll
            for (int c = 0; c < T::kStepTokens; ++c) mxs[c & 7] = fmaxf(mxs[c & 7], s[c]);
          } else {
            const uint32_t v0 = (uint32_t)vis, v1 = (uint32_t)(vis >> 32);
            // E4M3: each page's scores carry its K scale (and the Q row's 2^-k)
            float kmul[T::kTP];
#pragma unroll
            for (int pg = 0; pg < T::kTP; ++pg) kmul[pg] = FP8 ? ksc[pg] * qdiv * p.scale_log2 : p.scale_log2;
#pragma unroll
            for (int c = 0; c < T::kStepTokens; ++c) {
              const bool v = (((c < 32 ? v0 : v1) >> (c & 31)) & 1u) != 0;
              s[c] = v ? s[c] * kmul[c / T::kBS] : -INFINITY;
              mxs[c & 7] = fmaxf(mxs[c & 7], s[c]);
            }
          }
          float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                           fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
          if (raw) mx *= p.scale_log2;
          const float m_new = fmaxf(m_used, mx);
          const bool need = row_live && (m_used != -INFINITY) && (m_new > m_used + 8.f);

          if (__any_sync(0xffffffffu, need)) {
            // the O row is rescaled only once PV(gs - 1) has landed in it
            if (!(ok = wait_or_abort(bar_o_done + 8 * ((gs - 1) & 1), ((gs - 1) >> 1) & 1, abort_flag, p.err)))
              break;
            tc_fence_after();
            const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t raw[32];
              tmem_ld_x32(tO + lane_off + c0, raw);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) raw[c] = __float_as_uint(__uint_as_float(raw[c]) * alpha);
              tmem_st_x32(tO + lane_off + c0, raw);
            }
            tmem_wait_st();
            l *= alpha;
          }
          if (need || m_used == -INFINITY) m_used = m_new;
          const float basev = m_used == -INFINITY ? 0.f : m_used;

          // zero V rows of tokens that hold no data (block tails, stale stages): P is 0 there,
          // but 0 * NaN would still poison the product.  Thread r handles token r of the step,
          // after the step's V tile has landed.  (E4M3 tiles come zeroed from the conversion.)
          if constexpr (!FP8) {
            const int tok = tok0 + r;
            const bool tok_ok = ((pok >> (r >> 4)) & 1u) && tok < limit_tok;
            if (__any_sync(0xffffffffu, !tok_ok)) {
              if (!(ok = wait_or_abort(bar_vfull + 8 * (gs % T::kVStages), (gs / T::kVStages) & 1, abort_flag,
                                       p.err)))
                break;
              if (!tok_ok) {
                const uint32_t vrow = sV + (gs % T::kVStages) * T::kKTile + r * 128;
#pragma unroll
                for (int hh = 0; hh < T::kHalves; ++hh)
#pragma unroll
                  for (int c = 0; c < 8; ++c)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + hh * T::kRegion + c * 16),
                                 "r"(0u)
                                 : "memory");
              }
            }
          }
          // P row r as bf16 pairs over the first 32 columns of this step's S buffer; the V rows
          // zeroed above reach the MMA through the fence below
          uint32_t w[32];
          float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
          const float2 one2 = make_float2(1.f, 1.f);
          const float2 sc2 = raw ? make_float2(p.scale_log2, p.scale_log2) : one2;
          const float2 nb2 = make_float2(-basev, -basev);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sc2, nb2);
            const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            if constexpr (FP8) {  // f16 P carries each page's V scale; l sums the plain weights
              acc[c & 3] = ffma2(e, one2, acc[c & 3]);
              const float vm = vsc[(2 * c) / T::kBS];
              w[c] = pack_f16(e.x * vm, e.y * vm);
            } else {
              // l sums the bf16-rounded weights that P.V multiplies, so the row is normalised by
              // the sum of its own weights (the rounding then moves weight between tokens only)
              w[c] = pack_bf16(e.x, e.y);
              acc[c & 3] = add_bf16x2_f2(w[c], acc[c & 3]);
            }
          }
          l += ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
          tmem_st_x32(tS, w);
          tmem_wait_st();
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_p_ready + 8 * (gs & 1));
          if (r == 0) PA_ST(gs, kStP0);
          if (r == 32) PA_ST(gs, kStP1);
        }
        if (!ok) break;

        // ---- segment epilogue: O row / l, then release O to the next segment -------------
        const int gl = gs - 1;  // this segment's last step
        if (!(ok = wait_or_abort(bar_o_done + 8 * (gl & 1), (gl >> 1) & 1, abort_flag, p.err))) break;
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t orow = ((size_t)sg.b * QL + ri) * Hq + sg.g * G + rh;
        // partial slot of this segment (see the header): rows of kv head g, sequence b, CTA c
        const size_t slot = (size_t)sg.g * B + sg.b + blockIdx.x;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t raw[32];
          tmem_ld_x32(tO + lane_off + c0, raw);
          tmem_wait_ld();
          if (!row_live) continue;
          if (sg.whole) {
            __nv_bfloat16* dst = p.out + orow * D + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(raw[c + 0]) * inv, __uint_as_float(raw[c + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(raw[c + 2]) * inv, __uint_as_float(raw[c + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(raw[c + 4]) * inv, __uint_as_float(raw[c + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(raw[c + 6]) * inv, __uint_as_float(raw[c + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + c) = v;
            }
          } else {
            float* dst = p.part_o + (slot * R + r) * D + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(dst + c) =
                  make_float4(__uint_as_float(raw[c]) * inv, __uint_as_float(raw[c + 1]) * inv,
                              __uint_as_float(raw[c + 2]) * inv, __uint_as_float(raw[c + 3]) * inv);
          }
        }
        if (row_live && !sg.whole) p.part_lse[slot * R + r] = (l > 0.f) ? m_used + __log2f(l) : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_o_free);  // O is read out: the next segment may overwrite it

        if (!has_next) break;
        sg = sg_next;
        ++seg;
      }
      if (r == 0) {
        PA_TL_STAMP(3);
        PA_TL_VALUE(5, seg + 1);
        PA_TL_VALUE(6, gs);
      }
    }
  }

  // the merge kernel (launched as a programmatic dependent) may start its prologue now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T::kTmemCols) : "memory");
  }
  if (threadIdx.x == 0) PA_TL_STAMP(7);
}

// TP and the exclusive prefix of page counts of the (clamped) contexts: plan[0] = TP,
// plan[1 + b] = first page of sequence b, plan[1 + B] = TP.  One CTA of 1024 threads.
template <int D>
__global__ void __launch_bounds__(1024) verify_plan_kernel(const AttnParams p, int32_t* plan) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  __shared__ int empty_seqs[1024];
  __shared__ int n_empty;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row_elems = p.q_len * p.num_q_heads * D;
  if (tid == 0) carry = 0;
  if (tid == 0) n_empty = 0;
  __syncthreads();
  for (int base = 0; base < p.num_seqs; base += 1024) {
    const int b = base + tid;
    int pages = 0;
    if (b < p.num_seqs) {
      int L = p.context_lens[b];
      if (L > p.max_context_len) {
        record_error(p.err, kErrShortContext);
        L = p.max_context_len;
      }
      if (L < p.q_len) record_error(p.err, kErrShortContext);  // some row sees no token
      pages = L > 0 ? (L + 15) / 16 + kSegCost : 0;  // real pages plus the segment's header
      if (L <= 0) empty_seqs[atomicAdd(&n_empty, 1)] = b;
    }
    // block-wide inclusive scan
    int v = pages;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += t;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = v + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    if (b < p.num_seqs) plan[1 + b] = incl - pages;
    __syncthreads();
    if (tid == 1023) carry = incl;
    __syncthreads();
    // rows of sequences without any token: zeros (no CTA of the attention kernel visits them)
    for (int e = 0; e < n_empty; ++e)
      for (int i = tid; i < row_elems; i += 1024) p.out[(size_t)empty_seqs[e] * row_elems + i] = __float2bfloat16(0.f);
    __syncthreads();
    if (tid == 0) n_empty = 0;
    __syncthreads();
  }
  if (tid == 0) {
    plan[0] = carry;
    plan[1 + p.num_seqs] = carry;
  }

  // the verify kernel (launched as a programmatic dependent) waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Combine the pieces of each (sequence, row) split over several CTAs.  One warp per (sequence,
// query index, query head); the pieces are the partial slots g * B + b + c of the CTAs c whose
// ranges meet the sequence.
template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) verify_merge_kernel(const AttnParams p,
                                                                        const int32_t* __restrict__ plan, int ncta) {
  constexpr int kDPL = D / 32;
  __shared__ int32_t own[kOwnPlanMax + 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.num_q_heads, Hkv = p.num_kv_heads, G = Hq / Hkv, QL = p.q_len, R = G * QL;
  const long long rows = (long long)p.num_seqs * QL * Hq;
  const long long row = (long long)blockIdx.x * kMergeWarps + warp;
  // Up to kOwnPlanMax sequences the CTA rebuilds the plan from context_lens -- an input, so this
  // runs before the verify kernel ends and only the pieces are read after the wait; beyond that,
  // the planner kernel's copy is read after the wait.
  const bool own_plan = p.num_seqs <= kOwnPlanMax;
  if (own_plan) build_plan(p, own, -1);  // every thread of the CTA takes part
  if (row >= rows) return;
  const int h = (int)(row % Hq);
  const int i = (int)((row / Hq) % QL);
  const int b = (int)(row / ((long long)Hq * QL));
  const int g = h / G;
  const int rr = i * G + (h - g * G);  // row within the kv head's group
  if (!own_plan) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (own_plan) plan = own;
  const long long TP = plan[0];
  if (plan[2 + b] <= plan[1 + b]) return;  // the planner zeroed the rows of empty sequences
  const int sb = plan[1 + b] + kSegCost, npages = plan[2 + b] - sb;  // real pages of (g, b)
  const long long Ttot = TP * Hkv;
  const long long x0 = (long long)g * TP + sb;
  const int c0 = cta_of(x0, Ttot, ncta), c1 = cta_of(x0 + npages - 1, Ttot, ncta);
  if (c0 == c1) return;  // one segment held the whole sequence and wrote the row
  if (own_plan) asm volatile("griddepcontrol.wait;" ::: "memory");  // the pieces come from the verify kernel
  // with at least one page per CTA every CTA in [c0, c1] holds a piece; otherwise skip the empty
  const bool every_cta = every_range_nonempty(Ttot, ncta);
  auto has_piece = [&](int c) { return every_cta || range_start(c, Ttot, ncta) < range_start(c + 1, Ttot, ncta); };
  const size_t slot0 = (size_t)g * p.num_seqs + b;
  // one pass, four pieces per turn with their loads issued together; the running maximum M
  // rescales what was summed before it grew (log-sum-exp rule)
  float M = -INFINITY, wsum = 0.f;
  float acc[kDPL];
#pragma unroll
  for (int e = 0; e < kDPL; ++e) acc[e] = 0.f;
  for (int cb = c0; cb <= c1; cb += 4) {
    float lse[4];
    float vv[4][kDPL];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = cb + k;
      const bool valid = c <= c1 && has_piece(c);
      const size_t rix = (slot0 + (valid ? c : c0)) * R + rr;
      lse[k] = valid ? p.part_lse[rix] : -INFINITY;
      const float* src = p.part_o + rix * D + lane * kDPL;
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
    for (int k = 0; k < 4; ++k) mb = fmaxf(mb, lse[k]);
    if (mb == -INFINITY) continue;  // nothing with mass yet
    const float alpha = M == -INFINITY ? 0.f : fast_exp2(M - mb);
    wsum *= alpha;
#pragma unroll
    for (int e = 0; e < kDPL; ++e) acc[e] *= alpha;
    M = mb;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float w = lse[k] == -INFINITY ? 0.f : fast_exp2(lse[k] - M);
      wsum += w;
#pragma unroll
      for (int e = 0; e < kDPL; ++e) acc[e] += w * vv[k][e];
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = p.out + row * D + lane * kDPL;
#pragma unroll
  for (int e = 0; e < kDPL; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
#ifdef PA_TIMELINE
  if (lane == 0) atomicMax(&g_verify_merge_end, tl_now());
#endif
}

template <int D, bool FP8>
cudaError_t launch_d(const AttnParams& p, int32_t* plan, int ncta, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t st) {
  using T = TcTraits<D>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(verify_tc_kernel<D, FP8>), T::kSmem);
  if (e != cudaSuccess) return e;
  const bool own_plan = p.num_seqs <= kOwnPlanMax;
  if (!own_plan) {
    verify_plan_kernel<D><<<1, 1024, 0, st>>>(p, plan);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    AttnParams pp = p;
    int32_t* gplan = plan;
    CUtensorMap k = tk, v = tv;
    void* args[] = {&pp, &gplan, &k, &v};
    e = own_plan ? cudaLaunchKernel(reinterpret_cast<const void*>(verify_tc_kernel<D, FP8>), dim3(ncta),
                                    dim3(T::kThreads), args, T::kSmem, st)
                 : launch_pdl(reinterpret_cast<const void*>(verify_tc_kernel<D, FP8>), dim3(ncta), dim3(T::kThreads),
                              T::kSmem, st, args);
    if (e != cudaSuccess) return e;
  }
  const long long rows = (long long)p.num_seqs * p.q_len * p.num_q_heads;
  AttnParams pp = p;
  const int32_t* cplan = plan;
  int n = ncta;
  void* args[] = {&pp, &cplan, &n};
  return launch_pdl(reinterpret_cast<const void*>(verify_merge_kernel<D>),
                    dim3((unsigned)((rows + kMergeWarps - 1) / kMergeWarps)), dim3(32 * kMergeWarps), 0, st, args);
}

}  // namespace

int verify_resident_ctas(int num_sms) { return 2 * num_sms; }

size_t verify_scratch_bytes(int num_seqs, int q_len, int num_q_heads, int num_kv_heads, int head_dim, int ncta) {
  const size_t rows_per_slot = (size_t)(num_q_heads / num_kv_heads) * q_len;
  const size_t slots = (size_t)num_kv_heads * num_seqs + ncta;
  const size_t plan = ((size_t)num_seqs + 2) * sizeof(int32_t);
  const size_t plan_padded = (plan + 255) / 256 * 256;
  return plan_padded + slots * rows_per_slot * (head_dim + 1) * sizeof(float);
}

cudaError_t launch_verify_tc(const AttnParams& p, const Launch& l, void* scratch, int ncta, const CUtensorMap& tk,
                             const CUtensorMap& tv) {
  if (l.group * p.q_len > TcTraits<128>::kRows) return cudaErrorInvalidConfiguration;
  const size_t plan = ((size_t)p.num_seqs + 2) * sizeof(int32_t);
  const size_t plan_padded = (plan + 255) / 256 * 256;
  AttnParams q = p;
  int32_t* planp = static_cast<int32_t*>(scratch);
  const size_t rows_per_slot = (size_t)l.group * p.q_len;
  const size_t slots = (size_t)p.num_kv_heads * p.num_seqs + ncta;
  q.part_o = reinterpret_cast<float*>(static_cast<char*>(scratch) + plan_padded);
  q.part_lse = q.part_o + slots * rows_per_slot * l.head_dim;
  q.max_partitions = ncta;
  if (l.head_dim == 128)
    return l.fp8 ? launch_d<128, true>(q, planp, ncta, tk, tv, l.stream) : launch_d<128, false>(q, planp, ncta, tk, tv, l.stream);
  if (l.head_dim == 64)
    return l.fp8 ? launch_d<64, true>(q, planp, ncta, tk, tv, l.stream) : launch_d<64, false>(q, planp, ncta, tk, tv, l.stream);
  return cudaErrorInvalidConfiguration;
}

#ifdef PA_TIMELINE
}  // namespace pa
// Instrumented build only: copy the stamps of the last verify launch ([CTA][8] u64, then the
// merge's last row end) to host and reset the merge-end stamp.
extern "C" int paged_attn_timeline_read_verify(unsigned long long* host, int max_ctas) {
  const int n = max_ctas < pa::kTlCtas ? max_ctas : pa::kTlCtas;
  const size_t bytes = (size_t)n * pa::kTlSlots * sizeof(unsigned long long);
  if (cudaMemcpyFromSymbol(host, pa::g_verify_timeline, bytes) != cudaSuccess) return 3;
  if (cudaMemcpyFromSymbol(host + (size_t)n * pa::kTlSlots, pa::g_verify_merge_end, 8) != cudaSuccess) return 3;
  const unsigned long long zero = 0;
  return cudaMemcpyToSymbol(pa::g_verify_merge_end, &zero, 8) == cudaSuccess ? 0 : 3;
}
// Instrumented build only: copy the per-step stamps of the last verify launch ([16 CTAs][64 steps]
// [kStSlots] clock64 values; 0 where a CTA walked fewer steps) to host.
extern "C" int paged_attn_timeline_read_verify_steps(long long* host) {
  const size_t bytes = sizeof(pa::g_verify_steps);
  if (cudaMemcpyFromSymbol(host, pa::g_verify_steps, bytes) != cudaSuccess) return 3;
  return 0;
}
namespace pa {
#endif

}  // namespace pa
