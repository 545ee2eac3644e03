// Paged chunked-prefill attention on 5th-generation tensor cores (tcgen05), sm_103a.
//
// Chunked prefill splits a long prompt into chunks and runs each chunk as one forward next to the
// running decodes (aegloslab servingai 5.3.15, Sarathi-style chunking with piggybacked decode):
// the chunk's tokens attend to everything already in the paged cache and causally to each other.
// Queries are packed per sequence (varlen): sequence b owns rows [qsl[b], qsl[b+1]) of q, with
// q_len_b of them, and its context_lens[b] counts them (their K/V are in the cache already), so
// new token i sees n = L - q_len_b + i + 1 tokens -- decode (q_len 1), verify (K + 1) and a
// prefill chunk in one call.
//
// Tile: the G query heads of a kv head share every K/V page, so one CTA takes 128 / G new tokens
// of one (sequence, kv head) as 128 rows r = token * G + head (a full M = 128 MMA tile) and walks
// the context in 64-token steps (FlashAttention tiling with an online softmax, studybook
// fde-roadmap ch.10, section 10.1.2):
//   S[128 x 64]  = Q[128 x d] . K_step^T              (tcgen05.mma, operands in shared memory)
//   O[128 x d]  += P[128 x 64] . V_step[64 x d]        (P from tensor memory, V from shared)
// Tensor memory: two S buffers (columns 0-63, 64-127; P overwrites its S as bf16 pairs) and O
// (columns 128..128+d): QK of step k+1 runs while the softmax of step k works.  Shared memory
// (~97 KB: Q, 2-stage K and V rings) lets two CTAs share an SM, so one's softmax overlaps the
// other's products.  Warps: 0-3 softmax (thread r = row r = TMEM lane r), 4 K producer, 5 V
// producer (2-D TMA boxes of 16 tokens x 64 dims, 128-byte swizzle), 6 MMA issuer.
// Grid: x = rank * Hkv + kv head, the rank of the (sequence, tile) pair in the planner's work
// list, which orders the pairs by their number of steps, largest first.
// E4M3 caches (FP8), as in the verify kernel (study book ch.10, section 10.8.2: one symmetric
// scale per (block, kv head)): with head_dim 128, Q.K^T runs on the E4M3 codes of K
// (kind::f8f6f4; K pages copied as swizzled 2-D boxes, Q as two E4M3 terms after a power-of-two
// row scale) and each page's K scale multiplies its scores; the V pages are bulk-copied into the
// upper half of the step's f16 tile and both producer warps convert half of its rows in place to
// f16 (exact), zeroing pages without a block and tokens past the tile's last row; P.V runs on f16
// with P carrying each page's V scale.  With head_dim 64 K is converted the same way and Q.K^T
// runs on f16 (Q re-encoded after the row scale).
#include "pa_kernels.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

template <int D>
struct PfTraits {
  static constexpr int kBS = 16;
  static constexpr int kTP = 4;                          // pages per step
  static constexpr int kStepTokens = kTP * kBS;          // 64
  static constexpr int kHalves = D / 64;                 // 64-dim swizzle atoms across d
  static constexpr int kRegion = kStepTokens * 128;      // one half of a step tile
  static constexpr int kBoxBytes = kBS * 128;            // one half of one page
  static constexpr int kTile = kHalves * kRegion;        // K or V tile of one step
  static constexpr int kRows = 128;
  static constexpr int kQHalf = kRows * 128;
  static constexpr int kQBytes = kHalves * kQHalf;
  static constexpr int kOffK = 0;                        // K stages 0, 1
  static constexpr int kOffV = kOffK + 2 * kTile;        // V stages 0, 1
  static constexpr int kOffQ = kOffV + 2 * kTile;
  static constexpr int kOffBar = kOffQ + kQBytes;
  // kfull[2], vfull[2], kempty[2], o_done[2], s_ready[2], p_ready[2], q_ready, final, and for
  // E4M3 caches kready[2], vready[2] (tile converted to f16)
  static constexpr int kNumBars = 18;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmem = kOffMisc + 16 + 1024;       // + slack for 1024-byte alignment
  static constexpr int kSCol = 0;                          // S/P buffer j: columns 64 j ..
  static constexpr int kOCol = 128;
  static constexpr int kTmemCols = 256;
  static constexpr int kThreads = 224;
  // kind::f16: D fp32 (bit 4), A bf16 (7-9), B bf16 (10-12), B MN-major (16), N >> 3 (17), M >> 4 (24)
  static constexpr uint32_t kIdescQK =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kStepTokens >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static constexpr uint32_t kIdescPV =
      (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  // E4M3 caches: f16 operands (A and B type 0)
  static constexpr uint32_t kIdescQK16 = kIdescQK & ~((1u << 7) | (1u << 10));
  static constexpr uint32_t kIdescPV16 = kIdescPV & ~((1u << 7) | (1u << 10));
};

// Work order: the (sequence, tile) pairs sorted by their number of 64-token steps, largest first
// (longest-processing-time order: the block scheduler hands out CTAs in blockIdx order, so the
// heaviest tiles start first and the light ones fill the tail).  One CTA: per-sequence checks,
// a histogram of step counts, its exclusive scan from the top, a scatter.  tiles[0] = number of
// pairs, tiles[1 + k] = b | tile << 16.
constexpr int kCostBuckets = 8192;

__global__ void __launch_bounds__(1024) prefill_plan_kernel(const AttnParams p, int tiles_per_row, int32_t* tiles) {
  __shared__ int hist[kCostBuckets];
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kCostBuckets; i += 1024) hist[i] = 0;
  if (tid == 0) total = 0;
  __syncthreads();
  const int Tt = tiles_per_row;
  auto seq_info = [&](int b, int& QL, int& first_new) {
    const int qs = p.query_start_loc[b];
    QL = p.query_start_loc[b + 1] - qs;
    if (qs < 0 || QL < 0 || qs + QL > p.total_q || QL > p.q_len) {
      record_error(p.err, kErrBadInput);  // rows outside the packed q: the sequence is skipped
      QL = 0;
    }
    int L = p.context_lens[b];
    if (L > p.max_context_len) {
      record_error(p.err, kErrShortContext);
      L = p.max_context_len;
    }
    first_new = L - QL;
  };
  auto cost = [&](int QL, int first_new, int t) {
    const int n_max = first_new + min((t + 1) * Tt, QL);
    const int steps = n_max > 0 ? (n_max + 63) / 64 : 0;
    return kCostBuckets - 1 - min(steps, kCostBuckets - 1);  // order index: costliest first
  };
  for (int b = tid; b < p.num_seqs; b += 1024) {
    int QL, first_new;
    seq_info(b, QL, first_new);
    const int nt = (QL + Tt - 1) / Tt;
    for (int t = 0; t < nt; ++t) atomicAdd(&hist[cost(QL, first_new, t)], 1);
  }
  __syncthreads();
  // exclusive scan of the histogram (8 buckets per thread)
  int loc[kCostBuckets / 1024];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < kCostBuckets / 1024; ++i) {
    loc[i] = hist[tid * (kCostBuckets / 1024) + i];
    sum += loc[i];
  }
  int inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int run = inc - sum + (warp > 0 ? warp_tot[warp - 1] : 0);
#pragma unroll
  for (int i = 0; i < kCostBuckets / 1024; ++i) {
    hist[tid * (kCostBuckets / 1024) + i] = run;
    run += loc[i];
  }
  if (tid == 1023) total = run;
  __syncthreads();
  for (int b = tid; b < p.num_seqs; b += 1024) {
    int QL, first_new;
    seq_info(b, QL, first_new);
    const int nt = (QL + Tt - 1) / Tt;
    for (int t = 0; t < nt; ++t) {
      const int pos = atomicAdd(&hist[cost(QL, first_new, t)], 1);
      tiles[1 + pos] = b | (t << 16);
    }
  }
  if (tid == 0) tiles[0] = total;
  // the attention kernel (a programmatic dependent) waits for this grid before reading the list
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifdef PA_TIMELINE
// Instrumented build only (-DPA_TIMELINE, a separate library; the product build has none of
// it): per CTA of the last (non-split) prefill launch, by blockIdx.x, read by
// paged_attn_timeline_read_prefill.  Slots: 0 entry, 1 exit (%globaltimer), 2 SM id, 3 steps,
// and sums over the steps s >= 2 of thread 0 of the softmax and of the MMA issuer (SM cycles,
// clock64): 4 softmax busy (S(s) seen -> P(s) arrived), 5 softmax waiting for S(s) (P(s-1)
// arrived -> S(s) seen), 6 handoff (last softmax warp's P(s) arrival -> PV(s) issued), 7 chain
// (PV(s-2) issued -> S(s) seen), 8 QK lag (PV(s-2) issued -> QK(s) issued), 9 steps summed,
// 10-13 the softmax step's phases (S loaded from tensor memory; row max and rescale; weights;
// P stored to tensor memory), 14 skew of the four softmax warps' P(s) arrivals (last - first).
constexpr int kPfTlCtas = 8192, kPfTlSlots = 16;
__device__ unsigned long long g_prefill_timeline[kPfTlCtas * kPfTlSlots];
__device__ __forceinline__ unsigned long long pf_gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned long long pf_clock() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void pf_tl_put(int slot, unsigned long long v) {
  if (blockIdx.x < kPfTlCtas && gridDim.y == 1) g_prefill_timeline[blockIdx.x * kPfTlSlots + slot] = v;
}
#endif

// SPLIT = false: packed variable-length rows, one CTA per (kv head, (sequence, tile) pair) in the
// planner's order.  SPLIT = true (verify rows that exceed the verify kernel's 64: every sequence
// q_len rows, G * q_len <= 128, one tile): grid (partition, kv head, sequence) over the split-KV
// plan of decode -- the CTA walks the pages [part * ppp, part * ppp + ppp) of its sequence and,
// when the sequence has several partitions, writes the normalised partial rows and their
// log2-sum-exp for the log-sum-exp merge kernel; p.tree_mask, when set, replaces the causal mask.
template <int D, bool SPLIT, bool FP8>
__global__ void __launch_bounds__(224, 2) prefill_tc_kernel(const AttnParams p, const int32_t* __restrict__ tiles,
                                                            const __grid_constant__ CUtensorMap tmk,
                                                            const __grid_constant__ CUtensorMap tmv) {
  using T = PfTraits<D>;
  // E4M3 with head_dim 128: Q.K^T on the E4M3 codes of K (kind::f8f6f4, Q split into two E4M3
  // terms), P.V on f16; head_dim 64: both products on f16 (K and V converted)
  constexpr bool kKDirect = FP8 && D == 128;
  const int Hq = p.num_q_heads, Hkv = p.num_kv_heads, G = Hq / Hkv;
  const int Tt = T::kRows / G;  // new tokens per tile
  int g, b, tile, qs, QL, part = 0;
  if constexpr (SPLIT) {
    part = (int)blockIdx.x;
    g = (int)blockIdx.y;
    b = (int)blockIdx.z;
    tile = 0;
    QL = p.q_len;
    qs = b * QL;
  } else {
    g = (int)(blockIdx.x % (unsigned)Hkv);
    const int rank = (int)(blockIdx.x / (unsigned)Hkv);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the work list comes from the planner
    if (rank >= tiles[0]) return;                       // fewer tiles than the grid's bound (uniform)
    const int entry = tiles[1 + rank];
    b = entry & 0xffff;
    tile = entry >> 16;
    qs = p.query_start_loc[b];
    QL = p.query_start_loc[b + 1] - qs;
  }

  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
  const uint32_t sK = base + T::kOffK, sV = base + T::kOffV, sQ = base + T::kOffQ;
  const uint32_t bar_kfull = base + T::kOffBar;  // + 8 * stage
  const uint32_t bar_vfull = bar_kfull + 16;
  const uint32_t bar_kempty = bar_vfull + 16;    // QK of a step done: K stage reusable
  const uint32_t bar_o_done = bar_kempty + 16;   // PV of a step done: V stage and S/P buffer reusable
  const uint32_t bar_s_ready = bar_o_done + 16;  // S of a step in tensor memory
  const uint32_t bar_p_ready = bar_s_ready + 16; // P of a step in tensor memory (4 warps)
  const uint32_t bar_q_ready = bar_p_ready + 16; // Q written (4 warps)
  const uint32_t bar_final = bar_q_ready + 8;    // every MMA issued has completed
  const uint32_t bar_kready = bar_final + 8;     // E4M3: + 8 * stage: K tile converted to f16
  const uint32_t bar_vready = bar_kready + 16;   // E4M3: + 8 * stage: V tile converted to f16
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + T::kOffMisc);
  volatile uint32_t* abort_flag = misc + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef PA_TIMELINE
  // stamps handed between the softmax and the issuer: P(s) arrived, PV(s) issued (by s % 2)
  __shared__ volatile unsigned long long tl_pdone[2], tl_pvissue[2], tl_pwarp[2][4];
  if (threadIdx.x == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    pf_tl_put(0, pf_gtime());
    pf_tl_put(2, smid);
    for (int i = 3; i < kPfTlSlots; ++i) pf_tl_put(i, 0ull);
  }
  unsigned long long tl_a = 0, tl_b = 0, tl_c = 0, tl_d = 0;  // the role's sums
  unsigned long long tl_ph[4] = {0ull, 0ull, 0ull, 0ull}, tl_mark = 0;
#endif

  // a longer context is flagged by the planner (split: by partition 0 of kv head 0)
  const int L = SPLIT ? context_len(p, b, part == 0 && g == 0 && threadIdx.x == 0)
                      : min(p.context_lens[b], p.max_context_len);
  const int t0 = tile * Tt;
  const int first_new = L - QL;                       // cache position of new token 0
  const int n_max = first_new + min(t0 + Tt, QL);     // tokens the tile's last row sees
  const int npages = n_max > 0 ? (n_max + T::kBS - 1) / T::kBS : 0;
  // the CTA's pages [pfirst, plast): all of them, or its partition (a whole number of steps)
  const int ppp = SPLIT ? p.pages_per_partition : 0;
  const int pfirst = SPLIT ? part * ppp : 0;
  const int plast = SPLIT ? min(npages, pfirst + ppp) : npages;
  const int nparts = SPLIT ? (npages + ppp - 1) / ppp : 1;
  const int nsteps = plast > pfirst ? (plast - pfirst + T::kTP - 1) / T::kTP : 0;
  const int32_t* bt = p.block_table + (size_t)b * p.max_blocks_per_seq;

  if (first_new + t0 + 1 <= 0 && part == 0) {
    // the tile's first row sees no token (context shorter than the new tokens): its rows that see
    // nothing come out as zeros
    if (threadIdx.x == 0) record_error(p.err, kErrShortContext);
  }
  if (SPLIT && npages > 0 && nsteps == 0) return;  // a partition past the sequence's pages
  if (nsteps == 0) {
    if (part != 0) return;
    for (int r = threadIdx.x; r < T::kRows; r += blockDim.x) {
      const int t = t0 + r / G;
      if (t >= QL) continue;
      __nv_bfloat16* dst = p.out + ((size_t)(qs + t) * Hq + g * G + r % G) * D;
      for (int c = 0; c < D; ++c) dst[c] = __float2bfloat16(0.f);
    }
    return;
  }

  // ---- set-up: barriers, tensor memory -------------------------------------------------------
  if (threadIdx.x == 128) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
      mbar_init(bar_o_done + 8 * s, 1);
      mbar_init(bar_s_ready + 8 * s, 1);
      mbar_init(bar_p_ready + 8 * s, 4);
      mbar_init(bar_kready + 8 * s, 1);
      mbar_init(bar_vready + 8 * s, kKDirect ? 2 : 1);  // head_dim 128: both producer warps convert V
    }
    mbar_init(bar_q_ready, 4);
    mbar_init(bar_final, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    if constexpr (!FP8 || kKDirect) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    if constexpr (!FP8) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  if (warp == 6) {
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

  if ((warp == 4 || warp == 5) && FP8) {
    // ======== E4M3 producers: warp 4 copies the K ring, warp 5 the V ring (2 stages each).  A bulk
    // copy lands each fp8 page of a step in the upper half of the step's f16 tile; once it has
    // landed a warp reads its rows of the step into registers and writes them back in place as f16
    // (exact) in the 128-byte-swizzled layout the MMAs read -- zeroing pages without a block and
    // tokens past the tile's last row -- and marks the tile converted.  With head_dim 128 the K
    // pages need no conversion (Q.K^T runs on the E4M3 codes, kind::f8f6f4): warp 4 copies them as
    // 2-D boxes in the swizzled layout the MMA reads and converts token rows 0-31 of every V tile,
    // while warp 5 copies the V pages and converts rows 32-63.  Copies run up to the ring ahead of
    // the conversions: a warp polls both sides, so neither waits behind the other.
    const bool is_k = warp == 4;
    const uint32_t ring = is_k ? sK : sV;
    const uint32_t bar_full = is_k ? bar_kfull : bar_vfull;    // fp8 bytes landed
    const uint32_t bar_free = is_k ? bar_kempty : bar_o_done;  // QK / PV of the step two before done
    const uint8_t* cache = is_k ? p.k_cache : p.v_cache;
    // the ring this warp converts and its token rows [c_row0, c_row0 + kCRows)
    const bool conv_v = kKDirect || !is_k;
    const uint32_t c_ring = conv_v ? sV : sK;
    const uint32_t c_full = conv_v ? bar_vfull : bar_kfull;
    const uint32_t c_ready = conv_v ? bar_vready : bar_kready;
    const int c_row0 = kKDirect && !is_k ? 32 : 0;
    constexpr int kCRows = kKDirect ? 32 : T::kStepTokens;
    constexpr int kPageFp8 = T::kBS * D;              // bytes of one fp8 page
    constexpr int kStageFp8 = T::kTP * kPageFp8;      // one step: half the f16 tile
    constexpr int kCPR = D / 16;                      // 16-code chunks per token row
    constexpr int kPer = kCRows * kCPR / 32;          // chunks per lane per step
    static_assert(2 * kStageFp8 == T::kTile, "fp8 step in the upper half of its f16 tile");
    // block id of page pfirst + s * kTP + (lane & 3) for lanes 0-3 (-1: none, or outside the pool)
    auto step_id = [&](int s, bool flag) {
      const int page = pfirst + s * T::kTP + (lane & 3);
      int v = -1;
      if (lane < T::kTP && page < plast) {
        v = bt[page];
        if (v < 0 || v >= p.num_blocks) {
          if (flag) record_error(p.err, kErrBlockId);
          v = -1;
        }
      }
      return v;
    };
    // with head_dim 128 warp 4's copies (K) and conversions (V) are independent
    const bool own_conv = !(kKDirect && is_k);
    int gi = 0, gc = 0;  // steps copied, steps converted
    uint32_t idle = 0;
    while (gc < nsteps || gi < nsteps) {
      bool progressed = false;
      // (a) copy the next step's pages once its stage is free
      if (gi < nsteps && (gi < gc + 2 || !own_conv)) {
        bool free_ok = gi < 2;
        if (!free_ok && lane == 0) free_ok = mbar_test_wait(bar_free + 8 * (gi & 1), ((gi - 2) >> 1) & 1);
        if (__shfl_sync(0xffffffffu, free_ok, 0)) {
          const int v = step_id(gi, is_k);
          int pbs[T::kTP];
#pragma unroll
          for (int pg = 0; pg < T::kTP; ++pg) pbs[pg] = __shfl_sync(0xffffffffu, v, pg);
          if (lane == 0) {
            const uint32_t bar = bar_full + 8 * (gi & 1);
            int npg = 0;
#pragma unroll
            for (int pg = 0; pg < T::kTP; ++pg) npg += pbs[pg] >= 0;
            if (npg == 0) {
              mbar_arrive(bar);
            } else if (!own_conv) {
              // E4M3 K pages as 16 x 128-byte boxes, 128-byte swizzle: the MMA's K-major layout
              const uint32_t dst = ring + (gi & 1) * T::kTile;
              mbar_arrive_expect_tx(bar, npg * kPageFp8);
#pragma unroll
              for (int pg = 0; pg < T::kTP; ++pg)
                if (pbs[pg] >= 0) tma_load_2d(dst + pg * kPageFp8, &tmk, 0, (pbs[pg] * Hkv + g) * T::kBS, bar);
            } else {
              const uint32_t dst = ring + (gi & 1) * T::kTile + kStageFp8;
              mbar_arrive_expect_tx(bar, npg * kPageFp8);
#pragma unroll
              for (int pg = 0; pg < T::kTP; ++pg)
                if (pbs[pg] >= 0)
                  bulk_copy_g2s(dst + pg * kPageFp8, cache + ((size_t)pbs[pg] * Hkv + g) * kPageFp8, kPageFp8, bar);
            }
          }
          ++gi;
          progressed = true;
        }
      }
      // (b) convert this warp's rows of the oldest unconverted step once its bytes have landed (a
      // V step that warp 5 copied has landed once its full barrier's phase completed: warp 5
      // cannot copy into that stage again before this warp has converted it)
      if (gc < nsteps && (gc < gi || !own_conv)) {
        bool landed = false;
        if (lane == 0) landed = mbar_test_wait(c_full + 8 * (gc & 1), (gc >> 1) & 1);
        if (__shfl_sync(0xffffffffu, landed, 0)) {
          const uint32_t tile = c_ring + (gc & 1) * T::kTile;
          const uint32_t src = tile + kStageFp8;
          const unsigned okm = __ballot_sync(0xffffffffu, step_id(gc, false) >= 0) & ((1u << T::kTP) - 1u);
          const int ps = pfirst + gc * T::kTP;
          const int rows_ok = min(n_max, min(ps + T::kTP, plast) * T::kBS) - ps * T::kBS;  // token rows [0, rows_ok)
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
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c8 ^ (tr & 7)) << 4)), "r"(h[0]),
                           "r"(h[1]), "r"(h[2]), "r"(h[3])
                           : "memory");
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((c8 + 1) ^ (tr & 7)) << 4)),
                           "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                           : "memory");
            }
            __syncwarp();
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(c_ready + 8 * (gc & 1));
          ++gc;
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
      }
    }
    // every copy started has landed before the CTA's shared memory can go away (a copy is started
    // only once the copy two steps before it was consumed, so only the last two can be in flight)
    if (lane == 0)
      for (int k = max(0, gi - 2); k < gi; ++k) mbar_wait(bar_full + 8 * (k & 1), (k >> 1) & 1);
    __syncwarp();
  } else if (warp == 4 || warp == 5) {
    // ======== TMA producers: warp 4 fills the K ring, warp 5 the V ring (2 stages each) ========
    const bool is_k = warp == 4;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    const uint32_t ring = is_k ? sK : sV;
    const uint32_t bar_full = is_k ? bar_kfull : bar_vfull;
    const uint32_t bar_free = is_k ? bar_kempty : bar_o_done;
    auto load_ids = [&](int pbase) {
      const int pg = pbase + lane;
      int v = -1;
      if (pg < plast) {
        v = bt[pg];
        if (v < 0 || v >= p.num_blocks) {
          if (is_k) record_error(p.err, kErrBlockId);
          v = -1;
        }
      }
      return v;
    };
    int cbase = pfirst;
    int cur = load_ids(cbase);
    int s = 0;
    for (; s < nsteps; ++s) {
      const int pstep = pfirst + s * T::kTP;
      if (pstep >= cbase + 32) {
        cbase += 32;
        cur = load_ids(cbase);
      }
      int pbs[T::kTP];
      int npg = 0;
#pragma unroll
      for (int pg = 0; pg < T::kTP; ++pg) {
        pbs[pg] = __shfl_sync(0xffffffffu, cur, (pstep - cbase + pg) & 31);
        npg += pbs[pg] >= 0;
      }
      bool ready = true;
      if (lane == 0) {
        if (s >= 2) ready = wait_or_abort(bar_free + 8 * (s & 1), ((s - 2) >> 1) & 1, abort_flag, p.err);
        if (ready) {
          const uint32_t region = ring + (s & 1) * T::kTile;
          const uint32_t bar = bar_full + 8 * (s & 1);
          if (npg == 0) {
            mbar_arrive(bar);
          } else {
            mbar_arrive_expect_tx(bar, npg * T::kHalves * T::kBoxBytes);
#pragma unroll
            for (int pg = 0; pg < T::kTP; ++pg) {
              if (pbs[pg] < 0) continue;
              const int row = (pbs[pg] * Hkv + g) * T::kBS;
#pragma unroll
              for (int hh = 0; hh < T::kHalves; ++hh)
                tma_load_2d(region + hh * T::kRegion + pg * T::kBoxBytes, map, hh * 64, row, bar);
            }
          }
        }
      }
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (!ready) break;
    }
    // every copy started has landed before the CTA's shared memory can go away
    if (lane == 0)
      for (int k = max(0, s - 2); k < s; ++k) mbar_wait(bar_full + 8 * (k & 1), (k >> 1) & 1);
    __syncwarp();
  } else if (warp == 6) {
    // ======================= MMA issuer ========================================================
    if (lane == 0) {
      auto mma_qk = [&](int s) {
        const uint32_t kreg = sK + (s & 1) * T::kTile;
        const uint32_t tS = tmem + T::kSCol + (s & 1) * 64;
        if constexpr (kKDirect) {
          // S = Q_hi . K^T + Q_lo . K^T on E4M3 operands: each token row of K is one 128-byte
          // swizzled row (128 codes), 32 codes per instruction; Q_hi and Q_lo are 128-row E4M3
          // tiles one Q half apart
#pragma unroll
          for (int term = 0; term < 2; ++term)
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)
              umma_f8(tS, smem_desc(sQ + term * T::kQHalf + kk * 32, 16, 1024), smem_desc(kreg + kk * 32, 16, 1024),
                      T::kIdescQK16, (term > 0 || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * T::kRegion + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * T::kQHalf + (kk & 3) * 32;
            umma_bf16(tS, smem_desc(sQ + qoff, 16, 1024), smem_desc(kreg + koff, 16, 1024),
                      FP8 ? T::kIdescQK16 : T::kIdescQK, kk > 0 ? 1u : 0u);
          }
        }
        umma_commit(bar_s_ready + 8 * (s & 1));
        umma_commit(bar_kempty + 8 * (s & 1));
      };
      auto mma_pv = [&](int s) {
        const uint32_t vreg = sV + (s & 1) * T::kTile;
        const uint32_t tP = tmem + T::kSCol + (s & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < T::kStepTokens / 16; ++kk) {
          // A = P in tensor memory (16 tokens = 8 columns of bf16 pairs); B = V MN-major
          umma_bf16_tmem_a(tO, tP + kk * 8, smem_desc(vreg + kk * 2048, T::kRegion, 1024),
                           FP8 ? T::kIdescPV16 : T::kIdescPV, (s > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar_o_done + 8 * (s & 1));
      };
      int gq = 0, gp = 0;
      uint32_t idle = 0;
      while (gp < nsteps) {
        bool progressed = false;
        if (gq < nsteps && mbar_test_wait((FP8 && !kKDirect ? bar_kready : bar_kfull) + 8 * (gq & 1), (gq >> 1) & 1) &&
            (gq < 2 || mbar_test_wait(bar_o_done + 8 * (gq & 1), ((gq - 2) >> 1) & 1)) &&
            (gq > 0 || mbar_test_wait(bar_q_ready, 0))) {
          tc_fence_after();
#ifdef PA_TIMELINE
          if (gq >= 2) tl_b += pf_clock() - tl_pvissue[gq & 1];
#endif
          mma_qk(gq);
          ++gq;
          progressed = true;
        }
        if (gp < gq && mbar_test_wait(bar_p_ready + 8 * (gp & 1), (gp >> 1) & 1) &&
            mbar_test_wait((FP8 ? bar_vready : bar_vfull) + 8 * (gp & 1), (gp >> 1) & 1)) {
          tc_fence_after();
#ifdef PA_TIMELINE
          {
            const unsigned long long now = pf_clock();
            if (gp >= 2) {
              unsigned long long lo = tl_pwarp[gp & 1][0], hi = lo;
              for (int w = 1; w < 4; ++w) {
                lo = min(lo, (unsigned long long)tl_pwarp[gp & 1][w]);
                hi = max(hi, (unsigned long long)tl_pwarp[gp & 1][w]);
              }
              tl_a += now - hi;
              tl_d += hi - lo;
            }
            tl_pvissue[gp & 1] = now;
          }
#endif
          mma_pv(gp);
          ++gp;
          progressed = true;
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
#ifdef PA_TIMELINE
      pf_tl_put(6, tl_a);
      pf_tl_put(8, tl_b);
      pf_tl_put(14, tl_d);
#endif
    }
    __syncwarp();
  } else {
    // ======================= softmax: thread r owns row r ======================================
    const int r = threadIdx.x;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int t = t0 + r / G;          // new-token index of this row
    const int h = g * G + r % G;       // its query head
    const bool row_live = t < QL;
    const int n_r = row_live ? max(first_new + t + 1, 0) : 0;  // tokens this row sees
    // tree verify (split mode only): the new tokens the row sees are its ancestor bits; the chain
    // mask (bits 0 .. t) gives the causal row exactly
    const bool tree = SPLIT && p.tree_mask != nullptr;
    const uint32_t anc = (tree && row_live) ? p.tree_mask[(size_t)b * QL + t] : 0u;
    // Q row r: bf16, K-major 128-byte swizzle (halves of 64 dims, 8-row groups 1024 B apart).
    // E4M3: the row scaled by a power of two 2^k first (exact, no overflow for any bf16 q) and its
    // scores by qdiv = 2^-k; head_dim 128: two E4M3 terms hi = e4m3(q 2^k), lo = e4m3(q 2^k - hi)
    // (e4m3_prescale_exp), each a 128-byte row of codes, one Q half apart; head_dim 64: f16
    // (f16_prescale_exp).
    float qdiv = 1.f;
    {
      const __nv_bfloat16* qrow = row_live ? p.q + ((size_t)(qs + t) * Hq + h) * D : nullptr;
      float up = 1.f;
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
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint4 a = make_uint4(0u, 0u, 0u, 0u), b2 = a;
          if (qrow) {
            a = *reinterpret_cast<const uint4*>(qrow + c * 16);
            b2 = *reinterpret_cast<const uint4*>(qrow + c * 16 + 8);
          }
          const uint32_t wq[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 x0 = bf16x2_to_f2(wq[2 * j]), x1 = bf16x2_to_f2(wq[2 * j + 1]);
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
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sQ + T::kQHalf + off), "r"(lo[0]), "r"(lo[1]),
                       "r"(lo[2]), "r"(lo[3])
                       : "memory");
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (qrow) v = *reinterpret_cast<const uint4*>(qrow + c * 8);
          if constexpr (FP8) {
            const float2 a = bf16x2_to_f2(v.x), b2 = bf16x2_to_f2(v.y), c2 = bf16x2_to_f2(v.z), d2 = bf16x2_to_f2(v.w);
            v = make_uint4(pack_f16(a.x * up, a.y * up), pack_f16(b2.x * up, b2.y * up), pack_f16(c2.x * up, c2.y * up),
                           pack_f16(d2.x * up, d2.y * up));
          }
          const uint32_t dst = sQ + (c >> 3) * T::kQHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_q_ready);
    }
    // bf16: pages of a step that hold usable data (bit per page)
    auto pages_ok = [&](int s, float (&ksc)[T::kTP], float (&vsc)[T::kTP]) {
      unsigned okp = 0;
#pragma unroll
      for (int pg = 0; pg < T::kTP; ++pg) {
        ksc[pg] = 0.f;
        vsc[pg] = 0.f;
        const int page = pfirst + s * T::kTP + pg;
        if (page < plast) {
          const int pb = bt[page];
          if (pb >= 0 && pb < p.num_blocks) okp |= 1u << pg;
        }
      }
      return okp;
    };
    // bf16: one check of every block id of the tile's range by the 128 softmax threads (named
    // barrier 1); with a valid table the steps need no per-page lookups
    bool all_ok = false;
    if constexpr (!FP8) {
      unsigned bad = 0;
      for (int pg = pfirst + r; pg < plast; pg += T::kRows) {
        const int pb = bt[pg];
        bad |= (pb < 0 || pb >= p.num_blocks) ? 1u : 0u;
      }
      unsigned anybad;
      asm volatile(
          "{\n\t.reg .pred pb, pr;\n\tsetp.ne.u32 pb, %1, 0;\n\tbar.red.or.pred pr, 1, 128, pb;\n\tselp.u32 %0, 1, 0, pr;\n\t}"
          : "=r"(anybad)
          : "r"(bad)
          : "memory");
      all_ok = anybad == 0;
    }
    // pages of step s that lie in the tile's range (valid table)
    auto pages_in = [&](int s) {
      const int left = plast - (pfirst + s * T::kTP);
      return left >= T::kTP ? (1u << T::kTP) - 1u : (left > 0 ? (1u << left) - 1u : 0u);
    };
    // E4M3: the block ids of step s + 2 are loaded during step s, and the K and V scales of step
    // s + 1 from them (at clamped addresses, no branch on a loaded value), so neither dependent
    // round trip waits inside a step
    int ids_next[T::kTP];  // block ids of the step after the next one (-1: past the range)
    auto load_ids = [&](int s, int (&ids)[T::kTP]) {
#pragma unroll
      for (int pg = 0; pg < T::kTP; ++pg) {
        const int page = pfirst + s * T::kTP + pg;
        ids[pg] = page < plast ? bt[page] : -1;
      }
    };
    auto scales_of = [&](const int (&ids)[T::kTP], float (&ksc)[T::kTP], float (&vsc)[T::kTP]) {
      unsigned okp = 0;
#pragma unroll
      for (int pg = 0; pg < T::kTP; ++pg) {
        const bool v = ids[pg] >= 0 && ids[pg] < p.num_blocks;
        okp |= (v ? 1u : 0u) << pg;
        const size_t at = (size_t)(v ? ids[pg] : 0) * Hkv + g;
        ksc[pg] = p.k_scale[at];
        vsc[pg] = p.v_scale[at];
      }
      return okp;
    };
    bool ok = true;
    float m_used = -INFINITY, l = 0.f;
    float ks_next[T::kTP], vs_next[T::kTP];
    unsigned pok_next;
    if constexpr (FP8) {
      load_ids(0, ids_next);
      pok_next = scales_of(ids_next, ks_next, vs_next);
      if (nsteps > 1) load_ids(1, ids_next);
    } else {
      pok_next = all_ok ? pages_in(0) : pages_ok(0, ks_next, vs_next);
    }
    for (int s = 0; s < nsteps; ++s) {
      const unsigned pok = pok_next;
      float ksc[T::kTP], vsc[T::kTP];
#pragma unroll
      for (int pg = 0; pg < T::kTP; ++pg) {
        ksc[pg] = ks_next[pg];
        vsc[pg] = vs_next[pg];
      }
      const uint32_t tS = tmem + T::kSCol + (s & 1) * 64 + lane_off;
      if (!(ok = wait_or_abort(bar_s_ready + 8 * (s & 1), (s >> 1) & 1, abort_flag, p.err))) break;
      tc_fence_after();
#ifdef PA_TIMELINE
      unsigned long long tl_s = 0;
      if (r == 0) {
        tl_s = pf_clock();
        if (s >= 2) {
          tl_b += tl_s - tl_pdone[(s - 1) & 1];
          tl_c += tl_s - tl_pvissue[s & 1];
        }
      }
#endif
      float sc[T::kStepTokens];
      {
        uint32_t raw64[64];
        tmem_ld_x64(tS, raw64);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 64; ++c) sc[c] = __uint_as_float(raw64[c]);
      }
#ifdef PA_TIMELINE
      if (r == 0 && s >= 2) {
        tl_mark = pf_clock();
        tl_ph[0] += tl_mark - tl_s;
      }
#endif
      if (s + 1 < nsteps) {
        if constexpr (FP8) {
          pok_next = scales_of(ids_next, ks_next, vs_next);
          if (s + 2 < nsteps) load_ids(s + 2, ids_next);
        } else {
          pok_next = all_ok ? pages_in(s + 1) : pages_ok(s + 1, ks_next, vs_next);
        }
      }
      const int tok0 = (pfirst + s * T::kTP) * T::kBS;
      // visibility of the step's 64 tokens for this row: causal limit (or, for a tree, the whole
      // prefix and the ancestor bits of the new tokens) and pages holding data
      uint64_t vis;
      if (tree) {
        const int sh = first_new - tok0;  // bit of new token 0 within the step
        const uint64_t a = row_live ? (uint64_t)anc : 0ull;
        const uint64_t nb = sh >= 64 ? 0ull : sh >= 0 ? (a << sh) : (-sh >= 64 ? 0ull : (a >> -sh));
        vis = (row_live ? low_bits64(first_new - tok0) : 0ull) | nb;
      } else {
        vis = low_bits64(n_r - tok0);
      }
      {
        uint64_t pm = 0;
#pragma unroll
        for (int pg = 0; pg < T::kTP; ++pg)
          if ((pok >> pg) & 1u) pm |= 0xffffull << (16 * pg);
        vis &= pm;
      }
      // Full steps with a positive scale stay in raw scores: the row max of raw scores times the
      // scale is the max of the scaled ones, and each weight is ex2(s * scale - m) with the
      // scale folded into one packed FMA per pair.  Masked steps (the diagonal, block tails)
      // scale first and mask with -inf.
      const bool raw = !FP8 && vis == ~0ull && p.scale_log2 > 0.f;
      // E4M3: each page's scores carry its K scale
      float kmul[T::kTP];
#pragma unroll
      for (int pg = 0; pg < T::kTP; ++pg) kmul[pg] = FP8 ? ksc[pg] * qdiv * p.scale_log2 : p.scale_log2;
      // E4M3 full steps with positive scales stay in raw scores too: the page's max of raw scores
      // times its K multiplier is its scaled max, and each weight is ex2(s * kmul - m + log2
      // vscale), the V scale folded into the exponent's packed FMA, the row sum recovered per page
      // by dividing by the scale.  The V scales must be at least 2^-60: a folded weight then drops
      // below the smallest normal float (and out of the row sum) only where the weight itself is
      // under 2^-66; a smaller scale would lose the page's weights from the row sum.
      const bool fraw = FP8 && vis == ~0ull && p.scale_log2 > 0.f &&
                        fminf(fminf(ksc[0], ksc[1]), fminf(ksc[2], ksc[3])) > 0.f &&
                        fminf(fminf(vsc[0], vsc[1]), fminf(vsc[2], vsc[3])) >= 0x1p-60f;
      float mxs[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mxs[j] = -INFINITY;
      if (raw) {
#pragma unroll
        for (int c = 0; c < T::kStepTokens; ++c) mxs[c & 7] = fmaxf(mxs[c & 7], sc[c]);
      } else if (fraw) {
#pragma unroll
        for (int c = 0; c < T::kStepTokens; ++c) mxs[(c / T::kBS) * 2 + (c & 1)] = fmaxf(mxs[(c / T::kBS) * 2 + (c & 1)], sc[c]);
#pragma unroll
        for (int pg = 0; pg < T::kTP; ++pg) {
          mxs[2 * pg] = fmaxf(mxs[2 * pg], mxs[2 * pg + 1]) * kmul[pg];
          mxs[2 * pg + 1] = -INFINITY;
        }
      } else {
        const uint32_t v0 = (uint32_t)vis, v1 = (uint32_t)(vis >> 32);
#pragma unroll
        for (int c = 0; c < T::kStepTokens; ++c) {
          const bool v = (((c < 32 ? v0 : v1) >> (c & 31)) & 1u) != 0;
          sc[c] = v ? sc[c] * kmul[c / T::kBS] : -INFINITY;
          mxs[c & 7] = fmaxf(mxs[c & 7], sc[c]);
        }
      }
      float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                       fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
      if (raw) mx *= p.scale_log2;
      const float m_new = fmaxf(m_used, mx);
      const bool need = (m_used != -INFINITY) && (m_new > m_used + 8.f);
      if (__any_sync(0xffffffffu, need)) {
        // the O row is rescaled only once PV(s - 1) has landed in it
        if (!(ok = wait_or_abort(bar_o_done + 8 * ((s - 1) & 1), ((s - 1) >> 1) & 1, abort_flag, p.err))) break;
        tc_fence_after();
        const float alpha = need ? fast_exp2(m_used - m_new) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rw[32];
          tmem_ld_x32(tO + lane_off + c0, rw);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) rw[c] = __float_as_uint(__uint_as_float(rw[c]) * alpha);
          tmem_st_x32(tO + lane_off + c0, rw);
        }
        tmem_wait_st();
        l *= alpha;
      }
      if (need || m_used == -INFINITY) m_used = m_new;
      const float basev = m_used == -INFINITY ? 0.f : m_used;
#ifdef PA_TIMELINE
      if (r == 0 && s >= 2) {
        const unsigned long long now = pf_clock();
        tl_ph[1] += now - tl_mark;
        tl_mark = now;
      }
#endif

      // zero the V rows of tokens that hold no data (past the tile's range, or pages without a
      // block): P is 0 there, but 0 * NaN would still poison the product.  Thread r < 64 takes
      // token r of the step, after the step's V tile has landed; with a valid table only the last
      // step can hold such tokens.  (E4M3 tiles come zeroed from the conversion.)
      if (!FP8 && warp < 2 && (!all_ok || tok0 + T::kStepTokens > n_max)) {
        const int tok = tok0 + r;
        const bool tok_ok = ((pok >> (r >> 4)) & 1u) && tok < n_max;
        if (__any_sync(0xffffffffu, !tok_ok)) {
          if (!(ok = wait_or_abort(bar_vfull + 8 * (s & 1), (s >> 1) & 1, abort_flag, p.err))) break;
          if (!tok_ok) {
            const uint32_t vrow = sV + (s & 1) * T::kTile + r * 128;
#pragma unroll
            for (int hh = 0; hh < T::kHalves; ++hh)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + hh * T::kRegion + c * 16),
                             "r"(0u)
                             : "memory");
          }
          fence_proxy_async_smem();
        }
      }
      // P row r as bf16 pairs over the first 32 columns of this step's S buffer
      uint32_t w[32];
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      const float2 one2 = make_float2(1.f, 1.f);
      const float2 sc2 = raw ? make_float2(p.scale_log2, p.scale_log2) : one2;
      const float2 nb2 = make_float2(-basev, -basev);
      float lstep = 0.f;
      if (FP8 && fraw) {
        // pair c lies in page c / 8; acc[page] sums the weights times the page's V scale
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int pg = c / (T::kBS / 2);
          const float bias = __log2f(vsc[pg]) - basev;
          const float2 x = ffma2(make_float2(sc[2 * c], sc[2 * c + 1]), make_float2(kmul[pg], kmul[pg]),
                                 make_float2(bias, bias));
          const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          acc[pg] = ffma2(e, one2, acc[pg]);
          w[c] = pack_f16(e.x, e.y);
        }
#pragma unroll
        for (int pg = 0; pg < T::kTP; ++pg) lstep += (acc[pg].x + acc[pg].y) / vsc[pg];
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = ffma2(make_float2(sc[2 * c], sc[2 * c + 1]), sc2, nb2);
          const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          if constexpr (FP8) {  // f16 P carries each page's V scale; l sums the plain weights
            acc[c & 3] = ffma2(e, one2, acc[c & 3]);
            const float vm = vsc[(2 * c) / T::kBS];
            w[c] = pack_f16(e.x * vm, e.y * vm);
          } else {
            // l sums the bf16-rounded weights that P.V multiplies (normalised by its own weights)
            w[c] = pack_bf16(e.x, e.y);
            acc[c & 3] = add_bf16x2_f2(w[c], acc[c & 3]);
          }
        }
        lstep = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) + ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
      }
#ifdef PA_TIMELINE
      if (r == 0 && s >= 2) {
        const unsigned long long now = pf_clock();
        tl_ph[2] += now - tl_mark;
        tl_mark = now;
      }
#endif
      tmem_st_x32(tS, w);
      tmem_wait_st();
#ifdef PA_TIMELINE
      if (r == 0 && s >= 2) tl_ph[3] += pf_clock() - tl_mark;
#endif
      l += lstep;
      tc_fence_before();
      __syncwarp();
#ifdef PA_TIMELINE
      if (r == 0) {
        const unsigned long long now = pf_clock();
        if (s >= 2) tl_a += now - tl_s;
        tl_pdone[s & 1] = now;
      }
      if (lane == 0) tl_pwarp[s & 1][warp] = pf_clock();
#endif
      if (lane == 0) mbar_arrive(bar_p_ready + 8 * (s & 1));
    }
#ifdef PA_TIMELINE
    if (r == 0) {
      pf_tl_put(3, (unsigned long long)nsteps);
      pf_tl_put(4, tl_a);
      pf_tl_put(5, tl_b);
      pf_tl_put(7, tl_c);
      pf_tl_put(9, (unsigned long long)(nsteps > 2 ? nsteps - 2 : 0));
      for (int i = 0; i < 4; ++i) pf_tl_put(10 + i, tl_ph[i]);
    }
#endif
    if (ok) {
      // ---- epilogue: O row / l -> bf16 ------------------------------------------------------
      const int gl = nsteps - 1;
      ok = wait_or_abort(bar_o_done + 8 * (gl & 1), (gl >> 1) & 1, abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* dst = p.out + ((size_t)(qs + t) * Hq + h) * D;
        // split sequence: the partition's normalised rows and log2-sum-exp for the merge kernel
        const bool partial = SPLIT && nparts > 1;
        const size_t prow = ((size_t)(qs + t) * Hq + h) * p.max_partitions + part;
        if (partial && row_live) p.part_lse[prow] = l > 0.f ? m_used + __log2f(l) : -INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t raw[32];
          tmem_ld_x32(tO + lane_off + c0, raw);
          tmem_wait_ld();
          if (!row_live) continue;
          if (partial) {
            float* pdst = p.part_o + prow * D + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(pdst + c) =
                  make_float4(__uint_as_float(raw[c]) * inv, __uint_as_float(raw[c + 1]) * inv,
                              __uint_as_float(raw[c + 2]) * inv, __uint_as_float(raw[c + 3]) * inv);
            continue;
          }
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(raw[c + 0]) * inv, __uint_as_float(raw[c + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(raw[c + 2]) * inv, __uint_as_float(raw[c + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(raw[c + 4]) * inv, __uint_as_float(raw[c + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(raw[c + 6]) * inv, __uint_as_float(raw[c + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c0 + c) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 6) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T::kTmemCols) : "memory");
  }
#ifdef PA_TIMELINE
  if (threadIdx.x == 0) pf_tl_put(1, pf_gtime());
#endif
}

template <int D, bool FP8>
cudaError_t launch_d(const AttnParams& p, int max_q_len, int group, int32_t* tiles, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t st) {
  using T = PfTraits<D>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(prefill_tc_kernel<D, false, FP8>), T::kSmem);
  if (e != cudaSuccess) return e;
  const int tt = T::kRows / group;
  prefill_plan_kernel<<<1, 1024, 0, st>>>(p, tt, tiles);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long bound = (long long)p.num_seqs * ((max_q_len + tt - 1) / tt);
  AttnParams pp = p;
  const int32_t* ct = tiles;
  CUtensorMap k = tk, v = tv;
  void* args[] = {&pp, &ct, &k, &v};
  // x = rank * Hkv + kv head: the heaviest pairs, all heads of each, are dispatched first
  return launch_pdl(reinterpret_cast<const void*>(prefill_tc_kernel<D, false, FP8>),
                    dim3((unsigned)(bound * p.num_kv_heads)), dim3(T::kThreads), T::kSmem, st, args);
}

template <int D, bool FP8>
cudaError_t launch_split_d(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  using T = PfTraits<D>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(prefill_tc_kernel<D, true, FP8>), T::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_partitions, p.num_kv_heads, p.num_seqs);
  prefill_tc_kernel<D, true, FP8><<<grid, T::kThreads, T::kSmem, st>>>(p, nullptr, tk, tv);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_scratch_bytes(int num_seqs, int max_q_len, int group) {
  const int tt = PfTraits<128>::kRows / group;
  return (1 + (size_t)num_seqs * ((max_q_len + tt - 1) / tt)) * sizeof(int32_t);
}

cudaError_t launch_verify_split(const AttnParams& p, const Launch& l, const CUtensorMap& tk, const CUtensorMap& tv) {
  if (l.group * p.q_len > PfTraits<128>::kRows || p.pages_per_partition % PfTraits<128>::kTP != 0)
    return cudaErrorInvalidConfiguration;
  if (l.head_dim == 128)
    return l.fp8 ? launch_split_d<128, true>(p, tk, tv, l.stream) : launch_split_d<128, false>(p, tk, tv, l.stream);
  if (l.head_dim == 64)
    return l.fp8 ? launch_split_d<64, true>(p, tk, tv, l.stream) : launch_split_d<64, false>(p, tk, tv, l.stream);
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_prefill_tc(const AttnParams& p, const Launch& l, int max_q_len, void* scratch, const CUtensorMap& tk,
                              const CUtensorMap& tv) {
  if (l.group < 1 || PfTraits<128>::kRows % l.group != 0) return cudaErrorInvalidConfiguration;
  int32_t* tiles = static_cast<int32_t*>(scratch);
  if (l.head_dim == 128)
    return l.fp8 ? launch_d<128, true>(p, max_q_len, l.group, tiles, tk, tv, l.stream)
                 : launch_d<128, false>(p, max_q_len, l.group, tiles, tk, tv, l.stream);
  if (l.head_dim == 64)
    return l.fp8 ? launch_d<64, true>(p, max_q_len, l.group, tiles, tk, tv, l.stream)
                 : launch_d<64, false>(p, max_q_len, l.group, tiles, tk, tv, l.stream);
  return cudaErrorInvalidConfiguration;
}

#ifdef PA_TIMELINE
}  // namespace pa
// Instrumented build only: copy the per-CTA slots ([CTA][12] u64) to host, then zero them, so
// that CTAs of the next launch that return before their first stamp read as all-zero.
extern "C" int paged_attn_timeline_read_prefill(unsigned long long* host, int max_ctas) {
  const int n = max_ctas < pa::kPfTlCtas ? max_ctas : pa::kPfTlCtas;
  const size_t bytes = (size_t)n * pa::kPfTlSlots * sizeof(unsigned long long);
  if (cudaMemcpyFromSymbol(host, pa::g_prefill_timeline, bytes) != cudaSuccess) return 3;
  void* dev = nullptr;
  if (cudaGetSymbolAddress(&dev, pa::g_prefill_timeline) != cudaSuccess) return 3;
  if (cudaMemset(dev, 0, sizeof(unsigned long long) * pa::kPfTlCtas * pa::kPfTlSlots) != cudaSuccess) return 3;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
namespace pa {
#endif

}  // namespace pa
