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
// One CTA per (partition, kv head, sequence), five warps:
//   warps 3, 4     -- TMA producers (lane 0 of each): K and V pages (2-D tensor boxes of 16 tokens
//                     x 64 dims with the 128-byte swizzle, completion on mbarriers) into separate
//                     2-stage rings, so a K tile is refilled as soon as its scores are computed;
//   warp 2, lane 0 -- MMA issuer: tcgen05.mma for both products, completion via tcgen05.commit,
//                     issuing S(k+1) ahead of PV(k) whenever it is ready first;
//   warps 0, 1     -- softmax: thread r owns query row r (TMEM lane r); it reads its 64 scores
//                     with tcgen05.ld, masks (causal limit, block tail, partition end), keeps the
//                     row max m and sum l in base 2, writes P (bf16) into shared memory in the
//                     K-major 128-byte-swizzled layout the MMA reads, and rescales its O row in
//                     TMEM only when the max grows by more than 2^8 (a stale max is exact as long
//                     as l uses the same one).
// Shared operands use the canonical tcgen05 layouts: Q, K and P K-major with 128-byte swizzle
// (8-row groups 1024 B apart), V MN-major with 128-byte swizzle (64-dim atoms one region apart).
#include "pa_kernels.h"

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
  static constexpr int kStageBytes = 2 * kKTile;         // K tile then V tile
  static constexpr int kStages = 2;
  static constexpr int kRows = 64;                       // rows a CTA serves (G * q_len <= 64)
  static constexpr int kPBytes = kRows * 128;            // one P buffer: rows 0..63; MMA rows
  static constexpr int kQBytes = kHalves * kRows * 128;  //   64..127 read what follows (padding)
  static constexpr int kOffP = 0;                        // two P buffers
  static constexpr int kOffQ = kOffP + 2 * kPBytes;
  static constexpr int kOffStage = kOffQ + kQBytes;
  static constexpr int kOffBar = kOffStage + kStages * kStageBytes;
  // barriers: kfull[2], vfull[2], kempty[2], o_done[2], p_ready[2], s_ready, s_free, final
  static constexpr int kNumBars = 13;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kMaxPages = 256;                    // block ids of a partition, staged once
  static constexpr int kOffIds = kOffMisc + 16;
  static constexpr int kSmem = kOffIds + kMaxPages * 4 + 1024;  // + slack for 1024-B alignment
  static constexpr int kSCol = 0;                          // S: 64 fp32 columns
  static constexpr int kOCol = 64;                         // O: D fp32 columns
  static constexpr int kTmemCols = D == 128 ? 256 : 128;   // power of two >= 64 + D
  static constexpr int kThreads = 160;
  // instruction descriptors (kind::f16): D fp32 (bit 4), A bf16 (bits 7-9 = 1), B bf16 (bits
  // 10-12 = 1), B major bit 16 (1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24
  static constexpr uint32_t kIdescQK =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kStepTokens >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static constexpr uint32_t kIdescPV =
      (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
};

// ---- tcgen05 / TMA primitives ---------------------------------------------------------------

// Shared-memory matrix descriptor: start >> 4 (bits 0-13), leading byte offset >> 4 (16-29),
// stride byte offset >> 4 (32-45), fixed 0b001 at bits 46-48, swizzle mode at bits 61-63
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Bounded wait that also gives up once another thread has aborted the CTA.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                              unsigned* err) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 1023u) == 1023u && *abort_flag) return false;
  }
  *abort_flag = 1u;
  record_error(err, kErrTimeout);
  return false;
}

template <int D>
__global__ void __launch_bounds__(160, 2) verify_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                                                           const __grid_constant__ CUtensorMap tmv) {
  using T = TcTraits<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));  // generic pointer to `base`
  const uint32_t sP = base + T::kOffP;
  const uint32_t sQ = base + T::kOffQ;
  const uint32_t sStage = base + T::kOffStage;
  // barriers (each + 8 * (step % 2) where paired)
  const uint32_t bar_kfull = base + T::kOffBar;     // K tile of a stage landed
  const uint32_t bar_vfull = bar_kfull + 16;        // V tile of a stage landed
  const uint32_t bar_kempty = bar_vfull + 16;       // QK of a stage done: K tile reusable
  const uint32_t bar_o_done = bar_kempty + 16;      // PV of a step done: V tile and P buffer reusable
  const uint32_t bar_p_ready = bar_o_done + 16;     // softmax wrote P of a step
  const uint32_t bar_s_ready = bar_p_ready + 16;    // S of a step in tensor memory
  const uint32_t bar_s_free = bar_s_ready + 8;      // softmax copied S out of tensor memory
  const uint32_t bar_final = bar_s_free + 8;        // every MMA issued has completed
  uint32_t* misc = reinterpret_cast<uint32_t*>(gbase + T::kOffMisc);
  volatile uint32_t* abort_flag = misc + 1;

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

  // rows that see no token (context shorter than q_len) come out as zeros; flag them
  if (L < QL && part == 0 && g == 0 && threadIdx.x == 0) record_error(p.err, kErrShortContext);
  if (L <= 0) {  // no page at all: zero the group's rows once
    if (part == 0) {
      for (int idx = threadIdx.x; idx < R * D; idx += T::kThreads) {
        const int rr = idx / D, dd = idx - rr * D;
        const int i = rr / G, h = rr - i * G;
        p.out[(((size_t)b * QL + i) * Hq + g * G + h) * D + dd] = __float2bfloat16(0.f);
      }
    }
    return;
  }
  const int npages = (L + T::kBS - 1) / T::kBS;
  const int ppp = p.pages_per_partition;
  const int pbeg = part * ppp;
  if (pbeg >= npages) return;
  const int pend = min(npages, pbeg + ppp);
  const int nparts = (npages + ppp - 1) / ppp;
  if (pend - pbeg > T::kMaxPages) {  // the host plans at most kMaxPages pages per partition
    if (threadIdx.x == 0) record_error(p.err, kErrShortContext);
    return;
  }
  const int limit_tok = min(L, pend * T::kBS);  // tokens of this partition end here
  const int nsteps = (pend - pbeg + T::kTP - 1) / T::kTP;
  const int32_t* bt = p.block_table + (size_t)b * p.max_blocks_per_seq;
  int32_t* ids = reinterpret_cast<int32_t*>(gbase + T::kOffIds);  // physical block of each page, or -1

  // ---- set-up: block ids, barriers, Q rows, tensor-memory allocation --------------------------
  for (int pg = threadIdx.x; pg < pend - pbeg; pg += T::kThreads) {
    const int pb = bt[pbeg + pg];
    const bool okb = pb >= 0 && pb < p.num_blocks;
    if (!okb) record_error(p.err, kErrBlockId);
    ids[pg] = okb ? pb : -1;
  }
  if (threadIdx.x == 128) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
      mbar_init(bar_o_done + 8 * s, 1);
      mbar_init(bar_p_ready + 8 * s, 2);
    }
    mbar_init(bar_s_ready, 1);
    mbar_init(bar_s_free, 2);
    mbar_init(bar_final, 1);
    *abort_flag = 0u;
    fence_mbar_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  const int r = threadIdx.x;  // softmax threads: query row r (TMEM lane r)
  if (warp < 2) {
    // Q row r (zeros for padding rows) as K-major 128-byte-swizzled rows of 64 dims
    const __nv_bfloat16* qrow = nullptr;
    if (r < R) qrow = p.q + (((size_t)b * QL + r / G) * Hq + g * G + r % G) * D;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (qrow) v = *reinterpret_cast<const uint4*>(qrow + c * 8);
      const uint32_t dst = sQ + (c >> 3) * (T::kRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + T::kOffMisc),
                 "r"(T::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const uint32_t tS = tmem + T::kSCol;
  const uint32_t tO = tmem + T::kOCol;

  // physical block of page `pg` of step `st`, or -1 (past the partition, or out of range)
  auto page_block = [&](int st, int pg) {
    const int page = st * T::kTP + pg;
    return page < pend - pbeg ? ids[page] : -1;
  };

  if (warp >= 3) {
    // ========== TMA producers: warp 3 fills the K ring, warp 4 the V ring (2 stages each) ======
    if (lane == 0) {
      const bool is_k = warp == 3;
      const CUtensorMap* map = is_k ? &tmk : &tmv;
      const uint32_t tile_off = is_k ? 0u : (uint32_t)T::kKTile;
      const uint32_t bar_full = is_k ? bar_kfull : bar_vfull;
      // a stage is free once QK (K tile) or PV (V tile) of the step two before has completed
      const uint32_t bar_free = is_k ? bar_kempty : bar_o_done;
      int st = 0;
      uint32_t idle = 0;
      while (st < nsteps) {
        if (st >= 2 && !mbar_test_wait(bar_free + 8 * (st & 1), ((st - 2) >> 1) & 1)) {
          if (++idle >= kWaitLimit || ((idle & 1023u) == 0 && *abort_flag)) {
            if (!*abort_flag) record_error(p.err, kErrTimeout);
            *abort_flag = 1u;
            break;
          }
          continue;
        }
        idle = 0;
        const int s = st & 1;
        const uint32_t region = sStage + s * T::kStageBytes + tile_off;
        const uint32_t bar = bar_full + 8 * s;
        int pbs[T::kTP];
        int npg = 0;
#pragma unroll
        for (int pg = 0; pg < T::kTP; ++pg) {
          pbs[pg] = page_block(st, pg);
          npg += pbs[pg] >= 0;
        }
        if (npg == 0) {
          mbar_arrive(bar);
        } else {
          mbar_arrive_expect_tx(bar, npg * T::kHalves * T::kBoxBytes);
#pragma unroll
          for (int pg = 0; pg < T::kTP; ++pg) {
            if (pbs[pg] < 0) continue;
            const int row = (pbs[pg] * p.num_kv_heads + g) * T::kBS;
#pragma unroll
            for (int hh = 0; hh < T::kHalves; ++hh)
              tma_load_2d(region + hh * T::kRegion + pg * T::kBoxBytes, map, hh * 64, row, bar);
          }
        }
        ++st;
      }
      // every copy started has landed before the CTA's shared memory can go away
      for (int k = max(0, st - 2); k < st; ++k) mbar_wait(bar_full + 8 * (k & 1), (k >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ======================= MMA issuer ======================================================
    if (lane == 0) {
      auto mma_qk = [&](int st) {
        const uint32_t kreg = sStage + (st & 1) * T::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * T::kRegion + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * (T::kRows * 128) + (kk & 3) * 32;
          umma_bf16(tS, smem_desc(sQ + qoff, 16, 1024), smem_desc(kreg + koff, 16, 1024), T::kIdescQK,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(bar_s_ready);
        umma_commit(bar_kempty + 8 * (st & 1));
      };
      auto mma_pv = [&](int st) {
        const uint32_t vreg = sStage + (st & 1) * T::kStageBytes + T::kKTile;
        const uint32_t preg = sP + (st & 1) * T::kPBytes;
#pragma unroll
        for (int kk = 0; kk < T::kStepTokens / 16; ++kk) {
          // A = P (K-major, 16 tokens = 32 B per step); B = V (MN-major: 64-dim atoms one
          // half region apart, 8-token groups 1024 B apart, 16 tokens = 2048 B per step)
          umma_bf16(tO, smem_desc(preg + kk * 32, 16, 1024), smem_desc(vreg + kk * 2048, T::kRegion, 1024),
                    T::kIdescPV, (st > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar_o_done + 8 * (st & 1));
      };
      // S(k+1) is computed while the softmax warps still work on step k: QK(k+1) goes in as soon
      // as its K tile is there and S(k) has been copied out of tensor memory; PV(k) goes in once
      // P(k) and the V tile are there.  Whichever is ready first is issued first.
      int next_qk = 0, next_pv = 0;
      uint32_t idle = 0;
      while (next_pv < nsteps) {
        bool progressed = false;
        if (next_qk < nsteps && mbar_test_wait(bar_kfull + 8 * (next_qk & 1), (next_qk >> 1) & 1) &&
            (next_qk == 0 || mbar_test_wait(bar_s_free, (next_qk - 1) & 1))) {
          tc_fence_after();
          mma_qk(next_qk++);
          progressed = true;
        }
        if (next_pv < next_qk && mbar_test_wait(bar_p_ready + 8 * (next_pv & 1), (next_pv >> 1) & 1) &&
            mbar_test_wait(bar_vfull + 8 * (next_pv & 1), (next_pv >> 1) & 1)) {
          tc_fence_after();
          mma_pv(next_pv++);
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle >= kWaitLimit || ((idle & 1023u) == 0 && *abort_flag)) {
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
  } else {
    // ======================= softmax warps: thread r owns query row r =======================
    const bool row_live = r < R;
    const int n_r = row_live ? L - QL + r / G + 1 : 0;  // causal limit of this row
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    auto step_pages_ok = [&](int st) {
      unsigned okp = 0;
#pragma unroll
      for (int pg = 0; pg < T::kTP; ++pg)
        if (page_block(st, pg) >= 0) okp |= 1u << pg;
      return okp;
    };
    unsigned pok_next = step_pages_ok(0);
    for (int k = 0; k < nsteps; ++k) {
      const unsigned pok = pok_next;
      if (!(ok = wait_or_abort(bar_s_ready, k & 1, abort_flag, p.err))) break;
      tc_fence_after();
      float s[T::kStepTokens];
      {
        uint32_t raw0[32], raw1[32];
        tmem_ld_x32(tS + lane_off, raw0);
        tmem_ld_x32(tS + lane_off + 32, raw1);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(raw0[c]);
          s[32 + c] = __uint_as_float(raw1[c]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_s_free);
      if (k + 1 < nsteps) pok_next = step_pages_ok(k + 1);  // block-table reads for the next step

      const int tok0 = (pbeg + k * T::kTP) * T::kBS;
      // interior steps (every page present, inside the partition, before the causal band) need no
      // mask; padding rows are scaled by 0 and never used
      const bool full_step = pok == (1u << T::kTP) - 1 && tok0 + T::kStepTokens <= limit_tok &&
                             tok0 + T::kStepTokens <= L - QL + 1;
      float mxs[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mxs[j] = -INFINITY;
      if (full_step) {
        const float sc = row_live ? p.scale_log2 : 0.f;
#pragma unroll
        for (int c = 0; c < T::kStepTokens; ++c) {
          s[c] *= sc;
          mxs[c & 7] = fmaxf(mxs[c & 7], s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < T::kStepTokens; ++c) {
          const int tok = tok0 + c;
          const bool v = ((pok >> (c >> 4)) & 1u) && tok < limit_tok && tok < n_r;
          s[c] = v ? s[c] * p.scale_log2 : -INFINITY;
          mxs[c & 7] = fmaxf(mxs[c & 7], s[c]);
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                             fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
      const float m_new = fmaxf(m_used, mx);
      const bool need = row_live && (m_used != -INFINITY) && (m_new > m_used + 8.f);

      // P buffer k % 2 was last read by PV(k - 2)
      if (k >= 2) {
        if (!(ok = wait_or_abort(bar_o_done + 8 * (k & 1), ((k - 2) >> 1) & 1, abort_flag, p.err))) break;
      }
      if (__any_sync(0xffffffffu, need)) {
        // the O row is rescaled only once PV(k - 1) has landed in it
        if (!(ok = wait_or_abort(bar_o_done + 8 * ((k - 1) & 1), ((k - 1) >> 1) & 1, abort_flag, p.err))) break;
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

      // zero V rows of tokens that hold no data (block tails, stale stages): P is 0 there, but
      // 0 * NaN would still poison the product.  Thread r handles token r of the step, after the
      // step's V tile has landed.
      {
        const int tok = tok0 + r;
        const bool tok_ok = ((pok >> (r >> 4)) & 1u) && tok < limit_tok;
        if (__any_sync(0xffffffffu, !tok_ok)) {
          if (!(ok = wait_or_abort(bar_vfull + 8 * (k & 1), (k >> 1) & 1, abort_flag, p.err))) break;
          if (!tok_ok) {
            const uint32_t vrow = sStage + (k & 1) * T::kStageBytes + T::kKTile + r * 128;
#pragma unroll
            for (int hh = 0; hh < T::kHalves; ++hh)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + hh * T::kRegion + c * 16), "r"(0u)
                             : "memory");
          }
        }
      }
      // P row r: bf16, K-major 128-byte swizzle (64 tokens = 8 chunks of 16 B)
      float ps[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) ps[j] = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float e0 = fast_exp2(s[c * 8 + 2 * e] - basev);
          const float e1 = fast_exp2(s[c * 8 + 2 * e + 1] - basev);
          ps[2 * e] += e0;
          ps[2 * e + 1] += e1;
          w[e] = pack_bf16(e0, e1);
        }
        const uint32_t dst = sP + (k & 1) * T::kPBytes + r * 128 + ((c ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
      }
      const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      l += psum;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_ready + 8 * (k & 1));
    }

    // ---- epilogue: O row / l -----------------------------------------------------------
    if (ok) ok = wait_or_abort(bar_o_done + 8 * ((nsteps - 1) & 1), ((nsteps - 1) >> 1) & 1, abort_flag, p.err);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const int i = r / G, h = r - i * G;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t orow = ((size_t)b * QL + i) * Hq + g * G + h;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t raw[32];
        tmem_ld_x32(tO + lane_off + c0, raw);
        tmem_wait_ld();
        if (!row_live) continue;
        if (nparts == 1) {
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
          float* dst = p.part_o + (orow * p.max_partitions + part) * D + c0;
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(dst + c) =
                make_float4(__uint_as_float(raw[c]) * inv, __uint_as_float(raw[c + 1]) * inv,
                            __uint_as_float(raw[c + 2]) * inv, __uint_as_float(raw[c + 3]) * inv);
        }
      }
      if (row_live && nparts > 1)
        p.part_lse[orow * p.max_partitions + part] = (l > 0.f) ? m_used + __log2f(l) : -INFINITY;
    }
  }

  // the merge kernel (launched as a programmatic dependent) may start its prologue now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(T::kTmemCols) : "memory");
  }
}

template <int D>
cudaError_t launch_d(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  using T = TcTraits<D>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(verify_tc_kernel<D>), T::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_partitions, p.num_kv_heads, p.num_seqs);
  verify_tc_kernel<D><<<grid, T::kThreads, T::kSmem, st>>>(p, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify_tc(const AttnParams& p, const Launch& l, const CUtensorMap& tk, const CUtensorMap& tv) {
  if (l.group * p.q_len > TcTraits<128>::kRows) return cudaErrorInvalidConfiguration;
  if (l.head_dim == 128) return launch_d<128>(p, tk, tv, l.stream);
  if (l.head_dim == 64) return launch_d<64>(p, tk, tv, l.stream);
  return cudaErrorInvalidConfiguration;
}

}  // namespace pa
