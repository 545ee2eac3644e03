// Paged GQA decode (q_len = 1) on CUDA cores, sm_103a: the kernel of
// paged_attn_decode_static_scratch (paged_attn_decode runs the mma.sync kernel of pa_decode_mma.cu).
//
// One CTA per (partition, kv head, sequence).  A partition is a run of whole pages of one
// sequence; a page is the 16 x d slice of one physical block for one kv head, contiguous in
// the [num_blocks, Hkv, bs, d] pool, so the block-table gather (studybook fde-roadmap ch.10,
// section 10.4.2; aegloslab servingai 5.3.7) is one bulk copy per page for K and one for V.
//
// Four warps split the partition's pages round-robin.  Each warp owns a ring of page stages
// filled by the TMA unit (cp.async.bulk, completion on an mbarrier), so no thread spends
// instructions on moving bytes.  All G query heads of the group are scored against each K row
// while it sits in shared memory: one KV read serves the whole GQA group (section 10.1.2).
//
// Scores: 8 lanes per token, each holding d/8 dims of all G queries in registers; partial dot
// products are reduce-scattered across the 8 lanes so that each lane ends with one head's
// score.  Softmax: per-warp online softmax in base 2 (running max m, running sum l, rescale
// by 2^(m_old - m_new)) -- the tiling + online softmax of FlashAttention (section 10.1.2).
// Values: each lane owns d/32 output dims of all G heads and accumulates p * v with paired
// fp32 FMAs.  The four warps merge through shared memory; when the sequence has several
// partitions the CTA writes its normalised output and log2-sum-exp for the merge kernel.
#include "pa_kernels.h"

namespace pa {
namespace {

template <int D, int G, bool FP8>
struct DecodeTraits {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kBS = 16;
  static constexpr int kElt = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kPageBytes = kBS * kRowBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;
  // bf16: 3 CTAs per SM (12 warps) for G <= 4, 2-stage rings (shared memory bound).  E4M3 pages
  // are half the size, so G <= 4 runs 4 CTAs per SM (16 warps, 128 registers) with 3-stage
  // rings.  G = 8 needs ~255 registers: 2 CTAs with deeper rings.
  static constexpr int kMinBlocks = G >= 8 ? 2 : (FP8 ? 4 : 3);
  static constexpr int kStages = G >= 8 ? (FP8 ? 6 : 3) : (FP8 ? 3 : 2);
  static constexpr int kQD = D / 8;                       // QK dims per lane
  static constexpr int kLaneBytes = kQD * kElt;           // QK bytes per lane per row
  static constexpr int kPiece = kLaneBytes >= 16 ? 16 : kLaneBytes;
  static constexpr int kPieces = kLaneBytes / kPiece;
  static constexpr int kPieceElts = kPiece / kElt;
  static constexpr int kDPL = D / 32;                     // PV dims per lane
  static constexpr int kStageRegion = kWarps * kStages * kStageBytes;
  static constexpr int kPRegion = kWarps * (kBS * G + G) * 4;
  static constexpr int kBarRegion = kWarps * kStages * 8;
  static constexpr int kSmem = kStageRegion + kPRegion + kBarRegion;
  static_assert(kWarps * G * D * 4 + 2 * kWarps * G * 4 <= kStageRegion, "merge scratch fits");
  static_assert(kLaneBytes % kPiece == 0 && kPiece % 8 == 0, "lane slice layout");
  static_assert(kDPL % 2 == 0, "PV pairs");
};

// Head index a lane of an 8-lane token group holds after reduce_scatter8<G>.
template <int G>
__device__ __forceinline__ int head_of_lane(int j) {
  int h = 0, cnt = G;
#pragma unroll
  for (int lvl = 0; lvl < 3; ++lvl) {
    const int m = 4 >> lvl;
    if (cnt > 1) {
      const int half = cnt / 2;
      if (j & m) h += half;
      cnt = half;
    }
  }
  return h;
}

// Sum G partial dot products over the 8 lanes of a token group; each lane keeps one head.
template <int G>
__device__ __forceinline__ float reduce_scatter8(float (&a)[G], int j) {
  int cnt = G;
#pragma unroll
  for (int lvl = 0; lvl < 3; ++lvl) {
    const int m = 4 >> lvl;
    if (cnt > 1) {
      const int half = cnt / 2;
      const bool upper = (j & m) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float keep = upper ? a[half + i] : a[i];
        const float send = upper ? a[i] : a[half + i];
        a[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
      }
      cnt = half;
    } else {
      a[0] += __shfl_xor_sync(0xffffffffu, a[0], m);
    }
  }
  return a[0];
}

// The lane's QK slice of one K row, as fp32 pairs (raw E4M3 values for fp8: the page scale is
// applied to the finished score).
template <class T, bool FP8>
__device__ __forceinline__ void load_k_slice(const uint8_t* row, int j, float2 (&kf)[T::kQD / 2]) {
#pragma unroll
  for (int c = 0; c < T::kPieces; ++c) {
    const uint8_t* src = row + (j + 8 * c) * T::kPiece;
    uint32_t w[T::kPiece / 4];
    if constexpr (T::kPiece == 16) {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      w[0] = v.x; w[1] = v.y;
    }
#pragma unroll
    for (int i = 0; i < T::kPiece / 4; ++i) {
      if constexpr (FP8) {
        kf[c * (T::kPieceElts / 2) + 2 * i] = e4m3x2_to_f2(static_cast<uint16_t>(w[i] & 0xffffu));
        kf[c * (T::kPieceElts / 2) + 2 * i + 1] = e4m3x2_to_f2(static_cast<uint16_t>(w[i] >> 16));
      } else {
        kf[c * (T::kPieceElts / 2) + i] = bf16x2_to_f2(w[i]);
      }
    }
  }
}

// The lane's PV slice (dims [lane * kDPL, lane * kDPL + kDPL)) of one V row.
template <class T, bool FP8>
__device__ __forceinline__ void load_v_slice(const uint8_t* row, int lane, float2 (&vf)[T::kDPL / 2]) {
  if constexpr (FP8) {
    if constexpr (T::kDPL == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(row + 4 * lane);
      vf[0] = e4m3x2_to_f2(static_cast<uint16_t>(w & 0xffffu));
      vf[1] = e4m3x2_to_f2(static_cast<uint16_t>(w >> 16));
    } else {
      vf[0] = e4m3x2_to_f2(*reinterpret_cast<const uint16_t*>(row + 2 * lane));
    }
  } else {
    if constexpr (T::kDPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(row + 8 * lane);
      vf[0] = bf16x2_to_f2(w.x);
      vf[1] = bf16x2_to_f2(w.y);
    } else {
      vf[0] = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(row + 4 * lane));
    }
  }
}

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(128, (DecodeTraits<D, G, FP8>::kMinBlocks)) decode_kernel(const AttnParams p) {
  using T = DecodeTraits<D, G, FP8>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int part = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int Hq = p.num_q_heads;
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
  const int ppp = p.pages_per_partition;
  const int pbeg = part * ppp;
  if (pbeg >= npages) return;
  const int pend = min(npages, pbeg + ppp);
  const int nparts = (npages + ppp - 1) / ppp;

  uint8_t* stages = smem + warp * T::kStages * T::kStageBytes;
  float* p_s = reinterpret_cast<float*>(smem + T::kStageRegion) + warp * (T::kBS * G + G);
  float* alpha_s = p_s + T::kBS * G;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::kStageRegion + T::kPRegion) + warp * T::kStages;

  const int first = pbeg + warp;
  const int nk = first < pend ? (pend - first + T::kWarps - 1) / T::kWarps : 0;
  const int32_t* bt = p.block_table + (size_t)b * p.max_blocks_per_seq;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < T::kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Block ids of the warp's pages, 32 at a time in registers (one coalesced load per window):
  // lane i of idw0 holds the id of the warp's page wb + i, idw1 the next window.  Reading them
  // with a shuffle keeps the block-table latency out of the copy issue.
  auto load_window = [&](int kb) {
    const int kk = kb + lane;
    return kk < nk ? bt[first + T::kWarps * kk] : -1;
  };
  int wb = 0;
  int idw0 = load_window(0);
  int idw1 = load_window(32);
  auto id_of = [&](int k) {  // k in [wb, wb + 64), warp-uniform
    const int o = k - wb;
    return o < 32 ? __shfl_sync(0xffffffffu, idw0, o) : __shfl_sync(0xffffffffu, idw1, o - 32);
  };
  // fp8: the K and V scales of the window's pages, loaded with the window (a page's scale is then
  // a shuffle, not a dependent global load after its copy lands)
  auto load_scale = [&](const float* sc, int id) {
    return (FP8 && id >= 0 && id < p.num_blocks) ? sc[(size_t)id * p.num_kv_heads + g] : 1.f;
  };
  float ksw0 = load_scale(p.k_scale, idw0), vsw0 = load_scale(p.v_scale, idw0);
  float ksw1 = load_scale(p.k_scale, idw1), vsw1 = load_scale(p.v_scale, idw1);

  // whole warp: lane 0 starts the copies of the warp's k-th page into stage k % kStages
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
    const size_t off = ((size_t)pb * p.num_kv_heads + g) * T::kPageBytes;
    const uint32_t dst = smem_addr(stages + s * T::kStageBytes);
    mbar_arrive_expect_tx(bar, 2 * T::kPageBytes);
    bulk_copy_g2s(dst, p.k_cache + off, T::kPageBytes, bar);
    bulk_copy_g2s(dst + T::kPageBytes, p.v_cache + off, T::kPageBytes, bar);
  };
  {
    const int n0 = nk < T::kStages ? nk : T::kStages;
    for (int k = 0; k < n0; ++k) issue(k);
  }

  const int j = lane & 7;  // position in the 8-lane token group
  const int r = lane >> 3; // token slot of the group (tokens r, r+4, r+8, r+12 of a page)
  const int myh = head_of_lane<G>(j);

  // queries of the group, pre-scaled into base-2 score units, in the lane's QK dims
  float2 q2[G][T::kQD / 2];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const __nv_bfloat16* qrow = p.q + ((size_t)b * Hq + g * G + h) * D;
#pragma unroll
    for (int c = 0; c < T::kPieces; ++c) {
      const int d0 = ((j + 8 * c) * T::kPiece) / T::kElt;
#pragma unroll
      for (int e = 0; e < T::kPieceElts; e += 2) {
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(qrow + d0 + e));
        q2[h][(c * T::kPieceElts + e) / 2] = make_float2(v.x * p.scale_log2, v.y * p.scale_log2);
      }
    }
  }

  float m_run = -INFINITY;
  float l_part = 0.f;
  float2 acc[G][T::kDPL / 2];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < T::kDPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);

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
    if (k == wb + 32) {  // slide the id window (the issue below looks at most kStages ahead)
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
      float ks = 1.f, vs = 1.f;
      if constexpr (FP8) {
        const int o = k - wb;  // k is in [wb, wb + 32) here
        ks = __shfl_sync(0xffffffffu, ksw0, o);
        vs = __shfl_sync(0xffffffffu, vsw0, o);
      }
      float sc[4];
#pragma unroll
      for (int sub = 0; sub < 4; ++sub) {
        const int t = r + 4 * sub;
        float2 kf[T::kQD / 2];
        load_k_slice<T, FP8>(kp + t * T::kRowBytes, j, kf);
        float part_s[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float2 a = make_float2(0.f, 0.f);
#pragma unroll
          for (int i = 0; i < T::kQD / 2; ++i) a = ffma2(q2[h][i], kf[i], a);
          part_s[h] = a.x + a.y;
        }
        float sv = reduce_scatter8<G>(part_s, j);
        if constexpr (FP8) sv *= ks;
        sc[sub] = (t < valid) ? sv : -INFINITY;
      }
      float mloc = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 8));
      mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
      const float m_new = fmaxf(m_run, mloc);
      const float alpha = fast_exp2(m_run - m_new);
      m_run = m_new;
      float psum = 0.f;
#pragma unroll
      for (int sub = 0; sub < 4; ++sub) {
        const float pv = fast_exp2(sc[sub] - m_new);
        psum += pv;
        p_s[(r + 4 * sub) * G + myh] = pv * vs;
      }
      l_part = l_part * alpha + psum;
      if (r == 0) alpha_s[myh] = alpha;
      __syncwarp();
      if (__any_sync(0xffffffffu, alpha != 1.f)) {  // a running max moved: rescale the outputs
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float al = alpha_s[h];
#pragma unroll
          for (int e = 0; e < T::kDPL / 2; ++e) acc[h][e] = ffma2(make_float2(al, al), acc[h][e], make_float2(0.f, 0.f));
        }
      }
      // acc[h] += p[t][h] * v[t] for the page's valid tokens; a full page is unrolled so the
      // shared-memory loads of later tokens overlap the FMAs of earlier ones
      auto pv_token = [&](int t) {
        float2 vf[T::kDPL / 2];
        load_v_slice<T, FP8>(vp + t * T::kRowBytes, lane, vf);
        float pw[G];
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int h = 0; h < G; h += 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(p_s + t * G + h);
            pw[h] = v4.x; pw[h + 1] = v4.y; pw[h + 2] = v4.z; pw[h + 3] = v4.w;
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) pw[h] = p_s[t * G + h];
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < T::kDPL / 2; ++e)
            acc[h][e] = ffma2(make_float2(pw[h], pw[h]), vf[e], acc[h][e]);
      };
      if (valid == T::kBS) {
#pragma unroll
        for (int t = 0; t < T::kBS; ++t) pv_token(t);
      } else {
        for (int t = 0; t < valid; ++t) pv_token(t);
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
      for (int k = k_done; k < issued; ++k)
        mbar_wait(smem_addr(&bars[k % T::kStages]), (k / T::kStages) & 1);
    }
    __syncwarp();
  }

  // the merge kernel (launched as a programmatic dependent) may start its prologue now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // full l of this lane's head: sum over the four token slots
  float l_full = l_part;
  l_full += __shfl_xor_sync(0xffffffffu, l_full, 8);
  l_full += __shfl_xor_sync(0xffffffffu, l_full, 16);

  __syncthreads();  // every warp is done with its stages
  float* wacc = reinterpret_cast<float*>(smem);       // [kWarps][G][D]
  float* wm = wacc + T::kWarps * G * D;               // [kWarps][G]
  float* wl = wm + T::kWarps * G;                     // [kWarps][G]
  if (r == 0) {
    wm[warp * G + myh] = m_run;
    wl[warp * G + myh] = l_full;
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < T::kDPL / 2; ++e)
      *reinterpret_cast<float2*>(wacc + (warp * G + h) * D + lane * T::kDPL + 2 * e) = acc[h][e];
  __syncthreads();

  store_partition<G, D, T::kWarps>(p, wacc, wm, wl, b, g, part, nparts);
}

template <int D, int G, bool FP8>
cudaError_t launch_one(const AttnParams& p, cudaStream_t stream) {
  using T = DecodeTraits<D, G, FP8>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(decode_kernel<D, G, FP8>), T::kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_partitions, p.num_kv_heads, p.num_seqs);
  decode_kernel<D, G, FP8><<<grid, T::kThreads, T::kSmem, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t dispatch_group(const AttnParams& p, const Launch& l) {
  switch (l.group) {
    case 1: return launch_one<D, 1, FP8>(p, l.stream);
    case 2: return launch_one<D, 2, FP8>(p, l.stream);
    case 4: return launch_one<D, 4, FP8>(p, l.stream);
    case 8: return launch_one<D, 8, FP8>(p, l.stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace

cudaError_t launch_decode(const AttnParams& p, const Launch& l) {
  if (l.head_dim == 128) return l.fp8 ? dispatch_group<128, true>(p, l) : dispatch_group<128, false>(p, l);
  if (l.head_dim == 64) return l.fp8 ? dispatch_group<64, true>(p, l) : dispatch_group<64, false>(p, l);
  return cudaErrorInvalidConfiguration;
}

}  // namespace pa
