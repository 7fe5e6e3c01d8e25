// score_tc2.cu -- DSA indexer prefill scoring on CTA pairs (2-SM tcgen05 MMA).
//
// Same result as score_tc.cu (GLM5 TensorCast adaptation design, "性能模型设计" buckets
// 6 and 7: q-k index score MMA; head weight multiply, head reduce, FP8 relu / q-scale
// / k-scale shaping), organised for the prefill shape N = 256 (four queries of 64
// heads, or 256 / H queries):
//
//   a cluster of two CTAs on two SMs works on 256-key tiles.  Each CTA stages its
//   own 128 keys (MMA A rows) and half of the q tile (MMA B rows 0..127 or
//   128..255); the even CTA issues tcgen05.mma.cta_group::2 with M = 256, N = 256,
//   so each SM reads only its A half and its B half from shared memory while each
//   TMEM holds the accumulators of its own 128 keys for all 256 q columns.
//   Each SM reads a third less operand data per flop than with the single-SM
//   kernel.  Selected with DSA_PAIR_MMA=1; on GB300 it is currently slower than the
//   single-SM kernel (whose tensor pipe is not operand-bound once its issuing thread
//   is lean), so the single-SM kernel is the default.
//
// Warp roles per CTA (320 threads): warp 0 loads (TMA into its own shared memory,
// completion counted on the even CTA's barriers), warp 1 allocates TMEM (both CTAs,
// jointly) and, in the even CTA, issues the MMAs; warps 2..9 are the epilogue over
// the CTA's 128 keys, identical to the single-SM prefill epilogue.
// Barriers the peer arrives on are waited on with cluster-scope acquire; every wait
// is bounded and a timeout records kStatusTimeout.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kN2 = 256;          // q columns per tile (queries x heads)
constexpr int kHalfN = kN2 / 2;   // q rows staged per CTA
constexpr int kPairKeys = 2 * kBlockM;

struct Plan2 {
  uint32_t q[2];
  uint32_t k[kMaxKStages];
  uint32_t wbuf, qsbuf, ksbuf, bars, misc, total;
};

__host__ __device__ inline Plan2 plan2(int D, int q_fp8, int k_fp8, int nK) {
  Plan2 p{};
  uint32_t off = 0;
  const uint32_t qb = static_cast<uint32_t>(kHalfN) * D * (q_fp8 ? 1 : 2);
  const uint32_t kb = static_cast<uint32_t>(kBlockM) * D * (k_fp8 ? 1 : 2);
  for (int i = 0; i < 2; ++i) { p.q[i] = off; off += qb; }
  for (int i = 0; i < kMaxKStages; ++i) { p.k[i] = off; if (i < nK) off += kb; }
  p.wbuf = off;  off += 2u * kN2 * 4u;
  p.qsbuf = off; if (q_fp8) off += 2u * kN2 * 4u;
  p.ksbuf = off; if (k_fp8) off += static_cast<uint32_t>(nK) * kBlockM * 4u;
  p.bars = off;  off += 64u * 8u;
  p.misc = off;  off += 16u;
  p.total = off;
  return p;
}

enum {
  bQFull = 0,    // [2] even CTA: two arrive.expect_tx (one per CTA) + TMA bytes of both halves
  bQEmpty = 2,   // [2] each CTA: MMA commit (multicast) + 8 local epilogue warps
  bWFull = 4,    // [2] each CTA: 32 cp.async arrivals (w, q_scale of the item)
  bTFull = 6,    // [2] each CTA: MMA commit (multicast)
  bTEmpty = 8,   // [2] even CTA: 8 epilogue warps of each CTA
  bFold = 10,    // [2][2] each CTA, per epilogue half: q-scale folding done
  bDone = 14,    // even CTA: final commit
  bKFull = 15,   // [nK] even CTA: two arrive.expect_tx + TMA bytes of both key halves
  bKEmpty = 15 + kMaxKStages,   // [nK] each CTA: MMA commit (+ 8 epilogue warps for FP8 keys)
  bKSFull = 15 + 2 * kMaxKStages  // [nK] each CTA: 32 cp.async arrivals (k scales)
};
static_assert(15 + 3 * kMaxKStages <= 64, "barrier slots exceed the bars region");

struct Item2 {
  int row0, pos0, kt0, kt1, b, nrows;
};

template <int NQ>
__device__ __forceinline__ bool fetch_item2(const ScoreArgs& a, int n_items, int it, Item2& I) {
  const long long G = gridDim.x / 2, c = blockIdx.x / 2;  // one work stream per CTA pair
  const long long idx = static_cast<long long>(it) * G + ((it & 1) ? (G - 1 - c) : c);
  if (idx >= n_items) return false;
  if (!a.paged) {
    const int qb = a.n_dense_items - 1 - static_cast<int>(idx);
    I.row0 = qb * NQ;
    I.nrows = min(NQ, a.T - I.row0);
    I.pos0 = a.q_pos0 + I.row0;
    I.b = 0;
    const int last = min(I.pos0 + I.nrows - 1, a.S - 1);
    I.kt0 = 0;
    I.kt1 = (last + kPairKeys) / kPairKeys;
  } else {
    const WorkItem w = a.items[idx];
    I.row0 = w.row0;
    I.pos0 = w.pos0;
    I.kt0 = w.kt & 0xFFFF;
    I.kt1 = (w.kt >> 16) & 0xFFFF;
    I.b = w.bn & 0xFFFFFF;
    I.nrows = (w.bn >> 24) & 0xFF;
  }
  return true;
}

__device__ __forceinline__ bool warp_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* status) {
  const bool ok = ptx::mbar_wait_cluster(bar, parity, abort, status, kStatusTimeout);
  return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------------------ loads (warp 0, both CTAs)
template <int H>
__device__ __forceinline__ void producer2(const ScoreArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                                          uint8_t* smem, const Plan2& P, uint64_t* bars, volatile int* abort,
                                          int n_items, uint32_t rank) {
  constexpr int NQ = kN2 / H;
  const int lane = threadIdx.x & 31;
  const int nK = a.num_k_stages;
  const int q_esz = a.q_fp8 ? 1 : 2, k_esz = a.k_fp8 ? 1 : 2;
  const int n_atoms_q = a.D * q_esz / 128, n_atoms_k = a.D * k_esz / 128;
  const int box_q = 128 / q_esz, box_k = 128 / k_esz;
  const uint32_t q_bytes = static_cast<uint32_t>(kHalfN) * a.D * q_esz;
  float* wbuf = reinterpret_cast<float*>(smem + P.wbuf);
  float* qsbuf = reinterpret_cast<float*>(smem + P.qsbuf);
  float* ksbuf = reinterpret_cast<float*>(smem + P.ksbuf);
  const int PS = a.page_size;
  const int ppt = a.paged ? kBlockM / PS : 1;
  const uint32_t page_bytes = static_cast<uint32_t>(PS) * a.D * k_esz;
  const int key_off = static_cast<int>(rank) * kBlockM;  // this CTA's keys inside a pair tile

  uint32_t nq = 0, nk = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    Item2 I;
    if (!fetch_item2<NQ>(a, n_items, it, I)) break;
    {
      const int s = nq & 1;
      int good = 1;
      if (lane == 0) good = ptx::mbar_wait_cluster(&bars[bQEmpty + s], ((nq >> 1) & 1) ^ 1, abort, a.status, kStatusTimeout);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) { ok = false; break; }
      // w and q_scale of all N columns (this CTA's epilogue covers every query)
      const long long base = static_cast<long long>(I.row0) * H;
      const long long lim = static_cast<long long>(a.total_rows) * H;
      for (int c = lane; c < kN2 / 4; c += 32) {
        const long long e = base + 4ll * c;
        const bool v = e + 4 <= lim;
        ptx::cp_async_16(wbuf + s * kN2 + 4 * c, v ? static_cast<const void*>(a.w + e) : static_cast<const void*>(a.w),
                         v ? 16u : 0u);
        if (a.q_fp8)
          ptx::cp_async_16(qsbuf + s * kN2 + 4 * c,
                           v ? static_cast<const void*>(a.q_scale + e) : static_cast<const void*>(a.q_scale),
                           v ? 16u : 0u);
      }
      ptx::cp_async_mbar_arrive_noinc(&bars[bWFull + s]);
      if (lane == 0) {
        const uint32_t full = ptx::mapa_shared(ptx::smem_u32(&bars[bQFull + s]), 0);
        ptx::mbar_arrive_expect_tx_cluster(full, q_bytes);
        for (int at = 0; at < n_atoms_q; ++at)
          ptx::tma_load_2d_pair(smem + P.q[s] + at * kHalfN * 128, tq, full, at * box_q,
                                I.row0 * H + static_cast<int>(rank) * kHalfN);
      }
      ++nq;
    }
    const int32_t* bt_row = a.paged ? a.block_tables + static_cast<long long>(I.b) * a.max_pages_per_seq : nullptr;
    int win0 = -(1 << 30);
    int pg_win = -1;
    const int pos_last = I.pos0 + I.nrows - 1;
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int s = nk % nK;
      int good = 1;
      if (lane == 0) good = ptx::mbar_wait_cluster(&bars[bKEmpty + s], ((nk / nK) & 1) ^ 1, abort, a.status, kStatusTimeout);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) { ok = false; break; }
      const uint32_t full = ptx::mapa_shared(ptx::smem_u32(&bars[bKFull + s]), 0);
      uint8_t* dst = smem + P.k[s];
      const int key0 = kt * kPairKeys + key_off;  // first key of this CTA's 128
      if (!a.paged) {
        if (a.k_fp8) {
          const long long e = static_cast<long long>(key0) + 4 * lane;
          float* d4 = ksbuf + s * kBlockM + 4 * lane;
          if (e + 4 <= a.S) {
            ptx::cp_async_16(d4, a.k_scale + e, 16u);
          } else {
            for (int j = 0; j < 4; ++j) {
              const bool v = e + j < a.S;
              ptx::cp_async_4(d4 + j, v ? a.k_scale + e + j : a.k_scale, v ? 4u : 0u);
            }
          }
          ptx::cp_async_mbar_arrive_noinc(&bars[bKSFull + s]);
        }
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx_cluster(full, static_cast<uint32_t>(kBlockM) * a.D * k_esz);
          for (int at = 0; at < n_atoms_k; ++at)
            ptx::tma_load_2d_pair(dst + at * kBlockM * 128, tk, full, at * box_k, key0);
        }
      } else {
        const int lp0 = key0 / PS;
        if (lp0 < win0 || lp0 + ppt > win0 + 32) {
          win0 = lp0;
          const int lp = win0 + lane;
          pg_win = lp < a.max_pages_per_seq ? __ldg(bt_row + lp) : -1;
        }
        int phys = -1;
        bool valid = false;
        {
          const int j = lane;
          const int src_lane = (lp0 - win0 + (j < ppt ? j : 0)) & 31;
          const int pg = __shfl_sync(0xffffffffu, pg_win, src_lane);
          const bool needed = j < ppt && static_cast<long long>(lp0 + j) * PS <= pos_last;
          valid = needed && pg >= 0 && pg < a.num_pages;
          if (needed && !valid) atomicOr(a.status, kStatusBadPage);
          phys = valid ? pg : -1;
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        if (a.k_fp8) {
          const int j = (4 * lane) / PS;
          const int pj = __shfl_sync(0xffffffffu, phys, j);
          const bool v = (vmask >> j) & 1u;
          const float* src = v ? a.k_scale + static_cast<long long>(pj) * PS + (4 * lane) % PS : a.k_scale;
          ptx::cp_async_16(ksbuf + s * kBlockM + 4 * lane, src, v ? 16u : 0u);
          ptx::cp_async_mbar_arrive_noinc(&bars[bKSFull + s]);
        }
        int pj_all[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) pj_all[j] = __shfl_sync(0xffffffffu, phys, j);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx_cluster(full, static_cast<uint32_t>(__popc(vmask)) * page_bytes);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j < ppt && ((vmask >> j) & 1u)) {
              for (int at = 0; at < n_atoms_k; ++at)
                ptx::tma_load_3d_pair(dst + at * kBlockM * 128 + j * PS * 128, tk, full, at * box_k, 0, pj_all[j]);
            }
          }
        }
      }
      ++nk;
    }
  }
}

// ------------------------------------------------------------------ MMA issuer (even CTA, warp 1 lane 0)
// Kept lean like the single-SM issuer: incremental ring slots, descriptors by offset.
template <int H, bool F8, int NSTEPS>
__device__ __forceinline__ void mma2_loop(const ScoreArgs& a, uint8_t* smem, const Plan2& P, uint64_t* bars,
                                          volatile int* abort, int n_items, uint32_t tmem_base) {
  constexpr int NQ = kN2 / H;
  const int nK = a.num_k_stages;
  const uint32_t idesc = ptx::idesc_f32acc(2 * kBlockM, kN2, !F8);
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t k_stage_bytes = P.k[1] - P.k[0];
  const uint32_t k_base = sbase + P.k[0];
  uint32_t nq = 0, nt = 0;
  uint32_t sk = 0, kphase = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    Item2 I;
    if (!fetch_item2<NQ>(a, n_items, it, I)) break;
    const int sq = nq & 1;
    if (!ptx::mbar_wait_cluster(&bars[bQFull + sq], (nq >> 1) & 1, abort, a.status, kStatusTimeout)) break;
    const uint64_t bdesc0 = ptx::sw128_kmajor_desc(sbase + P.q[sq]);
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int acc = nt & 1;
      if (!ptx::mbar_wait_cluster(&bars[bKFull + sk], kphase, abort, a.status, kStatusTimeout) ||
          !ptx::mbar_wait_cluster(&bars[bTEmpty + acc], ((nt >> 1) & 1) ^ 1, abort, a.status, kStatusTimeout)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
      const uint64_t adesc0 = ptx::sw128_kmajor_desc(k_base + sk * k_stage_bytes);
#pragma unroll
      for (int j = 0; j < NSTEPS; ++j) {
        const uint64_t ad = adesc0 + static_cast<uint64_t>(((j >> 2) * (kBlockM * 128) + (j & 3) * 32) >> 4);
        const uint64_t bd = bdesc0 + static_cast<uint64_t>(((j >> 2) * (kHalfN * 128) + (j & 3) * 32) >> 4);
        if (F8) ptx::mma_f8_pair(d_tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
        else ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
      }
      ptx::mma_commit_pair(&bars[bKEmpty + sk], 3);
      ptx::mma_commit_pair(&bars[bTFull + acc], 3);
      if (++sk == static_cast<uint32_t>(nK)) { sk = 0; kphase ^= 1u; }
      ++nt;
    }
    if (!ok) break;
    ptx::mma_commit_pair(&bars[bQEmpty + sq], 3);
    ++nq;
  }
  ptx::mma_commit_pair(&bars[bDone], 1);
  ptx::mbar_wait_cluster_drain(&bars[bDone], 0, a.status, kStatusTimeout, 200000000ull);
}

template <int H>
__device__ __forceinline__ void mma2(const ScoreArgs& a, uint8_t* smem, const Plan2& P, uint64_t* bars,
                                     volatile int* abort, int n_items, uint32_t tmem_base) {
  if (a.k_fp8) mma2_loop<H, true, 4>(a, smem, P, bars, abort, n_items, tmem_base);
  else if (a.D == 128) mma2_loop<H, false, 8>(a, smem, P, bars, abort, n_items, tmem_base);
  else mma2_loop<H, false, 4>(a, smem, P, bars, abort, n_items, tmem_base);
}

// ------------------------------------------------------------------ epilogue (warps 2..9, both CTAs)
template <int H>
__device__ __forceinline__ void epilogue2(const ScoreArgs& a, uint8_t* smem, const Plan2& P, uint64_t* bars,
                                          volatile int* abort, int n_items, uint32_t tmem_base, uint32_t rank) {
  constexpr int NQ = kN2 / H;
  constexpr int NCOLS = kN2 / 2;
  constexpr int QH = NCOLS / H;
  constexpr int NCH = NCOLS / 32;
  constexpr int NP = (32 / (2 * QH)) > 4 ? 4 : ((32 / (2 * QH)) < 1 ? 1 : (32 / (2 * QH)));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = (warp - 2) >> 2;
  const int quarter = warp & 3;
  const int m = quarter * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int col0 = half * NCOLS;
  const int q0 = col0 / H;
  const int nK = a.num_k_stages;
  float* wbuf = reinterpret_cast<float*>(smem + P.wbuf);
  const float* qsbuf = reinterpret_cast<const float*>(smem + P.qsbuf);
  const float* ksbuf = reinterpret_cast<const float*>(smem + P.ksbuf);
  const int fold_t = static_cast<int>(threadIdx.x) - 64 - half * 128;
  const int key_off = static_cast<int>(rank) * kBlockM;

  uint32_t nq = 0, nk = 0, nt = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    Item2 I;
    if (!fetch_item2<NQ>(a, n_items, it, I)) break;
    const int sq = nq & 1;
    if (!warp_wait_cl(&bars[bWFull + sq], (nq >> 1) & 1, abort, a.status)) break;
    float* wq = wbuf + sq * kN2;
    if (a.q_fp8) {
      const int c = col0 + fold_t;
      wq[c] *= qsbuf[sq * kN2 + c];
      uint64_t* fb = &bars[bFold + sq * 2 + half];
      ptx::mbar_arrive(fb);
      if (!warp_wait_cl(fb, (nq >> 1) & 1, abort, a.status)) break;
    }
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int sk = nk % nK;
      const int acc = nt & 1;
      if (a.k_fp8 && !warp_wait_cl(&bars[bKSFull + sk], (nk / nK) & 1, abort, a.status)) {
        ok = false;
        break;
      }
      if (!warp_wait_cl(&bars[bTFull + acc], (nt >> 1) & 1, abort, a.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float2 part[QH][NP];
#pragma unroll
      for (int j = 0; j < QH; ++j)
#pragma unroll
        for (int p = 0; p < NP; ++p) part[j][p] = make_float2(0.f, 0.f);
      const uint32_t tcol = tmem_base + lane_addr + static_cast<uint32_t>(acc * 256 + col0);
      uint32_t xa[32], xb[32];
      ptx::tmem_ld_32x32b_x32(tcol, xa);
      ptx::tmem_ld_wait_regs(xa);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        if (c + 1 < NCH) ptx::tmem_ld_32x32b_x32(tcol + 32 * (c + 1), xb);
        const float4* w4 = reinterpret_cast<const float4*>(wq + col0 + 32 * c);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 wv = w4[i4];
          const int cc = 32 * c + 4 * i4;
          const int jq = cc / H;
          const int p0 = ((cc % H) / 2) % NP, p1 = ((cc % H) / 2 + 1) % NP;
          const float r0 = fmaxf(__uint_as_float(xa[4 * i4 + 0]), 0.f);
          const float r1 = fmaxf(__uint_as_float(xa[4 * i4 + 1]), 0.f);
          const float r2 = fmaxf(__uint_as_float(xa[4 * i4 + 2]), 0.f);
          const float r3 = fmaxf(__uint_as_float(xa[4 * i4 + 3]), 0.f);
          ptx::ffma2(part[jq][p0], make_float2(wv.x, wv.y), make_float2(r0, r1));
          ptx::ffma2(part[jq][p1], make_float2(wv.z, wv.w), make_float2(r2, r3));
        }
        if (c + 1 < NCH) {
          ptx::tmem_ld_wait_regs(xb);
#pragma unroll
          for (int i = 0; i < 32; ++i) xa[i] = xb[i];
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&bars[bTEmpty + acc]), 0));
      float ks = 1.f;
      if (a.k_fp8) {
        ks = ksbuf[sk * kBlockM + m];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars[bKEmpty + sk]);
      }
      const int s = kt * kPairKeys + key_off + m;
      const bool key_ok = a.paged || s < a.S;
#pragma unroll
      for (int j = 0; j < QH; ++j) {
        float t = 0.f;
#pragma unroll
        for (int p = 0; p < NP; ++p) t += part[j][p].x + part[j][p].y;
        const int qi = q0 + j;
        if (qi < I.nrows && key_ok && s <= I.pos0 + qi)
          a.scores[static_cast<long long>(I.row0 + qi - a.row_base) * a.ld + s] = t * ks;
      }
      ++nk;
      ++nt;
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&bars[bQEmpty + sq]);
    ++nq;
  }
}

template <int H>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel_pair(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const ScoreArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  // the same check in both CTAs, so both return together before any cluster barrier
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusSmemAlign);
    return;
  }
  const Plan2 P = plan2(a.D, a.q_fp8, a.k_fp8, a.num_k_stages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + P.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + P.misc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars[bQFull + s], 2);
      ptx::mbar_init(&bars[bQEmpty + s], 1 + 8);
      ptx::mbar_init(&bars[bWFull + s], 32);
      ptx::mbar_init(&bars[bTFull + s], 1);
      ptx::mbar_init(&bars[bTEmpty + s], 16);
      ptx::mbar_init(&bars[bFold + 2 * s + 0], 128);
      ptx::mbar_init(&bars[bFold + 2 * s + 1], 128);
    }
    ptx::mbar_init(&bars[bDone], 1);
    for (int s = 0; s < a.num_k_stages; ++s) {
      ptx::mbar_init(&bars[bKFull + s], 2);
      ptx::mbar_init(&bars[bKEmpty + s], 1 + (a.k_fp8 ? 8 : 0));
      ptx::mbar_init(&bars[bKSFull + s], 32);
    }
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_q);
    ptx::prefetch_tmap(&tmap_k);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int n_items = a.paged ? min(*a.n_items, a.items_cap) : a.n_dense_items;

  if ((tmem_base & 0xFFFFu) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTmemAlloc);
  } else if (warp == 0) {
    producer2<H>(a, &tmap_q, &tmap_k, smem, P, bars, abort, n_items, rank);
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) mma2<H>(a, smem, P, bars, abort, n_items, tmem_base);
    __syncwarp();
  } else {
    epilogue2<H>(a, smem, P, bars, abort, n_items, tmem_base, rank);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // no CTA leaves while its peer may still touch its barriers or TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <int H>
cudaError_t launch_pair_t(const ScoreArgs& a, const CUtensorMap* tq, const CUtensorMap* tk, int grid, size_t smem,
                          cudaStream_t st) {
  auto kern = score_kernel_pair<H>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kScoreThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, *tq, *tk, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

size_t score_pair_smem_bytes(const ScoreArgs& a, int num_k_stages) {
  return plan2(a.D, a.q_fp8, a.k_fp8, num_k_stages).total;
}

cudaError_t launch_score_pair(const ScoreArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k, int grid,
                              size_t smem_bytes, cudaStream_t st) {
  switch (a.H) {
    case 4: return launch_pair_t<4>(a, tmap_q, tmap_k, grid, smem_bytes, st);
    case 8: return launch_pair_t<8>(a, tmap_q, tmap_k, grid, smem_bytes, st);
    case 16: return launch_pair_t<16>(a, tmap_q, tmap_k, grid, smem_bytes, st);
    case 32: return launch_pair_t<32>(a, tmap_q, tmap_k, grid, smem_bytes, st);
    case 64: return launch_pair_t<64>(a, tmap_q, tmap_k, grid, smem_bytes, st);
    case 128: return launch_pair_t<128>(a, tmap_q, tmap_k, grid, smem_bytes, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dsa
