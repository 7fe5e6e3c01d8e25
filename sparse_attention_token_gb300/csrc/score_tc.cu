// score_tc.cu -- DSA indexer scoring on the sm_103a tensor cores.
//
// Computes, for a block of query rows and a range of 128-key tiles,
//     score[t, s] = ks[s] * sum_h w'[t, h] * max(sum_d q[t, h, d] * k[s, d], 0),   w' = w * q_scale
// (GLM5 TensorCast adaptation design, "性能模型设计" buckets 6 and 7: the q-k index
// score MMA, then head weight multiply, head reduce and the FP8 relu / q-scale /
// k-scale shaping).  The [T, H, S] intermediate never leaves the SM: it lives in
// TMEM and is reduced over heads by the epilogue warps.
//
// Tile orientation: MMA M = 128 keys (one TMEM lane per key), N = queries x heads
// (each query's H heads are H consecutive TMEM columns), K = D.  A TMEM lane then
// holds every head of one (key, query) pair, so the head reduction is in-thread.
//
// Warp roles (one CTA per SM, persistent over work items; 352 threads):
//   warp 0      TMA producer: q tile (N x D) per item into a 2-deep ring, key tiles
//               (128 x D, dense or gathered page by page through block_tables) into
//               an nK-deep ring, per-item w / q_scale by cp.async, per-tile k_scale by
//               cp.async (dense keys) or a bulk copy per page (paged keys).
//   warp 10     a second key producer when the key ring depth is even (decode tiles;
//               e4m3 prefill tiles): warp 0 takes the even key tiles, warp 10 the odd
//               ones (each owns alternate stages of the ring), so the address work and
//               TMA issue of one overlap the other's.
//   warp 1      TMEM allocator; lane 0 issues tcgen05.mma into two 256-column fp32
//               accumulators (double buffered) and commits to mbarriers.
//   warps 2..9  epilogue: tcgen05.ld, ReLU, head-weighted sum, k scale, causal mask,
//               coalesced fp32 stores.  bf16 prefill tiles (N = 256) are split by
//               columns between two warpgroups; decode tiles (N = max(64, H)) and e4m3
//               prefill tiles alternate between the warpgroups tile by tile.
//   bf16 queries against e4m3 keys (decode): the queries come as exact e4m3 hi / lo row
//               pairs (qsplit.cuh), so the MMAs are FP8 and the epilogue adds the pair
//               before the ReLU.
// Every wait is bounded; on a timeout the kernel records kStatusTimeout, all roles
// leave their loops, in-flight copies and MMAs are drained (bounded) and TMEM freed.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {

namespace {

struct SmemPlan {
  uint32_t q[2];
  uint32_t k[kMaxKStages];
  uint32_t wbuf, qsbuf, ksbuf, bars, misc, total;
};

__host__ __device__ inline SmemPlan plan_smem(int N, int D, int q_fp8, int k_fp8, int nK) {
  SmemPlan p{};
  uint32_t off = 0;
  const uint32_t qb = static_cast<uint32_t>(N) * D * (q_fp8 ? 1 : 2);
  const uint32_t kb = static_cast<uint32_t>(kBlockM) * D * (k_fp8 ? 1 : 2);
  for (int i = 0; i < 2; ++i) { p.q[i] = off; off += qb; }
  for (int i = 0; i < kMaxKStages; ++i) { p.k[i] = off; if (i < nK) off += kb; }
  p.wbuf = off;  off += 2u * N * 4u;
  p.qsbuf = off; if (q_fp8) off += 2u * N * 4u;
  p.ksbuf = off; if (k_fp8) off += static_cast<uint32_t>(nK) * kBlockM * 4u;
  p.bars = off;  off += 64u * 8u;
  p.misc = off;  off += 16u;
  p.total = off;
  return p;
}

// Barrier slots inside the bars region.
enum {
  kBarQFull = 0, kBarQEmpty = 2, kBarTFull = 4, kBarTEmpty = 6, kBarFold = 8,  // fold: 4 slots
  kBarDone = 12, kBarKFull = 13, kBarKEmpty = 13 + kMaxKStages, kBarProbe = 13 + 2 * kMaxKStages,
  kBarEnd = kBarProbe + 1
};
static_assert(kBarEnd <= 64, "barrier region");

// Advance a ring position (slot, phase parity) by one: no division on the per-tile path.
__device__ __forceinline__ void ring_next(uint32_t& slot, uint32_t& phase, int n) {
  if (++slot == static_cast<uint32_t>(n)) {
    slot = 0;
    phase ^= 1u;
  }
}

// A wait of a role that has slack.  e4m3 prefill tiles are bound by the epilogue: the
// producers (free ring slots) and the MMA issuer (free accumulators) wait most of the
// time, and spinning there takes issue slots from the epilogue warps sharing their
// schedulers, so those waits suspend in hardware until the phase completes.  Elsewhere
// these roles are on the critical path and poll.
__device__ __forceinline__ bool slack_wait(uint64_t* bar, uint32_t parity, bool suspend, volatile int* abort,
                                           unsigned* status) {
  return suspend ? ptx::mbar_wait_hint(bar, parity, abort, status, kStatusTimeout)
                 : ptx::mbar_wait(bar, parity, abort, status, kStatusTimeout);
}

struct ItemInfo {
  int row0, pos0, kt0, kt1, b, nrows;
};

template <int NQ>
__device__ __forceinline__ bool fetch_item(const ScoreArgs& a, int n_items, int it, ItemInfo& I) {
  const long long G = gridDim.x, c = blockIdx.x;
  long long idx;
  if (a.per_cta > 0) {
    // balanced list: this CTA's own items, in order
    if (it >= min(__ldg(a.cta_counts + c), a.per_cta)) return false;
    idx = c * a.per_cta + it;
  } else {
    // strided walk, alternating direction so CTAs share the tail of the list
    idx = static_cast<long long>(it) * G + ((it & 1) ? (G - 1 - c) : c);
    if (idx >= n_items) return false;
  }
  if (!a.paged) {
    // query blocks in decreasing order of causal work
    const int qb = a.n_dense_items - 1 - static_cast<int>(idx);
    I.row0 = qb * NQ;
    I.nrows = min(NQ, a.T - I.row0);
    I.pos0 = a.q_pos0 + I.row0;
    I.b = 0;
    const int last = min(I.pos0 + I.nrows - 1, a.S - 1);
    I.kt0 = 0;
    I.kt1 = (last + kBlockM) / kBlockM;
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

// SPLIT (decode, bf16 q against e4m3 keys): each query's H heads come as 2H e4m3 rows
// (hi rows, then lo rows), one query per tile: N = max(64, 2H).
template <int H, bool DECODE, bool SPLIT = false>
struct Cfg {
  static constexpr int N = SPLIT ? (2 * H >= 64 ? 2 * H : 64) : (DECODE ? (H >= 64 ? H : 64) : 256);
  static constexpr int NQ = SPLIT ? 1 : N / H;
  static constexpr int QROWS = SPLIT ? 2 * H : H;
  // decode tiles are short (16 or 32 KB) and HBM-bound: a second producer warp (warp 10)
  // takes every other key tile, which needs an even ring
  // a second key producer (warp 10) takes every other key tile when the ring depth is even:
  // decode tiles are short and HBM-bound, and paged e4m3 prefill tiles cost the copy
  // engine two instructions (page boxes, scale rows) per 16 KB, more than one warp's TMA
  // issue keeps up with at the e4m3 MMA rate
  static constexpr int NPROD = 2;
  static constexpr int THREADS = kScoreThreads + 32 * (NPROD - 1);
};

// ------------------------------------------------------------------ producer (warp 0)
template <int H, bool DECODE, bool SPLIT>
__device__ __forceinline__ void producer_role(const ScoreArgs& a, const CUtensorMap* tmap_q,
                                              const CUtensorMap* tmap_k, uint8_t* smem, const SmemPlan& P,
                                              uint64_t* bars, volatile int* abort, int n_items, int pw) {
  if (pw == 1 && !a.two_producers) return;  // one producer: warp 0 takes every tile
  using C = Cfg<H, DECODE, SPLIT>;
  constexpr int N = C::N;
  const int lane = threadIdx.x & 31;
  const int nK = a.num_k_stages;
  const int q_esz = a.q_fp8 ? 1 : 2, k_esz = a.k_fp8 ? 1 : 2;
  const int n_atoms_q = a.D * q_esz / 128, n_atoms_k = a.D * k_esz / 128;
  const int box_q = 128 / q_esz, box_k = 128 / k_esz;
  const uint32_t q_bytes = static_cast<uint32_t>(N) * a.D * q_esz;
  float* wbuf = reinterpret_cast<float*>(smem + P.wbuf);
  float* qsbuf = reinterpret_cast<float*>(smem + P.qsbuf);
  float* ksbuf = reinterpret_cast<float*>(smem + P.ksbuf);
  const int PS = a.page_size;
  const int ppt = a.paged ? kBlockM / PS : 1;
  const uint32_t page_bytes = static_cast<uint32_t>(PS) * a.D * k_esz;

  uint32_t nq = 0, nk = 0;
  uint32_t ks_slot = 0, ks_phase = 0;  // key ring slot of tile nk and its phase parity
  bool ok = true;
  for (int it = 0; ok; ++it) {
    ItemInfo I;
    if (!fetch_item<C::NQ>(a, n_items, it, I)) break;
    // ---- q tile, w and q_scale of this item (first producer)
    if (pw == 0) {
      const int s = nq & 1;
      int good = 1;
      if (lane == 0) good = ptx::mbar_wait(&bars[kBarQEmpty + s], ((nq >> 1) & 1) ^ 1, abort, a.status, kStatusTimeout);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) { ok = false; break; }
      const long long base = static_cast<long long>(I.row0) * H;
      const long long lim = static_cast<long long>(a.total_rows) * H;
      // w (and q_scale) for the item's columns; SPLIT: the query's H weights (w / s)
      for (int c = lane; c < (SPLIT ? H : N) / 4; c += 32) {
        const long long e = base + 4ll * c;
        const bool v = e + 4 <= lim;
        ptx::cp_async_16(wbuf + s * N + 4 * c, v ? static_cast<const void*>(a.w + e) : static_cast<const void*>(a.w),
                         v ? 16u : 0u);
        if (a.q_fp8 && !SPLIT)
          ptx::cp_async_16(qsbuf + s * N + 4 * c,
                           v ? static_cast<const void*>(a.q_scale + e) : static_cast<const void*>(a.q_scale),
                           v ? 16u : 0u);
      }
      ptx::cp_async_mbar_arrive_noinc(&bars[kBarQFull + s]);
      if (lane == 0) ptx::mbar_arrive_expect_tx(&bars[kBarQFull + s], q_bytes);
      __syncwarp();
      // one TMA instruction: lane `at` copies 128-byte atom column `at`
      if (lane < n_atoms_q)
        ptx::tma_load_2d(smem + P.q[s] + lane * N * 128, tmap_q, &bars[kBarQFull + s], lane * box_q,
                         I.row0 * C::QROWS);
      ++nq;
    }
    // ---- key tiles
    const int32_t* bt_row = a.paged ? a.block_tables + static_cast<long long>(I.b) * a.max_pages_per_seq : nullptr;
    int win0 = -(1 << 30);
    int pg_win = -1;
    const int pos_last = I.pos0 + I.nrows - 1;
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      if (a.two_producers && (nk & 1u) != static_cast<uint32_t>(pw)) {
        ++nk;  // the other producer's tile (and stage)
        ring_next(ks_slot, ks_phase, nK);
        continue;
      }
      const int s = static_cast<int>(ks_slot);
      int good = 1;
      if (lane == 0) {
        good = slack_wait(&bars[kBarKEmpty + s], ks_phase ^ 1u, a.q_fp8 && !DECODE, abort, a.status);
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) { ok = false; break; }
      uint64_t* full = &bars[kBarKFull + s];
      uint8_t* dst = smem + P.k[0] + s * (P.k[1] - P.k[0]);
      // Each TMA instruction costs the issuing warp a fixed time however many lanes
      // issue it, so every copy of a tile goes out in one instruction, one lane per copy.
      if (!a.paged) {
        if (a.k_fp8) {
          const long long e = static_cast<long long>(kt) * kBlockM + 4 * lane;
          float* d4 = ksbuf + s * kBlockM + 4 * lane;
          if (e + 4 <= a.S) {
            ptx::cp_async_16(d4, a.k_scale + e, 16u);
          } else {
            for (int j = 0; j < 4; ++j) {
              const bool v = e + j < a.S;
              ptx::cp_async_4(d4 + j, v ? a.k_scale + e + j : a.k_scale, v ? 4u : 0u);
            }
          }
          ptx::cp_async_mbar_arrive_noinc(full);
        }
        if (lane == 0) ptx::mbar_arrive_expect_tx(full, static_cast<uint32_t>(kBlockM) * a.D * k_esz);
        __syncwarp();
        if (lane < n_atoms_k) ptx::tma_load_2d(dst + lane * kBlockM * 128, tmap_k, full, lane * box_k, kt * kBlockM);
      } else {
        const int lp0 = kt * ppt;
        if (lp0 < win0 || lp0 + ppt > win0 + 32) {
          win0 = lp0;
          const int lp = win0 + lane;
          pg_win = lp < a.max_pages_per_seq ? __ldg(bt_row + lp) : -1;
        }
        // lane l copies atom column (l % n_atoms_k) of page (l / n_atoms_k) of this tile
        const int j = n_atoms_k == 2 ? (lane >> 1) : lane;
        const int at = lane - j * n_atoms_k;
        const int pg = __shfl_sync(0xffffffffu, pg_win, (lp0 - win0 + (j < ppt ? j : 0)) & 31);
        const bool needed = j < ppt && static_cast<long long>(lp0 + j) * PS <= pos_last;
        const bool valid = needed && pg >= 0 && pg < a.num_pages;
        if (needed && !valid && at == 0) atomicOr(a.status, kStatusBadPage);
        const unsigned vmask = __ballot_sync(0xffffffffu, valid && at == 0);
        // e4m3 key scales into ksbuf: one bulk copy of the page's scale row per page, on
        // the same barrier as the page's keys
        const bool ks_bulk = a.k_fp8;
        if (lane == 0) {
          const uint32_t per_page = page_bytes + (ks_bulk ? static_cast<uint32_t>(PS) * 4u : 0u);
          ptx::mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(vmask)) * per_page);
        }
        __syncwarp();
        if (valid) {
          ptx::tma_load_3d(dst + at * kBlockM * 128 + j * PS * 128, tmap_k, full, at * box_k, 0, pg);
          if (ks_bulk && at == 0)
            ptx::bulk_load(ksbuf + s * kBlockM + j * PS, a.k_scale + static_cast<long long>(pg) * PS,
                           static_cast<uint32_t>(PS) * 4u, full);
        }
      }
      ++nk;
      ring_next(ks_slot, ks_phase, nK);
    }
  }
  // Drain: wait (bounded) until the copies this warp issued into the rings have
  // landed, so none can write shared memory after the CTA exits.
  if (lane == 0) {
    const int kq = nq < 2 ? static_cast<int>(nq) : 2;
    for (int i = 1; i <= kq; ++i) {
      const uint32_t u = nq - i;
      ptx::mbar_wait_drain(&bars[kBarQFull + (u & 1)], (u >> 1) & 1, a.status, kStatusTimeout, 200000000ull);
    }
    const int kk = nk < static_cast<uint32_t>(nK) ? static_cast<int>(nk) : nK;
    for (int i = 1; i <= kk; ++i) {
      const uint32_t u = nk - i;
      if (a.two_producers && (u & 1u) != static_cast<uint32_t>(pw)) continue;  // the other producer's copy
      ptx::mbar_wait_drain(&bars[kBarKFull + (u % nK)], (u / nK) & 1, a.status, kStatusTimeout, 200000000ull);
    }
  }
}

// ------------------------------------------------------------------ MMA issuer (warp 1, lane 0)
// The single issuing thread is on the tensor core's critical path, so the loop keeps
// everything in registers: stage index and phase advance incrementally, stage
// addresses come from one multiply, and the per-step descriptors are the first
// step's descriptors plus a compile-time offset in their 16-byte address field.
template <int H, bool DECODE, bool SPLIT, bool F8, int NSTEPS>
__device__ __forceinline__ void mma_loop(const ScoreArgs& a, uint8_t* smem, const SmemPlan& P, uint64_t* bars,
                                         volatile int* abort, int n_items, uint32_t tmem_base) {
  using C = Cfg<H, DECODE, SPLIT>;
  constexpr int N = C::N;
  const int nK = a.num_k_stages;
  const uint32_t idesc = ptx::idesc_f32acc(kBlockM, N, !F8);
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t k_stage_bytes = P.k[1] - P.k[0];
  const uint32_t k_base = sbase + P.k[0];
  uint32_t nq = 0, nt = 0;
  uint32_t sk = 0, kphase = 0;  // key ring slot and its phase parity
  // test hook: a wait that nothing ends, bounded by probe_wait_ns, so the kernel records
  // a timeout and every role leaves its loop and drains
  bool ok = a.probe_wait_ns == 0 ||
            ptx::mbar_wait(&bars[kBarProbe], 0, abort, a.status, kStatusTimeout, a.probe_wait_ns);
  for (int it = 0; ok; ++it) {
    ItemInfo I;
    if (!fetch_item<C::NQ>(a, n_items, it, I)) break;
    const int sq = nq & 1;
    if (!ptx::mbar_wait(&bars[kBarQFull + sq], (nq >> 1) & 1, abort, a.status, kStatusTimeout)) break;
    const uint64_t bdesc0 = ptx::sw128_kmajor_desc(sbase + P.q[sq]);
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int acc = nt & 1;
      if (!ptx::mbar_wait(&bars[kBarKFull + sk], kphase, abort, a.status, kStatusTimeout) ||
          !slack_wait(&bars[kBarTEmpty + acc], ((nt >> 1) & 1) ^ 1, F8 && !DECODE, abort, a.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
      const uint64_t adesc0 = ptx::sw128_kmajor_desc(k_base + sk * k_stage_bytes);
#pragma unroll
      for (int j = 0; j < NSTEPS; ++j) {
        // step j reads 32 bytes of K at atom (j / 4), byte (j % 4) * 32 of each row
        const uint64_t ad = adesc0 + static_cast<uint64_t>(((j >> 2) * (kBlockM * 128) + (j & 3) * 32) >> 4);
        const uint64_t bd = bdesc0 + static_cast<uint64_t>(((j >> 2) * (N * 128) + (j & 3) * 32) >> 4);
        if (F8) ptx::mma_f8(d_tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
        else ptx::mma_bf16(d_tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
      }
      ptx::mma_commit(&bars[kBarKEmpty + sk]);
      ptx::mma_commit(&bars[kBarTFull + acc]);
      if (++sk == static_cast<uint32_t>(nK)) { sk = 0; kphase ^= 1u; }
      ++nt;
    }
    if (!ok) break;
    ptx::mma_commit(&bars[kBarQEmpty + sq]);
    ++nq;
  }
  // every MMA issued above has finished once this commit arrives
  ptx::mma_commit(&bars[kBarDone]);
  ptx::mbar_wait_drain(&bars[kBarDone], 0, a.status, kStatusTimeout, 200000000ull);
}

template <int H, bool DECODE, bool SPLIT>
__device__ __forceinline__ void mma_role(const ScoreArgs& a, uint8_t* smem, const SmemPlan& P, uint64_t* bars,
                                         volatile int* abort, int n_items, uint32_t tmem_base) {
  // 32 bytes of K per MMA: 16 bf16 or 32 e4m3 values (SPLIT: e4m3 queries, N = 2H)
  if (SPLIT || a.q_fp8) mma_loop<H, DECODE, SPLIT, true, 4>(a, smem, P, bars, abort, n_items, tmem_base);
  else if (a.D == 128) mma_loop<H, DECODE, SPLIT, false, 8>(a, smem, P, bars, abort, n_items, tmem_base);
  else mma_loop<H, DECODE, SPLIT, false, 4>(a, smem, P, bars, abort, n_items, tmem_base);
}

// Every lane waits (each observes the barrier itself); the outcome is made uniform
// across the warp so that .sync.aligned TMEM loads never run on a partial warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* status) {
  const bool ok = ptx::mbar_wait(bar, parity, abort, status, kStatusTimeout);
  return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------------------ epilogue (warps 2..9)
// ALT: whole tiles alternate between the two epilogue warpgroups (each thread reduces all
// N columns of its key); otherwise both warpgroups take every tile, split by columns.
// Decode tiles and e4m3 prefill tiles alternate: a tile's fixed per-warp work (waits,
// arrives, stores) is then spread over twice the columns.
template <int H, bool DECODE, bool SPLIT, bool ALT>
__device__ __forceinline__ void epilogue_role(const ScoreArgs& a, uint8_t* smem, const SmemPlan& P,
                                              uint64_t* bars, volatile int* abort, int n_items,
                                              uint32_t tmem_base) {
  using C = Cfg<H, DECODE, SPLIT>;
  constexpr int N = C::N;
  constexpr int NCOLS = ALT ? N : N / 2;     // columns one epilogue thread reduces
  constexpr int QH = SPLIT ? 1 : NCOLS / H;  // queries in those columns
  constexpr int NCH = NCOLS / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = (warp - 2) >> 2;
  const int quarter = warp & 3;            // TMEM lane quarter this warp may access
  const int m = quarter * 32 + lane;       // key row of the tile
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int col0 = ALT ? 0 : half * NCOLS;
  const int q0 = col0 / H;
  const int nK = a.num_k_stages;
  float* wbuf = reinterpret_cast<float*>(smem + P.wbuf);
  const float* qsbuf = reinterpret_cast<const float*>(smem + P.qsbuf);
  const float* ksbuf = reinterpret_cast<const float*>(smem + P.ksbuf);
  const int fold_t = ALT ? static_cast<int>(threadIdx.x) - 64 : static_cast<int>(threadIdx.x) - 64 - half * 128;

  uint32_t nq = 0, nk = 0, nt = 0;
  uint32_t ks_slot = 0, ks_phase = 0;  // key ring slot of tile nk and its phase parity
  bool ok = true;
  for (int it = 0; ok; ++it) {
    ItemInfo I;
    if (!fetch_item<C::NQ>(a, n_items, it, I)) break;
    const int sq = nq & 1;
    if (!warp_wait(&bars[kBarQFull + sq], (nq >> 1) & 1, abort, a.status)) break;
    float* wq = wbuf + sq * N;
    if (a.q_fp8 && !SPLIT) {
      // fold the q scale into w once per item (in place, each thread one column)
      const int c = ALT ? fold_t : col0 + fold_t;
      if (!ALT || fold_t < N) wq[c] *= qsbuf[sq * N + c];
      uint64_t* fb = &bars[kBarFold + sq * 2 + (ALT ? 0 : half)];
      ptx::mbar_arrive(fb);
      if (!warp_wait(fb, (nq >> 1) & 1, abort, a.status)) break;
    }
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int sk = static_cast<int>(ks_slot);
      const int acc = nt & 1;
      const bool mine = ALT ? (acc == half) : true;
      if (mine) {
        // e4m3 keys: take this key's scale and release the stage's scale slot before the
        // accumulator wait, so the ring turns over as soon as the MMA is done with it
        float ks = 1.f;
        if (a.k_fp8) {
          if (!warp_wait(&bars[kBarKFull + sk], ks_phase, abort, a.status)) {
            ok = false;
            break;
          }
          ks = ksbuf[sk * kBlockM + m];
          __syncwarp();
          ptx::mbar_arrive_elect(&bars[kBarKEmpty + sk]);
        }
        if (!warp_wait(&bars[kBarTFull + acc], (nt >> 1) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tcol = tmem_base + lane_addr + static_cast<uint32_t>(acc * 256 + col0);
        float accq[QH];
        if constexpr (SPLIT) {
          // head h: the hi part at column h, the lo part at column H + h; their sum is the
          // exact bf16 product up to fp32 rounding, and the ReLU takes the sum
          float2 part[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) part[p] = make_float2(0.f, 0.f);
          uint32_t xa[32], xb[32];
          if constexpr (H >= 32) {
#pragma unroll
            for (int j = 0; j < H / 32; ++j) {
              ptx::tmem_ld_32x32b_x32(tcol + 32 * j, xa);
              ptx::tmem_ld_32x32b_x32(tcol + H + 32 * j, xb);
              ptx::tmem_ld_wait_regs(xa);  // waits for both loads; the second ties xb's registers
              ptx::tmem_ld_wait_regs(xb);
              const float2* w2 = reinterpret_cast<const float2*>(wq + 32 * j);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float r0 = fmaxf(__uint_as_float(xa[2 * i]) + __uint_as_float(xb[2 * i]), 0.f);
                const float r1 = fmaxf(__uint_as_float(xa[2 * i + 1]) + __uint_as_float(xb[2 * i + 1]), 0.f);
                ptx::ffma2(part[i & 3], w2[i], make_float2(r0, r1));
              }
            }
          } else {
            ptx::tmem_ld_32x32b_x32(tcol, xa);
            ptx::tmem_ld_wait_regs(xa);
            const float2* w2 = reinterpret_cast<const float2*>(wq);
#pragma unroll
            for (int i = 0; i < H / 2; ++i) {
              const float r0 = fmaxf(__uint_as_float(xa[2 * i]) + __uint_as_float(xa[H + 2 * i]), 0.f);
              const float r1 = fmaxf(__uint_as_float(xa[2 * i + 1]) + __uint_as_float(xa[H + 2 * i + 1]), 0.f);
              ptx::ffma2(part[i & 3], w2[i], make_float2(r0, r1));
            }
          }
          accq[0] = (part[0].x + part[0].y) + (part[1].x + part[1].y) + (part[2].x + part[2].y) +
                    (part[3].x + part[3].y);
        } else {
        // NP packed (f32x2) partial sums per query: independent FMA chains
        constexpr int NP = (32 / (2 * QH)) > 4 ? 4 : ((32 / (2 * QH)) < 1 ? 1 : (32 / (2 * QH)));
        float2 part[QH][NP];
#pragma unroll
        for (int j = 0; j < QH; ++j)
#pragma unroll
          for (int p = 0; p < NP; ++p) part[j][p] = make_float2(0.f, 0.f);
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
            const int cc = 32 * c + 4 * i4;  // column (within this thread's range) of wv.x
            const int jq = cc / H;          // H >= 4, so the 4 columns share a query
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
#pragma unroll
        for (int j = 0; j < QH; ++j) {
          float t = 0.f;
#pragma unroll
          for (int p = 0; p < NP; ++p) t += part[j][p].x + part[j][p].y;
          accq[j] = t;
        }
        }
        ptx::tc_fence_before();
        __syncwarp();
        ptx::mbar_arrive_elect(&bars[kBarTEmpty + acc]);
        const int s = kt * kBlockM + m;
        const bool key_ok = a.paged || s < a.S;
#pragma unroll
        for (int j = 0; j < QH; ++j) {
          const int qi = q0 + j;
          float* dst = a.scores + static_cast<long long>(I.row0 + qi - a.row_base) * a.ld + s;
          ptx::st_global_if(dst, accq[j] * ks, qi < I.nrows && key_ok && s <= I.pos0 + qi);
        }
      }
      ++nk;
      ring_next(ks_slot, ks_phase, nK);
      ++nt;
    }
    if (!ok) break;
    __syncwarp();
    ptx::mbar_arrive_elect(&bars[kBarQEmpty + sq]);
    ++nq;
  }
}

template <int H, bool DECODE, bool SPLIT>
__global__ void __launch_bounds__(Cfg<H, DECODE, SPLIT>::THREADS, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const ScoreArgs a) {
  using C = Cfg<H, DECODE, SPLIT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusSmemAlign);
    return;
  }
  const SmemPlan P = plan_smem(C::N, a.D, SPLIT ? 1 : a.q_fp8, a.k_fp8, a.num_k_stages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + P.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + P.misc + 4);
  const bool alt = DECODE || a.q_fp8;  // whole tiles alternate between the epilogue warpgroups

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars[kBarQFull + s], 1 + 32);
      ptx::mbar_init(&bars[kBarQEmpty + s], 1 + 8);
      ptx::mbar_init(&bars[kBarTFull + s], 1);
      ptx::mbar_init(&bars[kBarTEmpty + s], alt ? 4 : 8);  // the warps that read the accumulator
      ptx::mbar_init(&bars[kBarFold + 2 * s + 0], alt ? 256 : 128);
      ptx::mbar_init(&bars[kBarFold + 2 * s + 1], 128);
    }
    ptx::mbar_init(&bars[kBarDone], 1);
    ptx::mbar_init(&bars[kBarProbe], 1);
    for (int s = 0; s < a.num_k_stages; ++s) {
      // e4m3 key scales of dense tiles come by cp.async (32 lane arrivals), those of
      // paged tiles by one bulk copy per page
      ptx::mbar_init(&bars[kBarKFull + s], 1 + ((a.k_fp8 && !a.paged) ? 32 : 0));
      // the epilogue also releases a stage when it reads that stage's key scales from ksbuf
      ptx::mbar_init(&bars[kBarKEmpty + s], 1 + (a.k_fp8 ? (alt ? 4 : 8) : 0));
    }
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_q);
    ptx::prefetch_tmap(&tmap_k);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // the prologue above overlaps the previous kernel's tail; its outputs (work lists,
  // split queries, the scores buffer it read) are safe to use from here on
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const int n_items = a.paged ? min(*a.n_items, a.items_cap) : a.n_dense_items;

  if ((tmem_base & 0xFFFFu) != 0) {
    // the two accumulators assume the allocation starts at column 0
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTmemAlloc);
  } else if (warp == 0) {
    producer_role<H, DECODE, SPLIT>(a, &tmap_q, &tmap_k, smem, P, bars, abort, n_items, 0);
  } else if (C::NPROD == 2 && warp == 10) {
    producer_role<H, DECODE, SPLIT>(a, &tmap_q, &tmap_k, smem, P, bars, abort, n_items, 1);
  } else if (warp == 1) {
    if (lane == 0) mma_role<H, DECODE, SPLIT>(a, smem, P, bars, abort, n_items, tmem_base);
    __syncwarp();
  } else {
    if constexpr (DECODE) epilogue_role<H, DECODE, SPLIT, true>(a, smem, P, bars, abort, n_items, tmem_base);
    else if (alt) epilogue_role<H, DECODE, SPLIT, true>(a, smem, P, bars, abort, n_items, tmem_base);
    else epilogue_role<H, DECODE, SPLIT, false>(a, smem, P, bars, abort, n_items, tmem_base);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int H, bool DECODE, bool SPLIT>
cudaError_t launch_t(const ScoreArgs& a, const CUtensorMap* tq, const CUtensorMap* tk, int grid, size_t smem,
                     cudaStream_t st) {
  auto kern = score_kernel<H, DECODE, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (a.two_producers && (a.num_k_stages & 1)) return cudaErrorInvalidValue;
  e = launch_pdl(kern, dim3(grid), dim3(Cfg<H, DECODE, SPLIT>::THREADS), smem, st, *tq, *tk, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

size_t score_smem_bytes(const ScoreArgs& a, int num_k_stages) {
  return plan_smem(a.N, a.D, a.split ? 1 : a.q_fp8, a.k_fp8, num_k_stages).total;
}

cudaError_t launch_score(const ScoreArgs& args, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k, int grid,
                         size_t smem_bytes, cudaStream_t st) {
  ScoreArgs a = args;
  a.probe_wait_ns = armed_probe_wait_ns();
  armed_probe_wait_ns() = 0;
  // decode tiles always use both producers (their ring depth is even); prefill tiles when
  // the ring depth is even (e4m3 tiles: ~10 stages; bf16 tiles fit 3 and keep one)
  a.two_producers = (a.num_k_stages % 2 == 0) ? 1 : 0;
  const bool dec = a.split || a.N != 256;
#define DSA_CASE(HH)                                                                        \
  case HH:                                                                                  \
    return dec ? (a.split ? launch_t<HH, true, true>(a, tmap_q, tmap_k, grid, smem_bytes, st)          \
                          : launch_t<HH, true, false>(a, tmap_q, tmap_k, grid, smem_bytes, st))        \
               : launch_t<HH, false, false>(a, tmap_q, tmap_k, grid, smem_bytes, st);
  switch (a.H) {
    DSA_CASE(4)
    DSA_CASE(8)
    DSA_CASE(16)
    DSA_CASE(32)
    DSA_CASE(64)
    DSA_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef DSA_CASE
}

}  // namespace dsa
