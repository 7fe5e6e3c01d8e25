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
// Warp roles (320 threads, 448 with the key converters; one CTA per SM, persistent
// over work items):
//   warp 0      TMA producer: q tile (N x D) per item into a 2-deep ring, key tiles
//               (128 x D, dense or gathered page by page through block_tables) into
//               an nK-deep ring, per-item w / q_scale by cp.async, per-tile k_scale by
//               cp.async (dense keys) or a bulk copy per page (paged prefill); decode
//               epilogue threads read their paged key scales from global memory.
//   warp 1      TMEM allocator; lane 0 issues tcgen05.mma into two 256-column fp32
//               accumulators (double buffered) and commits to mbarriers.
//   warps 2..9  epilogue: tcgen05.ld, ReLU, head-weighted sum, k scale, causal mask,
//               coalesced fp32 stores.  Prefill tiles (N = 256) are split by columns
//               between two warpgroups; decode tiles (N = max(64, H)) alternate
//               between the warpgroups tile by tile.
//   warps 10-13 only for bf16 queries against e4m3 keys (decode): widen each staged
//               e4m3 key tile to bf16 into TMEM, the MMA's A operand there.
// Every wait is bounded; on a timeout the kernel records kStatusTimeout, all roles
// leave their loops, in-flight copies and MMAs are drained (bounded) and TMEM freed.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {

namespace {

struct SmemPlan {
  uint32_t q[2];
  uint32_t k[kMaxKStages];
  uint32_t k8[kMaxK8Stages];  // e4m3 staging of the keys (mixed mode)
  uint32_t wbuf, qsbuf, ksbuf, bars, misc, total;
};

__host__ __device__ inline SmemPlan plan_smem(int N, int D, int q_fp8, int k_fp8, int nK, int mixed = 0) {
  SmemPlan p{};
  uint32_t off = 0;
  const uint32_t qb = static_cast<uint32_t>(N) * D * (q_fp8 ? 1 : 2);
  // mixed: the widened keys live in TMEM, only the e4m3 staging ring is in shared memory
  const uint32_t kb = mixed ? 0u : static_cast<uint32_t>(kBlockM) * D * (k_fp8 ? 1 : 2);
  for (int i = 0; i < 2; ++i) { p.q[i] = off; off += qb; }
  for (int i = 0; i < kMaxKStages; ++i) { p.k[i] = off; if (i < nK) off += kb; }
  for (int i = 0; i < kMaxK8Stages; ++i) { p.k8[i] = off; if (mixed && i < nK) off += static_cast<uint32_t>(kBlockM) * D; }
  p.wbuf = off;  off += 2u * N * 4u;
  p.qsbuf = off; if (q_fp8) off += 2u * N * 4u;
  p.ksbuf = off; if (k_fp8 && !mixed) off += static_cast<uint32_t>(nK) * kBlockM * 4u;  // mixed decode reads scales from global
  p.bars = off;  off += 64u * 8u;
  p.misc = off;  off += 16u;
  p.total = off;
  return p;
}

// Mixed mode: TMEM column of key stage s widened to bf16 (128 lanes x 64 columns).  The
// accumulators take columns [0, N) and [256, 256 + N); the stages fill the rest.
__device__ __forceinline__ uint32_t mixed_a_col(int s, int N) {
  const int per = (256 - N) / 64;
  return static_cast<uint32_t>(s < per ? N + 64 * s : 256 + N + 64 * (s - per));
}

// Barrier slots inside the bars region.
enum {
  kBarQFull = 0, kBarQEmpty = 2, kBarTFull = 4, kBarTEmpty = 6, kBarFold = 8,  // fold: 4 slots
  // key ring; in mixed mode the ring of widened tiles in TMEM (full: converted, empty: MMAs done)
  kBarDone = 12, kBarKFull = 13, kBarKEmpty = 13 + kMaxKStages,
  kBarK8Full = 13 + 2 * kMaxKStages,                  // mixed: e4m3 key tile landed in shared memory
  kBarK8Empty = 13 + 2 * kMaxKStages + kMaxK8Stages   // mixed: e4m3 staging slot converted
};
static_assert(kBarK8Empty + kMaxK8Stages <= 64, "barrier region");

struct ItemInfo {
  int row0, pos0, kt0, kt1, b, nrows;
};

template <int NQ>
__device__ __forceinline__ bool fetch_item(const ScoreArgs& a, int n_items, int it, ItemInfo& I) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long idx = static_cast<long long>(it) * G + ((it & 1) ? (G - 1 - c) : c);
  if (idx >= n_items) return false;
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

template <int H, bool DECODE>
struct Cfg {
  static constexpr int N = DECODE ? (H >= 64 ? H : 64) : 256;
  static constexpr int NQ = N / H;
  static constexpr int NCOLS = DECODE ? N : N / 2;  // columns one epilogue thread reduces
  static constexpr int QH = NCOLS / H;               // queries in those columns
  static constexpr int EPI_T_ARRIVALS = DECODE ? 4 : 8;
};

// ------------------------------------------------------------------ producer (warp 0)
template <int H, bool DECODE>
__device__ __forceinline__ void producer_role(const ScoreArgs& a, const CUtensorMap* tmap_q,
                                              const CUtensorMap* tmap_k, uint8_t* smem, const SmemPlan& P,
                                              uint64_t* bars, volatile int* abort, int n_items) {
  using C = Cfg<H, DECODE>;
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
  bool ok = true;
  for (int it = 0; ok; ++it) {
    ItemInfo I;
    if (!fetch_item<C::NQ>(a, n_items, it, I)) break;
    // ---- q tile, w and q_scale of this item
    {
      const int s = nq & 1;
      int good = 1;
      if (lane == 0) good = ptx::mbar_wait(&bars[kBarQEmpty + s], ((nq >> 1) & 1) ^ 1, abort, a.status, kStatusTimeout);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) { ok = false; break; }
      const long long base = static_cast<long long>(I.row0) * H;
      const long long lim = static_cast<long long>(a.total_rows) * H;
      for (int c = lane; c < N / 4; c += 32) {
        const long long e = base + 4ll * c;
        const bool v = e + 4 <= lim;
        ptx::cp_async_16(wbuf + s * N + 4 * c, v ? static_cast<const void*>(a.w + e) : static_cast<const void*>(a.w),
                         v ? 16u : 0u);
        if (a.q_fp8)
          ptx::cp_async_16(qsbuf + s * N + 4 * c,
                           v ? static_cast<const void*>(a.q_scale + e) : static_cast<const void*>(a.q_scale),
                           v ? 16u : 0u);
      }
      ptx::cp_async_mbar_arrive_noinc(&bars[kBarQFull + s]);
      if (lane == 0) ptx::mbar_arrive_expect_tx(&bars[kBarQFull + s], q_bytes);
      __syncwarp();
      // one TMA instruction: lane `at` copies 128-byte atom column `at`
      if (lane < n_atoms_q)
        ptx::tma_load_2d(smem + P.q[s] + lane * N * 128, tmap_q, &bars[kBarQFull + s], lane * box_q, I.row0 * H);
      ++nq;
    }
    // ---- key tiles
    const int32_t* bt_row = a.paged ? a.block_tables + static_cast<long long>(I.b) * a.max_pages_per_seq : nullptr;
    int win0 = -(1 << 30);
    int pg_win = -1;
    const int pos_last = I.pos0 + I.nrows - 1;
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int s = nk % nK;
      int good = 1;
      if (lane == 0) {
        // mixed: the staging slot is free once the converters have read it
        good = ptx::mbar_wait(&bars[(a.mixed ? kBarK8Empty : kBarKEmpty) + s], ((nk / nK) & 1) ^ 1, abort, a.status,
                              kStatusTimeout);
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) { ok = false; break; }
      // mixed: the e4m3 tile and its scales land in the staging slot; converters fill P.k
      uint64_t* full = a.mixed ? &bars[kBarK8Full + s] : &bars[kBarKFull + s];
      uint8_t* dst = smem + (a.mixed ? P.k8[0] + s * (P.k8[1] - P.k8[0]) : P.k[0] + s * (P.k[1] - P.k[0]));
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
        // e4m3 key scales: decode epilogue threads read their own from global memory;
        // prefill tiles take them by one bulk copy per page into ksbuf
        const bool ks_bulk = a.k_fp8 && !DECODE;
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
      ptx::mbar_wait_drain(&bars[(a.mixed ? kBarK8Full : kBarKFull) + (u % nK)], (u / nK) & 1, a.status, kStatusTimeout,
                           200000000ull);
    }
  }
}

// ------------------------------------------------------------------ MMA issuer (warp 1, lane 0)
// The single issuing thread is on the tensor core's critical path, so the loop keeps
// everything in registers: stage index and phase advance incrementally, stage
// addresses come from one multiply, and the per-step descriptors are the first
// step's descriptors plus a compile-time offset in their 16-byte address field.
template <int H, bool DECODE, bool F8, int NSTEPS, bool ATMEM = false>
__device__ __forceinline__ void mma_loop(const ScoreArgs& a, uint8_t* smem, const SmemPlan& P, uint64_t* bars,
                                         volatile int* abort, int n_items, uint32_t tmem_base) {
  using C = Cfg<H, DECODE>;
  constexpr int N = C::N;
  const int nK = ATMEM ? a.num_a_stages : a.num_k_stages;
  const uint32_t idesc = ptx::idesc_f32acc(kBlockM, N, !F8);
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t k_stage_bytes = P.k[1] - P.k[0];
  const uint32_t k_base = sbase + P.k[0];
  uint32_t nq = 0, nt = 0;
  uint32_t sk = 0, kphase = 0;  // key ring slot and its phase parity
  bool ok = true;
  for (int it = 0; ok; ++it) {
    ItemInfo I;
    if (!fetch_item<C::NQ>(a, n_items, it, I)) break;
    const int sq = nq & 1;
    if (!ptx::mbar_wait(&bars[kBarQFull + sq], (nq >> 1) & 1, abort, a.status, kStatusTimeout)) break;
    const uint64_t bdesc0 = ptx::sw128_kmajor_desc(sbase + P.q[sq]);
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int acc = nt & 1;
      if (!ptx::mbar_wait(&bars[kBarKFull + sk], kphase, abort, a.status, kStatusTimeout) ||
          !ptx::mbar_wait(&bars[kBarTEmpty + acc], ((nt >> 1) & 1) ^ 1, abort, a.status, kStatusTimeout)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
      if constexpr (ATMEM) {
        // keys widened into TMEM: step j takes columns [8j, 8j + 8) (16 bf16 of K)
        const uint32_t a_tmem = tmem_base + mixed_a_col(static_cast<int>(sk), N);
#pragma unroll
        for (int j = 0; j < NSTEPS; ++j) {
          const uint64_t bd = bdesc0 + static_cast<uint64_t>(((j >> 2) * (N * 128) + (j & 3) * 32) >> 4);
          ptx::mma_bf16_ts(d_tmem, a_tmem + 8 * j, bd, idesc, j > 0 ? 1u : 0u);
        }
      } else {
        const uint64_t adesc0 = ptx::sw128_kmajor_desc(k_base + sk * k_stage_bytes);
#pragma unroll
        for (int j = 0; j < NSTEPS; ++j) {
          // step j reads 32 bytes of K at atom (j / 4), byte (j % 4) * 32 of each row
          const uint64_t ad = adesc0 + static_cast<uint64_t>(((j >> 2) * (kBlockM * 128) + (j & 3) * 32) >> 4);
          const uint64_t bd = bdesc0 + static_cast<uint64_t>(((j >> 2) * (N * 128) + (j & 3) * 32) >> 4);
          if (F8) ptx::mma_f8(d_tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
          else ptx::mma_bf16(d_tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
        }
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

template <int H, bool DECODE>
__device__ __forceinline__ void mma_role(const ScoreArgs& a, uint8_t* smem, const SmemPlan& P, uint64_t* bars,
                                         volatile int* abort, int n_items, uint32_t tmem_base) {
  // 32 bytes of K per MMA: 16 bf16 or 32 e4m3 values; mixed mode multiplies bf16 by widened keys
  if (a.q_fp8) mma_loop<H, DECODE, true, 4>(a, smem, P, bars, abort, n_items, tmem_base);
  else if (DECODE && a.mixed) mma_loop<H, DECODE, false, 8, DECODE>(a, smem, P, bars, abort, n_items, tmem_base);
  else if (a.D == 128) mma_loop<H, DECODE, false, 8>(a, smem, P, bars, abort, n_items, tmem_base);
  else mma_loop<H, DECODE, false, 4>(a, smem, P, bars, abort, n_items, tmem_base);
}

// Every lane waits (each observes the barrier itself); the outcome is made uniform
// across the warp so that .sync.aligned TMEM loads never run on a partial warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned* status) {
  const bool ok = ptx::mbar_wait(bar, parity, abort, status, kStatusTimeout);
  return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------------------ key widening (mixed mode, warps 10..13)
// Two e4m3 codes -> two bf16, exactly (every e4m3 value, subnormals included, is a
// bf16 value).  `t` holds the codes in bits 15..8 and 31..24.  Moving the code's
// exponent and mantissa bits under bf16's exponent/mantissa boundary gives a bf16
// whose exponent is biased by 127 instead of 7 (an e4m3 subnormal lands on a bf16
// subnormal with the same mantissa); one multiply by 2^120 removes the bias gap.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t t) {
  const uint32_t v = (t & 0x80008000u) | ((t >> 4) & 0x07F007F0u);
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x7B807B80u));  // 0x7B80 = 2^120
  return r;
}

// Widen every staged e4m3 key tile (128 rows x D=128 bytes, 128-byte swizzle) to bf16
// straight into TMEM, where the MMA reads it as its A operand.  Warp w owns TMEM lanes
// [32 (w % 4), 32 (w % 4) + 32): lane l converts key row 32 (w % 4) + l, 64 columns.
template <int H, bool DECODE>
__device__ __forceinline__ void convert_role(const ScoreArgs& a, uint8_t* smem, const SmemPlan& P, uint64_t* bars,
                                             volatile int* abort, int n_items, uint32_t tmem_base) {
  using C = Cfg<H, DECODE>;
  const int quarter = (threadIdx.x >> 5) & 3;
  const int lane = threadIdx.x & 31;
  const int r = quarter * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int nK = a.num_k_stages;   // e4m3 staging ring (shared memory)
  const int nA = a.num_a_stages;   // widened tiles (TMEM)
  const uint32_t k8_stage = P.k8[1] - P.k8[0];
  uint32_t sk = 0, kph = 0, sa = 0, aph = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    ItemInfo I;
    if (!fetch_item<C::NQ>(a, n_items, it, I)) break;
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      // the staged tile has landed, and the MMAs that read this TMEM slot last are done
      if (!warp_wait(&bars[kBarK8Full + sk], kph, abort, a.status) ||
          !warp_wait(&bars[kBarKEmpty + sa], aph ^ 1u, abort, a.status)) {
        ok = false;
        break;
      }
      const uint8_t* row = smem + P.k8[0] + sk * k8_stage + r * 128;
      const uint32_t acol = tmem_base + lane_addr + mixed_a_col(static_cast<int>(sa), C::N);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o[32];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          // logical 16-byte chunk c = e4m3 elements [16c, 16c + 16) -> columns [8c, 8c + 8)
          const int c = 4 * hh + c4;
          const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
          o[8 * c4 + 0] = e4m3x2_to_bf16x2(__byte_perm(v.x, 0, 0x1404));
          o[8 * c4 + 1] = e4m3x2_to_bf16x2(__byte_perm(v.x, 0, 0x3424));
          o[8 * c4 + 2] = e4m3x2_to_bf16x2(__byte_perm(v.y, 0, 0x1404));
          o[8 * c4 + 3] = e4m3x2_to_bf16x2(__byte_perm(v.y, 0, 0x3424));
          o[8 * c4 + 4] = e4m3x2_to_bf16x2(__byte_perm(v.z, 0, 0x1404));
          o[8 * c4 + 5] = e4m3x2_to_bf16x2(__byte_perm(v.z, 0, 0x3424));
          o[8 * c4 + 6] = e4m3x2_to_bf16x2(__byte_perm(v.w, 0, 0x1404));
          o[8 * c4 + 7] = e4m3x2_to_bf16x2(__byte_perm(v.w, 0, 0x3424));
        }
        ptx::tmem_st_32x32b_x32(acol + 32 * hh, o);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(&bars[kBarKFull + sa]);
        ptx::mbar_arrive(&bars[kBarK8Empty + sk]);
      }
      if (++sk == static_cast<uint32_t>(nK)) { sk = 0; kph ^= 1u; }
      if (++sa == static_cast<uint32_t>(nA)) { sa = 0; aph ^= 1u; }
    }
  }
}

// ------------------------------------------------------------------ epilogue (warps 2..9)
template <int H, bool DECODE>
__device__ __forceinline__ void epilogue_role(const ScoreArgs& a, uint8_t* smem, const SmemPlan& P,
                                              uint64_t* bars, volatile int* abort, int n_items,
                                              uint32_t tmem_base) {
  using C = Cfg<H, DECODE>;
  constexpr int N = C::N;
  constexpr int NCOLS = C::NCOLS;
  constexpr int QH = C::QH;
  constexpr int NCH = NCOLS / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = (warp - 2) >> 2;
  const int quarter = warp & 3;            // TMEM lane quarter this warp may access
  const int m = quarter * 32 + lane;       // key row of the tile
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int col0 = DECODE ? 0 : half * NCOLS;
  const int q0 = col0 / H;
  const int nK = a.num_k_stages;
  float* wbuf = reinterpret_cast<float*>(smem + P.wbuf);
  const float* qsbuf = reinterpret_cast<const float*>(smem + P.qsbuf);
  const float* ksbuf = reinterpret_cast<const float*>(smem + P.ksbuf);
  const int fold_t = DECODE ? static_cast<int>(threadIdx.x) - 64 : static_cast<int>(threadIdx.x) - 64 - half * 128;

  uint32_t nq = 0, nk = 0, nt = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    ItemInfo I;
    if (!fetch_item<C::NQ>(a, n_items, it, I)) break;
    const int sq = nq & 1;
    if (!warp_wait(&bars[kBarQFull + sq], (nq >> 1) & 1, abort, a.status)) break;
    float* wq = wbuf + sq * N;
    if (a.q_fp8) {
      // fold the q scale into w once per item (in place, each thread one column)
      const int c = DECODE ? fold_t : col0 + fold_t;
      if (!DECODE || fold_t < N) wq[c] *= qsbuf[sq * N + c];
      uint64_t* fb = &bars[kBarFold + sq * 2 + (DECODE ? 0 : half)];
      ptx::mbar_arrive(fb);
      if (!warp_wait(fb, (nq >> 1) & 1, abort, a.status)) break;
    }
    for (int kt = I.kt0; kt < I.kt1; ++kt) {
      const int sk = nk % nK;
      const int acc = nt & 1;
      const bool mine = DECODE ? (acc == half) : true;
      if (mine) {
        // paged e4m3 keys: this thread's key scale straight from global memory (page
        // table, then the page's scale row), issued before the accumulator wait so the
        // two dependent loads overlap it; dense e4m3 keys: the staged copy in ksbuf
        float ks_g = 1.f;
        const bool ks_smem = a.k_fp8 && !(DECODE && a.paged);
        if (a.k_fp8 && !ks_smem) {
          const long long key = static_cast<long long>(kt) * kBlockM + m;
          const int lp = static_cast<int>(key / a.page_size);
          const int pg = (lp < a.max_pages_per_seq && key <= I.pos0 + I.nrows - 1)
                             ? __ldg(a.block_tables + static_cast<long long>(I.b) * a.max_pages_per_seq + lp)
                             : -1;
          ks_g = (pg >= 0 && pg < a.num_pages)
                     ? __ldg(a.k_scale + static_cast<long long>(pg) * a.page_size + (key - static_cast<long long>(lp) * a.page_size))
                     : 0.f;
        }
        if (ks_smem && !warp_wait(&bars[kBarKFull + sk], (nk / nK) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        if (!warp_wait(&bars[kBarTFull + acc], (nt >> 1) & 1, abort, a.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // NP packed (f32x2) partial sums per query: independent FMA chains
        constexpr int NP = (32 / (2 * QH)) > 4 ? 4 : ((32 / (2 * QH)) < 1 ? 1 : (32 / (2 * QH)));
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
        float accq[QH];
#pragma unroll
        for (int j = 0; j < QH; ++j) {
          float t = 0.f;
#pragma unroll
          for (int p = 0; p < NP; ++p) t += part[j][p].x + part[j][p].y;
          accq[j] = t;
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars[kBarTEmpty + acc]);
        float ks = ks_g;
        if (ks_smem) {
          ks = ksbuf[sk * kBlockM + m];
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bars[kBarKEmpty + sk]);
        }
        const int s = kt * kBlockM + m;
        const bool key_ok = a.paged || s < a.S;
#pragma unroll
        for (int j = 0; j < QH; ++j) {
          const int qi = q0 + j;
          if (qi < I.nrows && key_ok && s <= I.pos0 + qi) {
            float* dst = a.scores + static_cast<long long>(I.row0 + qi - a.row_base) * a.ld + s;
            *dst = accq[j] * ks;
          }
        }
      }
      ++nk;
      ++nt;
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&bars[kBarQEmpty + sq]);
    ++nq;
  }
}

template <int H, bool DECODE, bool MIXED>
__global__ void __launch_bounds__(MIXED ? kMixedThreads : kScoreThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const ScoreArgs a) {
  using C = Cfg<H, DECODE>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusSmemAlign);
    return;
  }
  const SmemPlan P = plan_smem(C::N, a.D, a.q_fp8, a.k_fp8, a.num_k_stages, MIXED ? 1 : 0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + P.misc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + P.misc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars[kBarQFull + s], 1 + 32);
      ptx::mbar_init(&bars[kBarQEmpty + s], 1 + 8);
      ptx::mbar_init(&bars[kBarTFull + s], 1);
      ptx::mbar_init(&bars[kBarTEmpty + s], C::EPI_T_ARRIVALS);
      ptx::mbar_init(&bars[kBarFold + 2 * s + 0], DECODE ? 256 : 128);
      ptx::mbar_init(&bars[kBarFold + 2 * s + 1], 128);
    }
    ptx::mbar_init(&bars[kBarDone], 1);
    const int n_ring = MIXED ? a.num_a_stages : a.num_k_stages;
    for (int s = 0; s < n_ring; ++s) {
      // dense e4m3 key scales come by cp.async (32 lane arrivals); paged ones by bulk copy;
      // mixed: the four converter warps fill a TMEM slot
      ptx::mbar_init(&bars[kBarKFull + s], MIXED ? 4 : 1 + ((a.k_fp8 && !a.paged) ? 32 : 0));
      // the epilogue also releases a stage when it reads that stage's key scales from ksbuf
      ptx::mbar_init(&bars[kBarKEmpty + s], 1 + ((a.k_fp8 && !(DECODE && a.paged)) ? C::EPI_T_ARRIVALS : 0));
    }
    if (MIXED) {
      for (int s = 0; s < a.num_k_stages; ++s) {
        ptx::mbar_init(&bars[kBarK8Full + s], 1);
        ptx::mbar_init(&bars[kBarK8Empty + s], 4);
      }
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
  const int n_items = a.paged ? min(*a.n_items, a.items_cap) : a.n_dense_items;

  if ((tmem_base & 0xFFFFu) != 0) {
    // the two accumulators assume the allocation starts at column 0
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTmemAlloc);
  } else if (warp == 0) {
    producer_role<H, DECODE>(a, &tmap_q, &tmap_k, smem, P, bars, abort, n_items);
  } else if (warp == 1) {
    if (lane == 0) mma_role<H, DECODE>(a, smem, P, bars, abort, n_items, tmem_base);
    __syncwarp();
  } else if (MIXED && warp >= 10) {
    convert_role<H, DECODE>(a, smem, P, bars, abort, n_items, tmem_base);
  } else {
    epilogue_role<H, DECODE>(a, smem, P, bars, abort, n_items, tmem_base);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int H, bool DECODE, bool MIXED>
cudaError_t launch_t(const ScoreArgs& a, const CUtensorMap* tq, const CUtensorMap* tk, int grid, size_t smem,
                     cudaStream_t st) {
  auto kern = score_kernel<H, DECODE, MIXED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, MIXED ? kMixedThreads : kScoreThreads, smem, st>>>(*tq, *tk, a);
  return cudaGetLastError();
}

}  // namespace

size_t score_smem_bytes(const ScoreArgs& a, int num_k_stages) {
  return plan_smem(a.N, a.D, a.q_fp8, a.k_fp8, num_k_stages, a.mixed).total;
}

cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap* tmap_q, const CUtensorMap* tmap_k, int grid,
                         size_t smem_bytes, cudaStream_t st) {
  const bool dec = a.N != 256;
#define DSA_CASE(HH)                                                                        \
  case HH:                                                                                  \
    return dec ? (a.mixed ? launch_t<HH, true, true>(a, tmap_q, tmap_k, grid, smem_bytes, st)          \
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
