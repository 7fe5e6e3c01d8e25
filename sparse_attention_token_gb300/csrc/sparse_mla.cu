// sparse_mla.cu -- multi-head latent attention over the indexer's top-k selection.
//
// GLM5 TensorCast adaptation design: the fused indexer hands topk_indices (and
// topk_limit) to the MLA backend, whose attention length is capped by the top-k width
// ("Sparse MLA 配置兼容", the _get_backend_kwargs hand-off; the performance model's
// sparse prefill / decode length).  Read as absorbed multi-head latent attention on the
// selected keys only:
//     logit[t, h, s] = scale * (q_nope[t, h] . c_kv[s] + q_rope[t, h] . k_rope[s])
//     out[t, h]      = sum_s softmax_s(logit[t, h, :]) * c_kv[s]          (latent output)
// over the logical key positions s = topk[t, j] >= 0 of token t's sequence, each read
// from the paged latent cache through block_tables.  An empty selection outputs zeros.
//
// One CTA per (query token, key split, group of up to 64 heads); its selected keys are
// taken 64 at a time (flash decoding with an exact combine across the splits):
//   warps 4..7  gather: each selected key's latent row (512 bf16) and rotary row (64
//               bf16) into a 128-byte-swizzled tile of 9 atom columns (16-byte cp.async,
//               zero-filled for padding), double buffered;
//   warp 8      TMEM allocator; lane 0 issues
//                 S  [heads x 64 keys]       = Q . K^T      (M = 128 rows of q, K-major A;
//                                                            the keys K-major B, K = 576)
//                 O^T[latent x heads]       += V^T . P^T    (M = 128 latent per MMA, the
//                                                            same key tile read MN-major as
//                                                            A; P K-major B, K = 64 keys)
//               with S double buffered and O^T (4 x heads columns) resident in TMEM;
//   warps 0..3  softmax and rescale: the threads of the head lanes take their head's 64
//               logits, keep a reference maximum and the sum (base-2 exponentials of the
//               scaled logits), write p as bf16 into P; when a head's reference moves,
//               every epilogue thread scales its O^T lanes by the heads' correction
//               factors before the next P . V accumulates; at the end they write the
//               unnormalised O, the reference maximum and the sum of the split.
// A second kernel combines the splits: out = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j.
// Every wait is bounded; on a timeout every role stops, copies and MMAs in flight are
// drained (bounded) and TMEM is freed.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "dsa_indexer.h"
#include "internal.h"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kKvRank = 512, kRopeDim = 64, kAtoms = 9;   // 576 = 9 atoms of 64 bf16
constexpr int kBlockKeys = 64;                           // keys per tile
constexpr int kHeadsPerCta = 64;
constexpr int kMlaThreads = 288;                         // warps 0-3 epilogue, 4-7 gather, 8 MMA
constexpr uint32_t kAtomBytes = kBlockKeys * 128;        // one atom column of a tile / of q
constexpr uint32_t kTileBytes = kAtoms * kAtomBytes;     // 73728
constexpr uint32_t kQBytes = kAtoms * kAtomBytes;        // q: 64 rows x 576
constexpr uint32_t kPBytes = kHeadsPerCta * 128;         // P: 64 heads x 64 keys bf16
constexpr uint32_t kOffQ = 0, kOffTile = kQBytes, kOffP = kOffTile + 2 * kTileBytes;
constexpr uint32_t kOffMisc = kOffP + kPBytes;
constexpr uint32_t kSCols = kBlockKeys;                  // one S buffer
constexpr uint32_t kOCol0 = 2 * kSCols;                  // O^T after the two S buffers

struct MlaArgs {
  int total_q, B, H, k, splits, keys_per_split, groups, page_size, num_pages, max_pages_per_seq;
  float scale_log2;          // scale * log2(e)
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  const int32_t* topk;
  const __nv_bfloat16* cache_c;
  const __nv_bfloat16* cache_r;
  float* part_o;             // [total_q, splits, H, 512]
  float* part_ml;            // [total_q, splits, H, 2]
  unsigned* status;
};

struct MlaBars {
  uint64_t qfull, tfull[2], tempty[2], sfull[2], sempty[2], pfull, ofree, done;
};

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ int seq_of_row(const MlaArgs& a, int r) {
  int lo = 0, hi = a.B;  // last b with cu_q_lens[b] <= r
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a.cu_q_lens + mid) <= r) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kMlaThreads, 1) sparse_mla_kernel(const __grid_constant__ CUtensorMap tmap_qn,
                                                                     const __grid_constant__ CUtensorMap tmap_qr,
                                                                     const MlaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusSmemAlign);
    return;
  }
  MlaBars* bars = reinterpret_cast<MlaBars*>(smem + kOffMisc);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kOffMisc + 128);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 132);
  volatile int* gather_ok = reinterpret_cast<volatile int*>(smem + kOffMisc + 136);
  float* corr = reinterpret_cast<float*>(smem + kOffMisc + 256);          // [64]
  long long* slot = reinterpret_cast<long long*>(smem + kOffMisc + 512);  // [64] cache row of each key, -1 none

  // work item: token t, key split j, head group g
  const int item = blockIdx.x;
  const int g = item % a.groups;
  const int j = (item / a.groups) % a.splits;
  const int t = item / (a.groups * a.splits);
  const int hg = min(kHeadsPerCta, a.H - g * kHeadsPerCta);  // heads of this CTA
  const int key0 = j * a.keys_per_split;
  const int nkeys = max(0, min(a.k, key0 + a.keys_per_split) - key0);
  const int nblk = (nkeys + kBlockKeys - 1) / kBlockKeys;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->qfull, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars->tfull[s], 128);  // every gather thread, after its copies landed
      ptx::mbar_init(&bars->tempty[s], 1);
      ptx::mbar_init(&bars->sfull[s], 1);
      ptx::mbar_init(&bars->sempty[s], 2);   // the two head-lane warps
    }
    ptx::mbar_init(&bars->pfull, 4);         // the four epilogue warps
    ptx::mbar_init(&bars->ofree, 1);
    ptx::mbar_init(&bars->done, 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 8) {
    ptx::tmem_alloc(tmem_holder, 512);
    ptx::tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    ptx::prefetch_tmap(&tmap_qn);
    ptx::prefetch_tmap(&tmap_qr);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  const int b = seq_of_row(a, t);
  const int seq_len = __ldg(a.seq_lens + b);
  const int32_t* sel = a.topk + static_cast<long long>(t) * a.k + key0;
  const long long part = (static_cast<long long>(t) * a.splits + j) * a.H + g * kHeadsPerCta;  // first head row

  if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sbase = ptx::smem_u32(smem);
      const uint32_t id1 = ptx::idesc_f32acc(128, kBlockKeys, true);   // S: 128 q rows x 64 keys
      const uint32_t id2 = ptx::idesc_f32acc_bf16_amn(128, hg);        // O^T: 128 latent x heads
      bool ok = nblk == 0 || ptx::mbar_wait(&bars->qfull, 0, abort, a.status, kStatusTimeout);
      auto gemm1 = [&](int blk) {
        const int tb = blk & 1;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + tb * kSCols;
        for (int at = 0; at < kAtoms; ++at) {
          const uint64_t ad = ptx::sw128_kmajor_desc(sbase + kOffQ + at * kAtomBytes);
          const uint64_t bd = ptx::sw128_kmajor_desc(sbase + kOffTile + tb * kTileBytes + at * kAtomBytes);
#pragma unroll
          for (int s = 0; s < 4; ++s)  // 16 bf16 of K per MMA inside the atom
            ptx::mma_bf16(d, ad + 2 * s, bd + 2 * s, id1, (at > 0 || s > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&bars->sfull[tb]);
      };
      auto gemm2 = [&](int blk) {
        ptx::tc_fence_after();
        const int tb = blk & 1;
        const uint32_t tile = sbase + kOffTile + tb * kTileBytes;
        const uint64_t bd0 = ptx::sw128_kmajor_desc(sbase + kOffP);
        for (int c = 0; c < 4; ++c) {  // latent 128c .. 128c + 127: atoms 2c and 2c + 1
          const uint32_t d = tmem_base + kOCol0 + c * kHeadsPerCta;
#pragma unroll
          for (int s = 0; s < 4; ++s) {  // 16 keys per MMA: two 8-key groups of 1024 bytes
            const uint64_t ad = ptx::sw128_mnmajor_desc(tile + 2 * c * kAtomBytes + s * 2048, kAtomBytes);
            ptx::mma_bf16(d, ad, bd0 + 2 * s, id2, (blk > 0 || s > 0) ? 1u : 0u);
          }
        }
        ptx::mma_commit(&bars->tempty[tb]);
        ptx::mma_commit(&bars->ofree);
      };
      // Issue whichever product has its inputs first: the next block's S (its key tile
      // gathered and its S buffer released) or this block's P . V (its P written), so
      // neither waits behind the other's inputs.  Bounded like every other wait.
      int n1 = 0, n2 = 0;
      uint64_t t0 = ptx::globaltimer();
      for (uint32_t spin = 0; ok && n2 < nblk; ++spin) {
        bool progress = false;
        if (n1 < nblk && n1 <= n2 + 1 && ptx::mbar_try_wait(&bars->tfull[n1 & 1], (n1 >> 1) & 1) &&
            ptx::mbar_try_wait(&bars->sempty[n1 & 1], ((n1 >> 1) & 1) ^ 1)) {
          gemm1(n1++);
          progress = true;
        }
        if (n2 < n1 && ptx::mbar_try_wait(&bars->pfull, n2 & 1)) {
          gemm2(n2++);
          progress = true;
        }
        if (progress) {
          t0 = ptx::globaltimer();
        } else if ((spin & 15u) == 15u) {
          if (*abort) break;
          if (ptx::globaltimer() - t0 > 2000000000ull) {
            *abort = 1;
            atomicOr(a.status, kStatusTimeout);
            break;
          }
        }
      }
      ptx::mma_commit(&bars->done);
      ptx::mbar_wait_drain(&bars->done, 0, a.status, kStatusTimeout, 200000000ull);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ gather (128 threads)
    const int gt = threadIdx.x - 128;
    if (gt == 0 && nblk > 0) {
      // this CTA's 64 q rows (heads of group g; rows past the group are not used), 9 atoms
      ptx::mbar_arrive_expect_tx(&bars->qfull, kQBytes);
      const int row0 = t * a.H + g * kHeadsPerCta;
      for (int at = 0; at < 8; ++at)
        ptx::tma_load_2d(smem + kOffQ + at * kAtomBytes, &tmap_qn, &bars->qfull, at * 64, row0);
      ptx::tma_load_2d(smem + kOffQ + 8 * kAtomBytes, &tmap_qr, &bars->qfull, 0, row0);
    }
    const int32_t* bt = a.block_tables + static_cast<long long>(b) * a.max_pages_per_seq;
    for (int blk = 0; blk < nblk; ++blk) {
      const int tb = blk & 1;
      int good = 1;
      if (gt == 0) good = ptx::mbar_wait(&bars->tempty[tb], ((blk >> 1) & 1) ^ 1, abort, a.status, kStatusTimeout);
      // the four gather warps agree before touching the buffer
      ptx::named_bar_sync(1, 128);
      if (gt == 0) *gather_ok = good;
      ptx::named_bar_sync(1, 128);
      if (!*gather_ok) break;  // the same decision in all four gather warps
      if (gt < kBlockKeys) {
        const int kk = blk * kBlockKeys + gt;
        long long sl = -1;
        if (kk < nkeys) {
          const int idx = __ldg(sel + kk);
          if (idx >= 0 && idx < seq_len) {
            const int lp = idx / a.page_size;
            const int pg = lp < a.max_pages_per_seq ? __ldg(bt + lp) : -1;
            if (pg >= 0 && pg < a.num_pages) sl = static_cast<long long>(pg) * a.page_size + idx % a.page_size;
            else atomicOr(a.status, kStatusBadPage);
          }
        }
        slot[gt] = sl;
      }
      ptx::named_bar_sync(1, 128);
      uint8_t* tile = smem + kOffTile + tb * kTileBytes;
      // 64 keys x 72 chunks of 16 bytes; consecutive threads take consecutive chunks of a key
      for (int e = gt; e < kBlockKeys * 72; e += 128) {
        const int key = e / 72, ch = e - key * 72;
        const int at = ch >> 3, c16 = ch & 7;
        const long long sl = slot[key];
        const void* src = at < 8 ? static_cast<const void*>(a.cache_c + (sl < 0 ? 0 : sl) * kKvRank + at * 64 + c16 * 8)
                                 : static_cast<const void*>(a.cache_r + (sl < 0 ? 0 : sl) * kRopeDim + c16 * 8);
        uint8_t* dst = tile + at * kAtomBytes + key * 128 + ((c16 ^ (key & 7)) << 4);
        ptx::cp_async_16(dst, src, sl < 0 ? 0u : 16u);
      }
      cp_async_wait_all();
      ptx::fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
      ptx::mbar_arrive(&bars->tfull[tb]);
    }
    // the q copy lands before the CTA can exit, whatever happened
    if (gt == 0 && nblk > 0) ptx::mbar_wait_drain(&bars->qfull, 0, a.status, kStatusTimeout, 200000000ull);
  } else {
    // ------------------------------------------------------------ softmax, rescale, output (warps 0..3)
    const int h = threadIdx.x;                  // head lane (warps 0, 1) / latent lane within a chunk
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const bool head_lane = warp < 2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // Every iteration runs both named barriers of the four warps whatever happened, so a
    // failed (timed-out) wait never leaves a warp behind at a barrier; after a failure the
    // warps only keep the barrier count.
    for (int blk = 0; blk < nblk; ++blk) {
      const int tb = blk & 1;
      float cr = 1.f;
      if (head_lane) {
        if (ok) ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->sfull[tb], (blk >> 1) & 1, abort, a.status,
                                                            kStatusTimeout)) != 0;
        if (ok) {
          ptx::tc_fence_after();
          uint32_t s0[32], s1[32];
          ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + tb * kSCols, s0);
          ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + tb * kSCols + 32, s1);
          ptx::tmem_ld_wait_regs(s0);
          ptx::tmem_ld_wait_regs(s1);
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&bars->sempty[tb]);
          // keys of this block past the split's selection, or padding, take no weight
          const int nvalid = min(kBlockKeys, nkeys - blk * kBlockKeys);
          float x[64];
          float mb = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = __uint_as_float(s0[i]) * a.scale_log2;
            x[32 + i] = __uint_as_float(s1[i]) * a.scale_log2;
          }
          const int32_t* selb = sel + blk * kBlockKeys;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            bool v = i < nvalid;
            if (v) {
              const int idx = __ldg(selb + i);
              v = idx >= 0 && idx < seq_len;
            }
            x[i] = v ? x[i] : -INFINITY;
            mb = fmaxf(mb, x[i]);
          }
          // The reference maximum moves only when the block's maximum exceeds it by more
          // than 8 (a factor 256 in probability): p stays below 256 and the output, which
          // divides by the sum taken against the same reference, is unchanged, while most
          // blocks need no rescaling of the accumulated output.
          float mn = m;
          if (m == -INFINITY) mn = mb;  // nothing accumulated yet (O is still zero)
          else if (mb > m + 8.f) mn = mb;
          cr = (m == -INFINITY || mn == m) ? 1.f : exp2f(m - mn);
          float ls = 0.f;
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float p0 = mn == -INFINITY ? 0.f : exp2f(x[2 * i] - mn);
            const float p1 = mn == -INFINITY ? 0.f : exp2f(x[2 * i + 1] - mn);
            ls += p0 + p1;
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
            pk[i] = *reinterpret_cast<const uint32_t*>(&pb);
          }
          l = l * cr + ls;
          m = mn;
          // P is free once the previous block's P . V has completed
          if (blk > 0)
            ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->ofree, (blk - 1) & 1, abort, a.status,
                                                        kStatusTimeout)) != 0;
          if (ok && h < hg) {
            // row h of P: 64 keys = 8 chunks of 16 bytes, swizzled by the row
            uint8_t* prow = smem + kOffP + h * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(prow + ((c ^ (h & 7)) << 4)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            corr[h] = cr;
          }
          ptx::fence_proxy_async_smem();
        }
      } else if (blk > 0 && ok) {
        ok = __all_sync(0xffffffffu, ptx::mbar_wait(&bars->ofree, (blk - 1) & 1, abort, a.status,
                                                    kStatusTimeout)) != 0;
      }
      // P and the correction factors are written; does any head need its output rescaled?
      uint32_t any;
      asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.f32 q, %1, 0f3F800000;\n\t"
                   "bar.red.or.pred p, 2, 128, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                   : "=r"(any) : "f"(head_lane && h < hg ? cr : 1.f) : "memory");
      if (any && blk > 0 && ok && !*abort) {
        // O^T *= corr per head column, for this thread's latent lane in each chunk
        ptx::tc_fence_after();
        for (int c = 0; c < 4; ++c) {
          const uint32_t col = tmem_base + lane_addr + kOCol0 + c * kHeadsPerCta;
          for (int h0 = 0; h0 < hg; h0 += 32) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(col + h0, r);
            ptx::tmem_ld_wait_regs(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr[h0 + i]);
            ptx::tmem_st_32x32b_x32(col + h0, r);
          }
        }
        ptx::tmem_st_wait();
      }
      ptx::tc_fence_before();
      if (any) ptx::named_bar_sync(2, 128);  // corr is read by everyone before the next block rewrites it
      if (lane == 0) ptx::mbar_arrive(&bars->pfull);
    }
    // the split's unnormalised output, maximum and sum
    bool fin = ok && (nblk == 0 || ptx::mbar_wait(&bars->ofree, (nblk - 1) & 1, abort, a.status, kStatusTimeout));
    fin = __all_sync(0xffffffffu, fin) != 0;
    if (head_lane && h < hg) {
      a.part_ml[(part + h) * 2] = m;
      a.part_ml[(part + h) * 2 + 1] = l;
    }
    if (fin) {
      ptx::tc_fence_after();
      for (int c = 0; c < 4; ++c) {
        const int lat = c * 128 + warp * 32 + lane;
        for (int h0 = 0; h0 < hg; h0 += 32) {
          uint32_t r[32];
          if (nblk > 0) {
            ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + kOCol0 + c * kHeadsPerCta + h0, r);
            ptx::tmem_ld_wait_regs(r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (h0 + i < hg) a.part_o[(part + h0 + i) * kKvRank + lat] = __uint_as_float(r[i]);
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

// out[t, h, :] = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j over the splits (0 when empty).
__global__ void sparse_mla_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                          int splits, int H, long long rows, float* __restrict__ out) {
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();
  const long long r = blockIdx.x;  // (t, h)
  if (r >= rows) return;
  const long long t = r / H, h = r - t * H;
  float M = -INFINITY;
  for (int jx = 0; jx < splits; ++jx) M = fmaxf(M, part_ml[((t * splits + jx) * H + h) * 2]);
  float L = 0.f;
  for (int jx = 0; jx < splits; ++jx) {
    const long long q = (t * splits + jx) * H + h;
    const float mj = part_ml[q * 2];
    if (mj != -INFINITY) L += exp2f(mj - M) * part_ml[q * 2 + 1];
  }
  for (int lat = threadIdx.x; lat < kKvRank; lat += blockDim.x) {
    float acc = 0.f;
    for (int jx = 0; jx < splits; ++jx) {
      const long long q = (t * splits + jx) * H + h;
      const float mj = part_ml[q * 2];
      if (mj != -INFINITY) acc += exp2f(mj - M) * part_o[q * kKvRank + lat];
    }
    out[r * kKvRank + lat] = L > 0.f ? acc / L : 0.f;
  }
}

bool mla_map(CUtensorMap* m, const void* base, long long rows, int cols) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct MlaPlan {
  int splits, keys_per_split, groups;
  size_t off_o, off_ml, total;
};

MlaPlan plan_mla(const dsa_sparse_mla_args* a, int sms) {
  MlaPlan p{};
  p.groups = (a->H + kHeadsPerCta - 1) / kHeadsPerCta;
  // Whole 64-key blocks per split.  One CTA fills an SM (shared memory), so the launch runs
  // in waves of `sms` CTAs, and a wave lasts as long as its CTAs' blocks plus about one
  // block's worth of fixed work (its q load, its partial output of 64 heads x 512 fp32,
  // which the combine reads back).  Take the blocks-per-split that minimises
  // waves x (blocks + 1); on a tie the larger one (fewer splits: the loop runs downwards).
  const long long base = std::max<long long>(1, static_cast<long long>(a->total_q) * p.groups);
  const int blocks = std::max(1, (a->topk_width + kBlockKeys - 1) / kBlockKeys);
  const long long n_sm = std::max(sms, 1);
  int best_bps = blocks;
  long long best_cost = -1;
  for (int bps = blocks; bps >= 1; --bps) {
    const long long splits = (blocks + bps - 1) / bps;
    const long long waves = (base * splits + n_sm - 1) / n_sm;
    const long long cost = waves * (bps + 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_bps = bps;
    }
  }
  const int bps = best_bps;
  p.keys_per_split = bps * kBlockKeys;
  p.splits = (blocks + bps - 1) / bps;
  const size_t rows = static_cast<size_t>(a->total_q) * p.splits * a->H;
  p.off_o = 0;
  p.off_ml = (rows * kKvRank * 4 + 255) / 256 * 256;
  p.total = p.off_ml + (rows * 2 * 4 + 255) / 256 * 256;
  return p;
}

dsa_status validate_mla(const dsa_sparse_mla_args* a) {
  if (!a) return DSA_ERR_INVALID_ARGUMENT;
  if (a->B < 0 || a->total_q < 0 || a->H <= 0 || a->topk_width < 1 || a->page_size <= 0 || a->num_pages < 0 ||
      a->max_pages_per_seq < 0 || !(a->scale > 0.f))
    return DSA_ERR_INVALID_ARGUMENT;
  if (a->kv_rank != kKvRank || a->rope_dim != kRopeDim) return DSA_ERR_UNSUPPORTED;
  if (a->H != 16 && a->H != 32 && a->H % 64 != 0) return DSA_ERR_UNSUPPORTED;
  if (static_cast<long long>(a->total_q) * a->H * kKvRank > (1LL << 40)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int mla_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return 148;
  return n > 0 ? n : 148;
}

}  // namespace

}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status dsa_sparse_mla_workspace_size(const dsa_sparse_mla_args* a, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARGUMENT;
  const dsa_status st = validate_mla(a);
  if (st != DSA_OK) return st;
  *bytes = plan_mla(a, mla_sms()).total;
  return DSA_OK;
}

dsa_status dsa_sparse_mla(const dsa_sparse_mla_args* a, dsa_stream_t stream) {
  dsa_status st = validate_mla(a);
  if (st != DSA_OK) return st;
  if (a->total_q == 0 || a->B == 0) return DSA_OK;
  if (!a->q_nope || !a->q_rope || !a->cache_c || !a->cache_r || !a->block_tables || !a->cu_q_lens ||
      !a->seq_lens || !a->topk || !a->out)
    return DSA_ERR_INVALID_ARGUMENT;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!al16(a->q_nope) || !al16(a->q_rope) || !al16(a->cache_c) || !al16(a->cache_r) || !al16(a->out))
    return DSA_ERR_INVALID_ARGUMENT;
  const MlaPlan p = plan_mla(a, mla_sms());
  if (!a->workspace || a->workspace_bytes < p.total || !al16(a->workspace)) return DSA_ERR_WORKSPACE;
  unsigned* status = device_status_ptr();
  if (!status) return DSA_ERR_CUDA;
  CUtensorMap tqn, tqr;
  const long long qrows = static_cast<long long>(a->total_q) * a->H;
  if (!mla_map(&tqn, a->q_nope, qrows, kKvRank) || !mla_map(&tqr, a->q_rope, qrows, kRopeDim)) return DSA_ERR_CUDA;
  MlaArgs k{};
  k.total_q = a->total_q;
  k.B = a->B;
  k.H = a->H;
  k.k = a->topk_width;
  k.splits = p.splits;
  k.keys_per_split = p.keys_per_split;
  k.groups = p.groups;
  k.page_size = a->page_size;
  k.num_pages = a->num_pages;
  k.max_pages_per_seq = a->max_pages_per_seq;
  k.scale_log2 = a->scale * 1.4426950408889634f;
  k.cu_q_lens = a->cu_q_lens;
  k.seq_lens = a->seq_lens;
  k.block_tables = a->block_tables;
  k.topk = a->topk;
  k.cache_c = static_cast<const __nv_bfloat16*>(a->cache_c);
  k.cache_r = static_cast<const __nv_bfloat16*>(a->cache_r);
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  k.part_o = reinterpret_cast<float*>(ws + p.off_o);
  k.part_ml = reinterpret_cast<float*>(ws + p.off_ml);
  k.status = status;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t smem = kOffMisc + 1024;
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  const long long items = static_cast<long long>(a->total_q) * p.splits * p.groups;
  if (items > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED;
  e = launch_pdl(sparse_mla_kernel, dim3(static_cast<unsigned>(items)), dim3(kMlaThreads), smem, s, tqn, tqr, k);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  e = launch_pdl(sparse_mla_combine_kernel, dim3(static_cast<unsigned>(qrows)), dim3(128), 0, s,
                 static_cast<const float*>(k.part_o), static_cast<const float*>(k.part_ml), p.splits, a->H, qrows,
                 static_cast<float*>(a->out));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // extern "C"
