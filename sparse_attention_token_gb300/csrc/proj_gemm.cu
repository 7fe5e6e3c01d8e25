// proj_gemm.cu -- the indexer front-end's projections on the sm_103a tensor cores.
//
// GLM5 TensorCast adaptation design, "性能模型设计" buckets 1-3 (the q, k and head-weight
// projection MMAs) and 4-5 (RoPE; on the FP8 path the rotation and the activation
// quantisation).  C[M, N] = A[M, K] . B[N, K]^T with A the token rows (qa_normed or
// hidden_states) and B the weight rows (wq_b, wk, weights_proj), both bf16 and K-major:
// exactly the operand layout of tcgen05.mma with M = 128 tokens per tile (one TMEM lane
// per token) and N = BN weight rows.
//
// Persistent kernel, one CTA per SM:
//   warp 0      TMA producer: 128 x 64 token slices and BN x 64 weight slices (one
//               128-byte swizzle atom of K) into an nS-deep ring;
//   warp 1      TMEM allocator; lane 0 issues the MMAs (4 per 64-wide K step) into two
//               BN-column fp32 accumulators, double buffered across tiles;
//   warps 2..9  epilogue, two warpgroups over the same token rows (one row per thread,
//               TMEM lane quarter = warp % 4), splitting the tile's columns between them:
//     kOutF32   fp32 rows into C (a K split s writes plane s; the row kernels add the
//               planes in order), or
//     kOutQRows the q rows finished in registers: RoPE on the first 2 HALF values of each
//               128-value head (pairs (i, i + HALF), or (2i, 2i + 1) when INTER), then
//               bf16, or the normalised Walsh-Hadamard rotation and the per-row e4m3
//               quantisation (scale = amax / 448, IEEE divisions, round to nearest even)
//               -- the same arithmetic, in the same order, as the q row kernel, without
//               the fp32 round trip through memory.
// Every wait is bounded; on a timeout every role stops, in-flight copies and MMAs are
// drained (bounded) and TMEM is freed.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {

namespace {

constexpr int kPM = 128;          // tokens per tile (TMEM lanes)
constexpr int kPK = 64;           // K per ring stage: one 128-byte atom of bf16
constexpr int kPThreads = 320;    // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue (two warpgroups)
constexpr int kPSmemBudget = 200 * 1024;

enum { kOutF32 = 0, kOutQRows = 1, kOutDual = 2 };

struct ProjArgs {
  int M, N, K;              // C[M, N] = A[M, K] . B[N, K]^T
  int ksteps, kc, splits;   // K in ksteps 64-wide steps, split into `splits` ranges of kc steps
  int n_mb, n_nb, n_tiles;  // tile = (mb * n_nb + nb) * splits + split
  int stages;
  int b_box;                // weight rows per TMA box: BN, or N when N < BN (rows past N are not stored)
  float* C;                 // kOutF32: plane s at C + s * plane, rows of ldc floats
  long long ldc, plane;
  // kOutDual: the weight rows are B's first 128 rows then B2's n2 rows; columns 0..127 go
  // to C as above, columns 128.. to C2 (plane s at C2 + s * plane2, rows of ldc2 floats)
  int n2;
  float* C2;
  long long ldc2, plane2;
  int H, fp8;               // kOutQRows: q_out [M, H, 128] (bf16, or e4m3 with q_scale [M, H])
  const float* cosb;
  const float* sinb;
  void* q_out;
  float* q_scale;
  unsigned* status;
};

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One 128-value q head row of token t in registers: RoPE, then bf16 or rotation +
// quantisation, then its store.
template <int HALF, bool INTER>
__device__ __forceinline__ void finish_q_row(float (&v)[128], const ProjArgs& a, long long t, int h) {
  if constexpr (HALF > 0) {
    const float* cs = a.cosb + t * HALF;
    const float* sn = a.sinb + t * HALF;
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
      const float c = __ldg(cs + i), s = __ldg(sn + i);
      const int i0 = INTER ? 2 * i : i, i1 = INTER ? 2 * i + 1 : i + HALF;
      const float x = v[i0], y = v[i1];
      v[i0] = x * c - y * s;
      v[i1] = x * s + y * c;
    }
  }
  const long long row = t * a.H + h;
  if (a.fp8) {
    // butterflies at distance 1, 2, 4, ..., 64 (Sylvester order), then 128^-1/2
#pragma unroll
    for (int len = 1; len < 128; len <<= 1) {
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        if ((i & len) == 0) {
          const float x = v[i], y = v[i + len];
          v[i] = x + y;
          v[i + len] = x - y;
        }
      }
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 128; ++i) {
      v[i] *= 0.08838834764831845f;
      m = max(m, __float_as_uint(fabsf(v[i])));
    }
    const float amax = __uint_as_float(m);
    const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.q_out) + row * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 16 * c + 4 * j;
        w[j] = e4m3x2(__fdiv_rn(v[i], scale), __fdiv_rn(v[i + 1], scale)) |
               (e4m3x2(__fdiv_rn(v[i + 2], scale), __fdiv_rn(v[i + 3], scale)) << 16);
      }
      dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    a.q_scale[row] = scale;
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.q_out) + row * 128);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * c + 2 * j], v[8 * c + 2 * j + 1]);
        w[j] = *reinterpret_cast<const uint32_t*>(&b);
      }
      dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

struct Tile {
  int mb, nb, s, k0, k1;
};

__device__ __forceinline__ Tile tile_of(const ProjArgs& a, int tile) {
  Tile T;
  T.s = tile % a.splits;
  const int mn = tile / a.splits;
  T.mb = mn / a.n_nb;
  T.nb = mn - T.mb * a.n_nb;
  T.k0 = T.s * a.kc;
  T.k1 = min(a.ksteps, T.k0 + a.kc);
  return T;
}

template <int BN, int OUT, int HALF, bool INTER>
__global__ void __launch_bounds__(kPThreads, 1) proj_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                             const __grid_constant__ CUtensorMap tmap_b,
                                                             const __grid_constant__ CUtensorMap tmap_b2,
                                                             const ProjArgs a) {
  constexpr uint32_t kAStage = kPM * 128, kBStage = BN * 128;
  constexpr uint32_t kCols = 2 * BN;  // two accumulators
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((ptx::smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusSmemAlign);
    return;
  }
  const int nS = a.stages;
  uint8_t* sa = smem;
  uint8_t* sb = smem + nS * kAStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sb + nS * kBStage);  // full[nS], empty[nS], tfull[2], tempty[2], done
  uint64_t* full = bars;
  uint64_t* empty = bars + nS;
  uint64_t* tfull = bars + 2 * nS;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < nS; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&tfull[s], 1);
      ptx::mbar_init(&tempty[s], 8);  // one arrival per epilogue warp
    }
    ptx::mbar_init(done, 1);
    *abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, kCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_b);
    if (OUT == kOutDual) ptx::prefetch_tmap(&tmap_b2);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  ptx::grid_dep_wait();  // the operands may come from the previous kernel on the stream
  ptx::grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      uint32_t n = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x) {
        const Tile T = tile_of(a, tile);
        for (int k = T.k0; k < T.k1; ++k, ++n) {
          const uint32_t s = n % nS;
          if (!ptx::mbar_wait(&empty[s], ((n / nS) & 1) ^ 1, abort, a.status, kStatusTimeout)) {
            ok = false;
            break;
          }
          const uint32_t b_rows = OUT == kOutDual ? 128u + static_cast<uint32_t>(a.n2) : static_cast<uint32_t>(a.b_box);
          ptx::mbar_arrive_expect_tx(&full[s], kAStage + b_rows * 128u);
          ptx::tma_load_2d(sa + s * kAStage, &tmap_a, &full[s], k * kPK, T.mb * kPM);
          ptx::tma_load_2d(sb + s * kBStage, &tmap_b, &full[s], k * kPK, T.nb * BN);
          if (OUT == kOutDual) ptx::tma_load_2d(sb + s * kBStage + 128 * 128, &tmap_b2, &full[s], k * kPK, 0);
        }
      }
      // drain: the copies issued into the ring land before the CTA can exit
      const uint32_t kk = n < static_cast<uint32_t>(nS) ? n : static_cast<uint32_t>(nS);
      for (uint32_t i = 1; i <= kk; ++i) {
        const uint32_t u = n - i;
        ptx::mbar_wait_drain(&full[u % nS], (u / nS) & 1, a.status, kStatusTimeout, 200000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_f32acc(kPM, BN, true);
      const uint32_t a0 = ptx::smem_u32(sa), b0 = ptx::smem_u32(sb);
      uint32_t n = 0, nt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < a.n_tiles && ok; tile += gridDim.x, ++nt) {
        const Tile T = tile_of(a, tile);
        const uint32_t acc = nt & 1;
        if (!ptx::mbar_wait(&tempty[acc], ((nt >> 1) & 1) ^ 1, abort, a.status, kStatusTimeout)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int k = T.k0; k < T.k1; ++k, ++n) {
          const uint32_t s = n % nS;
          if (!ptx::mbar_wait(&full[s], (n / nS) & 1, abort, a.status, kStatusTimeout)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ad = ptx::sw128_kmajor_desc(a0 + s * kAStage);
          const uint64_t bd = ptx::sw128_kmajor_desc(b0 + s * kBStage);
#pragma unroll
          for (int j = 0; j < 4; ++j)  // 16 bf16 (32 bytes) of K per MMA inside the 128-byte atom
            ptx::mma_bf16(d, ad + static_cast<uint64_t>(j * 2), bd + static_cast<uint64_t>(j * 2), idesc,
                          (k > T.k0 || j > 0) ? 1u : 0u);
          ptx::mma_commit(&empty[s]);
        }
        if (!ok) break;
        ptx::mma_commit(&tfull[acc]);
      }
      ptx::mma_commit(done);  // arrives once every MMA issued above has completed
      ptx::mbar_wait_drain(done, 0, a.status, kStatusTimeout, 200000000ull);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;  // the TMEM lane quarter this warp may read
    const int grp = (warp - 2) >> 2;  // epilogue warpgroup: 32-column chunks (heads) of its parity
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t nt = 0;
    for (int tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++nt) {
      const Tile T = tile_of(a, tile);
      const uint32_t acc = nt & 1;
      const bool ok = ptx::mbar_wait(&tfull[acc], (nt >> 1) & 1, abort, a.status, kStatusTimeout);
      if (__all_sync(0xffffffffu, ok) == 0) break;
      ptx::tc_fence_after();
      const long long t = static_cast<long long>(T.mb) * kPM + quarter * 32 + lane;
      const uint32_t tcol = tmem_base + lane_addr + acc * BN;
      if constexpr (OUT == kOutF32 || OUT == kOutDual) {
#pragma unroll 1
        for (int c = grp; c < BN / 32; c += 2) {
          // columns past N are not stored; kOutDual: columns 128.. belong to C2
          const bool second = OUT == kOutDual && c >= 4;
          const int ncols = OUT == kOutDual ? (second ? a.n2 : 128) : a.N;
          const int col0 = OUT == kOutDual ? 32 * (second ? c - 4 : c) : T.nb * BN + 32 * c;
          if (col0 >= ncols) break;
          float* crow = second ? a.C2 + T.s * a.plane2 + t * a.ldc2 + col0
                               : a.C + T.s * a.plane + t * a.ldc + col0;
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(tcol + 32 * c, r);
          ptx::tmem_ld_wait_regs(r);
          if (t < a.M) {
            if (col0 + 32 <= ncols && ((reinterpret_cast<uintptr_t>(crow) & 15u) == 0)) {
              float4* dst = reinterpret_cast<float4*>(crow);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                     __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (col0 + i < ncols) crow[i] = __uint_as_float(r[i]);
            }
          }
        }
      } else {
#pragma unroll 1
        for (int hh = grp; hh < BN / 128; hh += 2) {
          float v[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tcol + hh * 128 + 32 * c, r);
            ptx::tmem_ld_wait_regs(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
          }
          if (t < a.M) finish_q_row<HALF, INTER>(v, a, t, T.nb * (BN / 128) + hh);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kCols);
  }
}

bool proj_map(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
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
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kPK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

template <int BN, int OUT, int HALF, bool INTER>
cudaError_t launch_proj_t(const void* A, const void* B, ProjArgs a, cudaStream_t st, const void* B2 = nullptr) {
  CUtensorMap ta, tb, tb2;
  a.b_box = OUT == kOutDual ? 128 : (a.N < BN ? a.N : BN);
  if (!proj_map(&ta, A, a.M, a.K, kPM) || !proj_map(&tb, B, OUT == kOutDual ? 128 : a.N, a.K, a.b_box))
    return cudaErrorInvalidValue;
  if (OUT == kOutDual ? !proj_map(&tb2, B2, a.n2, a.K, a.n2) : false) return cudaErrorInvalidValue;
  if (OUT != kOutDual) tb2 = tb;
  const size_t stage = static_cast<size_t>(kPM) * 128 + static_cast<size_t>(BN) * 128;
  a.stages = static_cast<int>((kPSmemBudget - 256) / stage);
  if (a.stages > 8) a.stages = 8;
  const size_t smem = a.stages * stage + (2 * a.stages + 5) * 8 + 16;
  auto kern = proj_kernel<BN, OUT, HALF, INTER>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = std::min(a.n_tiles, sm_count());
  e = launch_pdl(kern, dim3(grid), dim3(kPThreads), smem, st, ta, tb, tb2, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

void fill_tiles(ProjArgs& a, int BN, int splits) {
  a.ksteps = (a.K + kPK - 1) / kPK;
  if (splits > a.ksteps) splits = a.ksteps;
  if (splits < 1) splits = 1;
  a.kc = (a.ksteps + splits - 1) / splits;
  a.splits = (a.ksteps + a.kc - 1) / a.kc;  // no empty split
  a.n_mb = (a.M + kPM - 1) / kPM;
  a.n_nb = (a.N + BN - 1) / BN;
  a.n_tiles = a.n_mb * a.n_nb * a.splits;
}

}  // namespace

int proj_bn(int N) { return N % 256 == 0 ? 256 : (N % 128 == 0 ? 128 : 64); }

int proj_splits(int M, int N, int K) {
  // with few token tiles, split K so that about 128 CTAs stream the weights (a fixed
  // target, so the workspace size depends on the shapes alone), each split at least 4
  // K steps; then drop splits that would be empty
  const int BN = proj_bn(N);
  const int tiles = ((M + kPM - 1) / kPM) * ((N + BN - 1) / BN);
  const int ksteps = (K + kPK - 1) / kPK;
  int s = 1;
  while (tiles * s * 2 <= 128 && (ksteps / (s * 2)) >= 4) s *= 2;
  const int kc = (ksteps + s - 1) / s;
  return (ksteps + kc - 1) / kc;
}

// C planes [splits][M, N] fp32 of A[M, K] . B[N, K]^T (K a multiple of 8); `splits` is
// proj_splits(M, N, K).
cudaError_t launch_proj_f32(const void* A, const void* B, int M, int N, int K, int splits, float* C,
                            unsigned* status, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (K % 8 || K <= 0 || (N % 4)) return cudaErrorInvalidValue;
  ProjArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.C = C;
  a.ldc = N;
  a.plane = static_cast<long long>(M) * N;
  a.status = status;
  const int BN = proj_bn(N);
  fill_tiles(a, BN, splits);
  if (a.splits != splits) return cudaErrorInvalidValue;  // the caller sized the planes for `splits`
  if (BN == 256) return launch_proj_t<256, kOutF32, 0, false>(A, B, a, st);
  if (BN == 128) return launch_proj_t<128, kOutF32, 0, false>(A, B, a, st);
  return launch_proj_t<64, kOutF32, 0, false>(A, B, a, st);
}

// The k and head-weight projections share their token operand: one pass over it.
// Kf planes [splits][M, 128] = A . Bk[128, K]^T, and W [M, n2] = A . Bw[n2, K]^T (planes
// [splits][M, n2] when split, else straight into W); n2 <= 128.
int proj_dual_splits(int M, int K) { return proj_splits(M, 256, K); }

cudaError_t launch_proj_dual(const void* A, const void* Bk, const void* Bw, int M, int n2, int K, int splits,
                             float* Kf, float* W, unsigned* status, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (K % 8 || K <= 0 || n2 < 1 || n2 > 128 || (n2 % 4)) return cudaErrorInvalidValue;
  ProjArgs a{};
  a.M = M;
  a.N = 128 + n2;
  a.K = K;
  a.C = Kf;
  a.ldc = 128;
  a.plane = static_cast<long long>(M) * 128;
  a.n2 = n2;
  a.C2 = W;
  a.ldc2 = n2;
  a.plane2 = static_cast<long long>(M) * n2;
  a.status = status;
  fill_tiles(a, 256, splits);
  if (a.splits != splits) return cudaErrorInvalidValue;
  return launch_proj_t<256, kOutDual, 0, false>(A, Bk, a, st, Bw);
}

// Whether the fused q projection covers this RoPE configuration.
bool proj_q_fused_supported(int H, int rope_dim) { return H % 2 == 0 && (rope_dim == 0 || rope_dim == 64 || rope_dim == 128); }

// q [M, H, 128] (bf16, or e4m3 with q_scale [M, H]) = the q row finish of A[M, K] . B[H * 128, K]^T.
cudaError_t launch_proj_q(const void* A, const void* B, int M, int H, int K, const float* cosb, const float* sinb,
                          int rope_dim, bool interleaved, bool fp8, void* q_out, float* q_scale, unsigned* status,
                          cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (!proj_q_fused_supported(H, rope_dim) || K % 8 || K <= 0) return cudaErrorInvalidValue;
  ProjArgs a{};
  a.M = M;
  a.N = H * 128;
  a.K = K;
  a.H = H;
  a.fp8 = fp8 ? 1 : 0;
  a.cosb = cosb;
  a.sinb = sinb;
  a.q_out = q_out;
  a.q_scale = q_scale;
  a.status = status;
  fill_tiles(a, 256, 1);
  if (rope_dim == 0) return launch_proj_t<256, kOutQRows, 0, false>(A, B, a, st);
  if (rope_dim == 64)
    return interleaved ? launch_proj_t<256, kOutQRows, 32, true>(A, B, a, st)
                       : launch_proj_t<256, kOutQRows, 32, false>(A, B, a, st);
  return interleaved ? launch_proj_t<256, kOutQRows, 64, true>(A, B, a, st)
                     : launch_proj_t<256, kOutQRows, 64, false>(A, B, a, st);
}

}  // namespace dsa
