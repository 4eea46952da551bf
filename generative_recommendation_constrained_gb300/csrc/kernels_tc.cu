// Full projection on the 5th-generation tensor cores (sm_103a):
//   Z[M][ldz] = H[M][d] . W[V][d]^T, fp32 accumulation in tensor memory.
//
// "ZeroGR: Filtering-First Constrained Decoding for Generative
// Recommendation" (paper-daily.com digest), section "Why computing fewer
// scores is not automatically faster": scoring every token is one regular
// large matrix product that GPUs execute best; steps with many legal tokens
// score everything, then pick the legal tokens.
//
// W_s is bf16 or fp16; the hidden vectors are fp32.  H is split as
// H = H_hi + H_lo with both halves in W's type, and both products are
// accumulated into the same fp32 accumulator, so the scores agree with the
// fp32 selective projection to ~1e-6 instead of the ~1e-3 a single rounding
// of H would give.
//
// Persistent CTAs (one per SM) walk 128 x 256 tiles: warp 0 issues TMA loads
// (128-byte swizzled K-major tiles) into a 3-stage shared-memory ring guarded
// by mbarriers, running ahead into the next tile; warp 1 owns two
// tensor-memory accumulators and issues tcgen05.mma from one thread into the
// one the epilogue has released; warps 2-9 (two per 32-lane quarter of the
// accumulator, one per 128-column half) read the other back with tcgen05.ld,
// fold the chunk partials, and store the fp32 scores as 32 x 32 blocks staged
// with the 128-byte swizzle and written by TMA stores (whole 128-byte lines),
// so a tile's epilogue overlaps the next tile's loads and MMAs.  Every wait is bounded; on
// expiry the kernel records kStatusTimeout, drains its own copies, frees its
// tensor memory and returns.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "zg_internal.h"

namespace zg {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;  // tile; kBK bf16 = 128 bytes = one swizzle row
constexpr int kTileA = kBM * kBK * 2;          // 16 KiB
constexpr int kTileB = kBN * kBK * 2;          // 32 KiB
constexpr int kTmemCols = 256;
constexpr int kStagingBytes = 8 * 4096;        // one 4 KiB store block per epilogue warp

// Shared-memory layout of one variant: SPLIT = the hidden as two half
// operands (two MMAs per K-step), else one (a single rounding of the hidden);
// ZSTORE = the scores are written out through staging blocks by TMA stores,
// else only the epilogue's per-chunk summaries leave the SM.
template <bool SPLIT, bool ZSTORE>
struct TcCfg {
  static constexpr int kA = SPLIT ? 2 : 1;                    // A operands a stage
  static constexpr int kStageBytes = kA * kTileA + kTileB;    // 64 or 48 KiB
  static constexpr int kStaging = ZSTORE ? kStagingBytes : 0;
  static constexpr int kStages = (227 * 1024 - 1024 - kStaging) / kStageBytes;  // 3 or 4
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + kStaging + 1024;
  static_assert(kStages >= 3, "a ring of three stages at least");
};
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA issuer, epilogue warps
constexpr uint32_t kSpinLimit = 1u << 26;  // default polls of a wait (seconds at most)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Bounded wait (`limit` polls) for the phase with the given parity; false on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(const void* p) {
  const uint64_t addr = smem_u32(p);
  uint64_t d = 0;
  d |= (addr & 0x3FFFFull) >> 4;          // start address
  d |= (uint64_t)(16 >> 4) << 16;         // leading byte offset (unused with swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor: f32 accumulate, A/B of type `ab` (0 f16, 1 bf16),
// both K-major, M = 128, N = 256.
__device__ __forceinline__ uint32_t instr_desc(uint32_t ab) {
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

// 2-D TMA store of a 32 x 32 fp32 block from shared memory (bulk group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <bool SPLIT, bool ZSTORE>
__global__ void __launch_bounds__(kThreads, 1)
    k_full_tc(const __grid_constant__ CUtensorMap map_hi, const __grid_constant__ CUtensorMap map_lo,
              const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_z, int M, int V,
              int d, int ldz, uint32_t ab_type, const FullEpi epi, uint32_t* status, uint32_t spin) {
  using Cfg = TcCfg<SPLIT, ZSTORE>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kStageBytes = Cfg::kStageBytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // stage buffers must sit on 1024-byte boundaries (swizzle atoms)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + kStages * kStageBytes;  // one 4 KiB block per epilogue warp (ZSTORE)
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (d + kBK - 1) / kBK;
  const int ntn = (V + kBN - 1) / kBN;
  const int ntiles = ntn * ((M + kBM - 1) / kBM);
  // tiles of this CTA: blockIdx.x, + gridDim.x, ...; tile t = (m-tile t / ntn, n-tile t % ntn)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], kEpiWarps);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(2 * kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;

  if (warp == 0 && lane == 0) {
    // producer: TMA ring, running ahead across tiles
    int kg = 0;  // k-blocks issued by this CTA
    for (int t = blockIdx.x; t < ntiles && !atomicAdd(&abort_flag, 0); t += gridDim.x) {
      const int m0 = (t / ntn) * kBM, n0 = (t % ntn) * kBN;
      for (int kb = 0; kb < nk; ++kb, ++kg) {
        const int st = kg % kStages;
        if (kg >= kStages && !mbar_wait(&empty_bar[st], ((kg / kStages) - 1) & 1, spin)) {
          atomicOr(status, kStatusTimeout);
          atomicExch(&abort_flag, 1);
          break;
        }
        uint8_t* sa_hi = smem + st * kStageBytes;
        uint8_t* sb = sa_hi + Cfg::kA * kTileA;
        mbar_expect_tx(&full_bar[st], kStageBytes);
        tma_load_2d(sa_hi, &map_hi, &full_bar[st], kb * kBK, m0);
        if constexpr (SPLIT) tma_load_2d(sa_hi + kTileA, &map_lo, &full_bar[st], kb * kBK, m0);
        tma_load_2d(sb, &map_w, &full_bar[st], kb * kBK, n0);
      }
    }
    // drain: every issued stage must have landed before the CTA may exit
    // (always the default limit, whatever the pipeline waits were given)
    for (int k = (kg > kStages ? kg - kStages : 0); k < kg; ++k)
      if (!mbar_wait(&full_bar[k % kStages], (k / kStages) & 1, kSpinLimit)) atomicOr(status, kStatusTimeout);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: accumulator buffer (i & 1) for the i-th tile of this CTA
    const uint32_t idesc = instr_desc(ab_type);
    int kg = 0, i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int b = i & 1;
      if (atomicAdd(&abort_flag, 0) || (i >= 2 && !mbar_wait(&tempty_bar[b], ((i >> 1) - 1) & 1, spin))) {
        atomicOr(status, kStatusTimeout);
        atomicExch(&abort_flag, 1);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t acc = tmem + (uint32_t)(b * kTmemCols);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb, ++kg) {
        const int st = kg % kStages;
        if (!mbar_wait(&full_bar[st], (kg / kStages) & 1, spin) || atomicAdd(&abort_flag, 0)) {
          atomicOr(status, kStatusTimeout);
          atomicExch(&abort_flag, 1);
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint8_t* sa_hi = smem + st * kStageBytes;
        const uint8_t* sb = sa_hi + Cfg::kA * kTileA;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t bd = smem_desc(sb + kk * 32);
          mma_f16(acc, smem_desc(sa_hi + kk * 32), bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          if constexpr (SPLIT) mma_f16(acc, smem_desc(sa_hi + kTileA + kk * 32), bd, idesc, 1u);
        }
        mma_commit(&empty_bar[st]);  // stage free once these MMAs have read it
      }
      mma_commit(&tfull_bar[b]);  // arrives once every MMA issued above has completed
      if (!ok) break;
    }
    // drain: every MMA this thread issued has finished with tensor memory and
    // the stage buffers before the accumulators are freed (default limit)
    mma_commit(&drain_bar);
    if (!mbar_wait(&drain_bar, 0, kSpinLimit)) atomicOr(status, kStatusTimeout);
  } else if (warp >= 2) {
    // epilogue: TMEM -> registers (one row a thread) -> partials, and the
    // scores through a swizzled staging block to TMA stores
    const int e = warp - 2;            // 0..7
    const int quarter = warp & 3;      // the accumulator lanes this warp may read
    const int half = e >> 2;           // 128-column half of the tile
    uint8_t* buf = staging + e * 4096;
    int issued = 0, i = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int b = i & 1;
      const int m0 = (t / ntn) * kBM, n0 = (t % ntn) * kBN;
      const int row = m0 + quarter * 32 + lane;
      // this row's legal-bitmap words for its four chunks, fetched while the
      // tile's MMAs run (they do not depend on the accumulator)
      uint32_t lmw[kBN / 64];
      bool dead = false;
#pragma unroll
      for (int ci = 0; ci < kBN / 64; ++ci) lmw[ci] = 0xFFFFFFFFu;
      if (epi.bitmap && row < M) {
        const uint32_t brow = epi.by_m ? (uint32_t)row : (epi.rows ? epi.rows[row] : 0u);
        dead = (brow == kDeadRow);
        if (!dead && brow >= epi.nrows) {  // never read past the table: flag, treat as dead
          atomicOr(status, kStatusRow);
          dead = true;
        }
        if (!dead) {
#pragma unroll
          for (int ci = 0; ci < kBN / 64; ++ci) {
            const int c0 = half * (kBN / 2) + ci * 32;
            if (n0 + c0 < V) lmw[ci] = epi.bitmap[(size_t)brow * epi.words + ((n0 + c0) >> 5)];
          }
        }
      }
      const bool got = mbar_wait(&tfull_bar[b], (i >> 1) & 1, spin);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (!got || atomicAdd(&abort_flag, 0)) {
        if (lane == 0) {
          atomicOr(status, kStatusTimeout);
          atomicExch(&abort_flag, 1);
        }
        break;
      }
      const uint32_t lane_addr = tmem + (uint32_t)(b * kTmemCols) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
      for (int ci = 0; ci < kBN / 64; ++ci) {
        const int c0 = half * (kBN / 2) + ci * 32;
        float v[32];
        tmem_ld32(lane_addr + (uint32_t)c0, v);
        if (n0 + c0 >= V) continue;  // uniform: a block wholly past the codebook
        const int chunk = (n0 + c0) >> 5;
        const int rem = V - (n0 + c0);
        const uint32_t vm = rem >= 32 ? 0xFFFFFFFFu : ((1u << rem) - 1u);
        if (row < M && epi.part) {
          // legal-only (max, sum exp) of this 32-token chunk (the fast
          // exponential: ~1e-6 relative, far inside the score tolerance);
          // with ptop also the second-largest legal z and the lowest token
          // offset holding the largest
          const uint32_t lm = dead ? 0u : (lmw[ci] & vm);
          float mx = -INFINITY, m2 = -INFINITY;
          int arg = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const bool l = (lm >> j) & 1u;
            const float x = v[j];
            if (l && x > mx) {
              m2 = mx;
              mx = x;
              arg = j;
            } else if (l && x > m2) {
              m2 = x;
            }
          }
          float sm = 0.f;
          if (mx != -INFINITY) {
#pragma unroll
            for (int j = 0; j < 32; ++j) sm += ((lm >> j) & 1u) ? __expf(v[j] - mx) : 0.f;
          }
          const size_t pi = (size_t)row * (ldz >> 5) + chunk;
          epi.part[pi] = make_float2(mx, sm);
          if (epi.ptop) epi.ptop[pi] = make_float2(m2, __int_as_float(arg));
        }
        if (row < M && epi.part_all) {
          // (max, sum exp) over every token of the chunk (score-first normaliser)
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) mx = ((vm >> j) & 1u) ? fmaxf(mx, v[j]) : mx;
          float sm = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) sm += ((vm >> j) & 1u) ? __expf(v[j] - mx) : 0.f;
          epi.part_all[(size_t)row * (ldz >> 5) + chunk] = make_float2(mx, sm);
        }
        if constexpr (ZSTORE) {
          // stage the 32 x 32 block (row = lane; 16-byte piece j of a row at
          // j ^ (row & 7): the 128-byte swizzle of the store map), then store
          if (issued > 0) {
            if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&map_z, buf, n0 + c0, m0 + quarter * 32);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
          ++issued;
        }
      }
      // this warp's part of accumulator b is read: let the MMA issuer reuse it
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&tempty_bar[b])) : "memory");
    }
    if constexpr (ZSTORE) {
      if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
    __syncwarp();
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * kTmemCols) : "memory");
  }
}

// H (fp32) -> H_hi + H_lo in the weights' half type.
template <typename HT>
__device__ __forceinline__ HT to_half(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 to_half<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half to_half<__half>(float x) {
  return __float2half_rn(x);
}
template <typename HT>
__device__ __forceinline__ float from_half(HT x);
template <>
__device__ __forceinline__ float from_half<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <>
__device__ __forceinline__ float from_half<__half>(__half x) {
  return __half2float(x);
}

template <typename HT>
__global__ void __launch_bounds__(256) k_split_h(const float* __restrict__ H, HT* __restrict__ hi, HT* __restrict__ lo,
                                                 size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float x = H[i];
    const HT h = to_half<HT>(x);
    hi[i] = h;
    if (lo) lo[i] = to_half<HT>(x - from_half<HT>(h));  // no lo: a single rounding of the hidden
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                              const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// 2-D K-major map: rows x d elements of 2 bytes, box box_rows x kBK, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, int rows, int d, int box_rows, bool bf16) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

std::atomic<uint32_t> g_wait_limit{kSpinLimit};

}  // namespace

cudaError_t launch_split_h(const float* H, void* hi, void* lo, size_t n, int w_dtype, cudaStream_t st) {
  const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
  if (w_dtype == ZG_BF16)
    k_split_h<__nv_bfloat16><<<blocks, 256, 0, st>>>(H, static_cast<__nv_bfloat16*>(hi),
                                                     static_cast<__nv_bfloat16*>(lo), n);
  else
    k_split_h<__half><<<blocks, 256, 0, st>>>(H, static_cast<__half*>(hi), static_cast<__half*>(lo), n);
  return cudaGetLastError();
}

namespace {

// Store map of the scores: fp32 [rows][ldz], 32 x 32 boxes, 128B swizzle.
bool make_store_map(CUtensorMap* m, float* Z, int rows, int ldz) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)ldz, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ldz * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, Z, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool SPLIT, bool ZSTORE>
cudaError_t launch_tc_t(const CUtensorMap& mh, const CUtensorMap& ml, const CUtensorMap& mw, const CUtensorMap& mz,
                        int M, int V, int d, int ldz, bool bf16, const FullEpi& epi, uint32_t* status,
                        cudaStream_t st) {
  auto kern = k_full_tc<SPLIT, ZSTORE>;
  constexpr size_t smem = TcCfg<SPLIT, ZSTORE>::kSmem;
  static bool attr_done = false;  // per instantiation
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  // persistent: one CTA per SM (shared memory admits one), tiles strided over the CTAs
  const int ntiles = ((V + kBN - 1) / kBN) * ((M + kBM - 1) / kBM);
  const int grid = std::max(1, std::min(ntiles, sm_count()));
  kern<<<grid, kThreads, smem, st>>>(mh, ml, mw, mz, M, V, d, ldz, bf16 ? 1u : 0u, epi, status,
                                     g_wait_limit.load(std::memory_order_relaxed));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_full_tc(const void* hi, const void* lo, const void* W, float* Z, int M, int V, int d, int ldz,
                           int w_dtype, const FullEpi& epi, uint32_t* status, cudaStream_t st) {
  const bool bf16 = (w_dtype == ZG_BF16);
  const bool split = (lo != nullptr);   // the hidden as hi + lo halves, else one rounding (hi)
  const bool zstore = (Z != nullptr);   // scores written out, else only the chunk summaries
  CUtensorMap mh, ml, mw, mz;
  if (ldz % 32 != 0 || !make_map(&mh, hi, M, d, kBM, bf16) || (split && !make_map(&ml, lo, M, d, kBM, bf16)) ||
      !make_map(&mw, W, V, d, kBN, bf16) || (zstore && !make_store_map(&mz, Z, M, ldz)))
    return cudaErrorInvalidValue;
  if (!zstore && !(epi.part && epi.ptop)) return cudaErrorInvalidValue;  // nothing would leave the kernel
  if (!split) ml = mh;
  if (!zstore) mz = mh;  // unused
  if (split)
    return zstore ? launch_tc_t<true, true>(mh, ml, mw, mz, M, V, d, ldz, bf16, epi, status, st)
                  : launch_tc_t<true, false>(mh, ml, mw, mz, M, V, d, ldz, bf16, epi, status, st);
  return zstore ? launch_tc_t<false, true>(mh, ml, mw, mz, M, V, d, ldz, bf16, epi, status, st)
                : launch_tc_t<false, false>(mh, ml, mw, mz, M, V, d, ldz, bf16, epi, status, st);
}

void set_wait_limit(uint32_t polls) { g_wait_limit.store(polls ? polls : kSpinLimit, std::memory_order_relaxed); }

}  // namespace zg
