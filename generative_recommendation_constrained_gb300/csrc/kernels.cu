// Decode-step kernels for sm_103a: selective projection into padded slots,
// prefix-state gather-add, SIMT full projection (fp32 weights), and the
// per-request select (masked log-softmax, cumulative add, top-K, emit).
//
// "ZeroGR: Filtering-First Constrained Decoding for Generative
// Recommendation" (paper-daily.com digest):
//   "Overall flow": per step, hidden vector -> legal tokens from the index ->
//     score the legal tokens -> log-softmax over the legal tokens only, add
//     to the cumulative log-probability, choose the next beams;
//   "Why computing fewer scores is not automatically faster": every beam of a
//     step gets the same number of slots (the step's largest fan-out, or the
//     whole codebook on dense steps), a candidate's slot depends only on its
//     beam and rank, empty slots score -inf, weight rows are read in place
//     (no compacted list, no temporary matrix);
//   "Why slice the index by decoding step": a beam carries only its row
//     number; the position of an entry is its next-step row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "zg_internal.h"

namespace zg {

__device__ uint32_t g_status;  // device status word, read by zg_check_device_status

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void flag(uint32_t* st, uint32_t bit) { atomicOr(st, bit); }

// Order-preserving map float -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f2ord(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// 16 bytes of weights -> fp32 lanes (exact widening for bf16/fp16).
template <typename WT>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int E = 4;
  __device__ __forceinline__ static void cvt(const uint4& r, float* o) {
    o[0] = __uint_as_float(r.x);
    o[1] = __uint_as_float(r.y);
    o[2] = __uint_as_float(r.z);
    o[3] = __uint_as_float(r.w);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ __forceinline__ static void cvt(const uint4& r, float* o) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Vec<__half> {
  static constexpr int E = 8;
  __device__ __forceinline__ static void cvt(const uint4& r, float* o) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h2 = *reinterpret_cast<const __half2*>(&w[i]);
      float2 f = __half22float2(h2);
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// (max, sum exp(x - max)) pairs combine associatively.
__device__ __forceinline__ float2 lse_combine(float2 a, float2 b) {
  float m = fmaxf(a.x, b.x);
  if (m == -INFINITY) return make_float2(-INFINITY, 0.f);
  float s = 0.f;
  if (a.y > 0.f) s += a.y * expf(a.x - m);
  if (b.y > 0.f) s += b.y * expf(b.x - m);
  return make_float2(m, s);
}

// State of beam k of request q entering step s.
struct BeamState {
  uint32_t row;
  float cum;
  int par, tok;
};
__device__ __forceinline__ BeamState load_beam(const StepLaunch& a, int q, int k) {
  BeamState bs;
  if (a.s == 1) {
    bs.row = 0;
    bs.cum = 0.f;
    bs.par = 0;
    bs.tok = 0;
  } else {
    const int i = q * a.beam + k;
    bs.row = a.row_in ? a.row_in[i] : 0u;
    bs.cum = a.cum_in[i];
    bs.par = a.par_in[i];
    bs.tok = a.tok_in[i];
    if (!a.row_in && bs.cum == -INFINITY) bs.row = kDeadRow;  // unconstrained: dead by score
  }
  return bs;
}

// ---------------------------------------------------------------------------
// Selective projection: one warp per (beam, 32-slot chunk).
// The warp gathers h_b = h_parent + C_{s-1}[token] (fp32, lane-sliced in
// registers), reads each legal token's weight row in place with coalesced
// 16-byte loads, accumulates per-lane partial dots for the 32 rows and
// reduce-scatters them with 31 shuffles so lane j ends with z of slot j.
// It writes the chunk's 32 slots (-inf where empty) and the chunk's
// (max, sum exp) partial of the legal-only log-sum-exp.
// ---------------------------------------------------------------------------
template <typename WT, int VPL>
__global__ void __launch_bounds__(256) k_selective(const StepLaunch a) {
  using VT = Vec<WT>;
  constexpr int E = VT::E;
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int N = a.B * a.Wc;
  const int d = a.d;
  const int nvec = d / E;
  const int64_t items = (int64_t)N * a.nch;
  const bool dense = (a.mode == kSelDense);
  for (int64_t it = wid; it < items; it += nw) {
    const int c = (int)(it / N);
    const int b = (int)(it - (int64_t)c * N);
    const int q = b / a.Wc, k = b - q * a.Wc;
    const BeamState bs = load_beam(a, q, k);
    if (bs.row == kDeadRow) continue;
    if (bs.row >= a.tab.rows) {
      if (lane == 0) flag(a.status, kStatusRow);
      continue;
    }
    const uint32_t rp0 = a.tab.rowptr[bs.row];
    const uint32_t F = a.tab.rowptr[bs.row + 1] - rp0;
    const int j0 = c * kChunk;
    uint32_t vmask;
    int t_lane = 0;
    if (dense) {
      const uint32_t bits = a.tab.bitmap[(size_t)bs.row * a.tab.words + c];
      const int tl = j0 + lane;
      vmask = bits;
      t_lane = tl;
      if (a.V - j0 < 32) vmask &= (a.V - j0 <= 0) ? 0u : ((1u << (a.V - j0)) - 1u);
    } else {
      if ((uint32_t)j0 >= F) continue;  // empty chunk: nothing to score or write
      const int nvalid = min(32, (int)F - j0);
      vmask = (nvalid == 32) ? kFull : ((1u << nvalid) - 1u);
      if (lane < nvalid) t_lane = a.tab.col[rp0 + j0 + lane];
    }
    if (((vmask >> lane) & 1u) && t_lane >= a.V) {
      flag(a.status, kStatusToken);
      vmask &= ~(1u << lane);
    }
    vmask = __ballot_sync(kFull, (vmask >> lane) & 1u);  // each lane vouches for its own slot

    // gather-add: this lane's slice of h_b
    float h[VPL][E];
    {
      const float* hp;
      const float* cr = nullptr;
      if (a.s == 1) {
        hp = a.u + (size_t)q * d;
      } else {
        hp = a.h_prev + ((size_t)q * a.Wp + bs.par) * d;
        cr = a.C_prev + (size_t)bs.tok * d;
      }
#pragma unroll
      for (int r = 0; r < VPL; ++r) {
        const int v = lane + 32 * r;
#pragma unroll
        for (int e = 0; e < E; ++e) h[r][e] = 0.f;
        if (v < nvec) {
#pragma unroll
          for (int e4 = 0; e4 < E; e4 += 4) {
            float4 x = *reinterpret_cast<const float4*>(hp + v * E + e4);
            if (cr) {
              float4 y = *reinterpret_cast<const float4*>(cr + v * E + e4);
              x.x += y.x;
              x.y += y.y;
              x.z += y.z;
              x.w += y.w;
            }
            h[r][e4] = x.x;
            h[r][e4 + 1] = x.y;
            h[r][e4 + 2] = x.z;
            h[r][e4 + 3] = x.w;
            if (c == 0 && a.h_out)
              *reinterpret_cast<float4*>(a.h_out + (size_t)b * d + v * E + e4) = x;
          }
        }
      }
    }

    float acc[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) acc[r] = 0.f;
    const WT* Wm = static_cast<const WT*>(a.W);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (((vmask >> (8 * g)) & 0xFFu) == 0u) continue;
      uint4 raw[8][VPL];
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = 8 * g + rr;
        const int t = __shfl_sync(kFull, t_lane, r);
        const bool ok = (vmask >> r) & 1u;
        const WT* wrow = Wm + (size_t)t * d;
#pragma unroll
        for (int vv = 0; vv < VPL; ++vv) {
          const int v = lane + 32 * vv;
          raw[rr][vv] = (ok && v < nvec) ? ldg_stream(wrow + v * E) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        float s = 0.f;
#pragma unroll
        for (int vv = 0; vv < VPL; ++vv) {
          float w[E];
          VT::cvt(raw[rr][vv], w);
#pragma unroll
          for (int e = 0; e < E; ++e) s = fmaf(w[e], h[vv][e], s);
        }
        acc[8 * g + rr] = s;
      }
    }
    // reduce-scatter: lane j ends with the full dot of row j
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const bool upper = lane & off;
#pragma unroll
      for (int i = 0; i < off; ++i) {
        const float send = upper ? acc[i] : acc[i + off];
        const float keep = upper ? acc[i + off] : acc[i];
        acc[i] = keep + __shfl_xor_sync(kFull, send, off);
      }
    }
    const bool valid = (vmask >> lane) & 1u;
    const float z = valid ? acc[0] : -INFINITY;
    float m = warp_max(z);
    float e = valid ? expf(z - m) : 0.f;
    float ssum = warp_sum(e);
    ssum = __shfl_sync(kFull, ssum, 0);
    a.Z[(size_t)b * a.S + j0 + lane] = z;
    if (lane == 0) a.part[(size_t)b * a.nch + c] = make_float2(m, vmask ? ssum : 0.f);
  }
}

// ---------------------------------------------------------------------------
// Gather-add for full-projection steps: H[b] = h_parent + C_{s-1}[token]
// (zero rows for dead beams).  One warp per beam, float4 accesses.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gather_add(const StepLaunch a, float* H) {
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int N = a.B * a.Wc;
  const int d4 = a.d / 4;
  for (int b = wid; b < N; b += nw) {
    const int q = b / a.Wc, k = b - q * a.Wc;
    const BeamState bs = load_beam(a, q, k);
    float4* out = reinterpret_cast<float4*>(H + (size_t)b * a.d);
    if (bs.row == kDeadRow || bs.cum == -INFINITY) {
      for (int v = lane; v < d4; v += 32) out[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    const float4* hp = reinterpret_cast<const float4*>(a.h_prev + ((size_t)q * a.Wp + bs.par) * a.d);
    const float4* cr = reinterpret_cast<const float4*>(a.C_prev + (size_t)bs.tok * a.d);
    for (int v = lane; v < d4; v += 32) {
      float4 x = hp[v], y = cr[v];
      out[v] = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
    }
  }
}

// ---------------------------------------------------------------------------
// SIMT full projection Z[M][ldz] = H[M][d] . W[V][d]^T in fp32 (fp32
// weights: the fp32 tolerance rules out tf32/bf16 tensor-core inputs).
// 64x64 tile, k-slab 16, 256 threads with 4x4 outputs each.
// ---------------------------------------------------------------------------
template <typename WT>
__global__ void __launch_bounds__(256) k_full_simt(const float* __restrict__ H, const WT* __restrict__ W,
                                                   float* __restrict__ Z, int M, int V, int d, int ldz) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += BK) {
    {  // A: 64 rows x 16 k = 256 float4
      const int r = tid >> 2, kq = (tid & 3) * 4;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m0 + r < M && k0 + kq < d) x = *reinterpret_cast<const float4*>(H + (size_t)(m0 + r) * d + k0 + kq);
      As[kq][r] = x.x;
      As[kq + 1][r] = x.y;
      As[kq + 2][r] = x.z;
      As[kq + 3][r] = x.w;
    }
    {  // B: 64 token rows x 16 k
      const int r = tid >> 2, kq = (tid & 3) * 4;
      float w[4] = {0.f, 0.f, 0.f, 0.f};
      if (n0 + r < V && k0 + kq < d) {
        const WT* p = W + (size_t)(n0 + r) * d + k0 + kq;
        if constexpr (sizeof(WT) == 4) {
          float4 x = *reinterpret_cast<const float4*>(p);
          w[0] = x.x;
          w[1] = x.y;
          w[2] = x.z;
          w[3] = x.w;
        } else {
          uint2 raw = *reinterpret_cast<const uint2*>(p);
          uint4 r4 = make_uint4(raw.x, raw.y, 0, 0);
          float t8[8];
          Vec<WT>::cvt(r4, t8);
          w[0] = t8[0];
          w[1] = t8[1];
          w[2] = t8[2];
          w[3] = t8[3];
        }
      }
      Bs[kq][r] = w[0];
      Bs[kq + 1][r] = w[1];
      Bs[kq + 2][r] = w[2];
      Bs[kq + 3][r] = w[3];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < V) Z[(size_t)m * ldz + n] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// Select: one CTA per request.
//  1. per beam: row, F (legal count), cumulative score, legal-only
//     log-sum-exp (from the selective chunk partials, or by a pass over the
//     legal full scores);
//  2. radix select (12+12+8 bits of an order-preserving key of
//     cand = cum + (z - lse)) of the keep-th best legal candidate;
//  3. collect the winners (ties at the threshold by lower flat slot index),
//     bitonic-sort them by (score desc, flat slot asc);
//  4. write the next beams (parent, token, next row, score) or, at the last
//     step, the output SIDs by following parent indices back.
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 512;

struct SelShared {
  int cnt[ZG_MAX_BEAM];
  int start[ZG_MAX_BEAM + 1];
  float cum[ZG_MAX_BEAM];
  float lse[ZG_MAX_BEAM];
  uint32_t rp[ZG_MAX_BEAM];
  uint32_t row[ZG_MAX_BEAM];
  int nleg[ZG_MAX_BEAM];
  uint32_t hist[4096];
  unsigned long long win[ZG_MAX_BEAM];
  int warp_tot[kSelThreads / 32];
  uint32_t prefix, prefmask;
  int need, cnt_gt, cnt_eq, nwin, nlegal, total;
};

__device__ __forceinline__ int find_beam(const SelShared& sh, int Wc, int c) {
  int lo = 0, hi = Wc - 1;  // largest k with start[k] <= c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sh.start[mid] <= c)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ bool is_legal_dense(const StepLaunch& a, uint32_t row, int t) {
  return (a.tab.bitmap[(size_t)row * a.tab.words + (t >> 5)] >> (t & 31)) & 1u;
}

// Key and legality of flat candidate c of request q.
__device__ __forceinline__ uint32_t cand_key(const StepLaunch& a, const SelShared& sh, int q, int c, bool* legal) {
  const int k = find_beam(sh, a.Wc, c);
  const int j = c - sh.start[k];
  const size_t zb = (size_t)(q * a.Wc + k) * a.S;
  float z;
  bool ok = true;
  switch (a.mode) {
    case kSelSparse:
    case kUncon:
      z = a.Z[zb + j];
      break;
    case kFullSparse:
      z = a.Z[zb + a.tab.col[sh.rp[k] + j]];
      break;
    default:  // kSelDense, kFullDense
      ok = is_legal_dense(a, sh.row[k], j);
      z = a.Z[zb + j];
      break;
  }
  *legal = ok;
  return f2ord(sh.cum[k] + (z - sh.lse[k]));
}

__global__ void __launch_bounds__(kSelThreads) k_select(const StepLaunch a) {
  __shared__ SelShared sh;
  const int q = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kSelThreads / 32;
  const int Wc = a.Wc;
  const bool constrained = (a.mode != kUncon);
  const bool sparse_slots = (a.mode == kSelSparse || a.mode == kFullSparse);

  // 1. beam setup
  for (int k = tid; k < Wc; k += kSelThreads) {
    const BeamState bs = load_beam(a, q, k);
    bool dead = (bs.row == kDeadRow) || (bs.cum == -INFINITY);
    uint32_t F = 0, rp = 0;
    if (!dead && constrained) {
      if (bs.row >= a.tab.rows) {
        flag(a.status, kStatusRow);
        dead = true;
      } else {
        rp = a.tab.rowptr[bs.row];
        F = a.tab.rowptr[bs.row + 1] - rp;
      }
    } else if (!dead) {
      F = (uint32_t)a.V;
    }
    sh.row[k] = bs.row;
    sh.rp[k] = rp;
    sh.cum[k] = bs.cum;
    sh.cnt[k] = dead ? 0 : (sparse_slots ? (int)F : a.V);
    sh.nleg[k] = dead ? 0 : (int)F;
    sh.lse[k] = 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    int s = 0, nl = 0;
    for (int k = 0; k < Wc; ++k) {
      sh.start[k] = s;
      s += sh.cnt[k];
      nl += sh.nleg[k];
    }
    sh.start[Wc] = s;
    sh.total = s;
    sh.nlegal = nl;
  }
  __syncthreads();
  // legal-only log-sum-exp per beam (one warp per beam)
  for (int k = warp; k < Wc; k += NW) {
    if (sh.cnt[k] == 0) continue;
    const int b = q * Wc + k;
    float2 acc = make_float2(-INFINITY, 0.f);
    if (a.mode == kSelSparse || a.mode == kSelDense) {
      const int nch = (a.mode == kSelSparse) ? (sh.cnt[k] + kChunk - 1) / kChunk : a.nch;
      for (int c = lane; c < nch; c += 32) acc = lse_combine(acc, a.part[(size_t)b * a.nch + c]);
    } else {
      const int n = sh.cnt[k];
      const size_t zb = (size_t)b * a.S;
      float m = -INFINITY;
      for (int j = lane; j < n; j += 32) {
        float z;
        if (a.mode == kFullSparse)
          z = a.Z[zb + a.tab.col[sh.rp[k] + j]];
        else if (a.mode == kFullDense)
          z = is_legal_dense(a, sh.row[k], j) ? a.Z[zb + j] : -INFINITY;
        else
          z = a.Z[zb + j];
        m = fmaxf(m, z);
      }
      float sm = 0.f;
      for (int j = lane; j < n; j += 32) {
        float z;
        if (a.mode == kFullSparse)
          z = a.Z[zb + a.tab.col[sh.rp[k] + j]];
        else if (a.mode == kFullDense)
          z = is_legal_dense(a, sh.row[k], j) ? a.Z[zb + j] : -INFINITY;
        else
          z = a.Z[zb + j];
        if (z != -INFINITY) sm += expf(z - m);
      }
      acc = make_float2(m, sm);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float2 other;
      other.x = __shfl_xor_sync(kFull, acc.x, o);
      other.y = __shfl_xor_sync(kFull, acc.y, o);
      acc = lse_combine(acc, other);
    }
    if (lane == 0) sh.lse[k] = acc.x + logf(acc.y);
  }
  __syncthreads();

  const int total = sh.total;
  const int keep_n = min(a.keep, sh.nlegal);
  if (tid == 0) {
    sh.nwin = 0;
    sh.prefix = 0;
    sh.prefmask = 0;
    sh.need = keep_n;
    sh.cnt_gt = 0;
    sh.cnt_eq = 0;
  }
  __syncthreads();

  bool take_all = (keep_n == sh.nlegal);
  if (!take_all && keep_n > 0) {
    // 2. radix select of the keep_n-th largest key
    const int shifts[3] = {20, 8, 0};
    const int widths[3] = {12, 12, 8};
    for (int p = 0; p < 3; ++p) {
      const int nb = 1 << widths[p];
      for (int i = tid; i < nb; i += kSelThreads) sh.hist[i] = 0;
      __syncthreads();
      const uint32_t pm = sh.prefmask, pv = sh.prefix;
      for (int c = tid; c < total; c += kSelThreads) {
        bool legal;
        const uint32_t key = cand_key(a, sh, q, c, &legal);
        if (legal && (key & pm) == pv) atomicAdd(&sh.hist[(key >> shifts[p]) & (nb - 1)], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // suffix scan from the top bin: lane l owns bins [nb - (l+1)*per, nb - l*per)
        const int per = nb / 32;
        const int hi = nb - lane * per;
        uint32_t mine = 0;
        for (int i = hi - per; i < hi; ++i) mine += sh.hist[i];
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t y = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - mine;
        const uint32_t target = (uint32_t)(sh.need - sh.cnt_gt);
        const bool here = (excl < target) && (incl >= target);
        const unsigned who = __ballot_sync(kFull, here);
        if (here && lane == __ffs(who) - 1) {
          uint32_t run = excl;
          for (int i = hi - 1; i >= hi - per; --i) {
            const uint32_t h = sh.hist[i];
            if (run + h >= target) {
              sh.cnt_gt += (int)run;
              sh.prefix |= (uint32_t)i << shifts[p];
              sh.prefmask |= (uint32_t)(nb - 1) << shifts[p];
              sh.cnt_eq = (int)h;
              break;
            }
            run += h;
          }
        }
      }
      __syncthreads();
    }
  }

  // 3. collect winners
  const uint32_t T = sh.prefix;
  const int need_eq = sh.need - sh.cnt_gt;
  const bool all_eq = take_all || (need_eq == sh.cnt_eq);
  if (keep_n > 0) {
    for (int c = tid; c < total; c += kSelThreads) {
      bool legal;
      const uint32_t key = cand_key(a, sh, q, c, &legal);
      if (!legal) continue;
      if (take_all || key > T || (all_eq && key == T)) {
        const int slot = atomicAdd(&sh.nwin, 1);
        sh.win[slot] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)c);
      }
    }
    __syncthreads();
    if (!all_eq) {
      // ties at the threshold: the need_eq lowest flat indices, in order
      int base = 0;
      for (int c0 = 0; c0 < total && base < need_eq; c0 += kSelThreads) {
        const int c = c0 + tid;
        bool f = false;
        uint32_t key = 0;
        if (c < total) {
          bool legal;
          key = cand_key(a, sh, q, c, &legal);
          f = legal && key == T;
        }
        const unsigned bal = __ballot_sync(kFull, f);
        if (lane == 0) sh.warp_tot[warp] = __popc(bal);
        __syncthreads();
        int before = base;
        for (int w = 0; w < warp; ++w) before += sh.warp_tot[w];
        before += __popc(bal & ((1u << lane) - 1u));
        if (f && before < need_eq) {
          const int slot = atomicAdd(&sh.nwin, 1);
          sh.win[slot] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)c);
        }
        int tile = 0;
        for (int w = 0; w < NW; ++w) tile += sh.warp_tot[w];
        __syncthreads();
        base += tile;
      }
    }
  }
  __syncthreads();
  const int nwin = keep_n;
  // bitonic sort (descending) of the winners
  int P = 1;
  while (P < nwin) P <<= 1;
  for (int i = nwin + tid; i < P; i += kSelThreads) sh.win[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += kSelThreads) {
        const int jx = i ^ stride;
        if (jx > i) {
          const bool desc = ((i & size) == 0);
          const unsigned long long x = sh.win[i], y = sh.win[jx];
          if (desc ? (x < y) : (x > y)) {
            sh.win[i] = y;
            sh.win[jx] = x;
          }
        }
      }
      __syncthreads();
    }
  }

  // 4. outputs
  const int s = a.s;
  const size_t BW = (size_t)a.B * a.beam;
  for (int i = tid; i < a.keep; i += kSelThreads) {
    if (i < nwin) {
      const unsigned long long w = sh.win[i];
      const uint32_t key = (uint32_t)(w >> 32);
      const int c = (int)(0xFFFFFFFFu - (uint32_t)(w & 0xFFFFFFFFu));
      const int k = find_beam(sh, Wc, c);
      const int j = c - sh.start[k];
      const float score = ord2f(key);
      int t;
      uint32_t nrow = 0;
      if (sparse_slots) {
        t = a.tab.col[sh.rp[k] + j];
        nrow = sh.rp[k] + (uint32_t)j;
      } else {
        t = j;
        if (constrained) {
          const uint32_t* bm = a.tab.bitmap + (size_t)sh.row[k] * a.tab.words;
          uint32_t rank = 0;
          for (int wd = 0; wd < (t >> 5); ++wd) rank += __popc(bm[wd]);
          rank += __popc(bm[t >> 5] & ((1u << (t & 31)) - 1u));
          nrow = sh.rp[k] + rank;
        }
      }
      if (s < a.L) {
        const size_t o = (size_t)q * a.beam + i;
        if (a.row_out) a.row_out[o] = nrow;
        a.cum_out[o] = score;
        a.tok_hist[(size_t)(s - 1) * BW + o] = t;
        a.par_hist[(size_t)(s - 1) * BW + o] = k;
      } else {
        a.out_scores[(size_t)q * a.K + i] = score;
        int32_t* sid = a.out_sids + ((size_t)q * a.K + i) * a.L;
        sid[a.L - 1] = t;
        int kc = k;
        for (int sp = a.L - 1; sp >= 1; --sp) {
          const size_t o = (size_t)(sp - 1) * BW + (size_t)q * a.beam + kc;
          sid[sp - 1] = a.tok_hist[o];
          kc = a.par_hist[o];
        }
      }
    } else {
      if (s < a.L) {
        const size_t o = (size_t)q * a.beam + i;
        if (a.row_out) a.row_out[o] = kDeadRow;
        a.cum_out[o] = -INFINITY;
        a.tok_hist[(size_t)(s - 1) * BW + o] = 0;
        a.par_hist[(size_t)(s - 1) * BW + o] = 0;
      } else {
        a.out_scores[(size_t)q * a.K + i] = -INFINITY;
        int32_t* sid = a.out_sids + ((size_t)q * a.K + i) * a.L;
        for (int sp = 0; sp < a.L; ++sp) sid[sp] = -1;
      }
    }
  }
}

// Tracing: counts of the work a step does, for roofline accounting.
__global__ void __launch_bounds__(256) k_trace_touch(const StepLaunch a, unsigned long long* cnt, uint32_t* mask) {
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int N = a.B * a.Wc;
  const int words = (a.V + 31) / 32;
  for (int b = wid; b < N; b += nw) {
    const int q = b / a.Wc, k = b - q * a.Wc;
    const BeamState bs = load_beam(a, q, k);
    if (bs.row == kDeadRow || bs.cum == -INFINITY) continue;
    unsigned long long F, chunks, ibytes;
    if (a.mode == kUncon) {
      F = (unsigned long long)a.V;
      chunks = 0;
      ibytes = 0;
      for (int w = lane; w < words; w += 32) {
        const int rem = a.V - 32 * w;
        atomicOr(&mask[w], rem >= 32 ? 0xFFFFFFFFu : ((1u << rem) - 1u));
      }
    } else {
      if (bs.row >= a.tab.rows) continue;
      const uint32_t rp = a.tab.rowptr[bs.row];
      F = a.tab.rowptr[bs.row + 1] - rp;
      if (a.tab.fmt == ZG_FMT_SPARSE) {
        for (uint32_t j = lane; j < F; j += 32) {
          const uint32_t t = a.tab.col[rp + j];
          if (t < (uint32_t)a.V) atomicOr(&mask[t >> 5], 1u << (t & 31));
        }
        chunks = (F + 31) / 32;
        ibytes = 8 + 2 * F;
      } else {
        for (int w = lane; w < words; w += 32) {
          const uint32_t bits = a.tab.bitmap[(size_t)bs.row * a.tab.words + w];
          if (bits) atomicOr(&mask[w], bits);
        }
        chunks = (unsigned long long)words;
        ibytes = 8 + 4ull * words;
      }
    }
    if (lane == 0) {
      atomicAdd(&cnt[0], 1ull);
      atomicAdd(&cnt[1], F);
      atomicAdd(&cnt[2], chunks);
      atomicAdd(&cnt[3], ibytes);
    }
  }
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <typename WT>
cudaError_t launch_sel_t(const StepLaunch& a, cudaStream_t st) {
  const int E = 16 / (int)sizeof(WT);
  const int nvec = a.d / E;
  const int vpl = (nvec + 31) / 32;
  const int64_t items = (int64_t)a.B * a.Wc * a.nch;
  if (items == 0) return cudaSuccess;
  const int64_t want = (items + 7) / 8;
  const int blocks = (int)std::min<int64_t>(want, (int64_t)sm_count() * 16);
  if (vpl <= 1)
    k_selective<WT, 1><<<blocks, 256, 0, st>>>(a);
  else if (vpl <= 2)
    k_selective<WT, 2><<<blocks, 256, 0, st>>>(a);
  else
    k_selective<WT, 4><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_selective(const StepLaunch& a, cudaStream_t st) {
  switch (a.w_dtype) {
    case ZG_F32:
      return launch_sel_t<float>(a, st);
    case ZG_BF16:
      return launch_sel_t<__nv_bfloat16>(a, st);
    default:
      return launch_sel_t<__half>(a, st);
  }
}

cudaError_t launch_gather_add(const StepLaunch& a, float* H, cudaStream_t st) {
  const int N = a.B * a.Wc;
  const int blocks = std::max(1, std::min((N + 7) / 8, sm_count() * 16));
  k_gather_add<<<blocks, 256, 0, st>>>(a, H);
  return cudaGetLastError();
}

cudaError_t launch_full_simt(const StepLaunch& a, const float* H, cudaStream_t st) {
  const int M = a.B * a.Wc;
  dim3 grid((a.V + 63) / 64, (M + 63) / 64);
  switch (a.w_dtype) {
    case ZG_F32:
      k_full_simt<float><<<grid, 256, 0, st>>>(H, static_cast<const float*>(a.W), a.Z, M, a.V, a.d, a.S);
      break;
    case ZG_BF16:
      k_full_simt<__nv_bfloat16><<<grid, 256, 0, st>>>(H, static_cast<const __nv_bfloat16*>(a.W), a.Z, M, a.V,
                                                       a.d, a.S);
      break;
    default:
      k_full_simt<__half><<<grid, 256, 0, st>>>(H, static_cast<const __half*>(a.W), a.Z, M, a.V, a.d, a.S);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_select(const StepLaunch& a, cudaStream_t st) {
  k_select<<<a.B, kSelThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_trace_touch(const StepLaunch& a, unsigned long long* counters, uint32_t* mask,
                               cudaStream_t st) {
  const int N = a.B * a.Wc;
  const int blocks = std::max(1, std::min((N + 7) / 8, sm_count() * 8));
  k_trace_touch<<<blocks, 256, 0, st>>>(a, counters, mask);
  return cudaGetLastError();
}

cudaError_t status_word(uint32_t** dev_ptr) { return cudaGetSymbolAddress((void**)dev_ptr, g_status); }

}  // namespace zg
