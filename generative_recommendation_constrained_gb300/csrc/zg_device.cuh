// Device building blocks shared by the per-step kernels and the cluster
// decode kernel: weight-row conversion, order-preserving score keys, the
// selective projection of one 32-slot chunk, and the CTA-level select.
//
// "ZeroGR: Filtering-First Constrained Decoding for Generative
// Recommendation" (paper-daily.com digest), section "Why computing fewer
// scores is not automatically faster": padded candidate slots (a slot
// depends only on its beam and rank, empty slots score -inf), weight rows
// read in place; section "Overall flow", stage 4: log-softmax over the
// legal tokens only, add to the cumulative log-probability, choose beams.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "zg_internal.h"

namespace zg {
namespace dev {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void flag(uint32_t* st, uint32_t bit) { atomicOr(st, bit); }

// Order-preserving map float -> uint32 (larger float -> larger key).  Every
// non-NaN float maps to a non-zero key, so 0 marks "no candidate".
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

// Accumulate the dot of 16 bytes of weights with the matching fp32 hidden
// lanes h[0..E) into the pair s (even elements into s.x, odd into s.y), one
// packed fp32x2 FMA per pair of elements; the caller adds s.x + s.y.
template <typename WT>
__device__ __forceinline__ void dot_pairs(const uint4& r, const float* h, float2& s) {
  float w[Vec<WT>::E];
  Vec<WT>::cvt(r, w);
#pragma unroll
  for (int e = 0; e < Vec<WT>::E; e += 2) s = __ffma2_rn(make_float2(w[e], w[e + 1]), make_float2(h[e], h[e + 1]), s);
}

// A weight row gathered in place: not kept in L1 (each SM meets a row only a
// few times), kept in L2 ahead of other lines (evict_last): every row of the
// step's codebook is gathered by many beams of the batch, and with normal
// priority the rows were evicted by one another inside a step whenever L2
// already held other data (about 9x the compulsory misses).
__device__ __forceinline__ uint4 ldg_wrow(const void* p) {
  uint4 r;
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
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

__device__ __forceinline__ float2 warp_lse(float2 acc) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    float2 other;
    other.x = __shfl_xor_sync(kFull, acc.x, o);
    other.y = __shfl_xor_sync(kFull, acc.y, o);
    acc = lse_combine(acc, other);
  }
  return acc;
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
    if (bs.cum == -INFINITY) bs.row = kDeadRow;
  }
  return bs;
}

// ---------------------------------------------------------------------------
// Selective projection of chunk c (slots 32c..32c+31) of beam k of request q
// by one warp.  The warp gathers h_b = h_parent + C_{s-1}[token] (fp32,
// lane-sliced in registers; written out once, by chunk 0, for the next step),
// reads each legal token's weight row in place with coalesced 16-byte loads,
// accumulates per-lane partial dots for the 32 rows and reduce-scatters them
// with 31 shuffles so lane j ends with z of slot j.  It writes the chunk's 32
// slots (-inf where empty) and its (max, sum exp) partial of the legal-only
// log-sum-exp.  `row`, `rp0`, `F` are the beam's index row, first entry and
// fan-out (checked by the caller).
// ---------------------------------------------------------------------------
// Destination of a chunk's scores inside the cluster: the rank-0 CTA's shared
// memory (reached through distributed shared memory), or none (global Z).
struct SlotSink {
  float* z;        // z of flat candidate start[k] + j, or null: the global slot buffer
  float2* part;    // chunk partials, by item istart[k] + c (also written to the global partials
                   // when z is null, for the selects that read them there)
  uint32_t* mask;  // chunk legal masks, by item
  int flat0;       // flat index of the chunk's first slot
  int item;        // item index of the chunk
  int cnt;         // slots of the beam (flat candidates it owns)
};

// The chunk's legal tokens: the lane mask and each lane's token (index
// column entries on a sparse step, a bitmap word on a dense one).
__device__ __forceinline__ uint32_t chunk_tokens(const StepLaunch& a, const BeamState& bs, uint32_t rp0, uint32_t F,
                                                 int c, int lane, int& t_lane) {
  const int j0 = c * kChunk;
  uint32_t vmask;
  t_lane = 0;
  if (a.mode == kSelDense) {
    vmask = a.tab.bitmap[(size_t)bs.row * a.tab.words + c];
    t_lane = j0 + lane;
    if (a.V - j0 < 32) vmask &= (1u << (a.V - j0)) - 1u;
  } else {
    const int nvalid = min(32, (int)F - j0);
    vmask = (nvalid >= 32) ? kFull : ((1u << nvalid) - 1u);
    if (lane < nvalid) t_lane = a.tab.col[rp0 + j0 + lane];
  }
  return vmask;
}

// The beam's hidden vector h_b = h_parent + C_{s-1}[token] (or the request
// vector at step 1, or the light decoder's output), lane-sliced: lane l holds
// elements (l + 32 r) * E .. + E.  write_h: also store it for the next step.
template <typename WT, int VPL>
__device__ __forceinline__ void load_hidden(const StepLaunch& a, int q, int k, const BeamState& bs, int lane,
                                            bool write_h, float (&h)[VPL][Vec<WT>::E]) {
  constexpr int E = Vec<WT>::E;
  const int d = a.d;
  const int nvec = d / E;
  const int b = q * a.Wc + k;
  const float* hp;
  const float* cr = nullptr;
  if (a.hpre) {  // the light decoder's hidden vector
    hp = a.hpre + (size_t)b * d;
  } else if (a.s == 1) {
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
          const float4 y = *reinterpret_cast<const float4*>(cr + v * E + e4);
          x.x += y.x;
          x.y += y.y;
          x.z += y.z;
          x.w += y.w;
        }
        h[r][e4] = x.x;
        h[r][e4 + 1] = x.y;
        h[r][e4 + 2] = x.z;
        h[r][e4 + 3] = x.w;
        if (write_h) *reinterpret_cast<float4*>(a.h_out + (size_t)b * d + v * E + e4) = x;
      }
    }
  }
}

// Scoring of chunk c of beam k once its tokens (vmask, t_lane) and hidden
// vector h are in registers.
template <typename WT, int VPL>
__device__ __forceinline__ void score_rows(const StepLaunch& a, int q, int k, int c, int lane, uint32_t vmask,
                                           int t_lane, const float (&h)[VPL][Vec<WT>::E],
                                           const SlotSink* sink = nullptr) {
  using VT = Vec<WT>;
  constexpr int E = VT::E;
  const int d = a.d;
  const int nvec = d / E;
  const int j0 = c * kChunk;
  if (((vmask >> lane) & 1u) && t_lane >= a.V) {
    flag(a.status, kStatusToken);
    vmask &= ~(1u << lane);
  }
  vmask = __ballot_sync(kFull, (vmask >> lane) & 1u);  // each lane vouches for its own slot

  float acc[32];
#pragma unroll
  for (int r = 0; r < 32; ++r) acc[r] = 0.f;
  const WT* Wm = static_cast<const WT*>(a.W);
  constexpr int GR = (VPL >= 4) ? 4 : 8;  // rows loaded together (16*VPL*GR bytes a lane)
  constexpr uint32_t GMASK = (1u << GR) - 1u;
#pragma unroll
  for (int g = 0; g < 32 / GR; ++g) {
    if (((vmask >> (GR * g)) & GMASK) == 0u) continue;
    uint4 raw[GR][VPL];
#pragma unroll
    for (int rr = 0; rr < GR; ++rr) {
      const int r = GR * g + rr;
      const int t = __shfl_sync(kFull, t_lane, r);
      const bool ok = (vmask >> r) & 1u;
      const WT* wrow = Wm + (size_t)t * d;
#pragma unroll
      for (int vv = 0; vv < VPL; ++vv) {
        const int v = lane + 32 * vv;
        raw[rr][vv] = (ok && v < nvec) ? ldg_wrow(wrow + v * E) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int rr = 0; rr < GR; ++rr) {
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int vv = 0; vv < VPL; ++vv) dot_pairs<WT>(raw[rr][vv], h[vv], s2);
      acc[GR * g + rr] = s2.x + s2.y;
    }
  }
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
  const float m = warp_max(z);
  const float e = valid ? expf(z - m) : 0.f;
  float ssum = warp_sum(e);
  ssum = __shfl_sync(kFull, ssum, 0);
  const float2 pc = make_float2(m, vmask ? ssum : 0.f);
  if (sink && sink->z) {
    if (j0 + lane < sink->cnt) sink->z[sink->flat0 + lane] = z;
  } else {
    a.Z[(size_t)q * a.zq + (size_t)k * a.S + j0 + lane] = z;
  }
  if (lane == 0) {
    if (sink) {
      sink->part[sink->item] = pc;
      sink->mask[sink->item] = vmask;
    }
    if (!sink || !sink->z) a.part[(size_t)q * a.pq + (size_t)k * a.nch + c] = pc;
  }
}

template <typename WT, int VPL>
__device__ __forceinline__ void score_chunk(const StepLaunch& a, int q, int k, const BeamState& bs, uint32_t rp0,
                                            uint32_t F, int c, int lane, const SlotSink* sink = nullptr) {
  // the chunk's legal tokens and the hidden vector are loaded together, then checked
  int t_lane;
  const uint32_t vmask = chunk_tokens(a, bs, rp0, F, c, lane, t_lane);
  float h[VPL][Vec<WT>::E];
  load_hidden<WT, VPL>(a, q, k, bs, lane, (c == 0) && a.h_out, h);
  score_rows<WT, VPL>(a, q, k, c, lane, vmask, t_lane, h, sink);
}

// ---------------------------------------------------------------------------
// Per-request beam table and select scratch (shared memory).
// ---------------------------------------------------------------------------
struct BeamTab {
  uint32_t row[ZG_MAX_BEAM];
  uint32_t rp[ZG_MAX_BEAM];
  int cnt[ZG_MAX_BEAM];        // candidate positions (slots) of the beam
  int nleg[ZG_MAX_BEAM];       // legal candidates of the beam
  int items[ZG_MAX_BEAM];      // 32-slot chunks to score (cluster kernel)
  float cum[ZG_MAX_BEAM];
  float lse[ZG_MAX_BEAM];
  int par[ZG_MAX_BEAM];
  int tok[ZG_MAX_BEAM];
  int start[ZG_MAX_BEAM + 1];  // flat candidate prefix
  int istart[ZG_MAX_BEAM + 1]; // chunk prefix
  int total, nlegal;
  // from the chunk partials (beam_lse_sel): the largest and the smallest
  // chunk-maximum key and the number of chunks holding a legal candidate
  uint32_t kceil, kfloor;
  int nne;
  // beam of every 32-slot chunk item, when the step has at most kItemMap
  // items (else items look their beam up in istart)
  static constexpr int kItemMap = 2048;
  int imap_ok;
  uint16_t ibeam[kItemMap];
};


template <int NW>
struct SelWorkT {
  alignas(16) uint32_t whist[NW][256];  // private radix histogram of each warp (or a histogram / list)
  unsigned long long win[ZG_MAX_BEAM];
  int warp_tot[32];
  uint32_t prefix, prefmask;
  int need, cnt_gt, cnt_eq, nwin;
  int all_eq;
};

// Legal-token bitmap row of beam k of request q on a dense-slot full step:
// the index row's bitmap, or the beam's own expanded row (mask_by_beam).
__device__ __forceinline__ const uint32_t* legal_bits(const StepLaunch& a, const BeamTab& bt, int q, int k) {
  return a.tab.bitmap + (a.mask_by_beam ? (size_t)q * a.Wc + k : (size_t)bt.row[k]) * a.tab.words;
}

// largest k with arr[k] <= c (arr ascending, arr[0] = 0)
__device__ __forceinline__ int upper_find(const int* arr, int n, int c) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (arr[mid] <= c)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Beam of chunk item i (items are numbered beam by beam: istart).
__device__ __forceinline__ int item_beam(const BeamTab& bt, int Wc, int i) {
  return bt.imap_ok ? (int)bt.ibeam[i] : upper_find(bt.istart, Wc, i);
}

// Fill the beam table of request q entering step s (threads k < Wc), then
// the flat-candidate and chunk prefixes.  Returns after __syncthreads.
template <int NT>
__device__ void build_beam_table(const StepLaunch& a, int q, BeamTab& bt) {
  const int tid = threadIdx.x;
  const bool constrained = (a.mode != kUncon);
  const bool sparse_slots = (a.mode == kSelSparse || a.mode == kFullSparse);
  for (int k = tid; k < a.Wc; k += NT) {
    const BeamState bs = load_beam(a, q, k);
    bool dead = (bs.row == kDeadRow);
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
    bt.row[k] = bs.row;
    bt.rp[k] = rp;
    bt.cum[k] = bs.cum;
    bt.par[k] = bs.par;
    bt.tok[k] = bs.tok;
    bt.cnt[k] = dead ? 0 : (sparse_slots ? (int)F : a.V);
    bt.nleg[k] = dead ? 0 : (int)F;
    bt.items[k] = dead ? 0 : (a.mode == kSelSparse ? (int)((F + kChunk - 1) / kChunk) : a.nch);
    bt.lse[k] = 0.f;
  }
  __syncthreads();
  if (tid < 32) {
    // warp prefix sums over Wc <= 512 beams, 16 consecutive beams a lane
    const int lane = tid;
    const int per = (a.Wc + 31) / 32;
    const int k0 = lane * per;
    int sc = 0, si = 0, sl = 0;
    for (int k = k0; k < min(k0 + per, a.Wc); ++k) {
      sc += bt.cnt[k];
      si += bt.items[k];
      sl += bt.nleg[k];
    }
    int ic = sc, ii = si, il = sl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yc = __shfl_up_sync(kFull, ic, o);
      const int yi = __shfl_up_sync(kFull, ii, o);
      const int yl = __shfl_up_sync(kFull, il, o);
      if (lane >= o) {
        ic += yc;
        ii += yi;
        il += yl;
      }
    }
    int rc = ic - sc, ri = ii - si;
    for (int k = k0; k < min(k0 + per, a.Wc); ++k) {
      bt.start[k] = rc;
      bt.istart[k] = ri;
      rc += bt.cnt[k];
      ri += bt.items[k];
    }
    if (lane == 31) {
      bt.start[a.Wc] = ic;
      bt.istart[a.Wc] = ii;
      bt.total = ic;
      bt.nlegal = il;
      bt.kceil = 0u;
      bt.kfloor = 0xFFFFFFFFu;
      bt.nne = 0;
      bt.imap_ok = (ii <= BeamTab::kItemMap) ? 1 : 0;
    }
  }
  __syncthreads();
  // chunk item -> beam, once per step, for every pass that walks items
  if (bt.imap_ok) {
    const int nitems = bt.istart[a.Wc];
    for (int i = tid; i < nitems; i += NT) bt.ibeam[i] = (uint16_t)upper_find(bt.istart, a.Wc, i);
    __syncthreads();
  }
}

// Log-sum-exp of every live beam from its chunk partials (m_c, s_c): lse =
// M + log(sum_c s_c exp(m_c - M)), M = max_c m_c, over the legal tokens
// (filter-first), or over every token from part_all (score-first).  Eight lanes a
// beam; each 8-lane group of the CTA takes up to two beams at once (their
// first partials loaded together and kept for the second pass), so every
// group has a beam before any has two; width-8 shuffle reductions.
// Partials come from shared memory by item (psm) or from the global partial
// buffer (psm == nullptr).  Also folds into bt.kceil / bt.kfloor / bt.nne the
// keys of each beam's best and weakest non-empty chunk maximum and its
// number of non-empty chunks.
template <int NT>
__device__ void beam_lse_sel(const StepLaunch& a, int q, BeamTab& bt, const float2* psm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  static_assert(NT >= 256, "eight warps at least");
  if (a.Wc <= 8) {
    // few beams (the first step's root beam): all 32 lanes of a warp on one
    // beam, width-32 reductions (the same threshold in every kernel keeps
    // the fused and stand-alone selects bit-identical)
    const int k = warp;
    const bool live = (k < a.Wc) && bt.cnt[k] > 0;
    if (!live) return;
    const int n = bt.items[k];
    const size_t go = (size_t)q * a.pq + (size_t)k * a.nch;
    const float2* pp = psm ? psm + bt.istart[k] : a.part + go;
    const bool all_v = (a.part_all != nullptr) && !psm;
    const float2* pa = all_v ? a.part_all + go : pp;
    float m = -INFINITY, mn = INFINITY, ma = -INFINITY;
    int ne = 0;
    for (int c = lane; c < n; c += 32) {
      const float2 p = pp[c];
      m = fmaxf(m, p.x);
      if (p.y > 0.f) {
        mn = fminf(mn, p.x);
        ++ne;
      }
      if (all_v) ma = fmaxf(ma, pa[c].x);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
      ne += __shfl_xor_sync(kFull, ne, o);
      ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, o));
    }
    if (!all_v) ma = m;
    float sum = 0.f;
    for (int c = lane; c < n; c += 32) {
      const float2 p = pa[c];
      if (p.y > 0.f) sum += p.y * expf(p.x - ma);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (lane == 0) {
      const float lse = ma + logf(sum);
      bt.lse[k] = lse;
      if (ne > 0) {
        atomicMax(&bt.kceil, f2ord(bt.cum[k] + (m - lse)));
        atomicMin(&bt.kfloor, f2ord(bt.cum[k] + (mn - lse)));
        atomicAdd(&bt.nne, ne);
      }
    }
    return;
  }
  const int sub = lane >> 3, sl = lane & 7;
  constexpr int NG = (NT / 32) * 4;  // 8-lane groups of the CTA
  const int g = warp * 4 + sub;
  for (int k0 = 0; k0 < a.Wc; k0 += 2 * NG) {
    int kb[2], n[2];
    const float2* pp[2];
    const float2* pa[2];
    float2 p0[2], a0[2];
    const bool all_v = (a.part_all != nullptr) && !psm;  // score-first: normaliser over the codebook
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int k = k0 + h * NG + g;  // every group takes a beam before any takes a second
      const bool live = (k < a.Wc) && bt.cnt[k] > 0;
      kb[h] = k;
      n[h] = live ? bt.items[k] : 0;
      const size_t go = (size_t)q * a.pq + (size_t)(live ? k : 0) * a.nch;
      pp[h] = psm ? psm + (live ? bt.istart[k] : 0) : a.part + go;
      pa[h] = all_v ? a.part_all + go : pp[h];
      p0[h] = (sl < n[h]) ? pp[h][sl] : make_float2(-INFINITY, 0.f);
      a0[h] = all_v ? ((sl < n[h]) ? pa[h][sl] : make_float2(-INFINITY, 0.f)) : p0[h];
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float m = p0[h].x, mn = (p0[h].y > 0.f) ? p0[h].x : INFINITY;
      int ne = (p0[h].y > 0.f) ? 1 : 0;  // a chunk with a legal candidate has sum >= 1
      // a beam with many chunks: four partials a lane in flight at a time
      for (int c0 = sl + 8; c0 < n[h]; c0 += 32) {
        float2 pv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) pv[u] = (c0 + 8 * u < n[h]) ? pp[h][c0 + 8 * u] : make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          m = fmaxf(m, pv[u].x);
          if (pv[u].y > 0.f) {
            mn = fminf(mn, pv[u].x);
            ++ne;
          }
        }
      }
      float ma = a0[h].x;  // maximum of the normalised set
      if (all_v)
        for (int c = sl + 8; c < n[h]; c += 8) ma = fmaxf(ma, pa[h][c].x);
#pragma unroll
      for (int o = 4; o; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
        ne += __shfl_xor_sync(kFull, ne, o);
        ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, o));
      }
      if (!all_v) ma = m;
      float sum = (a0[h].y > 0.f) ? a0[h].y * expf(a0[h].x - ma) : 0.f;
      for (int c0 = sl + 8; c0 < n[h]; c0 += 32) {
        float2 pv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) pv[u] = (c0 + 8 * u < n[h]) ? pa[h][c0 + 8 * u] : make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (pv[u].y > 0.f) sum += pv[u].y * expf(pv[u].x - ma);
      }
#pragma unroll
      for (int o = 4; o; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
      const int k = kb[h];
      // keys of the beam's best and of its weakest chunk maximum, as the
      // select computes them; folded over the warp's four beams first, so one
      // lane a warp updates the shared range
      uint32_t kc = 0u, kf = 0xFFFFFFFFu;
      int nn = 0;
      if (n[h] > 0) {
        const float lse = ma + logf(sum);
        if (sl == 0) bt.lse[k] = lse;
        if (ne > 0) {
          kc = f2ord(bt.cum[k] + (m - lse));
          kf = f2ord(bt.cum[k] + (mn - lse));
          nn = ne;
        }
      }
#pragma unroll
      for (int o = 8; o < 32; o <<= 1) {
        kc = max(kc, __shfl_xor_sync(kFull, kc, o));
        kf = min(kf, __shfl_xor_sync(kFull, kf, o));
        nn += __shfl_xor_sync(kFull, nn, o);
      }
      if (lane == 0 && nn > 0) {
        atomicMax(&bt.kceil, kc);
        atomicMin(&bt.kfloor, kf);
        atomicAdd(&bt.nne, nn);
      }
    }
  }
}

// Legal-only log-sum-exp of every live beam (one warp per beam): from the
// selective chunk partials, or by two passes over the full scores.
// Representative tiles of a step for the filtered select: rt tiles of tw
// slots (a multiple of 32) a beam, at most half of a cap-entry buffer.
__host__ __device__ __forceinline__ void tile_layout(int Wc, int S, int cap, int* rt, int* tw) {
  int max_rt = (cap / 2) / (Wc > 0 ? Wc : 1);
  if (max_rt < 1) max_rt = 1;
  int r = (S + 31) / 32;
  if (r > max_rt) r = max_rt;
  if (r < 1) r = 1;
  *rt = r;
  *tw = ((S + r - 1) / r + 31) & ~31;
}

// Legal-only log-sum-exp of every live beam (one warp per beam): from the
// selective chunk partials, or by two passes over the full scores.  For the
// full scores, when rep_z is given, the maximum legal z of every tw-slot
// tile of beam k is also stored (as float bits) at rep_z[k * rt + t]
// (-inf for a tile without legal tokens).
template <int NT>
__device__ void beam_lse(const StepLaunch& a, int q, BeamTab& bt, uint32_t* rep_z = nullptr, int rt = 0,
                         int tw = 256) {
  if (a.part) {  // selective steps, and full steps whose epilogue wrote chunk partials
    beam_lse_sel<NT>(a, q, bt, nullptr);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int k = warp; k < a.Wc; k += NT / 32) {
    if (bt.cnt[k] == 0) continue;
    const int n = bt.cnt[k];
    const size_t zb = (size_t)q * a.zq + (size_t)k * a.S;
    auto zval = [&](int j) -> float {
      if (a.mode == kFullSparse) return a.Z[zb + a.tab.col[bt.rp[k] + j]];
      if (a.mode == kFullDense)
        return ((legal_bits(a, bt, q, k)[j >> 5] >> (j & 31)) & 1u) ? a.Z[zb + j] : -INFINITY;
      return a.Z[zb + j];
    };
    float m = -INFINITY;
    for (int t = 0; t * tw < n; ++t) {
      float tm = -INFINITY;
      for (int i = 0; i < tw; i += 32) {
        const int j = t * tw + i + lane;
        if (j < n) tm = fmaxf(tm, zval(j));
      }
      tm = warp_max(tm);
      m = fmaxf(m, tm);
      if (rep_z && lane == 0) rep_z[k * rt + t] = __float_as_uint(tm);
    }
    float sm = 0.f;
    for (int j = lane; j < n; j += 32) {
      const float z = zval(j);
      if (z != -INFINITY) sm += expf(z - m);
    }
    sm = warp_sum(sm);
    if (lane == 0) bt.lse[k] = m + logf(sm);
  }
}

// Key of flat candidate c (0 = illegal slot).
__device__ __forceinline__ uint32_t cand_key_kj(const StepLaunch& a, const BeamTab& bt, int q, int k, int j);
__device__ __forceinline__ uint32_t cand_key(const StepLaunch& a, const BeamTab& bt, int q, int c) {
  const int k = upper_find(bt.start, a.Wc, c);
  return cand_key_kj(a, bt, q, k, c - bt.start[k]);
}
// Key of slot j of beam k (0 = illegal slot).
__device__ __forceinline__ uint32_t cand_key_kj(const StepLaunch& a, const BeamTab& bt, int q, int k, int j) {
  const size_t zb = (size_t)q * a.zq + (size_t)k * a.S;
  float z;
  switch (a.mode) {
    case kSelSparse:
    case kUncon:
      z = a.Z[zb + j];
      break;
    case kFullSparse:
      z = a.Z[zb + a.tab.col[bt.rp[k] + j]];
      break;
    default:  // kSelDense, kFullDense
      if (!((legal_bits(a, bt, q, k)[j >> 5] >> (j & 31)) & 1u)) return 0u;
      z = a.Z[zb + j];
      break;
  }
  return f2ord(bt.cum[k] + (z - bt.lse[k]));
}

// Keys of U candidates (slot jj[u] of beam kk[u]; jj[u] < 0: none, key 0),
// with the step format's branch taken once outside the per-candidate loops
// so that the U loads of each kind are issued together.
template <int U>
__device__ __forceinline__ void cand_keys_batch(const StepLaunch& a, const BeamTab& bt, int q, const int* kk,
                                                const int* jj, uint32_t* key) {
  float z[U];
  bool ok[U];
  if (a.mode == kSelSparse || a.mode == kUncon) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      ok[u] = jj[u] >= 0;
      z[u] = ok[u] ? a.Z[(size_t)q * a.zq + (size_t)kk[u] * a.S + jj[u]] : 0.f;
    }
  } else if (a.mode == kFullSparse) {
    uint32_t c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      ok[u] = jj[u] >= 0;
      c[u] = ok[u] ? a.tab.col[bt.rp[kk[u]] + jj[u]] : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) z[u] = ok[u] ? a.Z[(size_t)q * a.zq + (size_t)kk[u] * a.S + c[u]] : 0.f;
  } else {  // kSelDense, kFullDense: the legal word and the slot together
    uint32_t w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool any = jj[u] >= 0;
      w[u] = any ? legal_bits(a, bt, q, kk[u])[jj[u] >> 5] : 0u;
      z[u] = any ? a.Z[(size_t)q * a.zq + (size_t)kk[u] * a.S + jj[u]] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) ok[u] = jj[u] >= 0 && ((w[u] >> (jj[u] & 31)) & 1u);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) key[u] = ok[u] ? f2ord(bt.cum[kk[u]] + (z[u] - bt.lse[kk[u]])) : 0u;
}

// Stage the keys of every candidate in shared memory (eight independent
// candidates a thread in flight).
template <int NT>
__device__ void stage_keys_global(const StepLaunch& a, int q, const BeamTab& bt, uint32_t* keys) {
  constexpr int U = 8;
  const int total = bt.total;
  for (int c0 = threadIdx.x; c0 < total; c0 += U * NT) {
    int kk[U], jj[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * NT;
      kk[u] = 0;
      jj[u] = -1;
      if (c < total) {
        kk[u] = upper_find(bt.start, a.Wc, c);
        jj[u] = c - bt.start[kk[u]];
      }
    }
    uint32_t key[U];
    cand_keys_batch<U>(a, bt, q, kk, jj, key);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (c0 + u * NT < total) keys[c0 + u * NT] = key[u];
  }
}

// Descending bitonic sort of up to 32 values held one a lane (warp-wide).
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long o = __shfl_xor_sync(kFull, v, j);
      const bool desc = (lane & k) == 0;
      const bool lower = (lane & j) == 0;
      const bool take_max = (lower == desc);
      v = take_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Descending bitonic sort of list[0, P) in shared memory by the CTA (P a
// power of two).  Entry block [32w', 32w' + 32) is always handled by one
// warp, so a stage whose pairs stay inside a block, and whose successor does
// too, needs only that warp's barrier.  Returns after __syncthreads.
template <int NT>
__device__ void cta_bitonic_desc(unsigned long long* list, int P) {
  const int tid = threadIdx.x;
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += NT) {
        const int jx = i ^ stride;
        if (jx > i) {
          const bool desc = ((i & size) == 0);
          const unsigned long long x = list[i], y = list[jx];
          if (desc ? (x < y) : (x > y)) {
            list[i] = y;
            list[jx] = x;
          }
        }
      }
      const int next = (stride > 1) ? (stride >> 1) : size;  // stride of the following stage
      if (stride >= 32 || next >= 32)
        __syncthreads();
      else
        __syncwarp();
    }
  }
  __syncthreads();
}

// k-th largest (1 <= kth <= n) of the non-zero keys[0..n) in shared memory:
// returns T with count(> T) < kth <= count(>= T).  8-bit radix passes with
// per-warp histograms.
template <int NT, typename SW>
__device__ uint32_t cta_kth(const uint32_t* keys, int n, int kth, SW& sw) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    sw.prefix = 0;
    sw.prefmask = 0;
    sw.need = kth;
    sw.cnt_gt = 0;
  }
  __syncthreads();
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < NW * 256; i += NT) (&sw.whist[0][0])[i] = 0u;
    __syncthreads();
    const uint32_t pm = sw.prefmask, pv = sw.prefix;
    for (int c = tid; c < n; c += NT) {
      const uint32_t key = keys[c];
      if (key && (key & pm) == pv) atomicAdd(&sw.whist[warp][(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      const int hi = 256 - 8 * lane;
      uint32_t cnt8[8];
      uint32_t mine = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t h = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) h += sw.whist[w][hi - 1 - i];
        cnt8[i] = h;
        mine += h;
      }
      uint32_t incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - mine;
      const uint32_t target = (uint32_t)(sw.need - sw.cnt_gt);
      const bool here = (excl < target) && (incl >= target);
      const unsigned who = __ballot_sync(kFull, here);
      if (here && lane == __ffs(who) - 1) {
        uint32_t run = excl, bin = 0;
        bool found = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const bool hit = !found && (run + cnt8[i] >= target);
          bin = hit ? (uint32_t)(hi - 1 - i) : bin;
          found = found || hit;
          run += found ? 0u : cnt8[i];
        }
        sw.cnt_gt += (int)run;
        sw.prefix |= bin << shift;
        sw.prefmask |= 255u << shift;
      }
    }
    __syncthreads();
  }
  return sw.prefix;
}

// Select when the request's candidates do not fit in shared memory.  rep[0,
// nrep) holds, for tile t (tw slots) of beam k at k*rt + t (or, with rt = 0,
// for the i-th scored 32-slot chunk of the request), the key of the tile's
// best candidate; the keep-th largest of them is a lower bound on the
// keep-th largest candidate, so only tiles whose best clears it are read from
// the global slot buffer, and their candidates at or above it are kept as
// (key << 32 | ~flat) in buf after rep; they are bitonic-sorted descending
// and the first keep become the winners.  Returns -1 (nothing written) when
// more candidates pass than the space holds; the caller then runs the full
// radix select.
template <int NT, typename SW>
__device__ int cta_select_filtered(const StepLaunch& a, int q, BeamTab& bt, SW& sw, uint32_t* buf, int cap,
                                   int nrep, int rt, int tw) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int keep_n = min(a.keep, bt.nlegal);
  if (keep_n == 0) return 0;
  __syncthreads();
  const uint32_t tlb = (nrep >= keep_n) ? cta_kth<NT>(buf, nrep, keep_n, sw) : 1u;
  const int off = (nrep + 1) & ~1;  // u64 alignment
  unsigned long long* list = reinterpret_cast<unsigned long long*>(buf + off);
  int lcap = 1;
  while (lcap * 2 <= (cap - off) / 2) lcap *= 2;  // power of two, for the sort
  if (tid == 0) sw.nwin = 0;
  __syncthreads();
  // a tile whose best candidate is below the bound holds no winner: only the
  // tiles at or above it are read (one warp a tile)
  for (int i = warp; i < nrep; i += NT / 32) {
    if (buf[i] < tlb || buf[i] == 0u) continue;
    int k, j0;
    if (rt > 0) {
      k = i / rt;
      j0 = (i - k * rt) * tw;
    } else {  // one 32-slot chunk a representative, numbered by the chunk prefix
      k = item_beam(bt, a.Wc, i);
      j0 = (i - bt.istart[k]) * kChunk;
    }
    const int j1 = min(j0 + tw, bt.cnt[k]);
    for (int j = j0 + lane; j < j1; j += 32) {
      const uint32_t key = cand_key_kj(a, bt, q, k, j);
      if (key && key >= tlb) {
        const int pos = atomicAdd(&sw.nwin, 1);
        if (pos < lcap)
          list[pos] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)(bt.start[k] + j));
      }
    }
  }
  __syncthreads();
  const int nl = sw.nwin;
  if (nl > lcap || nl < keep_n) return -1;
  int P = 1;
  while (P < nl) P <<= 1;
  for (int i = nl + tid; i < P; i += NT) list[i] = 0ull;
  __syncthreads();
  cta_bitonic_desc<NT>(list, P);
  for (int i = tid; i < keep_n; i += NT) sw.win[i] = list[i];
  __syncthreads();
  return keep_n;
}

// Keys of the tile representatives for cta_select_filtered, in place in
// rep[k * rt + t]: from the tile maxima of full scores stored by beam_lse
// (float bits), or, for selective steps, from the maxima of each beam's
// chunk partials, tw/32 chunks a tile.  Returns the number of
// representatives (Wc * rt).
template <int NT>
__device__ int tile_rep_keys(const StepLaunch& a, int q, const BeamTab& bt, uint32_t* rep, int rt, int tw) {
  const bool sel = (a.part != nullptr);  // chunk partials exist
  const int n = a.Wc * rt;
  const int cpt = tw / kChunk;  // chunks a tile
  for (int i = threadIdx.x; i < n; i += NT) {
    const int k = i / rt, t = i - k * rt;
    uint32_t key = 0u;
    if (bt.cnt[k] > 0 && t * tw < bt.cnt[k]) {
      float m;
      if (sel) {
        const float2* pp = a.part + (size_t)q * a.pq + (size_t)k * a.nch;
        m = -INFINITY;
        const int c1 = min(bt.items[k], cpt * (t + 1));
        for (int c = cpt * t; c < c1; ++c) m = fmaxf(m, pp[c].x);
      } else {
        m = __uint_as_float(rep[i]);
      }
      if (m != -INFINITY) key = f2ord(bt.cum[k] + (m - bt.lse[k]));
    }
    rep[i] = key;
  }
  __syncthreads();
  return n;
}

// Keys of the scored chunks of a step with chunk partials as representatives
// for cta_select_filtered (rt = 0): rep[i] for the i-th chunk of the request
// in beam order, from the chunk's partial maximum.  Returns the chunk count.
template <int NT>
__device__ int chunk_rep_keys(const StepLaunch& a, int q, const BeamTab& bt, uint32_t* rep) {
  const int n = bt.istart[a.Wc];
  for (int i = threadIdx.x; i < n; i += NT) {
    const int k = item_beam(bt, a.Wc, i);
    const float m = a.part[(size_t)q * a.pq + (size_t)k * a.nch + (i - bt.istart[k])].x;
    rep[i] = (m != -INFINITY) ? f2ord(bt.cum[k] + (m - bt.lse[k])) : 0u;
  }
  __syncthreads();
  return n;
}

// Where cta_select finds the candidates' keys.
enum KeySrc { kKeysStaged = 0, kZStaged = 1, kGlobal = 2 };

// ---------------------------------------------------------------------------
// CTA-level select of the keep best legal candidates of request q.
//   kKeysStaged: keys[] holds every candidate's key;
//   kZStaged:    keys[] holds every candidate's z (-inf for an empty slot);
//                the first radix pass turns them into keys in place;
//   kGlobal:     keys are recomputed from the global slot buffer each pass.
// 8-bit radix passes from the top byte narrow the threshold key (stopping as
// soon as the threshold bin holds exactly the remainder); each warp counts
// into a private histogram.  Winners above the threshold are collected,
// threshold ties go to the lowest flat slot indices, and the winners are
// sorted by (score desc, flat asc).  Leaves sw.win[0..n) sorted; returns
// n = min(keep, legal candidates).
// ---------------------------------------------------------------------------
template <int NT, typename SW>
__device__ int cta_select(const StepLaunch& a, int q, BeamTab& bt, SW& sw, uint32_t* keys, KeySrc src) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int total = bt.total;
  const int keep_n = min(a.keep, bt.nlegal);
  if (tid == 0) {
    sw.nwin = 0;
    sw.prefix = 0;
    sw.prefmask = 0;
    sw.need = keep_n;
    sw.cnt_gt = 0;
    sw.cnt_eq = bt.nlegal;
    sw.all_eq = (keep_n == bt.nlegal) ? 1 : 0;
  }
  __syncthreads();
  if (keep_n == 0) return 0;
  bool z_pending = (src == kZStaged);
  if (sw.all_eq && z_pending) {
    // everything is kept: keys are still needed for the order
    for (int c = tid; c < total; c += NT) {
      const int k = upper_find(bt.start, a.Wc, c);
      const float z = __uint_as_float(keys[c]);
      keys[c] = (z == -INFINITY) ? 0u : f2ord(bt.cum[k] + (z - bt.lse[k]));
    }
    z_pending = false;
  }
  for (int shift = 24; shift >= 0 && !sw.all_eq; shift -= 8) {
    for (int i = tid; i < NW * 256; i += NT) (&sw.whist[0][0])[i] = 0u;
    __syncthreads();
    const uint32_t pm = sw.prefmask, pv = sw.prefix;
    uint32_t* wh = sw.whist[warp];
    if (z_pending) {
      int c = tid, k = (c < total) ? upper_find(bt.start, a.Wc, c) : 0;
      for (; c < total; c += NT) {
        while (bt.start[k + 1] <= c) ++k;
        const float z = __uint_as_float(keys[c]);
        const uint32_t key = (z == -INFINITY) ? 0u : f2ord(bt.cum[k] + (z - bt.lse[k]));
        keys[c] = key;
        if (key) atomicAdd(&wh[key >> 24], 1u);
      }
    } else {
      for (int c = tid; c < total; c += NT) {
        const uint32_t key = (src == kGlobal) ? cand_key(a, bt, q, c) : keys[c];
        if (key && (key & pm) == pv) atomicAdd(&wh[(key >> shift) & 255u], 1u);
      }
    }
    z_pending = false;
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins [248 - 8l, 256 - 8l), scanned from the top
      const int hi = 256 - 8 * lane;
      uint32_t cnt8[8];
      uint32_t mine = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t h = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) h += sw.whist[w][hi - 1 - i];
        cnt8[i] = h;
        mine += h;
      }
      uint32_t incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - mine;
      const uint32_t target = (uint32_t)(sw.need - sw.cnt_gt);
      const bool here = (excl < target) && (incl >= target);
      const unsigned who = __ballot_sync(kFull, here);
      if (here && lane == __ffs(who) - 1) {
        uint32_t run = excl, bin = 0, bc = 0;
        bool found = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t hc = cnt8[i];
          const bool hit = !found && (run + hc >= target);
          bin = hit ? (uint32_t)(hi - 1 - i) : bin;
          bc = hit ? hc : bc;
          found = found || hit;
          run += found ? 0u : hc;
        }
        sw.cnt_gt += (int)run;
        sw.prefix |= bin << shift;
        sw.prefmask |= 255u << shift;
        sw.cnt_eq = (int)bc;
        if ((int)bc == sw.need - sw.cnt_gt) sw.all_eq = 1;
      }
    }
    __syncthreads();
  }
  const uint32_t pm = sw.prefmask, pv = sw.prefix;
  const int need_eq = sw.need - sw.cnt_gt;
  const bool all_eq = sw.all_eq;
  for (int c = tid; c < total; c += NT) {
    const uint32_t key = (src == kGlobal) ? cand_key(a, bt, q, c) : keys[c];
    if (!key) continue;
    const uint32_t mk = key & pm;
    if (mk > pv || (all_eq && mk == pv)) {
      const int slot = atomicAdd(&sw.nwin, 1);
      if (slot < ZG_MAX_BEAM) sw.win[slot] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)c);
    }
  }
  __syncthreads();
  if (!all_eq) {
    // ties at the exact threshold key: the need_eq lowest flat indices
    int base = 0;
    for (int c0 = 0; c0 < total && base < need_eq; c0 += NT) {
      const int c = c0 + tid;
      uint32_t key = 0;
      if (c < total) key = (src == kGlobal) ? cand_key(a, bt, q, c) : keys[c];
      const bool f = key && key == pv;
      const unsigned bal = __ballot_sync(kFull, f);
      if (lane == 0) sw.warp_tot[warp] = __popc(bal);
      __syncthreads();
      int before = base;
      for (int w = 0; w < warp; ++w) before += sw.warp_tot[w];
      before += __popc(bal & ((1u << lane) - 1u));
      if (f && before < need_eq) {
        const int slot = atomicAdd(&sw.nwin, 1);
        if (slot < ZG_MAX_BEAM) sw.win[slot] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)c);
      }
      int tile = 0;
      for (int w = 0; w < NW; ++w) tile += sw.warp_tot[w];
      __syncthreads();
      base += tile;
    }
  }
  __syncthreads();
  if (keep_n <= 32) {
    if (warp == 0) {
      const unsigned long long v = warp_sort_desc(lane < keep_n ? sw.win[lane] : 0ull, lane);
      if (lane < keep_n) sw.win[lane] = v;
    }
    __syncthreads();
    return keep_n;
  }
  int P = 1;
  while (P < keep_n) P <<= 1;
  for (int i = keep_n + tid; i < P; i += NT) sw.win[i] = 0ull;
  __syncthreads();
  cta_bitonic_desc<NT>(sw.win, P);
  return keep_n;
}

// ---------------------------------------------------------------------------
// Histogram-cut selects.  Keys are cut by 2048 bins over a key range [lo, hi]
// (bin = min((key - lo) >> sh, 2047), sh the smallest shift that maps hi -
// lo below 2048): the bin where the count from the top reaches the target
// bounds the winners from below, and every key outside that bin and the bins
// above it is out.  The bin map is monotone, so the cut is exact.
// ---------------------------------------------------------------------------
constexpr int kBins = 2048;

__device__ __forceinline__ int bin_shift(uint32_t lo, uint32_t hi) {
  const uint32_t R = hi - lo;
  return (R < (uint32_t)kBins) ? 0 : (32 - __clz(R) - 11);
}
__device__ __forceinline__ uint32_t bin_of(uint32_t key, uint32_t lo, int sh) {
  return min((key - lo) >> sh, (uint32_t)(kBins - 1));
}

// Cut of a complete histogram (every thread past the barrier that completed
// it): the bin b where the count of the bins above stays below target and
// with b reaches it goes to sw.prefix, the count above to sw.cnt_gt, the
// count in b to sw.cnt_eq, and sw.nwin is zeroed.  Returns the histogram's
// total (the same in every thread; sw is not written when it is below
// target).  Thread t scans bins [top - PER, top), top = NB - PER * t, from
// the top.  On return every thread may overwrite the histogram.
template <int NT, typename SW, int NB = kBins>
__device__ uint32_t hist_cut(const uint32_t* hist, SW& sw, uint32_t target) {
  constexpr int NW = NT / 32;
  constexpr int PER = NB / NT;
  static_assert(PER >= 1 && NB % NT == 0, "bins a thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int top = NB - PER * tid;
  uint32_t cnt[PER];
  if constexpr (PER % 4 == 0) {
#pragma unroll
    for (int i = 0; i < PER; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(&hist[top - 4 - i]);
      cnt[i] = v.w;
      cnt[i + 1] = v.z;
      cnt[i + 2] = v.y;
      cnt[i + 3] = v.x;
    }
  } else {
#pragma unroll
    for (int i = 0; i < PER; ++i) cnt[i] = hist[top - 1 - i];
  }
  uint32_t mine = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) mine += cnt[i];
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sw.warp_tot[warp] = (int)incl;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t t = (uint32_t)sw.warp_tot[w];
    before += (w < warp) ? t : 0u;
    all += t;
  }
  const uint32_t excl = before + incl - mine;
  if (all >= target && excl < target && excl + mine >= target) {
    uint32_t run = excl;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (run + cnt[i] >= target) {
        sw.prefix = (uint32_t)(top - 1 - i);
        sw.cnt_gt = (int)run;
        sw.cnt_eq = (int)cnt[i];
        break;
      }
      run += cnt[i];
    }
    sw.nwin = 0;
  }
  __syncthreads();
  return all;
}

// Append (key << 32 | ~flat) of the lanes with f set to list (warp-wide).
__device__ __forceinline__ void warp_append(unsigned long long* list, int lcap, int& nwin, bool f, uint32_t key,
                                            int flat, int lane) {
  const unsigned bal = __ballot_sync(kFull, f);
  if (!bal) return;
  int pos = 0;
  if (lane == 0) pos = atomicAdd(&nwin, __popc(bal));
  pos = __shfl_sync(kFull, pos, 0) + __popc(bal & ((1u << lane) - 1u));
  if (f && pos < lcap) list[pos] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)flat);
}

// The keep_n best of nl distinct list entries, in descending order, into
// sw.win: a warp sort up to 32 entries, else every entry goes to the slot
// given by the number of entries above it.  Returns after __syncthreads.
template <int NT, typename SW>
__device__ void place_winners(const unsigned long long* list, int nl, int keep_n, SW& sw) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (nl <= 32) {
    if (warp == 0) {
      const unsigned long long v = warp_sort_desc(lane < nl ? list[lane] : 0ull, lane);
      if (lane < keep_n) sw.win[lane] = v;
    }
  } else if (2 * nl <= NT) {
    // two threads an entry, each counting over half of the list
    const int i = tid >> 1, half = tid & 1;
    const bool act = i < nl;
    const unsigned long long x = act ? list[i] : 0ull;
    int r = 0;
    if (act) {
      const int j0 = half ? (nl >> 1) : 0, j1 = half ? nl : (nl >> 1);
      for (int j = j0; j < j1; ++j) r += (list[j] > x);
    }
    r += __shfl_xor_sync(kFull, r, 1);
    if (act && !half && r < keep_n) sw.win[r] = x;
  } else if (nl <= NT) {
    if (tid < nl) {
      const unsigned long long x = list[tid];
      int r = 0;
      for (int j = 0; j < nl; ++j) r += (list[j] > x);
      if (r < keep_n) sw.win[r] = x;
    }
  } else {
    for (int i0 = tid; i0 < nl; i0 += 2 * NT) {
      const int i1 = i0 + NT;
      const unsigned long long x0 = list[i0], x1 = (i1 < nl) ? list[i1] : ~0ull;
      int r0 = 0, r1 = 0;
      for (int j = 0; j < nl; ++j) {
        const unsigned long long y = list[j];
        r0 += (y > x0);
        r1 += (y > x1);
      }
      if (r0 < keep_n) sw.win[r0] = x0;
      if (i1 < nl && r1 < keep_n) sw.win[r1] = x1;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// CTA-level select by one histogram pass over keys in shared memory, when
// the chunk partials gave the key range [kfloor, kceil] (the smallest and the
// largest chunk-maximum key; kfloor is at most the keep-th largest key when
// at least keep chunks hold a legal candidate).  One pass makes the keys
// (from z for kZStaged) and counts them; the cut bounds the winners; one more
// pass lists every key at or above the cut as (key << 32 | ~flat), whose
// descending order is the tie order (score desc, flat asc).  Falls back to
// cta_select when the range is unknown or the list does not fit.  Leaves
// sw.win[0..n) sorted; returns n = min(keep, legal candidates).
// ---------------------------------------------------------------------------
template <int NT, typename SW>
__device__ int cta_select_bins(const StepLaunch& a, int q, BeamTab& bt, SW& sw, uint32_t* keys, KeySrc src) {
  constexpr int NW = NT / 32;
  constexpr int LCAP = NW * 256 / 2;  // u64 list entries in the histogram's space
  static_assert(NW * 256 >= kBins, "histogram space");
  uint32_t* hist = &sw.whist[0][0];
  unsigned long long* list = reinterpret_cast<unsigned long long*>(hist);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int total = bt.total;
  const int keep_n = min(a.keep, bt.nlegal);
  if (keep_n == 0 || src == kGlobal) return cta_select<NT>(a, q, bt, sw, keys, src);
  for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
  __syncthreads();  // publishes the lse and the key range of beam_lse_sel (and staged keys)
  const uint32_t lo = bt.kfloor, hi = bt.kceil;
  if (bt.nne < keep_n || lo > hi) return cta_select<NT>(a, q, bt, sw, keys, src);
  const int sh = bin_shift(lo, hi);
  if (src == kZStaged) {
    // one warp a 32-slot chunk (the beam looked up once for 32 candidates)
    const int nitems = bt.istart[a.Wc];
    for (int i = warp; i < nitems; i += NW) {
      const int k = item_beam(bt, a.Wc, i);
      const int j = (i - bt.istart[k]) * kChunk + lane;
      if (j < bt.cnt[k]) {
        const int c = bt.start[k] + j;
        const float z = __uint_as_float(keys[c]);
        const uint32_t key = (z == -INFINITY) ? 0u : f2ord(bt.cum[k] + (z - bt.lse[k]));
        keys[c] = key;
        if (key >= lo) atomicAdd(&hist[bin_of(key, lo, sh)], 1u);
      }
    }
  } else {
    for (int c = tid; c < total; c += NT) {
      const uint32_t key = keys[c];
      if (key && key >= lo) atomicAdd(&hist[bin_of(key, lo, sh)], 1u);
    }
  }
  __syncthreads();
  const uint32_t all = hist_cut<NT>(hist, sw, (uint32_t)keep_n);
  if (all < (uint32_t)keep_n || sw.cnt_gt + sw.cnt_eq > LCAP)  // uniform: every thread read the same counts
    return cta_select<NT>(a, q, bt, sw, keys, kKeysStaged);
  const uint32_t tcut = lo + (sw.prefix << sh);  // smallest key in the cut bin or above
  const int nl = sw.cnt_gt + sw.cnt_eq;
  for (int c0 = warp * 32; c0 < total; c0 += NT) {
    const int c = c0 + lane;
    const uint32_t key = (c < total) ? keys[c] : 0u;
    warp_append(list, LCAP, sw.nwin, key && key >= tcut, key, c, lane);
  }
  __syncthreads();
  place_winners<NT>(list, nl, keep_n, sw);
  return keep_n;
}

// Staged second cut of the chunk-filtered select (scores in the global slot
// buffer): the chunks whose maximum key reaches tc are compacted into cid[],
// their candidates' keys (0 below tc or beyond the beam's slots) copied into
// kst[] by a flat pass, the keys cut for keep by 2,048 bins over [tc, kceil],
// and the keys at or above the cut listed and placed.  spare holds cid (at
// most spare_cap / 33 chunks) then kst.  Returns -1, having written nothing
// the caller needs, when the chunks or the final list do not fit.
template <int NT, typename SW>
__device__ int stage_passing_chunks(const StepLaunch& a, int q, BeamTab& bt, SW& sw, const uint32_t* ckb,
                                    const uint32_t* kb, int st, uint32_t tc, uint32_t* spare, int spare_cap) {
  constexpr int NW = NT / 32;
  constexpr int LCAP = NW * 256 / 2;
  uint32_t* hist = &sw.whist[0][0];
  unsigned long long* list = reinterpret_cast<unsigned long long*>(hist);
  const int tid = threadIdx.x, lane = tid & 31;
  const int keep_n = min(a.keep, bt.nlegal);
  const int maxc = spare ? spare_cap / 33 : 0;
  if (maxc == 0) return -1;
  const int nitems = bt.istart[a.Wc];
  int* cid = reinterpret_cast<int*>(spare);
  uint32_t* kst = spare + maxc;
  if (tid == 0) sw.nwin = 0;
  for (int i = tid; i < kBins; i += NT) hist[i] = 0u;  // counted while the keys are staged
  __syncthreads();
  for (int i0 = 0; i0 < nitems; i0 += NT) {
    const int i = i0 + tid;
    const bool f = (i < nitems) && ckb[(size_t)i * st] >= tc;
    const unsigned bal = __ballot_sync(kFull, f);
    int pos = 0;
    if (lane == 0 && bal) pos = atomicAdd(&sw.nwin, __popc(bal));
    pos = __shfl_sync(kFull, pos, 0) + __popc(bal & ((1u << lane) - 1u));
    if (f && pos < maxc) cid[pos] = i;
  }
  __syncthreads();
  const int npass = sw.nwin;
  if (npass > maxc) return -1;
  const int ne = npass * kChunk;
  const uint32_t hi = bt.kceil;
  const int sh = bin_shift(tc, hi);
  constexpr int UL = 16;  // global loads a thread keeps in flight
  for (int e0 = tid; e0 < ne; e0 += UL * NT) {
    int kk[UL], jj[UL];
#pragma unroll
    for (int u = 0; u < UL; ++u) {
      const int e = e0 + u * NT;
      kk[u] = 0;
      jj[u] = -1;  // no candidate
      if (e < ne) {
        const int item = cid[e >> 5];
        const int k = (int)kb[(size_t)item * st];
        const int j = (item - bt.istart[k]) * kChunk + (e & 31);
        kk[u] = k;
        if (j < bt.cnt[k]) jj[u] = j;
      }
    }
    uint32_t key[UL];
    cand_keys_batch<UL>(a, bt, q, kk, jj, key);
#pragma unroll
    for (int u = 0; u < UL; ++u) {
      const uint32_t k2 = key[u] >= tc ? key[u] : 0u;
      if (e0 + u * NT < ne) kst[e0 + u * NT] = k2;
      if (k2) atomicAdd(&hist[bin_of(k2, tc, sh)], 1u);
    }
  }
  __syncthreads();
  if (hist_cut<NT>(hist, sw, (uint32_t)keep_n) < (uint32_t)keep_n) return -1;
  if (sw.cnt_gt + sw.cnt_eq > LCAP) return -1;
  const uint32_t t2 = tc + (sw.prefix << sh);
  // hist_cut has zeroed sw.nwin and synchronised after its last histogram read
  for (int e0 = 0; e0 < ne; e0 += NT) {
    const int e = e0 + tid;
    const uint32_t key = (e < ne) ? kst[e] : 0u;
    int flat = 0;
    if (key >= t2 && key) {
      const int item = cid[e >> 5];
      const int k = (int)kb[(size_t)item * st];
      flat = bt.start[k] + (item - bt.istart[k]) * kChunk + (e & 31);
    }
    warp_append(list, LCAP, sw.nwin, key && key >= t2, key, flat, lane);
  }
  __syncthreads();
  place_winners<NT>(list, sw.nwin, keep_n, sw);
  return keep_n;
}

// ---------------------------------------------------------------------------
// Chunk-filtered select for steps with chunk partials (from shared memory
// `ps` by chunk item, or the global partial buffer when ps is null), with the
// slot scores in shared memory (kSmemZ: `zs` by flat candidate) or in the
// global slot buffer.
//   1. Every chunk's maximum key goes to ckb[i * st] and its beam to
//      kb[i * st]; the maxima are cut for keep: at least keep chunk maxima,
//      all true candidates, lie at or above the cut key tc, so the keep-th
//      largest candidate does too.
//   2. The candidates >= tc of the chunks whose maximum reaches tc are cut
//      again for keep over [tc, kceil]: cut key t2.
//   3. The candidates >= t2 are listed and placed in descending order.
// For a small keep (16 * keep within the list space) the candidates >= tc are
// listed and placed at once, and 2 and 3 run only if that list overflows.
// In 2 and 3 each warp tests 32 chunks at once (lane l: chunk i0 + l * NW +
// warp) and scores the passing ones U at a time.  Returns -1 (caller falls
// back) when the key range is unknown or the final list would not fit in the
// histogram's space.
// ---------------------------------------------------------------------------
template <int NT, bool kSmemZ, typename SW>
__device__ int cta_select_chunks(const StepLaunch& a, int q, BeamTab& bt, SW& sw, const float2* ps, const float* zs,
                                 uint32_t* ckb, uint32_t* kb, int st, uint32_t* spare = nullptr, int spare_cap = 0) {
  constexpr int NW = NT / 32;
  constexpr int LCAP = NW * 256 / 2;
  constexpr int U = 4;  // chunks a warp has in flight
  static_assert(NW * 256 >= kBins, "histogram space");
  uint32_t* hist = &sw.whist[0][0];
  unsigned long long* list = reinterpret_cast<unsigned long long*>(hist);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int keep_n = min(a.keep, bt.nlegal);
  if (keep_n == 0) return 0;
  for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
  __syncthreads();  // publishes the lse and the key range of beam_lse_sel
  const uint32_t lo = bt.kfloor, hi = bt.kceil;
  if (bt.nne < keep_n || lo > hi) return -1;
  const int nitems = bt.istart[a.Wc];
  const int sh = bin_shift(lo, hi);
  // 1. chunk maxima (a thread reads and then overwrites its own chunks' entries)
  for (int i0 = tid; i0 < nitems; i0 += U * NT) {
    float2 p[U];
    int kk[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * NT;
      p[u] = make_float2(-INFINITY, 0.f);
      kk[u] = 0;
      if (i < nitems) {
        kk[u] = item_beam(bt, a.Wc, i);
        p[u] = ps ? ps[i] : a.part[(size_t)q * a.pq + (size_t)kk[u] * a.nch + (i - bt.istart[kk[u]])];
      }
    }
    asm volatile("" ::: "memory");  // the entries below may overwrite ps[i] in place: reads first
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * NT;
      if (i >= nitems) continue;
      const int k = kk[u];
      const uint32_t ck = (p[u].y > 0.f) ? f2ord(bt.cum[k] + (p[u].x - bt.lse[k])) : 0u;
      ckb[(size_t)i * st] = ck;
      kb[(size_t)i * st] = (uint32_t)k;
      if (ck >= lo) atomicAdd(&hist[bin_of(ck, lo, sh)], 1u);
    }
  }
  __syncthreads();
  if (hist_cut<NT>(hist, sw, (uint32_t)keep_n) < (uint32_t)keep_n) return -1;
  const uint32_t tc = lo + (sw.prefix << sh);
  const int sh2 = bin_shift(tc, hi);
  // a small keep lists every candidate >= tc at once (pass 1) and cuts again
  // only when that list overflows; a large keep cuts again first (pass 2)
  if constexpr (!kSmemZ) {
    // scores in the global slot buffer: copy the candidates of the chunks
    // whose maximum reaches tc into shared memory in one flat pass (many
    // loads in flight), then cut, list and place from there
    const int n = stage_passing_chunks<NT>(a, q, bt, sw, ckb, kb, st, tc, spare, spare_cap);
    if (n >= 0) return n;
    if (tid == 0) sw.nwin = 0;  // the passes below list from an empty list
    __syncthreads();
  }
  const int first = (keep_n * 16 <= LCAP) ? 1 : 2;
  if (first == 2) {
    for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
    __syncthreads();
  }
  for (int pass = first; pass <= 3; ++pass) {
    uint32_t tmin = tc;  // >= lo >= 1
    if (pass == 3) {
      if (hist_cut<NT>(hist, sw, (uint32_t)keep_n) < (uint32_t)keep_n) return -1;
      if (sw.cnt_gt + sw.cnt_eq > LCAP) return -1;
      tmin = tc + (sw.prefix << sh2);
    }
    for (int i0 = 0; i0 < nitems; i0 += NT) {
      const int ic = i0 + lane * NW + warp;
      const bool pass_c = (ic < nitems) && ckb[(size_t)ic * st] >= tmin;
      const int kl = pass_c ? (int)kb[(size_t)ic * st] : 0;
      unsigned bal = __ballot_sync(kFull, pass_c);
      while (bal) {
        uint32_t key[U];
        int flat[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          key[u] = 0u;
          flat[u] = 0;
          if (bal) {  // warp-uniform
            const int src = __ffs(bal) - 1;
            bal &= bal - 1u;
            const int k = __shfl_sync(kFull, kl, src);
            const int j = (i0 + src * NW + warp - bt.istart[k]) * kChunk + lane;
            if (j < bt.cnt[k]) {
              flat[u] = bt.start[k] + j;
              if constexpr (kSmemZ) {
                const float z = zs[flat[u]];
                key[u] = (z == -INFINITY) ? 0u : f2ord(bt.cum[k] + (z - bt.lse[k]));
              } else {
                key[u] = cand_key_kj(a, bt, q, k, j);
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (pass == 2) {
            if (key[u] >= tc) atomicAdd(&hist[bin_of(key[u], tc, sh2)], 1u);
          } else {
            warp_append(list, LCAP, sw.nwin, key[u] >= tmin, key[u], flat[u], lane);
          }
        }
      }
    }
    __syncthreads();
    if (pass == 1) {
      const int nl = sw.nwin;  // the same in every thread
      if (nl <= LCAP) {
        if (nl > 2 * keep_n && nl > 64) {
          // a long list: cut it once more by a 1,024-bin histogram over
          // [tc, kceil] (in sw.win, spare until the placement), keep the
          // entries at or above the cut and place those
          constexpr int NB3 = 1024, EPT = (LCAP + NT - 1) / NT;
          uint32_t* h3 = reinterpret_cast<uint32_t*>(sw.win);
          const int sh3 = (hi - tc < (uint32_t)NB3) ? 0 : (32 - __clz(hi - tc) - 10);
          for (int i = tid; i < NB3; i += NT) h3[i] = 0u;
          unsigned long long mine[EPT];
#pragma unroll
          for (int u = 0; u < EPT; ++u) mine[u] = (tid + u * NT < nl) ? list[tid + u * NT] : 0ull;
          __syncthreads();
#pragma unroll
          for (int u = 0; u < EPT; ++u)
            if (mine[u]) atomicAdd(&h3[min(((uint32_t)(mine[u] >> 32) - tc) >> sh3, (uint32_t)(NB3 - 1))], 1u);
          __syncthreads();
          hist_cut<NT, SW, NB3>(h3, sw, (uint32_t)keep_n);  // total nl >= keep_n
          const uint32_t t3 = tc + (sw.prefix << sh3);
#pragma unroll
          for (int u = 0; u < EPT; ++u)
            warp_append(list, LCAP, sw.nwin, mine[u] && (uint32_t)(mine[u] >> 32) >= t3, (uint32_t)(mine[u] >> 32),
                        (int)(0xFFFFFFFFu - (uint32_t)(mine[u] & 0xFFFFFFFFu)), lane);
          __syncthreads();
          place_winners<NT>(list, sw.nwin, keep_n, sw);
          return keep_n;
        }
        place_winners<NT>(list, nl, keep_n, sw);
        return keep_n;
      }
      for (int i = tid; i < kBins; i += NT) hist[i] = 0u;  // overflow: cut again
      __syncthreads();
    }
  }
  place_winners<NT>(list, sw.cnt_gt + sw.cnt_eq, keep_n, sw);
  return keep_n;
}

// ---------------------------------------------------------------------------
// Chunk-top select: full steps whose scores were never written.  The full
// projection's epilogue left, per 32-token chunk of every beam row, the
// legal-only partial (max, sum exp) and the chunk's second-largest legal z
// with the offset of the lowest token holding the largest (a.ptop).
//
// Within one chunk all candidates share the beam's cumulative score and
// log-sum-exp, so their order is the order of z.  Let tc be the keep-th
// largest chunk-maximum key: at least keep candidates (those maxima) reach
// tc, so every winner does.  A chunk whose second-largest is below the cut
// holds at most one candidate above it, its maximum; only chunks whose second
// also clears the cut are re-scored token by token, from the same operands
// the projection used.  Re-scored values may differ from the projection's by
// rounding, so the cut is lowered by a margin (kTopMargin on the score): every
// candidate left out is then below the keep-th largest listed.
// Candidates at or above the lowered cut are listed as (key << 32 | ~flat)
// and placed; when the list overflows, 2,048-bin histograms over the same
// implicit candidate set narrow the cut (at most three rounds, to one key
// value), and ties at that key go to the lowest flat slots by an ordered walk.
// Exact for any data; deterministic (a re-score is recomputed identically).
// ---------------------------------------------------------------------------
constexpr float kTopMargin = 1e-4f;

// Sequential dot W_s[t] . h_b with the full projection's operands.  For fp32
// weights the order of accumulation is the SIMT projection's (one fused
// multiply-add per element, ascending), so the value is bit-identical to it.
template <typename WT>
__device__ __forceinline__ float rescore_token(const StepLaunch& a, size_t b, int t) {
  // loads are issued eight 16-byte vectors at a time (d is a multiple of 8,
  // so d/4 fp32 or d/8 half vectors), then consumed in order
  constexpr int U = 8;
  const WT* w = static_cast<const WT*>(a.W) + (size_t)t * a.d;
  float z = 0.f;
  if constexpr (sizeof(WT) == 4) {
    const float4* h4 = reinterpret_cast<const float4*>(a.hq + b * a.d);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const int n = a.d / 4;
    for (int e0 = 0; e0 < n; e0 += U) {
      float4 hv[U], wv[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (e0 + u < n) {
          hv[u] = h4[e0 + u];
          wv[u] = w4[e0 + u];
        }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (e0 + u < n) {
          z = fmaf(hv[u].x, wv[u].x, z);
          z = fmaf(hv[u].y, wv[u].y, z);
          z = fmaf(hv[u].z, wv[u].z, z);
          z = fmaf(hv[u].w, wv[u].w, z);
        }
    }
  } else {
    const uint4* hh = reinterpret_cast<const uint4*>(static_cast<const WT*>(a.hq_hi) + b * a.d);
    const uint4* hl = a.hq_lo ? reinterpret_cast<const uint4*>(static_cast<const WT*>(a.hq_lo) + b * a.d) : nullptr;
    const uint4* w8 = reinterpret_cast<const uint4*>(w);
    const int n = a.d / 8;
    for (int e0 = 0; e0 < n; e0 += U) {
      uint4 wv[U], hv[U], lv[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (e0 + u < n) {
          wv[u] = w8[e0 + u];
          hv[u] = hh[e0 + u];
          lv[u] = hl ? hl[e0 + u] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (e0 + u < n) {
          float wf[8], hf[8], lf[8];
          Vec<WT>::cvt(wv[u], wf);
          Vec<WT>::cvt(hv[u], hf);
          Vec<WT>::cvt(lv[u], lf);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            z = fmaf(hf[i], wf[i], z);
            if (hl) z = fmaf(lf[i], wf[i], z);
          }
        }
    }
  }
  return z;
}

__device__ __forceinline__ float rescore(const StepLaunch& a, size_t b, int t) {
  switch (a.w_dtype) {
    case ZG_F32:
      return rescore_token<float>(a, b, t);
    case ZG_BF16:
      return rescore_token<__nv_bfloat16>(a, b, t);
    default:
      return rescore_token<__half>(a, b, t);
  }
}

// Key of score s lowered by the re-score margin (0 stays 0).
__device__ __forceinline__ uint32_t key_lowered(uint32_t k) {
  if (!k) return 0u;
  const float s = ord2f(k);
  const uint32_t lk = f2ord(s - kTopMargin * (1.f + fabsf(s)));
  return lk ? lk : 1u;
}

// What the select needs of chunk item i: the keys of its maximum (ck) and of
// its second-largest (k2), 0 when absent, its beam k and the offset t1 of its
// maximum.  Read from the global partials, or from a shared-memory stage of
// three words an item ([ck], [k2], [k << 8 | t1]) filled by one flat pass.
struct ChunkTop {
  uint32_t ck, k2;
  int k, t1;
};

__device__ __forceinline__ ChunkTop chunk_top_global(const StepLaunch& a, const BeamTab& bt, int q, int i) {
  ChunkTop t;
  t.k = item_beam(bt, a.Wc, i);
  const size_t pi = (size_t)q * a.pq + (size_t)t.k * a.nch + (i - bt.istart[t.k]);
  const float2 p = a.part[pi];
  const float2 t2 = a.ptop[pi];
  const float cum = bt.cum[t.k], lse = bt.lse[t.k];
  t.ck = (p.y > 0.f) ? f2ord(cum + (p.x - lse)) : 0u;
  t.k2 = (p.y > 0.f && t2.x != -INFINITY) ? f2ord(cum + (t2.x - lse)) : 0u;
  t.t1 = __float_as_int(t2.y);
  return t;
}

struct TopStage {
  const uint32_t* st;  // null: read the global partials
  int n;
  __device__ __forceinline__ ChunkTop get(const StepLaunch& a, const BeamTab& bt, int q, int i) const {
    if (!st) return chunk_top_global(a, bt, q, i);
    ChunkTop t;
    t.ck = st[i];
    t.k2 = st[n + i];
    const uint32_t w = st[2 * n + i];
    t.k = (int)(w >> 8);
    t.t1 = (int)(w & 255u);
    return t;
  }
};

// Candidates of chunk item i (beam t.k, chunk c) at or above tmin, one a
// lane: lane j's (key, flat) for token 32c + j (key 0: none).  Warp-wide.
__device__ __forceinline__ uint32_t chunk_top_cands(const StepLaunch& a, const BeamTab& bt, int q, const ChunkTop& t,
                                                    int c, uint32_t tmin, int lane, int* flat) {
  const int k = t.k;
  *flat = bt.start[k] + c * kChunk + lane;
  if (t.ck < tmin) return 0u;
  if (t.k2 < tmin) return (lane == t.t1) ? t.ck : 0u;  // only the maximum can clear the cut
  // re-score the chunk: every legal token at or above the cut
  const int tok = c * kChunk + lane;
  bool legal = tok < a.V;
  if (legal && a.mode != kUncon) legal = (legal_bits(a, bt, q, k)[c] >> lane) & 1u;
  if (!legal) return 0u;
  const float z = rescore(a, (size_t)q * a.Wc + k, tok);
  const uint32_t kz = f2ord(bt.cum[k] + (z - bt.lse[k]));
  return kz >= tmin ? kz : 0u;
}

// stage: shared memory of stage_cap words for the per-chunk stage (used when
// three words an item fit), else null.
template <int NT, typename SW>
__device__ int cta_select_tops(const StepLaunch& a, int q, BeamTab& bt, SW& sw, uint32_t* stage, int stage_cap) {
  constexpr int NW = NT / 32;
  constexpr int LCAP = NW * 256 / 2;
  static_assert(NW * 256 >= kBins, "histogram space");
  uint32_t* hist = &sw.whist[0][0];
  unsigned long long* list = reinterpret_cast<unsigned long long*>(hist);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int keep_n = min(a.keep, bt.nlegal);
  if (keep_n == 0) return 0;
  const int nitems = bt.istart[a.Wc];
  for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
  __syncthreads();  // publishes the lse and the chunk-maximum key range of beam_lse_sel
  // 1. one flat pass over the chunks: stage their tops (when they fit) and
  //    count the maxima's keys over [kfloor, kceil]; cut tc = the keep-th
  //    largest chunk maximum
  TopStage ts{(stage && 3 * nitems <= stage_cap) ? stage : nullptr, nitems};
  const bool cut = bt.nne >= keep_n && bt.kfloor <= bt.kceil;
  const uint32_t lo = bt.kfloor, hi = bt.kceil;
  const int sh = cut ? bin_shift(lo, hi) : 0;
  for (int i0 = tid; i0 < nitems; i0 += 4 * NT) {
    ChunkTop t[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u * NT < nitems) t[u] = chunk_top_global(a, bt, q, i0 + u * NT);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * NT;
      if (i >= nitems) continue;
      if (ts.st) {
        stage[i] = t[u].ck;
        stage[nitems + i] = t[u].k2;
        stage[2 * nitems + i] = ((uint32_t)t[u].k << 8) | (uint32_t)t[u].t1;
      }
      if (cut && t[u].ck >= lo) atomicAdd(&hist[bin_of(t[u].ck, lo, sh)], 1u);
    }
  }
  __syncthreads();
  uint32_t tmin = 1u;
  if (cut) {
    if (hist_cut<NT>(hist, sw, (uint32_t)keep_n) >= (uint32_t)keep_n) tmin = key_lowered(lo + (sw.prefix << sh));
    __syncthreads();
  }
  // 2. the chunks whose maximum reaches tmin are compacted, then each warp
  //    produces their candidates once (re-scoring where needed) into a
  //    shared-memory list, which is cut and placed without touching the
  //    scores again.  The multi-pass route below is the fallback when the
  //    list space does not hold them.
  if (stage) {
    const int used = ts.st ? 3 * nitems : 0;
    const int room = stage_cap - used;
    if (tid == 0) sw.nwin = 0;
    __syncthreads();
    int* cid = reinterpret_cast<int*>(stage + used);
    const int maxc = room / 4;  // chunk ids, then candidates (two words each)
    for (int i0 = 0; i0 < nitems; i0 += NT) {
      const int i = i0 + tid;
      bool f = false;
      if (i < nitems) f = (ts.st ? ts.st[i] : chunk_top_global(a, bt, q, i).ck) >= tmin;
      const unsigned bal = __ballot_sync(kFull, f);
      int pos = 0;
      if (lane == 0 && bal) pos = atomicAdd(&sw.nwin, __popc(bal));
      pos = __shfl_sync(kFull, pos, 0) + __popc(bal & ((1u << lane) - 1u));
      if (f && pos < maxc) cid[pos] = i;
    }
    __syncthreads();
    const int npass = sw.nwin;
    if (npass <= maxc) {
      // candidates after the chunk ids, 8-byte aligned
      const int cofs = (used + npass + 1) & ~1;
      unsigned long long* cand = reinterpret_cast<unsigned long long*>(stage + cofs);
      const int ccap = (stage_cap - cofs) / 2;
      __syncthreads();
      if (tid == 0) sw.nwin = 0;
      __syncthreads();
      for (int w = warp; w < npass; w += NW) {
        const int i = cid[w];
        const ChunkTop t = ts.get(a, bt, q, i);
        int flat;
        const uint32_t key = chunk_top_cands(a, bt, q, t, i - bt.istart[t.k], tmin, lane, &flat);
        warp_append(cand, ccap, sw.nwin, key != 0u, key, flat, lane);
      }
      __syncthreads();
      const int nc = sw.nwin;
      if (nc <= ccap && nc >= keep_n) {
        // cut the list's keys for keep over [tmin, max] by 2,048 bins; keys
        // at or above the cut go to the list space and are placed
        for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
        if (tid == 0) sw.prefmask = 0u;
        __syncthreads();
        for (int e = tid; e < nc; e += NT) atomicMax(&sw.prefmask, (uint32_t)(cand[e] >> 32));
        __syncthreads();
        const uint32_t kmax = sw.prefmask;
        const int csh = bin_shift(tmin, kmax);
        for (int e = tid; e < nc; e += NT) atomicAdd(&hist[bin_of((uint32_t)(cand[e] >> 32), tmin, csh)], 1u);
        __syncthreads();
        hist_cut<NT>(hist, sw, (uint32_t)keep_n);
        const uint32_t cutk = tmin + (sw.prefix << csh);
        const int nlist = sw.cnt_gt + sw.cnt_eq;
        __syncthreads();
        if (nlist <= LCAP) {
          if (tid == 0) sw.nwin = 0;
          __syncthreads();
          for (int e0 = 0; e0 < nc; e0 += NT) {
            const int e = e0 + tid;
            const unsigned long long x = (e < nc) ? cand[e] : 0ull;
            const bool f = (e < nc) && (uint32_t)(x >> 32) >= cutk;
            const unsigned bal = __ballot_sync(kFull, f);
            int pos = 0;
            if (lane == 0 && bal) pos = atomicAdd(&sw.nwin, __popc(bal));
            pos = __shfl_sync(kFull, pos, 0) + __popc(bal & ((1u << lane) - 1u));
            if (f && pos < LCAP) list[pos] = x;
          }
          __syncthreads();
          place_winners<NT>(list, sw.nwin, keep_n, sw);
          return keep_n;
        }
      }
    }
    __syncthreads();
  }
  // fallback: every pass visits the chunks whose maximum reaches tmin: each
  // lane tests one chunk, the warp then takes the passing ones in turn
  auto for_chunks = [&](auto&& body) {
    for (int i0 = 0; i0 < nitems; i0 += NT) {
      const int ic = i0 + lane * NW + warp;
      ChunkTop t{0u, 0u, 0, 0};
      if (ic < nitems) t = ts.get(a, bt, q, ic);
      unsigned bal = __ballot_sync(kFull, ic < nitems && t.ck >= tmin);
      while (bal) {
        const int src = __ffs(bal) - 1;
        bal &= bal - 1u;
        ChunkTop tt;
        tt.ck = __shfl_sync(kFull, t.ck, src);
        tt.k2 = __shfl_sync(kFull, t.k2, src);
        tt.k = __shfl_sync(kFull, t.k, src);
        tt.t1 = __shfl_sync(kFull, t.t1, src);
        const int c = i0 + src * NW + warp - bt.istart[tt.k];
        int flat;
        const uint32_t key = chunk_top_cands(a, bt, q, tt, c, tmin, lane, &flat);
        body(key, flat);
      }
    }
  };
  // fallback 1: list every candidate at or above tmin
  if (tid == 0) sw.nwin = 0;
  __syncthreads();
  for_chunks([&](uint32_t key, int flat) { warp_append(list, LCAP, sw.nwin, key != 0u, key, flat, lane); });
  __syncthreads();
  int nl = sw.nwin;
  if (nl < keep_n) return -1;  // cannot happen (the keep chunk maxima are listed); caller flags it
  if (nl <= LCAP) {
    place_winners<NT>(list, nl, keep_n, sw);
    return keep_n;
  }
  // 3. overflow: narrow [lo, hi] by histograms of the same candidates until
  //    the keys at or above the cut fit the list, or the cut is one key value
  uint32_t rlo = tmin, rhi = 0xFFFFFFFFu;
  int above = 0;  // candidates with a key > rhi (all winners)
  for (int round = 0; round < 4; ++round) {
    const int rsh = bin_shift(rlo, rhi);
    for (int i = tid; i < kBins; i += NT) hist[i] = 0u;
    __syncthreads();
    for_chunks([&](uint32_t key, int flat) {
      if (key >= rlo && key <= rhi) atomicAdd(&hist[bin_of(key, rlo, rsh)], 1u);
    });
    __syncthreads();
    hist_cut<NT>(hist, sw, (uint32_t)(keep_n - above));  // total >= keep_n - above by construction
    const uint32_t b = sw.prefix;
    const uint32_t nlo = rlo + (b << rsh);
    const unsigned long long top = (unsigned long long)nlo + ((1ull << rsh) - 1ull);
    const uint32_t nhi = (b == (uint32_t)(kBins - 1)) ? rhi : (uint32_t)(top < rhi ? top : rhi);
    const int gt = sw.cnt_gt, eq = sw.cnt_eq;
    __syncthreads();
    if (above + gt + eq <= LCAP) {  // list everything at or above the cut bin
      if (tid == 0) sw.nwin = 0;
      __syncthreads();
      for_chunks([&](uint32_t key, int flat) { warp_append(list, LCAP, sw.nwin, key >= nlo, key, flat, lane); });
      __syncthreads();
      place_winners<NT>(list, sw.nwin, keep_n, sw);
      return keep_n;
    }
    above += gt;
    rlo = nlo;
    rhi = nhi;
    if (rlo == rhi) break;  // one key value: ties
  }
  // 4. ties at key value T = rlo: every key > T wins; the remaining winners
  //    are the lowest flat slots with key == T, found by one warp walking the
  //    chunks in order
  const uint32_t T = rlo;
  if (tid == 0) sw.nwin = 0;
  __syncthreads();
  for_chunks([&](uint32_t key, int flat) { warp_append(list, LCAP, sw.nwin, key > T, key, flat, lane); });
  __syncthreads();
  if (warp == 0) {
    int need = keep_n - sw.nwin;  // the same in every lane
    for (int i0 = 0; i0 < nitems && need > 0; i0 += 32) {
      const int ic = i0 + lane;
      ChunkTop t{0u, 0u, 0, 0};
      if (ic < nitems) t = ts.get(a, bt, q, ic);
      unsigned bal = __ballot_sync(kFull, ic < nitems && t.ck >= tmin);
      while (bal && need > 0) {
        const int src = __ffs(bal) - 1;  // ascending chunk order = ascending flat order
        bal &= bal - 1u;
        ChunkTop tt;
        tt.ck = __shfl_sync(kFull, t.ck, src);
        tt.k2 = __shfl_sync(kFull, t.k2, src);
        tt.k = __shfl_sync(kFull, t.k, src);
        tt.t1 = __shfl_sync(kFull, t.t1, src);
        int flat;
        const uint32_t key = chunk_top_cands(a, bt, q, tt, i0 + src - bt.istart[tt.k], tmin, lane, &flat);
        const unsigned tie = __ballot_sync(kFull, key == T && key != 0u);
        const int before = __popc(tie & ((1u << lane) - 1u));
        if (key == T && key != 0u && before < need) {
          const int pos = sw.nwin + before;
          if (pos < LCAP) list[pos] = ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)flat);
        }
        const int took = min(__popc(tie), need);
        need -= took;
        if (lane == 0) sw.nwin += took;
        __syncwarp();
      }
    }
  }
  __syncthreads();
  place_winners<NT>(list, min(sw.nwin, LCAP), keep_n, sw);
  return keep_n;
}

// Write the survivors (sorted winners) of request q, one thread a survivor:
// the next beams (parent, token, next-step row, score) or, at the last step,
// the output SIDs by following parent indices back; rows beyond n are dead
// beams / padding.  On dense steps the next-step row is the row's first entry
// plus the token's rank among the row's legal tokens: from the chunk legal
// masks in shared memory when given (cluster kernel), else from the bitmap.
template <int NT, typename SW>
__device__ void write_survivors(const StepLaunch& a, int q, const BeamTab& bt, const SW& sw, int n,
                                const uint32_t* msm = nullptr) {
  const int s = a.s;
  const size_t BW = (size_t)a.B * a.beam;
  const bool sparse_slots = (a.mode == kSelSparse || a.mode == kFullSparse);
  for (int i = threadIdx.x; i < a.keep; i += NT) {
    if (i < n) {
      const unsigned long long w = sw.win[i];
      const uint32_t key = (uint32_t)(w >> 32);
      const int c = (int)(0xFFFFFFFFu - (uint32_t)(w & 0xFFFFFFFFu));
      const int k = upper_find(bt.start, a.Wc, c);
      const int j = c - bt.start[k];
      int t;
      uint32_t nrow = 0;
      if (sparse_slots) {
        t = a.tab.col[bt.rp[k] + j];
        nrow = bt.rp[k] + (uint32_t)j;
      } else {
        t = j;
        if (a.mode != kUncon) {
          uint32_t rank = 0;
          if (msm) {
            const uint32_t* mk = msm + bt.istart[k];
            for (int wd = 0; wd < (t >> 5); ++wd) rank += __popc(mk[wd]);
            rank += __popc(mk[t >> 5] & ((1u << (t & 31)) - 1u));
          } else {
            const uint32_t* bm = legal_bits(a, bt, q, k);
            for (int wd = 0; wd < (t >> 5); ++wd) rank += __popc(bm[wd]);
            rank += __popc(bm[t >> 5] & ((1u << (t & 31)) - 1u));
          }
          nrow = bt.rp[k] + rank;
        }
      }
      const float score = ord2f(key);
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

}  // namespace dev
}  // namespace zg
