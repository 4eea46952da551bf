// Decode kernels for sm_103a.
//
//   k_decode_cluster  one thread-block cluster per request runs every
//                     selective step of the decode in a single launch:
//                     all CTAs of the cluster score the request's (beam,
//                     chunk) items, a hardware cluster barrier publishes the
//                     slots, the rank-0 CTA selects the next beams, another
//                     cluster barrier, next step.  No spin loops.
//   k_selective       the same scoring as a stand-alone step kernel
//   k_gather_add      hidden vectors of a full-projection step
//   k_full_simt       fp32 full projection (fp32 weights)
//   k_select          per-request select of a stand-alone step
//
// "ZeroGR: Filtering-First Constrained Decoding for Generative
// Recommendation" (paper-daily.com digest): "Overall flow" (four stages per
// step), "Why computing fewer scores is not automatically faster" (padded
// slots, in-place weight rows), "Why slice the index by decoding step" (a
// beam carries only its row; an entry's position is its next-step row).
#include <cooperative_groups.h>

#include "zg_device.cuh"

namespace zg {

__device__ uint32_t g_status;  // device status word, read by zg_check_device_status

namespace {

using namespace dev;
namespace cg = cooperative_groups;

// Programmatic dependent launch inside a selective step (k_beam_items ->
// k_selective -> k_select -> next step's k_beam_items): each of these kernels
// is launched so that it may start while its predecessor finishes.  It first
// waits for the predecessor's completion (griddepcontrol.wait) and only then
// lets its own successor launch, so a kernel that starts early knows that
// everything before its predecessor is complete; k_select builds its beam
// table (beam states of the previous select, index rows) before its wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kSelThreads = 512;
constexpr int kSelCap = 32768;       // keys staged in shared memory by k_select (one CTA a request)
constexpr int kClusterThreads = 256;
constexpr int kClusterCap = 11264;   // slot scores / keys held by the cluster kernel's rank-0 CTA
constexpr int kClusterPcap = 2048;   // chunk partials and masks held by the rank-0 CTA

// Select when the candidates do not fit in shared memory: filtered select
// on the maxima of the scored 32-slot chunks when there are chunk partials
// and their count fits in half the buffer, else on the maxima of tiles of
// whole chunks, else the radix select over the global slot buffer.  For
// full-score steps without chunk partials beam_lse has already stored the
// tile maxima in buf when tile_z_ready.
template <int NT, typename SW>
__device__ int select_large(const StepLaunch& a, int q, BeamTab& bt, SW& sw, uint32_t* buf, int cap,
                            bool tile_z_ready = false) {
  if (a.part && bt.istart[a.Wc] <= cap / 2) {
    const int nrep = chunk_rep_keys<NT>(a, q, bt, buf);
    const int n = cta_select_filtered<NT>(a, q, bt, sw, buf, cap, nrep, 0, kChunk);
    if (n >= 0) return n;
    return cta_select<NT>(a, q, bt, sw, buf, kGlobal);
  }
  const bool need_z = (a.part == nullptr);  // tile maxima come from partials when there are any
  int rt, tw;
  tile_layout(a.Wc, a.S, cap, &rt, &tw);
  if (a.Wc * rt <= cap / 2 && (!need_z || tile_z_ready)) {
    const int nrep = tile_rep_keys<NT>(a, q, bt, buf, rt, tw);
    const int n = cta_select_filtered<NT>(a, q, bt, sw, buf, cap, nrep, rt, tw);
    if (n >= 0) return n;
  }
  return cta_select<NT>(a, q, bt, sw, buf, kGlobal);
}

// ---------------------------------------------------------------------------
// Stand-alone selective step over every request at once: the non-empty
// (beam, 32-slot chunk) items of the whole batch are numbered by a scan of
// the beams' chunk counts, and every warp of the grid scores one contiguous
// range of them, so the work is balanced across requests (a beam with
// thousands of legal tokens is spread over many warps).
//   k_beam_items: per beam its first index entry, fan-out and chunk count
//                 (0 for a dead beam); each CTA scans its beams' counts into
//                 offsets within the CTA and writes its total;
//   k_selective:  every CTA scans the (at most kItemBlocks) CTA totals in
//                 shared memory, so a beam's first item is its CTA's offset
//                 plus its offset within the CTA; then the scoring.
// ---------------------------------------------------------------------------
// beams per k_beam_items CTA: a multiple of 256, enough for at most kItemBlocks CTAs
__host__ __device__ __forceinline__ int item_block_beams(int N) {
  const int per = (N + kItemBlocks - 1) / kItemBlocks;
  return ((per + 255) / 256) * 256;
}

// Exclusive scan of one value per thread over a 256-thread CTA; *total gets
// the CTA's sum.  wsum: 8 ints of shared memory, free again on return.
__device__ __forceinline__ int cta256_exclusive_scan(int v, int32_t* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int x = wsum[w];
    before += (w < warp) ? x : 0;
    all += x;
  }
  __syncthreads();
  *total = all;
  return before + incl - v;
}

__global__ void __launch_bounds__(256) k_beam_items(const __grid_constant__ StepLaunch a) {
  __shared__ int32_t wsum[8];
  pdl_wait();
  pdl_trigger();
  const int N = a.B * a.Wc;
  const int bper = item_block_beams(N);
  int32_t* loc = a.bscan;  // first item of each beam, counted from its CTA's first
  int32_t* rp = loc + N;
  int32_t* fo = rp + N;
  int32_t* bsum = fo + N;  // items per CTA
  const int b0 = blockIdx.x * bper, b1 = min(N, b0 + bper);
  int carry = 0;
  for (int base = b0; base < b1; base += 256) {
    const int b = base + (int)threadIdx.x;
    int items = 0;
    uint32_t r0 = 0, F = 0;
    if (b < b1) {
      const int q = b / a.Wc, k = b - q * a.Wc;
      const BeamState bs = load_beam(a, q, k);
      if (bs.row != kDeadRow) {
        if (bs.row >= a.tab.rows) {
          flag(a.status, kStatusRow);
        } else {
          r0 = a.tab.rowptr[bs.row];
          F = a.tab.rowptr[bs.row + 1] - r0;
          items = (a.mode == kSelSparse) ? (int)((F + kChunk - 1) / kChunk) : a.nch;
        }
      }
    }
    int sum;
    const int ex = cta256_exclusive_scan(items, wsum, &sum);
    if (b < b1) {
      loc[b] = carry + ex;
      rp[b] = (int32_t)r0;
      fo[b] = (int32_t)F;
    }
    carry += sum;
  }
  if (threadIdx.x == 0) bsum[blockIdx.x] = carry;
}

template <typename WT, int VPL>
__global__ void __launch_bounds__(256) k_selective(const __grid_constant__ StepLaunch a) {
  __shared__ int32_t boff[kItemBlocks + 1];  // exclusive offsets of the k_beam_items CTAs, then the total
  __shared__ int32_t wsum[8];
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int N = a.B * a.Wc;
  const int bper = item_block_beams(N);
  const int nblk = (N + bper - 1) / bper;
  const int32_t* loc = a.bscan;
  const int32_t* rp = loc + N;
  const int32_t* fo = rp + N;
  const int32_t* bsum = fo + N;
  pdl_wait();
  pdl_trigger();
  {
    constexpr int PT = kItemBlocks / 256;  // CTA totals per thread
    int v[PT], sum = 0;
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      const int i = (int)threadIdx.x * PT + j;
      v[j] = (i < nblk) ? bsum[i] : 0;
      sum += v[j];
    }
    int all;
    int run = cta256_exclusive_scan(sum, wsum, &all);
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      boff[threadIdx.x * PT + j] = run;
      run += v[j];
    }
    if (threadIdx.x == 0) boff[kItemBlocks] = all;
    __syncthreads();
  }
  const int total = boff[kItemBlocks];
  // first item of beam p (p = N: the total)
  auto off = [&](int p) { return (p >= N) ? total : boff[p / bper] + loc[p]; };
  const int per = (total + nw - 1) / nw;
  const int i0 = wid * per, i1 = min(total, i0 + per);
  if (i0 >= i1) return;
  // the beam of the range's first item (largest b with off(b) <= i0): a
  // 32-way search, each lane probing one point of the current interval
  int lo = 0, hi = N - 1;  // off(lo) <= i0 always holds
  while (hi > lo) {
    const int span = hi - lo;
    const int p = lo + (int)(((long long)span * (lane + 1)) / 32);  // lane 31 probes hi
    const unsigned ok = __ballot_sync(kFull, off(p) <= i0);
    const int top = ok ? 31 - __clz(ok) : -1;  // highest lane whose point is <= i0
    const int nlo = (top >= 0) ? lo + (int)(((long long)span * (top + 1)) / 32) : lo;
    const int nhi = (top < 31) ? lo + (int)(((long long)span * (top + 2)) / 32) - 1 : hi;
    lo = nlo;
    hi = max(nlo, nhi);
  }
  int b = lo, loaded = -1, ob = off(lo), onext = off(lo + 1);
  BeamState bs;
  float h[VPL][Vec<WT>::E];
  for (int it = i0; it < i1; ++it) {
    while (onext <= it) {
      ++b;
      ob = onext;
      onext = off(b + 1);
    }
    const int q = b / a.Wc, k = b - q * a.Wc;
    const int c = it - ob;
    const bool fresh = (b != loaded);  // consecutive chunks of one beam share its state and hidden vector
    if (fresh) bs = load_beam(a, q, k);
    int t_lane;
    const uint32_t vmask = chunk_tokens(a, bs, (uint32_t)rp[b], (uint32_t)fo[b], c, lane, t_lane);
    if (fresh) {
      // chunk 0 of a beam is the first of its chunks that its warp meets: that warp stores h
      load_hidden<WT, VPL>(a, q, k, bs, lane, (c == 0) && a.h_out, h);
      loaded = b;
    }
    score_rows<WT, VPL>(a, q, k, c, lane, vmask, t_lane, h);
  }
}

// ---------------------------------------------------------------------------
// Cluster decode of the selective steps s0..L (all steps selective).
//
// Per step: every CTA builds the request's beam table, the cluster's warps
// score its (beam, chunk) items and, when the request's candidates fit,
// write the slot scores, chunk partials and chunk legal masks straight into
// the rank-0 CTA's shared memory (distributed shared memory); a cluster
// barrier publishes them; the rank-0 CTA computes the legal-only
// log-sum-exps and keys in shared memory, selects and writes the next
// beams; a second cluster barrier publishes those.  Larger requests go
// through the global slot buffer instead.  At launch every CTA prefetches
// its share of the fused steps' tables into L2 with bulk prefetches.
// ---------------------------------------------------------------------------
struct MegaArgs {
  int32_t s0, L, cap, pcap;
  int32_t npf, pad;
  uint64_t pf_total;
  PrefetchRegion pf[kMaxPrefetch];
  StepLaunch st[ZG_MAX_STEPS];
};

__device__ __forceinline__ void l2_prefetch(const MegaArgs& A) {
  using u64 = unsigned long long;
  const u64 total = A.pf_total;
  if (!total) return;
  const u64 per = ((total + gridDim.x - 1) / gridDim.x + 15ull) & ~15ull;
  const u64 lo = (u64)blockIdx.x * per;
  const u64 hi = total < lo + per ? total : lo + per;
  if (lo >= hi) return;
  u64 piece = (((hi - lo) + blockDim.x - 1) / blockDim.x + 15ull) & ~15ull;
  if (piece < 4096ull) piece = 4096ull;
  const u64 my_lo = lo + (u64)threadIdx.x * piece;
  const u64 my_hi = hi < my_lo + piece ? hi : my_lo + piece;
  u64 off = 0;
  for (int i = 0; i < A.npf && my_lo < my_hi; ++i) {
    const u64 rb = A.pf[i].bytes;
    const u64 x = my_lo > off ? my_lo : off;
    const u64 y = my_hi < off + rb ? my_hi : off + rb;
    if (x < y) {
      const char* p = static_cast<const char*>(A.pf[i].ptr) + (x - off);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"((uint32_t)(y - x)) : "memory");
    }
    off += rb;
  }
}

template <typename WT, int VPL>
__global__ void __launch_bounds__(kClusterThreads, 2) k_decode_cluster(const __grid_constant__ MegaArgs A) {
  extern __shared__ __align__(16) uint32_t dyn[];
  uint32_t* zsm = dyn;                                        // [cap] slot scores, then keys
  float2* psm = reinterpret_cast<float2*>(dyn + A.cap);       // [pcap] chunk partials
  uint32_t* msm = reinterpret_cast<uint32_t*>(psm + A.pcap);  // [pcap] chunk legal masks
  constexpr int NT = kClusterThreads, NW = NT / 32;
  __shared__ BeamTab bt;
  __shared__ SelWorkT<NW> sw;
  cg::cluster_group cl = cg::this_cluster();
  const int G = (int)cl.num_blocks();
  const int r = (int)cl.block_rank();
  const int q = blockIdx.x / G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  l2_prefetch(A);
  for (int s = A.s0; s <= A.L; ++s) {
    const StepLaunch& a = A.st[s - 1];
    build_beam_table<NT>(a, q, bt);
    const int nitems = bt.istart[a.Wc];
    const bool p_smem = nitems <= A.pcap;              // chunk partials in rank 0's shared memory
    const bool in_smem = p_smem && bt.total <= A.cap;  // and the slot scores too
    SlotSink sink{};
    if (p_smem) {
      sink.z = in_smem ? cl.map_shared_rank(reinterpret_cast<float*>(zsm), 0) : nullptr;
      sink.part = cl.map_shared_rank(psm, 0);
      sink.mask = cl.map_shared_rank(msm, 0);
    }
    for (int it = r * NW + warp; it < nitems; it += G * NW) {
      const int k = item_beam(bt, a.Wc, it);
      const int c = it - bt.istart[k];
      BeamState bs;
      bs.row = bt.row[k];
      bs.cum = bt.cum[k];
      bs.par = bt.par[k];
      bs.tok = bt.tok[k];
      sink.flat0 = bt.start[k] + c * kChunk;
      sink.item = it;
      sink.cnt = bt.cnt[k];
      score_chunk<WT, VPL>(a, q, k, bs, bt.rp[k], (uint32_t)bt.nleg[k], c, lane, p_smem ? &sink : nullptr);
    }
    cl.sync();  // slots and partials of the whole request are now visible to rank 0
    if (r == 0) {
      int n;
      if (in_smem) {
        beam_lse_sel<NT>(a, q, bt, psm);
        // the chunk-maximum cut filters only when the chunks outnumber the
        // survivors well; otherwise one flat histogram pass over the staged
        // scores is faster.  Chunk beams and keys replace the spent partials
        // in place.
        n = -1;
        if (4 * min(a.keep, bt.nlegal) < nitems)
          n = cta_select_chunks<NT, true>(a, q, bt, sw, psm, reinterpret_cast<const float*>(zsm),
                                          reinterpret_cast<uint32_t*>(psm) + 1, reinterpret_cast<uint32_t*>(psm), 2);
        if (n < 0) n = cta_select_bins<NT>(a, q, bt, sw, zsm, kZStaged);
        write_survivors<NT>(a, q, bt, sw, n, msm);
      } else {
        // scores in the global slot buffer; the partials in shared memory too
        // when they fit (their log-sum-exp then reads no global memory)
        if (p_smem)
          beam_lse_sel<NT>(a, q, bt, psm);
        else
          beam_lse<NT>(a, q, bt);
        __syncthreads();
        const int ni = bt.istart[a.Wc];
        // spare: the rest of the slot stage plus the partial and mask stages,
        // contiguous after it (the partials are read before the spare is used)
        n = (a.part && 2 * ni <= A.cap)
                ? cta_select_chunks<NT, false>(a, q, bt, sw, p_smem ? psm : nullptr, nullptr, zsm, zsm + ni, 1,
                                               zsm + 2 * ni, A.cap - 2 * ni + 3 * A.pcap)
                : -1;
        if (n < 0) {
          if (bt.total <= A.cap) {
            stage_keys_global<NT>(a, q, bt, zsm);
            n = cta_select_bins<NT>(a, q, bt, sw, zsm, kKeysStaged);
          } else {
            n = select_large<NT>(a, q, bt, sw, zsm, A.cap);
          }
        }
        write_survivors<NT>(a, q, bt, sw, n);
      }
    }
    cl.sync();  // next beams visible to every CTA of the cluster; rank 0's buffers free again
  }
}

// ---------------------------------------------------------------------------
// Gather-add for full-projection steps: H[b] = h_parent + C_{s-1}[token]
// (zero rows for dead beams).  One warp per beam, float4 accesses.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gather_add(const __grid_constant__ StepLaunch a, float* H) {
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int N = a.B * a.Wc;
  const int d4 = a.d / 4;
  for (int b = wid; b < N; b += nw) {
    const int q = b / a.Wc, k = b - q * a.Wc;
    const BeamState bs = load_beam(a, q, k);
    float4* out = reinterpret_cast<float4*>(H + (size_t)b * a.d);
    if (bs.row == kDeadRow) {
      for (int v = lane; v < d4; v += 32) out[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    const float4* hp = reinterpret_cast<const float4*>(a.h_prev + ((size_t)q * a.Wp + bs.par) * a.d);
    const float4* cr = reinterpret_cast<const float4*>(a.C_prev + (size_t)bs.tok * a.d);
    for (int v = lane; v < d4; v += 32) {
      const float4 x = hp[v], y = cr[v];
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
                                                   float* __restrict__ Z, int M, int V, int d, int ldz,
                                                   const FullEpi epi) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += BK) {
    {
      const int r = tid >> 2, kq = (tid & 3) * 4;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m0 + r < M && k0 + kq < d) x = *reinterpret_cast<const float4*>(H + (size_t)(m0 + r) * d + k0 + kq);
      As[kq][r] = x.x;
      As[kq + 1][r] = x.y;
      As[kq + 2][r] = x.z;
      As[kq + 3][r] = x.w;
    }
    {
      const int r = tid >> 2, kq = (tid & 3) * 4;
      float w[4] = {0.f, 0.f, 0.f, 0.f};
      if (n0 + r < V && k0 + kq < d) {
        const WT* p = W + (size_t)(n0 + r) * d + k0 + kq;
        if constexpr (sizeof(WT) == 4) {
          const float4 x = *reinterpret_cast<const float4*>(p);
          w[0] = x.x;
          w[1] = x.y;
          w[2] = x.z;
          w[3] = x.w;
        } else {
          const uint2 raw = *reinterpret_cast<const uint2*>(p);
          float t8[8];
          Vec<WT>::cvt(make_uint4(raw.x, raw.y, 0, 0), t8);
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
  if (Z) {
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
  if (epi.part) {
    // legal-only (max, sum exp) of each 32-token chunk: 8 threads (4 tokens
    // each) share a chunk; lanes tx^1, tx^2, tx^4 hold its other tokens.
    // With ptop also the chunk's second-largest legal z and the offset of
    // the lowest token holding its largest.
    const int chunk = (n0 >> 5) + (tx >> 3);
    const int sh = (tx & 7) * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + ty * 4 + i;
      const uint32_t lm = (m < M) ? (epi_legal_mask(epi, m, chunk, V) >> sh) & 0xFu : 0u;
      float mx = -INFINITY, m2 = -INFINITY;
      int arg = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool l = (lm >> j) & 1u;
        if (l && acc[i][j] > mx) {
          m2 = mx;
          mx = acc[i][j];
          arg = sh + j;
        } else if (l && acc[i][j] > m2) {
          m2 = acc[i][j];
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {  // merge (largest, lowest offset, second) pairs
        const float omx = __shfl_xor_sync(0xFFFFFFFFu, mx, o);
        const float om2 = __shfl_xor_sync(0xFFFFFFFFu, m2, o);
        const int oarg = __shfl_xor_sync(0xFFFFFFFFu, arg, o);
        const bool mine = (mx > omx) || (mx == omx && arg < oarg);
        const float lose = mine ? omx : mx;
        m2 = fmaxf(fmaxf(m2, om2), lose);
        arg = mine ? arg : oarg;
        mx = mine ? mx : omx;
      }
      float sm = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int j = 0; j < 4; ++j) sm += ((lm >> j) & 1u) ? __expf(acc[i][j] - mx) : 0.f;
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) sm += __shfl_xor_sync(0xFFFFFFFFu, sm, o);
      if ((tx & 7) == 0 && m < M && chunk * 32 < V) {
        const size_t pi = (size_t)m * (ldz >> 5) + chunk;
        epi.part[pi] = make_float2(mx, sm);
        if (epi.ptop) epi.ptop[pi] = make_float2(m2, __int_as_float(arg));
      }
    }
  }
  if (epi.part_all) {
    // (max, sum exp) over every token of each chunk (score-first normaliser)
    const int chunk = (n0 >> 5) + (tx >> 3);
    const int sh = (tx & 7) * 4;
    const int rem = V - chunk * 32;
    const uint32_t vm = (rem >= 32 ? 0xFFFFFFFFu : (rem <= 0 ? 0u : ((1u << rem) - 1u))) >> sh & 0xFu;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + ty * 4 + i;
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) mx = ((vm >> j) & 1u) ? fmaxf(mx, acc[i][j]) : mx;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
      float sm = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int j = 0; j < 4; ++j) sm += ((vm >> j) & 1u) ? __expf(acc[i][j] - mx) : 0.f;
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) sm += __shfl_xor_sync(0xFFFFFFFFu, sm, o);
      if ((tx & 7) == 0 && m < M && chunk * 32 < V) epi.part_all[(size_t)m * (ldz >> 5) + chunk] = make_float2(mx, sm);
    }
  }
}

// ---------------------------------------------------------------------------
// Stand-alone select: one CTA per request.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) k_select(const __grid_constant__ StepLaunch a) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ BeamTab bt;
  __shared__ SelWorkT<kSelThreads / 32> sw;
  const int q = blockIdx.x;
  build_beam_table<kSelThreads>(a, q, bt);
  pdl_wait();  // the step's scores and partials
  pdl_trigger();
  const bool staged = bt.total <= kSelCap;
  int rt, tw;
  tile_layout(a.Wc, a.S, kSelCap, &rt, &tw);
  // without partials (full scores of a sparse step) the tile maxima land in
  // keys[] while the log-sum-exp is computed
  beam_lse<kSelThreads>(a, q, bt, (!staged && !a.part && a.Wc * rt <= kSelCap / 2) ? keys : nullptr, rt, tw);
  __syncthreads();
  const int ni = bt.istart[a.Wc];
  if (a.ptop) {  // the scores were never written: chunk-top select
    int n = cta_select_tops<kSelThreads>(a, q, bt, sw, keys, kSelCap);
    if (n < 0) {
      if (threadIdx.x == 0) flag(a.status, kStatusSelect);  // unreachable: the cut's own maxima are listed
      n = 0;
    }
    write_survivors<kSelThreads>(a, q, bt, sw, n);
    return;
  }
  int n = (a.part && 2 * ni <= kSelCap)
              ? cta_select_chunks<kSelThreads, false>(a, q, bt, sw, nullptr, nullptr, keys, keys + ni, 1, keys + 2 * ni,
                                                      kSelCap - 2 * ni)
              : -1;
  if (n < 0) {
    if (staged) {
      stage_keys_global<kSelThreads>(a, q, bt, keys);
      n = cta_select_bins<kSelThreads>(a, q, bt, sw, keys, kKeysStaged);
    } else {
      n = select_large<kSelThreads>(a, q, bt, sw, keys, kSelCap, true);
    }
  }
  write_survivors<kSelThreads>(a, q, bt, sw, n);
}

// ---------------------------------------------------------------------------
// Score-first order on a sparse-format step: expand every beam's legal list
// (the index row's column entries) into a token bitmap row of its own,
// tab.bitmap[b * words] for beam b = q*Wc + k (zeros for a dead beam), so
// the full projection's epilogue and the select mask tokens as on a dense
// step.  One warp per beam: clear the row, then set the bits.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_legal_mask(const __grid_constant__ StepLaunch a) {
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int N = a.B * a.Wc;
  uint32_t* mask = const_cast<uint32_t*>(a.tab.bitmap);
  for (int b = wid; b < N; b += nw) {
    const int q = b / a.Wc, k = b - q * a.Wc;
    uint32_t* row = mask + (size_t)b * a.tab.words;
    for (int w = lane; w < (int)a.tab.words; w += 32) row[w] = 0u;
    __syncwarp();
    const BeamState bs = load_beam(a, q, k);
    if (bs.row == kDeadRow) continue;
    if (bs.row >= a.tab.rows) {
      if (lane == 0) flag(a.status, kStatusRow);
      continue;
    }
    const uint32_t rp = a.tab.rowptr[bs.row];
    const uint32_t F = a.tab.rowptr[bs.row + 1] - rp;
    for (uint32_t j = lane; j < F; j += 32) {
      const uint32_t t = a.tab.col[rp + j];
      if (t < (uint32_t)a.V)
        atomicOr(&row[t >> 5], 1u << (t & 31));
      else
        flag(a.status, kStatusToken);
    }
  }
}

// Tracing: counts of the work a step does, for roofline accounting.
__global__ void __launch_bounds__(256) k_trace_touch(const __grid_constant__ StepLaunch a, unsigned long long* cnt,
                                                     uint32_t* mask) {
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int N = a.B * a.Wc;
  const int words = (a.V + 31) / 32;
  for (int b = wid; b < N; b += nw) {
    const int q = b / a.Wc, k = b - q * a.Wc;
    const BeamState bs = load_beam(a, q, k);
    if (bs.row == kDeadRow) continue;
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


template <typename WT>
int vpl_for(int d) {
  const int nvec = d / (16 / (int)sizeof(WT));
  const int v = (nvec + 31) / 32;
  return v <= 1 ? 1 : (v <= 2 ? 2 : 4);
}

template <typename WT>
cudaError_t launch_sel_t(const StepLaunch& a, cudaStream_t st, cudaEvent_t after_count) {
  const int N = a.B * a.Wc;
  if (N == 0 || a.nch == 0) return cudaSuccess;
  const int bper = item_block_beams(N);
  cudaError_t e = launch_pdl(k_beam_items, (unsigned)((N + bper - 1) / bper), 256, 0, st, a);
  if (e != cudaSuccess) return e;
  if (after_count) cudaEventRecord(after_count, st);
  // persistent: as many CTAs as are resident at once (the occupancy of this
  // instantiation), each warp one contiguous range of the items; fewer when
  // there cannot be that many items
  const int64_t items = (int64_t)N * a.nch;
  auto launch = [&](auto kern) {
    static int resident = 0;  // per instantiation
    if (!resident) {
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
      resident = per_sm * sm_count();
    }
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((items + 7) / 8, (int64_t)resident));
    return launch_pdl(kern, (unsigned)blocks, 256, 0, st, a);
  };
  switch (vpl_for<WT>(a.d)) {
    case 1:
      return launch(k_selective<WT, 1>);
    case 2:
      return launch(k_selective<WT, 2>);
    default:
      return launch(k_selective<WT, 4>);
  }
}

template <typename WT, int VPL>
cudaError_t launch_cluster_vpl(const MegaArgs& A, int B, int G, cudaStream_t st) {
  auto kern = k_decode_cluster<WT, VPL>;
  const size_t smem = (size_t)A.cap * 4 + (size_t)A.pcap * 12;
  static bool attr_done = false;  // per instantiation
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * G));
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)G;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, A);
}

template <typename WT>
cudaError_t launch_cluster_t(const MegaArgs& A, int B, int G, int d, cudaStream_t st) {
  switch (vpl_for<WT>(d)) {
    case 1:
      return launch_cluster_vpl<WT, 1>(A, B, G, st);
    case 2:
      return launch_cluster_vpl<WT, 2>(A, B, G, st);
    default:
      return launch_cluster_vpl<WT, 4>(A, B, G, st);
  }
}

}  // namespace

int sm_count() {
  static int n = 0;
  if (!n) {
    int dv = 0;
    cudaGetDevice(&dv);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dv);
    if (n <= 0) n = 148;
  }
  return n;
}

cudaError_t launch_selective(const StepLaunch& a, cudaStream_t st, cudaEvent_t after_count) {
  switch (a.w_dtype) {
    case ZG_F32:
      return launch_sel_t<float>(a, st, after_count);
    case ZG_BF16:
      return launch_sel_t<__nv_bfloat16>(a, st, after_count);
    default:
      return launch_sel_t<__half>(a, st, after_count);
  }
}

namespace {
__global__ void k_delay(unsigned long long ns) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int i = 0; i < (1 << 20); ++i) {  // 2^20 sleeps of at least 1 us: the bound, if the timer stalls
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= ns) break;
    __nanosleep(1000);
  }
}
}  // namespace

cudaError_t launch_delay(unsigned long long ns, cudaStream_t st) {
  k_delay<<<1, 1, 0, st>>>(ns);
  return cudaGetLastError();
}

cudaError_t launch_decode_cluster(const StepLaunch* steps, int s0, int L, int G, const PrefetchRegion* pf, int npf,
                                  cudaStream_t st) {
  MegaArgs A{};
  A.s0 = s0;
  A.L = L;
  A.cap = kClusterCap;
  A.pcap = kClusterPcap;
  A.npf = std::min(npf, kMaxPrefetch);
  for (int i = 0; i < A.npf; ++i) {
    A.pf[i] = pf[i];
    A.pf[i].bytes &= ~15ull;  // bulk prefetch sizes are multiples of 16 bytes
    A.pf_total += A.pf[i].bytes;
  }
  for (int s = 0; s < L; ++s) A.st[s] = steps[s];
  const StepLaunch& a = steps[L - 1];
  switch (a.w_dtype) {
    case ZG_F32:
      return launch_cluster_t<float>(A, a.B, G, a.d, st);
    case ZG_BF16:
      return launch_cluster_t<__nv_bfloat16>(A, a.B, G, a.d, st);
    default:
      return launch_cluster_t<__half>(A, a.B, G, a.d, st);
  }
}

cudaError_t launch_gather_add(const StepLaunch& a, float* H, cudaStream_t st) {
  const int N = a.B * a.Wc;
  const int blocks = std::max(1, std::min((N + 7) / 8, sm_count() * 16));
  k_gather_add<<<blocks, 256, 0, st>>>(a, H);
  return cudaGetLastError();
}

cudaError_t launch_full_simt(const StepLaunch& a, const float* H, const FullEpi& epi, cudaStream_t st) {
  const int M = a.B * a.Wc;
  dim3 grid((a.V + 63) / 64, (M + 63) / 64);
  switch (a.w_dtype) {
    case ZG_F32:
      k_full_simt<float><<<grid, 256, 0, st>>>(H, static_cast<const float*>(a.W), a.Z, M, a.V, a.d, a.S, epi);
      break;
    case ZG_BF16:
      k_full_simt<__nv_bfloat16><<<grid, 256, 0, st>>>(H, static_cast<const __nv_bfloat16*>(a.W), a.Z, M, a.V,
                                                       a.d, a.S, epi);
      break;
    default:
      k_full_simt<__half><<<grid, 256, 0, st>>>(H, static_cast<const __half*>(a.W), a.Z, M, a.V, a.d, a.S, epi);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_select(const StepLaunch& a, cudaStream_t st) {
  static bool attr_done = false;
  const size_t smem = (size_t)kSelCap * 4;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  return launch_pdl(k_select, (unsigned)a.B, kSelThreads, smem, st, a);
}

cudaError_t launch_trace_touch(const StepLaunch& a, unsigned long long* counters, uint32_t* mask, cudaStream_t st) {
  const int N = a.B * a.Wc;
  const int blocks = std::max(1, std::min((N + 7) / 8, sm_count() * 8));
  k_trace_touch<<<blocks, 256, 0, st>>>(a, counters, mask);
  return cudaGetLastError();
}

cudaError_t launch_legal_mask(const StepLaunch& a, cudaStream_t st) {
  const int N = a.B * a.Wc;
  const int blocks = std::max(1, std::min((N + 7) / 8, sm_count() * 8));
  k_legal_mask<<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t status_word(uint32_t** dev_ptr) { return cudaGetSymbolAddress((void**)dev_ptr, g_status); }

}  // namespace zg
