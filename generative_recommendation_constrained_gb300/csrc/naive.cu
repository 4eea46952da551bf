// Naive legal-only scoring, kept as a measured contrast to the padded slots.
//
// "ZeroGR: Filtering-First Constrained Decoding for Generative
// Recommendation" (paper-daily.com digest), section "Why computing fewer
// scores is not automatically faster" and its figure "compact list vs padded
// slots" (paper section 4 / Figure 9): scoring only the legal tokens the
// straightforward way first compacts every beam's candidates into one list
// (a candidate's place depends on the fan-outs of all beams before it) and
// builds a temporary matrix; the paper measures it 5.1x slower than scoring
// every token, and the padded slots 8.5x faster than it.
//
// The compaction here is a fan-out count, an exclusive scan and a list of
// (beam, slot, token); the temporary matrix is the listed tokens' weight
// rows copied out; each score is then one row of it times the beam's hidden
// vector, written to the beam's padded slot so the ordinary select follows.
#include <algorithm>

#include "zg_device.cuh"

namespace zg {
namespace {

using namespace dev;

// Fan-out of every beam of the step (0 for a dead beam).
__global__ void __launch_bounds__(256) k_naive_count(const __grid_constant__ StepLaunch a, int32_t* cnt) {
  const int N = a.B * a.Wc;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < N; b += gridDim.x * blockDim.x) {
    const int q = b / a.Wc, k = b - q * a.Wc;
    const BeamState bs = load_beam(a, q, k);
    int F = 0;
    if (bs.row != kDeadRow) {
      if (bs.row >= a.tab.rows)
        flag(a.status, kStatusRow);
      else
        F = (int)(a.tab.rowptr[bs.row + 1] - a.tab.rowptr[bs.row]);
    }
    cnt[b] = F;
  }
}

// Exclusive prefix sum off[0..N] of cnt[0..N) by one CTA (off[N] = total).
__global__ void __launch_bounds__(1024) k_naive_scan(const int32_t* cnt, int32_t* off, int N) {
  __shared__ int wsum[32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int per = (N + 1023) / 1024;
  const int lo = min(N, t * per), hi = min(N, lo + per);
  int mine = 0;
  for (int i = lo; i < hi; ++i) mine += cnt[i];
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  int run = base + incl - mine;
  for (int i = lo; i < hi; ++i) {
    off[i] = run;
    run += cnt[i];
  }
  if (t == 1023) off[N] = base + incl;
}

// The compact list: (beam, slot, token) of every legal candidate in beam
// order, one warp per beam.  Sparse steps: slot j is the j-th column entry;
// dense steps: slot = token, the row's set bits in ascending order.
__global__ void __launch_bounds__(256) k_naive_list(const __grid_constant__ StepLaunch a, const int32_t* off,
                                                    int4* list, int64_t cap) {
  const int lane = threadIdx.x & 31;
  const int N = a.B * a.Wc;
  for (int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < N; b += (gridDim.x * blockDim.x) >> 5) {
    const int F = off[b + 1] - off[b];
    if (F == 0) continue;
    if ((int64_t)off[b + 1] > cap) {  // more candidates than the workspace was sized for
      if (lane == 0) flag(a.status, kStatusRow);
      continue;
    }
    const int q = b / a.Wc, k = b - q * a.Wc;
    const BeamState bs = load_beam(a, q, k);
    const uint32_t rp = a.tab.rowptr[bs.row];
    int4* out = list + off[b];
    if (a.tab.fmt == ZG_FMT_SPARSE) {
      for (int j = lane; j < F; j += 32) out[j] = make_int4(b, j, (int)a.tab.col[rp + j], 0);
    } else {
      const uint32_t* bm = a.tab.bitmap + (size_t)bs.row * a.tab.words;
      int base = 0;
      for (int w0 = 0; w0 < (int)a.tab.words; w0 += 32) {
        const uint32_t bits = (w0 + lane < (int)a.tab.words) ? bm[w0 + lane] : 0u;
        const int c = __popc(bits);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += y;
        }
        int pos = base + incl - c;
        for (uint32_t x = bits; x; x &= x - 1u) {
          const int t = (w0 + lane) * 32 + __ffs(x) - 1;
          if (pos < F) out[pos] = make_int4(b, t, t, 0);
          ++pos;
        }
        base += __shfl_sync(kFull, incl, 31);
      }
    }
  }
}

// The temporary matrix: row i = the weight row of the i-th listed token.
__global__ void __launch_bounds__(256) k_naive_gather(const __grid_constant__ StepLaunch a, const int4* list,
                                                      const int32_t* total, uint4* temp, int64_t cap) {
  const int lane = threadIdx.x & 31;
  const int n = (int)min((int64_t)*total, cap);
  const int row16 = a.d * (a.w_dtype == ZG_F32 ? 4 : 2) / 16;  // 16-byte pieces a row
  const uint4* W = static_cast<const uint4*>(a.W);
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += (gridDim.x * blockDim.x) >> 5) {
    const int t = list[i].z;
    if (t < 0 || t >= a.V) continue;  // a row left unlisted after a capacity flag
    for (int v = lane; v < row16; v += 32) temp[(size_t)i * row16 + v] = W[(size_t)t * row16 + v];
  }
}

// Scores: z_i = temp_i . h_beam(i), written to the beam's padded slot.
template <typename WT>
__global__ void __launch_bounds__(256) k_naive_dot(const __grid_constant__ StepLaunch a, const int4* list,
                                                   const int32_t* total, const uint4* temp, const float* H,
                                                   int64_t cap) {
  using VT = Vec<WT>;
  constexpr int E = VT::E;
  const int lane = threadIdx.x & 31;
  const int n = (int)min((int64_t)*total, cap);
  const int nvec = a.d / E;
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += (gridDim.x * blockDim.x) >> 5) {
    const int4 c = list[i];
    if (c.x < 0 || c.x >= a.B * a.Wc || c.y < 0 || c.y >= a.S || c.z < 0 || c.z >= a.V) continue;
    const float* h = H + (size_t)c.x * a.d;
    float acc = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      float w[E];
      VT::cvt(temp[(size_t)i * nvec + v], w);
#pragma unroll
      for (int e = 0; e < E; ++e) acc = fmaf(w[e], h[v * E + e], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      const int q = c.x / a.Wc, k = c.x - q * a.Wc;
      a.Z[(size_t)q * a.zq + (size_t)k * a.S + c.y] = acc;
    }
  }
}

}  // namespace

cudaError_t launch_naive_compact(const StepLaunch& a, int32_t* cnt, int32_t* off, int4* list, void* temp,
                                 int64_t cap, cudaStream_t st) {
  const int N = a.B * a.Wc;
  const int blocks = std::max(1, std::min((N + 255) / 256, sm_count() * 4));
  k_naive_count<<<blocks, 256, 0, st>>>(a, cnt);
  k_naive_scan<<<1, 1024, 0, st>>>(cnt, off, N);
  const int wblocks = std::max(1, std::min((N + 7) / 8, sm_count() * 8));
  k_naive_list<<<wblocks, 256, 0, st>>>(a, off, list, cap);
  k_naive_gather<<<sm_count() * 8, 256, 0, st>>>(a, list, off + N, static_cast<uint4*>(temp), cap);
  return cudaGetLastError();
}

cudaError_t launch_naive_dot(const StepLaunch& a, const int32_t* off, const int4* list, const void* temp,
                             const float* H, int64_t cap, cudaStream_t st) {
  const int N = a.B * a.Wc;
  const uint4* t = static_cast<const uint4*>(temp);
  if (a.w_dtype == ZG_F32)
    k_naive_dot<float><<<sm_count() * 8, 256, 0, st>>>(a, list, off + N, t, H, cap);
  else if (a.w_dtype == ZG_BF16)
    k_naive_dot<__nv_bfloat16><<<sm_count() * 8, 256, 0, st>>>(a, list, off + N, t, H, cap);
  else
    k_naive_dot<__half><<<sm_count() * 8, 256, 0, st>>>(a, list, off + N, t, H, cap);
  return cudaGetLastError();
}

}  // namespace zg
