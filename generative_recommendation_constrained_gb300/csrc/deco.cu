// A light causal decoder producing each step's hidden vectors.
//
// "Separating Thinking from Spelling for Efficient Generative Recommendation"
// (AI Papers Daily digest): the backbone emits a fixed-size next-item concept
// once; a light 2-layer, 256-wide causal decoder conditioned on the concept
// and the generated prefix runs the trie-constrained beam search, so only the
// light decoder takes part in decoding.
//
// At step s every live beam contributes one new sequence position: the M
// concept positions of its request at s = 1 (computed once, shared by the
// request's beams), the embedding of its token of step s-1 afterwards.  Keys
// and values of a position are stored where the position was created: the
// concept rows per request, a token row at [step][beam entering that step].
// A beam attends to its request's concept rows and to the rows of its own
// ancestors, found by following the parent indices of the beam history, so no
// key/value rows are copied when the select reorders beams.
//
// Kernels: embedding, row RMS normalisation, a tiled fp32 GEMM (rows x W^T,
// optional accumulate / ReLU), causal multi-head attention over the gathered
// positions.
#include "zg_internal.h"

namespace zg {
namespace {

constexpr float kRmsEps = 1e-6f;

// X rows of the new positions: concept m of request q plus P[m] at s = 1
// (row q*M + m); E_{s-1}[token] plus P[M + s - 2] for every beam b entering
// step s >= 2 (zero for a dead beam).
__global__ void __launch_bounds__(256) k_deco_embed(const DecoStep a, const zg_deco w) {
  const int rows = (a.s == 1) ? a.B * a.M : a.B * a.Wc;
  const int d4 = a.d / 4;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < (size_t)rows * d4;
       i += (size_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / d4), e = (int)(i - (size_t)r * d4);
    float4 x, p;
    if (a.s == 1) {
      const int m = r % a.M;
      x = reinterpret_cast<const float4*>(a.concepts + (size_t)r * a.d)[e];
      p = reinterpret_cast<const float4*>(w.P + (size_t)m * a.d)[e];
    } else {
      if (a.cum_in[r] == -INFINITY) {
        reinterpret_cast<float4*>(a.X + (size_t)r * a.d)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const int t = a.tok_in[r];
      x = reinterpret_cast<const float4*>(w.E[a.s - 2] + (size_t)t * a.d)[e];
      p = reinterpret_cast<const float4*>(w.P + (size_t)(a.M + a.s - 2) * a.d)[e];
    }
    reinterpret_cast<float4*>(a.X + (size_t)r * a.d)[e] = make_float4(x.x + p.x, x.y + p.y, x.z + p.z, x.w + p.w);
  }
}

// out[i] = X[src(i)] / sqrt(mean(X[src(i)]^2) + eps), src(i) = i * sstride + soff.
// One warp a row.
__global__ void __launch_bounds__(256) k_rms_rows(const float* __restrict__ X, float* __restrict__ out, int rows,
                                                  int d, int sstride, int soff) {
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int i = wid; i < rows; i += nw) {
    const float* x = X + ((size_t)i * sstride + soff) * d;
    float ss = 0.f;
    for (int e = lane; e < d; e += 32) ss = fmaf(x[e], x[e], ss);
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    const float inv = rsqrtf(ss / (float)d + kRmsEps);
    for (int e = lane; e < d; e += 32) out[(size_t)i * d + e] = x[e] * inv;
  }
}

// C[r][n] (+)= sum_k A[r][k] W[n][k] (fp32), optional ReLU of the result.
// 64 x 64 tile, k-slab 16, 256 threads with 4 x 4 outputs each; K % 4 == 0.
__global__ void __launch_bounds__(256) k_gemm_xwt(const float* __restrict__ A, const float* __restrict__ W,
                                                  float* __restrict__ Cm, int R, int N, int K, int accumulate,
                                                  int relu) {
  // 64 x 64 output tile, 4 x 4 a thread; K in tiles of 32 staged transposed in
  // shared memory, the next tile's loads in flight (registers) while the
  // current one is multiplied.  K is a multiple of 4 (rows 16-byte aligned).
  constexpr int BM = 64, BN = 64, BK = 32;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int lr = tid >> 3, kq = (tid & 7) * 4;  // staging: rows lr and lr + 32, columns kq..kq+3
  float4 x[2], y[2];
  auto load = [&](int k0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = lr + 32 * h;
      x[h] = make_float4(0.f, 0.f, 0.f, 0.f);
      y[h] = x[h];
      if (m0 + r < R && k0 + kq < K) x[h] = *reinterpret_cast<const float4*>(A + (size_t)(m0 + r) * K + k0 + kq);
      if (n0 + r < N && k0 + kq < K) y[h] = *reinterpret_cast<const float4*>(W + (size_t)(n0 + r) * K + k0 + kq);
    }
  };
  float acc[4][4] = {};
  load(0);
  for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = lr + 32 * h;
      As[kq][r] = x[h].x;
      As[kq + 1][r] = x[h].y;
      As[kq + 2][r] = x[h].z;
      As[kq + 3][r] = x[h].w;
      Bs[kq][r] = y[h].x;
      Bs[kq + 1][r] = y[h].y;
      Bs[kq + 2][r] = y[h].z;
      Bs[kq + 3][r] = y[h].w;
    }
    __syncthreads();
    if (k0 + BK < K) load(k0 + BK);
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
    if (m >= R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc[i][j];
      if (accumulate) v += Cm[(size_t)m * N + n];
      if (relu) v = fmaxf(v, 0.f);
      Cm[(size_t)m * N + n] = v;
    }
  }
}

constexpr int kMaxPos = 8 + ZG_MAX_STEPS;  // concept positions + token positions

// O[row] = causal multi-head attention of Q[row] over the row's visible
// positions.  One warp per (row, head).  Step 1 (concept rows, row = q*M + m):
// the request's concept rows 0..m.  Step s >= 2 (row = beam b entering step
// s): the request's M concept rows, then the token rows of b's ancestors
// entering steps 2..s-1, then b's own row.
__global__ void __launch_bounds__(256) k_deco_attn(const DecoStep a, int layer) {
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int rows = (a.s == 1) ? a.B * a.M : a.B * a.Wc;
  const int dh = a.d / a.heads;
  const float scale = rsqrtf((float)dh);
  const size_t cstride = (size_t)a.B * a.M * a.d;                 // one layer of concept rows
  const size_t sstride = (size_t)a.B * a.beam * a.d;              // one step of token rows
  const float* Kc = a.Kc + layer * cstride;
  const float* Vc = a.Vc + layer * cstride;
  const float* Ks = a.Ks + (size_t)layer * (a.L + 1) * sstride;
  const float* Vs = a.Vs + (size_t)layer * (a.L + 1) * sstride;
  for (int it = wid; it < rows * a.heads; it += nw) {
    const int row = it / a.heads, h = it - row * a.heads;
    const float* kp[kMaxPos];
    const float* vp[kMaxPos];
    int np = 0;
    if (a.s == 1) {
      const int q = row / a.M, m = row - q * a.M;
      for (int j = 0; j <= m; ++j) {
        kp[np] = Kc + (size_t)(q * a.M + j) * a.d;
        vp[np] = Vc + (size_t)(q * a.M + j) * a.d;
        ++np;
      }
    } else {
      const int q = row / a.Wc;
      for (int j = 0; j < a.M; ++j) {
        kp[np] = Kc + (size_t)(q * a.M + j) * a.d;
        vp[np] = Vc + (size_t)(q * a.M + j) * a.d;
        ++np;
      }
      // ancestors: anc[s] = row; the parent of the beam entering step t + 1
      // is par_hist[t-1][it] of the beams entering step t
      int anc[ZG_MAX_STEPS + 1];
      anc[a.s] = row;
      for (int t = a.s - 1; t >= 2; --t) anc[t] = q * a.beam + a.par_hist[(size_t)(t - 1) * a.B * a.beam + anc[t + 1]];
      for (int t = 2; t <= a.s; ++t) {
        kp[np] = Ks + (size_t)t * sstride + (size_t)anc[t] * a.d;
        vp[np] = Vs + (size_t)t * sstride + (size_t)anc[t] * a.d;
        ++np;
      }
    }
    const float* qr = a.Q + (size_t)row * a.d + h * dh;
    float sc[kMaxPos];
    float mx = -INFINITY;
    for (int j = 0; j < np; ++j) {
      float p = 0.f;
      for (int e = lane; e < dh; e += 32) p = fmaf(qr[e], kp[j][h * dh + e], p);
#pragma unroll
      for (int o = 16; o; o >>= 1) p += __shfl_xor_sync(0xFFFFFFFFu, p, o);
      sc[j] = p * scale;
      mx = fmaxf(mx, sc[j]);
    }
    float den = 0.f;
    for (int j = 0; j < np; ++j) {
      sc[j] = expf(sc[j] - mx);
      den += sc[j];
    }
    const float inv = 1.f / den;
    for (int e = lane; e < dh; e += 32) {
      float o = 0.f;
      for (int j = 0; j < np; ++j) o = fmaf(sc[j], vp[j][h * dh + e], o);
      a.O[(size_t)row * a.d + h * dh + e] = o * inv;
    }
  }
}

int grid_for(size_t work, int per_block) {
  const size_t b = (work + per_block - 1) / per_block;
  return (int)std::max<size_t>(1, std::min<size_t>(b, (size_t)sm_count() * 8));
}

cudaError_t gemm(const float* A, const float* W, float* Cm, int R, int N, int K, bool acc, bool relu,
                 cudaStream_t st) {
  dim3 grid((N + 63) / 64, (R + 63) / 64);
  k_gemm_xwt<<<grid, 256, 0, st>>>(A, W, Cm, R, N, K, acc ? 1 : 0, relu ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_deco_step(const zg_deco& w, const DecoStep& a, cudaStream_t st) {
  const int rows = (a.s == 1) ? a.B * a.M : a.B * a.Wc;
  const size_t cstride = (size_t)a.B * a.M * a.d;
  const size_t sstride = (size_t)a.B * a.beam * a.d;
  k_deco_embed<<<grid_for((size_t)rows * a.d / 4, 256), 256, 0, st>>>(a, w);
  cudaError_t e = cudaGetLastError();
  for (int l = 0; l < w.layers && e == cudaSuccess; ++l) {
    float* Kdst = (a.s == 1) ? a.Kc + l * cstride : a.Ks + ((size_t)l * (a.L + 1) + a.s) * sstride;
    float* Vdst = (a.s == 1) ? a.Vc + l * cstride : a.Vs + ((size_t)l * (a.L + 1) + a.s) * sstride;
    k_rms_rows<<<grid_for((size_t)rows * 32, 256), 256, 0, st>>>(a.X, a.A, rows, a.d, 1, 0);
    if ((e = cudaGetLastError()) != cudaSuccess) break;
    if ((e = gemm(a.A, w.Wq[l], a.Q, rows, a.d, a.d, false, false, st)) != cudaSuccess) break;
    if ((e = gemm(a.A, w.Wk[l], Kdst, rows, a.d, a.d, false, false, st)) != cudaSuccess) break;
    if ((e = gemm(a.A, w.Wv[l], Vdst, rows, a.d, a.d, false, false, st)) != cudaSuccess) break;
    k_deco_attn<<<grid_for((size_t)rows * w.heads * 32, 256), 256, 0, st>>>(a, l);
    if ((e = cudaGetLastError()) != cudaSuccess) break;
    if ((e = gemm(a.O, w.Wo[l], a.X, rows, a.d, a.d, true, false, st)) != cudaSuccess) break;
    k_rms_rows<<<grid_for((size_t)rows * 32, 256), 256, 0, st>>>(a.X, a.A, rows, a.d, 1, 0);
    if ((e = cudaGetLastError()) != cudaSuccess) break;
    if ((e = gemm(a.A, w.W1[l], a.F, rows, w.ffn, a.d, false, true, st)) != cudaSuccess) break;
    if ((e = gemm(a.F, w.W2[l], a.X, rows, a.d, w.ffn, true, false, st)) != cudaSuccess) break;
  }
  if (e != cudaSuccess) return e;
  // hidden vectors: the last concept row of each request at s = 1, every beam's row after
  const int nh = (a.s == 1) ? a.B : rows;
  k_rms_rows<<<grid_for((size_t)nh * 32, 256), 256, 0, st>>>(a.X, a.H, nh, a.d, (a.s == 1) ? a.M : 1,
                                                               (a.s == 1) ? a.M - 1 : 0);
  return cudaGetLastError();
}

}  // namespace zg
