// Decode engine: argument checks, workspace layout, per-step kernel
// sequence, per-step variant tuning, and the C ABI around them.
//
// "ZeroGR: Filtering-First Constrained Decoding for Generative
// Recommendation" (paper-daily.com digest):
//   "Overall flow": the online engine runs four stages per decoding step;
//   "Why computing fewer scores is not automatically faster", last part:
//     before serving, warm-up requests time the variants of every step and
//     the fastest is kept until the next model update;
//   "Is the scheme really better": the unconstrained decode scores every
//     token at every step and serves as the speed reference.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "zg_internal.h"

namespace zg {

namespace {
thread_local std::string g_err;

int esize(int dt) { return dt == ZG_F32 ? 4 : 2; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Dims {
  int L, V, d, w_dtype, B, beam, K;
  bool constrained;
  bool score_first;      // ZG_ORDER_SCORE_FIRST plan
  bool naive[ZG_MAX_STEPS];  // ZG_NAIVE steps of the plan
  size_t naive_rows;     // listed candidates the naive steps' workspace holds
  int64_t nnz[ZG_MAX_STEPS];
  int S_full;            // padded token stride of full scores
  int nch_sel[ZG_MAX_STEPS];
  int S_sel[ZG_MAX_STEPS];
  bool tops[ZG_MAX_STEPS];   // a full step hands chunk tops (no written scores) to the select
  bool split_h;              // half weights: the hidden as hi + lo operands
  bool need_mask;            // per-beam legal bitmaps (score-first, or chunk tops on sparse tables)
  bool sparse[ZG_MAX_STEPS]; // the step's table is sparse (constrained)
  const zg_deco* deco;       // light decoder producing the hidden vectors, or null
  int dM, dffn, dlayers;     // its concept vectors, MLP width, layers
};

// The automatic choice of how a full step hands its scores to the select:
// written.  Chunk tops save the score stores (~9 us of a 69 us tensor-core
// step at the dense-early catalogue's step 2) but their select, which
// re-scores chunks from the weights, measured slower on every configuration
// (dense early, the unconstrained decodes of the large catalogue), so they
// are used only when a plan asks for them.
bool auto_tops(const Dims&, int) { return false; }

struct WsLayout {
  size_t dX, dA, dQ, dO, dF, dKc, dVc, dKs, dVs, dH;  // light decoder
  size_t bscan;
  size_t tok_hist, par_hist, row[2], cum[2], h[2], hhi, hlo, Z, part, ptop, part_all, mask, naive_cnt, naive_off,
      naive_list, naive_temp, trace, u_stage, o_sids, o_scores, total;
  size_t trace_bytes;
};

WsLayout layout(const Dims& m, bool host_io) {
  WsLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align256(off + std::max<size_t>(bytes, 1));
    return o;
  };
  const size_t BW = (size_t)m.B * m.beam;
  const size_t hist = (size_t)std::max(m.L - 1, 1) * BW * 4;
  w.tok_hist = take(hist);
  w.par_hist = take(hist);
  for (int i = 0; i < 2; ++i) {
    w.row[i] = take(BW * 4);
    w.cum[i] = take(BW * 4);
    w.h[i] = take(BW * m.d * 4);
  }
  const size_t half_bytes = (m.w_dtype == ZG_F32) ? 0 : BW * m.d * 2;  // tensor-core operand halves
  w.hhi = take(half_bytes);
  w.hlo = take(half_bytes);
  size_t zf = 0, pf = 0;
  for (int s = 1; s <= m.L; ++s) {
    const size_t N = (size_t)m.B * (s == 1 ? 1 : m.beam);
    size_t S = m.tops[s - 1] ? 0 : m.S_full;       // full scores are written only without chunk tops
    pf = std::max(pf, N * (m.S_full / kChunk));  // full-projection chunk partials
    if (m.constrained) {
      S = std::max<size_t>(S, m.S_sel[s - 1]);
      pf = std::max(pf, N * m.nch_sel[s - 1]);
    }
    zf = std::max(zf, N * S);
  }
  w.Z = take(zf * 4);
  w.part = take(pf * 8);
  w.ptop = take(pf * 8);
  if (m.score_first) w.part_all = take(BW * (m.S_full / kChunk) * 8);  // codebook-wide partials
  if (m.need_mask) w.mask = take(BW * (size_t)((m.V + 31) / 32) * 4);  // per-beam token bitmaps
  if (m.naive_rows) {  // fan-outs, offsets, compact list, temporary matrix
    w.naive_cnt = take((BW + 1) * 4);
    w.naive_off = take((BW + 1) * 4);
    w.naive_list = take(m.naive_rows * 16);
    w.naive_temp = take(m.naive_rows * (size_t)m.d * esize(m.w_dtype));
  }
  if (m.deco) {  // work rows, keys and values by position, hidden vectors
    const size_t rows = std::max((size_t)m.B * m.dM, BW);
    w.dX = take(rows * m.d * 4);
    w.dA = take(rows * m.d * 4);
    w.dQ = take(rows * m.d * 4);
    w.dO = take(rows * m.d * 4);
    w.dF = take(rows * (size_t)m.dffn * 4);
    w.dKc = take((size_t)m.dlayers * m.B * m.dM * m.d * 4);
    w.dVc = take((size_t)m.dlayers * m.B * m.dM * m.d * 4);
    w.dKs = take((size_t)m.dlayers * (m.L + 1) * BW * m.d * 4);
    w.dVs = take((size_t)m.dlayers * (m.L + 1) * BW * m.d * 4);
    w.dH = take(BW * m.d * 4);
  }
  w.bscan = take((3 * BW + kItemBlocks) * 4);  // stand-alone selective steps: chunk offsets, first entries, fan-outs, CTA totals
  w.trace_bytes = 32 + (size_t)((m.V + 31) / 32) * 4;  // 4 counters + token mask
  w.trace = take(w.trace_bytes);
  if (host_io) {
    w.u_stage = take((size_t)m.B * (m.deco ? m.dM : 1) * m.d * 4);
    w.o_sids = take((size_t)m.B * m.K * m.L * 4);
    w.o_scores = take((size_t)m.B * m.K * 4);
  }
  w.total = off;
  return w;
}

zg_status check_common(const zg_index* idx, const zg_model* model, int B, int beam, int K, Dims* out) {
  if (!model) return fail(ZG_ERR_INVALID_ARG, "model is NULL");
  const zg_model& m = *model;
  if (m.L < 1 || m.L > ZG_MAX_STEPS) return fail(ZG_ERR_INVALID_ARG, "model.L must be in [1, 8]");
  if (m.V < 1 || m.V > 65536) return fail(ZG_ERR_INVALID_ARG, "model.V must be in [1, 65536]");
  if (m.w_dtype != ZG_F32 && m.w_dtype != ZG_BF16 && m.w_dtype != ZG_F16)
    return fail(ZG_ERR_INVALID_ARG, "model.w_dtype must be ZG_F32, ZG_BF16 or ZG_F16");
  if (m.d < 8 || m.d % 8 != 0 || m.d * esize(m.w_dtype) > 2048)
    return fail(ZG_ERR_INVALID_ARG, "model.d must be a multiple of 8 with d * sizeof(weight) <= 2048");
  for (int s = 0; s < m.L; ++s) {
    if (!m.W[s]) return fail(ZG_ERR_INVALID_ARG, "model.W[s] is NULL");
    if (reinterpret_cast<uintptr_t>(m.W[s]) % 16) return fail(ZG_ERR_INVALID_ARG, "model.W[s] not 16-byte aligned");
    if (s < m.L - 1 && !m.deco) {
      if (!m.C[s]) return fail(ZG_ERR_INVALID_ARG, "model.C[s] is NULL");
      if (reinterpret_cast<uintptr_t>(m.C[s]) % 16) return fail(ZG_ERR_INVALID_ARG, "model.C[s] not 16-byte aligned");
    }
  }
  if (B < 1) return fail(ZG_ERR_INVALID_ARG, "B must be >= 1");
  if (beam < 1 || beam > ZG_MAX_BEAM) return fail(ZG_ERR_INVALID_ARG, "beam must be in [1, 512]");
  if (K < 1 || K > beam) return fail(ZG_ERR_INVALID_ARG, "K must be in [1, beam]");
  if (idx) {
    if (idx->residency != ZG_RESIDENT_DEVICE || !idx->dev)
      return fail(ZG_ERR_INVALID_ARG, "index is host-resident; build or load it with ZG_RESIDENT_DEVICE");
    if (idx->L != m.L || idx->V != m.V) return fail(ZG_ERR_INVALID_ARG, "index and model disagree on L or V");
  }
  if (m.deco) {
    const zg_deco& w = *m.deco;
    if (w.M < 1 || w.M > 8) return fail(ZG_ERR_INVALID_ARG, "deco.M must be in [1, 8]");
    if (w.layers < 1 || w.layers > ZG_MAX_DECO_LAYERS) return fail(ZG_ERR_INVALID_ARG, "deco.layers must be in [1, 4]");
    if (w.heads < 1 || m.d % w.heads != 0 || m.d / w.heads > 256)
      return fail(ZG_ERR_INVALID_ARG, "deco.heads must divide d with d / heads <= 256");
    if (w.ffn < 4 || w.ffn % 4 != 0) return fail(ZG_ERR_INVALID_ARG, "deco.ffn must be a positive multiple of 4");
    auto bad = [](const float* p) { return !p || reinterpret_cast<uintptr_t>(p) % 16; };
    if (bad(w.P)) return fail(ZG_ERR_INVALID_ARG, "deco.P is NULL or not 16-byte aligned");
    for (int s = 0; s < m.L - 1; ++s)
      if (bad(w.E[s])) return fail(ZG_ERR_INVALID_ARG, "deco.E[s] is NULL or not 16-byte aligned");
    for (int l = 0; l < w.layers; ++l)
      if (bad(w.Wq[l]) || bad(w.Wk[l]) || bad(w.Wv[l]) || bad(w.Wo[l]) || bad(w.W1[l]) || bad(w.W2[l]))
        return fail(ZG_ERR_INVALID_ARG, "deco weight matrix is NULL or not 16-byte aligned");
  }
  Dims d{};
  d.deco = m.deco;
  if (m.deco) {
    d.dM = m.deco->M;
    d.dffn = m.deco->ffn;
    d.dlayers = m.deco->layers;
  }
  d.L = m.L;
  d.V = m.V;
  d.d = m.d;
  d.w_dtype = m.w_dtype;
  d.B = B;
  d.beam = beam;
  d.K = K;
  d.constrained = idx != nullptr;
  d.S_full = (m.V + kChunk - 1) / kChunk * kChunk;
  for (int s = 1; s <= m.L; ++s) {
    int nch = 0;
    if (idx) {
      const StepMeta& sm = idx->steps[s - 1];
      nch = sm.fmt == ZG_FMT_SPARSE ? (int)((sm.max_fanout + kChunk - 1) / kChunk) : (m.V + kChunk - 1) / kChunk;
    }
    d.nch_sel[s - 1] = nch;
    d.S_sel[s - 1] = nch * kChunk;
    d.nnz[s - 1] = idx ? (int64_t)idx->steps[s - 1].nnz : 0;
    d.sparse[s - 1] = idx && idx->steps[s - 1].fmt == ZG_FMT_SPARSE;
  }
  d.split_h = true;
  for (int s = 1; s <= m.L; ++s) d.tops[s - 1] = auto_tops(d, s);
  d.need_mask = false;
  for (int s = 1; s <= m.L; ++s) d.need_mask = d.need_mask || (d.tops[s - 1] && d.sparse[s - 1]);
  *out = d;
  return ZG_OK;
}

// What the plan changes in the decode's shape: the order, and the naive
// steps' workspace (a request's beams are distinct prefixes, so its listed
// candidates are at most min(beams * max_fanout, nnz) of the step).
zg_status apply_plan(Dims& m, const zg_index* idx, const zg_plan* plan) {
  m.score_first = idx && plan && plan->order == ZG_ORDER_SCORE_FIRST;
  if (plan) {
    m.split_h = plan->hidden != ZG_HIDDEN_SINGLE;
    for (int s = 1; s <= m.L; ++s)
      m.tops[s - 1] = plan->scores == ZG_SCORES_CHUNK_TOPS || (plan->scores == ZG_SCORES_AUTO && auto_tops(m, s));
  }
  m.need_mask = m.score_first;
  for (int s = 1; s <= m.L; ++s) m.need_mask = m.need_mask || (m.tops[s - 1] && m.sparse[s - 1]);
  m.naive_rows = 0;
  for (int s = 1; s <= m.L; ++s) {
    m.naive[s - 1] = idx && plan && !m.score_first && plan->variant[s - 1] == ZG_NAIVE;
    if (!m.naive[s - 1]) continue;
    const int64_t Wc = (s == 1) ? 1 : m.beam;
    const int64_t per = std::min<int64_t>(Wc * m.S_sel[s - 1], m.nnz[s - 1]);
    m.naive_rows = std::max<size_t>(m.naive_rows, (size_t)m.B * (size_t)std::max<int64_t>(per, 1));
  }
  if ((double)m.naive_rows * m.d * esize(m.w_dtype) > 16.0 * (1ull << 30))
    return fail(ZG_ERR_UNSUPPORTED, "naive variant: the temporary matrix would exceed 16 GiB; use a smaller batch");
  return ZG_OK;
}

std::mutex g_status_mu;
uint32_t* g_status_ptr[64] = {};
unsigned long long g_status_ctx[64] = {};

zg_status get_status_ptr(uint32_t** p) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(ZG_ERR_UNSUPPORTED, "device ordinal >= 64");
  unsigned long long ctx = 0;
  if ((e = current_context_id(&ctx)) != cudaSuccess) return cuda_fail(e, "current context id");
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev] || g_status_ctx[dev] != ctx) {  // first use, or a new context (device reset)
    e = status_word(&g_status_ptr[dev]);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
    g_status_ctx[dev] = ctx;
  }
  *p = g_status_ptr[dev];
  return ZG_OK;
}

// Everything one decode needs, resolved once.
struct Run {
  Dims m;
  WsLayout w;
  uint8_t* ws;
  const zg_index* idx;
  const zg_model* model;
  const float* u;
  int32_t* out_sids;
  float* out_scores;
  uint32_t* status;
};

// Events around the kernels of one step (tracing only).
struct StepTimer {
  cudaEvent_t ev[4];  // start, after gather-add, after projection, after select
};

StepLaunch make_launch(const Run& r, int s, int variant) {
  const Dims& m = r.m;
  StepLaunch a{};
  a.s = s;
  a.L = m.L;
  a.V = m.V;
  a.d = m.d;
  a.w_dtype = m.w_dtype;
  a.B = m.B;
  a.beam = m.beam;
  a.K = m.K;
  a.Wc = (s == 1) ? 1 : m.beam;
  a.Wp = (s <= 2) ? 1 : m.beam;
  a.keep = (s < m.L) ? m.beam : m.K;
  if (r.idx) a.tab = r.idx->dev_step(s);
  const size_t BW = (size_t)m.B * m.beam;
  auto F32 = [&](size_t off) { return reinterpret_cast<float*>(r.ws + off); };
  auto U32 = [&](size_t off) { return reinterpret_cast<uint32_t*>(r.ws + off); };
  auto I32 = [&](size_t off) { return reinterpret_cast<int32_t*>(r.ws + off); };
  if (s >= 2) {
    const int pi = (s - 1) & 1;
    a.row_in = r.idx ? U32(r.w.row[pi]) : nullptr;
    a.cum_in = F32(r.w.cum[pi]);
    a.par_in = I32(r.w.par_hist) + (size_t)(s - 2) * BW;
    a.tok_in = I32(r.w.tok_hist) + (size_t)(s - 2) * BW;
    a.h_prev = (s == 2) ? r.u : F32(r.w.h[pi]);
    a.C_prev = r.model->C[s - 2];
  }
  if (m.deco) {  // hidden vectors from the light decoder, computed before the step
    a.hpre = F32(r.w.dH);
    a.h_prev = nullptr;
    a.C_prev = nullptr;
  }
  a.u = r.u;
  a.W = r.model->W[s - 1];
  const bool full = (variant == ZG_FULL) || !r.idx || m.score_first;
  const bool naive = !full && variant == ZG_NAIVE;
  // hidden of this step's beams: the next step's parents (s < L) and the
  // full projection's (or naive scores') input; at step 1 it is u itself
  a.h_out = (!m.deco && s >= 2 && (s < m.L || full || naive)) ? F32(r.w.h[s & 1]) : nullptr;
  a.Z = F32(r.w.Z);
  a.row_out = r.idx ? U32(r.w.row[s & 1]) : nullptr;
  a.cum_out = F32(r.w.cum[s & 1]);
  a.tok_hist = I32(r.w.tok_hist);
  a.par_hist = I32(r.w.par_hist);
  a.out_sids = r.out_sids;
  a.out_scores = r.out_scores;
  a.status = r.status;
  if (naive) {
    // scores land in padded slots (sparse: slot = rank, dense: slot = token);
    // no chunk partials: the select computes its log-sum-exp from the slots
    if (r.idx->steps[s - 1].fmt == ZG_FMT_SPARSE) {
      a.mode = kSelSparse;
      a.nch = m.nch_sel[s - 1];
      a.S = m.S_sel[s - 1];
    } else {
      a.mode = kFullDense;
      a.nch = m.S_full / kChunk;
      a.S = m.S_full;
    }
    a.part = nullptr;
  } else if (!full) {
    const StepMeta& sm = r.idx->steps[s - 1];
    a.bscan = I32(r.w.bscan);
    a.mode = sm.fmt == ZG_FMT_SPARSE ? kSelSparse : kSelDense;
    a.nch = m.nch_sel[s - 1];
    a.S = m.S_sel[s - 1];
    a.part = reinterpret_cast<float2*>(r.ws + r.w.part);
  } else if ((m.score_first || m.tops[s - 1]) && r.idx) {
    // token slots with a legal bitmap: the score-first order (project every
    // token, normalise over the codebook, mask, select) and full steps that
    // hand chunk tops to the select; sparse-format steps expand their legal
    // lists into per-beam bitmap rows first
    a.mode = kFullDense;
    a.S = m.S_full;
    a.nch = m.S_full / kChunk;
    a.part = reinterpret_cast<float2*>(r.ws + r.w.part);
    if (m.score_first) a.part_all = reinterpret_cast<const float2*>(r.ws + r.w.part_all);
    if (r.idx->steps[s - 1].fmt == ZG_FMT_SPARSE) {
      a.mask_by_beam = 1;
      a.tab.bitmap = U32(r.w.mask);
      a.tab.words = (uint32_t)((m.V + 31) / 32);
    }
  } else {
    a.mode = !r.idx ? kUncon : (r.idx->steps[s - 1].fmt == ZG_FMT_SPARSE ? kFullSparse : kFullDense);
    a.S = m.S_full;
    if (a.mode == kFullSparse) {  // few legal tokens a beam: the select gathers them
      a.nch = 0;
      a.part = nullptr;
    } else {  // the full projection's epilogue writes chunk partials
      a.nch = m.S_full / kChunk;
      a.part = reinterpret_cast<float2*>(r.ws + r.w.part);
    }
  }
  a.zq = (int64_t)a.Wc * a.S;      // contiguous beam rows (the full projection's layout)
  a.pq = (int64_t)a.Wc * a.nch;
  if (full && m.tops[s - 1]) {
    // no scores written: the select works from the chunk tops and re-scores
    // from the projection's own operands
    a.ptop = reinterpret_cast<const float2*>(r.ws + r.w.ptop);
    a.Z = nullptr;
    const float* H = a.hpre ? a.hpre : ((s >= 2) ? a.h_out : r.u);
    a.hq = H;
    if (m.w_dtype != ZG_F32) {
      a.hq_hi = r.ws + r.w.hhi;
      a.hq_lo = m.split_h ? r.ws + r.w.hlo : nullptr;
    }
  }
  return a;
}

zg_status run_step(const Run& r, int s, int variant, cudaStream_t st, const StepTimer* tm = nullptr) {
  const StepLaunch a = make_launch(r, s, variant);
  cudaError_t e;
  if (tm) cudaEventRecord(tm->ev[0], st);
  if (variant == ZG_NAIVE && r.m.naive[s - 1]) {
    const float* H = a.hpre ? a.hpre : r.u;
    if (s >= 2 && !a.hpre) {
      e = launch_gather_add(a, a.h_out, st);
      if (e != cudaSuccess) return cuda_fail(e, "gather-add launch");
      H = a.h_out;
    }
    auto* cnt = reinterpret_cast<int32_t*>(r.ws + r.w.naive_cnt);
    auto* off = reinterpret_cast<int32_t*>(r.ws + r.w.naive_off);
    auto* list = reinterpret_cast<int4*>(r.ws + r.w.naive_list);
    void* temp = r.ws + r.w.naive_temp;
    e = launch_naive_compact(a, cnt, off, list, temp, (int64_t)r.m.naive_rows, st);
    if (e != cudaSuccess) return cuda_fail(e, "naive compaction launch");
    if (tm) cudaEventRecord(tm->ev[1], st);
    e = launch_naive_dot(a, off, list, temp, H, (int64_t)r.m.naive_rows, st);
    if (e != cudaSuccess) return cuda_fail(e, "naive scoring launch");
  } else if (a.mode == kSelSparse || a.mode == kSelDense) {
    e = launch_selective(a, st, tm ? tm->ev[1] : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "selective projection launch");
  } else {
    const float* H = a.hpre ? a.hpre : r.u;
    if (s >= 2 && !a.hpre) {
      e = launch_gather_add(a, a.h_out, st);
      if (e != cudaSuccess) return cuda_fail(e, "gather-add launch");
      H = a.h_out;
    }
    const int M = a.B * a.Wc;
    void* hlo = r.m.split_h ? r.ws + r.w.hlo : nullptr;  // none: a single rounding of the hidden
    if (a.w_dtype != ZG_F32) {
      e = launch_split_h(H, r.ws + r.w.hhi, hlo, (size_t)M * a.d, a.w_dtype, st);
      if (e != cudaSuccess) return cuda_fail(e, "hidden split launch");
    }
    FullEpi epi{};
    epi.part = a.part;
    epi.ptop = const_cast<float2*>(a.ptop);
    epi.part_all = const_cast<float2*>(a.part_all);
    if (a.mode == kFullDense) {
      epi.bitmap = a.tab.bitmap;
      epi.words = (int)a.tab.words;
      epi.rows = (s >= 2) ? a.row_in : nullptr;  // beam b = q*beam + k at s >= 2; the root's row 0 at s = 1
      epi.nrows = a.tab.rows;
      epi.status = a.status;
      if (a.mask_by_beam) {
        e = launch_legal_mask(a, st);
        if (e != cudaSuccess) return cuda_fail(e, "legal-mask launch");
        epi.by_m = 1;
        epi.nrows = (uint32_t)M;
      }
    }
    if (tm) cudaEventRecord(tm->ev[1], st);
    if (a.w_dtype != ZG_F32)
      e = launch_full_tc(r.ws + r.w.hhi, hlo, a.W, a.Z, M, a.V, a.d, a.S, a.w_dtype, epi, a.status, st);
    else
      e = launch_full_simt(a, H, epi, st);
    if (e != cudaSuccess) return cuda_fail(e, "full projection launch");
  }
  if (tm) cudaEventRecord(tm->ev[2], st);
  e = launch_select(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "select launch");
  if (tm) cudaEventRecord(tm->ev[3], st);
  return ZG_OK;
}

zg_status prepare(const zg_index* idx, const zg_plan* plan, const zg_model* model, const float* u, int B, int beam,
                  int K, int32_t* out_sids, float* out_scores, void* ws, size_t ws_bytes, bool host_io, Run* r) {
  Dims m;
  zg_status st = check_common(idx, model, B, beam, K, &m);
  if (st != ZG_OK) return st;
  if (plan && plan->L != m.L) return fail(ZG_ERR_INVALID_ARG, "plan has a different number of steps");
  if ((st = apply_plan(m, idx, plan)) != ZG_OK) return st;
  if (!u || !out_sids || !out_scores) return fail(ZG_ERR_INVALID_ARG, "u, out_sids and out_scores must not be NULL");
  if (!host_io && reinterpret_cast<uintptr_t>(u) % 16) return fail(ZG_ERR_INVALID_ARG, "u must be 16-byte aligned");
  if (!ws) return fail(ZG_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(ZG_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  WsLayout w = layout(m, host_io);
  if (ws_bytes < w.total) return fail(ZG_ERR_INVALID_ARG, "workspace too small");
  r->m = m;
  r->w = w;
  r->ws = static_cast<uint8_t*>(ws);
  r->idx = idx;
  r->model = model;
  r->u = u;
  r->out_sids = out_sids;
  r->out_scores = out_scores;
  return get_status_ptr(&r->status);
}

// The light decoder's step s: hidden vectors of the beams entering step s.
zg_status run_deco_step(const Run& r, int s, cudaStream_t st) {
  const Dims& m = r.m;
  const size_t BW = (size_t)m.B * m.beam;
  auto F32 = [&](size_t off) { return reinterpret_cast<float*>(r.ws + off); };
  DecoStep a{};
  a.s = s;
  a.L = m.L;
  a.B = m.B;
  a.Wc = (s == 1) ? 1 : m.beam;
  a.beam = m.beam;
  a.M = m.dM;
  a.d = m.d;
  a.heads = m.deco->heads;
  a.concepts = r.u;
  if (s >= 2) {
    a.tok_in = reinterpret_cast<const int32_t*>(r.ws + r.w.tok_hist) + (size_t)(s - 2) * BW;
    a.cum_in = F32(r.w.cum[(s - 1) & 1]);
  }
  a.par_hist = reinterpret_cast<const int32_t*>(r.ws + r.w.par_hist);
  a.X = F32(r.w.dX);
  a.A = F32(r.w.dA);
  a.Q = F32(r.w.dQ);
  a.O = F32(r.w.dO);
  a.F = F32(r.w.dF);
  a.Kc = F32(r.w.dKc);
  a.Vc = F32(r.w.dVc);
  a.Ks = F32(r.w.dKs);
  a.Vs = F32(r.w.dVs);
  a.H = F32(r.w.dH);
  cudaError_t e = launch_deco_step(*m.deco, a, st);
  if (e != cudaSuccess) return cuda_fail(e, "light decoder launch");
  return ZG_OK;
}

constexpr int kClusterCTAs = 8;  // default CTAs of the fused kernel's cluster (one cluster per request)

int variant_of(const Run& r, const zg_plan* plan, int s) {
  return (!r.idx || r.m.score_first) ? ZG_FULL : (plan ? plan->variant[s - 1] : ZG_SELECTIVE);
}

// First step of the trailing run of selective steps that zg_decode fuses
// (L+1: none).
int fused_from(const Run& r, const zg_plan* plan) {
  if (!r.idx || r.m.score_first || r.m.deco || (plan && !plan->fused)) return r.m.L + 1;
  int s0 = r.m.L + 1;
  while (s0 > 1 && variant_of(r, plan, s0 - 1) == ZG_SELECTIVE) --s0;
  return s0;
}

// Launch descriptions of the fused steps s0..L.  Clusters of different
// requests run through the steps independently, so every fused step uses one
// per-request stride for the slots and partials (the largest of the steps).
void fused_launches(const Run& r, int s0, StepLaunch* steps) {
  int64_t zq = 0, pq = 0;
  for (int s = 1; s <= r.m.L; ++s) {
    steps[s - 1] = make_launch(r, s, ZG_SELECTIVE);
    if (s >= s0) {
      zq = std::max(zq, steps[s - 1].zq);
      pq = std::max(pq, steps[s - 1].pq);
    }
  }
  for (int s = s0; s <= r.m.L; ++s) {
    steps[s - 1].zq = zq;
    steps[s - 1].pq = pq;
  }
}

// Tables the fused kernel prefetches into L2 at launch, in priority order,
// up to a budget of about 60 % of the L2: the output heads W_s of the fused
// steps (every legal row is read by some beam), the token tables C_{s-1}
// their gather-add reads (every beam reads one row), then the index tables of
// at most 8 MiB (a large table is touched only at the live beams' rows, so
// fetching all of it would evict useful lines).
int prefetch_set(const Run& r, int s0, PrefetchRegion* pf) {
  constexpr uint64_t kBudget = 80ull << 20;
  constexpr uint64_t kSmallTable = 8ull << 20;
  uint64_t used = 0;
  int n = 0;
  auto add = [&](const void* p, uint64_t bytes) {
    if (!p || n >= kMaxPrefetch || used + bytes > kBudget) return;
    pf[n].ptr = p;
    pf[n].bytes = bytes;
    used += bytes;
    ++n;
  };
  const uint64_t wrow = (uint64_t)r.m.d * (r.m.w_dtype == ZG_F32 ? 4 : 2);
  for (int s = s0; s <= r.m.L; ++s) add(r.model->W[s - 1], wrow * r.m.V);
  for (int s = std::max(s0, 2); s <= r.m.L; ++s) add(r.model->C[s - 2], (uint64_t)r.m.d * 4 * r.m.V);
  for (int s = s0; s <= r.m.L; ++s) {
    const StepMeta& sm = r.idx->steps[s - 1];
    const uint64_t bytes = sm.off_payload + sm.bytes_payload - sm.off_rowptr;
    if (bytes <= kSmallTable) add(r.idx->dev + sm.off_rowptr, bytes);
  }
  return n;
}

// An NVTX range for the host-side span of a call (profiler timelines); a
// no-op unless a tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

const char* step_range_name(int s, int variant) {
  static const char* names[ZG_MAX_STEPS][3] = {
      {"zg step 1 selective", "zg step 1 full", "zg step 1 naive"}, {"zg step 2 selective", "zg step 2 full", "zg step 2 naive"},
      {"zg step 3 selective", "zg step 3 full", "zg step 3 naive"}, {"zg step 4 selective", "zg step 4 full", "zg step 4 naive"},
      {"zg step 5 selective", "zg step 5 full", "zg step 5 naive"}, {"zg step 6 selective", "zg step 6 full", "zg step 6 naive"},
      {"zg step 7 selective", "zg step 7 full", "zg step 7 naive"}, {"zg step 8 selective", "zg step 8 full", "zg step 8 naive"}};
  return names[s - 1][variant];
}

// zg_decode's launch sequence: stand-alone steps, then the fused suffix.
zg_status decode_steps(const Run& r, const zg_plan* plan, cudaStream_t st, cudaEvent_t* fuse_ev = nullptr) {
  NvtxRange whole("zg_decode");
  const int s0 = fused_from(r, plan);
  for (int s = 1; s < s0; ++s) {
    const int v = variant_of(r, plan, s);
    NvtxRange step(step_range_name(s, v));
    if (r.m.deco) {
      zg_status e = run_deco_step(r, s, st);
      if (e != ZG_OK) return e;
    }
    zg_status e = run_step(r, s, v, st);
    if (e != ZG_OK) return e;
  }
  if (s0 <= r.m.L) {
    NvtxRange fused("zg fused selective steps");
    StepLaunch steps[ZG_MAX_STEPS];
    fused_launches(r, s0, steps);
    PrefetchRegion pf[kMaxPrefetch];
    const int npf = prefetch_set(r, s0, pf);
    if (fuse_ev) cudaEventRecord(fuse_ev[0], st);
    const int G = plan ? plan->fused : kClusterCTAs;
    cudaError_t e = launch_decode_cluster(steps, s0, r.m.L, G, pf, npf, st);
    if (e != cudaSuccess) return cuda_fail(e, "fused cluster decode launch");
    if (fuse_ev) cudaEventRecord(fuse_ev[1], st);
  }
  return ZG_OK;
}

}  // namespace

cudaError_t current_context_id(unsigned long long* id) {
  using GetCurrent = int (*)(void**);                      // cuCtxGetCurrent(CUcontext*)
  using GetId = int (*)(void*, unsigned long long*);       // cuCtxGetId(CUcontext, unsigned long long*)
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (!get_current || !get_id) return cudaErrorNotSupported;
  // make the runtime's primary context of the current device current on this
  // thread (cudaSetDevice initialises it; nothing is allocated)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  if (e != cudaSuccess) return e;
  void* ctx = nullptr;
  if (get_current(&ctx) != 0 || !ctx) return cudaErrorDeviceUninitialized;
  if (get_id(ctx, id) != 0) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

zg_status fail(zg_status code, const std::string& msg) {
  g_err = msg;
  return code;
}

zg_status cuda_fail(cudaError_t e, const char* what) {
  g_err = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return e == cudaErrorMemoryAllocation ? ZG_ERR_OUT_OF_MEMORY : ZG_ERR_CUDA;
}

}  // namespace zg

using namespace zg;

extern "C" {

const char* zg_last_error(void) { return g_err.c_str(); }
const char* zg_version(void) { return "zerogr-gb300 0.1 (sm_103a)"; }

zg_status zg_plan_force(const zg_index* idx, int32_t B, int32_t beam, const uint8_t* variant, zg_plan** out) {
  if (!out) return fail(ZG_ERR_INVALID_ARG, "zg_plan_force: out is NULL");
  *out = nullptr;
  if (!idx || !variant) return fail(ZG_ERR_INVALID_ARG, "zg_plan_force: idx and variant must not be NULL");
  for (int s = 0; s < idx->L; ++s)
    if (variant[s] != ZG_SELECTIVE && variant[s] != ZG_FULL && variant[s] != ZG_NAIVE)
      return fail(ZG_ERR_INVALID_ARG, "zg_plan_force: variant must be ZG_SELECTIVE, ZG_FULL or ZG_NAIVE");
  auto* p = new zg_plan();
  p->L = idx->L;
  p->B = B;
  p->beam = beam;
  p->variant.assign(variant, variant + idx->L);
  p->step_ms.assign((size_t)idx->L * 2, -1.f);
  *out = p;
  return ZG_OK;
}

zg_status zg_plan_describe(const zg_plan* plan, uint8_t* variant, float* step_ms, int32_t* cluster_ctas,
                           float* fused_ms) {
  if (!plan) return fail(ZG_ERR_INVALID_ARG, "zg_plan_describe: plan is NULL");
  if (variant) std::memcpy(variant, plan->variant.data(), plan->L);
  if (step_ms) std::memcpy(step_ms, plan->step_ms.data(), plan->step_ms.size() * sizeof(float));
  if (cluster_ctas) *cluster_ctas = plan->fused;
  if (fused_ms) std::memcpy(fused_ms, plan->fused_ms, sizeof(plan->fused_ms));
  return ZG_OK;
}

void zg_plan_free(zg_plan* plan) { delete plan; }

}  // extern "C"

namespace {
const char kPlanMagic[8] = {'Z', 'G', 'P', 'L', 'A', 'N', 0, 2};

uint64_t plan_fnv1a(const std::vector<uint8_t>& b) {
  uint64_t h = 1469598103934665603ull;
  for (uint8_t x : b) {
    h ^= x;
    h *= 1099511628211ull;
  }
  return h;
}

template <typename T>
void put(std::vector<uint8_t>& b, const T& v) {
  const uint8_t* p = reinterpret_cast<const uint8_t*>(&v);
  b.insert(b.end(), p, p + sizeof(T));
}

template <typename T>
bool get(const std::vector<uint8_t>& b, size_t& at, T* v) {
  if (at + sizeof(T) > b.size()) return false;
  std::memcpy(v, b.data() + at, sizeof(T));
  at += sizeof(T);
  return true;
}
}  // namespace

extern "C" {

zg_status zg_plan_save(const zg_plan* plan, const char* path) {
  if (!plan || !path) return fail(ZG_ERR_INVALID_ARG, "zg_plan_save: NULL argument");
  std::vector<uint8_t> body;
  put(body, plan->L);
  put(body, plan->B);
  put(body, plan->beam);
  put(body, plan->fused);
  put(body, plan->order);
  put(body, plan->hidden);
  put(body, plan->scores);
  put(body, plan->plan_ms);
  for (float x : plan->fused_ms) put(body, x);
  for (uint8_t v : plan->variant) put(body, v);
  for (float x : plan->step_ms) put(body, x);
  const uint64_t h = plan_fnv1a(body);
  FILE* f = std::fopen(path, "wb");
  if (!f) return fail(ZG_ERR_IO, std::string("zg_plan_save: cannot open ") + path);
  bool ok = std::fwrite(kPlanMagic, 1, 8, f) == 8 && std::fwrite(body.data(), 1, body.size(), f) == body.size() &&
            std::fwrite(&h, 8, 1, f) == 1;
  ok = (std::fclose(f) == 0) && ok;
  if (!ok) return fail(ZG_ERR_IO, std::string("zg_plan_save: write failed for ") + path);
  return ZG_OK;
}

zg_status zg_plan_load(const char* path, zg_plan** out) {
  if (!path || !out) return fail(ZG_ERR_INVALID_ARG, "zg_plan_load: NULL argument");
  *out = nullptr;
  FILE* f = std::fopen(path, "rb");
  if (!f) return fail(ZG_ERR_IO, std::string("zg_plan_load: cannot open ") + path);
  std::vector<uint8_t> raw;
  uint8_t buf[4096];
  size_t n;
  while ((n = std::fread(buf, 1, sizeof buf, f)) > 0 && raw.size() < (1u << 20)) raw.insert(raw.end(), buf, buf + n);
  std::fclose(f);
  auto bad = [&]() { return fail(ZG_ERR_IO, std::string("zg_plan_load: short, corrupt or foreign file ") + path); };
  if (raw.size() < 16 || std::memcmp(raw.data(), kPlanMagic, 8) != 0) return bad();
  std::vector<uint8_t> body(raw.begin() + 8, raw.end() - 8);
  uint64_t h = 0;
  std::memcpy(&h, raw.data() + raw.size() - 8, 8);
  if (h != plan_fnv1a(body)) return bad();
  auto p = std::make_unique<zg_plan>();
  size_t at = 0;
  bool ok = get(body, at, &p->L) && get(body, at, &p->B) && get(body, at, &p->beam) && get(body, at, &p->fused) &&
            get(body, at, &p->order) && get(body, at, &p->hidden) && get(body, at, &p->scores) &&
            get(body, at, &p->plan_ms);
  for (float& x : p->fused_ms) ok = ok && get(body, at, &x);
  ok = ok && p->L >= 1 && p->L <= ZG_MAX_STEPS && p->B >= 1 && p->beam >= 1 && p->beam <= ZG_MAX_BEAM &&
       (p->order == ZG_ORDER_FILTER_FIRST || p->order == ZG_ORDER_SCORE_FIRST) &&
       (p->hidden == ZG_HIDDEN_SPLIT || p->hidden == ZG_HIDDEN_SINGLE) &&
       (p->scores == ZG_SCORES_AUTO || p->scores == ZG_SCORES_WRITTEN || p->scores == ZG_SCORES_CHUNK_TOPS) &&
       (p->fused == 0 || p->fused == 1 || p->fused == 2 || p->fused == 4 || p->fused == 8 || p->fused == 16);
  if (ok) {
    p->variant.resize(p->L);
    p->step_ms.resize((size_t)p->L * 2);
    for (auto& v : p->variant) ok = ok && get(body, at, &v) && (v == ZG_SELECTIVE || v == ZG_FULL || v == ZG_NAIVE);
    for (auto& x : p->step_ms) ok = ok && get(body, at, &x);
  }
  if (!ok || at != body.size()) return bad();
  *out = p.release();
  return ZG_OK;
}

zg_status zg_plan_set_fusion(zg_plan* plan, int32_t cluster_ctas) {
  if (!plan) return fail(ZG_ERR_INVALID_ARG, "zg_plan_set_fusion: plan is NULL");
  if (cluster_ctas != 0 && cluster_ctas != 1 && cluster_ctas != 2 && cluster_ctas != 4 && cluster_ctas != 8 &&
      cluster_ctas != 16)
    return fail(ZG_ERR_INVALID_ARG, "zg_plan_set_fusion: cluster_ctas must be 0, 1, 2, 4, 8 or 16");
  plan->fused = cluster_ctas;
  return ZG_OK;
}

zg_status zg_plan_set_full_projection(zg_plan* plan, int32_t hidden_rounding, int32_t scores) {
  if (!plan) return fail(ZG_ERR_INVALID_ARG, "zg_plan_set_full_projection: plan is NULL");
  if (hidden_rounding != ZG_HIDDEN_SPLIT && hidden_rounding != ZG_HIDDEN_SINGLE)
    return fail(ZG_ERR_INVALID_ARG, "zg_plan_set_full_projection: hidden_rounding must be ZG_HIDDEN_SPLIT or ZG_HIDDEN_SINGLE");
  if (scores != ZG_SCORES_AUTO && scores != ZG_SCORES_WRITTEN && scores != ZG_SCORES_CHUNK_TOPS)
    return fail(ZG_ERR_INVALID_ARG, "zg_plan_set_full_projection: scores must be ZG_SCORES_AUTO, _WRITTEN or _CHUNK_TOPS");
  plan->hidden = hidden_rounding;
  plan->scores = scores;
  return ZG_OK;
}

zg_status zg_plan_set_order(zg_plan* plan, int32_t order) {
  if (!plan) return fail(ZG_ERR_INVALID_ARG, "zg_plan_set_order: plan is NULL");
  if (order != ZG_ORDER_FILTER_FIRST && order != ZG_ORDER_SCORE_FIRST)
    return fail(ZG_ERR_INVALID_ARG, "zg_plan_set_order: order must be ZG_ORDER_FILTER_FIRST or ZG_ORDER_SCORE_FIRST");
  plan->order = order;
  return ZG_OK;
}

zg_status zg_decode_workspace_size(const zg_index* idx, const zg_plan* plan, const zg_model* model, int32_t B,
                                   int32_t beam, int32_t K, size_t* bytes) {
  if (!bytes) return fail(ZG_ERR_INVALID_ARG, "bytes is NULL");
  Dims m;
  zg_status st = check_common(idx, model, B, beam, K, &m);
  if (st != ZG_OK) return st;
  if (plan && plan->L != m.L) return fail(ZG_ERR_INVALID_ARG, "plan has a different number of steps");
  if ((st = apply_plan(m, idx, plan)) != ZG_OK) return st;
  *bytes = layout(m, false).total;
  return ZG_OK;
}

zg_status zg_decode_host_workspace_size(const zg_index* idx, const zg_plan* plan, const zg_model* model, int32_t B,
                                        int32_t beam, int32_t K, size_t* bytes) {
  if (!bytes) return fail(ZG_ERR_INVALID_ARG, "bytes is NULL");
  Dims m;
  zg_status st = check_common(idx, model, B, beam, K, &m);
  if (st != ZG_OK) return st;
  if (plan && plan->L != m.L) return fail(ZG_ERR_INVALID_ARG, "plan has a different number of steps");
  if ((st = apply_plan(m, idx, plan)) != ZG_OK) return st;
  *bytes = layout(m, true).total;
  return ZG_OK;
}

zg_status zg_decode(const zg_index* idx, const zg_plan* plan, const zg_model* model, const float* u, int32_t B,
                    int32_t beam, int32_t K, int32_t* out_sids, float* out_scores, void* workspace, size_t ws_bytes,
                    void* stream) {
  Run r;
  zg_status st = prepare(idx, plan, model, u, B, beam, K, out_sids, out_scores, workspace, ws_bytes, false, &r);
  if (st != ZG_OK) return st;
  return decode_steps(r, plan, static_cast<cudaStream_t>(stream));
}

zg_status zg_decode_host(const zg_index* idx, const zg_plan* plan, const zg_model* model, const float* u_host,
                         int32_t B, int32_t beam, int32_t K, int32_t* out_sids_host, float* out_scores_host,
                         void* workspace, size_t ws_bytes, void* stream) {
  Run r;
  zg_status st =
      prepare(idx, plan, model, u_host, B, beam, K, out_sids_host, out_scores_host, workspace, ws_bytes, true, &r);
  if (st != ZG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* u_dev = reinterpret_cast<float*>(r.ws + r.w.u_stage);
  int32_t* sids_dev = reinterpret_cast<int32_t*>(r.ws + r.w.o_sids);
  float* sc_dev = reinterpret_cast<float*>(r.ws + r.w.o_scores);
  cudaError_t e = cudaMemcpyAsync(u_dev, u_host, (size_t)B * (r.m.deco ? r.m.dM : 1) * r.m.d * 4,
                                  cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "zg_decode_host: copy of u");
  r.u = u_dev;
  r.out_sids = sids_dev;
  r.out_scores = sc_dev;
  st = decode_steps(r, plan, s);
  if (st != ZG_OK) return st;
  e = cudaMemcpyAsync(out_sids_host, sids_dev, (size_t)B * K * r.m.L * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_scores_host, sc_dev, (size_t)B * K * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "zg_decode_host: copy back");
  return ZG_OK;
}

zg_status zg_tune(const zg_index* idx, const zg_model* model, const float* warm_u, int32_t B, int32_t beam, int32_t K,
                  int32_t reps, void* stream, zg_plan** out) {
  if (!out) return fail(ZG_ERR_INVALID_ARG, "zg_tune: out is NULL");
  *out = nullptr;
  NvtxRange range("zg_tune");
  if (!idx) return fail(ZG_ERR_INVALID_ARG, "zg_tune: idx is NULL (the unconstrained decode has one variant)");
  if (!warm_u) return fail(ZG_ERR_INVALID_ARG, "zg_tune: warm_u is NULL");
  if (reps < 1) reps = 1;
  Dims m;
  zg_status st = check_common(idx, model, B, beam, K, &m);
  if (st != ZG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsLayout w = layout(m, true);
  void* ws = nullptr;
  cudaError_t e = cudaMalloc(&ws, w.total);
  if (e != cudaSuccess) return cuda_fail(e, "zg_tune: workspace allocation");
  cudaEvent_t ev[2] = {nullptr, nullptr};
  auto cleanup = [&]() {
    for (auto& x : ev)
      if (x) cudaEventDestroy(x);
    cudaFree(ws);
  };
  if ((e = cudaEventCreate(&ev[0])) != cudaSuccess || (e = cudaEventCreate(&ev[1])) != cudaSuccess) {
    cleanup();
    return cuda_fail(e, "zg_tune: cudaEventCreate");
  }
  Run r;
  r.m = m;
  r.w = w;
  r.ws = static_cast<uint8_t*>(ws);
  r.idx = idx;
  r.model = model;
  r.u = warm_u;
  r.out_sids = reinterpret_cast<int32_t*>(r.ws + w.o_sids);
  r.out_scores = reinterpret_cast<float*>(r.ws + w.o_scores);
  if ((st = get_status_ptr(&r.status)) != ZG_OK) {
    cleanup();
    return st;
  }
  auto* plan = new zg_plan();
  plan->L = m.L;
  plan->B = B;
  plan->beam = beam;
  plan->variant.assign(m.L, ZG_SELECTIVE);
  plan->step_ms.assign((size_t)m.L * 2, -1.f);
  for (int step = 1; step <= m.L && st == ZG_OK; ++step) {
    float best = INFINITY;
    int best_v = ZG_SELECTIVE;
    if (m.deco && (st = run_deco_step(r, step, s)) != ZG_OK) break;  // the entering beams' hidden vectors
    for (int v = ZG_SELECTIVE; v <= ZG_FULL && st == ZG_OK; ++v) {
      for (int i = 0; i < 2 && st == ZG_OK; ++i) st = run_step(r, step, v, s);
      if (st != ZG_OK) break;
      cudaEventRecord(ev[0], s);
      for (int i = 0; i < reps && st == ZG_OK; ++i) st = run_step(r, step, v, s);
      cudaEventRecord(ev[1], s);
      if ((e = cudaEventSynchronize(ev[1])) != cudaSuccess) {
        st = cuda_fail(e, "zg_tune: timing");
        break;
      }
      float ms = 0.f;
      cudaEventElapsedTime(&ms, ev[0], ev[1]);
      ms /= reps;
      plan->step_ms[(size_t)(step - 1) * 2 + v] = ms;
      if (ms < best) {
        best = ms;
        best_v = v;
      }
    }
    if (st != ZG_OK) break;
    plan->variant[step - 1] = (uint8_t)best_v;
    st = run_step(r, step, best_v, s);  // advance the state with the kept variant
  }
  // Whole-decode candidates: for every split point s0, the per-step best
  // variants before s0 and selective steps from s0 on, fused with each
  // cluster size (or, for s0 = L+1, no fused part).  The fastest decode wins.
  if (st == ZG_OK) {
    const std::vector<uint8_t> best_steps = plan->variant;
    const int sizes[5] = {1, 2, 4, 8, 16};
    float best_total = INFINITY;
    std::vector<uint8_t> best_v = best_steps;
    int best_g = 0;
    float best_gms[5] = {-1, -1, -1, -1, -1};
    zg_plan cand = *plan;
    for (int s0 = 1; s0 <= m.L + 1 && st == ZG_OK; ++s0) {
      bool best_here = false;
      for (int step = 1; step <= m.L; ++step)
        cand.variant[step - 1] = step < s0 ? best_steps[step - 1] : (uint8_t)ZG_SELECTIVE;
      if (s0 > 1 && s0 <= m.L && cand.variant[s0 - 2] == ZG_SELECTIVE) continue;  // same as a smaller s0
      float gms[5] = {-1, -1, -1, -1, -1};
      for (int gi = 0; gi < 5 && st == ZG_OK; ++gi) {
        if (s0 > m.L && gi > 0) break;
        cand.fused = (s0 > m.L) ? 0 : sizes[gi];
        float sum = 0.f;
        bool ok = true;
        for (int i = 0; i < reps + 2 && ok; ++i) {
          cudaEventRecord(ev[0], s);
          st = decode_steps(r, &cand, s);
          cudaEventRecord(ev[1], s);
          if (st != ZG_OK || cudaEventSynchronize(ev[1]) != cudaSuccess) {
            ok = false;  // e.g. this cluster size cannot be scheduled
            st = ZG_OK;
            cudaGetLastError();
            break;
          }
          float ms = 0.f;
          cudaEventElapsedTime(&ms, ev[0], ev[1]);
          if (i >= 2) sum += ms;
        }
        if (!ok) continue;
        const float avg = sum / reps;
        if (s0 <= m.L) gms[gi] = avg;
        if (avg < best_total) {
          best_total = avg;
          best_v = cand.variant;
          best_g = cand.fused;
          best_here = true;
        }
      }
      if (best_here) std::memcpy(best_gms, gms, sizeof gms);  // every cluster size timed at this split
    }
    plan->variant = best_v;
    plan->fused = best_g;
    std::memcpy(plan->fused_ms, best_gms, sizeof best_gms);
    plan->plan_ms = best_total;
  }
  if (st == ZG_OK && (e = cudaStreamSynchronize(s)) != cudaSuccess) st = cuda_fail(e, "zg_tune: synchronise");
  cleanup();
  if (st != ZG_OK) {
    delete plan;
    return st;
  }
  *out = plan;
  return ZG_OK;
}

zg_status zg_decode_trace(const zg_index* idx, const zg_plan* plan, const zg_model* model, const float* u, int32_t B,
                          int32_t beam, int32_t K, int32_t* out_sids, float* out_scores, void* workspace,
                          size_t ws_bytes, void* stream, zg_trace* trace) {
  if (!trace) return fail(ZG_ERR_INVALID_ARG, "zg_decode_trace: trace is NULL");
  Run r;
  zg_status st = prepare(idx, plan, model, u, B, beam, K, out_sids, out_scores, workspace, ws_bytes, false, &r);
  if (st != ZG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::memset(trace, 0, sizeof(*trace));
  trace->L = r.m.L;
  constexpr int kEv = 6 * ZG_MAX_STEPS + 4;  // 4 a step, 2 a step for the light decoder, 4 for the whole
  cudaEvent_t ev[kEv] = {};
  int made = 0;
  cudaError_t e = cudaSuccess;
  for (; made < kEv && e == cudaSuccess; ++made) e = cudaEventCreate(&ev[made]);
  auto cleanup = [&]() {
    for (int i = 0; i < kEv; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);
  };
  if (e != cudaSuccess) {
    cleanup();
    return cuda_fail(e, "zg_decode_trace: cudaEventCreate");
  }
  // pass 1: zg_decode's own launch sequence
  const int s0 = fused_from(r, plan);
  if ((e = launch_delay(50000ull, s)) != cudaSuccess) st = cuda_fail(e, "zg_decode_trace: delay launch");
  cudaEventRecord(ev[kEv - 2], s);
  if (st == ZG_OK) st = decode_steps(r, plan, s, s0 <= r.m.L ? &ev[kEv - 4] : nullptr);
  cudaEventRecord(ev[kEv - 1], s);
  if (st == ZG_OK && (e = cudaEventSynchronize(ev[kEv - 1])) != cudaSuccess) st = cuda_fail(e, "zg_decode_trace");
  if (st != ZG_OK) {
    cleanup();
    return st;
  }
  cudaEventElapsedTime(&trace->ms_total, ev[kEv - 2], ev[kEv - 1]);
  if (s0 <= r.m.L) {
    trace->fused_from = s0;
    cudaEventElapsedTime(&trace->ms_fused, ev[kEv - 4], ev[kEv - 3]);
  }
  // pass 2: stand-alone step kernels, each timed, with work counts
  auto* cnt = reinterpret_cast<unsigned long long*>(r.ws + r.w.trace);
  auto* mask = reinterpret_cast<uint32_t*>(r.ws + r.w.trace + 32);
  const int words = (r.m.V + 31) / 32;
  std::vector<uint32_t> hmask(words);
  for (int step = 1; step <= r.m.L; ++step) {
    const int v = variant_of(r, plan, step);
    StepTimer tm;
    for (int j = 0; j < 4; ++j) tm.ev[j] = ev[4 * (step - 1) + j];
    cudaEvent_t* mev = &ev[4 * ZG_MAX_STEPS + 2 * (step - 1)];
    // the step's launches are enqueued behind a delay, so the events time kernels, not launch gaps
    if ((e = launch_delay(50000ull, s)) != cudaSuccess) {
      st = cuda_fail(e, "zg_decode_trace: delay launch");
      break;
    }
    if (r.m.deco) {
      cudaEventRecord(mev[0], s);
      if ((st = run_deco_step(r, step, s)) != ZG_OK) break;
      cudaEventRecord(mev[1], s);
    }
    st = run_step(r, step, v, s, &tm);
    if (st != ZG_OK) break;
    // untimed: what this step worked on (its entering state is still intact)
    const StepLaunch a = make_launch(r, step, v);
    unsigned long long hc[4];
    e = cudaMemsetAsync(r.ws + r.w.trace, 0, r.w.trace_bytes, s);
    if (e == cudaSuccess) e = launch_trace_touch(a, cnt, mask, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hc, cnt, 32, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hmask.data(), mask, (size_t)words * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
      st = cuda_fail(e, "zg_decode_trace: counting");
      break;
    }
    zg_step_trace& t = trace->step[step - 1];
    t.variant = v;
    t.live_beams = (int32_t)hc[0];
    t.legal_slots = (int64_t)hc[1];
    t.chunks = (v == ZG_SELECTIVE) ? (int64_t)hc[2] : 0;
    t.index_bytes = (int64_t)hc[3];
    int64_t ut = 0;
    for (uint32_t w : hmask) ut += __builtin_popcount(w);
    t.unique_tokens = ut;
    float g = 0.f, pj = 0.f, q = 0.f;
    cudaEventElapsedTime(&g, tm.ev[0], tm.ev[1]);
    cudaEventElapsedTime(&pj, tm.ev[1], tm.ev[2]);
    cudaEventElapsedTime(&q, tm.ev[2], tm.ev[3]);
    t.ms_gather = (v == ZG_NAIVE || v == ZG_SELECTIVE || (v == ZG_FULL && (step >= 2 || r.m.w_dtype != ZG_F32))) ? g : 0.f;
    t.ms_project = pj;
    t.ms_select = q;
    if (r.m.deco) cudaEventElapsedTime(&t.ms_model, mev[0], mev[1]);
  }
  cleanup();
  return st;
}

void zg_debug_set_wait_limit(uint32_t polls) { set_wait_limit(polls); }

zg_status zg_check_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "zg_check_device_status: synchronise");
  uint32_t* p = nullptr;
  zg_status st = get_status_ptr(&p);
  if (st != ZG_OK) return st;
  uint32_t v = 0;
  e = cudaMemcpy(&v, p, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "zg_check_device_status: read");
  if (!v) return ZG_OK;
  cudaMemset(p, 0, 4);
  std::string msg = "device status:";
  if (v & kStatusRow) msg += " row out of range;";
  if (v & kStatusToken) msg += " token out of range;";
  if (v & kStatusTimeout) msg += " tensor-core wait expired;";
  if (v & kStatusTmem) msg += " tensor-memory allocation failed;";
  if (v & kStatusSelect) msg += " select found fewer candidates than its cut;";
  return fail(ZG_ERR_DEVICE_STATUS, msg);
}

}  // extern "C"
