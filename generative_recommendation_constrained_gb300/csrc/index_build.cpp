// Host-side builder of the step-sliced filter index, its statistics, export,
// and save/load.
//
// "ZeroGR: Filtering-First Constrained Decoding for Generative
// Recommendation" (paper-daily.com digest):
//   section "Why slice the index by decoding step": one table per decoding
//     step; a row is a prefix; the position of an entry is its next-step row;
//     dense tables for steps with many legal tokens, sparse (CSR) otherwise;
//   section "Is the scheme really better", last part: the index is rebuilt
//     on the CPU in chunks, in parallel, first computing where each chunk goes
//     in the final index, then filling two buffers in turn while the other is
//     sent to the GPU, without taking the serving GPU.
//
// Chunks here are first-token subtrees ("buckets"): after a parallel radix
// partition by the first token every later prefix lives inside one bucket,
// so rows and entries of every step can be counted per bucket (pass 1), laid
// out by exclusive prefix sums, and filled independently (pass 2).
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <new>
#include <thread>

#include <nvtx3/nvToolsExt.h>

#include "zg_internal.h"

namespace zg {
namespace {

using clk = std::chrono::steady_clock;
double ms_since(clk::time_point t0) {
  return std::chrono::duration<double, std::milli>(clk::now() - t0).count();
}

int bits_for(int V) {
  int b = 0;
  while ((1LL << b) < V) ++b;
  return b == 0 ? 1 : b;
}

uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Dynamic parallel loop over [0, n).
template <class F>
void parallel_for(int T, int64_t n, F fn) {
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      int64_t i = next.fetch_add(1, std::memory_order_relaxed);
      if (i >= n) break;
      fn(i);
    }
  };
  int nt = (int)std::min<int64_t>(T, n);
  if (nt <= 1) {
    worker();
    return;
  }
  std::vector<std::thread> th;
  th.reserve(nt - 1);
  for (int t = 1; t < nt; ++t) th.emplace_back(worker);
  worker();
  for (auto& x : th) x.join();
}

// Static split of [0, n) into T contiguous ranges; fn(t, lo, hi).
template <class F>
void parallel_ranges(int T, int64_t n, F fn) {
  std::vector<std::thread> th;
  int64_t per = (n + T - 1) / T;
  for (int t = 1; t < T; ++t) {
    int64_t lo = std::min(n, per * t), hi = std::min(n, per * (t + 1));
    th.emplace_back([&, t, lo, hi]() { fn(t, lo, hi); });
  }
  fn(0, 0, std::min(n, per));
  for (auto& x : th) x.join();
}

// 1-based step at which key a first differs from key b (L+1 if equal).
inline int first_diff_step(uint64_t a, uint64_t b, int L, int bits) {
  uint64_t x = a ^ b;
  if (!x) return L + 1;
  int hb = 63 - __builtin_clzll(x);
  int pos = (L - 1) - hb / bits;  // 0-based token position
  return pos + 1;
}

struct Bucket {
  int64_t start = 0;  // offset in the key array
  int64_t count = 0;  // distinct keys after merging duplicates
  uint32_t tok = 0;   // first token
};

struct Layout {
  int L, V, bits, words;
  std::vector<Bucket> buckets;                 // nonempty, ascending first token
  std::vector<std::vector<uint32_t>> cnt;      // [nb][L+1]: distinct s-prefixes (s=1..L)
  std::vector<std::vector<uint32_t>> maxf;     // [nb][L+1]
  std::vector<std::vector<uint64_t>> rowoff;   // [L+1][nb]
  std::vector<std::vector<uint64_t>> entoff;   // [L+1][nb]
};

// Fill bucket b's slice of step s (s >= 2).
void fill_bucket(const Layout& lay, const uint64_t* keys, int b, int s, int fmt, uint32_t* rowptr_dst,
                 void* pay_dst) {
  const Bucket& bk = lay.buckets[b];
  const int L = lay.L, bits = lay.bits;
  const uint64_t mask = (bits >= 64) ? ~0ull : ((1ull << bits) - 1);
  const uint64_t ent_base = lay.entoff[s][b];
  const uint32_t words = (uint32_t)lay.words;
  int64_t row = -1, ent = -1;
  uint16_t* col = static_cast<uint16_t*>(pay_dst);
  uint32_t* bm = static_cast<uint32_t*>(pay_dst);
  if (fmt == ZG_FMT_DENSE) std::memset(bm, 0, (size_t)lay.cnt[b][s - 1] * words * 4);
  const uint64_t* k = keys + bk.start;
  for (int64_t i = 0; i < bk.count; ++i) {
    int s0 = (i == 0) ? 1 : first_diff_step(k[i], k[i - 1], L, bits);
    if (s0 <= s - 1) {
      ++row;
      rowptr_dst[row] = (uint32_t)(ent_base + (uint64_t)(ent + 1));
    }
    if (s0 <= s) {
      ++ent;
      uint32_t tok = (uint32_t)((k[i] >> ((L - s) * bits)) & mask);
      if (fmt == ZG_FMT_SPARSE)
        col[ent] = (uint16_t)tok;
      else
        bm[(uint64_t)row * words + tok / 32] |= 1u << (tok % 32);
    }
  }
}

// Host-side failure injection for tests (zg_debug_inject_build_failure):
// the `after`-th next call at `point` reports a failure instead of running.
std::atomic<int> g_inject_point{0}, g_inject_after{0};

bool injected(int point) {
  if (g_inject_point.load(std::memory_order_relaxed) != point) return false;
  if (g_inject_after.fetch_sub(1) > 0) return false;
  g_inject_point.store(0);  // fires once
  return true;
}

struct Pinned {
  uint8_t* p = nullptr;
  size_t n = 0;
  ~Pinned() {
    if (p) cudaFreeHost(p);
  }
  cudaError_t ensure(size_t bytes) {
    if (bytes <= n) return cudaSuccess;
    if (p) cudaFreeHost(p);
    p = nullptr;
    n = 0;
    if (injected(ZG_INJECT_PINNED_ALLOC)) return cudaErrorMemoryAllocation;
    cudaError_t e = cudaHostAlloc((void**)&p, bytes, cudaHostAllocDefault);
    if (e == cudaSuccess) n = bytes;
    return e;
  }
};

zg_status build_impl(const int32_t* sids, int64_t n, int L, int V, const zg_build_opts& o,
                     cudaStream_t stream, zg_index** out) {
  auto t_all = clk::now();
  if (!out) return fail(ZG_ERR_INVALID_ARG, "zg_index_build: out is NULL");
  *out = nullptr;
  if (!sids) return fail(ZG_ERR_INVALID_ARG, "zg_index_build: sids is NULL");
  if (n < 1) return fail(ZG_ERR_INVALID_ARG, "zg_index_build: empty catalogue (n < 1)");
  if (L < 1 || L > ZG_MAX_STEPS) return fail(ZG_ERR_INVALID_ARG, "zg_index_build: L must be in [1, 8]");
  if (V < 1 || V > 65536) return fail(ZG_ERR_INVALID_ARG, "zg_index_build: V must be in [1, 65536]");
  if (o.format_mode < ZG_FORMAT_AUTO || o.format_mode > ZG_FORMAT_ALL_DENSE)
    return fail(ZG_ERR_INVALID_ARG, "zg_index_build: bad format_mode");
  if (o.residency != ZG_RESIDENT_DEVICE && o.residency != ZG_RESIDENT_HOST)
    return fail(ZG_ERR_INVALID_ARG, "zg_index_build: bad residency");
  const int bits = bits_for(V);
  if (L * bits > 64) return fail(ZG_ERR_UNSUPPORTED, "zg_index_build: L * ceil(log2 V) exceeds 64 key bits");
  int T = o.n_threads > 0 ? o.n_threads : (int)std::thread::hardware_concurrency();
  if (T < 1) T = 1;
  if (T > 256) T = 256;
  const int words = (V + 31) / 32;

  int device = -1;
  if (o.residency == ZG_RESIDENT_DEVICE) {
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_fail(e, "zg_index_build: cudaGetDevice");
  }

  // ---- pack, validate and partition by first token (radix pass) -------------
  auto t0 = clk::now();
  std::vector<uint64_t> keys((size_t)n);
  std::vector<int64_t> hist((size_t)T * V, 0);
  std::atomic<int64_t> bad{-1};
  parallel_ranges(T, n, [&](int t, int64_t lo, int64_t hi) {
    int64_t* h = &hist[(size_t)t * V];
    for (int64_t i = lo; i < hi; ++i) {
      const int32_t* r = sids + i * L;
      for (int s = 0; s < L; ++s)
        if (r[s] < 0 || r[s] >= V) {
          bad.store(i);
          return;
        }
      ++h[r[0]];
    }
  });
  if (bad.load() >= 0) {
    char msg[160];
    std::snprintf(msg, sizeof msg, "zg_index_build: SID %lld has a token outside [0, %d)",
                  (long long)bad.load(), V);
    return fail(ZG_ERR_INVALID_ARG, msg);
  }
  std::vector<int64_t> bstart(V + 1, 0);
  for (int v = 0; v < V; ++v) {
    int64_t tot = 0;
    for (int t = 0; t < T; ++t) tot += hist[(size_t)t * V + v];
    bstart[v + 1] = bstart[v] + tot;
  }
  std::vector<int64_t> cursor((size_t)T * V);
  for (int v = 0; v < V; ++v) {
    int64_t c = bstart[v];
    for (int t = 0; t < T; ++t) {
      cursor[(size_t)t * V + v] = c;
      c += hist[(size_t)t * V + v];
    }
  }
  parallel_ranges(T, n, [&](int t, int64_t lo, int64_t hi) {
    int64_t* cur = &cursor[(size_t)t * V];
    for (int64_t i = lo; i < hi; ++i) {
      const int32_t* r = sids + i * L;
      uint64_t k = 0;
      for (int s = 0; s < L; ++s) k = (k << bits) | (uint64_t)r[s];
      keys[(size_t)cur[r[0]]++] = k;
    }
  });
  Layout lay;
  lay.L = L;
  lay.V = V;
  lay.bits = bits;
  lay.words = words;
  for (int v = 0; v < V; ++v)
    if (bstart[v + 1] > bstart[v]) {
      Bucket b;
      b.start = bstart[v];
      b.count = bstart[v + 1] - bstart[v];
      b.tok = (uint32_t)v;
      lay.buckets.push_back(b);
    }
  const int nb = (int)lay.buckets.size();
  // sort + merge duplicates inside each bucket, largest buckets first
  std::vector<int> by_size(nb);
  for (int i = 0; i < nb; ++i) by_size[i] = i;
  std::sort(by_size.begin(), by_size.end(),
            [&](int a, int b) { return lay.buckets[a].count > lay.buckets[b].count; });
  parallel_for(T, nb, [&](int64_t i) {
    Bucket& b = lay.buckets[by_size[i]];
    uint64_t* p = keys.data() + b.start;
    std::sort(p, p + b.count);
    b.count = std::unique(p, p + b.count) - p;
  });
  double ms_sort = ms_since(t0);

  // ---- pass 1: count rows / entries per bucket and step ----------------------
  nvtxMarkA("zg_index_build: pass 1 (count)");
  t0 = clk::now();
  lay.cnt.assign(nb, std::vector<uint32_t>(L + 1, 0));
  lay.maxf.assign(nb, std::vector<uint32_t>(L + 1, 0));
  std::atomic<int> overflow{0};
  parallel_for(T, nb, [&](int64_t bi) {
    const Bucket& b = lay.buckets[bi];
    const uint64_t* k = keys.data() + b.start;
    std::vector<uint64_t> c(L + 1, 0), run(L + 1, 0), mx(L + 1, 0);
    for (int64_t i = 0; i < b.count; ++i) {
      int s0 = (i == 0) ? 1 : first_diff_step(k[i], k[i - 1], L, bits);
      for (int s = s0; s <= L; ++s) {
        ++c[s];
        if (s >= 2) {
          if (s0 <= s - 1) run[s] = 0;
          ++run[s];
          mx[s] = std::max(mx[s], run[s]);
        }
      }
    }
    for (int s = 1; s <= L; ++s) {
      if (c[s] > 0xFFFFFFFFull) overflow.store(1);
      lay.cnt[bi][s] = (uint32_t)c[s];
      lay.maxf[bi][s] = (uint32_t)mx[s];
    }
  });
  if (overflow.load()) return fail(ZG_ERR_UNSUPPORTED, "zg_index_build: a step has 2^32 or more entries");

  auto* idx = new (std::nothrow) zg_index();
  if (!idx) return fail(ZG_ERR_OUT_OF_MEMORY, "zg_index_build: host allocation");
  std::unique_ptr<zg_index> guard(idx);
  idx->L = L;
  idx->V = V;
  idx->residency = o.residency;
  idx->n_input = n;
  idx->device = device;
  idx->steps.resize(L);
  lay.rowoff.assign(L + 1, std::vector<uint64_t>(nb + 1, 0));
  lay.entoff.assign(L + 1, std::vector<uint64_t>(nb + 1, 0));
  int64_t nuniq = 0;
  for (int b = 0; b < nb; ++b) nuniq += lay.buckets[b].count;
  idx->n_unique = nuniq;
  uint64_t off = 0;
  for (int s = 1; s <= L; ++s) {
    StepMeta& m = idx->steps[s - 1];
    uint64_t rows = 0, nnz = 0;
    uint32_t mf = 0;
    if (s == 1) {
      rows = 1;
      nnz = (uint64_t)nb;
      mf = (uint32_t)nb;
    } else {
      for (int b = 0; b < nb; ++b) {
        lay.rowoff[s][b] = rows;
        lay.entoff[s][b] = nnz;
        rows += lay.cnt[b][s - 1];
        nnz += lay.cnt[b][s];
        mf = std::max(mf, lay.maxf[b][s]);
      }
      lay.rowoff[s][nb] = rows;
      lay.entoff[s][nb] = nnz;
    }
    if (nnz >= 0xFFFFFFFFull || rows >= 0xFFFFFFFFull)
      return fail(ZG_ERR_UNSUPPORTED, "zg_index_build: a step has 2^32 or more entries");
    m.rows = (uint32_t)rows;
    m.nnz = (uint32_t)nnz;
    m.words = (uint32_t)words;
    m.max_fanout = mf;
    if (o.format_mode == ZG_FORMAT_ALL_SPARSE)
      m.fmt = ZG_FMT_SPARSE;
    else if (o.format_mode == ZG_FORMAT_ALL_DENSE)
      m.fmt = ZG_FMT_DENSE;
    else
      m.fmt = (4ull * rows * (uint64_t)words < 2ull * nnz) ? ZG_FMT_DENSE : ZG_FMT_SPARSE;
    m.bytes_rowptr = (rows + 1) * 4;
    m.bytes_payload = (m.fmt == ZG_FMT_SPARSE) ? nnz * 2 : rows * (uint64_t)words * 4;
    m.off_rowptr = off;
    off = align_up(off + m.bytes_rowptr, 256);
    m.off_payload = off;
    off = align_up(off + m.bytes_payload, 256);
  }
  idx->total_bytes = off;
  double ms_count = ms_since(t0);

  // ---- pass 2: fill, streamed through two pinned buffers ---------------------
  nvtxMarkA("zg_index_build: pass 2 (fill + copy)");
  t0 = clk::now();
  const bool dev = (o.residency == ZG_RESIDENT_DEVICE);
  if (dev) {
    cudaError_t e = cudaMalloc((void**)&idx->dev, idx->total_bytes);
    if (e != cudaSuccess) {
      idx->dev = nullptr;
      return e == cudaErrorMemoryAllocation ? fail(ZG_ERR_OUT_OF_MEMORY, "zg_index_build: cudaMalloc of the index")
                                            : cuda_fail(e, "zg_index_build: cudaMalloc");
    }
  } else {
    try {
      idx->host.assign(idx->total_bytes, 0);
    } catch (const std::bad_alloc&) {
      return fail(ZG_ERR_OUT_OF_MEMORY, "zg_index_build: host image");
    }
  }
  struct DevFree {
    zg_index* i;
    bool armed = true;
    ~DevFree() {
      if (armed && i->dev) {
        cudaFree(i->dev);
        i->dev = nullptr;
      }
    }
  } dev_guard{idx};

  // segment byte sizes of bucket b at step s
  auto seg_rows = [&](int s, int b) -> uint64_t { return lay.cnt[b][s - 1]; };
  auto seg_pay = [&](int s, int b, int fmt) -> uint64_t {
    return fmt == ZG_FMT_SPARSE ? (uint64_t)lay.cnt[b][s] * 2 : (uint64_t)lay.cnt[b][s - 1] * words * 4;
  };
  uint64_t cap = o.pinned_chunk_bytes ? o.pinned_chunk_bytes : (64ull << 20);
  for (int s = 2; s <= L; ++s)
    for (int b = 0; b < nb; ++b) {
      uint64_t need = align_up(seg_rows(s, b) * 4 + 4, 16) + seg_pay(s, b, idx->steps[s - 1].fmt) + 16;
      cap = std::max(cap, need);
    }
  {
    uint64_t need1 = 16 + (uint64_t)std::max<int>(nb * 2, words * 4) + 32;
    cap = std::max(cap, need1);
  }
  Pinned buf[2];
  cudaEvent_t ev[2] = {nullptr, nullptr};
  bool ev_live[2] = {false, false};
  int cur = 0;
  zg_status st = ZG_OK;
  auto cleanup_events = [&]() {
    for (int i = 0; i < 2; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);
  };
  if (dev) {
    for (int i = 0; i < 2; ++i) {
      cudaError_t e = buf[i].ensure(cap);
      if (e != cudaSuccess) {
        cleanup_events();
        return e == cudaErrorMemoryAllocation ? fail(ZG_ERR_OUT_OF_MEMORY, "zg_index_build: cudaHostAlloc of a staging buffer")
                                              : cuda_fail(e, "zg_index_build: cudaHostAlloc of a staging buffer");
      }
      e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
      if (e != cudaSuccess) {
        cleanup_events();
        return cuda_fail(e, "zg_index_build: cudaEventCreate");
      }
    }
  }
  // Returns a staging area (device residency) or the host image location.
  auto begin_batch = [&](uint8_t** base) -> zg_status {
    if (!dev) return ZG_OK;
    if (ev_live[cur]) {
      cudaError_t e = cudaEventSynchronize(ev[cur]);
      if (e != cudaSuccess) return cuda_fail(e, "zg_index_build: staging event");
      ev_live[cur] = false;
    }
    *base = buf[cur].p;
    return ZG_OK;
  };
  auto end_batch = [&](uint64_t dst_rp, const uint8_t* src_rp, uint64_t n_rp, uint64_t dst_pay,
                       const uint8_t* src_pay, uint64_t n_pay) -> zg_status {
    if (!dev) return ZG_OK;
    cudaError_t e = cudaSuccess;
    if (injected(ZG_INJECT_COPY)) e = cudaErrorUnknown;
    if (e == cudaSuccess && n_rp) e = cudaMemcpyAsync(idx->dev + dst_rp, src_rp, n_rp, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && n_pay)
      e = cudaMemcpyAsync(idx->dev + dst_pay, src_pay, n_pay, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaEventRecord(ev[cur], stream);
    if (e != cudaSuccess) return cuda_fail(e, "zg_index_build: cudaMemcpyAsync to HBM");
    ev_live[cur] = true;
    cur ^= 1;
    return ZG_OK;
  };

  // step 1: the single empty-prefix row lists every first token present
  {
    const StepMeta& m = idx->steps[0];
    uint8_t* base = nullptr;
    if ((st = begin_batch(&base)) != ZG_OK) {
      cleanup_events();
      return st;
    }
    uint8_t* rp = dev ? base : idx->host.data() + m.off_rowptr;
    uint8_t* pay = dev ? base + 16 : idx->host.data() + m.off_payload;
    uint32_t r2[2] = {0u, (uint32_t)nb};
    std::memcpy(rp, r2, 8);
    if (m.fmt == ZG_FMT_SPARSE) {
      uint16_t* c = reinterpret_cast<uint16_t*>(pay);
      for (int b = 0; b < nb; ++b) c[b] = (uint16_t)lay.buckets[b].tok;
    } else {
      uint32_t* w = reinterpret_cast<uint32_t*>(pay);
      std::memset(w, 0, (size_t)words * 4);
      for (int b = 0; b < nb; ++b) w[lay.buckets[b].tok / 32] |= 1u << (lay.buckets[b].tok % 32);
    }
    if ((st = end_batch(m.off_rowptr, rp, 8, m.off_payload, pay, m.bytes_payload)) != ZG_OK) {
      cleanup_events();
      return st;
    }
  }
  for (int s = 2; s <= L; ++s) {
    const StepMeta& m = idx->steps[s - 1];
    int b0 = 0;
    while (b0 < nb) {
      // grow the batch while it fits the staging buffer
      int b1 = b0;
      uint64_t rows = 0, pay = 0;
      while (b1 < nb) {
        uint64_t r2 = rows + seg_rows(s, b1), p2 = pay + seg_pay(s, b1, m.fmt);
        if (b1 > b0 && align_up(r2 * 4 + 4, 16) + p2 + 16 > cap) break;
        rows = r2;
        pay = p2;
        ++b1;
      }
      const bool last = (b1 == nb);
      uint8_t* base = nullptr;
      if ((st = begin_batch(&base)) != ZG_OK) {
        cleanup_events();
        return st;
      }
      const uint64_t row0 = lay.rowoff[s][b0];
      const uint64_t pay0 = (m.fmt == ZG_FMT_SPARSE) ? lay.entoff[s][b0] * 2 : row0 * words * 4;
      uint8_t* rp = dev ? base : idx->host.data() + m.off_rowptr + row0 * 4;
      uint8_t* pp = dev ? base + align_up(rows * 4 + 4, 16) : idx->host.data() + m.off_payload + pay0;
      parallel_for(T, b1 - b0, [&](int64_t i) {
        int b = b0 + (int)i;
        uint32_t* rpd = reinterpret_cast<uint32_t*>(rp) + (lay.rowoff[s][b] - row0);
        uint8_t* pd = pp + ((m.fmt == ZG_FMT_SPARSE) ? (lay.entoff[s][b] * 2 - pay0)
                                                     : (lay.rowoff[s][b] * words * 4 - pay0));
        fill_bucket(lay, keys.data(), b, s, m.fmt, rpd, pd);
      });
      uint64_t n_rp = rows * 4;
      if (last) {
        reinterpret_cast<uint32_t*>(rp)[rows] = m.nnz;  // rowptr[rows] = nnz
        n_rp += 4;
      }
      if ((st = end_batch(m.off_rowptr + row0 * 4, rp, n_rp, m.off_payload + pay0, pp, pay)) != ZG_OK) {
        cleanup_events();
        return st;
      }
      b0 = b1;
    }
  }
  if (dev) {
    cudaError_t e = cudaStreamSynchronize(stream);
    cleanup_events();
    if (e != cudaSuccess) return cuda_fail(e, "zg_index_build: final synchronise");
  }
  idx->ms_sort = ms_sort;
  idx->ms_count = ms_count;
  idx->ms_fill = ms_since(t0);
  idx->ms_total = ms_since(t_all);
  dev_guard.armed = false;
  *out = guard.release();
  return ZG_OK;
}

uint64_t fnv1a(const uint8_t* p, size_t n, uint64_t h = 1469598103934665603ull) {
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 1099511628211ull;
  }
  return h;
}

const char kMagic[8] = {'Z', 'G', 'I', 'D', 'X', 0, 0, 1};

zg_status read_step_bytes(const zg_index* idx, int s, std::vector<uint8_t>* rp, std::vector<uint8_t>* pay) {
  const StepMeta& m = idx->steps[s - 1];
  rp->resize(m.bytes_rowptr);
  pay->resize(m.bytes_payload);
  if (idx->residency == ZG_RESIDENT_HOST) {
    std::memcpy(rp->data(), idx->host.data() + m.off_rowptr, m.bytes_rowptr);
    if (m.bytes_payload) std::memcpy(pay->data(), idx->host.data() + m.off_payload, m.bytes_payload);
    return ZG_OK;
  }
  cudaError_t e = cudaMemcpy(rp->data(), idx->dev + m.off_rowptr, m.bytes_rowptr, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && m.bytes_payload)
    e = cudaMemcpy(pay->data(), idx->dev + m.off_payload, m.bytes_payload, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the index back from the device");
  return ZG_OK;
}

}  // namespace
}  // namespace zg

zg::DevStep zg_index::dev_step(int s) const {
  const zg::StepMeta& m = steps[s - 1];
  zg::DevStep d;
  d.rowptr = reinterpret_cast<const uint32_t*>(dev + m.off_rowptr);
  d.col = m.fmt == ZG_FMT_SPARSE ? reinterpret_cast<const uint16_t*>(dev + m.off_payload) : nullptr;
  d.bitmap = m.fmt == ZG_FMT_DENSE ? reinterpret_cast<const uint32_t*>(dev + m.off_payload) : nullptr;
  d.rows = m.rows;
  d.nnz = m.nnz;
  d.words = m.words;
  d.max_fanout = m.max_fanout;
  d.fmt = m.fmt;
  return d;
}

using namespace zg;

extern "C" {

zg_status zg_index_build(const int32_t* sids, int64_t n, int32_t L, int32_t V, const zg_build_opts* opts,
                         void* stream, zg_index** out) {
  zg_build_opts o{};
  if (opts) o = *opts;
  try {
    return build_impl(sids, n, L, V, o, static_cast<cudaStream_t>(stream), out);
  } catch (const std::bad_alloc&) {
    return fail(ZG_ERR_OUT_OF_MEMORY, "zg_index_build: host allocation failed");
  } catch (const std::exception& e) {
    return fail(ZG_ERR_INVALID_ARG, std::string("zg_index_build: ") + e.what());
  }
}

void zg_debug_inject_build_failure(int32_t point, int32_t after) {
  g_inject_after.store(after < 0 ? 0 : after);
  g_inject_point.store(point);
}

zg_status zg_index_stats(const zg_index* idx, int32_t step, zg_step_stats* out) {
  if (!idx || !out) return fail(ZG_ERR_INVALID_ARG, "zg_index_stats: NULL argument");
  if (step < 1 || step > idx->L) return fail(ZG_ERR_INVALID_ARG, "zg_index_stats: step out of range");
  const StepMeta& m = idx->steps[step - 1];
  out->format = m.fmt;
  out->rows = m.rows;
  out->nnz = m.nnz;
  out->words_per_row = m.words;
  out->max_fanout = m.max_fanout;
  out->reserved = 0;
  out->mean_fanout = m.rows ? (double)m.nnz / m.rows : 0.0;
  out->legal_fraction = m.rows ? (double)m.nnz / ((double)m.rows * idx->V) : 0.0;
  out->bytes = m.bytes_rowptr + m.bytes_payload;
  return ZG_OK;
}

zg_status zg_index_info_get(const zg_index* idx, zg_index_info* out) {
  if (!idx || !out) return fail(ZG_ERR_INVALID_ARG, "zg_index_info_get: NULL argument");
  out->L = idx->L;
  out->V = idx->V;
  out->residency = idx->residency;
  out->reserved = 0;
  out->n_input = idx->n_input;
  out->n_unique = idx->n_unique;
  out->bytes = 0;
  out->dense_trie_bytes = 0;
  for (const auto& m : idx->steps) {
    out->bytes += m.bytes_rowptr + m.bytes_payload;
    out->dense_trie_bytes += (uint64_t)m.rows * (uint64_t)idx->V * 4;
  }
  out->ms_sort = idx->ms_sort;
  out->ms_count = idx->ms_count;
  out->ms_fill = idx->ms_fill;
  out->ms_total = idx->ms_total;
  return ZG_OK;
}

zg_status zg_index_export(const zg_index* idx, int32_t step, void* buf, size_t* bytes) {
  if (!idx || !bytes) return fail(ZG_ERR_INVALID_ARG, "zg_index_export: NULL argument");
  if (step < 1 || step > idx->L) return fail(ZG_ERR_INVALID_ARG, "zg_index_export: step out of range");
  const StepMeta& m = idx->steps[step - 1];
  const size_t pay = m.fmt == ZG_FMT_SPARSE ? (size_t)align_up(m.bytes_payload, 4) : (size_t)m.bytes_payload;
  const size_t need = 16 + (size_t)m.bytes_rowptr + pay;
  if (!buf) {
    *bytes = need;
    return ZG_OK;
  }
  if (*bytes < need) {
    *bytes = need;
    return fail(ZG_ERR_INVALID_ARG, "zg_index_export: buffer too small");
  }
  std::vector<uint8_t> rp, py;
  zg_status st = read_step_bytes(idx, step, &rp, &py);
  if (st != ZG_OK) return st;
  uint8_t* o = static_cast<uint8_t*>(buf);
  uint32_t head[4] = {(uint32_t)m.fmt, m.rows, m.nnz, m.words};
  std::memcpy(o, head, 16);
  std::memcpy(o + 16, rp.data(), rp.size());
  std::memset(o + 16 + rp.size(), 0, pay);
  if (!py.empty()) std::memcpy(o + 16 + rp.size(), py.data(), py.size());
  *bytes = need;
  return ZG_OK;
}

zg_status zg_index_save(const zg_index* idx, const char* path) {
  if (!idx || !path) return fail(ZG_ERR_INVALID_ARG, "zg_index_save: NULL argument");
  std::vector<uint8_t> img(idx->total_bytes);
  if (idx->residency == ZG_RESIDENT_HOST) {
    std::memcpy(img.data(), idx->host.data(), img.size());
  } else {
    cudaError_t e = cudaMemcpy(img.data(), idx->dev, img.size(), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "zg_index_save: reading the device image");
  }
  FILE* f = std::fopen(path, "wb");
  if (!f) return fail(ZG_ERR_IO, std::string("zg_index_save: cannot open ") + path);
  bool ok = std::fwrite(kMagic, 1, 8, f) == 8;
  int32_t hdr32[2] = {idx->L, idx->V};
  int64_t hdr64[2] = {idx->n_input, idx->n_unique};
  uint64_t tot = idx->total_bytes;
  ok = ok && std::fwrite(hdr32, 4, 2, f) == 2 && std::fwrite(hdr64, 8, 2, f) == 2 && std::fwrite(&tot, 8, 1, f) == 1;
  for (const auto& m : idx->steps) {
    int32_t a[1] = {m.fmt};
    uint32_t b[4] = {m.rows, m.nnz, m.words, m.max_fanout};
    uint64_t c[4] = {m.off_rowptr, m.off_payload, m.bytes_rowptr, m.bytes_payload};
    ok = ok && std::fwrite(a, 4, 1, f) == 1 && std::fwrite(b, 4, 4, f) == 4 && std::fwrite(c, 8, 4, f) == 4;
  }
  ok = ok && std::fwrite(img.data(), 1, img.size(), f) == img.size();
  uint64_t h = fnv1a(img.data(), img.size());
  ok = ok && std::fwrite(&h, 8, 1, f) == 1;
  ok = (std::fclose(f) == 0) && ok;
  if (!ok) return fail(ZG_ERR_IO, std::string("zg_index_save: write failed for ") + path);
  return ZG_OK;
}

}  // extern "C"

namespace {

// Structural check of a loaded image before anything reads it on the device:
// the invariants of the step-sliced index ("Why slice the index by decoding
// step": one row per (s-1)-prefix, a row's legal tokens ascending, entry e of
// step s is row e of step s+1).  Any table that passes keeps every kernel
// read in bounds: rowptr is non-decreasing from 0 to nnz, every token is
// below V, and every next-step row (an entry position) is below the next
// step's row count.
bool tables_valid(const zg_index& idx, const std::vector<uint8_t>& img) {
  const int L = idx.L;
  const uint32_t V = (uint32_t)idx.V;
  const uint32_t words = (V + 31) / 32;
  for (int s = 1; s <= L; ++s) {
    const StepMeta& m = idx.steps[s - 1];
    if (m.words != words) return false;
    if (s == 1 && m.rows != 1) return false;
    if (s < L && idx.steps[s].rows != m.nnz) return false;
    const uint64_t want_pay = (m.fmt == ZG_FMT_SPARSE) ? (uint64_t)m.nnz * 2 : (uint64_t)m.rows * words * 4;
    if (m.bytes_payload != want_pay || m.off_rowptr % 4 || m.off_payload % 4) return false;
    const uint32_t* rp = reinterpret_cast<const uint32_t*>(img.data() + m.off_rowptr);
    if (rp[0] != 0 || rp[m.rows] != m.nnz) return false;
    uint32_t mf = 0;
    for (uint32_t r = 0; r < m.rows; ++r) {
      if (rp[r + 1] < rp[r]) return false;
      const uint32_t F = rp[r + 1] - rp[r];
      if (F > V) return false;
      mf = std::max(mf, F);
      if (m.fmt == ZG_FMT_SPARSE) {
        const uint16_t* col = reinterpret_cast<const uint16_t*>(img.data() + m.off_payload) + rp[r];
        for (uint32_t j = 0; j < F; ++j)
          if (col[j] >= V || (j > 0 && col[j] <= col[j - 1])) return false;
      } else {
        const uint32_t* bm = reinterpret_cast<const uint32_t*>(img.data() + m.off_payload) + (uint64_t)r * words;
        uint32_t pc = 0;
        for (uint32_t w = 0; w < words; ++w) pc += (uint32_t)__builtin_popcount(bm[w]);
        if (V % 32 && (bm[words - 1] >> (V % 32))) return false;  // no bit at a token >= V
        if (pc != F) return false;
      }
    }
    if (mf != m.max_fanout) return false;
  }
  return true;
}

}  // namespace

extern "C" {

zg_status zg_index_load(const char* path, int32_t residency, void* stream, zg_index** out) {
  if (!path || !out) return fail(ZG_ERR_INVALID_ARG, "zg_index_load: NULL argument");
  *out = nullptr;
  if (residency != ZG_RESIDENT_DEVICE && residency != ZG_RESIDENT_HOST)
    return fail(ZG_ERR_INVALID_ARG, "zg_index_load: bad residency");
  FILE* f = std::fopen(path, "rb");
  if (!f) return fail(ZG_ERR_IO, std::string("zg_index_load: cannot open ") + path);
  std::unique_ptr<zg_index> idx(new zg_index());
  char mg[8];
  int32_t hdr32[2];
  int64_t hdr64[2];
  uint64_t tot = 0;
  bool ok = std::fread(mg, 1, 8, f) == 8 && std::memcmp(mg, kMagic, 8) == 0;
  ok = ok && std::fread(hdr32, 4, 2, f) == 2 && std::fread(hdr64, 8, 2, f) == 2 && std::fread(&tot, 8, 1, f) == 1;
  ok = ok && hdr32[0] >= 1 && hdr32[0] <= ZG_MAX_STEPS && hdr32[1] >= 1 && hdr32[1] <= 65536 &&
       tot < (1ull << 40);
  if (ok) {
    idx->L = hdr32[0];
    idx->V = hdr32[1];
    idx->n_input = hdr64[0];
    idx->n_unique = hdr64[1];
    idx->total_bytes = tot;
    idx->steps.resize(idx->L);
    for (auto& m : idx->steps) {
      int32_t a[1];
      uint32_t b[4];
      uint64_t c[4];
      ok = ok && std::fread(a, 4, 1, f) == 1 && std::fread(b, 4, 4, f) == 4 && std::fread(c, 8, 4, f) == 4;
      if (!ok) break;
      m.fmt = a[0];
      m.rows = b[0];
      m.nnz = b[1];
      m.words = b[2];
      m.max_fanout = b[3];
      m.off_rowptr = c[0];
      m.off_payload = c[1];
      m.bytes_rowptr = c[2];
      m.bytes_payload = c[3];
      ok = ok && (m.fmt == 0 || m.fmt == 1) && m.off_rowptr + m.bytes_rowptr <= tot &&
           m.off_payload + m.bytes_payload <= tot && m.bytes_rowptr == 4ull * ((uint64_t)m.rows + 1);
    }
  }
  std::vector<uint8_t> img;
  if (ok) {
    img.resize(tot);
    uint64_t h = 0;
    ok = std::fread(img.data(), 1, tot, f) == tot && std::fread(&h, 8, 1, f) == 1 && h == fnv1a(img.data(), tot);
  }
  ok = ok && tables_valid(*idx, img);
  std::fclose(f);
  if (!ok) return fail(ZG_ERR_IO, std::string("zg_index_load: short, corrupt or foreign file ") + path);
  idx->residency = residency;
  if (residency == ZG_RESIDENT_HOST) {
    idx->host = std::move(img);
  } else {
    cudaError_t e = cudaGetDevice(&idx->device);
    if (e == cudaSuccess) e = cudaMalloc((void**)&idx->dev, tot);
    if (e != cudaSuccess) {
      idx->dev = nullptr;
      return cuda_fail(e, "zg_index_load: cudaMalloc");
    }
    e = cudaMemcpyAsync(idx->dev, img.data(), tot, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      cudaFree(idx->dev);
      idx->dev = nullptr;
      return cuda_fail(e, "zg_index_load: upload");
    }
  }
  *out = idx.release();
  return ZG_OK;
}

void zg_index_free(zg_index* idx) {
  if (!idx) return;
  if (idx->dev) cudaFree(idx->dev);
  delete idx;
}

}  // extern "C"
