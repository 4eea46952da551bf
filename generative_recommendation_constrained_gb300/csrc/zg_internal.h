// Internal declarations of the zerogr library (host engine <-> kernels).
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/zerogr.h"

namespace zg {

constexpr uint32_t kDeadRow = 0xFFFFFFFFu;
constexpr int kChunk = 32;  // slots scored by one warp work item (one per lane)
constexpr int kItemBlocks = 1024;  // CTAs of a stand-alone selective step's item count, at most

// Device status bits (see zg_check_device_status).
constexpr uint32_t kStatusRow = 1u;
constexpr uint32_t kStatusToken = 2u;
constexpr uint32_t kStatusTimeout = 4u;
constexpr uint32_t kStatusTmem = 8u;
constexpr uint32_t kStatusSelect = 16u;  // a select found fewer candidates than its own cut guarantees

// Host-side metadata of one step table.
struct StepMeta {
  int32_t fmt = 0;
  uint32_t rows = 0, nnz = 0, words = 0, max_fanout = 0;
  uint64_t off_rowptr = 0, off_payload = 0;      // byte offsets in the image
  uint64_t bytes_rowptr = 0, bytes_payload = 0;  // payload bytes without padding
};

// Device view of one step table, passed to kernels by value.
struct DevStep {
  const uint32_t* rowptr;
  const uint16_t* col;     // sparse steps
  const uint32_t* bitmap;  // dense steps
  uint32_t rows, nnz, words, max_fanout;
  int32_t fmt;
};

// Per-step launch description built by the engine.
enum SelectMode : int32_t {
  kSelSparse = 0,   // selective scores, slot j = j-th legal token
  kSelDense = 1,    // selective scores, slot = token, illegal slots -inf
  kFullSparse = 2,  // full scores indexed by token, legal set from col[]
  kFullDense = 3,   // full scores indexed by token, legal set from bitmap
  kUncon = 4        // full scores, every token legal
};

struct StepLaunch {
  int32_t s, L, V, d, w_dtype;
  int32_t B, Wc, Wp;    // requests; beams per request now / at the previous step
  int32_t keep;         // survivors per request (beam, or K at the last step)
  int32_t beam;         // beam width (stride of state arrays)
  int32_t K;
  DevStep tab;          // zeroed in unconstrained mode
  int32_t mode;         // SelectMode
  int32_t S;            // slot stride of a beam's row of Z (selective) or padded V (full)
  int32_t nch;          // chunks per beam (selective), else 0
  int64_t zq;           // stride of a request's rows of Z (floats): the slots of beam k of
                        // request q start at q*zq + k*S.  Constant across the steps a fused
                        // kernel runs, so requests never overwrite each other's slots.
  int64_t pq;           // stride of a request's chunk partials (float2): q*pq + k*nch + c
  // state entering the step (NULL at s = 1: one root beam, row 0, cum 0, h = u)
  const uint32_t* row_in;
  const float* cum_in;
  const int32_t* par_in;   // parent index (within the request) of each beam
  const int32_t* tok_in;   // token chosen at step s-1
  const float* u;          // [B][d]
  const float* hpre;       // [B*Wc][d] hidden vectors given by the light decoder (then no gather-add), or null
  const float* h_prev;     // [B*Wp][d] hidden of the previous step's beams (s >= 3)
  const float* C_prev;     // C_{s-1} [V][d] (s >= 2)
  const void* W;           // W_s [V][d]
  float* h_out;            // [B*Wc][d] hidden of this step's beams, or NULL
  // scores
  float* Z;                // [B][zq]
  float2* part;            // [B][pq] (max, sum exp) of the legal tokens per chunk
  const float2* part_all;  // [B][pq] (max, sum exp) of every token per chunk: score-first
                           // order (log-softmax over the codebook), else NULL
  int32_t* bscan;          // stand-alone selective steps: [B*Wc] each beam's first non-empty
                           // chunk counted from the first of its counting CTA, [B*Wc] its first
                           // index entry, [B*Wc] its fan-out, [kItemBlocks] chunks per CTA
  int32_t mask_by_beam;    // tab.bitmap holds one row per beam (b = q*Wc + k), not per
                           // index row: a sparse step's legal lists expanded (score-first)
  // chunk-top select (full steps whose scores were not written): ptop[q*pq +
  // k*nch + c] = (second-largest legal z, offset of the lowest token holding the
  // largest) of each chunk, and the operands the projection used, to re-score a
  // chunk: hq (fp32 hidden, fp32 weights) or hq_hi (+ hq_lo when split) [B*Wc][d]
  const float2* ptop;
  const float* hq;
  const void* hq_hi;
  const void* hq_lo;
  // outputs
  uint32_t* row_out;       // [B*beam] (s < L)
  float* cum_out;          // [B*beam]
  int32_t* tok_hist;       // [L-1][B*beam] token chosen at step j (j = 1..L-1)
  int32_t* par_hist;       // [L-1][B*beam] parent index of that beam
  int32_t* out_sids;       // [B][K][L] (s = L)
  float* out_scores;       // [B][K]
  uint32_t* status;        // device status word
};

// What the full-projection epilogues write besides the scores: for every
// 32-token chunk of every beam row, (max, sum exp(z - max)) over the legal
// tokens of the chunk, the same partials the selective kernels produce.
struct FullEpi {
  float2* part;            // [M][ldz/32], or null (no partials)
  float2* ptop;            // [M][ldz/32] (second-largest legal z, offset 0..31 of the lowest token holding the
                           // largest, as int bits) of every chunk, or null; with it the scores need not be
                           // written (chunk-top select)
  float2* part_all;        // [M][ldz/32] (max, sum exp) over every token < V, or null
  const uint32_t* bitmap;  // dense step's bitmap rows; null: every token < V is legal
  const uint32_t* rows;    // [M] index row of each beam (kDeadRow: dead); null: row 0
  int words;               // bitmap words a row
  int by_m;                // bitmap row m belongs to beam row m (rows unused)
  uint32_t nrows;          // bitmap rows: an index row at or beyond it is flagged kStatusRow
                           // and treated as dead (never read)
  uint32_t* status;        // device status word (for that flag)
};

#ifdef __CUDACC__
// Legal tokens of chunk `chunk` of beam row `m` as a 32-bit mask.
__device__ __forceinline__ uint32_t epi_legal_mask(const FullEpi& e, int m, int chunk, int V) {
  uint32_t mask = 0xFFFFFFFFu;
  if (e.bitmap) {
    const uint32_t r = e.by_m ? (uint32_t)m : (e.rows ? e.rows[m] : 0u);
    if (r == kDeadRow) return 0u;
    if (r >= e.nrows) {
      atomicOr(e.status, kStatusRow);
      return 0u;
    }
    mask = e.bitmap[(size_t)r * e.words + chunk];
  }
  const int rem = V - chunk * 32;
  if (rem < 32) mask &= (rem <= 0) ? 0u : ((1u << rem) - 1u);
  return mask;
}
#endif

// kernels (kernels.cu)
// after_count (optional): an event recorded between the chunk-counting and the scoring kernel
cudaError_t launch_selective(const StepLaunch& a, cudaStream_t st, cudaEvent_t after_count = nullptr);
// a one-thread kernel that returns once `ns` nanoseconds of the GPU's global timer have passed
// (at most about a second), so that the host can enqueue the launches behind it
cudaError_t launch_delay(unsigned long long ns, cudaStream_t st);
cudaError_t launch_gather_add(const StepLaunch& a, float* H, cudaStream_t st);
cudaError_t launch_full_simt(const StepLaunch& a, const float* H, const FullEpi& epi, cudaStream_t st);
cudaError_t launch_select(const StepLaunch& a, cudaStream_t st);
cudaError_t launch_legal_mask(const StepLaunch& a, cudaStream_t st);
int sm_count();  // streaming multiprocessors of the current device
// naive legal-only contrast (naive.cu): compaction + temporary matrix, then the scores
// (cap: rows the list and the temporary matrix hold; candidates beyond it are
// dropped and flagged kStatusRow)
cudaError_t launch_naive_compact(const StepLaunch& a, int32_t* cnt, int32_t* off, int4* list, void* temp,
                                 int64_t cap, cudaStream_t st);
cudaError_t launch_naive_dot(const StepLaunch& a, const int32_t* off, const int4* list, const void* temp,
                             const float* H, int64_t cap, cudaStream_t st);
// A device region the fused kernel prefetches into L2 (16-byte aligned).
struct PrefetchRegion {
  const void* ptr;
  uint64_t bytes;
};
constexpr int kMaxPrefetch = 24;
// Steps s0..L (all selective) in one cluster kernel, G CTAs per request;
// steps[] holds the launch description of every step (1-based s at [s-1]);
// pf[] lists the tables to prefetch into L2 at launch.
cudaError_t launch_decode_cluster(const StepLaunch* steps, int s0, int L, int G, const PrefetchRegion* pf, int npf,
                                  cudaStream_t st);
cudaError_t status_word(uint32_t** dev_ptr);   // per-device status word address
// One step of the light decoder (deco.cu): the new positions' rows through
// every layer, keys and values stored, hidden vectors of the beams entering
// step s into H.
struct DecoStep {
  int32_t s, L, B, Wc, beam, M, d, heads;
  const float* concepts;   // [B][M][d] (the decode's input)
  const int32_t* tok_in;   // [B*beam] token chosen at step s-1 (s >= 2)
  const float* cum_in;     // [B*beam] entering scores (-inf: dead beam), s >= 2
  const int32_t* par_hist; // [L-1][B*beam] parent index history
  float *X, *A, *Q, *O, *F;                 // [rows][d] (F: [rows][ffn]) work rows
  float *Kc, *Vc;                           // [layers][B*M][d] concept keys / values
  float *Ks, *Vs;                           // [layers][L+1][B*beam][d] token keys / values by step
  float* H;                                 // [B*Wc][d] output hidden vectors
};
cudaError_t launch_deco_step(const zg_deco& w, const DecoStep& a, cudaStream_t st);
// tensor-core full projection (kernels_tc.cu): H = hi + lo in W's half type
cudaError_t launch_split_h(const float* H, void* hi, void* lo, size_t n, int w_dtype, cudaStream_t st);
cudaError_t launch_full_tc(const void* hi, const void* lo, const void* W, float* Z, int M, int V, int d, int ldz,
                           int w_dtype, const FullEpi& epi, uint32_t* status, cudaStream_t st);
// polls of an mbarrier before a pipeline wait of the tensor-core kernel gives
// up (0: the default); the drain waits before exit always use the default
void set_wait_limit(uint32_t polls);
// Unique id of the calling thread's current CUDA context (the driver's
// cuCtxGetId; a context created after cudaDeviceReset gets a new id).  Device
// addresses of __device__ variables are cached per context under this id.
cudaError_t current_context_id(unsigned long long* id);
// Work counts of the beams entering a step (tracing only): counters[0..3] =
// live beams, legal slots, chunks, index bytes; mask = V-bit set of touched
// tokens.  Both must be zeroed by the caller.
cudaError_t launch_trace_touch(const StepLaunch& a, unsigned long long* counters, uint32_t* mask,
                               cudaStream_t st);

// error reporting (engine.cpp)
zg_status fail(zg_status code, const std::string& msg);
zg_status cuda_fail(cudaError_t e, const char* what);

}  // namespace zg

struct zg_index {
  int32_t L = 0, V = 0, residency = 0;
  int64_t n_input = 0, n_unique = 0;
  std::vector<zg::StepMeta> steps;
  uint64_t total_bytes = 0;
  uint8_t* dev = nullptr;          // device image (residency device)
  std::vector<uint8_t> host;       // host image (residency host)
  int32_t device = -1;
  double ms_sort = 0, ms_count = 0, ms_fill = 0, ms_total = 0;

  zg::DevStep dev_step(int s) const;  // s is 1-based
};

struct zg_plan {
  int32_t L = 0, B = 0, beam = 0;
  int32_t fused = 8;            // CTAs per cluster of the fused kernel; 0 = no fusion
  int32_t order = 0;            // zg_order
  int32_t hidden = 0;           // zg_hidden_rounding of the tensor-core full projection
  int32_t scores = 0;           // zg_full_scores: how full steps hand their scores to the select
  float fused_ms[5] = {-1, -1, -1, -1, -1};  // tuned decode times with 1, 2, 4, 8, 16 CTAs a cluster
  float plan_ms = -1.f;                      // tuned decode time of the kept plan
  std::vector<uint8_t> variant;  // [L]
  std::vector<float> step_ms;    // [L][2]
};
