// C-ABI entry points: argument checks, workspace planning, tensor-map encoding and
// the launch sequence of the forward and backward passes.  All device work is
// enqueued on the caller's stream; nothing here synchronises the host.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "flce.h"
#include "host_internal.h"
#include "internal.cuh"
#include "ptx.cuh"
#include "small_kernels.cuh"
#include "vocab_order.cuh"

namespace flce {

// One thread waits, with the same bounded wait the tensor-core kernels use, on an
// mbarrier that nothing ever arrives on: after the limit it sets the error bit and the
// kernel returns (nothing faults or hangs).
__global__ void k_wait_timeout_selftest(unsigned long long* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
}

namespace {

constexpr size_t kAlign = 256;
constexpr int kLseGroupMin = 4;  // vocabulary tiles per forward unit: range searched
constexpr int kLseGroupMax = 8;
constexpr int kPlanPairs = 76;   // SM pairs of a GB300 (152 SMs), for the planner
// Token tiles per band of the M-first schedules (linear-LSE, dZ): 16 tiles of 256 rows
// keep 16 x 256 x Hd x 2 bytes of H (32 MiB at Hd 4096) in L2 while W streams past
// once per band, instead of H streaming past once per vocabulary tile when it does
// not fit in L2 (N = 32768: 224 MiB).
constexpr int kBandM = 16;
// bf16 dZ chunk bytes.  Measured sustained on one GB300 (forward + backward per step,
// 100-step runs at the power cap): 512 MiB runs the Llama-3-, Gemma-2- and packed-shaped
// heads within 0.7-1.0% of 1 GiB for 27-45% less peak extra memory; 384 and 256 MiB cost
// 0.5-1.7% and 1.1-2.1% more (more launches, and a dH read-modify-write per chunk).
constexpr size_t kDefaultChunkBudget = size_t(512) << 20;
constexpr int kMaxDevices = 64;

thread_local int t_last_cuda = 0;
thread_local uint64_t t_launches = 0;
struct EventSink {
  void* const* start = nullptr;
  void* const* end = nullptr;
  int* ids = nullptr;
  int cap = 0;
  int used = 0;
};
thread_local EventSink t_sink;

struct DeviceState {
  bool initialized = false;
  flce_status status = FLCE_OK;
  int sms = 0;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool mul_ok(size_t a, size_t b, size_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(size_t a, size_t b, size_t* out) { return !__builtin_add_overflow(a, b, out); }

// Reserve `bytes` at 256-byte alignment; false on overflow.
bool reserve(size_t* cursor, size_t bytes, size_t* offset) {
  *offset = align_up(*cursor);
  return add_ok(*offset, bytes, cursor);
}

flce_status cuda_fail(cudaError_t e) {
  t_last_cuda = static_cast<int>(e);
  return FLCE_ERR_CUDA;
}

// Launch bookkeeping: optional event pair around the launch, launch counter.
template <class F>
cudaError_t launch(int kernel_id, cudaStream_t st, F&& f) {
  const bool rec = t_sink.cap > 0 && t_sink.used < t_sink.cap;
  if (rec) cudaEventRecord(static_cast<cudaEvent_t>(t_sink.start[t_sink.used]), st);
  cudaError_t e = f();
  if (rec) {
    cudaEventRecord(static_cast<cudaEvent_t>(t_sink.end[t_sink.used]), st);
    t_sink.ids[t_sink.used] = kernel_id;
    ++t_sink.used;
  }
  ++t_launches;
  return e;
}

flce_status device_setup(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceState& d = g_dev[dev];
  if (!d.initialized) {
    int major = 0, minor = 0, count = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e);
    if (major != 10 || minor != 3) {
      d.status = FLCE_ERR_UNSUPPORTED;
    } else {
      if ((e = set_gemm_smem_attributes_fwd()) != cudaSuccess) return cuda_fail(e);
      if ((e = set_gemm_smem_attributes_bwd()) != cudaSuccess) return cuda_fail(e);
      std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
          g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      });
      d.status = g_encode ? FLCE_OK : FLCE_ERR_CUDA;
    }
    d.sms = count;
    d.initialized = true;
  }
  *sms = d.sms;
  return d.status;
}

// 2-D bf16 tensor map with 128-byte swizzle: dims {inner, outer}, row pitch in bytes.
bool tmap_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
             uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  std::memset(tm, 0, sizeof(*tm));
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int cdiv(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// CTA pairs run one 256-row tile each: an even grid of at most one CTA per SM.
int pair_grid(int units, int sms) { return 2 * std::max(1, std::min(units, sms / 2)); }

// ------------------------------------------------------------------ planning
struct FwdPlan {
  int m_tiles = 0, v_tiles = 0, group = 0, n_groups = 0, k_blocks = 0;
  int dot_blocks = 0, merge_blocks = 0;
  size_t off_pm = 0, off_ps = 0, off_t = 0, off_sums = 0, off_counts = 0, total = 0;
};

flce_status check_sizes(int64_t N, int64_t Hd, int64_t V) {
  if (N < 0 || Hd <= 0 || V <= 0) return FLCE_ERR_ARG;
  if (Hd % 8 != 0) return FLCE_ERR_ALIGN;
  // TMA coordinates are int32 and the label is kept as int32 on the device.
  const int64_t lim = (int64_t(1) << 31) - 512;
  if (N > lim || Hd > lim || V > lim) return FLCE_ERR_OVERFLOW;
  size_t b;
  if (!mul_ok(size_t(N), size_t(Hd), &b) || !mul_ok(b, 4, &b)) return FLCE_ERR_OVERFLOW;
  if (!mul_ok(size_t(V), size_t(Hd), &b) || !mul_ok(b, 4, &b)) return FLCE_ERR_OVERFLOW;
  return FLCE_OK;
}

// Vocabulary tiles per forward unit (4..8): the count whose round-robin assignment of
// units to the SM pairs has the smallest makespan in tiles (ties: the larger count,
// which means fewer partials).  Units of one group index share their W tiles.
int64_t count_congruent(int64_t lo, int64_t hi, int64_t r, int64_t mod) {  // #{u in [lo, hi): u % mod == r}
  if (hi <= lo) return 0;
  auto upto = [&](int64_t x) { return x <= r ? int64_t(0) : (x - 1 - r) / mod + 1; };  // #{u in [0, x)}
  return upto(hi) - upto(lo);
}

// Makespan in tiles of the banded M-first unit order for G tiles per unit.  Every unit
// has G tiles except those of the last group, which sit at the end of each band; with
// more than kMaxBandsExact bands the tail is counted as if the order were unbanded
// (the choice of G then hardly matters).
constexpr int64_t kMaxBandsExact = 64;
int64_t lse_makespan(int m_tiles, int v_tiles, int G, int band, int pairs) {
  const int64_t ng = cdiv(v_tiles, G);
  const int64_t units = int64_t(m_tiles) * ng;
  const int64_t last = v_tiles - (ng - 1) * G;  // tiles in each unit of the last group
  const int64_t bw = (band > 0 && band < m_tiles && cdiv(m_tiles, band) <= kMaxBandsExact) ? band : m_tiles;
  int64_t t = 0;
  for (int p = 0; p < pairs; ++p) {
    int64_t tail = 0;
    for (int64_t b0 = 0; b0 < m_tiles; b0 += bw) {  // the band of M-tiles [b0, b0 + w)
      const int64_t w = std::min<int64_t>(bw, m_tiles - b0);
      const int64_t start = b0 * ng + (ng - 1) * w;  // its last group's first unit
      tail += count_congruent(start, start + w, p, pairs);
    }
    t = std::max(t, G * count_congruent(0, units, p, pairs) - (G - last) * tail);
  }
  return t;
}

int pick_lse_group(int m_tiles, int v_tiles, int pairs) {
  int best_g = kLseGroupMin;
  int64_t best_t = -1;
  for (int G = kLseGroupMin; G <= kLseGroupMax; ++G) {
    const int64_t t = lse_makespan(m_tiles, v_tiles, G, kBandM, pairs);
    if (best_t < 0 || t <= best_t) {
      best_t = t;
      best_g = G;
    }
  }
  return best_g;
}

flce_status plan_forward(int64_t N, int64_t Hd, int64_t V, int pairs, FwdPlan* p) {
  flce_status s = check_sizes(N, Hd, V);
  if (s != FLCE_OK) return s;
  p->m_tiles = cdiv(N, kPairM);  // CTA pairs: 256 token rows per tile
  p->v_tiles = cdiv(V, kBN);
  p->group = pick_lse_group(p->m_tiles, p->v_tiles, pairs);
  p->n_groups = cdiv(p->v_tiles, p->group);
  p->k_blocks = cdiv(Hd, kBK);
  p->dot_blocks = static_cast<int>(std::min<int64_t>(std::max<int64_t>(cdiv(N, kDotWarps), 1), kDotMaxBlocks));
  p->merge_blocks = std::max(cdiv(N, kMergeRows), 1);
  size_t cur = 0, part;
  if (!mul_ok(size_t(p->n_groups) * kEpiSplit, size_t(N), &part) || !mul_ok(part, 4, &part))
    return FLCE_ERR_OVERFLOW;
  if (!reserve(&cur, part, &p->off_pm) || !reserve(&cur, part, &p->off_ps) ||
      !reserve(&cur, size_t(N) * 4, &p->off_t) || !reserve(&cur, size_t(p->merge_blocks) * 8, &p->off_sums) ||
      !reserve(&cur, size_t(p->dot_blocks) * 8, &p->off_counts))
    return FLCE_ERR_OVERFLOW;
  p->total = align_up(cur);
  return FLCE_OK;
}

// Scratch of the vocabulary order, at offsets from `base` inside a larger workspace.
struct VocabPlan {
  int n_seg = 0;
  int64_t rows_per_seg = 0;
  size_t off_key = 0, off_word0 = 0, off_word1 = 0, off_perm = 0, off_inv = 0, off_part = 0, off_hbar = 0;
};

bool plan_vocab(int64_t N, int64_t Hd, int64_t V, size_t* cur, VocabPlan* p) {
  p->n_seg = static_cast<int>(std::min<int64_t>(128, std::max<int64_t>(1, cdiv(N, 64))));
  p->rows_per_seg = std::max<int64_t>(1, cdiv(N, p->n_seg));
  size_t part;
  if (!mul_ok(size_t(p->n_seg), size_t(Hd), &part) || !mul_ok(part, 4, &part)) return false;
  return reserve(cur, size_t(V) * 4, &p->off_key) && reserve(cur, size_t(V) * 8, &p->off_word0) &&
         reserve(cur, size_t(V) * 8, &p->off_word1) && reserve(cur, size_t(V) * 4, &p->off_perm) &&
         reserve(cur, size_t(V) * 4, &p->off_inv) && reserve(cur, part, &p->off_part) &&
         reserve(cur, size_t(Hd) * 4, &p->off_hbar);
}

struct BwdPlan {
  int64_t Vc = 0;              // widest chunk: the dZ buffer's row pitch in elements
  int n_chunks = 0;
  int64_t v_tiles = 0;         // 256-column tiles of the vocabulary, split over the chunks
  // Chunk c covers vocabulary columns [chunk_begin(c), chunk_begin(c + 1)): the tiles are
  // dealt out as evenly as whole tiles allow, so widths differ by at most one tile.
  int64_t chunk_begin(int c, int64_t V) const {
    return c >= n_chunks ? V : (int64_t(c) * v_tiles / n_chunks) * kBN;
  }
  int dh_split = 1;            // K parts per dH output tile (1: no split)
  int nz_rows = 0, nz_ld = 0;  // token blocks x vocabulary blocks of the dZ block flags
  int dh_mask_ld = 0, dw_mask_ld = 0, mask_tok_tiles = 0, mask_voc_tiles = 0;
  bool sort = false, split = false;
  VocabPlan vocab;
  size_t off_rows = 0, off_dz = 0, off_dz_lo = 0, off_dh = 0, off_dh_parts = 0, off_nz = 0, off_dh_mask = 0,
         off_dw_mask = 0, off_wperm = 0, total = 0;
  // row compaction: compact RowInfo [n_cap], row map [N], compact H [n_cap][Hd] bf16,
  // per-block counts and the compact row count
  int64_t n_cap = 0;
  int compact_blocks = 0;
  size_t off_rows_c = 0, off_map = 0, off_hc = 0, off_blk = 0, off_nrows = 0;
};

// K parts per dH output tile: the count (1 .. kMaxDhSplit, at most the chunk's K blocks)
// whose units fill the launch's waves best, in waves of whole-K tiles.  A split costs
// (parts - 1) fp32 [N, Hd] buffers and a pass that adds them, so it is taken only when it
// shortens the launch by at least kMinDhSplitGain: 256 tiles on 76 pairs (4 waves ->
// 3.5) split in 2, 128 tiles (2 -> 1.75) in 4, 512 tiles (7 -> 6.75) not at all.
constexpr int kMaxDhSplit = 4;
constexpr double kMinDhSplitGain = 0.05;
int choose_dh_split(int64_t tiles, int pairs, int64_t k_blocks) {
  const double whole = static_cast<double>(cdiv(tiles, pairs));
  int best = 1;
  double best_t = whole;
  for (int S = 2; S <= kMaxDhSplit && S <= k_blocks; ++S) {
    const double t = static_cast<double>(cdiv(tiles * S, pairs)) / S;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = S;
    }
  }
  return best_t <= (1.0 - kMinDhSplitGain) * whole ? best : 1;
}

// The chunk budget covers the bf16 dZ chunk (two of them, value and rounding remainder, in
// the compensated mode) and, with the sorted vocabulary, the bf16 copy of the chunk's
// weight rows in sorted order: at most budget / (2N (x2) (+ 2Hd)) columns, a multiple of
// 256.  The vocabulary's 256-column tiles are then dealt out over the fewest chunks that
// bound allows, as evenly as whole tiles allow, so the last chunk is not a thin remainder
// with its own launch tails.
flce_status plan_backward(int64_t N, int64_t Hd, int64_t V, size_t budget, unsigned options, BwdPlan* p) {
  flce_status s = check_sizes(N, Hd, V);
  if (s != FLCE_OK) return s;
  if ((options & ~unsigned(FLCE_BWD_SORT_VOCAB | FLCE_BWD_COMPENSATED)) != 0) return FLCE_ERR_ARG;
  p->sort = (options & FLCE_BWD_SORT_VOCAB) != 0;
  p->split = (options & FLCE_BWD_COMPENSATED) != 0;
  if (budget == 0) budget = kDefaultChunkBudget;
  const int64_t v_round = int64_t(cdiv(V, kBN)) * kBN;
  const size_t per_col = size_t(N) * (p->split ? 4 : 2) + (p->sort ? size_t(Hd) * 2 : 0);
  int64_t vc_max = N > 0 ? static_cast<int64_t>(std::min<size_t>(budget / per_col, size_t(v_round))) : v_round;
  vc_max = vc_max / kBN * kBN;
  if (vc_max < kBN) vc_max = kBN;
  p->v_tiles = cdiv(V, kBN);
  p->n_chunks = cdiv(V, vc_max);                                 // fewest chunks within the bound
  const int64_t vc = int64_t(cdiv(p->v_tiles, p->n_chunks)) * kBN;  // widest chunk, <= vc_max
  p->Vc = vc;
  // the compensated mode's two-part A operand is not split
  p->dh_split = p->split ? 1 : choose_dh_split(int64_t(cdiv(N, kPairM)) * cdiv(Hd, kBN), kPlanPairs, cdiv(vc, kBK));
  p->nz_rows = cdiv(N, 64);
  p->nz_ld = static_cast<int>(vc / 64);
  p->dh_mask_ld = cdiv(p->nz_ld, 32);
  p->dw_mask_ld = cdiv(p->nz_rows, 32);
  p->mask_tok_tiles = cdiv(N, kPairM);
  p->mask_voc_tiles = static_cast<int>(vc / kPairM);
  size_t cur = 0, dz, dh = 0, parts = 0;
  if (!mul_ok(size_t(N), size_t(vc), &dz) || !mul_ok(dz, 2, &dz)) return FLCE_ERR_OVERFLOW;
  if ((p->n_chunks > 1 || p->dh_split > 1) && (!mul_ok(size_t(N), size_t(Hd), &dh) || !mul_ok(dh, 4, &dh)))
    return FLCE_ERR_OVERFLOW;
  if (p->dh_split > 1 && !mul_ok(dh, size_t(p->dh_split - 1), &parts)) return FLCE_ERR_OVERFLOW;
  p->n_cap = int64_t(cdiv(N, kPairM)) * kPairM;
  p->compact_blocks = std::max(cdiv(N, kCompactRows), 1);
  size_t hc;
  if (!mul_ok(size_t(p->n_cap), size_t(Hd), &hc) || !mul_ok(hc, 2, &hc)) return FLCE_ERR_OVERFLOW;
  if (!reserve(&cur, size_t(p->n_cap) * sizeof(RowInfo), &p->off_rows_c) ||
      !reserve(&cur, size_t(N) * 4, &p->off_map) || !reserve(&cur, hc, &p->off_hc) ||
      !reserve(&cur, size_t(p->compact_blocks) * 4, &p->off_blk) || !reserve(&cur, 4, &p->off_nrows))
    return FLCE_ERR_OVERFLOW;
  if (!reserve(&cur, size_t(N) * sizeof(RowInfo), &p->off_rows) || !reserve(&cur, dz, &p->off_dz) ||
      !reserve(&cur, p->split ? dz : 0, &p->off_dz_lo) || !reserve(&cur, dh, &p->off_dh) ||
      !reserve(&cur, parts, &p->off_dh_parts) || !reserve(&cur, size_t(p->nz_rows) * size_t(p->nz_ld), &p->off_nz) ||
      !reserve(&cur, size_t(p->mask_tok_tiles) * p->dh_mask_ld * 4, &p->off_dh_mask) ||
      !reserve(&cur, size_t(p->mask_voc_tiles) * p->dw_mask_ld * 4, &p->off_dw_mask))
    return FLCE_ERR_OVERFLOW;
  if (p->sort) {
    size_t wp;
    if (!mul_ok(size_t(vc), size_t(Hd), &wp) || !mul_ok(wp, 2, &wp) || !reserve(&cur, wp, &p->off_wperm) ||
        !plan_vocab(N, Hd, V, &cur, &p->vocab))
      return FLCE_ERR_OVERFLOW;
  }
  p->total = align_up(cur);
  return FLCE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

int check_device() {
  int sms = 0;
  return device_setup(&sms);
}

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

// Sort keys (mean raw logit per vocabulary row), then the stable descending order:
// perm[position] = row, inv[row] = position (inv may be null).
flce_status vocab_order_impl(const void* H, const void* W, int64_t N, int64_t Hd, int64_t V, const VocabPlan& vp,
                             uint8_t* ws, float* key, int32_t* perm, int32_t* inv, unsigned long long* err, int sms,
                             cudaStream_t st) {
  const __nv_bfloat16* Hb = static_cast<const __nv_bfloat16*>(H);
  const __nv_bfloat16* Wb = static_cast<const __nv_bfloat16*>(W);
  unsigned long long* w0 = reinterpret_cast<unsigned long long*>(ws + vp.off_word0);
  unsigned long long* w1 = reinterpret_cast<unsigned long long*>(ws + vp.off_word1);
  float* part = reinterpret_cast<float*>(ws + vp.off_part);
  float* hbar = reinterpret_cast<float*>(ws + vp.off_hbar);
  cudaError_t e;
  if (N == 0) {  // no rows: every key is 0 (hbar = 0), the order is the identity
    if ((e = cudaMemsetAsync(hbar, 0, size_t(Hd) * 4, st)) != cudaSuccess) return cuda_fail(e);
  } else {
    e = launch(FLCE_KERNEL_VOCAB_KEYS, st, [&] {
      k_col_partial<<<dim3(cdiv(Hd, 8 * kColThreads), vp.n_seg), kColThreads, 0, st>>>(Hb, N, Hd, vp.rows_per_seg,
                                                                                        part);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch(FLCE_KERNEL_VOCAB_KEYS, st, [&] {
      k_col_mean<<<cdiv(Hd, 256), 256, 0, st>>>(part, vp.n_seg, Hd, N, hbar);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return cuda_fail(e);
  }
  const int row_blocks = std::min(cdiv(V, kRowCopyThreads / 32), 8 * sms);
  e = launch(FLCE_KERNEL_VOCAB_KEYS, st, [&] {
    k_vocab_keys<<<row_blocks, kRowCopyThreads, 0, st>>>(Wb, hbar, V, Hd, key, w0);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch(FLCE_KERNEL_VOCAB_SORT, st, [&] {
    k_sort_runs<<<cdiv(V, kSortSeg), kSortThreads, 0, st>>>(w0, w1, V);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned long long* cur = w1;
  unsigned long long* nxt = w0;
  const int merge_blocks = std::min(cdiv(V, kMergeSortThreads), 8 * sms);
  for (int64_t L = kSortSeg; L < V; L *= 2) {
    e = launch(FLCE_KERNEL_VOCAB_SORT, st, [&] {
      k_merge_runs<<<merge_blocks, kMergeSortThreads, 0, st>>>(cur, nxt, V, L);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return cuda_fail(e);
    std::swap(cur, nxt);
  }
  e = launch(FLCE_KERNEL_VOCAB_SORT, st, [&] {
    k_order_finish<<<merge_blocks, kMergeSortThreads, 0, st>>>(cur, V, perm, inv, err);
    return cudaGetLastError();
  });
  return e == cudaSuccess ? FLCE_OK : cuda_fail(e);
}

// Forward over the weight rows [v_offset, v_offset + V) of a vocabulary of V_total
// (v_offset = 0 and V_total = V without sharding).  reduction -1: no loss output (the
// sharded forward, whose per-shard LSE and target logits are merged later).
flce_status forward_impl(const void* H, const void* W, const int64_t* labels, int64_t N, int64_t Hd, int64_t V,
                         int64_t v_offset, int64_t V_total, int64_t ignore_index, float softcap, int reduction,
                         float* loss, float* lse, float* target_logit, int64_t* counts, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (reduction < -1 || reduction > 2 || softcap != softcap) return FLCE_ERR_ARG;
  FwdPlan pl;
  flce_status s = plan_forward(N, Hd, V, kPlanPairs, &pl);
  if (s != FLCE_OK) return s;
  if (!W || (reduction >= 0 && !loss) || !counts) return FLCE_ERR_ARG;
  if (N > 0 && (!H || !labels || !lse || !workspace)) return FLCE_ERR_ARG;
  if (!aligned(W, 16) || (H && !aligned(H, 16)) || !aligned(counts, 8) || (labels && !aligned(labels, 8)) ||
      (loss && !aligned(loss, 4)) || (lse && !aligned(lse, 4)) || (target_logit && !aligned(target_logit, 4)))
    return FLCE_ERR_ALIGN;
  if (N > 0 && (workspace_bytes < pl.total || !aligned(workspace, kAlign))) return FLCE_ERR_WORKSPACE;
  int sms = 0;
  if ((s = device_setup(&sms)) != FLCE_OK) return s;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(counts, 0, 3 * sizeof(int64_t), st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (N == 0) {
    if ((reduction == FLCE_REDUCTION_MEAN || reduction == FLCE_REDUCTION_SUM) &&
        (e = cudaMemsetAsync(loss, 0, sizeof(float), st)) != cudaSuccess)
      return cuda_fail(e);
    return FLCE_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* part_m = reinterpret_cast<float*>(ws + pl.off_pm);
  float* part_s = reinterpret_cast<float*>(ws + pl.off_ps);
  float* t_ws = reinterpret_cast<float*>(ws + pl.off_t);
  double* sums = reinterpret_cast<double*>(ws + pl.off_sums);
  int2* blk_counts = reinterpret_cast<int2*>(ws + pl.off_counts);
  unsigned long long* err = reinterpret_cast<unsigned long long*>(counts + 2);
  const auto* Hb = static_cast<const __nv_bfloat16*>(H);
  const auto* Wb = static_cast<const __nv_bfloat16*>(W);

  // (1) label scan + indexed dot
  e = launch(FLCE_KERNEL_LABEL_DOT, st, [&] {
    k_label_dot<<<pl.dot_blocks, 32 * kDotWarps, 0, st>>>(Hb, Wb, labels, N, Hd, V, v_offset, V_total,
                                                          ignore_index, softcap, t_ws, target_logit, blk_counts);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);

  // (2) tensor-core linear-LSE
  CUtensorMap tmH, tmW;
  if (!tmap_2d(&tmH, H, Hd, N, Hd * 2, kBK, kBM) || !tmap_2d(&tmW, W, Hd, V, Hd * 2, kBK, kBN / 2))
    return FLCE_ERR_CUDA;
  Sched sc{};
  sc.m_tiles = pl.m_tiles;
  sc.n_tiles = pl.v_tiles;
  sc.k_blocks = pl.k_blocks;
  sc.group = pl.group;
  sc.n_groups = pl.n_groups;
  sc.units = pl.m_tiles * pl.n_groups;
  sc.order = 0;
  sc.band = kBandM;
  EpiLseParams lp{N, V, softcap, part_m, part_s};
  const int grid = pair_grid(sc.units, sms);
  e = launch(FLCE_KERNEL_LINEAR_LSE, st, [&] { return launch_linear_lse(tmH, tmW, sc, lp, err, grid, st); });
  if (e != cudaSuccess) return cuda_fail(e);

  // (3) fixed-order merge, per-row loss, block sums
  float* loss_rows = reduction == FLCE_REDUCTION_NONE ? loss : nullptr;
  e = launch(FLCE_KERNEL_LSE_MERGE, st, [&] {
    const auto merge = pl.merge_blocks <= 2 * sms ? k_lse_merge<true> : k_lse_merge<false>;
    merge<<<pl.merge_blocks, kMergeRows * kMergeSlices, 0, st>>>(part_m, part_s, pl.n_groups * kEpiSplit, N, t_ws,
                                                                 labels, ignore_index, V_total, lse, loss_rows, sums);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);

  // (4) totals, counts, mean
  e = launch(FLCE_KERNEL_REDUCE, st, [&] {
    k_reduce<<<1, 256, 0, st>>>(sums, pl.merge_blocks, blk_counts, pl.dot_blocks, reduction, loss, counts);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  return FLCE_OK;
}

// Backward over the weight rows [v_offset, v_offset + V) of a vocabulary of V_total, from
// the global LSE.  dh_partial (sharded backward): dH is written there in fp32 as this
// shard's partial sum over its vocabulary rows instead of as bf16 into dH.
flce_status backward_impl(const void* H, const void* W, const int64_t* labels, const float* lse, int64_t* counts,
                          int64_t N, int64_t Hd, int64_t V, int64_t v_offset, int64_t V_total, int64_t ignore_index,
                          float softcap, int reduction, const float* grad_out, float filter_threshold,
                          unsigned options, void* dH, float* dh_partial, void* dW, void* workspace,
                          size_t workspace_bytes, size_t chunk_budget_bytes, void* stream) {
  if (reduction < 0 || reduction > 2 || softcap != softcap || !(filter_threshold >= 0.0f)) return FLCE_ERR_ARG;
  const bool filter = filter_threshold > 0.0f;
  if (filter && (options & FLCE_BWD_COMPENSATED) != 0) return FLCE_ERR_ARG;  // exact gradients only
  BwdPlan pl;
  flce_status s = plan_backward(N, Hd, V, chunk_budget_bytes, options, &pl);
  if (s != FLCE_OK) return s;
  const bool want_dh = dH != nullptr || dh_partial != nullptr;  // either gradient may be skipped
  if (!W || !counts || (!dW && !want_dh)) return FLCE_ERR_ARG;
  if (N > 0 && (!H || !labels || !lse || !grad_out || !workspace)) return FLCE_ERR_ARG;
  if (!aligned(W, 16) || (dW && !aligned(dW, 16)) || (H && !aligned(H, 16)) || (dH && !aligned(dH, 16)) ||
      (dh_partial && !aligned(dh_partial, 16)) ||
      !aligned(counts, 8) || (labels && !aligned(labels, 8)) || (lse && !aligned(lse, 4)) ||
      (grad_out && !aligned(grad_out, 4)))
    return FLCE_ERR_ALIGN;
  if (N > 0 && (workspace_bytes < pl.total || !aligned(workspace, kAlign))) return FLCE_ERR_WORKSPACE;
  int sms = 0;
  if ((s = device_setup(&sms)) != FLCE_OK) return s;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (N == 0) {  // no tokens: the weight gradient is an empty sum
    e = dW ? cudaMemsetAsync(dW, 0, size_t(V) * size_t(Hd) * 2, st) : cudaSuccess;
    return e == cudaSuccess ? FLCE_OK : cuda_fail(e);
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  RowInfo* rows = reinterpret_cast<RowInfo*>(ws + pl.off_rows);
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_dz);
  __nv_bfloat16* dz_lo = pl.split ? reinterpret_cast<__nv_bfloat16*>(ws + pl.off_dz_lo) : nullptr;
  float* dh32 = (pl.n_chunks > 1 || pl.dh_split > 1) ? reinterpret_cast<float*>(ws + pl.off_dh) : nullptr;
  float* dh_parts = pl.dh_split > 1 ? reinterpret_cast<float*>(ws + pl.off_dh_parts) : nullptr;
  uint8_t* nz = filter ? ws + pl.off_nz : nullptr;
  uint32_t* dh_mask = reinterpret_cast<uint32_t*>(ws + pl.off_dh_mask);
  uint32_t* dw_mask = reinterpret_cast<uint32_t*>(ws + pl.off_dw_mask);
  // skipping needs a tile's mask to fit the kernels' shared-memory copy
  const bool skip = filter && pl.dh_mask_ld <= kMaskWords && pl.dw_mask_ld <= kMaskWords;
  unsigned long long* err = reinterpret_cast<unsigned long long*>(counts + 2);

  // Sorted vocabulary: chunk c covers positions [c Vc, (c + 1) Vc) of the order; its
  // weight rows are gathered into wperm, labels become positions, dW rows go back to ids.
  int32_t* perm = nullptr;
  int32_t* inv = nullptr;
  __nv_bfloat16* wperm = nullptr;
  if (pl.sort) {
    perm = reinterpret_cast<int32_t*>(ws + pl.vocab.off_perm);
    inv = reinterpret_cast<int32_t*>(ws + pl.vocab.off_inv);
    wperm = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_wperm);
    s = vocab_order_impl(H, W, N, Hd, V, pl.vocab, ws, reinterpret_cast<float*>(ws + pl.vocab.off_key), perm, inv,
                         err, sms, st);
    if (s != FLCE_OK) return s;
  }

  e = launch(FLCE_KERNEL_BWD_PREP, st, [&] {
    k_bwd_prep<<<cdiv(N, 256), 256, 0, st>>>(labels, lse, counts, grad_out, reduction, N, V, v_offset, V_total,
                                             ignore_index, inv, rows);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);

  // Row compaction: the rows that carry a gradient (scale != 0) are gathered to the front of
  // a compact copy of H, in their original order, with their RowInfo; their count stays on
  // the device, where the tensor-core kernels read it.  Every other row contributes exact
  // zeros (its dZ row is zero), so the products run on the compact rows only and dH is
  // scattered back through the row map; the other rows of dH are written as zeros here.
  RowInfo* rows_c = reinterpret_cast<RowInfo*>(ws + pl.off_rows_c);
  int32_t* rmap = reinterpret_cast<int32_t*>(ws + pl.off_map);
  __nv_bfloat16* Hc = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_hc);
  int* blk = reinterpret_cast<int*>(ws + pl.off_blk);
  int* n_rows = reinterpret_cast<int*>(ws + pl.off_nrows);
  const auto* Hb = static_cast<const __nv_bfloat16*>(H);
  e = launch(FLCE_KERNEL_COMPACT, st, [&] {
    k_compact_count<<<pl.compact_blocks, kCompactRows, 0, st>>>(rows, N, blk);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch(FLCE_KERNEL_COMPACT, st, [&] {
    k_compact_scan<<<1, kCompactRows, 0, st>>>(blk, pl.compact_blocks, n_rows);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch(FLCE_KERNEL_COMPACT, st, [&] {
    k_compact_place<<<pl.compact_blocks, kCompactRows, 0, st>>>(rows, N, blk, rmap, rows_c);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch(FLCE_KERNEL_COMPACT, st, [&] {
    k_compact_gather<<<static_cast<int>(std::min<int64_t>(cdiv(pl.n_cap, 8), 8 * int64_t(sms))), 256, 0, st>>>(
        Hb, N, Hd, rmap, n_rows, pl.n_cap, Hc, rows_c);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  if (want_dh) {
    e = launch(FLCE_KERNEL_DH_ZERO, st, [&] {
      k_zero_dead_rows<<<static_cast<int>(std::min<int64_t>(cdiv(N, 8), 8 * int64_t(sms))), 256, 0, st>>>(
          rows, N, Hd, static_cast<__nv_bfloat16*>(dH), dh_partial);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return cuda_fail(e);
  }

  CUtensorMap tmH_k, tmW_k, tmH_mn, tmW_mn;
  if (!tmap_2d(&tmH_k, Hc, Hd, pl.n_cap, Hd * 2, kBK, kBM) || !tmap_2d(&tmH_mn, Hc, Hd, pl.n_cap, Hd * 2, 64, kBK) ||
      (!pl.sort && (!tmap_2d(&tmW_k, W, Hd, V, Hd * 2, kBK, kBN / 2) || !tmap_2d(&tmW_mn, W, Hd, V, Hd * 2, 64, kBK))))
    return FLCE_ERR_CUDA;

  const int m_tiles_tok = cdiv(N, kPairM);
  const int d_tiles = cdiv(Hd, kBN);
  for (int c = 0; c < pl.n_chunks; ++c) {
    const int64_t v0 = pl.chunk_begin(c, V);
    const int64_t wc = pl.chunk_begin(c + 1, V) - v0;
    CUtensorMap tmDz_k, tmDz_mn, tmLo_k, tmLo_mn;
    if (!tmap_2d(&tmDz_k, dz, wc, N, pl.Vc * 2, kBK, kBM) || !tmap_2d(&tmDz_mn, dz, wc, N, pl.Vc * 2, 64, kBK))
      return FLCE_ERR_CUDA;
    if (pl.split) {
      if (!tmap_2d(&tmLo_k, dz_lo, wc, N, pl.Vc * 2, kBK, kBM) || !tmap_2d(&tmLo_mn, dz_lo, wc, N, pl.Vc * 2, 64, kBK))
        return FLCE_ERR_CUDA;
    } else {
      tmLo_k = tmDz_k;
      tmLo_mn = tmDz_mn;
    }
    int64_t w_off = v0;  // first weight row of the chunk in the tensor maps
    if (pl.sort) {
      e = launch(FLCE_KERNEL_GATHER, st, [&] {
        k_gather_rows<<<std::min(cdiv(wc, kRowCopyThreads / 32), 8 * sms), kRowCopyThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(W), V, Hd, perm, v0, wc, wperm, err);
        return cudaGetLastError();
      });
      if (e != cudaSuccess) return cuda_fail(e);
      if (!tmap_2d(&tmW_k, wperm, Hd, wc, Hd * 2, kBK, kBN / 2) || !tmap_2d(&tmW_mn, wperm, Hd, wc, Hd * 2, 64, kBK))
        return FLCE_ERR_CUDA;
      w_off = 0;
    }

    // dZ chunk = f(H W_chunk^T)
    Sched s4{};
    s4.m_tiles = m_tiles_tok;
    s4.n_tiles = cdiv(wc, kBN);
    s4.k_blocks = cdiv(Hd, kBK);
    s4.group = 1;
    s4.n_groups = s4.n_tiles;
    s4.units = s4.m_tiles * s4.n_groups;
    s4.order = 0;
    s4.band = kBandM;
    s4.b_n_off = static_cast<int>(w_off);
    s4.n_dev = n_rows;  // M walks the compact rows
    s4.n_role = 1;
    if (filter && (e = cudaMemsetAsync(nz, 0, size_t(pl.nz_rows) * size_t(pl.nz_ld), st)) != cudaSuccess)
      return cuda_fail(e);
    EpiDzParams p4{N, V, v0, wc, pl.Vc, softcap, rows_c, dz, dz_lo, filter_threshold, nz, pl.nz_ld};
    e = launch(FLCE_KERNEL_DZ, st,
               [&] { return launch_dz(tmH_k, tmW_k, s4, p4, err, pair_grid(s4.units, sms), st); });
    if (e != cudaSuccess) return cuda_fail(e);

    if (skip) {  // per-tile K-step masks of the dW and dH products
      const int kb_dh = cdiv(wc, kBK);
      const int vt = cdiv(wc, kPairM);
      const int total = pl.mask_tok_tiles * pl.dh_mask_ld + vt * pl.dw_mask_ld;
      e = launch(FLCE_KERNEL_BLOCK_MASK, st, [&] {
        k_block_masks<<<std::min(cdiv(total, 256), 4 * sms), 256, 0, st>>>(
            nz, pl.nz_rows, pl.nz_ld, kb_dh, pl.mask_tok_tiles, vt, dh_mask, pl.dh_mask_ld, dw_mask, pl.dw_mask_ld);
        return cudaGetLastError();
      });
      if (e != cudaSuccess) return cuda_fail(e);
    }

    // dW rows [v0, v0 + wc) = dZ_chunk^T H
    Sched s5{};
    s5.m_tiles = cdiv(wc, kPairM);
    s5.n_tiles = d_tiles;
    s5.k_blocks = cdiv(N, kBK);
    s5.group = 1;
    s5.n_groups = d_tiles;
    s5.units = s5.m_tiles * s5.n_groups;
    s5.order = 1;
    s5.n_dev = n_rows;  // K walks the compact rows
    s5.n_role = 2;
    if (skip) {
      s5.kmask = dw_mask;
      s5.kmask_ld = pl.dw_mask_ld;
    }
    if (pl.split) {  // dZ^T H + dZ_lo^T H in one accumulator
      s5.k_half = s5.k_blocks;
      s5.k_blocks *= 2;
    }
    EpiDwParams p5{wc, v0, Hd, static_cast<__nv_bfloat16*>(dW), perm, V};
    if (dW) {
      e = launch(FLCE_KERNEL_DW, st,
                 [&] { return launch_dw(tmDz_mn, tmLo_mn, tmH_mn, s5, p5, err, pair_grid(s5.units, sms), st); });
      if (e != cudaSuccess) return cuda_fail(e);
    }

    // dH (+)= dZ_chunk W_chunk
    Sched s6{};
    s6.m_tiles = m_tiles_tok;
    s6.n_tiles = d_tiles;
    s6.k_blocks = cdiv(wc, kBK);
    s6.group = 1;
    s6.n_groups = d_tiles;
    s6.units = s6.m_tiles * s6.n_groups;
    s6.order = 1;
    s6.b_k_off = static_cast<int>(w_off);
    s6.n_dev = n_rows;  // M walks the compact rows
    s6.n_role = 1;
    if (skip) {
      s6.kmask = dh_mask;
      s6.kmask_ld = pl.dh_mask_ld;
    }
    if (pl.split) {  // dZ W + dZ_lo W in one accumulator
      s6.k_half = s6.k_blocks;
      s6.k_blocks *= 2;
    }
    // K split of the exact product (the filtered mode keeps whole tiles for its K-step masks;
    // a shard's fp32 partial is accumulated in dH's own rows, without part sums)
    const int ksplit = (filter || dh_partial != nullptr) ? 1 : std::min(pl.dh_split, s6.k_blocks);
    s6.k_split = ksplit;
    s6.units *= ksplit;
    float* dh_acc = dh_partial != nullptr ? dh_partial : dh32;
    const bool last = c == pl.n_chunks - 1;
    EpiDhParams p6 = dh_partial != nullptr
                         ? EpiDhParams{N, Hd, dh_partial, nullptr, c == 0, 0, dh_parts, rmap, n_rows, 1}
                         : EpiDhParams{N, Hd, dh32, static_cast<__nv_bfloat16*>(dH), c == 0, last && ksplit == 1,
                                       dh_parts, rmap, n_rows, 0};
    if (want_dh) {
      e = launch(FLCE_KERNEL_DH, st,
                 [&] { return launch_dh(tmDz_k, tmLo_k, tmW_mn, s6, p6, err, pair_grid(s6.units, sms), st); });
      if (e != cudaSuccess) return cuda_fail(e);
      if (ksplit > 1) {  // parts 1 .. ksplit - 1 into the running sum, or into the bf16 dH at the last chunk
        __nv_bfloat16* out = (dh_partial == nullptr && last) ? static_cast<__nv_bfloat16*>(dH) : nullptr;
        const int64_t count = N * Hd;
        e = launch(FLCE_KERNEL_DH_COMBINE, st, [&] {
          k_dh_combine<<<static_cast<int>(std::min<int64_t>(std::max<int64_t>(count / 4 / 256, 1), 8 * sms)), 256, 0,
                         st>>>(dh_acc, dh_parts, ksplit - 1, count, Hd, out, rmap, n_rows);
          return cudaGetLastError();
        });
        if (e != cudaSuccess) return cuda_fail(e);
      }
    }
  }
  return FLCE_OK;
}

}  // namespace flce

using namespace flce;

extern "C" {

size_t flce_forward_workspace_size(int64_t N, int64_t Hd, int64_t V) {
  FwdPlan p;
  return plan_forward(N, Hd, V, kPlanPairs, &p) == FLCE_OK ? p.total : 0;
}

size_t flce_backward_workspace_size(int64_t N, int64_t Hd, int64_t V, size_t chunk_budget_bytes, unsigned options) {
  BwdPlan p;
  return plan_backward(N, Hd, V, chunk_budget_bytes, options, &p) == FLCE_OK ? p.total : 0;
}

size_t flce_vocab_order_workspace_size(int64_t N, int64_t Hd, int64_t V) {
  VocabPlan p;
  size_t cur = 0;
  if (check_sizes(N, Hd, V) != FLCE_OK || !plan_vocab(N, Hd, V, &cur, &p)) return 0;
  return align_up(cur);
}

flce_status flce_vocab_order(const void* H, const void* W, int64_t N, int64_t Hd, int64_t V, float* keys,
                             int32_t* perm, int32_t* inv, void* workspace, size_t workspace_bytes, void* stream) {
  flce_status s = check_sizes(N, Hd, V);
  if (s != FLCE_OK) return s;
  VocabPlan vp;
  size_t cur = 0;
  if (!plan_vocab(N, Hd, V, &cur, &vp)) return FLCE_ERR_OVERFLOW;
  if (!W || !perm || !workspace || (N > 0 && !H)) return FLCE_ERR_ARG;
  if (!aligned(W, 16) || (H && !aligned(H, 16)) || !aligned(perm, 4) || (keys && !aligned(keys, 4)) ||
      (inv && !aligned(inv, 4)))
    return FLCE_ERR_ALIGN;
  if (workspace_bytes < align_up(cur) || !aligned(workspace, kAlign)) return FLCE_ERR_WORKSPACE;
  int sms = 0;
  if ((s = device_setup(&sms)) != FLCE_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return vocab_order_impl(H, W, N, Hd, V, vp, ws, keys ? keys : reinterpret_cast<float*>(ws + vp.off_key), perm, inv,
                          nullptr, sms, static_cast<cudaStream_t>(stream));
}

flce_status flce_forward(const void* H, const void* W, const int64_t* labels, int64_t N, int64_t Hd, int64_t V,
                         int64_t ignore_index, float softcap, int reduction, float* loss, float* lse,
                         float* target_logit, int64_t* counts, void* workspace, size_t workspace_bytes,
                         void* stream) {
  if (reduction < 0 || reduction > 2) return FLCE_ERR_ARG;
  return forward_impl(H, W, labels, N, Hd, V, 0, V, ignore_index, softcap, reduction, loss, lse, target_logit, counts,
                      workspace, workspace_bytes, stream);
}

flce_status flce_backward(const void* H, const void* W, const int64_t* labels, const float* lse, int64_t* counts,
                          int64_t N, int64_t Hd, int64_t V, int64_t ignore_index, float softcap, int reduction,
                          const float* grad_out, float filter_threshold, unsigned options, void* dH, void* dW,
                          void* workspace, size_t workspace_bytes, size_t chunk_budget_bytes, void* stream) {
  return backward_impl(H, W, labels, lse, counts, N, Hd, V, 0, V, ignore_index, softcap, reduction, grad_out,
                       filter_threshold, options, dH, nullptr, dW, workspace, workspace_bytes, chunk_budget_bytes,
                       stream);
}

namespace {
flce_status check_shard(int64_t V_shard, int64_t v_offset, int64_t V_total) {
  if (V_shard <= 0 || v_offset < 0 || V_total <= 0) return FLCE_ERR_ARG;
  if (V_total > (int64_t(1) << 31) - 512) return FLCE_ERR_OVERFLOW;
  if (v_offset > V_total - V_shard) return FLCE_ERR_ARG;
  return FLCE_OK;
}
}  // namespace

flce_status flce_forward_shard(const void* H, const void* W_shard, const int64_t* labels, int64_t N, int64_t Hd,
                               int64_t V_shard, int64_t v_offset, int64_t V_total, int64_t ignore_index,
                               float softcap, float* lse_shard, float* target_shard, int64_t* counts,
                               void* workspace, size_t workspace_bytes, void* stream) {
  flce_status s = check_shard(V_shard, v_offset, V_total);
  if (s != FLCE_OK) return s;
  if (N > 0 && !target_shard) return FLCE_ERR_ARG;
  return forward_impl(H, W_shard, labels, N, Hd, V_shard, v_offset, V_total, ignore_index, softcap, -1, nullptr,
                      lse_shard, target_shard, counts, workspace, workspace_bytes, stream);
}

size_t flce_merge_shards_workspace_size(int64_t N) {
  if (N < 0) return 0;
  const size_t blocks = std::max(cdiv(N, kMergeThreads), 1);
  return align_up(blocks * sizeof(double)) + align_up(blocks * sizeof(int2));
}

flce_status flce_merge_shards(const float* lse_parts, const float* target_parts, int64_t n_shards,
                              const int64_t* labels, int64_t N, int64_t V_total, int64_t ignore_index, int reduction,
                              float* loss, float* lse, int64_t* counts, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (reduction < 0 || reduction > 2 || n_shards <= 0 || n_shards > (int64_t(1) << 20) || N < 0 || V_total <= 0)
    return FLCE_ERR_ARG;
  if (!loss || !counts) return FLCE_ERR_ARG;
  if (N > 0 && (!lse_parts || !target_parts || !labels || !lse || !workspace)) return FLCE_ERR_ARG;
  if (!aligned(counts, 8) || !aligned(loss, 4) || (labels && !aligned(labels, 8))) return FLCE_ERR_ALIGN;
  size_t total;
  if (!mul_ok(size_t(n_shards), size_t(N), &total)) return FLCE_ERR_OVERFLOW;
  const size_t need = flce_merge_shards_workspace_size(N);
  if (N > 0 && (workspace_bytes < need || !aligned(workspace, kAlign))) return FLCE_ERR_WORKSPACE;
  int sms = 0;
  flce_status s = device_setup(&sms);
  if (s != FLCE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(counts, 0, 3 * sizeof(int64_t), st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (N == 0) {
    if (reduction != FLCE_REDUCTION_NONE && (e = cudaMemsetAsync(loss, 0, sizeof(float), st)) != cudaSuccess)
      return cuda_fail(e);
    return FLCE_OK;
  }
  const int blocks = std::max(cdiv(N, kMergeThreads), 1);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  double* sums = reinterpret_cast<double*>(ws);
  int2* blk_counts = reinterpret_cast<int2*>(ws + align_up(size_t(blocks) * sizeof(double)));
  float* loss_rows = reduction == FLCE_REDUCTION_NONE ? loss : nullptr;
  e = launch(FLCE_KERNEL_SHARD_MERGE, st, [&] {
    k_shard_merge<<<blocks, kMergeThreads, 0, st>>>(lse_parts, target_parts, static_cast<int>(n_shards), N, labels,
                                                    ignore_index, V_total, lse, loss_rows, sums, blk_counts);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch(FLCE_KERNEL_REDUCE, st, [&] {
    k_reduce<<<1, 256, 0, st>>>(sums, blocks, blk_counts, blocks, reduction, loss, counts);
    return cudaGetLastError();
  });
  return e == cudaSuccess ? FLCE_OK : cuda_fail(e);
}

flce_status flce_backward_shard(const void* H, const void* W_shard, const int64_t* labels, const float* lse,
                                int64_t* counts, int64_t N, int64_t Hd, int64_t V_shard, int64_t v_offset,
                                int64_t V_total, int64_t ignore_index, float softcap, int reduction,
                                const float* grad_out, float filter_threshold, unsigned options,
                                float* dH_partial, void* dW_shard, void* workspace, size_t workspace_bytes,
                                size_t chunk_budget_bytes, void* stream) {
  flce_status s = check_shard(V_shard, v_offset, V_total);
  if (s != FLCE_OK) return s;
  return backward_impl(H, W_shard, labels, lse, counts, N, Hd, V_shard, v_offset, V_total, ignore_index, softcap,
                       reduction, grad_out, filter_threshold, options, nullptr, dH_partial, dW_shard, workspace,
                       workspace_bytes, chunk_budget_bytes, stream);
}

flce_status flce_stage_h2d(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return FLCE_OK;
  if (!dst || !src) return FLCE_ERR_ARG;
  if (!aligned(dst, 16) || !aligned(src, 16)) return FLCE_ERR_ALIGN;
  int sms = 0;
  flce_status s = device_setup(&sms);
  if (s != FLCE_OK) return s;
  // src: page-locked host memory (pageable memory is reachable from the GPU on systems
  // with address translation services too, but is refused); dst: this device's memory
  int dev = 0;
  cudaPointerAttributes as{}, ad{};
  if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&as, src) != cudaSuccess ||
      cudaPointerGetAttributes(&ad, dst) != cudaSuccess) {
    (void)cudaGetLastError();  // clear the (non-sticky) lookup error
    return FLCE_ERR_ARG;
  }
  if (as.type != cudaMemoryTypeHost || as.devicePointer == nullptr) return FLCE_ERR_ARG;
  if ((ad.type != cudaMemoryTypeDevice && ad.type != cudaMemoryTypeManaged) || ad.device != dev) return FLCE_ERR_ARG;
  const void* dsrc = as.devicePointer;
  if (!aligned(dsrc, 16)) return FLCE_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((n16 + kStageThreads - 1) / kStageThreads, sms)));
  const cudaError_t e = launch(FLCE_KERNEL_STAGE, st, [&] {
    k_stage_h2d<<<blocks, kStageThreads, 0, st>>>(static_cast<const uint4*>(dsrc), static_cast<uint4*>(dst), n16,
                                                  static_cast<int>(bytes % 16));
    return cudaGetLastError();
  });
  return e == cudaSuccess ? FLCE_OK : cuda_fail(e);
}

flce_status flce_selftest_wait_timeout(int64_t* status_word, void* stream) {
  if (!status_word) return FLCE_ERR_ARG;
  if (!aligned(status_word, 8)) return FLCE_ERR_ALIGN;
  int sms = 0;
  flce_status s = device_setup(&sms);
  if (s != FLCE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(status_word, 0, sizeof(int64_t), st);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch(FLCE_KERNEL_SELFTEST, st, [&] {
    k_wait_timeout_selftest<<<1, 32, 0, st>>>(reinterpret_cast<unsigned long long*>(status_word));
    return cudaGetLastError();
  });
  return e == cudaSuccess ? FLCE_OK : cuda_fail(e);
}

const char* flce_strerror(int status) {
  switch (status) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_ARG: return "invalid argument (null pointer, negative size, unknown reduction, NaN or negative threshold)";
    case FLCE_ERR_ALIGN: return "misaligned pointer or hidden size not a multiple of 8";
    case FLCE_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case FLCE_ERR_OVERFLOW: return "sizes overflow the 64-bit byte counts or the 2^31 index limits";
    case FLCE_ERR_CUDA: return "a CUDA runtime call failed (see flce_last_cuda_error)";
    case FLCE_ERR_UNSUPPORTED: return "unsupported device (needs sm_103)";
    default: return "unknown status";
  }
}

int flce_last_cuda_error(void) { return t_last_cuda; }

uint64_t flce_launch_count(void) { return t_launches; }

int flce_set_event_sink(void* const* start_events, void* const* end_events, int* kernel_ids, int capacity) {
  if (capacity <= 0 || !start_events || !end_events || !kernel_ids) {
    t_sink = EventSink{};
    return 0;
  }
  t_sink.start = start_events;
  t_sink.end = end_events;
  t_sink.ids = kernel_ids;
  t_sink.cap = capacity;
  t_sink.used = 0;
  return 0;
}

int flce_event_sink_used(void) { return t_sink.used; }

}  // extern "C"
