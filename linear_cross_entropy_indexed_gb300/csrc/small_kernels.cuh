// Memory- and latency-bound kernels of the path: label scan + indexed dot, the
// fixed-order (max, sum) merge with the per-row loss, the final reduction, and the
// per-row backward preparation.
#pragma once

#include "internal.cuh"

namespace flce {

constexpr int kDotWarps = 8;        // rows per block of the indexed-dot kernel
constexpr int kDotMaxBlocks = 2048; // grid cap (grid-stride beyond)
constexpr int kMergeThreads = 256;
constexpr int kMergeRows = 32;     // rows per block of the (m, s) merge: one per lane
constexpr int kMergeSlices = 8;    // warps per merge block: each merges every 8th partial
constexpr int kMergeBatch = 16;    // partials a warp loads before merging them (short grids)

__device__ __forceinline__ float softcap_exact(float x, float c) {
  return c > 0.0f ? c * tanhf(x / c) : x;
}

// Label scan + indexed dot: for every row i, valid_i = (y_i != ignore) && 0 <= y_i < V_total,
// bad_i = (y_i != ignore) && !valid_i, and t_i = cap(h_i . w_{y_i - v_offset}) when the label
// falls in this weight's rows [v_offset, v_offset + V) (0 otherwise).  Without vocabulary
// sharding v_offset = 0 and V_total = V.  One warp per row, 16-byte loads, fp32 FMA,
// butterfly sum.  Per-block (n_valid, n_bad) go to blk_counts for the fixed-order final
// reduction.
__global__ void __launch_bounds__(32 * kDotWarps)
    k_label_dot(const __nv_bfloat16* __restrict__ H, const __nv_bfloat16* __restrict__ W,
                const int64_t* __restrict__ labels, int64_t N, int64_t Hd, int64_t V, int64_t v_offset,
                int64_t V_total, int64_t ignore, float softcap, float* __restrict__ t_ws,
                float* __restrict__ t_user, int2* __restrict__ blk_counts) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int n_valid = 0, n_bad = 0;
  const int64_t vec = Hd / 8;  // 16-byte vectors per row
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kDotWarps + warp; i < N;
       i += static_cast<int64_t>(gridDim.x) * kDotWarps) {
    const int64_t y = labels[i];
    const bool ignored = y == ignore;
    const bool in_range = y >= 0 && y < V_total;
    const bool valid = !ignored && in_range;
    const int64_t yl = y - v_offset;
    const bool local = valid && yl >= 0 && yl < V;
    float acc = 0.0f;
    if (local) {
      const uint4* hp = reinterpret_cast<const uint4*>(H + i * Hd);
      const uint4* wp = reinterpret_cast<const uint4*>(W + yl * Hd);
      for (int64_t k = lane; k < vec; k += 32) {
        const uint4 a = __ldg(hp + k);
        const uint4 b = __ldg(wp + k);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = __bfloat1622float2(a2[e]);
          const float2 fb = __bfloat1622float2(b2[e]);
          acc = fmaf(fa.x, fb.x, acc);
          acc = fmaf(fa.y, fb.y, acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      acc = softcap_exact(acc, softcap);
    }
    if (lane == 0) {
      t_ws[i] = acc;
      if (t_user) t_user[i] = acc;
      n_valid += valid ? 1 : 0;
      n_bad += (!ignored && !in_range) ? 1 : 0;
    }
  }
  __shared__ int sv[kDotWarps], sb[kDotWarps];
  if (lane == 0) {
    sv[warp] = n_valid;
    sb[warp] = n_bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0, b = 0;
    for (int w = 0; w < kDotWarps; ++w) {
      a += sv[w];
      b += sb[w];
    }
    blk_counts[blockIdx.x] = make_int2(a, b);
  }
}

// Fixed-order merge of the per-group (max, sum) partials into lse_i, then the per-row
// loss and a fixed-tree block sum (double) of the losses.  A block takes 32 rows, one
// per lane, so every partial is read as one coalesced 128-byte line per warp; its 8 warps
// split the partials (warp j merges groups j, j + 8, j + 16, ... in increasing order) so
// that each row has 8 chains of loads in flight instead of one, and warp 0 then merges
// the 8 slices in slice order.  The order of every merge is fixed: results are bitwise
// reproducible.
__device__ __forceinline__ void merge_ms(float& m, float& s, float mg, float sg) {
  if (mg == -INFINITY) return;  // a group (or slice) that saw nothing
  const float mn = fmaxf(m, mg);
  s = s * exp2f(m - mn) + sg * exp2f(mg - mn);  // 2^-inf = 0 for the first merge
  m = mn;
}

// BATCH (short grids, at most two blocks per SM): a warp issues the loads of kMergeBatch
// partials before merging them, since its own loads are all that hides the latency; else
// it streams them (with enough blocks resident, occupancy hides it and the batch's
// registers only lower occupancy).  Both merge in the same order: bitwise the same result.
template <bool BATCH>
__global__ void __launch_bounds__(kMergeRows * kMergeSlices)
    k_lse_merge(const float* __restrict__ part_m, const float* __restrict__ part_s, int n_groups,
                int64_t N, const float* __restrict__ t, const int64_t* __restrict__ labels,
                int64_t ignore, int64_t V_total, float* __restrict__ lse_out, float* __restrict__ loss_rows,
                double* __restrict__ blk_sums) {
  __shared__ float sm[kMergeSlices][kMergeRows], ss[kMergeSlices][kMergeRows];
  const int lane = threadIdx.x & 31;
  const int slice = threadIdx.x >> 5;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kMergeRows + lane;
  float m = -INFINITY, s = 0.0f;
  if (i < N && !BATCH) {
#pragma unroll 4
    for (int g = slice; g < n_groups; g += kMergeSlices)
      merge_ms(m, s, part_m[static_cast<int64_t>(g) * N + i], part_s[static_cast<int64_t>(g) * N + i]);
  } else if (i < N) {
    // kMergeBatch groups of the slice at a time: all their loads are issued (past the last
    // group, the batch's first group is read again and dropped) before the merges, which
    // run in increasing group order as ever
    for (int g0 = slice; g0 < n_groups; g0 += kMergeBatch * kMergeSlices) {
      float bm[kMergeBatch], bs[kMergeBatch];
#pragma unroll
      for (int b = 0; b < kMergeBatch; ++b) {
        const int g = g0 + b * kMergeSlices;
        const int64_t at = static_cast<int64_t>(g < n_groups ? g : g0) * N + i;
        bm[b] = part_m[at];
        bs[b] = part_s[at];
      }
#pragma unroll
      for (int b = 0; b < kMergeBatch; ++b)
        if (g0 + b * kMergeSlices < n_groups) merge_ms(m, s, bm[b], bs[b]);
    }
  }
  sm[slice][lane] = m;
  ss[slice][lane] = s;
  __syncthreads();
  if (slice != 0) return;
  double mine = 0.0;
  if (i < N) {
    m = -INFINITY;
    s = 0.0f;
#pragma unroll
    for (int k = 0; k < kMergeSlices; ++k) merge_ms(m, s, sm[k][lane], ss[k][lane]);
    const float lse = (m + log2f(s)) * kLn2;
    lse_out[i] = lse;
    const int64_t y = labels[i];
    const bool valid = y != ignore && y >= 0 && y < V_total;
    const float l = valid ? lse - t[i] : 0.0f;
    if (loss_rows) loss_rows[i] = l;
    mine = l;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mine += __shfl_down_sync(0xffffffffu, mine, off);
  if (lane == 0) blk_sums[blockIdx.x] = mine;
}

// dH split: acc += parts[0] + parts[1] + ... in part order, 4 elements per thread per
// step (16-byte loads; count = N Hd, Hd a multiple of 8).  At the last vocabulary chunk
// (out != null) the sum goes to the bf16 dH instead of back into the running sum: the
// rows are compact, row r < *n_rows going to dH row row_map[r] (rows past *n_rows hold
// no gradient and are not written).
__global__ void __launch_bounds__(256)
    k_dh_combine(float* __restrict__ acc, const float* __restrict__ parts, int n_parts, int64_t count, int64_t Hd,
                 __nv_bfloat16* __restrict__ out, const int32_t* __restrict__ row_map, const int* __restrict__ n_rows) {
  const int64_t n4 = count / 4;
  const int64_t nr = (out != nullptr && row_map != nullptr) ? static_cast<int64_t>(*n_rows) : 0;
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < n4;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t oq = q;  // destination float4 index (in dH's rows)
    if (out != nullptr && row_map != nullptr) {
      const int64_t r = (4 * q) / Hd;
      if (r >= nr) continue;
      const int64_t o = row_map[r];
      if (o < 0 || o >= count / Hd) continue;
      oq = (o * Hd + (4 * q - r * Hd)) / 4;
    }
    float4 v = reinterpret_cast<const float4*>(acc)[q];
    for (int j = 0; j < n_parts; ++j) {
      const float4 w = reinterpret_cast<const float4*>(parts + static_cast<int64_t>(j) * count)[q];
      v.x += w.x;
      v.y += w.y;
      v.z += w.z;
      v.w += w.w;
    }
    if (out != nullptr) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 packed;
      packed.x = *reinterpret_cast<const uint32_t*>(&lo);
      packed.y = *reinterpret_cast<const uint32_t*>(&hi);
      reinterpret_cast<uint2*>(out)[oq] = packed;
    } else {
      reinterpret_cast<float4*>(acc)[q] = v;
    }
  }
}

// ------------------------------------------------------------------ host-to-device staging
// Grid-stride copy of n16 16-byte words from a pinned host buffer (read through its
// device mapping) to device memory, four independent loads in flight per thread; block 0
// copies the last `tail` (< 16) bytes one by one.
constexpr int kStageThreads = 128;
__global__ void __launch_bounds__(kStageThreads)
    k_stage_h2d(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16, int tail) {
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * step < n16; i += 4 * step) {
    const uint4 a = src[i];
    const uint4 b = src[i + step];
    const uint4 c = src[i + 2 * step];
    const uint4 d = src[i + 3 * step];
    dst[i] = a;
    dst[i + step] = b;
    dst[i + 2 * step] = c;
    dst[i + 3 * step] = d;
  }
  for (; i < n16; i += step) dst[i] = src[i];
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail)
    reinterpret_cast<uint8_t*>(dst + n16)[threadIdx.x] = reinterpret_cast<const uint8_t*>(src + n16)[threadIdx.x];
}

// ------------------------------------------------------------------ row compaction
// The backward runs only on the rows that carry a gradient (scale != 0: a valid label and
// a non-zero upstream gradient); every other row's dZ row, dH row and share of dW are
// exactly zero.  The rows that do are gathered to the front in their original order: a
// count per block of kCompactRows rows, an exclusive scan of the counts (one block), then
// each row's place.  The count of such rows stays on the device.
constexpr int kCompactRows = 1024;

__global__ void __launch_bounds__(kCompactRows)
    k_compact_count(const RowInfo* __restrict__ rows, int64_t N, int* __restrict__ blk_cnt) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kCompactRows + threadIdx.x;
  const int live = (i < N && rows[i].scale != 0.0f) ? 1 : 0;
  const int c = __syncthreads_count(live);
  if (threadIdx.x == 0) blk_cnt[blockIdx.x] = c;
}

// Exclusive scan of nblk block counts in place (blocks of kCompactRows values, each
// scanned in shared memory, carried in order); the total goes to *n_rows.
__global__ void __launch_bounds__(kCompactRows) k_compact_scan(int* __restrict__ blk, int nblk, int* __restrict__ n_rows) {
  __shared__ int sh[kCompactRows];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < nblk; base += kCompactRows) {
    const int k = base + static_cast<int>(threadIdx.x);
    const int v = k < nblk ? blk[k] : 0;
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < kCompactRows; off <<= 1) {  // inclusive Hillis-Steele scan
      const int t = threadIdx.x >= static_cast<unsigned>(off) ? sh[threadIdx.x - off] : 0;
      __syncthreads();
      sh[threadIdx.x] += t;
      __syncthreads();
    }
    if (k < nblk) blk[k] = carry + sh[threadIdx.x] - v;
    __syncthreads();
    if (threadIdx.x == kCompactRows - 1) carry += sh[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_rows = carry;
}

// Row i that carries a gradient goes to position blk_off[block] + its rank in the block:
// map[pos] = i, rows_c[pos] = rows[i].
__global__ void __launch_bounds__(kCompactRows)
    k_compact_place(const RowInfo* __restrict__ rows, int64_t N, const int* __restrict__ blk_off,
                    int32_t* __restrict__ map, RowInfo* __restrict__ rows_c) {
  __shared__ int warp_sum[kCompactRows / 32];
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kCompactRows + threadIdx.x;
  const bool live = i < N && rows[i].scale != 0.0f;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned ball = __ballot_sync(0xffffffffu, live);
  if (lane == 0) warp_sum[w] = __popc(ball);
  __syncthreads();
  if (w == 0) {  // exclusive scan of the 32 warp sums
    const int v = warp_sum[lane];
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    warp_sum[lane] = incl - v;
  }
  __syncthreads();
  if (live) {
    const int pos = blk_off[blockIdx.x] + warp_sum[w] + __popc(ball & ((1u << lane) - 1u));
    map[pos] = static_cast<int32_t>(i);
    rows_c[pos] = rows[i];
  }
}

// One warp per compact row p < ceil256(max(n, 1)) (n = *n_rows), bounded by n_cap: rows
// p < n copy H row map[p] into Hc row p; the rest of the last 256-row tile is zeroed
// (Hc and rows_c: no gradient, finite logits), so that the tile computes exact zeros.
__global__ void __launch_bounds__(256)
    k_compact_gather(const __nv_bfloat16* __restrict__ H, int64_t N, int64_t Hd, const int32_t* __restrict__ map,
                     const int* __restrict__ n_rows, int64_t n_cap, __nv_bfloat16* __restrict__ Hc,
                     RowInfo* __restrict__ rows_c) {
  const int64_t n = *n_rows;
  const int64_t end = min(n_cap, ((max(n, int64_t(1)) + 255) / 256) * 256);
  const int lane = threadIdx.x & 31;
  const int64_t vec = Hd / 8;
  for (int64_t p = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; p < end;
       p += static_cast<int64_t>(gridDim.x) * blockDim.x / 32) {
    uint4* dst = reinterpret_cast<uint4*>(Hc + p * Hd);
    if (p < n) {
      const int64_t src_row = map[p];
      if (src_row < 0 || src_row >= N) continue;  // (never: map holds rows of H)
      const uint4* src = reinterpret_cast<const uint4*>(H + src_row * Hd);
      for (int64_t k = lane; k < vec; k += 32) dst[k] = __ldg(src + k);
    } else {
      for (int64_t k = lane; k < vec; k += 32) dst[k] = make_uint4(0u, 0u, 0u, 0u);
      if (lane == 0) rows_c[p] = RowInfo{0.0f, 0.0f, -1, 0};
    }
  }
}

// Rows that carry no gradient get an exactly zero output row: one warp per row, bf16 dH
// or fp32 dH partial (whichever is given).
__global__ void __launch_bounds__(256)
    k_zero_dead_rows(const RowInfo* __restrict__ rows, int64_t N, int64_t Hd, __nv_bfloat16* __restrict__ dh_bf16,
                     float* __restrict__ dh_f32) {
  const int lane = threadIdx.x & 31;
  for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32; i < N;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x / 32) {
    if (rows[i].scale != 0.0f) continue;
    if (dh_bf16 != nullptr) {
      uint4* d = reinterpret_cast<uint4*>(dh_bf16 + i * Hd);
      for (int64_t k = lane; k < Hd / 8; k += 32) d[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (dh_f32 != nullptr) {
      float4* d = reinterpret_cast<float4*>(dh_f32 + i * Hd);
      for (int64_t k = lane; k < Hd / 4; k += 32) d[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// Single block: fixed-order totals of the block sums and block counts, then the
// reduction (mean divides once by n_valid; 0 when n_valid == 0).
__global__ void __launch_bounds__(256)
    k_reduce(const double* __restrict__ blk_sums, int n_sum_blocks, const int2* __restrict__ blk_counts,
             int n_count_blocks, int reduction, float* __restrict__ loss, int64_t* __restrict__ counts) {
  __shared__ double ss[256];
  __shared__ long long sv[256], sb[256];
  double s = 0.0;
  long long v = 0, b = 0;
  for (int k = threadIdx.x; k < n_sum_blocks; k += 256) s += blk_sums[k];
  for (int k = threadIdx.x; k < n_count_blocks; k += 256) {
    v += blk_counts[k].x;
    b += blk_counts[k].y;
  }
  ss[threadIdx.x] = s;
  sv[threadIdx.x] = v;
  sb[threadIdx.x] = b;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      ss[threadIdx.x] += ss[threadIdx.x + w];
      sv[threadIdx.x] += sv[threadIdx.x + w];
      sb[threadIdx.x] += sb[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    counts[0] = sv[0];
    counts[1] = sb[0];
    if (reduction == 0) loss[0] = sv[0] > 0 ? static_cast<float>(ss[0] / static_cast<double>(sv[0])) : 0.0f;
    if (reduction == 1) loss[0] = static_cast<float>(ss[0]);
  }
}

// Backward per-row data: scale_i (0 for ignored rows), the label as a row of this weight
// (-1 when ignored or, with vocabulary sharding, held by another shard), lse * log2 e.
__global__ void k_bwd_prep(const int64_t* __restrict__ labels, const float* __restrict__ lse,
                           const int64_t* __restrict__ counts, const float* __restrict__ grad,
                           int reduction, int64_t N, int64_t V, int64_t v_offset, int64_t V_total, int64_t ignore,
                           const int32_t* __restrict__ inv, RowInfo* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const int64_t y = labels[i];
  const bool valid = y != ignore && y >= 0 && y < V_total;
  const int64_t yl = y - v_offset;
  float scale = 0.0f;
  if (valid) {
    if (reduction == 0) {
      const long long nv = counts[0];
      scale = nv > 0 ? static_cast<float>(static_cast<double>(grad[0]) / static_cast<double>(nv)) : 0.0f;
    } else if (reduction == 1) {
      scale = grad[0];
    } else {
      scale = grad[i];
    }
  }
  RowInfo r;
  r.lse2 = lse[i] * kLog2e;
  r.scale = scale;
  // the target's column: its id in this vocabulary, or its position when sorted (inv)
  r.label = (valid && yl >= 0 && yl < V) ? (inv ? inv[yl] : static_cast<int32_t>(yl)) : -1;
  r.pad = 0;
  out[i] = r;
}

// Vocabulary-sharded forward: fixed-order merge (shard 0, 1, ...) of the per-shard row
// LSEs into the global one, lse = m + log sum_r exp(lse_r - m), the target logit as the
// sum of the per-shard ones (exactly one shard holds it), the per-row loss, and
// per-block loss sums (double) and (n_valid, n_bad) counts.
__global__ void __launch_bounds__(kMergeThreads)
    k_shard_merge(const float* __restrict__ lse_parts, const float* __restrict__ t_parts, int n_shards, int64_t N,
                  const int64_t* __restrict__ labels, int64_t ignore, int64_t V_total, float* __restrict__ lse_out,
                  float* __restrict__ loss_rows, double* __restrict__ blk_sums, int2* __restrict__ blk_counts) {
  __shared__ double sh[kMergeThreads];
  __shared__ int sv[kMergeThreads], sb[kMergeThreads];
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x;
  double mine = 0.0;
  int v = 0, b = 0;
  if (i < N) {
    float m = -INFINITY;
    for (int r = 0; r < n_shards; ++r) m = fmaxf(m, lse_parts[static_cast<int64_t>(r) * N + i]);
    float s = 0.0f, t = 0.0f;
    for (int r = 0; r < n_shards; ++r) {
      s += expf(lse_parts[static_cast<int64_t>(r) * N + i] - m);
      t += t_parts[static_cast<int64_t>(r) * N + i];
    }
    const float lse = m + logf(s);
    lse_out[i] = lse;
    const int64_t y = labels[i];
    const bool ignored = y == ignore;
    const bool valid = !ignored && y >= 0 && y < V_total;
    const float l = valid ? lse - t : 0.0f;
    if (loss_rows) loss_rows[i] = l;
    mine = l;
    v = valid ? 1 : 0;
    b = (!ignored && !valid) ? 1 : 0;
  }
  sh[threadIdx.x] = mine;
  sv[threadIdx.x] = v;
  sb[threadIdx.x] = b;
  __syncthreads();
  for (int w = kMergeThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      sh[threadIdx.x] += sh[threadIdx.x + w];
      sv[threadIdx.x] += sv[threadIdx.x + w];
      sb[threadIdx.x] += sb[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    blk_sums[blockIdx.x] = sh[0];
    blk_counts[blockIdx.x] = make_int2(sv[0], sb[0]);
  }
}

// Bitmasks of the live K steps of the dW and dH products over a filtered dZ chunk.
// nz is [TB][VB] bytes, one per 64 x 64 (token x vocabulary) block, non-zero when the
// block holds a non-zero dZ entry.
//   dH pair tile mt (token blocks 4mt..4mt+3), K steps = vocabulary blocks kb < kb_dh:
//     dh_mask[mt * dh_ld + kb / 32] bit kb % 32
//   dW pair tile vt (vocabulary blocks 4vt..4vt+3), K steps = token blocks tb < TB:
//     dw_mask[vt * dw_ld + tb / 32] bit tb % 32
__global__ void k_block_masks(const uint8_t* __restrict__ nz, int TB, int VB, int kb_dh, int MT, int VT,
                              uint32_t* __restrict__ dh_mask, int dh_ld, uint32_t* __restrict__ dw_mask, int dw_ld) {
  const int total_dh = MT * dh_ld;
  const int total = total_dh + VT * dw_ld;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    uint32_t bits = 0;
    if (i < total_dh) {
      const int mt = i / dh_ld, w = i - (i / dh_ld) * dh_ld;
      for (int j = 0; j < 32; ++j) {
        const int kb = w * 32 + j;
        if (kb >= kb_dh) break;
        uint32_t any = 0;
        for (int t = 0; t < 4; ++t) {
          const int tb = mt * 4 + t;
          if (tb < TB) any |= nz[static_cast<int64_t>(tb) * VB + kb];
        }
        bits |= (any != 0 ? 1u : 0u) << j;
      }
      dh_mask[i] = bits;
    } else {
      const int k = i - total_dh;
      const int vt = k / dw_ld, w = k - (k / dw_ld) * dw_ld;
      for (int j = 0; j < 32; ++j) {
        const int tb = w * 32 + j;
        if (tb >= TB) break;
        const uint32_t v4 = *reinterpret_cast<const uint32_t*>(nz + static_cast<int64_t>(tb) * VB + vt * 4);
        bits |= (v4 != 0 ? 1u : 0u) << j;
      }
      dw_mask[k] = bits;
    }
  }
}

}  // namespace flce
