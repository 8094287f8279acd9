// Vocabulary order for block-aligned gradient filtering (Liger-CCE blog, §三 "CCE": the
// mean logit of every word, tallied over the batch, orders the vocabulary so that the
// words whose probabilities survive the filter share blocks and the rest of the blocks
// can be skipped whole).
//
// key_v = (1/N) sum_i x_iv, the raw logit averaged over all N rows.  By linearity it is
// hbar . w_v with hbar the column mean of H, which needs one pass over H and one over W
// instead of a reduction across the rows of every logit tile.  The order is keys
// descending, equal keys by ascending id: each entry becomes the 64-bit word
// (descending image of its key) << 32 | id, all words are distinct, and an ascending
// sort of the words is the order.  The sort is a shared-memory bitonic sort of runs of
// kSortSeg words followed by merge passes that place each word by binary search in its
// partner run; every step has a fixed order, so the permutation is deterministic.
#pragma once

#include "internal.cuh"

namespace flce {

constexpr int kColThreads = 128;    // 8 columns of H per thread
constexpr int kSortSeg = 4096;      // words sorted per block in shared memory
constexpr int kSortThreads = 1024;
constexpr int kMergeSortThreads = 256;
constexpr int kRowCopyThreads = 256;  // 8 rows (one per warp) per block
constexpr unsigned long long kDevErrBadIndex = 2ull;  // FLCE_DEVERR_BAD_INDEX

// Column sums of H over the rows of segment blockIdx.y: part[seg][c .. c + 8).
// Hd % 8 == 0 and a 16-byte aligned H make every 8-column group one 16-byte load.
__global__ void __launch_bounds__(kColThreads)
    k_col_partial(const __nv_bfloat16* __restrict__ H, int64_t N, int64_t Hd, int64_t rows_per_seg,
                  float* __restrict__ part) {
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * kColThreads + threadIdx.x) * 8;
  if (c >= Hd) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_seg;
  const int64_t r1 = r0 + rows_per_seg < N ? r0 + rows_per_seg : N;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int64_t r = r0; r < r1; ++r) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(H + r * Hd + c));
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      acc[2 * j] += f.x;
      acc[2 * j + 1] += f.y;
    }
  }
  float* out = part + static_cast<int64_t>(blockIdx.y) * Hd + c;
#pragma unroll
  for (int j = 0; j < 8; ++j) out[j] = acc[j];
}

// hbar[c] = (segment sums added in segment order) / N.
__global__ void k_col_mean(const float* __restrict__ part, int n_seg, int64_t Hd, int64_t N,
                           float* __restrict__ hbar) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= Hd) return;
  float s = 0.0f;
  for (int k = 0; k < n_seg; ++k) s += part[static_cast<int64_t>(k) * Hd + c];
  hbar[c] = s / static_cast<float>(N);
}

// Ascending order of the returned word = descending order of k; -0 and +0 are one key.
__device__ __forceinline__ uint32_t descending_image(float k) {
  uint32_t u = __float_as_uint(k);
  if ((u << 1) == 0u) u = 0u;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // ascending in k
  return ~u;
}

// One warp per vocabulary row: key[v] = hbar . w_v in fp32 (each lane sums its
// 8-column groups in order, then a fixed shuffle tree; lane 0's total is stored).
__global__ void __launch_bounds__(kRowCopyThreads)
    k_vocab_keys(const __nv_bfloat16* __restrict__ W, const float* __restrict__ hbar, int64_t V, int64_t Hd,
                 float* __restrict__ key, unsigned long long* __restrict__ word) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t v = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; v < V; v += n_warps) {
    const __nv_bfloat16* w = W + v * Hd;
    float acc = 0.0f;
#pragma unroll 8
    for (int64_t c = lane * 8; c < Hd; c += 256) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(w + c));
      const float4 h0 = __ldg(reinterpret_cast<const float4*>(hbar + c));
      const float4 h1 = __ldg(reinterpret_cast<const float4*>(hbar + c + 4));
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&q);
      const float2 f0 = __bfloat1622float2(b[0]), f1 = __bfloat1622float2(b[1]);
      const float2 f2 = __bfloat1622float2(b[2]), f3 = __bfloat1622float2(b[3]);
      acc = fmaf(f0.x, h0.x, acc);
      acc = fmaf(f0.y, h0.y, acc);
      acc = fmaf(f1.x, h0.z, acc);
      acc = fmaf(f1.y, h0.w, acc);
      acc = fmaf(f2.x, h1.x, acc);
      acc = fmaf(f2.y, h1.y, acc);
      acc = fmaf(f3.x, h1.z, acc);
      acc = fmaf(f3.y, h1.w, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      key[v] = acc;
      word[v] = (static_cast<unsigned long long>(descending_image(acc)) << 32) | static_cast<unsigned long long>(v);
    }
  }
}

// Sort runs of kSortSeg words per block in shared memory (bitonic network, ascending).
// The last run is padded with all-ones words, which sort last and are not written back
// (a real word's low half is an id below 2^31, so no real word is all ones).
__global__ void __launch_bounds__(kSortThreads)
    k_sort_runs(const unsigned long long* __restrict__ in, unsigned long long* __restrict__ out, int64_t n) {
  __shared__ unsigned long long s[kSortSeg];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kSortSeg;
  for (int i = threadIdx.x; i < kSortSeg; i += kSortThreads) s[i] = base + i < n ? in[base + i] : ~0ull;
  __syncthreads();
  for (int k = 2; k <= kSortSeg; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = threadIdx.x; t < kSortSeg / 2; t += kSortThreads) {
        const int i = 2 * t - (t & (j - 1));  // bit j of i is clear; its partner is i + j
        const unsigned long long a = s[i], b = s[i + j];
        const bool up = (i & k) == 0;
        if ((a > b) == up) {
          s[i] = b;
          s[i + j] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < kSortSeg; i += kSortThreads)
    if (base + i < n) out[base + i] = s[i];
}

// Merge neighbouring sorted runs of length L into runs of 2L: a word's position is its
// index in its own run plus the number of smaller words in the partner run.
__global__ void __launch_bounds__(kMergeSortThreads)
    k_merge_runs(const unsigned long long* __restrict__ in, unsigned long long* __restrict__ out, int64_t n,
                 int64_t L) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n; idx += stride) {
    const int64_t base = idx / (2 * L) * (2 * L);
    const int64_t mid = base + L < n ? base + L : n;
    const int64_t end = base + 2 * L < n ? base + 2 * L : n;
    const unsigned long long x = in[idx];
    int64_t lo = mid, hi = end, own = idx - base;
    if (idx >= mid) {
      lo = base;
      hi = mid;
      own = idx - mid;
    }
    const int64_t first = lo;
    while (lo < hi) {
      const int64_t m = (lo + hi) >> 1;
      if (in[m] < x)
        lo = m + 1;
      else
        hi = m;
    }
    out[base + own + (lo - first)] = x;
  }
}

// perm[p] = id at position p; inv[id] = p (inv may be null).
__global__ void k_order_finish(const unsigned long long* __restrict__ sorted, int64_t n, int32_t* __restrict__ perm,
                               int32_t* __restrict__ inv, unsigned long long* __restrict__ err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < n; p += stride) {
    const int64_t v = static_cast<int64_t>(sorted[p] & 0xffffffffull);
    if (v >= n) {  // cannot happen for a permutation; recorded, never used as an index
      if (err) atomicOr(err, kDevErrBadIndex);
      perm[p] = 0;
      continue;
    }
    perm[p] = static_cast<int32_t>(v);
    if (inv) inv[v] = static_cast<int32_t>(p);
  }
}

// out[j] = W[perm[j0 + j]] for j < rows (one warp per row, 16-byte vectors).  An id
// outside [0, V) sets the error bit and leaves the row as it was.
__global__ void __launch_bounds__(kRowCopyThreads)
    k_gather_rows(const __nv_bfloat16* __restrict__ W, int64_t V, int64_t Hd, const int32_t* __restrict__ perm,
                  int64_t j0, int64_t rows, __nv_bfloat16* __restrict__ out, unsigned long long* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t j = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; j < rows; j += n_warps) {
    const int64_t v = perm[j0 + j];
    if (v < 0 || v >= V) {
      if (lane == 0) atomicOr(err, kDevErrBadIndex);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(W + v * Hd);
    uint4* dst = reinterpret_cast<uint4*>(out + j * Hd);
#pragma unroll 4
    for (int64_t c = lane; c < Hd / 8; c += 32) dst[c] = __ldg(src + c);
  }
}

}  // namespace flce
