// Persistent, warp-specialised tcgen05 GEMM engine with pluggable epilogues, run on
// CTA pairs (a 2-CTA cluster, cta_group::2).
//
// Each pair computes 256 x 256 output tiles: CTA r of the pair owns output rows
// [128 r, 128 r + 128) of the tile (its TMEM lanes) and stages, per K step of 64, its
// own 128 rows of A and its own 128 rows (half) of B, so a stage is 32 KiB and the
// ring is six stages deep.
//   warp 0      TMA producer (both CTAs): 128-byte-swizzled boxes into the ring; the
//               bytes of both CTAs complete on CTA 0's "full" barrier.
//   warp 1      MMA issuer (one thread of CTA 0): tcgen05.mma.cta_group::2 (M = 256,
//               N = 256, K = 16) into one of two TMEM accumulators (2 x 256 fp32
//               columns, allocated pair-wide), committing to both CTAs' barriers.
//   warps 2..5  epilogue (both CTAs): each warp owns the 32 TMEM lanes of its lane
//               quadrant, pulls 32 columns at a time with tcgen05.ld and runs the
//               epilogue (online LSE, dZ, dW store, dH accumulate) while the MMA warp
//               fills the other accumulator; one lane per warp then arrives on CTA 0's
//               "accumulator empty" barrier.
//
// Operands are K-major ([rows, K] with K contiguous) or MN-major ([K, rows] with rows
// contiguous); both use the 128-byte swizzle that the TMA writes:
//   K-major : one box {64 K, 128 rows};  8-row groups 1024 B apart (SBO), K step = +32 B
//   MN-major: two boxes {64 rows, 64 K}; 64-row atoms 8 KiB apart (LBO), 8-K groups
//             1024 B apart (SBO), K step of 16 = +2 KiB
#pragma once

#include "internal.cuh"
#include "ptx.cuh"

namespace flce {

__device__ __forceinline__ void decode_unit(const Sched& s, int u, int& mt, int& g, int& ks) {
  ks = 0;
  if (s.k_split > 1) {  // the K part is the slowest index
    const int per_part = s.m_tiles * s.n_groups;
    ks = u / per_part;
    u -= ks * per_part;
  }
  const int fast = s.order == 0 ? s.m_tiles : s.n_groups;  // dimension walked first
  const int slow = s.order == 0 ? s.n_groups : s.m_tiles;
  int f, sl;
  if (s.band > 0 && s.band < fast) {
    // band b holds fast-dimension tiles [b band, b band + width) crossed with every
    // slow-dimension index; inside it the fast index varies first
    const int per_band = s.band * slow;
    const int b = u / per_band;
    const int r = u - b * per_band;
    const int width = min(s.band, fast - b * s.band);
    sl = r / width;
    f = b * s.band + (r - sl * width);
  } else {
    sl = u / fast;
    f = u - sl * fast;
  }
  if (s.order == 0) {
    mt = f;
    g = sl;
  } else {
    g = f;
    mt = sl;
  }
}

template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int k) {
  if constexpr (!MN) {
    return smem_desc_sw128(base + k * 32, 16, 1024);
  } else {
    return smem_desc_sw128(base + k * 2048, 8192, 1024);
  }
}

// ====================================================================== epilogues
// Every epilogue thread owns one TMEM lane (output row) and drains slices
// [h * kSlicesPerWarp, (h + 1) * kSlicesPerWarp) of 32 fp32 columns, h = its warp's
// column half.  Per-element work is kept to a few FMAs around the MUFU operations.

// tanh(u) = 1 - 2 / (e^{2u} + 1); the caller passes a = 2u log2(e), so e^{2u} = 2^a.
// Absolute error a few fp32 ulps of 1 (no cancellation blow-up for small u); saturates
// to +-1 for large |u|.
__device__ __forceinline__ float tanh_from_exp2_arg(float a) {
  return fmaf(-2.0f, rcp_approx(ex2_approx(a) + 1.0f), 1.0f);
}

template <class F>
__device__ __forceinline__ void for_each_slice(uint32_t taddr, int h, F&& f) {
#pragma unroll 1
  for (int c = h * kSlicesPerWarp; c < (h + 1) * kSlicesPerWarp; ++c) {
    float x[32];
    __syncwarp();  // tcgen05.ld is warp-collective: reconverge first
    tmem_ld32(taddr + c * 32, x);
    f(c, x);
  }
}

// Forward: running (max, sum) of 2^(z log2 e) over the unit's vocabulary tiles.
struct EpiLse {
  using Params = EpiLseParams;
  struct State {
    float m;  // running max of z*log2e
    float s;  // sum of 2^(z*log2e - m)
  };
  __device__ static void unit_begin(const Params&, State& st) {
    st.m = -INFINITY;
    st.s = 0.0f;
  }
  // z is monotone in its key k (k = x without softcap, k = tanh(x/c) with it), so the
  // slice max is taken on k and z*log2e = k * zs.
  template <bool CAP>
  __device__ static void slices(const Params& p, State& st, uint32_t taddr, int nt, int h) {
    const int64_t v_tile = static_cast<int64_t>(nt) * kBN;
    const float k_tanh = CAP ? 2.0f * kLog2e / p.softcap : 0.0f;
    const float zs = CAP ? p.softcap * kLog2e : kLog2e;
    for_each_slice(taddr, h, [&](int c, float(&x)[32]) {
      const int64_t v0 = v_tile + c * 32;
      if (v0 >= p.V) return;  // the whole slice is past V
      if (CAP) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = tanh_from_exp2_arg(x[j] * k_tanh);
      }
      if (v0 + 32 > p.V) {
        const int n = static_cast<int>(p.V - v0);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j >= n) x[j] = -INFINITY;
      }
      float kmax = x[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) kmax = fmaxf(kmax, x[j]);
      const float mn = fmaxf(st.m, kmax * zs);
      float acc = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) acc += ex2_approx(fmaf(x[j], zs, -mn));
      st.s = st.s * ex2_approx(st.m - mn) + acc;  // 2^-inf = 0 for the first slice
      st.m = mn;
    });
  }
  __device__ static void tile(const Params& p, State& st, uint32_t taddr, int64_t, int nt, int h, uint8_t*, int) {
    if (p.softcap > 0.0f)
      slices<true>(p, st, taddr, nt, h);
    else
      slices<false>(p, st, taddr, nt, h);
  }
  __device__ static void unit_end(const Params& p, State& st, int64_t row, int g, int h) {
    if (row < p.N) {
      const int64_t k = static_cast<int64_t>(g) * kEpiSplit + h;
      p.part_m[k * p.N + row] = st.m;
      p.part_s[k * p.N + row] = st.s;
    }
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Backward: recompute the logit tile, dZ = (p - onehot) * scale * cap', bf16 store.
// With filtering, entries with p below the threshold (other than the target) are
// dropped and each warp marks the 64 x 64 blocks it wrote a non-zero into.
struct EpiDz {
  using Params = EpiDzParams;
  struct State {};
  __device__ static void unit_begin(const Params&, State&) {}
  __device__ static void unit_end(const Params&, State&, int64_t, int, int) {}
  template <bool CAP, bool FILTER, bool SPLIT>
  __device__ static void slices(const Params& p, uint32_t taddr, int64_t row, int nt, int h) {
    RowInfo ri{0.0f, 0.0f, -1, 0};
    const bool row_ok = row < p.N;
    if (row_ok) ri = p.rows[row];
    const float k_tanh = CAP ? 2.0f * kLog2e / p.softcap : 0.0f;
    const float zs = CAP ? p.softcap * kLog2e : kLog2e;
    const float neg_scale = -ri.scale;
    const int64_t vl_tile = static_cast<int64_t>(nt) * kBN;
    const int64_t y_local = ri.label >= 0 ? static_cast<int64_t>(ri.label) - p.v0 : -1;
    __nv_bfloat16* out_row = p.dz + (row_ok ? row : 0) * p.ldz;
    __nv_bfloat16* lo_row = SPLIT ? p.dz_lo + (row_ok ? row : 0) * p.ldz : nullptr;
    for_each_slice(taddr, h, [&](int c, float(&x)[32]) {
      const int64_t vl = vl_tile + c * 32;
      if (vl >= p.wc) return;  // same for the whole warp
      const int yrel = (y_local >= vl && y_local < vl + 32) ? static_cast<int>(y_local - vl) : -1;
      uint32_t pk[16];
      uint32_t pl[SPLIT ? 16 : 1];
      bool nonzero = false;
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        float d[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float dv, pr;
          if (CAP) {
            const float t = tanh_from_exp2_arg(x[j + e] * k_tanh);
            pr = ex2_approx(fmaf(t, zs, -ri.lse2));
            dv = fmaf(pr, ri.scale, (j + e == yrel) ? neg_scale : 0.0f) * fmaf(-t, t, 1.0f);
          } else {
            pr = ex2_approx(fmaf(x[j + e], zs, -ri.lse2));
            dv = fmaf(pr, ri.scale, (j + e == yrel) ? neg_scale : 0.0f);
          }
          if (FILTER) {
            if (pr < p.filter && j + e != yrel) dv = 0.0f;
            nonzero |= dv != 0.0f;
          }
          d[e] = dv;
        }
        pk[j / 2] = pack_bf16x2(d[0], d[1]);
        if (SPLIT) {  // remainder of the bf16 rounding, itself rounded to bf16
          const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&pk[j / 2]);
          const float2 hf = __bfloat1622float2(hb);
          pl[j / 2] = pack_bf16x2(d[0] - hf.x, d[1] - hf.y);
        }
      }
      if (FILTER) {
        const unsigned any = __ballot_sync(0xffffffffu, nonzero && row_ok);
        if (any != 0 && (threadIdx.x & 31) == 0) p.nz[(row / 64) * p.nz_ld + vl / 64] = 1;
      }
      if (!row_ok) return;
      if (vl + 32 <= p.wc) {
        uint4* dst = reinterpret_cast<uint4*>(out_row + vl);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        if (SPLIT) {
          uint4* dlo = reinterpret_cast<uint4*>(lo_row + vl);
#pragma unroll
          for (int k = 0; k < 4; ++k) dlo[k] = make_uint4(pl[4 * k], pl[4 * k + 1], pl[4 * k + 2], pl[4 * k + 3]);
        }
      } else {
        for (int j = 0; j < 32 && vl + j < p.wc; ++j) {
          const uint32_t w = pk[j / 2];
          const uint16_t hbits = static_cast<uint16_t>((j & 1) ? (w >> 16) : (w & 0xFFFFu));
          reinterpret_cast<uint16_t*>(out_row)[vl + j] = hbits;
          if (SPLIT) {
            const uint32_t wl = pl[j / 2];
            reinterpret_cast<uint16_t*>(lo_row)[vl + j] = static_cast<uint16_t>((j & 1) ? (wl >> 16) : (wl & 0xFFFFu));
          }
        }
      }
    });
  }
  __device__ static void tile(const Params& p, State&, uint32_t taddr, int64_t row, int nt, int h, uint8_t*, int) {
    const bool cap = p.softcap > 0.0f;
    if (p.nz != nullptr) {  // filtering (the backward never combines it with the split)
      if (cap)
        slices<true, true, false>(p, taddr, row, nt, h);
      else
        slices<false, true, false>(p, taddr, row, nt, h);
    } else if (p.dz_lo != nullptr) {
      if (cap)
        slices<true, false, true>(p, taddr, row, nt, h);
      else
        slices<false, false, true>(p, taddr, row, nt, h);
    } else {
      if (cap)
        slices<true, false, false>(p, taddr, row, nt, h);
      else
        slices<false, false, false>(p, taddr, row, nt, h);
    }
  }
};

// Backward: dW chunk = dZ^T H, converted to bf16 and written once.
// The dW and dH epilogues write through a per-warp staging buffer: each thread drops its
// row's slice (32 columns) into shared memory, then the warp writes rows back as whole
// 64- or 128-byte segments (8 or 4 rows per store instruction) instead of one 16-byte
// piece of 32 different rows.  The 16-byte chunks of a staged row are XOR-swizzled by the
// row index so that both the row-wise writes and the chunk-wise reads are free of bank
// conflicts.

// Backward: dW rows of the chunk = dZ_chunk^T H, bf16.
struct EpiDw {
  using Params = EpiDwParams;
  struct State {};
  __device__ static void unit_begin(const Params&, State&) {}
  __device__ static void unit_end(const Params&, State&, int64_t, int, int) {}
  __device__ static void tile(const Params& p, State&, uint32_t taddr, int64_t row, int nt, int h, uint8_t* stage,
                                   int) {
    const int lane = threadIdx.x & 31;
    bool row_ok = row < p.rows_valid;
    int64_t orow = p.row0 + (row_ok ? row : 0);
    if (p.perm != nullptr && row_ok) {  // sorted vocabulary: position -> id
      orow = p.perm[orow];
      row_ok = orow >= 0 && orow < p.out_rows;
    }
    const int64_t mine = row_ok ? orow : -1;
    // store step i writes rows 8i .. 8i+7 of the warp: lane -> row 8i + lane/4, chunk lane%4
    int64_t dst[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = __shfl_sync(0xffffffffu, mine, 8 * i + (lane >> 2));
    const int ch = lane & 3;
    for_each_slice(taddr, h, [&](int c, float(&x)[32]) {
      const int64_t col = static_cast<int64_t>(nt) * kBN + c * 32;
      if (col >= p.cols) return;  // same for the whole warp
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint4*>(stage + lane * 64 + 16 * (k ^ ((lane >> 1) & 3))) =
            make_uint4(pack_bf16x2(x[8 * k], x[8 * k + 1]), pack_bf16x2(x[8 * k + 2], x[8 * k + 3]),
                       pack_bf16x2(x[8 * k + 4], x[8 * k + 5]), pack_bf16x2(x[8 * k + 6], x[8 * k + 7]));
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = 8 * i + (lane >> 2);
        const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * 64 + 16 * (ch ^ ((rr >> 1) & 3)));
        if (dst[i] >= 0 && col + 8 * ch + 8 <= p.cols)
          *reinterpret_cast<uint4*>(p.out + dst[i] * p.cols + col + 8 * ch) = v;
      }
      __syncwarp();
    });
  }
};

// Backward: dH += dZ_chunk W_chunk; fp32 running sum across chunks, bf16 at the end.
// The running sum's values for the next slice are loaded while the current one is
// added, so the read-modify-write costs one memory latency per tile, not per slice.
// With a K split, part 0 updates the running sum (never the bf16 output: the parts are
// added afterwards) and part ks > 0 stores its fp32 sum into its own slice of `parts`.
struct EpiDh {
  using Params = EpiDhParams;
  struct State {};
  __device__ static void unit_begin(const Params&, State&) {}
  __device__ static void unit_end(const Params&, State&, int64_t, int, int) {}
  __device__ static void tile(const Params& pp, State&, uint32_t taddr, int64_t row, int nt, int h, uint8_t* stage,
                              int ks) {
    Params p = pp;
    if (ks > 0) {
      p.acc32 = pp.parts + static_cast<int64_t>(ks - 1) * pp.N * pp.Hd;
      p.first = 1;
      p.last = 0;
      p.acc_mapped = 0;
    }
    const int lane = threadIdx.x & 31;
    const int64_t mine = row < p.N ? row : -1;
    // the row of dH this product row lands in (compact rows: through the row map; rows
    // past the compact count hold no gradient and land nowhere)
    int64_t out_mine = mine, acc_mine = mine;
    if (p.row_map != nullptr && (p.last || p.acc_mapped)) {
      const int64_t nr = *p.n_rows;
      const int64_t o = (mine >= 0 && row < nr) ? static_cast<int64_t>(p.row_map[row]) : -1;
      out_mine = (o >= 0 && o < p.N) ? o : -1;
      if (p.acc_mapped) acc_mine = out_mine;
    }
    // step i moves rows 4i .. 4i+3 of the warp: lane -> row 4i + lane/8, 4-column chunk lane%8
    int64_t dst[8], odst[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      dst[i] = __shfl_sync(0xffffffffu, acc_mine, 4 * i + (lane >> 3));
      odst[i] = __shfl_sync(0xffffffffu, out_mine, 4 * i + (lane >> 3));
    }
    const int ch = lane & 7;
    const int64_t col_tile = static_cast<int64_t>(nt) * kBN;
    const int c_end = (h + 1) * kSlicesPerWarp;
    float4 pre[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) pre[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    auto load_sum = [&](int c) {  // this lane's part of slice c of the running sum
      const int64_t cc = col_tile + c * 32 + 4 * ch;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pre[i] = (dst[i] >= 0 && cc + 4 <= p.Hd) ? *reinterpret_cast<const float4*>(p.acc32 + dst[i] * p.Hd + cc)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    if (!p.first) load_sum(h * kSlicesPerWarp);
    for_each_slice(taddr, h, [&](int c, float(&x)[32]) {
      const int64_t col = col_tile + c * 32;
      if (col >= p.Hd) return;  // same for the whole warp
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<float4*>(stage + lane * 128 + 16 * (k ^ (lane & 7))) =
            make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
      __syncwarp();
      float4 cur[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = pre[i];
      if (!p.first && c + 1 < c_end && col + 32 < p.Hd) load_sum(c + 1);
      const int64_t cc = col + 4 * ch;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3);
        float4 v = *reinterpret_cast<const float4*>(stage + rr * 128 + 16 * (ch ^ (rr & 7)));
        if (dst[i] < 0 || cc + 4 > p.Hd) continue;
        if (!p.first) {
          v.x += cur[i].x;
          v.y += cur[i].y;
          v.z += cur[i].z;
          v.w += cur[i].w;
        }
        if (p.last) {
          if (odst[i] >= 0)
            *reinterpret_cast<uint2*>(p.out + odst[i] * p.Hd + cc) =
                make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        } else {
          *reinterpret_cast<float4*>(p.acc32 + dst[i] * p.Hd + cc) = v;
        }
      }
      __syncwarp();
    });
  }
};

// ====================================================================== engine
static_assert(kPairSmemBytes <= 232448, "pair pipeline exceeds shared memory");

// Block skipping over a filtered dZ chunk: sched.kmask holds, per pair tile (M index),
// a bitmask of the K steps whose dZ slab has a non-zero entry (built by k_block_masks).
// At each tile start the issuing thread copies the tile's words to shared memory with
// independent loads; producer and MMA thread copy the same words, so they take the
// same decisions.
__device__ __forceinline__ void load_kmask(const Sched& s, int mt, uint32_t* mask) {
  const uint32_t* src = s.kmask + static_cast<int64_t>(mt) * s.kmask_ld;
  const int words = (s.k_blocks + 31) / 32;
  for (int w = 0; w < words; ++w) mask[w] = __ldg(src + w);
}

// Calls f(kb), in increasing order, for every K step the tile runs: the steps whose
// mask bit is set, or the last step alone when no bit is set (so that the accumulator
// of an all-zero tile is initialised, to zero).  The mask is read one 32-step word at
// a time and only set bits are visited, so a skipped step costs nothing.  Returns false
// as soon as f does.
template <class F>
__device__ __forceinline__ bool for_each_live_kblock(const Sched& s, const uint32_t* mask, F&& f) {
  const int words = (s.k_blocks + 31) / 32;
  const uint32_t tail = (s.k_blocks & 31) ? ((1u << (s.k_blocks & 31)) - 1u) : 0xffffffffu;
  bool any = false;
  for (int wd = 0; wd < words; ++wd) {
    uint32_t bits = mask[wd];
    if (wd == words - 1) {
      bits &= tail;
      if (!any && bits == 0) bits = 1u << ((s.k_blocks - 1) & 31);
    }
    while (bits != 0) {
      const int j = __ffs(bits) - 1;
      bits &= bits - 1u;
      any = true;
      if (!f(wd * 32 + j)) return false;
    }
  }
  return true;
}

template <bool MN>
__device__ __forceinline__ void load_half_pair(uint32_t dst, const CUtensorMap* tm, uint32_t bar_cluster, int row0,
                                               int k0) {
  if constexpr (!MN) {
    tma_load_2d_pair(dst, tm, bar_cluster, k0, row0);
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j) tma_load_2d_pair(dst + j * 8192, tm, bar_cluster, row0 + j * 64, k0);
  }
}

template <class Epi, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB,
                        const Sched sched_in, const typename Epi::Params ep, unsigned long long* err) {
  extern __shared__ uint8_t smem_raw[];
  // the token extent of a compacted backward is read here, before any role uses the schedule
  Sched sched = sched_in;
  if (sched.n_dev != nullptr) {
    const int n = max(0, *sched.n_dev);
    if (sched.n_role == 1) {
      sched.m_tiles = max(1, (n + kPairM - 1) / kPairM);
      sched.units = (sched.k_split > 1 ? sched.k_split : 1) * sched.m_tiles * sched.n_groups;
    } else if (sched.n_role == 2) {
      const int kb = max(1, (n + kBK - 1) / kBK);
      if (sched.k_half > 0) {
        sched.k_half = kb;
        sched.k_blocks = 2 * kb;
      } else {
        sched.k_blocks = kb;
      }
    }
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kPairStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* kmask = reinterpret_cast<uint32_t*>(smem + kPairStages * kPairStageBytes + kBarrierBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int ksplit = sched.k_split > 1 ? sched.k_split : 1;  // Sched{} leaves it 0: no split
  const uint32_t tiles_u32 = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kPairStages;
  const uint32_t tfull0 = empty0 + 8 * kPairStages;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    if (sched.k_half > 0) tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised before any remote arrive / complete_tx
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t full0_lead = mapa_shared(full0, 0);
  const uint32_t tempty0_lead = mapa_shared(tempty0, 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      for (int u = pair; ok && u < sched.units; u += npairs) {
        int mt, g, ks;
        decode_unit(sched, u, mt, g, ks);
        const int kb0 = ks * sched.k_blocks / ksplit;  // K split: this part's K blocks
        const int kb1 = (ks + 1) * sched.k_blocks / ksplit;
        const int nt0 = g * sched.group;
        const int nt1 = min(nt0 + sched.group, sched.n_tiles);
        for (int nt = nt0; ok && nt < nt1; ++nt) {
          // one K step: wait for a free slot, arm the full barrier, load both halves of A
          // (through map ta) and of B, at K block kb
          auto load_k = [&](const CUtensorMap* ta, int kb) -> bool {
            if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, err)) return false;
            if (leader) mbar_arrive_expect_tx(full0 + 8 * stage, 2 * kPairStageBytes);
            const uint32_t a = tiles_u32 + stage * kPairStageBytes;
            const uint32_t fb = full0_lead + 8 * stage;
            load_half_pair<A_MN>(a, ta, fb, mt * kPairM + int(rank) * kBM, kb * kBK);
            load_half_pair<B_MN>(a + kATileBytes, &tmB, fb, nt * kBN + int(rank) * kPairBRows + sched.b_n_off,
                                 kb * kBK + sched.b_k_off);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1;
            }
            return true;
          };
          auto load_step = [&](int kb) -> bool { return load_k(&tmA, kb); };
          if (sched.kmask == nullptr && sched.k_half == 0) {
            for (int kb = kb0; kb < kb1; ++kb)
              if (!load_step(kb)) {
                ok = false;
                break;
              }
          } else if (sched.kmask == nullptr) {  // two-part A: A1 B over all K blocks, then A2 B
            for (int kb = 0; kb < sched.k_blocks; ++kb) {
              const bool second = kb >= sched.k_half;
              if (!load_k(second ? &tmA2 : &tmA, second ? kb - sched.k_half : kb)) {
                ok = false;
                break;
              }
            }
          } else {  // filtered dZ: only the K steps of the tile's mask
            uint32_t* mask = kmask;
            load_kmask(sched, mt, mask);
            if (!for_each_live_kblock(sched, mask, load_step)) ok = false;
          }
        }
      }
      if (!ok && leader) {
        volatile int never = 0;
        for (int s = 0; s < kPairStages; ++s)
          if (armed & (1u << s)) mbar_wait(full0 + 8 * s, (armed_parity >> s) & 1u, &never, err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA issuer (CTA 0)
      constexpr uint32_t idesc = idesc_bf16_f32(kPairM, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int u = pair; ok && u < sched.units; u += npairs) {
        int mt, g, ks;
        decode_unit(sched, u, mt, g, ks);
        const int kb0 = ks * sched.k_blocks / ksplit;
        const int kb1 = (ks + 1) * sched.k_blocks / ksplit;
        const int nt0 = g * sched.group;
        const int nt1 = min(nt0 + sched.group, sched.n_tiles);
        for (int nt = nt0; ok && nt < nt1; ++nt) {
          if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * kBN;
          if (sched.kmask == nullptr) {
            for (int kb = kb0; kb < kb1; ++kb) {
              if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a = tiles_u32 + stage * kPairStageBytes;
              const uint32_t b = a + kATileBytes;
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                mma_bf16_pair(d, operand_desc<A_MN>(a, k), operand_desc<B_MN>(b, k), idesc,
                              ((kb - kb0) | k) != 0 ? 1u : 0u);
              issued = true;
              mma_commit_pair(empty0 + 8 * stage, 0x3);
              if (++stage == kPairStages) {
                stage = 0;
                phase ^= 1;
              }
            }
          } else {  // filtered dZ: only the K steps of the tile's mask
            uint32_t* mask = kmask + kMaskWords;
            load_kmask(sched, mt, mask);
            int done = 0;
            ok = for_each_live_kblock(sched, mask, [&](int) -> bool {
              if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, err)) return false;
              tc_fence_after();
              const uint32_t a = tiles_u32 + stage * kPairStageBytes;
              const uint32_t b = a + kATileBytes;
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                mma_bf16_pair(d, operand_desc<A_MN>(a, k), operand_desc<B_MN>(b, k), idesc,
                              (done | k) != 0 ? 1u : 0u);
              ++done;
              issued = true;
              mma_commit_pair(empty0 + 8 * stage, 0x3);
              if (++stage == kPairStages) {
                stage = 0;
                phase ^= 1;
              }
              return true;
            });
          }
          if (!ok) break;
          mma_commit_pair(tfull0 + 8 * acc, 0x3);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1;
          }
        }
      }
      if (!ok && issued) {
        volatile int never = 0;
        mma_commit_pair(drain, 0x1);
        mbar_wait(drain, 0, &never, err);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;               // TMEM lane quadrant this warp may access
    const int h = (warp - 2) / 4;         // column half of the tile this warp drains
    const int row_in_tile = int(rank) * kBM + q * 32 + lane;
    uint8_t* epi_stage = smem + kPairStages * kPairStageBytes + kBarrierBytes + 2 * kMaskWords * sizeof(uint32_t) +
                         (warp - 2) * kEpiStageBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int u = pair; ok && u < sched.units; u += npairs) {
      int mt, g, ks;
      decode_unit(sched, u, mt, g, ks);
      const int nt0 = g * sched.group;
      const int nt1 = min(nt0 + sched.group, sched.n_tiles);
      const int64_t row = static_cast<int64_t>(mt) * (2 * kBM) + row_in_tile;
      typename Epi::State st;
      Epi::unit_begin(ep, st);
      for (int nt = nt0; nt < nt1; ++nt) {
        if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
        Epi::tile(ep, st, taddr, row, nt, h, epi_stage, ks);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0_lead + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) break;
      Epi::unit_end(ep, st, row, g, h);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its barriers or TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

template <class Epi, bool A_MN, bool B_MN>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmA2, const CUtensorMap& tmB, const Sched& s,
                             const typename Epi::Params& p, unsigned long long* err, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<Epi, A_MN, B_MN>, tmA, tmA2, tmB, s, p, err);
}

template <class Epi, bool A_MN, bool B_MN>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(tc_gemm_kernel<Epi, A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kPairSmemBytes));
}

}  // namespace flce
