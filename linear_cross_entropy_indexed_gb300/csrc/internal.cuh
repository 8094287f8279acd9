// Shared definitions between the host entry points and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace flce {

// Tile shape of every tensor-core kernel: a CTA pair computes 256 x 256 fp32 tiles;
// each CTA owns 128 of the rows (its TMEM lanes) and stages K 64 bf16 (one 128-byte
// swizzle row) at a time: its 128 rows of A and its 128-row half of B per stage.
constexpr int kBM = 128;                                   // rows per CTA
constexpr int kPairM = 2 * kBM;                            // rows per pair tile
constexpr int kBN = 256;                                   // columns per tile
constexpr int kBK = 64;
constexpr int kPairBRows = kBN / 2;                        // B rows staged by each CTA
constexpr int kATileBytes = kBM * kBK * 2;                 // 16 KiB
constexpr int kPairStageBytes = kATileBytes + kPairBRows * kBK * 2;  // 32 KiB
constexpr int kPairStages = 6;
constexpr int kEpiWarps = 4;                               // a multiple of 4
constexpr int kEpiSplit = kEpiWarps / 4;                   // warps per TMEM lane quadrant
constexpr int kSlices = kBN / 32;                          // 32-column slices per tile
constexpr int kSlicesPerWarp = kSlices / kEpiSplit;        // slices each epilogue warp drains
constexpr int kThreads = 64 + 32 * kEpiWarps;              // TMA warp, MMA warp, epilogue
constexpr int kTmemCols = 2 * kBN;                         // double-buffered accumulator
constexpr int kBarrierBytes = 256;
constexpr int kMaskWords = 512;                            // K-step bitmask words (16384 steps)
constexpr int kEpiStageBytes = 4096;                       // per epilogue warp: 32 rows x 128 B
constexpr size_t kPairSmemBytes = 1024 + size_t(kPairStages) * kPairStageBytes + kBarrierBytes +
                                  2 * kMaskWords * sizeof(uint32_t) + size_t(kEpiWarps) * kEpiStageBytes;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Persistent tile schedule.  Work is split into units; a unit is one 256-row M-tile and
// a run of `group` consecutive N-tiles (the LSE kernel keeps a running (max, sum)
// across them).  CTA pair p takes units p, p + pairs, ...
struct Sched {
  int m_tiles;
  int n_tiles;
  int k_blocks;
  int group;
  int n_groups;
  int units;
  int order;     // 0: consecutive units walk M first (share the B operand); 1: walk N first
  // > 0: the dimension walked first is walked in bands of this many tiles: all units of
  // one band (every tile of the other dimension) come before the next band's, so the
  // band's operand tiles stay in L2 while the other operand streams past once per band.
  int band;
  int b_n_off;   // added to the B operand's N coordinate (rows of W, K-major B)
  int b_k_off;   // added to the B operand's K coordinate (rows of W, MN-major B)
  // Block skipping over a filtered dZ chunk (null: off): per pair tile (M index), a
  // bitmask of its K steps whose dZ slab holds a non-zero entry, kmask_ld words per tile.
  // A K step whose slab is all zero is neither loaded nor multiplied.
  const uint32_t* kmask;
  int kmask_ld;
  // K split (1: off; the exact dH product only): every output tile's K steps are split
  // into k_split ranges run as separate units (units = k_split * m_tiles * n_groups, part
  // index slowest); part ks covers K blocks [ks k_blocks / k_split, (ks + 1) k_blocks /
  // k_split).  Fills the last wave of a launch that has few output tiles.
  int k_split;
  // Two-part A operand (0: off): K steps [0, k_half) read A through the first tensor map,
  // steps [k_half, 2 k_half) the same coordinates through the second; B is read at the
  // step index modulo k_half, so the accumulator sums A1 B + A2 B.
  int k_half;
  // Token extent read on the device at launch (null: the fields above stand).  The
  // backward runs on the rows that carry a gradient, compacted to the front; their count
  // is known only on the device.  n_role 1: M walks those rows, m_tiles = max(1,
  // ceil(n / 256)) and units = k_split * m_tiles * n_groups; n_role 2: K walks them,
  // k_blocks = max(1, ceil(n / 64)) (doubled with a two-part A operand).
  const int* n_dev;
  int n_role;
};

// Per-row data the dZ epilogue needs, packed in one 16-byte load.
struct RowInfo {
  float lse2;    // lse * log2(e)
  float scale;   // grad / n_valid, grad, grad_i, or 0 for an ignored row
  int32_t label; // y_i, or -1 when the row is ignored
  int32_t pad;
};

struct EpiLseParams {
  int64_t N, V;
  float softcap;        // <= 0: off
  float* part_m;        // [n_groups * kEpiSplit][N], running max in log2 units
  float* part_s;        // [n_groups * kEpiSplit][N], sum of 2^(z*log2e - max)
};

struct EpiDzParams {
  int64_t N, V;
  int64_t v0;           // first vocabulary row of this chunk
  int64_t wc;           // chunk width (columns of dZ that exist)
  int64_t ldz;          // row pitch of the dZ buffer in elements
  float softcap;
  const RowInfo* rows;
  __nv_bfloat16* dz;
  __nv_bfloat16* dz_lo;  // compensated mode: bf16 rounding remainder of dZ (same layout), else null
  float filter;         // drop entries with p < filter off the target (0: exact)
  uint8_t* nz;          // block flags written when filtering, else null
  int nz_ld;            // vocabulary blocks per token-block row of nz
};

struct EpiDwParams {
  int64_t rows_valid;    // chunk width: dZ^T rows that exist
  int64_t row0;          // first output row (vocabulary index, or position when sorted)
  int64_t cols;          // Hd
  __nv_bfloat16* out;    // dW, row pitch Hd
  const int32_t* perm;   // sorted vocabulary: output row of position q is perm[q]; else null
  int64_t out_rows;      // rows of dW (bound for the perm indirection)
};

struct EpiDhParams {
  int64_t N, Hd;
  float* acc32;         // [N, Hd] fp32 running sum across vocabulary chunks (compact rows)
  __nv_bfloat16* out;   // dH (rows of the original order)
  int first, last;
  float* parts;         // K split: fp32 sums of K parts 1 .. k_split - 1, [k_split - 1][N][Hd]
  // Compact rows: row r < *n_rows of the product is row row_map[r] of dH; rows from
  // *n_rows on are not written to dH.  Null: rows are dH's own.  acc_mapped: the running
  // sum acc32 is in dH's rows too (the fp32 partial of a vocabulary shard), else compact.
  const int32_t* row_map;
  const int* n_rows;
  int acc_mapped;
};

// Launchers (defined in the kernel translation units).  Each returns the launch error.
cudaError_t launch_linear_lse(const CUtensorMap& tmH, const CUtensorMap& tmW, const Sched& s,
                              const EpiLseParams& p, unsigned long long* err, int grid,
                              cudaStream_t st);
cudaError_t launch_dz(const CUtensorMap& tmH, const CUtensorMap& tmW, const Sched& s,
                      const EpiDzParams& p, unsigned long long* err, int grid, cudaStream_t st);
// tmDz2: second part of the A operand when s.k_half > 0 (see Sched), else unused.
cudaError_t launch_dw(const CUtensorMap& tmDz, const CUtensorMap& tmDz2, const CUtensorMap& tmH, const Sched& s,
                      const EpiDwParams& p, unsigned long long* err, int grid, cudaStream_t st);
cudaError_t launch_dh(const CUtensorMap& tmDz, const CUtensorMap& tmDz2, const CUtensorMap& tmW, const Sched& s,
                      const EpiDhParams& p, unsigned long long* err, int grid, cudaStream_t st);
cudaError_t set_gemm_smem_attributes_fwd();
cudaError_t set_gemm_smem_attributes_bwd();

}  // namespace flce
