// Internal launch interface between the C ABI (phobos_gemm.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/phobos_gemm.h"

namespace phobos {

// ---------------------------------------------------------------- FFMA path
struct FfmaArgs {
  const float *A;
  const float *B;
  float *C;
  int64_t lda, ldb, ldc;
  int M, N, K;
  float alpha, beta;
  int tile;        // 128 (128x128 tile, 256 threads) or 64 (64x64 tile, 64 threads)
  int k_begin;     // first k of this launch
  int k_len;       // number of k of this launch
  int vec_a, vec_b, vec_c;  // 16-byte vector access allowed for A / B / C
  // 64x64 tiles only: K slices per tile (1 = off, 2..8).  The slices of a tile
  // form one thread-block cluster and are summed through distributed shared
  // memory by the cluster's rank 0, in rank order.
  int kslices;
};
cudaError_t launch_ffma(const FfmaArgs &a, cudaStream_t stream);

// ------------------------------------------------------ split / pack pre-pass
// A (M x K, row-major, lda) -> big/small [Mp][Kp]; zero padding.
cudaError_t launch_split_rows(const float *A, int64_t lda, int M, int K, int Mp, int Kp,
                              float *big, float *small, int vec, cudaStream_t stream);
// B (K x N, row-major, ldb) -> transposed big/small [Np][Kp] (K-major); zero padding.
cudaError_t launch_split_cols(const float *B, int64_t ldb, int K, int N, int Np, int Kp,
                              float *big, float *small, cudaStream_t stream);
// Both splits and the zeroing of the tail-split flags in one launch.  The
// launcher fills a_blocks and b_tiles_*; split_a / split_b select the parts
// (a launch with neither only zeroes the flags).
struct SplitArgs {
  const float *A;
  int64_t lda;
  int M, K, Mp, Kp;
  float *a_big, *a_small;  // a_small may be null (one-pass TF32)
  int vec_a;               // 16-byte loads of A allowed
  const float *B;
  int64_t ldb;
  int N, Np;
  float *b_big, *b_small;  // b_small may be null
  unsigned *flags;
  int64_t n_flags;
  int a_blocks, b_tiles_k, b_tiles_n;
};
cudaError_t launch_split_ab(SplitArgs a, int split_a, int split_b, cudaStream_t stream);
// The same layouts with one 16-bit operand (fp16 when bf16 == 0, else bf16),
// each element rounded to nearest, ties to even.  `out` holds 2-byte elements.
cudaError_t launch_convert_rows(const float *A, int64_t lda, int M, int K, int Mp, int Kp,
                                void *out, int bf16, cudaStream_t stream);
cudaError_t launch_convert_cols(const float *B, int64_t ldb, int K, int N, int Np, int Kp,
                                void *out, int bf16, cudaStream_t stream);
// C = beta * C (beta == 0: C = 0 without reading C).
cudaError_t launch_scale(float *C, int64_t ldc, int M, int N, float beta, cudaStream_t stream);

// ------------------------------------------------------- tensor-core path
// Shortest K piece (in K blocks) of a tail tile split among workers, and the
// most workers that can share the tail of one launch.
constexpr int kMinPieceBlocks = 4;
constexpr int kMaxTailUnits = 160;
struct TcArgs {
  CUtensorMap tmap_ab, tmap_as, tmap_bb, tmap_bs;  // K-major operand maps
  float *C;
  int64_t ldc;
  int M, N;
  int k_block0, k_blocks;  // k blocks (128 bytes of K each) of this launch
  int tiles_m, tiles_n, group_m;
  float alpha, beta;
  int vec_c;
  int promote_blocks;  // K blocks per TMEM partial sum before it is added into registers
  int sm_count;        // SMs of the device: the persistent grid size
  // testing only: 1 = skip the first operand load, 2 = never publish the flag of
  // the first in-kernel split item; either way a bounded wait then expires
  int withhold_first_load;
  // Split of the last, partial wave along K.  Tiles [0, full_tiles) are
  // computed whole, strided over the workers (CTAs, or CTA pairs).  The K
  // blocks of the remaining tiles, laid end to end, are dealt evenly to
  // workers 0 .. tail_units-1 (0 = no split): worker w's share runs from tail
  // tile tail_tile[w], K block tail_k[w] (tile counted from full_tiles, k in
  // [0, k_blocks)) to the start of worker w + 1's share; entry tail_units is
  // (tail tiles, 0).  A piece that starts at k = 0 owns its tile; a later
  // piece is the first piece of its worker w, writes its sum to partials slot
  // w (tile_m x BN floats), and each accumulator warp stores `epoch` into
  // flags[(w * 2 + cta rank) * 8 + warp - 2]; the owner adds the slots in K
  // order and stores C.
  int full_tiles, tail_units;
  int tail_tile[kMaxTailUnits + 1], tail_k[kMaxTailUnits + 1];
  int grid_units;  // CTAs (pairs) to launch; 0 = min(tiles, SMs (pairs))
  // 1: tmap_ab maps the caller's raw fp32 A (K x M extents, zero fill outside)
  // and the kernel splits it into tf32 big/small in shared memory; tmap_as is
  // unused.  0: both A maps point at the pre-split workspace.
  int a_inline;
  // CTA-pair kernels only.  1: clusters of two pairs computing tiles (tm, 2 tn)
  // and (tm, 2 tn + 1), which TMA-multicast their shared A panels: tiles_n
  // counts such tile pairs, the A maps have 64-row boxes, grid_units counts
  // clusters, and partials slots are per pair (slot 2 w + pair of worker w).
  int multicast;
  float *partials;
  unsigned *flags;
  unsigned epoch;
  int *err;
  // In-kernel panel split (CTA pairs, tf32 operands).  1: warps 10 and 11 of
  // every CTA split the caller's raw A (and B when split_b) into the
  // workspace buffers that the operand maps cover, while the GEMM runs: an
  // item is one 32-row slice of a 256-row A panel, or one 32-column slice of
  // a 256-column B panel (written transposed, K-major), over a K chunk of
  // kSplitChunkBlocks k blocks of this launch, padding written as zeros.
  // Items are claimed from the counter split_next[epoch - 1] in the order the
  // persistent tiles first need them (by wave, then K chunk); each publishes
  // `epoch` in its flag once its stores are visible:
  //   A: split_flags[(tm * KC + kc) * 8 + slice]
  //   B: split_flags[((tiles_m + tn) * KC + kc) * 8 + slice]
  // with KC = ceil(k_blocks / kSplitChunkBlocks).  A CTA's producer waits for
  // the four flags of its 128 rows of A and 128 rows of B (transposed) at
  // the start of every K chunk of a tile.  The host zeroes flags and counters
  // before each call.
  int split_inline, split_b;
  const float *A_raw, *B_raw;
  int64_t lda, ldb;
  int K;   // K of the whole problem: the raw operands' extent
  int kp;  // row length of the workspace operand buffers (K rounded up to 32)
  float *a_big, *a_small, *b_big, *b_small;
  int vec_a, vec_b;  // 16-byte loads of the raw operands allowed
  unsigned *split_flags;
  unsigned *split_next;
  // split_done[epoch - 1] counts the launch's published items; once it equals
  // their number, a producer stops waiting on flags for the rest of the launch
  unsigned *split_done;
  // Cluster Launch Control (CTA pairs of split TF32 without the shared-memory A
  // split or multicast).  1: the grid holds one pair per output tile; a
  // resident pair starts on its own tile and takes every further tile from
  // the hardware by cancelling the launch of a pair that has not started, so
  // tiles are dealt to pairs as they free up.  clc_units: the pairs that fit
  // on the device at once (the in-kernel split orders its items by their
  // waves).  clc_pieces P > 1: work items [0, full_tiles) are whole tiles,
  // and item full_tiles + j * P + q is K piece q (k blocks [q kb / P,
  // (q+1) kb / P)) of tile full_tiles + j.  Every piece leaves its partial sum
  // in partials slot j * P + q and counts itself in on the tile's counter
  // flags[(j * 2 + rank) * 8 + warp - 2]; the last to arrive adds the P slots
  // in order, stores C and resets the counter.  No piece waits for another.
  int clc, clc_units, clc_pieces;
  // Instrumentation (nullptr = off): thread 0 of CTA 0 adds the SM cycles
  // (clock64) and the nanoseconds (%globaltimer) of its CTA's lifetime to
  // clock_acc[0] and clock_acc[1], which gives the SM clock the kernel ran at;
  // with Cluster Launch Control every tile taken from a cancelled launch adds
  // one to clock_acc[2].
  unsigned long long *clock_acc;
};
// K blocks per item of the in-kernel panel split (256 of K).  Measured on
// GB300: items of 64 of K spent more time in their flag fences and round trips
// than they saved at the start (4096^3: 0.542 against 0.447 ms per call), and
// items of 128 of K still did (4096^3 0.455 against 0.433 ms, 8192^3 3.11
// against 3.04 ms).
constexpr int kSplitChunkBlocks = 8;
// Operand types of the tensor-core kernel: tf32 from fp32 containers (one or
// three passes), or pre-converted fp16 / bf16 (one pass, MMA kind::f16).
enum TcKind : int { kTcTf32 = 0, kTcF16 = 1, kTcBf16 = 2 };
// passes: 1 (tf32, fp16, bf16) or 3 (split tf32); bn: 128 or 256.  A k block
// is 128 bytes of K: 32 fp32 elements, or 64 fp16/bf16 elements, and k_block0
// and k_blocks count those.
cudaError_t launch_tc(const TcArgs &a, int passes, int bn, int stages, cudaStream_t stream,
                      int kind = kTcTf32);
int tc_max_stages(int passes, int bn);
// CTA-pair (cluster of 2, tcgen05 cta_group::2) variant: tiles_m counts
// 256-row pair tiles; bn: 256.
cudaError_t launch_tc_pair(const TcArgs &a, int passes, int bn, int stages, cudaStream_t stream,
                           int kind = kTcTf32);
int tc_pair_max_stages(int passes, int bn);
// Clusters of the multicast pair kernel (passes 1 or 3, bn 256, deepest ring)
// that can be resident at once on the current device; -1 if the query failed.
int tc_multicast_clusters(int passes, int bn, cudaStream_t stream);

// Frees the workspace cached for `stream` on the current device (stream-ordered);
// for code in this library that destroys a stream it created.
phobos_status_t release_stream_workspace(cudaStream_t stream);

}  // namespace phobos
