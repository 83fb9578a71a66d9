// Host-side rules shared by the entry points (phobos_gemm.cu, noalloc.cu):
// size limits and the split-TF32 partial length.  No kernel includes this
// header.  Not installed; not part of the ABI.
#pragma once

#include <cstdint>

namespace phobos {

// Largest M, N or K a call accepts: the kernels index rows and columns with
// 32-bit ints.
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1024;

// K blocks (of 32) summed in TMEM before the partial sum is added into fp32
// registers with round-to-nearest adds, for split TF32; every entry point that
// runs the split-TF32 kernel takes its partial length from here.  The
// truncation error of one partial is largest relative to sum|a||b| when the
// whole K spans few partials.  Measured on GB300 (max over 4 M outputs, normal
// data, bar 2^-20 = 9.5e-7):
//   partials of 8 blocks: 1.07e-6 at K = 256, 4.9e-7 at K = 1024, 2.4e-7 at K = 4096
//   partials of 4 blocks: 8.9e-7 at K = 128, 5.6e-7 at K = 256, 2.5e-7 at K = 1024
//   partials of 2 blocks: 6.9e-7 at K = 64, 3.2e-7 at K = 256, 1.9e-7 at K = 512
//   partials of 1 block:  3.7e-7 at K = 64, 2.4e-7 at K = 128
// while shorter partials cost speed (8192^3: 367, 355, 322, 204 TFLOP/s).  So
// the length follows K, keeping every case at 5e-7 or below.  Two partials
// are also the slack the next tile's MMAs have while the accumulator warps
// store a tile, so above K = 1024 the longer partials are used: 8 blocks
// measured 4.7e-7 at K = 1025, 3.3e-7 at K = 2000 (2 M outputs each).
inline int promote_blocks_for(int64_t k) {
  if (k <= 128) return 1;
  if (k <= 512) return 2;
  if (k <= 1024) return 4;
  return 8;
}

// Device address of the no-allocation entry point's status word on device
// `dev` (noalloc.cu), or null before that entry point first ran there.
int *noalloc_status_word(int dev);

}  // namespace phobos
