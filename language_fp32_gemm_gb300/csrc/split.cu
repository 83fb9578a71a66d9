// Operand pre-pass of the tensor-core path and the beta-scaling leaf.
//
// Split TF32: every fp32 operand value x is written as two tf32 values,
//   big = rna_tf32(x),  small = rna_tf32(x - big)
// (x - big is exact in fp32), so x = big + small up to 2^-22 |x|.  Both are
// stored as 32-bit containers whose low 13 bits are zero, in K-major buffers
// padded with zeros to whole tiles: A stays row-major [Mp][Kp], B is
// transposed to [Np][Kp].  Padded rows and the K tail are zero, so the main
// kernel never needs bounds checks on its operands and TMA boxes never leave
// the buffers.  The pages convert fp32 operands before the tensor cores too,
// and note the single conversion is lossy ("Show HN: Phobos", footnote 14);
// the two-term split recovers fp32-level products.
//
// 16-bit inputs ("Show HN: Phobos", "Side-quest: Cheating": cast to a 16-bit
// type before the tensor cores): the same two layouts hold one fp16 or bf16
// value per element, rounded to nearest with ties to even.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace phobos {

namespace {

__global__ void __launch_bounds__(256) split_rows_kernel(const float *__restrict__ A, int64_t lda,
                                                         int M, int K, int Mp, int Kp,
                                                         float *__restrict__ big,
                                                         float *__restrict__ small, int vec) {
  const int64_t groups_per_row = Kp / 4;
  const int64_t total = static_cast<int64_t>(Mp) * groups_per_row;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(g / groups_per_row);
    const int k = static_cast<int>(g - static_cast<int64_t>(i) * groups_per_row) * 4;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (i < M) {
      const float *src = A + static_cast<int64_t>(i) * lda + k;
      if (vec && k + 3 < K) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (k + t < K) x[t] = __ldg(src + t);
      }
    }
    float4 b, s;
    b.x = tf32_rna_bits(x[0]); s.x = tf32_rna_bits(x[0] - b.x);
    b.y = tf32_rna_bits(x[1]); s.y = tf32_rna_bits(x[1] - b.y);
    b.z = tf32_rna_bits(x[2]); s.z = tf32_rna_bits(x[2] - b.z);
    b.w = tf32_rna_bits(x[3]); s.w = tf32_rna_bits(x[3] - b.w);
    const int64_t o = static_cast<int64_t>(i) * Kp + k;
    *reinterpret_cast<float4 *>(big + o) = b;
    if (small) *reinterpret_cast<float4 *>(small + o) = s;
  }
}

// B (K x N) -> K-major [Np][Kp] through a 32 x 32 shared-memory tile.
__global__ void __launch_bounds__(256) split_cols_kernel(const float *__restrict__ B, int64_t ldb,
                                                         int K, int N, int Kp,
                                                         float *__restrict__ big,
                                                         float *__restrict__ small) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32;
  const int n0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;  // 0..7
#pragma unroll
  for (int r = 0; r < 32; r += 8) {
    const int k = k0 + ty + r;
    const int n = n0 + tx;
    tile[ty + r][tx] = (k < K && n < N) ? __ldg(B + static_cast<int64_t>(k) * ldb + n) : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 32; r += 8) {
    const int n = n0 + ty + r;
    const int k = k0 + tx;
    const float x = tile[tx][ty + r];
    const float b = tf32_rna_bits(x);
    const int64_t o = static_cast<int64_t>(n) * Kp + k;
    big[o] = b;
    if (small) small[o] = tf32_rna_bits(x - b);
  }
}

// The whole split-TF32 pre-pass in one launch: blocks [0, a_blocks) split A
// row by row (a grid-stride loop over A's float4 groups, as split_rows_kernel),
// the next b_tiles_k * b_tiles_n blocks each split and transpose one 32 x 32
// tile of B (as split_cols_kernel), and every thread also zeroes its share of
// the tail-split flags.  One launch instead of a flag memset and two kernels
// saves their launch gaps on the stream.
__global__ void __launch_bounds__(256) split_ab_kernel(const SplitArgs a) {
  __shared__ float tile[32][33];
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < a.n_flags;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    a.flags[i] = 0u;
  if (static_cast<int>(blockIdx.x) < a.a_blocks) {
    const int64_t groups_per_row = a.Kp / 4;
    const int64_t total = static_cast<int64_t>(a.Mp) * groups_per_row;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(a.a_blocks) * blockDim.x) {
      const int i = static_cast<int>(g / groups_per_row);
      const int k = static_cast<int>(g - static_cast<int64_t>(i) * groups_per_row) * 4;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (i < a.M) {
        const float *src = a.A + static_cast<int64_t>(i) * a.lda + k;
        if (a.vec_a && k + 3 < a.K) {
          const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
          x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (k + t < a.K) x[t] = __ldg(src + t);
        }
      }
      float4 b, s;
      b.x = tf32_rna_bits(x[0]); s.x = tf32_rna_bits(x[0] - b.x);
      b.y = tf32_rna_bits(x[1]); s.y = tf32_rna_bits(x[1] - b.y);
      b.z = tf32_rna_bits(x[2]); s.z = tf32_rna_bits(x[2] - b.z);
      b.w = tf32_rna_bits(x[3]); s.w = tf32_rna_bits(x[3] - b.w);
      const int64_t o = static_cast<int64_t>(i) * a.Kp + k;
      *reinterpret_cast<float4 *>(a.a_big + o) = b;
      if (a.a_small) *reinterpret_cast<float4 *>(a.a_small + o) = s;
    }
    return;
  }
  const int t = static_cast<int>(blockIdx.x) - a.a_blocks;
  if (t >= a.b_tiles_k * a.b_tiles_n) return;
  const int k0 = (t % a.b_tiles_k) * 32;
  const int n0 = (t / a.b_tiles_k) * 32;
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;  // 0..7
#pragma unroll
  for (int r = 0; r < 32; r += 8) {
    const int k = k0 + ty + r;
    const int n = n0 + tx;
    tile[ty + r][tx] = (k < a.K && n < a.N) ? __ldg(a.B + static_cast<int64_t>(k) * a.ldb + n) : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 32; r += 8) {
    const int n = n0 + ty + r;
    const int k = k0 + tx;
    const float x = tile[tx][ty + r];
    const float b = tf32_rna_bits(x);
    const int64_t o = static_cast<int64_t>(n) * a.Kp + k;
    a.b_big[o] = b;
    if (a.b_small) a.b_small[o] = tf32_rna_bits(x - b);
  }
}

template <bool BF16>
__device__ __forceinline__ unsigned short to_16bit(float x) {
  if (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  return __half_as_ushort(__float2half_rn(x));
}

// A (M x K) -> [Mp][Kp] 16-bit, four elements (8 bytes) per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) convert_rows_kernel(const float *__restrict__ A, int64_t lda,
                                                           int M, int K, int Mp, int Kp,
                                                           unsigned short *__restrict__ out, int vec) {
  const int64_t groups_per_row = Kp / 4;
  const int64_t total = static_cast<int64_t>(Mp) * groups_per_row;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(g / groups_per_row);
    const int k = static_cast<int>(g - static_cast<int64_t>(i) * groups_per_row) * 4;
    float x[4] = {0.f, 0.f, 0.f, 0.f};
    if (i < M) {
      const float *src = A + static_cast<int64_t>(i) * lda + k;
      if (vec && k + 3 < K) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t)
          if (k + t < K) x[t] = __ldg(src + t);
      }
    }
    uint2 w;
    w.x = static_cast<uint32_t>(to_16bit<BF16>(x[0])) | (static_cast<uint32_t>(to_16bit<BF16>(x[1])) << 16);
    w.y = static_cast<uint32_t>(to_16bit<BF16>(x[2])) | (static_cast<uint32_t>(to_16bit<BF16>(x[3])) << 16);
    *reinterpret_cast<uint2 *>(out + static_cast<int64_t>(i) * Kp + k) = w;
  }
}

// B (K x N) -> K-major [Np][Kp] 16-bit through a 32 x 32 shared-memory tile.
template <bool BF16>
__global__ void __launch_bounds__(256) convert_cols_kernel(const float *__restrict__ B, int64_t ldb,
                                                           int K, int N, int Kp,
                                                           unsigned short *__restrict__ out) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32;
  const int n0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;  // 0..7
#pragma unroll
  for (int r = 0; r < 32; r += 8) {
    const int k = k0 + ty + r;
    const int n = n0 + tx;
    tile[ty + r][tx] = (k < K && n < N) ? __ldg(B + static_cast<int64_t>(k) * ldb + n) : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < 32; r += 8) {
    const int n = n0 + ty + r;
    const int k = k0 + tx;
    out[static_cast<int64_t>(n) * Kp + k] = to_16bit<BF16>(tile[tx][ty + r]);
  }
}

__global__ void __launch_bounds__(256) scale_kernel(float *C, int64_t ldc, int M, int N,
                                                    float beta) {
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = e / N;
    const int64_t j = e - i * N;
    float *c = C + i * ldc + j;
    *c = beta == 0.0f ? 0.0f : beta * *c;
  }
}

unsigned grid_for(int64_t work, int per_block) {
  int64_t blocks = (work + per_block - 1) / per_block;
  // enough blocks to fill every SM several times; the kernels stride the rest
  const int64_t cap = 152 * 32;
  if (blocks > cap) blocks = cap;
  return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_split_rows(const float *A, int64_t lda, int M, int K, int Mp, int Kp,
                              float *big, float *small, int vec, cudaStream_t stream) {
  const int64_t groups = static_cast<int64_t>(Mp) * (Kp / 4);
  split_rows_kernel<<<grid_for(groups, 256), 256, 0, stream>>>(A, lda, M, K, Mp, Kp, big, small,
                                                               vec);
  return cudaGetLastError();
}

cudaError_t launch_split_cols(const float *B, int64_t ldb, int K, int N, int Np, int Kp,
                              float *big, float *small, cudaStream_t stream) {
  dim3 grid(Kp / 32, Np / 32);
  split_cols_kernel<<<grid, 256, 0, stream>>>(B, ldb, K, N, Kp, big, small);
  return cudaGetLastError();
}

cudaError_t launch_split_ab(SplitArgs a, int split_a, int split_b, cudaStream_t stream) {
  a.a_blocks = split_a ? static_cast<int>(grid_for(static_cast<int64_t>(a.Mp) * (a.Kp / 4), 256)) : 0;
  a.b_tiles_k = split_b ? a.Kp / 32 : 0;
  a.b_tiles_n = split_b ? a.Np / 32 : 0;
  const int64_t blocks = a.a_blocks + static_cast<int64_t>(a.b_tiles_k) * a.b_tiles_n;
  const int64_t flag_blocks = (a.n_flags + 255) / 256;
  const int64_t grid = blocks > flag_blocks ? blocks : flag_blocks;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  split_ab_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_convert_rows(const float *A, int64_t lda, int M, int K, int Mp, int Kp,
                                void *out, int bf16, cudaStream_t stream) {
  const int64_t groups = static_cast<int64_t>(Mp) * (Kp / 4);
  const int vec = (lda % 4 == 0) && (reinterpret_cast<uintptr_t>(A) & 15u) == 0;
  unsigned short *o = static_cast<unsigned short *>(out);
  if (bf16)
    convert_rows_kernel<true><<<grid_for(groups, 256), 256, 0, stream>>>(A, lda, M, K, Mp, Kp, o, vec);
  else
    convert_rows_kernel<false><<<grid_for(groups, 256), 256, 0, stream>>>(A, lda, M, K, Mp, Kp, o, vec);
  return cudaGetLastError();
}

cudaError_t launch_convert_cols(const float *B, int64_t ldb, int K, int N, int Np, int Kp,
                                void *out, int bf16, cudaStream_t stream) {
  dim3 grid(Kp / 32, Np / 32);
  unsigned short *o = static_cast<unsigned short *>(out);
  if (bf16)
    convert_cols_kernel<true><<<grid, 256, 0, stream>>>(B, ldb, K, N, Kp, o);
  else
    convert_cols_kernel<false><<<grid, 256, 0, stream>>>(B, ldb, K, N, Kp, o);
  return cudaGetLastError();
}

cudaError_t launch_scale(float *C, int64_t ldc, int M, int N, float beta, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(M) * N;
  scale_kernel<<<grid_for(total, 256), 256, 0, stream>>>(C, ldc, M, N, beta);
  return cudaGetLastError();
}

}  // namespace phobos
