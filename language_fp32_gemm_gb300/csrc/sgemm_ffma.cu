// Register-tiled fp32 SGEMM on the CUDA cores (fused multiply-add), for small
// problems and for callers who ask for plain fp32 products.
//
// This is the pages' own fp32 path ("Show HN: Phobos", "GPU Performance"):
// coalesced global loads, a shared-memory tile per CTA, a per-thread register
// micro-tile (8 x 8 outputs) read from shared memory without bank conflicts,
// and ping-pong buffering of the K tiles ("Are we cuBLAS yet?": ping-pong
// buffering and pipelining).  The CTA tile is 128 x 128 x 16 (256 threads) or
// 64 x 64 x 16 (64 threads); the pages' tuned winner on their GPU was
// 64 x 128 x 8.  With the fragments of the next k step loaded during the
// current one, 16-deep K tiles measured 1 % faster than 8-deep ones.  Any M, N, K and leading dimension is accepted: loads outside
// the matrix read zero and stores outside it are skipped.
//
// Small problems, with fewer tiles than SMs, split K across the CTAs of a
// thread-block cluster (up to 8): each CTA sums its K slice, leaves the
// partial tile in its shared memory, and the cluster's rank 0 adds the other
// ranks' tiles through distributed shared memory, in rank order
// (deterministic), before the epilogue.  This is the cluster-level reduction
// of the "Clusters et DSMEM" chapter, section 3.4 (reduce inside the cluster
// instead of one atomic per block).
#include "internal.h"
#include "ptx.cuh"

namespace phobos {

namespace {

constexpr int kBK = 16;

template <int BM, int BN, bool KSPLIT>
__global__ void __launch_bounds__((BM / 8) * (BN / 8), BM == 128 ? 2 : 1)
    sgemm_ffma_kernel(const FfmaArgs p) {
  constexpr int NT = (BM / 8) * (BN / 8);
  constexpr int PAD = 4;
  constexpr int A_LOADS = BM * kBK / 4 / NT;  // float4 groups of A per thread
  constexpr int B_LOADS = BN * kBK / 4 / NT;  // float4 groups of B per thread
  static_assert(A_LOADS >= 1 && B_LOADS >= 1, "tile too small for the thread count");
  __shared__ __align__(16) float As[2][kBK][BM + PAD];
  __shared__ __align__(16) float Bs[2][kBK][BN + PAD];

  const int tid = threadIdx.x;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int slice = KSPLIT ? static_cast<int>(cluster_ctarank()) : 0;
  const int tile = KSPLIT ? static_cast<int>(blockIdx.x) / p.kslices : static_cast<int>(blockIdx.x);
  const int tm = tile / tiles_n;
  const int tn = tile - tm * tiles_n;
  // this CTA's K range (slices are whole multiples of kBK)
  int k_lo = p.k_begin, k_hi = p.k_begin + p.k_len;
  if (KSPLIT) {
    const int per = ((p.k_len + p.kslices - 1) / p.kslices + kBK - 1) / kBK * kBK;
    k_lo = min(p.k_begin + slice * per, k_hi);
    k_hi = min(k_lo + per, k_hi);
  }
  const int m0 = tm * BM, n0 = tn * BN;
  const int tx = tid % (BN / 8);
  const int ty = tid / (BN / 8);

  float a_reg[A_LOADS][4];
  float b_reg[B_LOADS][4];

  // Tiles wholly inside the matrix (the common case) load without the
  // per-element bounds checks.
  const bool a_rows_in = p.vec_a && m0 + BM <= p.M;
  const bool b_cols_in = p.vec_b && n0 + BN <= p.N;
  auto load_tiles = [&](int k0) {
    if (k0 + kBK <= k_hi && a_rows_in && b_cols_in) {
#pragma unroll
      for (int l = 0; l < A_LOADS; ++l) {
        const int g = tid + l * NT;
        const float4 v = __ldg(reinterpret_cast<const float4 *>(
            p.A + static_cast<int64_t>(m0 + g / (kBK / 4)) * p.lda + k0 + (g % (kBK / 4)) * 4));
        a_reg[l][0] = v.x; a_reg[l][1] = v.y; a_reg[l][2] = v.z; a_reg[l][3] = v.w;
      }
#pragma unroll
      for (int l = 0; l < B_LOADS; ++l) {
        const int g = tid + l * NT;
        const float4 v = __ldg(reinterpret_cast<const float4 *>(
            p.B + static_cast<int64_t>(k0 + g / (BN / 4)) * p.ldb + n0 + (g % (BN / 4)) * 4));
        b_reg[l][0] = v.x; b_reg[l][1] = v.y; b_reg[l][2] = v.z; b_reg[l][3] = v.w;
      }
      return;
    }
#pragma unroll
    for (int l = 0; l < A_LOADS; ++l) {
      const int g = tid + l * NT;       // group index in the BM x 8 tile
      const int row = g / (kBK / 4);
      const int kq = (g % (kBK / 4)) * 4;
      const int gi = m0 + row, gk = k0 + kq;
      const float *src = p.A + static_cast<int64_t>(gi) * p.lda + gk;
      if (gi < p.M && p.vec_a && gk + 3 < k_hi) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
        a_reg[l][0] = v.x; a_reg[l][1] = v.y; a_reg[l][2] = v.z; a_reg[l][3] = v.w;
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t)
          a_reg[l][t] = (gi < p.M && gk + t < k_hi) ? __ldg(src + t) : 0.f;
      }
    }
#pragma unroll
    for (int l = 0; l < B_LOADS; ++l) {
      const int g = tid + l * NT;       // group index in the 8 x BN tile
      const int k = g / (BN / 4);
      const int nq = (g % (BN / 4)) * 4;
      const int gk = k0 + k, gj = n0 + nq;
      const float *src = p.B + static_cast<int64_t>(gk) * p.ldb + gj;
      const bool krow = gk < k_hi;
      if (krow && p.vec_b && gj + 3 < p.N) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
        b_reg[l][0] = v.x; b_reg[l][1] = v.y; b_reg[l][2] = v.z; b_reg[l][3] = v.w;
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) b_reg[l][t] = (krow && gj + t < p.N) ? __ldg(src + t) : 0.f;
      }
    }
  };

  auto store_tiles = [&](int buf) {
#pragma unroll
    for (int l = 0; l < A_LOADS; ++l) {
      const int g = tid + l * NT;
      const int row = g / (kBK / 4);
      const int kq = (g % (kBK / 4)) * 4;
#pragma unroll
      for (int t = 0; t < 4; ++t) As[buf][kq + t][row] = a_reg[l][t];
    }
#pragma unroll
    for (int l = 0; l < B_LOADS; ++l) {
      const int g = tid + l * NT;
      const int k = g / (BN / 4);
      const int nq = (g % (BN / 4)) * 4;
      *reinterpret_cast<float4 *>(&Bs[buf][k][nq]) =
          make_float4(b_reg[l][0], b_reg[l][1], b_reg[l][2], b_reg[l][3]);
    }
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  const int k_end = k_hi;
  int buf = 0;
  load_tiles(k_lo);
  store_tiles(0);
  __syncthreads();
  // The fragments of step k + 1 are read from shared memory while step k's
  // FMAs run, so the FMAs do not wait on the shared-memory latency (which
  // was the kernel's main stall).
  float4 fa[2][2], fb[2][2];
  auto load_frag = [&](int b, int k, int slot) {
    fa[slot][0] = *reinterpret_cast<const float4 *>(&As[b][k][ty * 4]);
    fa[slot][1] = *reinterpret_cast<const float4 *>(&As[b][k][ty * 4 + BM / 2]);
    fb[slot][0] = *reinterpret_cast<const float4 *>(&Bs[b][k][tx * 4]);
    fb[slot][1] = *reinterpret_cast<const float4 *>(&Bs[b][k][tx * 4 + BN / 2]);
  };
  for (int k0 = k_lo; k0 < k_end; k0 += kBK) {
    const bool more = k0 + kBK < k_end;
    if (more) load_tiles(k0 + kBK);  // global loads in flight during the FMAs
    load_frag(buf, 0, 0);
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      if (k + 1 < kBK) load_frag(buf, k + 1, (k + 1) & 1);
      const float4 a0 = fa[k & 1][0], a1 = fa[k & 1][1];
      const float4 b0 = fb[k & 1][0], b1 = fb[k & 1][1];
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
      // column-outer order measured 1-2 % faster than row-outer
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) {
      store_tiles(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
  }

  if (KSPLIT) {
    // Cluster reduction of the K slices through distributed shared memory.
    // Every rank reduces its own share of the tile's rows: it reads that
    // share from every rank's partial tile (its own included), adds the
    // slices in rank order (deterministic), and stores those rows of C.
    __shared__ __align__(16) float part[BM * BN];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4);
#pragma unroll
      for (int h = 0; h < 2; ++h)
        *reinterpret_cast<float4 *>(&part[r * BN + tx * 4 + h * (BN / 2)]) =
            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
    }
    cluster_sync();  // every slice's partial tile is in place
    const int rows_per = (BM + p.kslices - 1) / p.kslices;
    const int r_lo = slice * rows_per;
    const int r_hi = min(BM, r_lo + rows_per);
    constexpr int kVecPerRow = BN / 4;
#pragma unroll 1
    for (int e = r_lo * kVecPerRow + tid; e < r_hi * kVecPerRow; e += NT) {
      const int r = e / kVecPerRow, c = (e - r * kVecPerRow) * 4;
      const uint32_t local = smem_u32(&part[r * BN + c]);
      float4 v[8];
#pragma unroll
      for (int rk = 0; rk < 8; ++rk)
        if (rk < p.kslices) v[rk] = ld_shared_cluster_v4(mapa_shared(local, rk));
      float4 t = v[0];
#pragma unroll
      for (int rk = 1; rk < 8; ++rk)
        if (rk < p.kslices) {
          t.x += v[rk].x;
          t.y += v[rk].y;
          t.z += v[rk].z;
          t.w += v[rk].w;
        }
      const int row = m0 + r, col = n0 + c;
      if (row < p.M) {
        float *crow = p.C + static_cast<int64_t>(row) * p.ldc;
        const float tv[4] = {t.x, t.y, t.z, t.w};
        if (p.vec_c && col + 3 < p.N) {
          float4 *dst = reinterpret_cast<float4 *>(crow + col);
          float4 o;
          if (p.beta != 0.0f) {
            const float4 old = *dst;
            o.x = fmaf(p.alpha, tv[0], p.beta * old.x);
            o.y = fmaf(p.alpha, tv[1], p.beta * old.y);
            o.z = fmaf(p.alpha, tv[2], p.beta * old.z);
            o.w = fmaf(p.alpha, tv[3], p.beta * old.w);
          } else {
            o.x = p.alpha * tv[0];
            o.y = p.alpha * tv[1];
            o.z = p.alpha * tv[2];
            o.w = p.alpha * tv[3];
          }
          *dst = o;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (col + q < p.N)
              crow[col + q] = p.beta != 0.0f ? fmaf(p.alpha, tv[q], p.beta * crow[col + q])
                                             : p.alpha * tv[q];
        }
      }
    }
    cluster_sync();  // the peers' shared memory stays valid until every rank has read it
    return;
  }

  // Epilogue: C = alpha * acc + beta * C_old; beta == 0 does not read C.
  // Old C of all the thread's rows is loaded before any store: a store could
  // alias a later load as far as the compiler knows, which would otherwise
  // serialise one memory round trip per row.  The 128-row tile (two CTAs per
  // SM, fewer registers) does it half a micro-tile at a time.
  constexpr int kHalfRows = BM == 128 ? 4 : 8;
#pragma unroll
  for (int i0 = 0; i0 < 8; i0 += kHalfRows) {
    float4 old[kHalfRows][2];
    if (p.beta != 0.0f) {
#pragma unroll
      for (int i = i0; i < i0 + kHalfRows; ++i) {
        const int row = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
        const float *crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int col = n0 + tx * 4 + h * (BN / 2);
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (row < p.M) {
            if (p.vec_c && col + 3 < p.N) {
              o = *reinterpret_cast<const float4 *>(crow + col);
            } else {
              if (col + 0 < p.N) o.x = crow[col + 0];
              if (col + 1 < p.N) o.y = crow[col + 1];
              if (col + 2 < p.N) o.z = crow[col + 2];
              if (col + 3 < p.N) o.w = crow[col + 3];
            }
          }
          old[i - i0][h] = o;
        }
      }
    }
#pragma unroll
    for (int i = i0; i < i0 + kHalfRows; ++i) {
      const int row = m0 + (i < 4 ? ty * 4 + i : BM / 2 + ty * 4 + (i - 4));
      if (row >= p.M) continue;
      float *crow = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = n0 + tx * 4 + h * (BN / 2);
        const float4 od = old[i - i0][h];
        const float oldv[4] = {od.x, od.y, od.z, od.w};
        float o[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          o[t] = p.beta != 0.0f ? fmaf(p.alpha, acc[i][4 * h + t], p.beta * oldv[t])
                                : p.alpha * acc[i][4 * h + t];
        if (p.vec_c && col + 3 < p.N) {
          *reinterpret_cast<float4 *>(crow + col) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (col + t < p.N) crow[col + t] = o[t];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_ffma(const FfmaArgs &a, cudaStream_t stream) {
  if (a.tile == 128) {
    const int64_t tiles = static_cast<int64_t>((a.M + 127) / 128) * ((a.N + 127) / 128);
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    sgemm_ffma_kernel<128, 128, false><<<static_cast<unsigned>(tiles), 256, 0, stream>>>(a);
  } else if (a.tile == 64) {
    const int64_t tiles = static_cast<int64_t>((a.M + 63) / 64) * ((a.N + 63) / 64);
    if (a.kslices > 1) {
      if (a.kslices > 8 || tiles * a.kslices > 0x7fffffff) return cudaErrorInvalidValue;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(tiles * a.kslices), 1, 1);
      cfg.blockDim = dim3(64, 1, 1);
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(a.kslices);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, sgemm_ffma_kernel<64, 64, true>, a);
    }
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    sgemm_ffma_kernel<64, 64, false><<<static_cast<unsigned>(tiles), 64, 0, stream>>>(a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace phobos
