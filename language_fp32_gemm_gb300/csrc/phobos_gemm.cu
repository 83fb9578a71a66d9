// C ABI of libphobos_gemm: argument checks, the planner, workspace handling
// and dispatch to the FFMA and tensor-core kernels.  See include/phobos_gemm.h
// for the contract of every entry point.
#include "../../include/phobos_gemm.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "host_rules.h"
#include "internal.h"

namespace phobos {
namespace {

constexpr int kTcBK = 32;
constexpr int kTcBM = 128;
constexpr int64_t kFfmaMacLimit = int64_t{1} << 25;     // DEFAULT: FFMA up to 32 Mi MACs
constexpr int64_t kDefaultSuper = 4096;                 // super-tile edge (raster group)
// Single TF32 (bound 2^-10) promotes every K = 1024.
constexpr int kTf32PromoteBlocks = 32;
// fp16 / bf16 inputs promote every 8 blocks of 64 (K = 512): a partial's
// truncating fp32 accumulation then stays within 512 * 2^-23 = 2^-14 of
// sum|a||b|, far inside the inputs' own rounding (2^-11, 2^-8).
constexpr int kHalfPromoteBlocks = 8;

bool half_path(int path) { return path == PHOBOS_PATH_FP16 || path == PHOBOS_PATH_BF16; }
// K elements in one 128-byte k block of a tensor-core path.
int tc_bk(int path) { return half_path(path) ? 2 * kTcBK : kTcBK; }
int tc_elem_bytes(int path) { return half_path(path) ? 2 : 4; }
int tc_kind(int path) {
  return path == PHOBOS_PATH_FP16 ? kTcF16 : path == PHOBOS_PATH_BF16 ? kTcBf16 : kTcTf32;
}
// Tail split: at most this many K pieces per tile, each at least this many K blocks.
constexpr int kMaxTailSplit = 8;
// Workers (CTAs or CTA pairs) that share the `tail` tiles of the last, partial
// wave, each taking an even share of the tail's K blocks (0 = no split).
// split: the plan's tail_split (0 = automatic, 1 = off, S = S pieces per tile
// when S workers per tail tile are free, else an even share for every worker).
// S is capped so that a share spans at least kMinPieceBlocks.  With more
// workers than tail tiles a share is shorter than a tile; moving its ends onto
// tile boundaries (the kernel does that for pieces shorter than
// kMinPieceBlocks) lengthens it by less than 2 * kMinPieceBlocks <= one tile,
// so a share never reaches into a third tile.
int tail_workers(int split, int tail, int units, int k_blocks) {
  if (split == 1 || tail == 0) return 0;
  int S = split;
  if (split == 0) {
    // S pieces per tile shorten the tail from k_blocks to about k_blocks / S
    // blocks of MMA work, and each piece after the first costs its owner about
    // 2.5 blocks' time to add (1.6 to 2.3 us measured on GB300, a block being
    // 0.8 us): k_blocks / S + 2.5 * (S - 1) is least at S = sqrt(k_blocks / 2.5).
    S = static_cast<int>(std::lround(std::sqrt(k_blocks / 2.5)));
    if (S > kMaxTailSplit) S = kMaxTailSplit;
    // Whole pieces: every tail tile is then cut at the same K offsets, so
    // tiles that share an A or B panel read it at the same time, as whole
    // tiles do.  Even shares across tile boundaries put concurrent pieces at
    // different K offsets: on a 1024 x 8192 x 8192 band the tail then read its
    // B panels from DRAM again and the kernel took 500 us instead of 438 us.
    // With short K that costs less than leaving SMs idle: when whole pieces
    // would leave a fifth of the workers idle and K is at most 128 blocks,
    // one more piece per tile deals the tail evenly to every worker.
    // Measured on GB300 (main kernel, 28 tail tiles over 76 pairs, 128 K
    // blocks): 4096^3 390 us instead of 404 (beta 0) and 405 instead of 416
    // (beta 1), 65536 x 256 x 4096 441 instead of 472.  With 256 K blocks
    // (8192^3, 36 tail tiles) the even shares were no faster.
    const int whole = units / tail;
    if (S > whole) {
      const bool idle_fifth = static_cast<int64_t>(tail) * whole * 5 <= static_cast<int64_t>(units) * 4;
      S = (k_blocks <= 128 && idle_fifth) ? whole + 1 : whole;
    }
  }
  if (S > k_blocks / kMinPieceBlocks) S = k_blocks / kMinPieceBlocks;
  if (S < 2) return 0;
  int64_t w = static_cast<int64_t>(tail) * S < units ? static_cast<int64_t>(tail) * S : units;
  if (w > kMaxTailUnits) w = kMaxTailUnits;
  return w > tail ? static_cast<int>(w) : 0;
}

// Worker w's share of the tail starts at K block floor(w * T / tail_units) of
// the T = tail * k_blocks blocks of the tail tiles laid end to end; a start
// closer than kMinPieceBlocks to a tile boundary moves onto it (a monotone
// map, so shares stay ordered).  Every piece then spans at least
// kMinPieceBlocks, or a whole tile.  Two starts can land on the same boundary
// when shares are short; the kernel wants no empty share (the later pieces of
// a tile are then consecutive workers), so fewer workers are used until none
// is empty.  Returns the number of workers (0 = no split).
int fill_tail_shares(TcArgs &t, int tail, int workers) {
  const int64_t kb = t.k_blocks, total = static_cast<int64_t>(tail) * kb;
  for (; workers > tail; --workers) {
    bool empty = false;
    for (int w = 0; w <= workers; ++w) {
      int64_t s = total * w / workers;
      const int64_t r = s % kb;
      if (r != 0 && r < kMinPieceBlocks) s -= r;
      else if (r != 0 && kb - r < kMinPieceBlocks) s += kb - r;
      t.tail_tile[w] = static_cast<int>(s / kb);
      t.tail_k[w] = static_cast<int>(s % kb);
      if (w > 0 && t.tail_tile[w] == t.tail_tile[w - 1] && t.tail_k[w] == t.tail_k[w - 1])
        empty = true;
    }
    if (!empty) return workers;
  }
  return 0;
}

constexpr int kEpiWarps = 8;  // accumulator warps of the tensor-core kernel (one flag each)
// Automatic a_split: split A inside the kernel up to this N.  A pre-pass over
// A costs about 6 * (TF32/3 rate) / (N * HBM bandwidth) of the GEMM time,
// ~300/N on GB300; splitting inside the kernel slows the main loop by about
// 15-20 % (the converter warps' share of the SM), measured on GB300 at
// M = 16384, K = 4096.  They cross between N = 1536 and N = 2048.
constexpr int64_t kInlineSplitMaxN = 1536;

std::mutex g_mutex;       // planner caches, device state, workspaces
std::mutex g_host_mutex;  // serialises the host-buffer entry point (shared staging)

struct DeviceState {
  bool checked = false;
  bool supported = false;
  int sm_count = 0;
  int *err = nullptr;  // device status word
  // SM cycles, nanoseconds and tiles taken from cancelled launches, summed by
  // the tensor-core kernels while timing events are set (allocated on first use)
  unsigned long long *clock_acc = nullptr;
  // resident clusters of the multicast pair kernel, one pass / three passes
  // (0 = not queried yet)
  int mc_clusters[2] = {0, 0};
};
std::map<int, DeviceState> g_devices;

struct Buffer {
  void *ptr = nullptr;
  size_t bytes = 0;
};
// workspace per (device, stream)
std::map<std::pair<int, uintptr_t>, Buffer> g_workspaces;
// staging buffers of the host-pointer entry point, per device
struct Staging {
  Buffer a, b, c;
};
std::map<int, Staging> g_staging;
// Copy streams and events of the host-buffer entry point, per device.
constexpr int kMaxBands = 8;
constexpr int kMaxBChunks = 8;  // K chunks of B for the first band (see phobos_sgemm_host)
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t ev[2 * kMaxBands + 2 + kMaxBChunks] = {};
  bool ready = false;
};
std::map<int, HostPipe> g_pipes;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

std::atomic<uint64_t> g_launches{0};
cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;  // instrumentation

cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

cudaError_t mark(cudaEvent_t ev, cudaStream_t stream) {
  return ev ? cudaEventRecord(ev, stream) : cudaSuccess;
}

bool env_flag(const char *name) {
  const char *v = std::getenv(name);
  return v && v[0] && std::strcmp(v, "0") != 0;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

phobos_status_t device_state(DeviceState **out, int *dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PHOBOS_ERR_CUDA;
  DeviceState &st = g_devices[dev];
  if (!st.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    st.supported = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    st.checked = true;
  }
  if (!st.supported) return PHOBOS_ERR_UNSUPPORTED;
  if (!st.err) {
    if (cudaMalloc(&st.err, sizeof(int)) != cudaSuccess) return PHOBOS_ERR_OUT_OF_MEMORY;
    if (cudaMemset(st.err, 0, sizeof(int)) != cudaSuccess) return PHOBOS_ERR_CUDA;
  }
  *out = &st;
  if (dev_out) *dev_out = dev;
  return PHOBOS_OK;
}

phobos_status_t ensure_buffer(Buffer &b, size_t bytes, cudaStream_t stream) {
  if (b.bytes >= bytes && b.ptr) return PHOBOS_OK;
  if (b.ptr) {
    // stream-ordered: work already enqueued on `stream` keeps the old buffer
    if (cudaFreeAsync(b.ptr, stream) != cudaSuccess) return PHOBOS_ERR_CUDA;
    b.ptr = nullptr;
    b.bytes = 0;
  }
  void *p = nullptr;
  if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return PHOBOS_ERR_OUT_OF_MEMORY;
  }
  b.ptr = p;
  b.bytes = bytes;
  return PHOBOS_OK;
}

}  // namespace

// The workspace cached for `stream` on the current device, released
// stream-ordered: for callers that are about to destroy a stream they made.
phobos_status_t release_stream_workspace(cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PHOBOS_ERR_CUDA;
  auto it = g_workspaces.find({device, reinterpret_cast<uintptr_t>(stream)});
  if (it == g_workspaces.end()) return PHOBOS_OK;
  phobos_status_t st = PHOBOS_OK;
  if (it->second.ptr && cudaFreeAsync(it->second.ptr, stream) != cudaSuccess) st = PHOBOS_ERR_CUDA;
  g_workspaces.erase(it);
  return st;
}

namespace {

phobos_status_t get_encoder() {
  if (g_encode) return PHOBOS_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return PHOBOS_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PHOBOS_OK;
}

// Tensor map of a K-major buffer [rows][kp] of the kernel's operand type
// (fp32 containers for tf32, or fp16 / bf16): boxes of one 128-byte k block
// x box_rows, 128B swizzle.
phobos_status_t make_kmajor_map(CUtensorMap *map, const void *base, int64_t rows, int64_t kp,
                                int box_rows, int kind = kTcTf32) {
  const int elem = kind == kTcTf32 ? 4 : 2;
  const CUtensorMapDataType type = kind == kTcTf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : kind == kTcF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kp), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kp) * elem};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, type, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PHOBOS_OK : PHOBOS_ERR_CUDA;
}

// Tensor map of a caller's row-major matrix read as a K-major operand: `rows`
// x `k` elements with leading dimension `ld` (a multiple of 4), boxes of 32 x
// box_rows, 128B swizzle; reads outside the matrix return zeros.
phobos_status_t make_kmajor_map_strided(CUtensorMap *map, const float *base, int64_t rows,
                                        int64_t k, int64_t ld, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PHOBOS_OK : PHOBOS_ERR_CUDA;
}

phobos_status_t check_sizes(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                            int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return PHOBOS_ERR_INVALID_VALUE;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return PHOBOS_ERR_INVALID_VALUE;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return PHOBOS_ERR_UNSUPPORTED;
  return PHOBOS_OK;
}

size_t tc_workspace(int64_t M, int64_t N, int64_t K, int bm, int bn, int passes, int path) {
  const int e = tc_elem_bytes(path);
  const int64_t Mp = round_up(M, bm), Np = round_up(N, bn), Kp = round_up(K, tc_bk(path));
  const int64_t a = round_up(Mp * Kp * e, 256), b = round_up(Np * Kp * e, 256);
  return static_cast<size_t>((a + b) * (passes == 3 ? 2 : 1));
}

phobos_status_t make_plan(int64_t M, int64_t N, int64_t K, phobos_math_t math,
                          phobos_gemm_plan_t *p) {
  std::memset(p, 0, sizeof(*p));
  int path;
  switch (math) {
    case PHOBOS_MATH_FFMA: path = PHOBOS_PATH_FFMA; break;
    case PHOBOS_MATH_TF32: path = PHOBOS_PATH_TF32; break;
    case PHOBOS_MATH_3XTF32: path = PHOBOS_PATH_3XTF32; break;
    case PHOBOS_MATH_FP16: path = PHOBOS_PATH_FP16; break;
    case PHOBOS_MATH_BF16: path = PHOBOS_PATH_BF16; break;
    case PHOBOS_MATH_DEFAULT: {
      const double macs = static_cast<double>(M) * static_cast<double>(N) * static_cast<double>(K);
      path = (macs <= static_cast<double>(kFfmaMacLimit) || M < 16 || N < 16) ? PHOBOS_PATH_FFMA
                                                                               : PHOBOS_PATH_3XTF32;
      break;
    }
    default: return PHOBOS_ERR_INVALID_VALUE;
  }
  p->path = path;
  p->cluster_m = 1;
  p->cluster_n = 1;
  p->multicast = 0;
  p->super_k = K;
  if (path == PHOBOS_PATH_FFMA) {
    const int t = (M >= 1024 && N >= 1024) ? 128 : 64;
    p->tile_m = t;
    p->tile_n = t;
    p->tile_k = 16;
    p->stages = 2;
    p->super_m = round_up(kDefaultSuper, t);
    p->super_n = round_up(kDefaultSuper, t);
    p->workspace_bytes = 0;
  } else {
    const int passes = path == PHOBOS_PATH_3XTF32 ? 3 : 1;
    const int bn = N <= 128 ? 128 : 256;
    // A CTA pair (256-row tile, tcgen05 cta_group::2) when both extents fill it.
    const bool pair = bn == 256 && M > kTcBM;
    p->tile_m = pair ? 2 * kTcBM : kTcBM;
    p->cluster_m = pair ? 2 : 1;
    p->tile_n = bn;
    p->tile_k = tc_bk(path);
    p->stages = pair ? tc_pair_max_stages(passes, bn) : tc_max_stages(passes, bn);
    // Raster groups (super-tiles on one GPU) of 4096 rows, the pages' smallest
    // super-tile.  When the kernel splits A and B itself (split TF32, pairs,
    // N > 1536) and one such group would cover all of M, the first wave would
    // need every A panel split at once; groups of 2048 rows cut that demand
    // (measured on GB300, 4096^3 per call: 0.4431 -> 0.4338 ms; 8192^3 and
    // 3001 x 5003 x 1999 unchanged within noise).
    const bool split_inside = pair && passes == 3 && N > kInlineSplitMaxN;
    p->super_m = split_inside && M <= kDefaultSuper ? kDefaultSuper / 2 : kDefaultSuper;
    p->super_n = kDefaultSuper;
    p->workspace_bytes = tc_workspace(M, N, K, p->tile_m, bn, passes, path);
  }
  return PHOBOS_OK;
}

// True in a process launched as one rank of a multi-process (multi-GPU) job,
// as torchrun and similar launchers announce it.
bool in_multi_rank_job() {
  for (const char *name : {"WORLD_SIZE", "LOCAL_WORLD_SIZE"}) {
    const char *v = std::getenv(name);
    if (v && std::atoll(v) > 1) return true;
  }
  return false;
}

phobos_status_t validate_plan(int64_t M, int64_t N, int64_t K, phobos_math_t math,
                              const phobos_gemm_plan_t &p) {
  if (math == PHOBOS_MATH_FFMA && p.path != PHOBOS_PATH_FFMA) return PHOBOS_ERR_INVALID_VALUE;
  if (math == PHOBOS_MATH_TF32 && p.path != PHOBOS_PATH_TF32) return PHOBOS_ERR_INVALID_VALUE;
  if (math == PHOBOS_MATH_3XTF32 && p.path != PHOBOS_PATH_3XTF32) return PHOBOS_ERR_INVALID_VALUE;
  if (math == PHOBOS_MATH_FP16 && p.path != PHOBOS_PATH_FP16) return PHOBOS_ERR_INVALID_VALUE;
  if (math == PHOBOS_MATH_BF16 && p.path != PHOBOS_PATH_BF16) return PHOBOS_ERR_INVALID_VALUE;
  if (math == PHOBOS_MATH_DEFAULT && half_path(p.path)) return PHOBOS_ERR_INVALID_VALUE;
  if (p.multicast != 0 && p.multicast != 1) return PHOBOS_ERR_INVALID_VALUE;
  const bool mc = p.multicast == 1;
  // TMA multicast stays a one-GPU option: never in a rank of a multi-GPU job.
  if (mc && in_multi_rank_job()) return PHOBOS_ERR_UNSUPPORTED;
  // multicast: two CTA pairs side by side along N (cluster 2 x 2), tf32 operands
  // split by the pre-pass
  if ((p.cluster_m != 1 && p.cluster_m != 2) || p.cluster_n != (mc ? 2 : 1))
    return PHOBOS_ERR_UNSUPPORTED;
  if (mc && (p.cluster_m != 2 || (p.path != PHOBOS_PATH_TF32 && p.path != PHOBOS_PATH_3XTF32) ||
             p.a_split == 2))
    return PHOBOS_ERR_UNSUPPORTED;
  if (p.super_k <= 0 || p.super_m <= 0 || p.super_n <= 0) return PHOBOS_ERR_INVALID_VALUE;
  if (p.tail_split < 0 || p.tail_split > kMaxTailSplit) return PHOBOS_ERR_INVALID_VALUE;
  if (p.a_split < 0 || p.a_split > 3) return PHOBOS_ERR_INVALID_VALUE;
  if (p.clc != 0 && p.clc != 1) return PHOBOS_ERR_INVALID_VALUE;
  // Cluster Launch Control deals tiles to split-TF32 CTA pairs that read A
  // from the workspace, with the deepest ring (checked below)
  if (p.clc == 1 && (p.cluster_m != 2 || mc || p.path != PHOBOS_PATH_3XTF32 || p.a_split == 2))
    return PHOBOS_ERR_UNSUPPORTED;
  // the in-kernel panel split runs in tf32 CTA pairs without multicast
  if (p.a_split == 3 && (p.cluster_m != 2 || mc ||
                         (p.path != PHOBOS_PATH_TF32 && p.path != PHOBOS_PATH_3XTF32)))
    return PHOBOS_ERR_UNSUPPORTED;
  if (p.path == PHOBOS_PATH_FFMA) {
    if (p.cluster_m != 1) return PHOBOS_ERR_UNSUPPORTED;
    if (!((p.tile_m == 128 && p.tile_n == 128) || (p.tile_m == 64 && p.tile_n == 64)))
      return PHOBOS_ERR_INVALID_VALUE;
    if (p.tile_k != 16 || (p.super_k < K && p.super_k % 8 != 0)) return PHOBOS_ERR_INVALID_VALUE;
  } else if (p.path == PHOBOS_PATH_TF32 || p.path == PHOBOS_PATH_3XTF32 || half_path(p.path)) {
    const int passes = p.path == PHOBOS_PATH_3XTF32 ? 3 : 1;
    const bool pair = p.cluster_m == 2;
    const int bk = tc_bk(p.path);
    if (p.tile_m != (pair ? 2 * kTcBM : kTcBM) || (p.tile_n != 128 && p.tile_n != 256) ||
        p.tile_k != bk || (pair && p.tile_n != 256))
      return PHOBOS_ERR_INVALID_VALUE;
    const int max_st = pair ? tc_pair_max_stages(passes, p.tile_n) : tc_max_stages(passes, p.tile_n);
    if (p.stages < 2 || p.stages > max_st) return PHOBOS_ERR_INVALID_VALUE;
    if ((p.a_split >= 2 || mc || p.clc) && p.stages != max_st) return PHOBOS_ERR_INVALID_VALUE;
    // 16-bit inputs: pre-converted A, deepest ring
    if (half_path(p.path) && (p.a_split == 2 || (p.stages != max_st && p.stages != 4)))
      return PHOBOS_ERR_INVALID_VALUE;
    if (p.super_k < K && p.super_k % bk != 0) return PHOBOS_ERR_INVALID_VALUE;
    if (round_up(N, p.tile_n) / 32 > 65535) return PHOBOS_ERR_UNSUPPORTED;
  } else {
    return PHOBOS_ERR_INVALID_VALUE;
  }
  return PHOBOS_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

phobos_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PHOBOS_OK;
  if (e == cudaErrorMemoryAllocation) return PHOBOS_ERR_OUT_OF_MEMORY;
  return PHOBOS_ERR_CUDA;
}

void log_plan(int64_t M, int64_t N, int64_t K, const phobos_gemm_plan_t &p) {
  std::fprintf(stderr,
               "[phobos] M=%lld N=%lld K=%lld path=%d tile=%dx%dx%d cluster=%dx%d stages=%d "
               "super=%lldx%lldx%lld workspace=%zu\n",
               (long long)M, (long long)N, (long long)K, p.path, p.tile_m, p.tile_n, p.tile_k,
               p.cluster_m, p.cluster_n, p.stages, (long long)p.super_m, (long long)p.super_n,
               (long long)p.super_k, p.workspace_bytes);
}

// K slices per 64x64 FFMA tile (a cluster summed through DSMEM) when there are
// fewer tiles than SMs: enough clusters to fill the SMs, each slice at least
// four K blocks of 8.
int ffma_kslices(int64_t M, int64_t N, int64_t k_len, const phobos_gemm_plan_t &p,
                 int sm_count) {
  if (p.tile_m != 64 || p.tail_split == 1) return 1;
  const int64_t tiles = ((M + 63) / 64) * ((N + 63) / 64);
  int64_t S = p.tail_split >= 2 ? p.tail_split : (tiles > 0 ? sm_count / tiles : 1);
  if (S > 8) S = 8;
  if (S > (k_len + 31) / 32) S = (k_len + 31) / 32;
  return S >= 2 ? static_cast<int>(S) : 1;
}

phobos_status_t run_ffma(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                         int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                         int64_t ldc, cudaStream_t stream, const phobos_gemm_plan_t &p,
                         const DeviceState &dev) {
  FfmaArgs a{};
  a.A = A; a.B = B; a.C = C;
  a.lda = lda; a.ldb = ldb; a.ldc = ldc;
  a.M = static_cast<int>(M); a.N = static_cast<int>(N); a.K = static_cast<int>(K);
  a.tile = p.tile_m;
  a.vec_a = (lda % 4 == 0) && aligned16(A);
  a.vec_b = (ldb % 4 == 0) && aligned16(B);
  a.vec_c = (ldc % 4 == 0) && aligned16(C);
  if (p.super_k >= K) {
    a.alpha = alpha; a.beta = beta; a.k_begin = 0; a.k_len = static_cast<int>(K);
    a.kslices = ffma_kslices(M, N, K, p, dev.sm_count);
    if (mark(g_ev_start, stream) != cudaSuccess) return PHOBOS_ERR_CUDA;
    phobos_status_t st = cuda_status(counted(launch_ffma(a, stream)));
    if (st == PHOBOS_OK && mark(g_ev_stop, stream) != cudaSuccess) st = PHOBOS_ERR_CUDA;
    return st;
  }
  // cluster split: init leaf, then one step leaf per K chunk with beta = 1
  phobos_status_t st = cuda_status(counted(launch_scale(C, ldc, a.M, a.N, beta, stream)));
  if (st == PHOBOS_OK && mark(g_ev_start, stream) != cudaSuccess) st = PHOBOS_ERR_CUDA;
  for (int64_t k0 = 0; st == PHOBOS_OK && k0 < K; k0 += p.super_k) {
    a.alpha = alpha; a.beta = 1.0f;
    a.k_begin = static_cast<int>(k0);
    a.k_len = static_cast<int>(K - k0 < p.super_k ? K - k0 : p.super_k);
    a.kslices = ffma_kslices(M, N, a.k_len, p, dev.sm_count);
    st = cuda_status(counted(launch_ffma(a, stream)));
  }
  if (st == PHOBOS_OK && mark(g_ev_stop, stream) != cudaSuccess) st = PHOBOS_ERR_CUDA;
  return st;
}

// reuse_b: the previous call on this stream split the same B (same N, K, ldb,
// mode) into the workspace; skip that pre-pass unless the workspace moved.
// k_ready (K-chunked plans only): event c is waited for before the step leaf
// of K chunk c, for callers whose operands arrive chunk by chunk.
phobos_status_t run_tc(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                       const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                       cudaStream_t stream, const phobos_gemm_plan_t &p, DeviceState &dev,
                       int device, bool reuse_b = false, const cudaEvent_t *k_ready = nullptr) {
  const int passes = p.path == PHOBOS_PATH_3XTF32 ? 3 : 1;
  const bool pair = p.cluster_m == 2;
  const bool mc = p.multicast == 1;  // clusters of two pairs sharing A (validated: pairs, tf32)
  const int bm = pair ? 2 * kTcBM : kTcBM;
  const int bn = p.tile_n;
  const bool half = half_path(p.path);
  const int bk = tc_bk(p.path), elem = tc_elem_bytes(p.path), kind = tc_kind(p.path);
  const int64_t Mp = round_up(M, bm), Np = round_up(N, bn), Kp = round_up(K, bk);
  // Where A is split: inside the kernel (TMA reads the caller's A directly)
  // or by the pre-pass into the workspace.  16-bit inputs are always
  // converted by the pre-pass.
  const bool a_tma_ok = (lda % 4 == 0) && aligned16(A);
  const int max_st = pair ? tc_pair_max_stages(passes, bn) : tc_max_stages(passes, bn);
  bool a_inline = false;      // A split in shared memory, B by the pre-pass
  bool split_inline = false;  // A and B split into the workspace by the GEMM kernel itself
  if (half) {
    if (p.a_split >= 2) return PHOBOS_ERR_UNSUPPORTED;
  } else if (p.a_split == 2) {
    if (!a_tma_ok) return PHOBOS_ERR_UNSUPPORTED;
    a_inline = true;
  } else if (p.a_split == 3) {
    split_inline = true;  // validated: tf32 CTA pairs, no multicast, deepest ring
  } else if (p.a_split == 0 && !mc && p.stages == max_st) {
    a_inline = !p.clc && a_tma_ok && N <= kInlineSplitMaxN;
    split_inline = !a_inline && pair && passes == 3;
  }
  const int64_t a_bytes = round_up(Mp * Kp * elem, 256), b_bytes = round_up(Np * Kp * elem, 256);
  const int ops = passes == 3 ? 2 : 1;  // big (+ small)
  // workspace: [B big][B small][A big][A small] (no A part when A is split in-kernel)
  const size_t ops_bytes = static_cast<size_t>(ops * b_bytes + (a_inline ? 0 : ops * a_bytes));

  // Persistent grid: one CTA (pair) per SM (pair), or one multicast cluster
  // per four SMs, as many as can be resident together.  The tiles of the
  // last, partial wave are split along K so that idle SMs share the tail.
  // With multicast a tile of the walk is two pair tiles side by side.
  int units = pair ? dev.sm_count / 2 : dev.sm_count;
  if (mc) {
    int &resident = dev.mc_clusters[passes == 3 ? 1 : 0];
    if (resident == 0) resident = tc_multicast_clusters(passes, bn, stream);
    if (resident <= 0) return PHOBOS_ERR_CUDA;
    units = dev.sm_count / 4 < resident ? dev.sm_count / 4 : resident;
    if (units <= 0) return PHOBOS_ERR_UNSUPPORTED;
    if (env_flag("PHOBOS_LOG"))
      std::fprintf(stderr, "[phobos] multicast clusters: %d resident at once, %d used\n", resident,
                   units);
  }
  const int64_t walk_n = mc ? (Np / bn + 1) / 2 : Np / bn;  // tile columns of the walk
  const int total_tiles = static_cast<int>((Mp / bm) * walk_n);
  const int chunk_blocks_max =
      static_cast<int>(round_up(p.super_k < K ? p.super_k : K, bk) / bk);
  // the static walk's tail split (Cluster Launch Control cuts its own, below)
  const int tail = units > 0 && !p.clc ? total_tiles % units : 0;
  const int tail_units = tail_workers(p.tail_split, tail, units, chunk_blocks_max);
  const int full_tiles = tail_units > 0 ? total_tiles - tail : total_tiles;
  // Cluster Launch Control: the last partial wave's tiles cut into P K
  // pieces of at least 4 k blocks, enough to give every resident pair work
  // (tail_split 1: off; 2..8: P)
  int clc_pieces = 1;
  const int clc_tail = p.clc && units > 0 ? total_tiles % units : 0;
  if (clc_tail > 0 && p.tail_split != 1) {
    int P = p.tail_split >= 2 ? p.tail_split : units / clc_tail;
    if (P > chunk_blocks_max / 4) P = chunk_blocks_max / 4;
    if (P > kMaxTailSplit) P = kMaxTailSplit;
    clc_pieces = P > 1 ? P : 1;
  }
  const int64_t slots = clc_pieces > 1 ? static_cast<int64_t>(clc_tail) * clc_pieces
                                       : static_cast<int64_t>(tail_units) * (mc ? 2 : 1);
  const size_t part_bytes = static_cast<size_t>(round_up(slots * bm * bn * 4, 256));
  // flags: the tail split's, then (in-kernel panel split) one per item of the
  // longest launch and two item counters per launch (claimed, done)
  const int64_t tail_flags = slots * 2 * kEpiWarps;
  const int64_t chunk_kc = (chunk_blocks_max + kSplitChunkBlocks - 1) / kSplitChunkBlocks;
  const int64_t launches = p.super_k < K ? (Kp / bk + chunk_blocks_max - 1) / chunk_blocks_max : 1;
  const int64_t split_flags = split_inline ? (Mp / bm + Np / bn) * chunk_kc * 8 : 0;
  const int64_t split_counters = split_inline ? 2 * launches : 0;  // claimed, done
  const size_t flag_bytes =
      static_cast<size_t>(round_up((tail_flags + split_flags + split_counters) * 4, 256));
  const size_t need = ops_bytes + part_bytes + flag_bytes;
  Buffer &ws = g_workspaces[{device, reinterpret_cast<uintptr_t>(stream)}];
  void *const old_ws = ws.ptr;
  phobos_status_t st = ensure_buffer(ws, need, stream);
  if (st != PHOBOS_OK) return st;
  if (ws.ptr != old_ws) reuse_b = false;
  float *partials = reinterpret_cast<float *>(static_cast<char *>(ws.ptr) + ops_bytes);
  unsigned *flags =
      reinterpret_cast<unsigned *>(static_cast<char *>(ws.ptr) + ops_bytes + part_bytes);
  if ((st = get_encoder()) != PHOBOS_OK) return st;

  char *base = static_cast<char *>(ws.ptr);
  float *b_big = reinterpret_cast<float *>(base);
  float *b_small = passes == 3 ? reinterpret_cast<float *>(base + b_bytes) : nullptr;
  float *a_big = reinterpret_cast<float *>(base + ops * b_bytes);
  float *a_small = passes == 3 ? reinterpret_cast<float *>(base + ops * b_bytes + a_bytes) : nullptr;

  // Flags must not hold a value a launch of this call will wait for: the
  // split-TF32 / TF32 pre-pass zeroes them in the same launch; without a
  // pre-pass a memset does.
  if (split_inline) {
    if (cudaMemsetAsync(flags, 0, flag_bytes, stream) != cudaSuccess) return PHOBOS_ERR_CUDA;
  } else if (half) {
    if (flag_bytes && cudaMemsetAsync(flags, 0, flag_bytes, stream) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    st = cuda_status(counted(launch_convert_rows(A, lda, static_cast<int>(M), static_cast<int>(K),
                                                 static_cast<int>(Mp), static_cast<int>(Kp), a_big,
                                                 kind == kTcBf16, stream)));
    if (st != PHOBOS_OK) return st;
    if (!reuse_b) {
      st = cuda_status(counted(launch_convert_cols(B, ldb, static_cast<int>(K), static_cast<int>(N),
                                                   static_cast<int>(Np), static_cast<int>(Kp), b_big,
                                                   kind == kTcBf16, stream)));
      if (st != PHOBOS_OK) return st;
    }
  } else if (!a_inline || !reuse_b || flag_bytes) {
    SplitArgs sa{};
    sa.A = A;
    sa.lda = lda;
    sa.M = static_cast<int>(M);
    sa.K = static_cast<int>(K);
    sa.Mp = static_cast<int>(Mp);
    sa.Kp = static_cast<int>(Kp);
    sa.a_big = a_big;
    sa.a_small = a_small;
    sa.vec_a = a_tma_ok ? 1 : 0;
    sa.B = B;
    sa.ldb = ldb;
    sa.N = static_cast<int>(N);
    sa.Np = static_cast<int>(Np);
    sa.b_big = b_big;
    sa.b_small = b_small;
    sa.flags = flags;
    sa.n_flags = tail_flags;
    st = cuda_status(counted(launch_split_ab(sa, a_inline ? 0 : 1, reuse_b ? 0 : 1, stream)));
    if (st != PHOBOS_OK) return st;
  }

  TcArgs t{};
  // each CTA loads 128 rows of A and, in a pair, half of the tile's B rows
  const int b_box = pair ? bn / 2 : bn;
  // with multicast each CTA loads half of its 128 A rows (and receives the
  // other half from the other pair)
  const int a_box = mc ? kTcBM / 2 : kTcBM;
  if (a_inline) {
    // the caller's A: K x M extents with its own stride; TMA fills zeros outside
    if ((st = make_kmajor_map_strided(&t.tmap_ab, A, M, K, lda, kTcBM)) != PHOBOS_OK) return st;
    t.tmap_as = t.tmap_ab;
  } else {
    if ((st = make_kmajor_map(&t.tmap_ab, a_big, Mp, Kp, a_box, kind)) != PHOBOS_OK) return st;
    t.tmap_as = t.tmap_ab;
    if (passes == 3 && (st = make_kmajor_map(&t.tmap_as, a_small, Mp, Kp, a_box)) != PHOBOS_OK)
      return st;
  }
  if ((st = make_kmajor_map(&t.tmap_bb, b_big, Np, Kp, b_box, kind)) != PHOBOS_OK) return st;
  t.tmap_bs = t.tmap_bb;
  if (passes == 3 && (st = make_kmajor_map(&t.tmap_bs, b_small, Np, Kp, b_box)) != PHOBOS_OK)
    return st;
  t.a_inline = a_inline ? 1 : 0;
  t.multicast = mc ? 1 : 0;
  if (split_inline) {
    t.split_inline = 1;
    t.split_b = reuse_b ? 0 : 1;  // a reused B was split by an earlier call on this stream
    t.A_raw = A;
    t.B_raw = B;
    t.lda = lda;
    t.ldb = ldb;
    t.K = static_cast<int>(K);
    t.kp = static_cast<int>(Kp);
    t.a_big = a_big;
    t.a_small = a_small;
    t.b_big = b_big;
    t.b_small = b_small;
    t.vec_a = a_tma_ok ? 1 : 0;
    t.vec_b = (ldb % 4 == 0) && aligned16(B) ? 1 : 0;
    t.split_flags = flags + tail_flags;
    t.split_next = flags + tail_flags + split_flags;
    t.split_done = t.split_next + launches;
  }
  t.C = C;
  t.ldc = ldc;
  t.M = static_cast<int>(M);
  t.N = static_cast<int>(N);
  t.tiles_m = static_cast<int>(Mp / bm);
  t.tiles_n = static_cast<int>(walk_n);
  int64_t gm = p.super_m / bm;
  if (gm < 1) gm = 1;
  if (gm > t.tiles_m) gm = t.tiles_m;
  t.group_m = static_cast<int>(gm);
  t.vec_c = (ldc % 4 == 0) && aligned16(C);
  // Split TF32 needs short TMEM partial sums to stay at fp32 accuracy.
  t.promote_blocks = passes == 3 ? promote_blocks_for(p.super_k < K ? p.super_k : K)
                     : half      ? kHalfPromoteBlocks
                                 : kTf32PromoteBlocks;
  t.sm_count = dev.sm_count;
  t.withhold_first_load = env_flag("PHOBOS_TEST_WITHHOLD_LOAD")    ? 1
                          : env_flag("PHOBOS_TEST_WITHHOLD_SPLIT") ? 2
                                                                   : 0;
  t.full_tiles = full_tiles;
  t.tail_units = tail_units;
  // whole tiles stride over all SMs (pairs); with no whole tiles, only the
  // workers sharing the tail are launched
  t.grid_units = tail_units > 0 ? (full_tiles > 0 ? units : tail_units)
                                : (total_tiles < units ? total_tiles : units);
  if (p.clc) {  // a pair per work item; the resident ones take the rest
    t.clc = 1;
    t.clc_units = units;
    t.clc_pieces = clc_pieces;
    t.full_tiles = clc_pieces > 1 ? total_tiles - clc_tail : total_tiles;
    t.grid_units = t.full_tiles + (clc_pieces > 1 ? clc_tail * clc_pieces : 0);
  }
  t.partials = partials;
  t.flags = flags;
  t.epoch = 1;
  t.err = dev.err;
  if (g_ev_start) {  // instrumentation on: the kernels also sum their SM cycles
    if (!dev.clock_acc) {
      if (cudaMalloc(&dev.clock_acc, 3 * sizeof(unsigned long long)) != cudaSuccess)
        return PHOBOS_ERR_OUT_OF_MEMORY;
      if (cudaMemset(dev.clock_acc, 0, 3 * sizeof(unsigned long long)) != cudaSuccess)
        return PHOBOS_ERR_CUDA;
    }
    t.clock_acc = dev.clock_acc;
  }
  const int total_blocks = static_cast<int>(Kp / bk);
  if (p.super_k >= K) {
    t.alpha = alpha;
    t.beta = beta;
    t.k_block0 = 0;
    t.k_blocks = total_blocks;
    if (t.tail_units > 0) {
      t.tail_units = fill_tail_shares(t, tail, t.tail_units);
      if (t.tail_units == 0) t.full_tiles = total_tiles;
    }
    if (mark(g_ev_start, stream) != cudaSuccess) return PHOBOS_ERR_CUDA;
    st = cuda_status(counted(pair ? launch_tc_pair(t, passes, bn, p.stages, stream, kind)
                                   : launch_tc(t, passes, bn, p.stages, stream, kind)));
    if (st == PHOBOS_OK && mark(g_ev_stop, stream) != cudaSuccess) st = PHOBOS_ERR_CUDA;
    return st;
  }
  // cluster split: init leaf C = beta*C, then step leaves C += alpha * A_c B_c
  st = cuda_status(counted(launch_scale(C, ldc, t.M, t.N, beta, stream)));
  if (st == PHOBOS_OK && mark(g_ev_start, stream) != cudaSuccess) st = PHOBOS_ERR_CUDA;
  const int chunk_blocks = static_cast<int>(p.super_k / bk);
  for (int kb = 0; st == PHOBOS_OK && kb < total_blocks; kb += chunk_blocks, ++t.epoch) {
    t.alpha = alpha;
    t.beta = 1.0f;
    t.k_block0 = kb;
    t.k_blocks = total_blocks - kb < chunk_blocks ? total_blocks - kb : chunk_blocks;
    // a short last chunk may not afford as many pieces
    if (t.tail_units > 0) {
      int w = tail_workers(p.tail_split, tail, units, t.k_blocks);
      if (w > tail_units) w = tail_units;  // the slots sized above
      t.tail_units = w > 0 ? fill_tail_shares(t, tail, w) : 0;
      if (t.tail_units == 0) t.full_tiles = total_tiles;
    }
    if (k_ready && cudaStreamWaitEvent(stream, k_ready[t.epoch - 1], 0) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    st = cuda_status(counted(pair ? launch_tc_pair(t, passes, bn, p.stages, stream, kind)
                                   : launch_tc(t, passes, bn, p.stages, stream, kind)));
  }
  if (st == PHOBOS_OK && mark(g_ev_stop, stream) != cudaSuccess) st = PHOBOS_ERR_CUDA;
  return st;
}

phobos_status_t read_status_word(DeviceState &dev, cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PHOBOS_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, dev.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PHOBOS_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(dev.err, 0, sizeof(int)) != cudaSuccess) return PHOBOS_ERR_CUDA;
    if (env_flag("PHOBOS_LOG")) std::fprintf(stderr, "[phobos] device status word 0x%x\n", word);
    return PHOBOS_ERR_TIMEOUT;
  }
  return PHOBOS_OK;
}

phobos_status_t sgemm_impl(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                           int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                           int64_t ldc, void *stream_ptr, phobos_math_t math,
                           const phobos_gemm_plan_t *user_plan, bool reuse_b = false,
                           const cudaEvent_t *k_ready = nullptr) {
  phobos_status_t st = check_sizes(M, N, K, lda, ldb, ldc);
  if (st != PHOBOS_OK) return st;
  if (math < PHOBOS_MATH_DEFAULT || math > PHOBOS_MATH_BF16) return PHOBOS_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return PHOBOS_OK;
  if (!C) return PHOBOS_ERR_INVALID_VALUE;
  const bool products = K > 0 && alpha != 0.0f;
  if (products && (!A || !B)) return PHOBOS_ERR_INVALID_VALUE;

  phobos_gemm_plan_t plan;
  if (user_plan) {
    plan = *user_plan;
    if ((st = validate_plan(M, N, K, math, plan)) != PHOBOS_OK) return st;
  } else if ((st = make_plan(M, N, K, math, &plan)) != PHOBOS_OK) {
    return st;
  }

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState *dev = nullptr;
  int device = 0;
  if ((st = device_state(&dev, &device)) != PHOBOS_OK) return st;
  if (env_flag("PHOBOS_LOG")) log_plan(M, N, K, plan);

  if (!products) {
    st = cuda_status(counted(launch_scale(C, ldc, static_cast<int>(M), static_cast<int>(N), beta, stream)));
  } else if (plan.path == PHOBOS_PATH_FFMA) {
    st = run_ffma(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, plan, *dev);
  } else {
    st = run_tc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, plan, *dev, device,
                reuse_b, plan.super_k < K ? k_ready : nullptr);
  }
  if (st == PHOBOS_OK && env_flag("PHOBOS_DEBUG_SYNC")) st = read_status_word(*dev, stream);
  return st;
}

}  // namespace
}  // namespace phobos

using namespace phobos;

extern "C" {

phobos_status_t phobos_gemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                 int64_t ldc, phobos_math_t math, phobos_gemm_plan_t *out) {
  if (!out) return PHOBOS_ERR_INVALID_VALUE;
  const phobos_status_t st = check_sizes(M, N, K, lda, ldb, ldc);
  if (st != PHOBOS_OK) return st;
  return make_plan(M, N, K, math, out);
}

phobos_status_t phobos_sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                             int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                             int64_t ldc, void *stream) {
  return sgemm_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, PHOBOS_MATH_DEFAULT,
                    nullptr);
}

phobos_status_t phobos_sgemm_ex(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                                int64_t ldc, void *stream, phobos_math_t math,
                                const phobos_gemm_plan_t *plan) {
  return sgemm_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, math, plan);
}

phobos_status_t phobos_sgemm_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                  int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                                  int64_t ldc, void *stream_ptr, phobos_math_t math) {
  phobos_status_t st = check_sizes(M, N, K, lda, ldb, ldc);
  if (st != PHOBOS_OK) return st;
  if (math < PHOBOS_MATH_DEFAULT || math > PHOBOS_MATH_BF16) return PHOBOS_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return PHOBOS_OK;
  if (!C) return PHOBOS_ERR_INVALID_VALUE;
  const bool products = K > 0 && alpha != 0.0f;
  if (products && (!A || !B)) return PHOBOS_ERR_INVALID_VALUE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  std::lock_guard<std::mutex> host_lock(g_host_mutex);
  // extents of the strided host arrays, in elements
  const size_t a_elems = products ? static_cast<size_t>((M - 1) * lda + K) : 0;
  const size_t b_elems = products ? static_cast<size_t>((K - 1) * ldb + N) : 0;
  const size_t c_elems = static_cast<size_t>((M - 1) * ldc + N);
  float *dA = nullptr, *dB = nullptr, *dC = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *dev = nullptr;
    int device = 0;
    if ((st = device_state(&dev, &device)) != PHOBOS_OK) return st;
    Staging &s = g_staging[device];
    if (products && (st = ensure_buffer(s.a, a_elems * 4, stream)) != PHOBOS_OK) return st;
    if (products && (st = ensure_buffer(s.b, b_elems * 4, stream)) != PHOBOS_OK) return st;
    if ((st = ensure_buffer(s.c, c_elems * 4, stream)) != PHOBOS_OK) return st;
    dA = static_cast<float *>(s.a.ptr);
    dB = static_cast<float *>(s.b.ptr);
    dC = static_cast<float *>(s.c.ptr);
  }
  // Large tensor-core problems run as row bands so that copies overlap the
  // compute: B goes in first, then every band's rows of A (and C) on a copy
  // stream; band i's GEMM runs on the caller's stream as soon as its rows are
  // in (bands after the first reuse the first band's split of B), and its rows
  // of C go back on a second copy stream while later bands compute.
  phobos_gemm_plan_t plan;
  if (products && (st = make_plan(M, N, K, math, &plan)) != PHOBOS_OK) return st;
  int bands = 1;
  if (products && plan.path != PHOBOS_PATH_FFMA && M >= 2048) {
    bands = static_cast<int>(M / 1024);
    if (bands > kMaxBands) bands = kMaxBands;
  }
  if (bands <= 1) {
    if (products) {
      if (cudaMemcpyAsync(dA, A, a_elems * 4, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
          cudaMemcpyAsync(dB, B, b_elems * 4, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return PHOBOS_ERR_CUDA;
    }
    if (beta != 0.0f &&
        cudaMemcpyAsync(dC, C, c_elems * 4, cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    st = sgemm_impl(M, N, K, alpha, dA, lda, dB, ldb, beta, dC, ldc, stream_ptr, math, nullptr);
    if (st != PHOBOS_OK) return st;
    if (cudaMemcpyAsync(C, dC, c_elems * 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PHOBOS_ERR_CUDA;
    return PHOBOS_OK;
  }
  HostPipe *pipe = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return PHOBOS_ERR_CUDA;
    pipe = &g_pipes[device];
    if (!pipe->ready) {
      if (cudaStreamCreateWithFlags(&pipe->in, cudaStreamNonBlocking) != cudaSuccess ||
          cudaStreamCreateWithFlags(&pipe->out, cudaStreamNonBlocking) != cudaSuccess)
        return PHOBOS_ERR_CUDA;
      for (cudaEvent_t &e : pipe->ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
          return PHOBOS_ERR_CUDA;
      pipe->ready = true;
    }
  }
  cudaEvent_t ev_start = pipe->ev[0], ev_end = pipe->ev[1];
  cudaEvent_t *ev_in = pipe->ev + 2, *ev_done = pipe->ev + 2 + kMaxBands;
  cudaEvent_t *ev_b = pipe->ev + 2 + 2 * kMaxBands;
  const int64_t rows = ((M + bands - 1) / bands + 255) / 256 * 256;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // When the first band's kernel splits its own operands (split TF32 with CTA
  // pairs and N > 1536), it runs in K chunks: B crosses the link chunk by
  // chunk right after that band's rows of A and C, and each chunk's step leaf
  // waits only for its rows of B, so the GEMM starts long before all of B is
  // in.  The later bands reuse the split of B that those steps leave in the
  // workspace.  Otherwise all of B goes first.
  phobos_gemm_plan_t band0_plan;
  int64_t kc = 0;
  int n_kc = 0;
  if (make_plan(rows < M ? rows : M, N, K, math, &band0_plan) == PHOBOS_OK &&
      band0_plan.path == PHOBOS_PATH_3XTF32 && band0_plan.cluster_m == 2 &&
      N > kInlineSplitMaxN && K >= 2048) {
    kc = round_up((K + kMaxBChunks - 1) / kMaxBChunks, 256);
    n_kc = static_cast<int>((K + kc - 1) / kc);
    band0_plan.super_k = kc;
  }
  if (!ok(cudaEventRecord(ev_start, stream)) || !ok(cudaStreamWaitEvent(pipe->in, ev_start, 0)) ||
      !ok(cudaStreamWaitEvent(pipe->out, ev_start, 0)) ||
      (n_kc == 0 && !ok(cudaMemcpyAsync(dB, B, b_elems * 4, cudaMemcpyHostToDevice, pipe->in))))
    return PHOBOS_ERR_CUDA;
  int used = 0;
  for (int64_t r0 = 0; r0 < M; r0 += rows, ++used) {
    const int64_t r1 = r0 + rows < M ? r0 + rows : M;
    const size_t a_off = static_cast<size_t>(r0 * lda), a_len = static_cast<size_t>((r1 - 1 - r0) * lda + K);
    const size_t c_off = static_cast<size_t>(r0 * ldc), c_len = static_cast<size_t>((r1 - 1 - r0) * ldc + N);
    if (!ok(cudaMemcpyAsync(dA + a_off, A + a_off, a_len * 4, cudaMemcpyHostToDevice, pipe->in)) ||
        (beta != 0.0f &&
         !ok(cudaMemcpyAsync(dC + c_off, C + c_off, c_len * 4, cudaMemcpyHostToDevice, pipe->in))) ||
        !ok(cudaEventRecord(ev_in[used], pipe->in)))
      return PHOBOS_ERR_CUDA;
    for (int c = 0; used == 0 && c < n_kc; ++c) {  // B's K rows, chunk by chunk
      const int64_t k0 = c * kc, k1 = k0 + kc < K ? k0 + kc : K;
      const size_t b_off = static_cast<size_t>(k0 * ldb), b_len = static_cast<size_t>((k1 - 1 - k0) * ldb + N);
      if (!ok(cudaMemcpyAsync(dB + b_off, B + b_off, b_len * 4, cudaMemcpyHostToDevice, pipe->in)) ||
          !ok(cudaEventRecord(ev_b[c], pipe->in)))
        return PHOBOS_ERR_CUDA;
    }
  }
  int band = 0;
  for (int64_t r0 = 0; r0 < M; r0 += rows, ++band) {
    const int64_t r1 = r0 + rows < M ? r0 + rows : M;
    const size_t a_off = static_cast<size_t>(r0 * lda);
    const size_t c_off = static_cast<size_t>(r0 * ldc), c_len = static_cast<size_t>((r1 - 1 - r0) * ldc + N);
    if (!ok(cudaStreamWaitEvent(stream, ev_in[band], 0))) return PHOBOS_ERR_CUDA;
    if (band == 0 && n_kc > 0)
      st = sgemm_impl(r1 - r0, N, K, alpha, dA + a_off, lda, dB, ldb, beta, dC + c_off, ldc,
                      stream_ptr, math, &band0_plan, false, ev_b);
    else
      st = sgemm_impl(r1 - r0, N, K, alpha, dA + a_off, lda, dB, ldb, beta, dC + c_off, ldc,
                      stream_ptr, math, nullptr, band > 0);
    if (st != PHOBOS_OK) return st;
    if (!ok(cudaEventRecord(ev_done[band], stream)) ||
        !ok(cudaStreamWaitEvent(pipe->out, ev_done[band], 0)) ||
        !ok(cudaMemcpyAsync(C + c_off, dC + c_off, c_len * 4, cudaMemcpyDeviceToHost, pipe->out)))
      return PHOBOS_ERR_CUDA;
  }
  if (!ok(cudaEventRecord(ev_end, pipe->out)) || !ok(cudaStreamWaitEvent(stream, ev_end, 0)) ||
      !ok(cudaStreamSynchronize(stream)))
    return PHOBOS_ERR_CUDA;
  return PHOBOS_OK;
}

phobos_status_t phobos_check_device(void *stream) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState *dev = nullptr;
  int device = 0;
  phobos_status_t st = device_state(&dev, &device);
  if (st != PHOBOS_OK) return st;
  st = read_status_word(*dev, static_cast<cudaStream_t>(stream));
  // The no-allocation entry point keeps its own word inside its fixed
  // scratch; read and clear it too, so an expired wait there is reported here.
  if (int *word = noalloc_status_word(device)) {
    int v = 0;
    if (cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    if (v != 0) {
      if (cudaMemset(word, 0, sizeof(int)) != cudaSuccess) return PHOBOS_ERR_CUDA;
      if (st == PHOBOS_OK) st = PHOBOS_ERR_TIMEOUT;
    }
  }
  return st;
}

phobos_status_t phobos_set_timing_events(void *start, void *stop) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_ev_start = static_cast<cudaEvent_t>(start);
  g_ev_stop = static_cast<cudaEvent_t>(stop);
  return PHOBOS_OK;
}

phobos_status_t phobos_kernel_clock_mhz(double *mhz) {
  if (!mhz) return PHOBOS_ERR_INVALID_VALUE;
  *mhz = 0.0;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState *dev = nullptr;
  phobos_status_t st = device_state(&dev, nullptr);
  if (st != PHOBOS_OK) return st;
  if (!dev->clock_acc) return PHOBOS_OK;
  unsigned long long acc[2] = {0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(acc, dev->clock_acc, sizeof(acc), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(dev->clock_acc, 0, sizeof(acc)) != cudaSuccess)
    return PHOBOS_ERR_CUDA;
  if (acc[1] > 0) *mhz = 1e3 * static_cast<double>(acc[0]) / static_cast<double>(acc[1]);
  return PHOBOS_OK;
}

phobos_status_t phobos_kernel_clc_tiles(uint64_t *tiles) {
  if (!tiles) return PHOBOS_ERR_INVALID_VALUE;
  *tiles = 0;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState *dev = nullptr;
  phobos_status_t st = device_state(&dev, nullptr);
  if (st != PHOBOS_OK) return st;
  if (!dev->clock_acc) return PHOBOS_OK;
  unsigned long long n = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&n, dev->clock_acc + 2, sizeof(n), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(dev->clock_acc + 2, 0, sizeof(n)) != cudaSuccess)
    return PHOBOS_ERR_CUDA;
  *tiles = n;
  return PHOBOS_OK;
}

uint64_t phobos_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

phobos_status_t phobos_release(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int current = 0;
  if (cudaGetDevice(&current) != cudaSuccess) return PHOBOS_ERR_CUDA;
  phobos_status_t st = PHOBOS_OK;
  auto free_on = [&](int device, Buffer &b) {
    if (!b.ptr) return;
    if (cudaSetDevice(device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
        cudaFree(b.ptr) != cudaSuccess)
      st = PHOBOS_ERR_CUDA;
    b.ptr = nullptr;
    b.bytes = 0;
  };
  for (auto &kv : g_workspaces) free_on(kv.first.first, kv.second);
  g_workspaces.clear();
  for (auto &kv : g_staging) {
    free_on(kv.first, kv.second.a);
    free_on(kv.first, kv.second.b);
    free_on(kv.first, kv.second.c);
  }
  g_staging.clear();
  cudaSetDevice(current);
  return st;
}

const char *phobos_status_string(phobos_status_t status) {
  switch (status) {
    case PHOBOS_OK: return "PHOBOS_OK: success";
    case PHOBOS_ERR_INVALID_VALUE: return "PHOBOS_ERR_INVALID_VALUE: invalid argument or plan";
    case PHOBOS_ERR_UNSUPPORTED: return "PHOBOS_ERR_UNSUPPORTED: device or shape not supported";
    case PHOBOS_ERR_CUDA: return "PHOBOS_ERR_CUDA: a CUDA call failed";
    case PHOBOS_ERR_OUT_OF_MEMORY: return "PHOBOS_ERR_OUT_OF_MEMORY: workspace allocation failed";
    case PHOBOS_ERR_TIMEOUT: return "PHOBOS_ERR_TIMEOUT: a device-side bounded wait expired";
  }
  return "unknown phobos status";
}

}  // extern "C"
