// Split-TF32 SGEMM with no device allocation: the entry point
// phobos_sgemm_noalloc runs the same operand pre-pass and tcgen05 main kernel
// as the 3xTF32 path of phobos_sgemm_ex, but its scratch (the tf32 big/small
// operand copies and a device status word) lives in one file-scope
// `__device__` array instead of a workspace obtained from cudaMallocAsync.
//
// Who needs this: callers that may not allocate device memory themselves --
// a serving process whose device memory was reserved up front by its own
// allocator (a caching allocator or an inference engine that claimed most of
// HBM at start-up, so a fresh cudaMalloc can fail or fragment the pool), and
// latency-critical loops that cannot take the implicit synchronisation and
// allocator latency of cudaMalloc/cudaFree.  They still pass their own A, B
// and C.
#include "../../include/phobos_gemm.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "host_rules.h"
#include "internal.h"

namespace phobos {
namespace {

constexpr size_t kHeadBytes = 256;  // status word, padded to keep the operands aligned
constexpr size_t kScratchBytes = PHOBOS_NOALLOC_SCRATCH_BYTES;
constexpr int kBM = 128, kBK = 32;
constexpr int64_t kSuper = 4096;
constexpr int kMaxDevices = 64;

// The scratch.  Every GPU that loads this library holds it until the process
// exits.  Layout: [0, 4) device status word; [256, 256 + kScratchBytes) the
// split operands of the current call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kHeadBytes + kScratchBytes];

std::mutex g_setup_mutex;
// Device address of g_noalloc_scratch per device ordinal (0 = not set up yet).
void *g_scratch_addr[kMaxDevices] = {};
bool g_device_ok[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Once per device, with that device current: find the scratch array's device
// address (the host-side symbol is only a stand-in and must never be passed
// to a kernel) and check the device.
phobos_status_t set_up(int dev, void **scratch) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (dev < 0 || dev >= kMaxDevices) return PHOBOS_ERR_UNSUPPORTED;
  if (!g_scratch_addr[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    g_device_ok[dev] = (major == 10 && minor == 3);
    if (!g_device_ok[dev]) return PHOBOS_ERR_UNSUPPORTED;
    if (cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return PHOBOS_ERR_CUDA;
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) {
      cudaGetLastError();
      return PHOBOS_ERR_CUDA;
    }
    if (!g_encode_fn) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return PHOBOS_ERR_CUDA;
      g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    g_scratch_addr[dev] = addr;
  }
  if (!g_device_ok[dev]) return PHOBOS_ERR_UNSUPPORTED;
  *scratch = g_scratch_addr[dev];
  return PHOBOS_OK;
}

phobos_status_t kmajor_map(CUtensorMap *map, const float *base, int64_t rows, int64_t kp,
                           int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kp), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kp) * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode_fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PHOBOS_OK : PHOBOS_ERR_CUDA;
}

phobos_status_t ok(cudaError_t e) { return e == cudaSuccess ? PHOBOS_OK : PHOBOS_ERR_CUDA; }

// Bytes of split operands a call needs: tf32 big and small copies of A
// ([Mp][Kp]) and of B transposed ([Np][Kp]), each copy padded to 256 bytes.
size_t scratch_bytes(int64_t M, int64_t N, int64_t K) {
  const int bn = N <= 128 ? 128 : 256;
  const int64_t Mp = round_up(M, kBM), Np = round_up(N, bn), Kp = round_up(K, kBK);
  return static_cast<size_t>(2 * (round_up(Mp * Kp * 4, 256) + round_up(Np * Kp * 4, 256)));
}

}  // namespace

// The status word of the no-allocation entry point on device `dev`, or null
// when that entry point has not run on the device yet; phobos_check_device
// reads and clears it beside the library's own word.
int *noalloc_status_word(int dev) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  return static_cast<int *>(g_scratch_addr[dev]);
}

}  // namespace phobos

using namespace phobos;

extern "C" phobos_status_t phobos_sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                                const float *A, int64_t lda, const float *B,
                                                int64_t ldb, float beta, float *C, int64_t ldc,
                                                void *stream_ptr) {
  if (M < 0 || N < 0 || K < 0) return PHOBOS_ERR_INVALID_VALUE;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return PHOBOS_ERR_INVALID_VALUE;
  // the same limit as every other entry point, before any size is narrowed to int
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return PHOBOS_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return PHOBOS_OK;
  if (!C) return PHOBOS_ERR_INVALID_VALUE;
  const bool products = K > 0 && alpha != 0.0f;
  if (products && (!A || !B)) return PHOBOS_ERR_INVALID_VALUE;
  if (products && scratch_bytes(M, N, K) > kScratchBytes)
    return PHOBOS_ERR_UNSUPPORTED;  // the split operands would not fit the fixed scratch

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PHOBOS_ERR_CUDA;
  void *scratch = nullptr;
  phobos_status_t st = set_up(dev, &scratch);
  if (st != PHOBOS_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int *status_word = static_cast<int *>(scratch);

  if (!products) {
    st = ok(launch_scale(C, ldc, static_cast<int>(M), static_cast<int>(N), beta, stream));
  } else {
    const int bn = N <= 128 ? 128 : 256;
    const int64_t Mp = round_up(M, kBM), Np = round_up(N, bn), Kp = round_up(K, kBK);
    const int64_t a_bytes = round_up(Mp * Kp * 4, 256), b_bytes = round_up(Np * Kp * 4, 256);
    char *base = static_cast<char *>(scratch) + kHeadBytes;
    float *a_big = reinterpret_cast<float *>(base);
    float *a_small = reinterpret_cast<float *>(base + a_bytes);
    float *b_big = reinterpret_cast<float *>(base + 2 * a_bytes);
    float *b_small = reinterpret_cast<float *>(base + 2 * a_bytes + b_bytes);
    // The pre-pass writes every element of the padded operand buffers (the
    // padding as zeros), so nothing left in the scratch by an earlier call is
    // read by this one.
    st = ok(launch_split_rows(A, lda, static_cast<int>(M), static_cast<int>(K),
                              static_cast<int>(Mp), static_cast<int>(Kp), a_big, a_small,
                              (lda % 4 == 0) && aligned16(A), stream));
    if (st == PHOBOS_OK)
      st = ok(launch_split_cols(B, ldb, static_cast<int>(K), static_cast<int>(N),
                                static_cast<int>(Np), static_cast<int>(Kp), b_big, b_small,
                                stream));
    TcArgs t{};
    if (st == PHOBOS_OK) st = kmajor_map(&t.tmap_ab, a_big, Mp, Kp, kBM);
    if (st == PHOBOS_OK) st = kmajor_map(&t.tmap_as, a_small, Mp, Kp, kBM);
    if (st == PHOBOS_OK) st = kmajor_map(&t.tmap_bb, b_big, Np, Kp, bn);
    if (st == PHOBOS_OK) st = kmajor_map(&t.tmap_bs, b_small, Np, Kp, bn);
    if (st == PHOBOS_OK) {
      t.C = C;
      t.ldc = ldc;
      t.M = static_cast<int>(M);
      t.N = static_cast<int>(N);
      t.k_block0 = 0;
      t.k_blocks = static_cast<int>(Kp / kBK);
      t.tiles_m = static_cast<int>(Mp / kBM);
      t.tiles_n = static_cast<int>(Np / bn);
      int64_t gm = kSuper / kBM;
      t.group_m = static_cast<int>(gm > t.tiles_m ? t.tiles_m : gm);
      t.alpha = alpha;
      t.beta = beta;
      t.vec_c = (ldc % 4 == 0) && aligned16(C);
      t.promote_blocks = promote_blocks_for(K);  // the rule of every split-TF32 call
      t.sm_count = g_sm_count[dev];
      t.err = status_word;
      st = ok(launch_tc(t, 3, bn, tc_max_stages(3, bn), stream));
    }
  }
  if (st == PHOBOS_OK) {
    const char *dbg = std::getenv("PHOBOS_DEBUG_SYNC");
    if (dbg && dbg[0] && std::strcmp(dbg, "0") != 0) {
      int word = 0;
      if (cudaStreamSynchronize(stream) != cudaSuccess ||
          cudaMemcpy(&word, status_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PHOBOS_ERR_CUDA;
      if (word != 0) {
        if (cudaMemset(status_word, 0, sizeof(int)) != cudaSuccess) return PHOBOS_ERR_CUDA;
        return PHOBOS_ERR_TIMEOUT;
      }
    }
  }
  return st;
}
