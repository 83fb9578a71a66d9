/*
 * libphobos_gemm -- fp32 GEMM  C = alpha * A * B + beta * C  on one GB300
 * (sm_103a), as a C ABI.
 *
 * The operation is the tiled matrix multiply that the Phobos pages use as
 * their running example: the `matmul` kernel of the "@cluster" attribute page
 * (phobos-lang.dev, "What the cluster compiler accepts": an accumulator tile
 * summed over a K loop, stored once as alpha * acc + beta * c_old) and the
 * "Matrix Multiplication" section of "Show HN: Phobos - A tiny scale-free
 * kernel language with tile-DAG support" (C = alpha A B + beta C with A of
 * M x K, B of K x N, C of M x N).
 *
 * Conventions shared by every entry point:
 *  - Layout: all matrices are row-major.  A[i][k] = A[i*lda + k],
 *    B[k][j] = B[k*ldb + j], C[i][j] = C[i*ldc + j].  Any size and leading
 *    dimension is accepted (the pages' multiple-of-four restriction is lifted)
 *    provided lda >= max(1,K), ldb >= max(1,N), ldc >= max(1,N).
 *  - Degenerate sizes: M == 0 or N == 0 is a no-op.  K == 0 or alpha == 0
 *    gives C = beta * C (an empty sum is zero).  beta == 0 means C is not read
 *    (so NaN or garbage in C is overwritten), following the init leaf of the
 *    cluster split, which "zeroes the output super-tile, or scales it by beta".
 *  - Ownership: A, B and C are caller-owned device pointers; the library never
 *    frees or retains them.  A and B are read only.  C must not overlap A or B
 *    (not checked; the result is undefined).  The library owns its workspace
 *    (per device and stream, grown on demand, released by phobos_release).
 *  - Execution: asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream).  The call returns after enqueueing.
 *    The current device must be compute capability 10.3 (sm_103); there is no
 *    CPU fallback.
 *  - Errors: a phobos_status_t; nothing is enqueued when the status is not
 *    PHOBOS_OK, except that PHOBOS_ERR_CUDA may follow a partial enqueue.
 *    Device-side bounded waits that expire set a device status word; it is
 *    read (and cleared) by phobos_check_device, and by every call when the
 *    environment variable PHOBOS_DEBUG_SYNC=1 is set.  For testing that path,
 *    PHOBOS_TEST_WITHHOLD_LOAD=1 makes the tensor-core kernel skip its first
 *    operand load: its wait on that load expires after about two seconds, the
 *    kernel stops without writing C, and the status word reports it.
 *    PHOBOS_TEST_WITHHOLD_SPLIT=1 does the same through the in-kernel panel
 *    split (a_split = 3): the first split item is never marked done.
 *  - Thread safety: calls may come from several host threads.  Calls that
 *    share one stream are ordered by it; calls on different streams use
 *    different workspaces.
 */
#ifndef PHOBOS_GEMM_H
#define PHOBOS_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PHOBOS_OK = 0,
  PHOBOS_ERR_INVALID_VALUE = 1, /* negative size, small leading dimension, NULL pointer, bad plan */
  PHOBOS_ERR_UNSUPPORTED = 2,   /* device is not sm_103, or the plan cannot run this shape */
  PHOBOS_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
  PHOBOS_ERR_OUT_OF_MEMORY = 4, /* the workspace could not be allocated */
  PHOBOS_ERR_TIMEOUT = 5        /* a device-side bounded wait expired (see phobos_check_device) */
} phobos_status_t;

/* How the products are formed.  DEFAULT picks FFMA for small problems and
 * split TF32 (3xTF32) on the tensor cores otherwise.
 *
 * FP16 and BF16 are the reduced-precision tensor-core mode of "Show HN:
 * Phobos", section "Side-quest: Cheating": the fp32 inputs are cast to a
 * 16-bit type before the tensor cores, the products are accumulated in fp32,
 * and the result is fp32.  Here the pre-pass rounds A and B to nearest
 * (ties to even).  Each product of two 16-bit values is exact in fp32.  The
 * result is therefore alpha * sum(r(a) * r(b)) + beta * C up to the fp32
 * accumulation, with r() the rounding (relative error <= 2^-11 for fp16,
 * 2^-8 for bf16).  This is not the fp32 accuracy of the other modes: it is
 * the mode the pages call apples to oranges.  fp16 keeps 5 exponent bits:
 * inputs beyond +-65504 become infinities, and tiny inputs lose precision.
 * bf16 keeps fp32's exponent range. */
typedef enum {
  PHOBOS_MATH_DEFAULT = 0,
  PHOBOS_MATH_3XTF32 = 1, /* a = a_big + a_small, three tf32 products, fp32-level accuracy */
  PHOBOS_MATH_TF32 = 2,   /* one tf32 product per term (10-bit mantissa operands) */
  PHOBOS_MATH_FFMA = 3,   /* fp32 fused multiply-add on the CUDA cores */
  PHOBOS_MATH_FP16 = 4,   /* inputs rounded to fp16, fp32 accumulation on the tensor cores */
  PHOBOS_MATH_BF16 = 5    /* inputs rounded to bf16, fp32 accumulation on the tensor cores */
} phobos_math_t;

typedef enum {
  PHOBOS_PATH_FFMA = 1,
  PHOBOS_PATH_TF32 = 2,
  PHOBOS_PATH_3XTF32 = 3,
  PHOBOS_PATH_FP16 = 4,
  PHOBOS_PATH_BF16 = 5
} phobos_path_t;

/*
 * A plan: which kernel runs and how the problem is tiled.
 *  path            phobos_path_t.
 *  tile_m, tile_n  output tile of one CTA (tile_m = 256 for a 2-CTA pair).
 *  tile_k          K depth of one shared-memory stage: 16 for FFMA, 32 for
 *                  the tf32 paths, 64 for FP16 and BF16 (128 bytes of K
 *                  either way on the tensor cores).
 *  cluster_m/_n    CTAs per thread-block cluster along M and N: 1 x 1, 2 x 1
 *                  (a CTA pair), or 2 x 2 with multicast.
 *  stages          depth of the shared-memory ring.
 *  multicast       0 (the planner's choice) or 1: split TF32 and TF32 with CTA
 *                  pairs only (tile 256 x 256, cluster 2 x 2, deepest ring, A
 *                  split by the pre-pass).  A cluster then holds two CTA pairs
 *                  that compute horizontally adjacent tiles; each pair
 *                  TMA-loads half of the A rows both need and multicasts it
 *                  to both pairs, so A crosses from L2 once per two tiles.
 *                  Results equal the pair kernel's bit for bit on tiles
 *                  computed whole.  Only as many clusters as fit on the GPU
 *                  at once are launched (36 on GB300, i.e. 144 of the 152
 *                  SMs), so the planner leaves it off: measured against the
 *                  pair kernel it is 5 % slower at 8192^3, 10 % at 4096^3 and
 *                  even at 16384^3.  Multicast is a one-GPU option: its
 *                  tensor maps cover this GPU's own memory only, and a plan
 *                  with multicast = 1 is refused (PHOBOS_ERR_UNSUPPORTED)
 *                  in a process that is one rank of a multi-process job
 *                  (environment WORLD_SIZE or LOCAL_WORLD_SIZE above 1).
 *  super_m/_n      super-tile: the output tiles are walked super-tile by
 *                  super-tile (an L2-locality group on one GPU).  The planner
 *                  takes 4096, the pages' smallest super-tile, and super_m =
 *                  2048 when the kernel splits A and B itself (a_split 3) and
 *                  M <= 4096, so that the first wave of tiles needs fewer
 *                  A panels split at once.
 *  super_k         K chunk of the cluster split: super_k < K runs an init
 *                  leaf C = beta*C then one step leaf C += alpha*A_c*B_c per
 *                  chunk (results equal up to rounding order).
 *  workspace_bytes device workspace of the operand pre-pass, for A and B
 *                  (less when A is split inside the kernel; the tail split
 *                  below adds at most one tile of partial sums per CTA pair,
 *                  about 20 MB on GB300, plus flags).
 *  tail_split      FFMA path with 64 x 64 tiles: K slices per tile, summed
 *                  inside a thread-block cluster through distributed shared
 *                  memory (0 = enough to fill the SMs, 1 = off, 2..8).
 *                  Tensor-core paths: each tile of the last, partial wave of
 *                  the persistent grid is cut along K into pieces for the
 *                  CTAs (pairs) that would otherwise idle (0 = automatic:
 *                  about sqrt(K / 80) pieces, as many as the idle CTAs
 *                  allow, at most 8, or, for K <= 4096 when those whole
 *                  pieces would leave a fifth of the CTAs idle, one more
 *                  piece per tile; 1 = off; S = 2..8: S pieces per tile,
 *                  or, when fewer than S CTAs per tail tile are free, the
 *                  tail's K blocks dealt evenly to every CTA).  Every piece
 *                  spans at least K = 128.  Results are equal up to rounding
 *                  order and deterministic.
 *  a_split         tensor-core paths: where A (and B) are split into tf32
 *                  big/small.
 *                   0 = chosen per call: 2 when N <= 1536 and A's rows are
 *                       16-byte aligned (a separate pass over A would cost a
 *                       large share of the GEMM there), else 3 for split TF32
 *                       with CTA pairs, else 1.
 *                   1 = a pre-pass kernel splits A and B into the workspace
 *                       before the GEMM kernel starts.
 *                   2 = A is split in shared memory inside the GEMM kernel,
 *                       B by the pre-pass; needs lda % 4 == 0 and a
 *                       16-byte-aligned A, else PHOBOS_ERR_UNSUPPORTED.
 *                   3 = the GEMM kernel splits A and B into the workspace
 *                       itself, overlapped with its own tiles: two extra
 *                       warps per CTA split the panels in the order the tiles
 *                       first need them, and each CTA waits only for the
 *                       panels of its current tile; tf32 CTA pairs without
 *                       multicast only (else PHOBOS_ERR_UNSUPPORTED), any
 *                       leading dimension and alignment.
 *                  Identical results whichever is used.  FP16 and BF16 always
 *                  convert A in the pre-pass (0 or 1).
 *  clc             split-TF32 CTA pairs without multicast or a_split = 2:
 *                  1 = Cluster Launch Control deals the tiles ("Clusters et
 *                  DSMEM", 3.7, Cluster Launch Control).  The grid holds one
 *                  CTA pair per output tile; each resident pair starts on its
 *                  own tile and then takes tiles from the hardware's queue of
 *                  pairs not yet launched (it cancels their launch), so pairs
 *                  that finish early, or start late because other work holds
 *                  SMs, take more tiles.  With a_split = 0 the kernel splits
 *                  A and B itself.  tail_split cuts the tiles of the last
 *                  partial wave into K pieces (0: enough to give every
 *                  resident pair work, at most 8, each at least 4 k blocks;
 *                  1: off; 2..8: that many), each dealt like a tile: every
 *                  piece leaves its partial sum in the workspace and the
 *                  last to finish adds them in K order and stores the tile,
 *                  so no piece waits for another and the result is
 *                  deterministic.  With tail_split = 1 each tile's result
 *                  equals the static walk's (tail_split = 1) bit for bit.
 *                  0 (the planner's choice) = a static persistent walk: one
 *                  pair per SM pair, tiles strided over the pairs.  Other
 *                  plans with clc = 1 give PHOBOS_ERR_UNSUPPORTED.
 *  FP16 and BF16 plans run the tensor-core kernel with its deepest stage ring
 *  only (stages must equal the planner's value).
 */
typedef struct {
  int32_t path;
  int32_t tile_m, tile_n, tile_k;
  int32_t cluster_m, cluster_n;
  int32_t stages;
  int32_t multicast;
  int64_t super_m, super_n, super_k;
  size_t workspace_bytes;
  int32_t tail_split;
  int32_t a_split;
  int32_t clc;
} phobos_gemm_plan_t;

/*
 * Choose a plan for an M x N x K problem with the given leading dimensions and
 * math mode (host logic only; no device call).  Tile choice follows the
 * pages' split into CTA tiles (@autotune) and super-tiles (@cluster): "@cluster"
 * attribute page, "A minimal kernel" and "What runs today" (a dimension takes
 * its first value without tuning); "Show HN: Phobos", "Clustering".
 * Errors: PHOBOS_ERR_INVALID_VALUE for bad sizes/leading dimensions, an
 * unknown math mode or out == NULL; PHOBOS_ERR_UNSUPPORTED when M, N or K
 * exceeds 2^31 - 1024 (the kernels index rows and columns with 32-bit ints).
 */
phobos_status_t phobos_gemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda,
                                 int64_t ldb, int64_t ldc, phobos_math_t math,
                                 phobos_gemm_plan_t *out);

/*
 * C = alpha * A * B + beta * C with the default math mode and an automatic
 * plan.  See the conventions above for layout, ownership and errors.
 * Definition: "@cluster" attribute page, the `matmul` listing; "Show HN:
 * Phobos", "Matrix Multiplication".
 */
phobos_status_t phobos_sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                             const float *A, int64_t lda, const float *B,
                             int64_t ldb, float beta, float *C, int64_t ldc,
                             void *stream);

/*
 * As phobos_sgemm with an explicit math mode and, optionally, a plan (NULL =
 * automatic).  A caller-supplied plan is validated against the shape and the
 * mode before anything is enqueued: PHOBOS_ERR_INVALID_VALUE if a field is out
 * of range for it, PHOBOS_ERR_UNSUPPORTED for a cluster shape this build does
 * not run (see cluster_m/_n and multicast above).  A plan with
 * super_k < K runs the cluster split of the "@cluster" page ("the init leaf
 * zeroes the output super-tile, or scales it by beta, and the step leaf adds
 * one chunk of K per launch"; "Show HN: Phobos", "Clustering": the beta term
 * is hoisted into the init leaf and each chunk applies an implicit beta of 1).
 */
phobos_status_t phobos_sgemm_ex(int64_t M, int64_t N, int64_t K, float alpha,
                                const float *A, int64_t lda, const float *B,
                                int64_t ldb, float beta, float *C, int64_t ldc,
                                void *stream, phobos_math_t math,
                                const phobos_gemm_plan_t *plan);

/*
 * Host-buffer form: A, B and C are HOST pointers (pinned memory gives the
 * fastest copies).  The call copies A, B (and C when beta != 0) to device
 * buffers owned by the library, runs the GEMM on `stream`, copies C back and
 * synchronizes `stream` before returning.  Problems on the tensor-core path
 * with M >= 2048 run as up to 8 row bands on two internal copy streams so
 * that the copies of later bands overlap the compute of earlier ones; when
 * the kernel splits its own operands and K >= 2048, the first band runs in K
 * chunks that each start as soon as their rows of B have arrived.  Same
 * layout and errors as phobos_sgemm_ex, plus PHOBOS_ERR_OUT_OF_MEMORY for
 * the staging buffers.  Calls are serialised inside the library.
 */
phobos_status_t phobos_sgemm_host(int64_t M, int64_t N, int64_t K, float alpha,
                                  const float *A, int64_t lda, const float *B,
                                  int64_t ldb, float beta, float *C, int64_t ldc,
                                  void *stream, phobos_math_t math);

/*
 * Synchronize `stream`, then read and clear the device status words of the
 * current device (the library's, and the no-allocation entry point's once it
 * has run there).  PHOBOS_ERR_TIMEOUT if a kernel's bounded wait expired since
 * the last check, PHOBOS_ERR_CUDA if synchronization failed, else PHOBOS_OK.
 */
phobos_status_t phobos_check_device(void *stream);

/*
 * Instrumentation.  With non-NULL events (cudaEvent_t passed as void*), every
 * following call of this library on any stream records `start` on its stream
 * just before its main GEMM kernel (after the operand pre-pass, if any) and
 * `stop` just after the last main kernel, so that cudaEventElapsedTime gives
 * the main kernel's device time.  NULL, NULL switches recording off.  The
 * events stay owned by the caller.  Always PHOBOS_OK.
 */
phobos_status_t phobos_set_timing_events(void *start, void *stop);

/*
 * Instrumentation: the SM clock the tensor-core GEMM kernels ran at.  While
 * timing events are set (phobos_set_timing_events), thread 0 of the first
 * CTA of every tensor-core GEMM launch on the current device adds the SM
 * cycles (clock64) and the nanoseconds (%globaltimer) of its CTA's lifetime
 * to a device-side sum.  This call waits for the current device, stores the
 * sum's cycles per microsecond in *mhz (0 when no launch was counted since the
 * last call) and clears the sum.  Under a power cap the SM clock changes
 * within milliseconds, faster than nvidia-smi samples it; this is the clock of
 * the kernels themselves.  Returns PHOBOS_ERR_INVALID_VALUE for a NULL mhz,
 * PHOBOS_ERR_CUDA if a copy fails.
 */
phobos_status_t phobos_kernel_clock_mhz(double *mhz);

/*
 * Instrumentation: the output tiles that Cluster Launch Control launches
 * (plan clc = 1) on the current device took from cancelled pair launches
 * while timing events were set, since the last call.  Waits for the device,
 * stores the count in *tiles and clears it.  A grid of T tiles of which P
 * pairs start at once hands out T - P tiles this way.  Returns
 * PHOBOS_ERR_INVALID_VALUE for a NULL tiles, PHOBOS_ERR_CUDA if a copy fails.
 */
phobos_status_t phobos_kernel_clc_tiles(uint64_t *tiles);

/* Number of CUDA kernels this library has launched since it was loaded. */
uint64_t phobos_kernel_launches(void);

/* Free every workspace and staging buffer the library holds (all devices).
 * Must not be called while a call of this library is running on any stream. */
phobos_status_t phobos_release(void);

/*
 * No-allocation form of the split-TF32 (3xTF32) GEMM.  The pages have no
 * counterpart; it exists for callers that may not allocate device memory
 * themselves: a serving process whose device memory was reserved up front by
 * its own allocator (a caching allocator or an engine that claimed most of
 * HBM at start-up, where a new cudaMalloc can fail or fragment the pool), and
 * latency-critical loops that cannot take the implicit synchronisation and
 * latency of cudaMalloc/cudaFree.
 *
 * Same arguments, layout and ownership as phobos_sgemm_ex with
 * PHOBOS_MATH_3XTF32, and a result within the same 3xTF32 bound: the same
 * operand split and TMEM partial lengths, but single-CTA tiles without the
 * tail split, so the rounding order (not the accuracy) may differ from the
 * automatic plan's.  The call allocates nothing:
 * no cudaMalloc, cudaMallocAsync, cudaFree or other allocating routine.  Its
 * scratch is one fixed device array inside the library
 * (PHOBOS_NOALLOC_SCRATCH_BYTES of split operands plus a status word).  Every
 * GPU that loads the library holds that array until the process exits.
 *  - Limit: the split operands take 8 * (Mp + Np) * Kp bytes, where
 *    Mp = M rounded up to 128, Np = N rounded up to 128 (N <= 128) or 256,
 *    and Kp = K rounded up to 32.  Larger problems return
 *    PHOBOS_ERR_UNSUPPORTED with nothing enqueued.
 *    2048 x 2048 x 2048 fits exactly.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (with that device current).  Make that first call before any
 *    stream capture.
 *  - Sharing: every call, on every stream, uses the same array, and the array
 *    keeps what the last call left there.  The operand pre-pass overwrites
 *    every element a call reads, padding included.  Calls whose work overlaps
 *    on the GPU (for example on two streams at once) race on the array:
 *    serialise them.
 *  - Errors: as phobos_sgemm_ex, including PHOBOS_ERR_UNSUPPORTED when M, N
 *    or K exceeds 2^31 - 1024.  An expired device-side wait is recorded in
 *    the array's status word.  phobos_check_device reads and clears that word
 *    beside the library's own; with PHOBOS_DEBUG_SYNC=1 every call also
 *    synchronises and reports it as PHOBOS_ERR_TIMEOUT.
 */
#define PHOBOS_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
phobos_status_t phobos_sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                     const float *A, int64_t lda, const float *B,
                                     int64_t ldb, float beta, float *C, int64_t ldc,
                                     void *stream);

/* A static, NUL-terminated description of a status code. */
const char *phobos_status_string(phobos_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* PHOBOS_GEMM_H */
