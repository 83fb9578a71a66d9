/*
 * phobos_cluster.h -- super-tile cluster runtime for the fp32 GEMM
 * C = alpha*A*B + beta*C on nodes that share storage.
 *
 * What the runtime computes is the K-chunked form of the GEMM from "Show HN:
 * Phobos", section "Matrix Multiplication" and its cluster-IR listing. The
 * output is cut into super-tiles of SUPER_M x SUPER_N. Each one is seeded
 * with beta*C_old (the init leaf), then accumulated over K chunks of SUPER_K
 * with C += alpha*A_chunk*B_chunk (the step leaves), then written back.
 *
 * How the work is planned and run follows the "@cluster" attribute page,
 * sections "What runs today" and "Cost and interactions", and "Show HN:
 * Phobos", sections "The DAG Compiler" and "The Cluster Prototype":
 *   - a scheduler plans every output super-tile and deals the super-tiles
 *     round robin over the nodes by their row-major index;
 *   - each node gets its own instruction list (ALLOC, LOAD, COMPUTE, STORE,
 *     FREE), and a backward pass over the dependency graph places each FREE
 *     after the last use of its tile;
 *   - a pod runs its list as dependencies complete;
 *   - when a node stops heart-beating, the scheduler re-plans the outputs it
 *     had not stored onto the nodes that are left.
 *
 * This header is the native core of that runtime: the planner (pure host
 * logic) and the pod executor (device arena, storage I/O, leaves through
 * phobos_sgemm_ex). The control plane that moves segments, heartbeats and
 * completion marks between processes lives in the Python package
 * (language_fp32_gemm_gb300.cluster).
 *
 * Storage: a tensor is a raw little-endian fp32 file holding a row-major
 * matrix with no header (file:// is the only storage the pages describe).
 *
 * Every function returns PHOBOS_OK (0) on success or a phobos_status_t code.
 */
#ifndef PHOBOS_CLUSTER_H_
#define PHOBOS_CLUSTER_H_

#include <stddef.h>
#include <stdint.h>

#include "phobos_gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Instruction kinds. The pages' COMPUTE is split into its two leaves. */
typedef enum {
  PHOBOS_CL_ALLOC = 0, /* reserve a tile buffer in the node's device arena */
  PHOBOS_CL_LOAD = 1,  /* storage -> host staging -> device buffer */
  PHOBOS_CL_INIT = 2,  /* init leaf: C_tile = beta*C_tile (zeros when beta == 0) */
  PHOBOS_CL_STEP = 3,  /* step leaf: C_tile += alpha * A_tile * B_tile */
  PHOBOS_CL_STORE = 4, /* device buffer -> storage (two-phase, see phobos_pod_run) */
  PHOBOS_CL_FREE = 5   /* return the buffer to the arena after its last use */
} phobos_cl_op_t;

typedef enum { PHOBOS_CL_A = 0, PHOBOS_CL_B = 1, PHOBOS_CL_C = 2 } phobos_cl_tensor_t;

/* A problem and how to plan it. Sizes are element counts. */
typedef struct {
  int64_t M, N, K;
  float alpha, beta;
  int32_t nodes; /* nodes of the cluster, numbered 0 .. nodes-1 */
  /* Super-tile search space per axis, as in @cluster(NAME in [lo, hi]): lo
   * and hi are inclusive bounds searched in doubling steps. Without
   * autotune each axis takes lo. A value above the problem extent is cut to
   * the extent. */
  int64_t super_lo[3]; /* M, N, K */
  int64_t super_hi[3];
  int32_t autotune;           /* 0: first value of each axis; 1: model-ranked search */
  int64_t node_budget_bytes;  /* device memory each node may hold at once */
  double node_tflops;         /* cost model: leaf rate per node */
  double storage_gbs;         /* cost model: storage read/write rate per node */
} phobos_cl_job_t;

/* One instruction of a node's segment. Buffers are named by the index of the
 * ALLOC instruction that reserved them. */
typedef struct {
  int32_t op;     /* phobos_cl_op_t */
  int32_t tensor; /* phobos_cl_tensor_t of the tile this instruction handles */
  uint64_t tile;  /* deterministic tile id, see phobos_cl_tile_id */
  int64_t row0, col0, rows, cols; /* the tile's region of its tensor */
  int32_t buf;    /* ALLOC: itself; LOAD/INIT/STORE/FREE: the buffer; STEP: the C buffer */
  int32_t buf_a, buf_b; /* STEP: the A and B buffers; -1 otherwise */
  int32_t dep_begin, dep_count; /* this instruction's dependencies in the segment's list */
} phobos_cl_instr_t;

/* Deterministic tile id: tensor in bits 62..63, K chunk (A, B) or output
 * version (C) in bits 42..61, row index of the super-tile grid in bits 21..41,
 * column index in bits 0..20. Equal ids mean equal tiles on every node and in
 * every plan, so re-running a lost part of the graph reproduces its tiles. */
uint64_t phobos_cl_tile_id(int32_t tensor, int64_t version, int64_t row, int64_t col);

typedef struct phobos_cl_plan phobos_cl_plan_t;

/* Plan `job`. `outputs` lists the output super-tiles (row-major indices) to
 * plan, or is NULL for all of them. `live` lists the nodes that may take
 * work, or is NULL for all nodes. Output super-tiles are dealt round robin
 * over `live` in increasing index order. The chosen super-tile sizes are
 * written to `super_out` (M, N, K) when it is not NULL. Errors:
 * PHOBOS_ERR_INVALID_VALUE for bad sizes, ranges or node lists;
 * PHOBOS_ERR_OUT_OF_MEMORY when no candidate fits node_budget_bytes. The plan
 * is owned by the caller and released with phobos_cl_plan_free. */
phobos_status_t phobos_cl_plan(const phobos_cl_job_t *job, const int32_t *outputs,
                               int64_t n_outputs, const int32_t *live, int32_t n_live,
                               int64_t super_out[3], phobos_cl_plan_t **plan);

void phobos_cl_plan_free(phobos_cl_plan_t *plan);

/* Size of node `node`'s segment, then the segment itself as a self-contained
 * byte blob (header, instructions, dependency list) that phobos_pod_run
 * takes. `bytes` must be at least the size returned. */
phobos_status_t phobos_cl_segment_size(const phobos_cl_plan_t *plan, int32_t node, size_t *bytes);
phobos_status_t phobos_cl_segment_write(const phobos_cl_plan_t *plan, int32_t node, void *out,
                                        size_t bytes);

/* Figures of a node's segment: instruction count, the count of each op
 * (indexed by phobos_cl_op_t, 6 entries), the peak bytes held in the arena when
 * the segment runs in list order, and the bytes it loads and stores. */
typedef struct {
  int64_t instrs;
  int64_t op_count[6];
  int64_t peak_bytes;
  int64_t load_bytes, store_bytes;
  int64_t flops;
  int64_t outputs; /* output super-tiles */
} phobos_cl_segment_info_t;

phobos_status_t phobos_cl_segment_info(const void *segment, size_t bytes,
                                       phobos_cl_segment_info_t *info);

/* Instruction `i` of a segment blob, and dependency `j` of its list. */
phobos_status_t phobos_cl_segment_instr(const void *segment, size_t bytes, int64_t i,
                                        phobos_cl_instr_t *out);
phobos_status_t phobos_cl_segment_dep(const void *segment, size_t bytes, int64_t j, int32_t *out);

/* Where a pod runs its leaves. */
typedef enum {
  PHOBOS_POD_CUDA = 0, /* arena in device memory of the current device; leaves via phobos_sgemm_ex */
  PHOBOS_POD_HOST = 1  /* arena in host memory; leaves via the host_gemm hook (host-logic tests) */
} phobos_pod_device_t;

/* Callbacks into the control plane. Each returns 0 to continue; anything else
 * stops the pod with PHOBOS_ERR_INVALID_VALUE after the current instruction. */
typedef struct {
  void *ctx;
  /* STORE, phase 1 done: the tile is complete in its side file. */
  int (*on_staged)(void *ctx, uint64_t tile);
  /* STORE, phase 2 done: the tile is in the output file. */
  int (*on_stored)(void *ctx, uint64_t tile);
  /* PHOBOS_POD_HOST only: C = alpha*A*B + beta*C on host memory (row-major). */
  int (*host_gemm)(void *ctx, int64_t m, int64_t n, int64_t k, float alpha, const float *a,
                   int64_t lda, const float *b, int64_t ldb, float beta, float *c, int64_t ldc);
} phobos_pod_hooks_t;

typedef struct {
  int32_t device;            /* phobos_pod_device_t */
  int64_t arena_bytes;       /* arena size; at least the segment's peak_bytes */
  const char *paths[3];      /* storage files of A, B and C */
  int64_t staging_bytes;     /* host staging chunk per transfer (0: 32 MiB) */
  void *stream;              /* PHOBOS_POD_CUDA: cudaStream_t for the leaves (NULL: a new one) */
} phobos_pod_config_t;

/* Run one segment to completion on this process's current device.
 *
 * Order: an instruction starts once its dependencies have. Device work is
 * chained with events, so LOADs of later tiles overlap earlier leaves
 * whenever the arena has room. ALLOCs start in list order, so the peak never
 * exceeds the segment's list-order peak.
 *
 * STORE is two-phase:
 *   1. the tile is written to "<C path>.tile-<id as 16 hex digits>", then
 *      on_staged is called;
 *   2. the tile is written into the C file, on_stored is called, and the
 *      side file is removed.
 * A tile is therefore either untouched in C, complete in its side file, or
 * complete in C, whenever the process stops.
 *
 * Errors:
 *   - PHOBOS_ERR_INVALID_VALUE: a malformed segment or a hook that asked to stop;
 *   - PHOBOS_ERR_OUT_OF_MEMORY: the arena is too small or fragmented;
 *   - PHOBOS_ERR_CUDA: a storage or CUDA failure;
 *   - or the status of a failed phobos_sgemm_ex. */
phobos_status_t phobos_pod_run(const void *segment, size_t bytes, const phobos_pod_config_t *cfg,
                               const phobos_pod_hooks_t *hooks);

#ifdef __cplusplus
}
#endif

#endif /* PHOBOS_CLUSTER_H_ */
