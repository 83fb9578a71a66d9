// Pod executor of the super-tile cluster runtime: runs one node's segment.
//
// "@cluster" attribute page, "What runs today": a pod runs its instructions
// as their dependencies complete. "Show HN: Phobos", "Where Does This Fit
// In?": there is no barrier instruction; dependencies are the only
// synchronisation, and a tile's next LOADs, which do not depend on the
// previous leaf, are prefetched.
//
// Here, on one GB300:
//   - one device arena per pod (first-fit, 256-byte granules), reserved once;
//   - LOAD: storage rows -> pinned staging (two chunks in flight) -> device on a copy stream;
//   - INIT and STEP: phobos_sgemm_ex on the compute stream, after the events of their inputs;
//   - STORE: device -> pinned staging -> side file, then into the C file (two-phase);
//   - FREE: the range goes back to the arena once every user's event has completed.
// ALLOCs start in list order, so the arena never holds more than the
// segment's list-order peak. Any LOAD that finds room runs ahead of the
// leaves that precede it in the list.

#include <cuda_runtime.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <cerrno>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <thread>
#include <vector>

#include "../../include/phobos_cluster.h"
#include "cluster_internal.h"
#include "internal.h"

namespace phobos {
namespace cluster {
namespace {

constexpr int64_t kGranule = 256;
constexpr int64_t kDefaultStaging = int64_t(32) << 20;

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// First-fit allocator over offsets [0, size).
class Arena {
 public:
  explicit Arena(int64_t size) { free_[0] = size; }
  bool alloc(int64_t bytes, int64_t *off) {
    bytes = round_up(bytes, kGranule);
    for (auto it = free_.begin(); it != free_.end(); ++it) {
      if (it->second < bytes) continue;
      *off = it->first;
      const int64_t rest = it->second - bytes, start = it->first + bytes;
      free_.erase(it);
      if (rest > 0) free_[start] = rest;
      return true;
    }
    return false;
  }
  void release(int64_t off, int64_t bytes) {
    bytes = round_up(bytes, kGranule);
    auto it = free_.emplace(off, bytes).first;
    auto next = std::next(it);
    if (next != free_.end() && it->first + it->second == next->first) {
      it->second += next->second;
      free_.erase(next);
    }
    if (it != free_.begin()) {
      auto prev = std::prev(it);
      if (prev->first + prev->second == it->first) {
        prev->second += it->second;
        free_.erase(it);
      }
    }
  }

 private:
  std::map<int64_t, int64_t> free_;
};

// Whole-range positional file I/O (retries short transfers).
bool pread_all(int fd, void *dst, int64_t bytes, int64_t off) {
  char *p = static_cast<char *>(dst);
  while (bytes > 0) {
    const ssize_t n = ::pread(fd, p, static_cast<size_t>(bytes), off);
    if (n < 0 && errno == EINTR) continue;
    if (n <= 0) return false;
    p += n;
    off += n;
    bytes -= n;
  }
  return true;
}

bool pwrite_all(int fd, const void *src, int64_t bytes, int64_t off) {
  const char *p = static_cast<const char *>(src);
  while (bytes > 0) {
    const ssize_t n = ::pwrite(fd, p, static_cast<size_t>(bytes), off);
    if (n < 0 && errno == EINTR) continue;
    if (n <= 0) return false;
    p += n;
    off += n;
    bytes -= n;
  }
  return true;
}

// Rows [r, r + nr) of a tile whose rows live at (row0 + r) * ld + col0 in a
// row-major file; the host side is packed (row stride = cols).
bool read_rows(int fd, int64_t ld, int64_t row0, int64_t col0, int64_t cols, int64_t r, int64_t nr,
               float *dst) {
  if (cols == ld) return pread_all(fd, dst, 4 * nr * cols, 4 * ((row0 + r) * ld + col0));
  for (int64_t i = 0; i < nr; ++i)
    if (!pread_all(fd, dst + i * cols, 4 * cols, 4 * ((row0 + r + i) * ld + col0))) return false;
  return true;
}

bool write_rows(int fd, int64_t ld, int64_t row0, int64_t col0, int64_t cols, int64_t r, int64_t nr,
                const float *src) {
  if (cols == ld) return pwrite_all(fd, src, 4 * nr * cols, 4 * ((row0 + r) * ld + col0));
  for (int64_t i = 0; i < nr; ++i)
    if (!pwrite_all(fd, src + i * cols, 4 * cols, 4 * ((row0 + r + i) * ld + col0))) return false;
  return true;
}

std::string side_path(const char *c_path, uint64_t tile) {
  char hex[17];
  std::snprintf(hex, sizeof(hex), "%016llx", static_cast<unsigned long long>(tile));
  return std::string(c_path) + ".tile-" + hex;
}

enum State { kPending = 0, kIssued = 1, kDone = 2 };

class Pod {
 public:
  Pod(const SegmentHeader &h, const phobos_cl_instr_t *recs, const int32_t *deps,
      const phobos_pod_config_t &cfg, const phobos_pod_hooks_t *hooks)
      : h_(h), recs_(recs), deps_(deps), cfg_(cfg), hooks_(hooks),
        cuda_(cfg.device == PHOBOS_POD_CUDA), arena_(cfg.arena_bytes),
        state_(h.n_instr, kPending), offset_(h.n_instr, -1), event_(h.n_instr, nullptr) {
    staging_bytes_ = cfg.staging_bytes > 0 ? cfg.staging_bytes : kDefaultStaging;
    ld_[PHOBOS_CL_A] = h.K;
    ld_[PHOBOS_CL_B] = h.N;
    ld_[PHOBOS_CL_C] = h.N;
    extent_[PHOBOS_CL_A][0] = h.M; extent_[PHOBOS_CL_A][1] = h.K;
    extent_[PHOBOS_CL_B][0] = h.K; extent_[PHOBOS_CL_B][1] = h.N;
    extent_[PHOBOS_CL_C][0] = h.M; extent_[PHOBOS_CL_C][1] = h.N;
  }

  ~Pod() {
    if (cuda_) {
      if (copy_in_) cudaStreamSynchronize(copy_in_);
      if (copy_out_) cudaStreamSynchronize(copy_out_);
      if (compute_) cudaStreamSynchronize(compute_);
      for (cudaEvent_t e : event_)
        if (e) cudaEventDestroy(e);
      for (int i = 0; i < 2; ++i) {
        if (stage_ev_[i]) cudaEventDestroy(stage_ev_[i]);
        if (stage_in_[i]) cudaFreeHost(stage_in_[i]);
      }
      if (stage_out_) cudaFreeHost(stage_out_);
      if (copy_in_) cudaStreamDestroy(copy_in_);
      if (copy_out_) cudaStreamDestroy(copy_out_);
      if (compute_ && own_compute_) {
        // the leaves' workspace is cached per stream: free it with the stream
        phobos::release_stream_workspace(compute_);
        cudaStreamSynchronize(compute_);
        cudaStreamDestroy(compute_);
      }
      if (base_) cudaFree(base_);
    } else {
      std::free(base_);
    }
    for (int fd : fd_)
      if (fd >= 0) ::close(fd);
  }

  phobos_status_t setup() {
    for (int t = 0; t < 3; ++t) {
      if (!cfg_.paths[t]) return PHOBOS_ERR_INVALID_VALUE;
      fd_[t] = ::open(cfg_.paths[t], t == PHOBOS_CL_C ? O_RDWR : O_RDONLY);
      if (fd_[t] < 0) return PHOBOS_ERR_CUDA;
      struct stat st;
      if (::fstat(fd_[t], &st) != 0 || st.st_size < 4 * extent_[t][0] * extent_[t][1])
        return PHOBOS_ERR_INVALID_VALUE;
    }
    for (int64_t i = 0; i < h_.n_instr; ++i) {
      const phobos_cl_instr_t &r = recs_[i];
      if (r.row0 + r.rows > extent_[r.tensor][0] || r.col0 + r.cols > extent_[r.tensor][1])
        return PHOBOS_ERR_INVALID_VALUE;
    }
    if (cfg_.arena_bytes < h_.peak) return PHOBOS_ERR_OUT_OF_MEMORY;
    if (!cuda_) {
      if (!hooks_ || !hooks_->host_gemm) return PHOBOS_ERR_INVALID_VALUE;
      base_ = static_cast<char *>(std::malloc(static_cast<size_t>(std::max<int64_t>(cfg_.arena_bytes, 1))));
      return base_ ? PHOBOS_OK : PHOBOS_ERR_OUT_OF_MEMORY;
    }
    if (cudaMalloc(reinterpret_cast<void **>(&base_), static_cast<size_t>(cfg_.arena_bytes)) != cudaSuccess)
      return PHOBOS_ERR_OUT_OF_MEMORY;
    if (cfg_.stream) {
      compute_ = static_cast<cudaStream_t>(cfg_.stream);
    } else {
      if (cudaStreamCreateWithFlags(&compute_, cudaStreamNonBlocking) != cudaSuccess) return PHOBOS_ERR_CUDA;
      own_compute_ = true;
    }
    if (cudaStreamCreateWithFlags(&copy_in_, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&copy_out_, cudaStreamNonBlocking) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    for (int i = 0; i < 2; ++i) {
      if (cudaMallocHost(reinterpret_cast<void **>(&stage_in_[i]), static_cast<size_t>(staging_bytes_)) !=
              cudaSuccess ||
          cudaEventCreateWithFlags(&stage_ev_[i], cudaEventDisableTiming) != cudaSuccess)
        return PHOBOS_ERR_OUT_OF_MEMORY;
    }
    if (cudaMallocHost(reinterpret_cast<void **>(&stage_out_), static_cast<size_t>(staging_bytes_)) !=
        cudaSuccess)
      return PHOBOS_ERR_OUT_OF_MEMORY;
    return PHOBOS_OK;
  }

  phobos_status_t run() {
    int64_t done = 0, next_alloc = 0;
    while (done < h_.n_instr) {
      bool progress = false;
      for (int64_t i = 0; i < h_.n_instr; ++i) {
        if (state_[i] != kPending) continue;
        const phobos_cl_instr_t &r = recs_[i];
        if (r.op == PHOBOS_CL_ALLOC) {
          if (i != first_pending_alloc(next_alloc)) continue;  // list order
        }
        if (!ready(i)) continue;
        bool started = false;
        const phobos_status_t st = issue(i, &started);
        if (st != PHOBOS_OK) return st;
        if (started) progress = true;
      }
      // Device work that has finished.
      for (int64_t i = 0; i < h_.n_instr; ++i) {
        if (state_[i] != kIssued) continue;
        const cudaError_t q = cudaEventQuery(event_[i]);
        if (q == cudaSuccess) {
          state_[i] = kDone;
          progress = true;
        } else if (q != cudaErrorNotReady) {
          return PHOBOS_ERR_CUDA;
        }
      }
      done = 0;
      for (int64_t i = 0; i < h_.n_instr; ++i) done += state_[i] == kDone;
      if (progress) continue;
      // Nothing could start: wait for the oldest device work in flight, or
      // report that the arena cannot hold the next ALLOC.
      int64_t oldest = -1;
      for (int64_t i = 0; i < h_.n_instr && oldest < 0; ++i)
        if (state_[i] == kIssued) oldest = i;
      if (oldest < 0) return PHOBOS_ERR_OUT_OF_MEMORY;
      if (cudaEventSynchronize(event_[oldest]) != cudaSuccess) return PHOBOS_ERR_CUDA;
    }
    return PHOBOS_OK;
  }

 private:
  int64_t first_pending_alloc(int64_t &next_alloc) const {
    while (next_alloc < h_.n_instr &&
           (recs_[next_alloc].op != PHOBOS_CL_ALLOC || state_[next_alloc] != kPending))
      ++next_alloc;
    return next_alloc;
  }

  // LOAD, INIT and STEP chain their device work on events, so they may start
  // once their inputs have started. STORE reads the result on the host and
  // FREE hands memory back, so both wait until their inputs have finished.
  bool ready(int64_t i) const {
    const phobos_cl_instr_t &r = recs_[i];
    const bool need_done = r.op == PHOBOS_CL_STORE || r.op == PHOBOS_CL_FREE;
    for (int32_t k = 0; k < r.dep_count; ++k) {
      const int32_t d = deps_[r.dep_begin + k];
      if (state_[d] == kPending) return false;
      if (need_done && state_[d] != kDone) return false;
    }
    return true;
  }

  float *buffer(int32_t alloc_index) const {
    return reinterpret_cast<float *>(base_ + offset_[alloc_index]);
  }

  // The instruction's device work has been enqueued: record its event.
  phobos_status_t mark_issued(int64_t i, cudaStream_t s) {
    if (!cuda_) {
      state_[i] = kDone;
      return PHOBOS_OK;
    }
    if (!event_[i] && cudaEventCreateWithFlags(&event_[i], cudaEventDisableTiming) != cudaSuccess)
      return PHOBOS_ERR_CUDA;
    if (cudaEventRecord(event_[i], s) != cudaSuccess) return PHOBOS_ERR_CUDA;
    state_[i] = kIssued;
    return PHOBOS_OK;
  }

  phobos_status_t wait_deps(int64_t i, cudaStream_t s) {
    if (!cuda_) return PHOBOS_OK;
    const phobos_cl_instr_t &r = recs_[i];
    for (int32_t k = 0; k < r.dep_count; ++k) {
      const int32_t d = deps_[r.dep_begin + k];
      if (event_[d] && state_[d] != kDone && cudaStreamWaitEvent(s, event_[d], 0) != cudaSuccess)
        return PHOBOS_ERR_CUDA;
    }
    return PHOBOS_OK;
  }

  phobos_status_t issue(int64_t i, bool *started) {
    const phobos_cl_instr_t &r = recs_[i];
    *started = true;
    switch (r.op) {
      case PHOBOS_CL_ALLOC: {
        int64_t off = 0;
        if (!arena_.alloc(4 * r.rows * r.cols, &off)) {
          *started = false;
          return PHOBOS_OK;
        }
        offset_[i] = off;
        state_[i] = kDone;
        return PHOBOS_OK;
      }
      case PHOBOS_CL_LOAD:
        return load(i);
      case PHOBOS_CL_INIT:
        return init(i);
      case PHOBOS_CL_STEP:
        return step(i);
      case PHOBOS_CL_STORE:
        return store(i);
      case PHOBOS_CL_FREE:
        arena_.release(offset_[r.buf], 4 * r.rows * r.cols);
        state_[i] = kDone;
        return PHOBOS_OK;
      default:
        return PHOBOS_ERR_INVALID_VALUE;
    }
  }

  phobos_status_t load(int64_t i) {
    const phobos_cl_instr_t &r = recs_[i];
    const phobos_cl_instr_t &b = recs_[r.buf];
    if (b.rows != r.rows || b.cols != r.cols) return PHOBOS_ERR_INVALID_VALUE;
    float *dst = buffer(r.buf);
    const int fd = fd_[r.tensor];
    const int64_t ld = ld_[r.tensor];
    if (!cuda_) {
      if (!read_rows(fd, ld, r.row0, r.col0, r.cols, 0, r.rows, dst)) return PHOBOS_ERR_CUDA;
      return mark_issued(i, nullptr);
    }
    if (wait_deps(i, copy_in_) != PHOBOS_OK) return PHOBOS_ERR_CUDA;
    const int64_t chunk_rows = std::max<int64_t>(1, staging_bytes_ / (4 * r.cols));
    if (4 * r.cols > staging_bytes_) return PHOBOS_ERR_INVALID_VALUE;
    for (int64_t row = 0; row < r.rows; row += chunk_rows) {
      const int64_t nr = std::min(chunk_rows, r.rows - row);
      const int k = stage_next_;
      stage_next_ ^= 1;
      // The previous copy out of this staging buffer must have finished.
      if (stage_used_[k] && cudaEventSynchronize(stage_ev_[k]) != cudaSuccess) return PHOBOS_ERR_CUDA;
      if (!read_rows(fd, ld, r.row0, r.col0, r.cols, row, nr, stage_in_[k])) return PHOBOS_ERR_CUDA;
      if (cudaMemcpyAsync(dst + row * r.cols, stage_in_[k], static_cast<size_t>(4 * nr * r.cols),
                          cudaMemcpyHostToDevice, copy_in_) != cudaSuccess ||
          cudaEventRecord(stage_ev_[k], copy_in_) != cudaSuccess)
        return PHOBOS_ERR_CUDA;
      stage_used_[k] = true;
    }
    return mark_issued(i, copy_in_);
  }

  phobos_status_t init(int64_t i) {
    const phobos_cl_instr_t &r = recs_[i];
    float *c = buffer(r.buf);
    if (!cuda_) {
      for (int64_t e = 0; e < r.rows * r.cols; ++e) c[e] = h_.beta == 0.0f ? 0.0f : h_.beta * c[e];
      return mark_issued(i, nullptr);
    }
    if (wait_deps(i, compute_) != PHOBOS_OK) return PHOBOS_ERR_CUDA;
    // K = 0: C = beta*C, and zeros without reading C when beta == 0.
    const phobos_status_t st = phobos_sgemm_ex(r.rows, r.cols, 0, 1.0f, nullptr, 1, nullptr, r.cols,
                                               h_.beta, c, r.cols, compute_, PHOBOS_MATH_DEFAULT, nullptr);
    if (st != PHOBOS_OK) return st;
    return mark_issued(i, compute_);
  }

  phobos_status_t step(int64_t i) {
    const phobos_cl_instr_t &r = recs_[i];
    const phobos_cl_instr_t &ca = recs_[r.buf], &aa = recs_[r.buf_a], &ba = recs_[r.buf_b];
    if (aa.rows != ca.rows || ba.cols != ca.cols || aa.cols != ba.rows) return PHOBOS_ERR_INVALID_VALUE;
    const int64_t kc = aa.cols;
    float *c = buffer(r.buf);
    const float *a = buffer(r.buf_a), *b = buffer(r.buf_b);
    if (!cuda_) {
      if (hooks_->host_gemm(hooks_->ctx, ca.rows, ca.cols, kc, h_.alpha, a, kc, b, ca.cols, 1.0f, c,
                            ca.cols) != 0)
        return PHOBOS_ERR_INVALID_VALUE;
      return mark_issued(i, nullptr);
    }
    if (wait_deps(i, compute_) != PHOBOS_OK) return PHOBOS_ERR_CUDA;
    // The step leaf: C += alpha * A_chunk * B_chunk (implicit beta = 1).  Pods
    // may run as ranks of a multi-GPU job, so leaves always take the automatic
    // plan, which never turns on TMA multicast (and the library refuses a
    // multicast plan in such a rank).
    const phobos_status_t st = phobos_sgemm_ex(ca.rows, ca.cols, kc, h_.alpha, a, kc, b, ca.cols, 1.0f, c,
                                               ca.cols, compute_, PHOBOS_MATH_DEFAULT, nullptr);
    if (st != PHOBOS_OK) return st;
    return mark_issued(i, compute_);
  }

  // Write the buffer's tile through `write(r, nr, host_rows)` in chunks.
  template <class Write>
  phobos_status_t drain(const phobos_cl_instr_t &r, const float *src, Write write) {
    if (!cuda_) return write(0, r.rows, src) ? PHOBOS_OK : PHOBOS_ERR_CUDA;
    if (4 * r.cols > staging_bytes_) return PHOBOS_ERR_INVALID_VALUE;
    const int64_t chunk_rows = std::max<int64_t>(1, staging_bytes_ / (4 * r.cols));
    for (int64_t row = 0; row < r.rows; row += chunk_rows) {
      const int64_t nr = std::min(chunk_rows, r.rows - row);
      if (cudaMemcpyAsync(stage_out_, src + row * r.cols, static_cast<size_t>(4 * nr * r.cols),
                          cudaMemcpyDeviceToHost, copy_out_) != cudaSuccess ||
          cudaStreamSynchronize(copy_out_) != cudaSuccess)
        return PHOBOS_ERR_CUDA;
      if (!write(row, nr, stage_out_)) return PHOBOS_ERR_CUDA;
    }
    return PHOBOS_OK;
  }

  phobos_status_t store(int64_t i) {
    const phobos_cl_instr_t &r = recs_[i];
    const float *src = buffer(r.buf);
    const std::string side = side_path(cfg_.paths[PHOBOS_CL_C], r.tile);
    // Phase 1: the whole tile into its side file.
    const int sfd = ::open(side.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (sfd < 0) return PHOBOS_ERR_CUDA;
    phobos_status_t st = drain(r, src, [&](int64_t row, int64_t nr, const float *h) {
      return pwrite_all(sfd, h, 4 * nr * r.cols, 4 * row * r.cols);
    });
    ::close(sfd);
    if (st != PHOBOS_OK) return st;
    if (hooks_ && hooks_->on_staged && hooks_->on_staged(hooks_->ctx, r.tile) != 0)
      return PHOBOS_ERR_INVALID_VALUE;
    // Phase 2: into the output.
    st = drain(r, src, [&](int64_t row, int64_t nr, const float *h) {
      return write_rows(fd_[PHOBOS_CL_C], ld_[PHOBOS_CL_C], r.row0, r.col0, r.cols, row, nr, h);
    });
    if (st != PHOBOS_OK) return st;
    if (hooks_ && hooks_->on_stored && hooks_->on_stored(hooks_->ctx, r.tile) != 0)
      return PHOBOS_ERR_INVALID_VALUE;
    ::unlink(side.c_str());
    state_[i] = kDone;
    return PHOBOS_OK;
  }

  const SegmentHeader h_;
  const phobos_cl_instr_t *recs_;
  const int32_t *deps_;
  const phobos_pod_config_t cfg_;
  const phobos_pod_hooks_t *hooks_;
  const bool cuda_;
  Arena arena_;
  std::vector<int> state_;
  std::vector<int64_t> offset_;
  std::vector<cudaEvent_t> event_;
  int64_t ld_[3];
  int64_t extent_[3][2];
  int fd_[3] = {-1, -1, -1};
  char *base_ = nullptr;
  int64_t staging_bytes_ = kDefaultStaging;
  cudaStream_t compute_ = nullptr, copy_in_ = nullptr, copy_out_ = nullptr;
  bool own_compute_ = false;
  float *stage_in_[2] = {nullptr, nullptr};
  cudaEvent_t stage_ev_[2] = {nullptr, nullptr};
  bool stage_used_[2] = {false, false};
  int stage_next_ = 0;
  float *stage_out_ = nullptr;
};

}  // namespace
}  // namespace cluster
}  // namespace phobos

extern "C" phobos_status_t phobos_pod_run(const void *segment, size_t bytes,
                                          const phobos_pod_config_t *cfg,
                                          const phobos_pod_hooks_t *hooks) {
  using namespace phobos::cluster;
  SegmentHeader h;
  const phobos_cl_instr_t *recs = nullptr;
  const int32_t *deps = nullptr;
  if (!cfg || !parse_segment(segment, bytes, &h, &recs, &deps)) return PHOBOS_ERR_INVALID_VALUE;
  if (cfg->device != PHOBOS_POD_CUDA && cfg->device != PHOBOS_POD_HOST) return PHOBOS_ERR_INVALID_VALUE;
  if (cfg->arena_bytes <= 0) return PHOBOS_ERR_INVALID_VALUE;
  Pod pod(h, recs, deps, *cfg, hooks);
  phobos_status_t st = pod.setup();
  if (st != PHOBOS_OK) return st;
  return pod.run();
}
