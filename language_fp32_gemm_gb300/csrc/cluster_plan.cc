// Planner of the super-tile cluster runtime: from a problem and a set of live
// nodes to one instruction list ("segment") per node.
//
// The program each node runs is the cluster-IR of "Show HN: Phobos", section
// "The DAG Compiler". For an output super-tile (pm, pn):
//   - the accumulator is seeded with beta*C[pm, pn] (version 0), by the init leaf;
//   - for every K chunk kt, version kt+1 = version kt + alpha*A[pm, kt]*B[kt, pn],
//     by a step leaf that reads and writes the accumulator in place;
//   - the last version is written back to C[pm, pn].
// Unrolled, that gives ALLOC, LOAD, INIT, STEP, STORE instructions. Each
// buffer's users are known exactly, so a backward pass over the list puts
// every FREE right after the last use of its buffer. The FREE waits for all
// of those users: there is no lifetime syntax, lifetimes fall out of the
// graph ("The DAG Compiler").
//
// Placement and tuning follow the "@cluster" attribute page, "What runs
// today":
//   - output super-tiles are dealt round robin over the nodes by their row-major index;
//   - without autotune each axis takes the first value of its range;
//   - with it, every combination on the doubling ladder is planned, and those
//     whose list-order peak does not fit a node's budget, or that leave a node
//     without a super-tile, are dropped;
//   - the rest are ranked by a model of the busiest node's compute and storage
//     time. Nothing is run to measure.
// The pages require every dimension to be a whole multiple of its super-tile;
// here the last super-tile of an axis may be shorter (the leaves accept any size).

#include <algorithm>
#include <cstring>
#include <limits>
#include <new>
#include <vector>

#include "../../include/phobos_cluster.h"
#include "cluster_internal.h"

namespace phobos {
namespace cluster {
namespace {

struct Instr {
  phobos_cl_instr_t rec;
  std::vector<int32_t> deps;
};

struct Segment {
  int32_t node = 0;
  std::vector<Instr> ins;
  int64_t peak = 0, load = 0, store = 0, flops = 0, outputs = 0;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace cluster
}  // namespace phobos

struct phobos_cl_plan {
  phobos_cl_job_t job;
  int64_t sm = 0, sn = 0, sk = 0;
  std::vector<phobos::cluster::Segment> segs;  // indexed by node
};

namespace phobos {
namespace cluster {
namespace {

class Builder {
 public:
  Builder(const phobos_cl_job_t &job, int64_t sm, int64_t sn, int64_t sk)
      : job_(job), sm_(sm), sn_(sn), sk_(sk) {}

  // Append the program of output super-tile (pm, pn) to `seg`.
  void output(Segment &seg, int64_t pm, int64_t pn) const {
    const int64_t gk = ceil_div(job_.K, sk_);
    const int64_t r0 = pm * sm_, c0 = pn * sn_;
    const int64_t rows = std::min(sm_, job_.M - r0), cols = std::min(sn_, job_.N - c0);
    const int32_t c = emit(seg, PHOBOS_CL_ALLOC, PHOBOS_CL_C, phobos_cl_tile_id(PHOBOS_CL_C, 0, pm, pn),
                           r0, c0, rows, cols, -1, -1, -1, {});
    int32_t last = c;
    if (job_.beta != 0.0f)
      last = emit(seg, PHOBOS_CL_LOAD, PHOBOS_CL_C, phobos_cl_tile_id(PHOBOS_CL_C, 0, pm, pn), r0, c0,
                  rows, cols, c, -1, -1, {c});
    last = emit(seg, PHOBOS_CL_INIT, PHOBOS_CL_C, phobos_cl_tile_id(PHOBOS_CL_C, 0, pm, pn), r0, c0,
                rows, cols, c, -1, -1, {last});
    for (int64_t kt = 0; kt < gk; ++kt) {
      const int64_t k0 = kt * sk_, kc = std::min(sk_, job_.K - k0);
      const uint64_t ta = phobos_cl_tile_id(PHOBOS_CL_A, 0, pm, kt);
      const uint64_t tb = phobos_cl_tile_id(PHOBOS_CL_B, 0, kt, pn);
      const int32_t a = emit(seg, PHOBOS_CL_ALLOC, PHOBOS_CL_A, ta, r0, k0, rows, kc, -1, -1, -1, {});
      const int32_t la = emit(seg, PHOBOS_CL_LOAD, PHOBOS_CL_A, ta, r0, k0, rows, kc, a, -1, -1, {a});
      const int32_t b = emit(seg, PHOBOS_CL_ALLOC, PHOBOS_CL_B, tb, k0, c0, kc, cols, -1, -1, -1, {});
      const int32_t lb = emit(seg, PHOBOS_CL_LOAD, PHOBOS_CL_B, tb, k0, c0, kc, cols, b, -1, -1, {b});
      last = emit(seg, PHOBOS_CL_STEP, PHOBOS_CL_C, phobos_cl_tile_id(PHOBOS_CL_C, kt + 1, pm, pn), r0,
                  c0, rows, cols, c, a, b, {last, la, lb});
      seg.flops += 2 * rows * cols * kc;
    }
    emit(seg, PHOBOS_CL_STORE, PHOBOS_CL_C, phobos_cl_tile_id(PHOBOS_CL_C, gk, pm, pn), r0, c0, rows,
         cols, c, -1, -1, {last});
    seg.outputs += 1;
  }

  // The backward pass: the last use of every buffer gets a FREE right after
  // it, depending on every instruction that uses the buffer. Then the
  // list-order figures (peak arena bytes, bytes loaded and stored).
  static void place_frees(Segment &seg) {
    const int n = static_cast<int>(seg.ins.size());
    std::vector<std::vector<int32_t>> users(n);
    auto use = [&](int32_t buf, int32_t i) {
      if (buf >= 0) users[buf].push_back(i);
    };
    for (int i = 0; i < n; ++i) {
      const phobos_cl_instr_t &r = seg.ins[i].rec;
      if (r.op == PHOBOS_CL_ALLOC) continue;
      use(r.buf, i);
      use(r.buf_a, i);
      use(r.buf_b, i);
    }
    std::vector<std::vector<int32_t>> frees_after(n);  // buffers whose last use is i
    std::vector<bool> seen(n, false);
    for (int i = n - 1; i >= 0; --i) {
      const phobos_cl_instr_t &r = seg.ins[i].rec;
      if (r.op == PHOBOS_CL_ALLOC) continue;
      for (int32_t buf : {r.buf, r.buf_a, r.buf_b})
        if (buf >= 0 && !seen[buf]) {
          seen[buf] = true;
          frees_after[i].push_back(buf);
        }
    }
    // Rebuild the list with the FREEs in place; indices shift, so remap.
    std::vector<Instr> out;
    std::vector<int32_t> remap(n, -1);
    std::vector<std::pair<int32_t, int32_t>> pending;  // (new FREE index, old buffer index)
    for (int i = 0; i < n; ++i) {
      remap[i] = static_cast<int32_t>(out.size());
      out.push_back(seg.ins[i]);
      for (int32_t buf : frees_after[i]) {
        const phobos_cl_instr_t &b = seg.ins[buf].rec;
        Instr f;
        f.rec = b;
        f.rec.op = PHOBOS_CL_FREE;
        f.rec.buf = buf;  // remapped below
        f.rec.buf_a = f.rec.buf_b = -1;
        f.deps = users[buf];  // remapped below
        pending.emplace_back(static_cast<int32_t>(out.size()), buf);
        out.push_back(f);
      }
    }
    for (Instr &in : out) {
      if (in.rec.op == PHOBOS_CL_FREE) continue;
      for (int32_t &d : in.deps) d = remap[d];
      if (in.rec.op == PHOBOS_CL_ALLOC) {
        in.rec.buf = -1;
      } else {
        if (in.rec.buf >= 0) in.rec.buf = remap[in.rec.buf];
        if (in.rec.buf_a >= 0) in.rec.buf_a = remap[in.rec.buf_a];
        if (in.rec.buf_b >= 0) in.rec.buf_b = remap[in.rec.buf_b];
      }
    }
    for (auto &pf : pending) {
      Instr &f = out[pf.first];
      f.rec.buf = remap[pf.second];
      for (int32_t &d : f.deps) d = remap[d];
    }
    for (size_t i = 0; i < out.size(); ++i)
      if (out[i].rec.op == PHOBOS_CL_ALLOC) out[i].rec.buf = static_cast<int32_t>(i);
    seg.ins.swap(out);

    int64_t held = 0;
    seg.peak = seg.load = seg.store = 0;
    for (const Instr &in : seg.ins) {
      const int64_t bytes = 4 * in.rec.rows * in.rec.cols;
      switch (in.rec.op) {
        case PHOBOS_CL_ALLOC: held += bytes; seg.peak = std::max(seg.peak, held); break;
        case PHOBOS_CL_FREE: held -= bytes; break;
        case PHOBOS_CL_LOAD: seg.load += bytes; break;
        case PHOBOS_CL_STORE: seg.store += bytes; break;
        default: break;
      }
    }
  }

 private:
  int32_t emit(Segment &seg, int op, int tensor, uint64_t tile, int64_t row0, int64_t col0,
               int64_t rows, int64_t cols, int32_t buf, int32_t buf_a, int32_t buf_b,
               std::vector<int32_t> deps) const {
    Instr in;
    std::memset(&in.rec, 0, sizeof(in.rec));
    in.rec.op = op;
    in.rec.tensor = tensor;
    in.rec.tile = tile;
    in.rec.row0 = row0;
    in.rec.col0 = col0;
    in.rec.rows = rows;
    in.rec.cols = cols;
    in.rec.buf = buf;
    in.rec.buf_a = buf_a;
    in.rec.buf_b = buf_b;
    in.deps = std::move(deps);
    seg.ins.push_back(std::move(in));
    return static_cast<int32_t>(seg.ins.size() - 1);
  }

  const phobos_cl_job_t &job_;
  int64_t sm_, sn_, sk_;
};

// Build every node's segment for the given super-tile sizes.
void build(const phobos_cl_job_t &job, int64_t sm, int64_t sn, int64_t sk,
           const std::vector<int32_t> &outputs, const std::vector<int32_t> &live,
           std::vector<Segment> &segs) {
  segs.assign(job.nodes, Segment());
  for (int32_t n = 0; n < job.nodes; ++n) segs[n].node = n;
  const int64_t gn = ceil_div(job.N, sn);
  Builder b(job, sm, sn, sk);
  for (size_t i = 0; i < outputs.size(); ++i) {
    const int32_t node = live[i % live.size()];
    b.output(segs[node], outputs[i] / gn, outputs[i] % gn);
  }
  for (Segment &s : segs) Builder::place_frees(s);
}

std::vector<int64_t> ladder(int64_t lo, int64_t hi, int64_t extent) {
  std::vector<int64_t> v;
  for (int64_t x = lo; x <= hi; x *= 2) {
    const int64_t c = std::min(x, extent);
    if (v.empty() || v.back() != c) v.push_back(c);
    if (x > std::numeric_limits<int64_t>::max() / 2) break;
  }
  return v;
}

// The cost model: the busiest node's leaf time plus its storage time.
double busiest_node_seconds(const phobos_cl_job_t &job, const std::vector<Segment> &segs) {
  double worst = 0.0;
  for (const Segment &s : segs) {
    const double t = static_cast<double>(s.flops) / (job.node_tflops * 1e12) +
                     static_cast<double>(s.load + s.store) / (job.storage_gbs * 1e9);
    worst = std::max(worst, t);
  }
  return worst;
}

}  // namespace
}  // namespace cluster
}  // namespace phobos

using namespace phobos::cluster;

extern "C" {

uint64_t phobos_cl_tile_id(int32_t tensor, int64_t version, int64_t row, int64_t col) {
  return (static_cast<uint64_t>(tensor & 3) << 62) |
         ((static_cast<uint64_t>(version) & ((1ull << 20) - 1)) << 42) |
         ((static_cast<uint64_t>(row) & ((1ull << 21) - 1)) << 21) |
         (static_cast<uint64_t>(col) & ((1ull << 21) - 1));
}

phobos_status_t phobos_cl_plan(const phobos_cl_job_t *job, const int32_t *outputs,
                               int64_t n_outputs, const int32_t *live, int32_t n_live,
                               int64_t super_out[3], phobos_cl_plan_t **plan) {
  if (!job || !plan) return PHOBOS_ERR_INVALID_VALUE;
  *plan = nullptr;
  const phobos_cl_job_t &j = *job;
  if (j.M <= 0 || j.N <= 0 || j.K <= 0 || j.nodes <= 0 || j.node_budget_bytes <= 0)
    return PHOBOS_ERR_INVALID_VALUE;
  const int64_t extent[3] = {j.M, j.N, j.K};
  for (int a = 0; a < 3; ++a)
    if (j.super_lo[a] <= 0 || j.super_hi[a] < j.super_lo[a]) return PHOBOS_ERR_INVALID_VALUE;
  if (j.autotune && (!(j.node_tflops > 0.0) || !(j.storage_gbs > 0.0)))
    return PHOBOS_ERR_INVALID_VALUE;

  std::vector<int32_t> nodes;
  if (live) {
    if (n_live <= 0) return PHOBOS_ERR_INVALID_VALUE;
    std::vector<bool> used(j.nodes, false);
    for (int32_t i = 0; i < n_live; ++i) {
      if (live[i] < 0 || live[i] >= j.nodes || used[live[i]]) return PHOBOS_ERR_INVALID_VALUE;
      used[live[i]] = true;
      nodes.push_back(live[i]);
    }
  } else {
    for (int32_t n = 0; n < j.nodes; ++n) nodes.push_back(n);
  }

  auto output_list = [&](int64_t sm, int64_t sn, std::vector<int32_t> &out) -> bool {
    const int64_t total = ceil_div(j.M, sm) * ceil_div(j.N, sn);
    if (total > std::numeric_limits<int32_t>::max()) return false;
    out.clear();
    if (!outputs) {
      for (int64_t s = 0; s < total; ++s) out.push_back(static_cast<int32_t>(s));
      return true;
    }
    for (int64_t i = 0; i < n_outputs; ++i) {
      if (outputs[i] < 0 || outputs[i] >= total) return false;
      if (i > 0 && outputs[i] <= outputs[i - 1]) return false;  // increasing, no repeats
      out.push_back(outputs[i]);
    }
    return true;
  };

  std::vector<int64_t> cand[3];
  for (int a = 0; a < 3; ++a) {
    cand[a] = j.autotune ? ladder(j.super_lo[a], j.super_hi[a], extent[a])
                         : std::vector<int64_t>{std::min(j.super_lo[a], extent[a])};
  }

  phobos_cl_plan_t *best = nullptr;
  double best_cost = 0.0;
  bool best_covers = false;
  bool any_valid_outputs = false;
  for (int64_t sm : cand[0])
    for (int64_t sn : cand[1])
      for (int64_t sk : cand[2]) {
        std::vector<int32_t> outs;
        if (!output_list(sm, sn, outs)) continue;
        any_valid_outputs = true;
        phobos_cl_plan_t *p = new (std::nothrow) phobos_cl_plan_t();
        if (!p) {
          delete best;
          return PHOBOS_ERR_OUT_OF_MEMORY;
        }
        p->job = j;
        p->sm = sm;
        p->sn = sn;
        p->sk = sk;
        build(j, sm, sn, sk, outs, nodes, p->segs);
        bool fits = true;
        for (const Segment &s : p->segs) fits = fits && s.peak <= j.node_budget_bytes;
        // Every live node gets a super-tile; where no candidate manages that
        // (fewer outputs than nodes), the fitting candidates are still ranked.
        const bool covers = outs.size() >= nodes.size();
        const double cost = j.autotune ? busiest_node_seconds(j, p->segs) : 0.0;
        const bool better = fits && (!best || (covers && !best_covers) ||
                                     (covers == best_covers && cost < best_cost));
        if (better) {
          delete best;
          best = p;
          best_cost = cost;
          best_covers = covers;
        } else {
          delete p;
        }
      }
  if (!any_valid_outputs) return PHOBOS_ERR_INVALID_VALUE;
  if (!best) return PHOBOS_ERR_OUT_OF_MEMORY;
  if (super_out) {
    super_out[0] = best->sm;
    super_out[1] = best->sn;
    super_out[2] = best->sk;
  }
  *plan = best;
  return PHOBOS_OK;
}

void phobos_cl_plan_free(phobos_cl_plan_t *plan) { delete plan; }

phobos_status_t phobos_cl_segment_size(const phobos_cl_plan_t *plan, int32_t node, size_t *bytes) {
  if (!plan || !bytes || node < 0 || node >= static_cast<int32_t>(plan->segs.size()))
    return PHOBOS_ERR_INVALID_VALUE;
  const Segment &s = plan->segs[node];
  size_t deps = 0;
  for (const Instr &in : s.ins) deps += in.deps.size();
  *bytes = sizeof(SegmentHeader) + s.ins.size() * sizeof(phobos_cl_instr_t) + deps * sizeof(int32_t);
  return PHOBOS_OK;
}

phobos_status_t phobos_cl_segment_write(const phobos_cl_plan_t *plan, int32_t node, void *out,
                                        size_t bytes) {
  size_t need = 0;
  phobos_status_t st = phobos_cl_segment_size(plan, node, &need);
  if (st != PHOBOS_OK) return st;
  if (!out || bytes < need) return PHOBOS_ERR_INVALID_VALUE;
  const Segment &s = plan->segs[node];
  SegmentHeader h;
  std::memset(&h, 0, sizeof(h));
  h.magic = kMagic;
  h.version = kVersion;
  h.node = node;
  h.n_instr = static_cast<int64_t>(s.ins.size());
  h.M = plan->job.M;
  h.N = plan->job.N;
  h.K = plan->job.K;
  h.sm = plan->sm;
  h.sn = plan->sn;
  h.sk = plan->sk;
  h.alpha = plan->job.alpha;
  h.beta = plan->job.beta;
  h.peak = s.peak;
  h.load = s.load;
  h.store = s.store;
  h.flops = s.flops;
  h.outputs = s.outputs;
  char *p = static_cast<char *>(out);
  phobos_cl_instr_t *recs = reinterpret_cast<phobos_cl_instr_t *>(p + sizeof(h));
  int32_t *deps = reinterpret_cast<int32_t *>(recs + s.ins.size());
  int32_t nd = 0;
  for (size_t i = 0; i < s.ins.size(); ++i) {
    phobos_cl_instr_t r = s.ins[i].rec;
    r.dep_begin = nd;
    r.dep_count = static_cast<int32_t>(s.ins[i].deps.size());
    std::memcpy(recs + i, &r, sizeof(r));
    for (int32_t d : s.ins[i].deps) std::memcpy(deps + nd++, &d, sizeof(d));
  }
  h.n_deps = nd;
  std::memcpy(p, &h, sizeof(h));
  return PHOBOS_OK;
}

}  // extern "C"

// ------------------------------------------------------------ segment reading

namespace phobos {
namespace cluster {

bool parse_segment(const void *segment, size_t bytes, SegmentHeader *h,
                   const phobos_cl_instr_t **recs, const int32_t **deps) {
  if (!segment || bytes < sizeof(SegmentHeader)) return false;
  std::memcpy(h, segment, sizeof(*h));
  if (h->magic != kMagic || h->version != kVersion || h->n_instr < 0 || h->n_deps < 0)
    return false;
  const size_t need = sizeof(SegmentHeader) + static_cast<size_t>(h->n_instr) * sizeof(phobos_cl_instr_t) +
                      static_cast<size_t>(h->n_deps) * sizeof(int32_t);
  if (bytes < need) return false;
  const char *p = static_cast<const char *>(segment);
  *recs = reinterpret_cast<const phobos_cl_instr_t *>(p + sizeof(SegmentHeader));
  *deps = reinterpret_cast<const int32_t *>(*recs + h->n_instr);
  for (int64_t i = 0; i < h->n_instr; ++i) {
    const phobos_cl_instr_t &r = (*recs)[i];
    if (r.op < PHOBOS_CL_ALLOC || r.op > PHOBOS_CL_FREE) return false;
    if (r.tensor < PHOBOS_CL_A || r.tensor > PHOBOS_CL_C) return false;
    if (r.rows <= 0 || r.cols <= 0 || r.row0 < 0 || r.col0 < 0) return false;
    if (r.dep_begin < 0 || r.dep_count < 0 || r.dep_begin + static_cast<int64_t>(r.dep_count) > h->n_deps)
      return false;
    for (int32_t k = 0; k < r.dep_count; ++k) {
      const int32_t d = (*deps)[r.dep_begin + k];
      if (d < 0 || d >= i) return false;  // dependencies point backwards
    }
    auto buf_ok = [&](int32_t b, bool required) {
      if (b < 0) return !required;
      return b < i && (*recs)[b].op == PHOBOS_CL_ALLOC;
    };
    switch (r.op) {
      case PHOBOS_CL_ALLOC:
        if (r.buf != i) return false;
        break;
      case PHOBOS_CL_STEP:
        if (!buf_ok(r.buf, true) || !buf_ok(r.buf_a, true) || !buf_ok(r.buf_b, true)) return false;
        break;
      default:
        if (!buf_ok(r.buf, true)) return false;
        break;
    }
  }
  return true;
}

}  // namespace cluster
}  // namespace phobos

extern "C" {

phobos_status_t phobos_cl_segment_info(const void *segment, size_t bytes,
                                       phobos_cl_segment_info_t *info) {
  SegmentHeader h;
  const phobos_cl_instr_t *recs = nullptr;
  const int32_t *deps = nullptr;
  if (!info || !parse_segment(segment, bytes, &h, &recs, &deps)) return PHOBOS_ERR_INVALID_VALUE;
  std::memset(info, 0, sizeof(*info));
  info->instrs = h.n_instr;
  for (int64_t i = 0; i < h.n_instr; ++i) info->op_count[recs[i].op] += 1;
  info->peak_bytes = h.peak;
  info->load_bytes = h.load;
  info->store_bytes = h.store;
  info->flops = h.flops;
  info->outputs = h.outputs;
  return PHOBOS_OK;
}

phobos_status_t phobos_cl_segment_instr(const void *segment, size_t bytes, int64_t i,
                                        phobos_cl_instr_t *out) {
  SegmentHeader h;
  const phobos_cl_instr_t *recs = nullptr;
  const int32_t *deps = nullptr;
  if (!out || !parse_segment(segment, bytes, &h, &recs, &deps) || i < 0 || i >= h.n_instr)
    return PHOBOS_ERR_INVALID_VALUE;
  std::memcpy(out, recs + i, sizeof(*out));
  return PHOBOS_OK;
}

phobos_status_t phobos_cl_segment_dep(const void *segment, size_t bytes, int64_t j, int32_t *out) {
  SegmentHeader h;
  const phobos_cl_instr_t *recs = nullptr;
  const int32_t *deps = nullptr;
  if (!out || !parse_segment(segment, bytes, &h, &recs, &deps) || j < 0 || j >= h.n_deps)
    return PHOBOS_ERR_INVALID_VALUE;
  *out = deps[j];
  return PHOBOS_OK;
}

}  // extern "C"
