// Shared between the cluster planner and the pod executor: the segment blob's
// header and its checked reader.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/phobos_cluster.h"

namespace phobos {
namespace cluster {

constexpr uint32_t kMagic = 0x4c434850u;  // "PHCL"
constexpr uint32_t kVersion = 1;

// Self-contained header of a segment blob; the instructions and the
// dependency list follow it.
struct SegmentHeader {
  uint32_t magic, version;
  int32_t node, reserved;
  int64_t n_instr, n_deps;
  int64_t M, N, K, sm, sn, sk;
  float alpha, beta;
  int64_t peak, load, store, flops, outputs;
};

// Checks a segment blob and returns its header, instructions and dependency
// list, or false when it is malformed: wrong magic or sizes, an unknown op or
// tensor, an empty region, or a buffer or dependency index that does not
// point backwards to the right kind of instruction.
bool parse_segment(const void *segment, size_t bytes, SegmentHeader *h,
                   const phobos_cl_instr_t **recs, const int32_t **deps);

}  // namespace cluster
}  // namespace phobos
